// Chunked prefill over the position-free paged cache, warp-specialised tcgen05
// form (two 128-row query tiles per CTA sharing every rotated key tile).
//
// Method (MiniPIC summary, gist.science 2606.13126, section 2.1): stored keys
// are unrotated; each key is rotated at its logical position
// pi(j) = start[r][j / 16] + j % 16 with cos/sin values and multiply-adds per
// element, then softmax attention runs.  A request's query chunk (the last
// q_len of its kv_len keys) attends causally: chunk query i sees keys
// j <= kv_len - q_len + i.
//
// CTA = (request r, kv head hk, query-tile pair): query tile i (i = 0, 1) holds
// TQ = 128 / G consecutive tokens x the G query heads of kv head hk.  Roles:
//   warps 0-3   softmax of query tile 0 (thread = TMEM lane = query row)
//   warps 4-7   softmax of query tile 1
//   warps 8-13  query preparation, then rotation of every staged key tile
//   warp 14     TMA producer (K~ tiles + block-start cos/sin rows, V tiles)
//   warp 15     TMEM allocation and tcgen05 MMA issue
// A key tile is NB blocks (16 NB keys); K~ has NSK stages and V NSV stages, so
// a stage freed by the products of tile t is refilled while tiles t+1..t+NSK-1
// are in flight.  Per key tile t the MMA warp issues
//   S0 = Q0 K_t^T, S1 = Q1 K_t^T, then O0 += P0 V_t, S0' = Q0 K_{t+1}^T,
//   O1 += P1 V_t, S1' = Q1 K_{t+1}^T ...
// so that each softmax warpgroup works on its tile while the tensor core runs
// the other tile's products.  S/P share TMEM columns (P = bf16 over S), O is
// accumulated in TMEM and rescaled only when a row max grows by more than 2^8.
#pragma once

#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace minipic {
namespace prefill2_impl {

using ptx::U4;

constexpr int kSoftThreads = 256;                 // two softmax warpgroups
constexpr int kRotBase = 256;                     // first thread of the six rotation warps
constexpr int kRotThreads = 192;
constexpr int kTmaWarp = 14, kMmaWarp = 15;
constexpr int kThreads = 16 * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;

constexpr int kMaskRing = 8;  // key-valid masks of tiles t & 7

// Shared memory, barriers and TMEM plan of one CTA.
// Default tile plan: 96-key tiles, four K~ stages, two V stages (about 222 KB
// of shared memory for d = 128).
constexpr int kNB = 6, kNSK = 4, kNSV = 2;

template <int D, int NB = kNB, int NSK = kNSK, int NSV = kNSV>
struct PG2 {
  // a mask slot is rewritten for tile t + kMaskRing once K~ stage of tile t + kMaskRing - NSK
  // is free, i.e. both softmax groups are past tile t + kMaskRing - NSK - 1 >= t
  static_assert(NB % 2 == 0 && NSK >= NSV && NSV >= 2 && kMaskRing > NSK && (8 * NB) % 16 == 0, "tile plan");
  static constexpr int BN = 16 * NB;                   // keys per tile
  static constexpr int HALVES = D / 64;
  static constexpr int QTILE = HALVES * 128 * 128;     // one 128-row query tile
  static constexpr int KTILE = HALVES * BN * 128;      // one K or V tile
  static constexpr int ROWB = 4 * D;                   // one cos|sin table row
  static constexpr int OFF_Q = 0;                      // [2] query tiles
  static constexpr int OFF_K = OFF_Q + 2 * QTILE;      // [NSK] K stages
  static constexpr int OFF_V = OFF_K + NSK * KTILE;    // [NSV] V stages
  static constexpr int OFF_RS = OFF_V + NSV * KTILE;   // [NSK][NB] block-start rows
  static constexpr int OFF_META = OFF_RS + NSK * NB * ROWB;  // [NSK] int start[NB], flag[NB], vblock[NB]
  static constexpr int OFF_MASK = OFF_META + NSK * 3 * NB * 4;  // [ring][NB] uint16 key-valid bits
  // barriers
  static constexpr int B_Q = 0, B_KFULL = 1, B_KROT = B_KFULL + NSK, B_KFREE = B_KROT + NSK;
  static constexpr int B_VFULL = B_KFREE + NSK, B_VFREE = B_VFULL + NSV, B_S = B_VFREE + NSV, B_P = B_S + 2;
  static constexpr int B_ODONE = B_P + 2, B_MASK = B_ODONE + 1, NBARS = B_MASK + kMaskRing;
  static constexpr int OFF_BAR = (OFF_MASK + kMaskRing * NB * 2 + 15) / 16 * 16;
  static constexpr int OFF_TSLOT = OFF_BAR + NBARS * 8;
  static constexpr int TOTAL = OFF_TSLOT + 16;
  // rotation split: thread = (frequency group of 8, slot pair, block group)
  static constexpr int NFG = D / 16;
  static constexpr int BG = kRotThreads / (NFG * 8);   // block groups (3 for d 128, 6 for d 64)
  static constexpr int BPG = NB / BG;                  // blocks per group
  static_assert(BG * NFG * 8 == kRotThreads && NB % BG == 0, "rotation split");
  // S_i at [128 i, 128 i + BN), P_i (bf16 pairs) over its first BN / 2 columns,
  // O_i at [256 + 128 i, 256 + 128 i + D)
  static constexpr uint32_t TCOLS = 512;
  static_assert(BN <= 128 && BN % 32 == 0, "TMEM plan");
  static_assert(BN <= 128 && TOTAL + 1024 <= 232448, "tile plan");
};

struct PrefillLaunch2 {
  PrefillArgs a;
  int tq;  // tokens per 128-row query tile (= 128 / G)
};

__device__ __forceinline__ uint32_t swz(int key, int chunk) {
  return (uint32_t)(key * 128 + ((chunk ^ (key & 7)) << 4));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void sts128(uint32_t addr, const U4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Rotate a pair of 8-element chunks (bf16 in) and pack the result: f16 for the
// rotated product (ROPE), bf16 unchanged otherwise.
__device__ __forceinline__ void rot_pack(U4& x, U4& y, const uint64_t (&c2)[4], const uint64_t (&s2)[4]) {
  uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t xv = ptx::bf2_to_f2(xw[k]), yv = ptx::bf2_to_f2(yw[k]);
    xw[k] = ptx::f2_to_h2(ptx::sub2(ptx::mul2(xv, c2[k]), ptx::mul2(yv, s2[k])));
    yw[k] = ptx::f2_to_h2(ptx::fma2(xv, s2[k], ptx::mul2(yv, c2[k])));
  }
  x = U4{xw[0], xw[1], xw[2], xw[3]};
  y = U4{yw[0], yw[1], yw[2], yw[3]};
}

// One CTA computes query-tile pair `pair` of request r and kv head hk and
// loads every K~/V box it reads itself.  vmap_p is the block view of the V pool
// (make_pool_block_map).
template <int D, bool ROPE, int NB = kNB, int NSK = kNSK, int NSV = kNSV>
__device__ __forceinline__ void prefill2_cta(const CUtensorMap* kmap_p, const CUtensorMap* vmap_p,
                                             const PrefillLaunch2& L, const int pair, const int n_pairs,
                                             const int hk, const int r, uint8_t* smem_raw) {
  using G_ = PG2<D, NB, NSK, NSV>;
  constexpr int BN = G_::BN;
  const PrefillArgs& a = L.a;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const uint32_t sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sbase - ptx::smem_addr(smem_raw));
  int* meta = reinterpret_cast<int*>(sg + G_::OFF_META);  // [stage][3 NB]: start, flag, V block id
  uint16_t* mask16 = reinterpret_cast<uint16_t*>(sg + G_::OFF_MASK);  // [ring][NB] key-valid bits
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sg + G_::OFF_TSLOT);
  const uint32_t bar0 = sbase + G_::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, TQ = L.tq, mb = a.max_blocks;
  const int q0 = a.cu_q_lens[r];
  const int ql = a.cu_q_lens[r + 1] - q0;
  const int tok0 = 2 * pair * TQ;  // first token of query tile 0
  if (tid == 0 && pair == n_pairs - 1 && ql > n_pairs * 2 * TQ) atomicOr(a.err, kErrSeqLen);
  auto has_rows = [&](int pr) { return pr >= 0 && ql > 0 && 2 * pr * TQ < ql; };
  if (!has_rows(pair)) return;
  int kvl = a.kv_lens[r];
  if (kvl < ql || kvl > mb * 16) {
    if (tid == 0 && pair == 0) atomicOr(a.err, kErrSeqLen);
    kvl = min(kvl, mb * 16);
  }
  const int nblk = (kvl + 15) >> 4;
  auto tiles_of = [&](int pr) {  // key tiles the rows of query-tile pair pr reach
    if (!has_rows(pr)) return 0;
    const int t0 = 2 * pr * TQ;
    const int lim_last = kvl - ql + t0 + min(2 * TQ, ql - t0) - 1;
    return lim_last >= 0 ? lim_last / BN + 1 : 0;
  };
  const int n_kt = tiles_of(pair);  // key tiles this CTA loads and computes on

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    ptx::mbar_init(bar(G_::B_Q), kRotThreads);
    for (int s = 0; s < NSK; ++s) {
      ptx::mbar_init(bar(G_::B_KFULL + s), 1);
      ptx::mbar_init(bar(G_::B_KROT + s), kRotThreads);
      ptx::mbar_init(bar(G_::B_KFREE + s), 1);
    }
    for (int s = 0; s < NSV; ++s) {
      ptx::mbar_init(bar(G_::B_VFULL + s), 1);
      ptx::mbar_init(bar(G_::B_VFREE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(G_::B_S + i), 1);
      ptx::mbar_init(bar(G_::B_P + i), kSoftThreads / 2);
    }
    ptx::mbar_init(bar(G_::B_ODONE), 1);
    for (int k = 0; k < kMaskRing; ++k) ptx::mbar_init(bar(G_::B_MASK + k), kRotThreads);
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(ptx::smem_addr(tslot), G_::TCOLS);
    umma::tmem_relinquish();
  }
  // zero K and V stages once so that never-loaded blocks hold finite values
  for (int i = tid; i < (NSK + NSV) * G_::KTILE / 16; i += kThreads)
    reinterpret_cast<uint4*>(sg + G_::OFF_K)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kTmaWarp) {
    // ======================================================== TMA producer
    // Step u loads K~ tile u (once the products of tile u - NSK freed its stage)
    // and V tile u - LAG (once tile u - LAG - NSV freed its stage): K~ runs LAG
    // tiles ahead of V so that rotation has time to work on it.  The whole warp
    // issues a tile's copies together (lane -> block lane % NB, half lane / NB;
    // the lanes after those fetch the block-start cos/sin rows): one thread
    // issuing every copy in turn cannot keep up with the tensor core.
    constexpr int LAG = NSK - NSV;
    constexpr unsigned FULL = 0xffffffffu;
    static_assert(NB * G_::HALVES + NB <= 32, "one lane per copy");
    if (n_kt > 0) {
      const int* bt = a.block_tables + (size_t)r * mb;
      const int* bs = a.block_starts + (size_t)r * mb;
      const int blk = lane % NB, hh = lane / NB;
      int my_ph = -1, my_st = 0;  // lanes < NB: block NB u + lane of the next K~ tile
      auto fetch = [&](int t) {
        const int b = NB * t + lane;
        const bool in = lane < NB && b < nblk;
        my_ph = in ? __ldg(bt + b) : -1;
        my_st = in ? __ldg(bs + b) : 0;
      };
      bool ok = true;
      fetch(0);
      for (int u = 0; u < n_kt + LAG; ++u) {
        if (u < n_kt) {
          const int s = u % NSK;
          bool w = true;
          if (lane == 0 && u >= NSK) w = ptx::mbar_wait(bar(G_::B_KFREE + s), ((u / NSK) - 1) & 1);
          if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
          int flag = 0;
          if (lane < NB && NB * u + lane < nblk) {
            if (my_ph >= 0 && my_ph < a.num_blocks) flag |= 1;
            else atomicOr(a.err, kErrBlockId);
            if (!ROPE || (my_st >= 0 && my_st < a.max_pos)) flag |= 2;
          }
          int* m = meta + 3 * NB * s;
          if (lane < NB) {
            m[lane] = my_st;
            m[NB + lane] = flag;
            m[2 * NB + lane] = (flag & 1) ? my_ph : -1;
          }
          const unsigned kv = __ballot_sync(FULL, flag & 1);
          const unsigned rw = __ballot_sync(FULL, ROPE && (flag & 3) == 3);
          const int ph_l = __shfl_sync(FULL, my_ph, blk);
          const int st_l = __shfl_sync(FULL, my_st, blk);
          __syncwarp();
          if (lane == 0)
            ptx::mbar_arrive_expect_tx(bar(G_::B_KFULL + s), __popc(kv) * G_::HALVES * 2048 + __popc(rw) * G_::ROWB);
          __syncwarp();
          if (lane < NB * G_::HALVES) {
            if ((kv >> blk) & 1u) {
              const uint32_t dst = sbase + G_::OFF_K + s * G_::KTILE + hh * (BN * 128) + blk * 2048;
              ptx::tma_load_2d(dst, &kmap, 64 * hh, (ph_l * a.Hkv + hk) * 16, bar(G_::B_KFULL + s));
            }
          } else if (ROPE && lane < NB * G_::HALVES + NB) {
            if ((rw >> blk) & 1u) {
              const uint32_t dst = sbase + G_::OFF_RS + (s * NB + blk) * G_::ROWB;
              ptx::bulk_load(dst, a.cos_sin + (size_t)st_l * D, G_::ROWB, bar(G_::B_KFULL + s));
            }
          }
          if (u + 1 < n_kt) fetch(u + 1);
        }
        const int tv = u - LAG;
        if (tv >= 0) {
          const int sv = tv % NSV;
          bool w = true;
          if (lane == 0 && tv >= NSV) w = ptx::mbar_wait(bar(G_::B_VFREE + sv), ((tv / NSV) - 1) & 1);
          if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
          // the meta of tile tv is rewritten only for tile tv + NSK > u
          const int ph = meta[3 * NB * (tv % NSK) + 2 * NB + blk];
          const unsigned vv = __ballot_sync(FULL, lane < NB && ph >= 0);
          if (lane == 0) ptx::mbar_arrive_expect_tx(bar(G_::B_VFULL + sv), __popc(vv) * G_::HALVES * 2048);
          __syncwarp();
          if (lane < NB && ph >= 0) {  // one box per block: [half][16 rows][64]
            const uint32_t dst = sbase + G_::OFF_V + sv * G_::KTILE + blk * (G_::HALVES * 2048);
            ptx::tma_load_3d(dst, &vmap, 0, (ph * a.Hkv + hk) * 16, 0, bar(G_::B_VFULL + sv));
          }
        }
      }
      if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ======================================================== MMA issue
    if (lane == 0 && n_kt > 0) {
      // release a K~ / V stage once the products that read it are done
      auto free_k = [&](int u) { umma::commit(bar(G_::B_KFREE + u % NSK)); };
      auto free_v = [&](int u) { umma::commit(bar(G_::B_VFREE + u % NSV)); };
      const uint32_t id_qk = ROPE ? umma::idesc_f16_f32(128, BN, false, false)
                                  : umma::idesc_bf16_f32(128, BN, false, false);
      const uint32_t id_pv = umma::idesc_bf16_f32(128, D, false, true);
      auto qk = [&](int i, int t) {
        const uint32_t kb = sbase + G_::OFF_K + (t % NSK) * G_::KTILE;
        const uint32_t qb = sbase + G_::OFF_Q + i * G_::QTILE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t cb = (ks & 3) * 32;
          umma::mma_ss(tmem + 128 * i, umma::smem_desc_sw128(qb + (ks >> 2) * (128 * 128) + cb, 16, 1024),
                       umma::smem_desc_sw128(kb + (ks >> 2) * (BN * 128) + cb, 16, 1024), id_qk, ks > 0);
        }
        umma::commit(bar(G_::B_S + i));
      };
      auto pv = [&](int i, int t) {  // V stage: [block][half][16 keys][64]
        const uint32_t vb = sbase + G_::OFF_V + (t % NSV) * G_::KTILE;
#pragma unroll
        for (int ks = 0; ks < NB; ++ks)
          umma::mma_ts(tmem + 256 + 128 * i, tmem + 128 * i + 8 * ks,
                       umma::smem_desc_sw128(vb + ks * (G_::HALVES * 2048), 2048, 1024), id_pv,
                       (t > 0 || ks > 0) ? 1u : 0u);
      };
      bool ok = true;
      if (n_kt > 0) {
        ok = ptx::mbar_wait(bar(G_::B_Q), 0) && ptx::mbar_wait(bar(G_::B_KROT), 0);
        if (ok) {
          umma::fence_after_sync();
          qk(0, 0);
          qk(1, 0);
          free_k(0);
        }
        for (int t = 0; t < n_kt && ok; ++t) {
          const int sv = t % NSV, sk1 = (t + 1) % NSK;
          const bool more = t + 1 < n_kt;
          if (!ptx::mbar_wait(bar(G_::B_P + 0), t & 1) || !ptx::mbar_wait(bar(G_::B_VFULL + sv), (t / NSV) & 1)) {
            ok = false;
            break;
          }
          umma::fence_after_sync();
          pv(0, t);
          if (more) {
            if (!ptx::mbar_wait(bar(G_::B_KROT + sk1), ((t + 1) / NSK) & 1)) { ok = false; break; }
            umma::fence_after_sync();
            qk(0, t + 1);
          }
          if (!ptx::mbar_wait(bar(G_::B_P + 1), t & 1)) { ok = false; break; }
          umma::fence_after_sync();
          pv(1, t);
          free_v(t);
          if (more) {
            qk(1, t + 1);
            free_k(t + 1);
          }
        }
        umma::commit(bar(G_::B_ODONE));
      }
      if (!ok) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (tid >= kRotBase) {
    // ======================================================== query preparation + key rotation
    const int rt = tid - kRotBase;  // 0..255
    const int rw = rt >> 5;         // warp within the group
    const float qs = a.scale * kLog2e;
#pragma unroll 1
    for (int qr = rt; qr < 256; qr += kRotThreads) {  // ---- query tiles: row qr % 128 of tile qr / 128
      const int i = qr >> 7, row = qr & 127;
      const int rtok = row / G, rh = row - rtok * G;
      const int tq = tok0 + i * TQ + rtok;
      const bool row_ok = rtok < TQ && tq < ql;
      U4 qc[D / 8];
      int pos = 0;
      if (row_ok) {
        const __nv_bfloat16* qp =
            static_cast<const __nv_bfloat16*>(a.q) + ((size_t)(q0 + tq) * a.Hq + (size_t)hk * G + rh) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qp) + c);
          qc[c] = U4{v.x, v.y, v.z, v.w};
        }
        if (ROPE) {
          pos = a.q_pos[q0 + tq];
          if (pos < 0 || pos >= a.max_pos) {
            atomicOr(a.err, kErrPosition);
            pos = 0;
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) qc[c] = U4{0u, 0u, 0u, 0u};
      }
      if constexpr (ROPE) {
        const float* trow = a.cos_sin + (size_t)pos * D;
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {  // chunk c pairs with chunk c + D/16
          uint64_t c2[4], s2[4];
          const float4 ca = __ldg(reinterpret_cast<const float4*>(trow + 8 * c));
          const float4 cb = __ldg(reinterpret_cast<const float4*>(trow + 8 * c + 4));
          const float4 sa = __ldg(reinterpret_cast<const float4*>(trow + D / 2 + 8 * c));
          const float4 sb = __ldg(reinterpret_cast<const float4*>(trow + D / 2 + 8 * c + 4));
          c2[0] = ptx::f2(ca.x * qs, ca.y * qs); c2[1] = ptx::f2(ca.z * qs, ca.w * qs);
          c2[2] = ptx::f2(cb.x * qs, cb.y * qs); c2[3] = ptx::f2(cb.z * qs, cb.w * qs);
          s2[0] = ptx::f2(sa.x * qs, sa.y * qs); s2[1] = ptx::f2(sa.z * qs, sa.w * qs);
          s2[2] = ptx::f2(sb.x * qs, sb.y * qs); s2[3] = ptx::f2(sb.z * qs, sb.w * qs);
          rot_pack(qc[c], qc[c + D / 16], c2, s2);
        }
        uint32_t wq = 0u;  // fp16 range watch over the rotated, scaled query
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
          wq = ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(wq, qc[c].x), qc[c].y), qc[c].z), qc[c].w);
        if (row_ok && wq != 0u) atomicOr(a.err, kErrRange);
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          U4& x = qc[c];
          x = U4{ptx::pack_bf16(ptx::bf_lo(x.x) * qs, ptx::bf_hi(x.x) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.y) * qs, ptx::bf_hi(x.y) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.z) * qs, ptx::bf_hi(x.z) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.w) * qs, ptx::bf_hi(x.w) * qs)};
        }
      }
#pragma unroll
      for (int c = 0; c < D / 8; ++c)
        sts128(sbase + G_::OFF_Q + i * G_::QTILE + (c >> 3) * (128 * 128) + swz(row, c & 7), qc[c]);
    }
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(bar(G_::B_Q));

    // ---- key rotation: thread -> (frequency group fg, slot pair sp, block group
    // bg): slots 2 sp and 2 sp + 1 of blocks BPG bg .. BPG bg + BPG - 1, so the
    // slots' own cos/sin(slot theta_f), f = 8 fg .. 8 fg + 7, stay in registers
    const int fg = rt % G_::NFG;
    const int sp = (rt / G_::NFG) & 7;
    const int bg = rt / (G_::NFG * 8);
    uint64_t rsc[2][4], rss[2][4];
    if constexpr (ROPE) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const float* tr = a.cos_sin + (size_t)min(2 * sp + k, a.max_pos - 1) * D;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 c = __ldg(reinterpret_cast<const float2*>(tr + 8 * fg + 2 * e));
          const float2 sn = __ldg(reinterpret_cast<const float2*>(tr + D / 2 + 8 * fg + 2 * e));
          rsc[k][e] = ptx::f2(c.x, c.y);
          rss[k][e] = ptx::f2(sn.x, sn.y);
        }
      }
    }
    for (int t = 0; t < n_kt; ++t) {
      const int s = t % NSK;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(G_::B_KFULL + s), (t / NSK) & 1))) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        break;
      }
      const int* m = meta + 3 * NB * s;
      uint8_t* sk = sg + G_::OFF_K + s * G_::KTILE;
      if constexpr (ROPE) {
        // loads for every key first (stage and start rows are always addressable),
        // stores only for valid keys: no branch between keys, so their loads overlap
        uint32_t wk = 0u;  // fp16 range watch over the stored keys
#pragma unroll
        for (int b = 0; b < G_::BPG; ++b) {
          const int blk = bg * G_::BPG + b;
          const int flag = m[NB + blk];
          const int start = m[blk];
          const uint8_t* rb = sg + G_::OFF_RS + (s * NB + blk) * G_::ROWB;
          const U4 c0 = *reinterpret_cast<const U4*>(rb + 32 * fg);
          const U4 c1 = *reinterpret_cast<const U4*>(rb + 32 * fg + 16);
          const U4 s0 = *reinterpret_cast<const U4*>(rb + 2 * D + 32 * fg);
          const U4 s1 = *reinterpret_cast<const U4*>(rb + 2 * D + 32 * fg + 16);
          const uint64_t ac[4] = {((uint64_t)c0.y << 32) | c0.x, ((uint64_t)c0.w << 32) | c0.z,
                                  ((uint64_t)c1.y << 32) | c1.x, ((uint64_t)c1.w << 32) | c1.z};
          const uint64_t as[4] = {((uint64_t)s0.y << 32) | s0.x, ((uint64_t)s0.w << 32) | s0.z,
                                  ((uint64_t)s1.y << 32) | s1.x, ((uint64_t)s1.w << 32) | s1.z};
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int slot = 2 * sp + k;
            const int key = blk * 16 + slot;
            const bool v = (flag & 3) == 3 && t * BN + key < kvl && start + slot < a.max_pos;
            U4* px = reinterpret_cast<U4*>(sk + swz(key, fg));
            U4* py = reinterpret_cast<U4*>(sk + ((D == 128) ? BN * 128 + swz(key, fg) : swz(key, fg + 4)));
            U4 x = *px, y = *py;
            uint64_t c2[4], s2[4];  // cos/sin((start + slot) theta) by angle addition
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              c2[e] = ptx::sub2(ptx::mul2(ac[e], rsc[k][e]), ptx::mul2(as[e], rss[k][e]));
              s2[e] = ptx::fma2(as[e], rsc[k][e], ptx::mul2(ac[e], rss[k][e]));
            }
            rot_pack(x, y, c2, s2);
            if (v) {
              *px = x;
              *py = y;
              wk = ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(wk, x.x), x.y), x.z), x.w);
              wk = ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(wk, y.x), y.y), y.z), y.w);
            }
          }
        }
        if (wk != 0u) atomicOr(a.err, kErrRange);
      }
      // key-valid bits: warp rw covers blocks rw, rw + 6, ...; lane = slot
#pragma unroll
      for (int blk = rw; blk < NB; blk += kRotThreads / 32) {
        const int flag = m[NB + blk];
        const int start = m[blk];
        const bool v = lane < 16 && (flag & 3) == 3 && t * BN + blk * 16 + lane < kvl &&
                       (!ROPE || start + lane < a.max_pos);
        const uint32_t bits = __ballot_sync(0xffffffffu, v);
        if (lane == 0) mask16[(t % kMaskRing) * NB + blk] = (uint16_t)bits;
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(G_::B_MASK + t % kMaskRing));
      ptx::mbar_arrive(bar(G_::B_KROT + s));
    }
  } else {
    // ======================================================== softmax of query tile i
    // The row's BN scores are read from TMEM once; the max, the reference
    // update and P (packed in place over the scores) all come from registers.
    constexpr int NP = BN / 32;  // 32-key parts of a tile
    const int i = warp >> 2;      // 0 or 1
    const int row = tid & 127;    // TMEM lane
    const int rtok = row / G, rh = row - rtok * G;
    const int tq = tok0 + i * TQ + rtok;
    const bool row_ok = rtok < TQ && tq < ql;
    const int lim = kvl - ql + tq;                        // last key this row attends
    const int lim_first = kvl - ql + tok0 + i * TQ;       // ... the tile's first row attends
    const uint32_t lane_base = ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t t_s = tmem + 128 * i + lane_base;
    const uint32_t t_o = tmem + 256 + 128 * i + lane_base;
    float m_run = -CUDART_INF_F, m_use = -CUDART_INF_F, l_run = 0.f;
    bool failed = false;
    for (int t = 0; t < n_kt; ++t) {
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(G_::B_S + i), t & 1))) {
        failed = true;
        break;
      }
      // the mask of tile t is rewritten for tile t + kMaskRing, which needs this group past tile t + 3
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(G_::B_MASK + t % kMaskRing), (t / kMaskRing) & 1))) {
        failed = true;
        break;
      }
      umma::fence_after_sync();
      uint32_t v[BN];
#pragma unroll
      for (int part = 0; part < NP; ++part)
        umma::tmem_ld32(t_s + 32 * part, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * part));
      const uint16_t* mk = mask16 + (t % kMaskRing) * NB;
      uint32_t mw[NP];
      uint32_t mall = 0xffffffffu;
#pragma unroll
      for (int w = 0; w < NP; ++w) {
        mw[w] = (uint32_t)mk[2 * w] | ((uint32_t)mk[2 * w + 1] << 16);
        mall &= mw[w];
      }
      const bool full = mall == 0xffffffffu && t * BN + BN - 1 <= lim_first;
      const int kb0 = t * BN;
      umma::tmem_wait_ld();
      float mx;
      if (full) {
        float pm[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int j = 0; j < BN; j += 2)
          pm[(j >> 1) & 3] = ptx::fmax3(pm[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
      } else if (mall == 0xffffffffu) {
        // every block usable: the valid keys are the causal prefix j < nv
        const int nv = row_ok ? lim - kb0 + 1 : 0;
        mx = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          v[j] = j < nv ? v[j] : __float_as_uint(-CUDART_INF_F);
          mx = fmaxf(mx, __uint_as_float(v[j]));
        }
      } else {
        // invalid keys become -inf in place, so that both passes treat them alike
        mx = -CUDART_INF_F;
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const bool ok = row_ok && ((mw[j >> 5] >> (j & 31)) & 1u) && kb0 + j <= lim;
          v[j] = ok ? v[j] : __float_as_uint(-CUDART_INF_F);
          mx = fmaxf(mx, __uint_as_float(v[j]));
        }
      }
      m_run = fmaxf(m_run, mx);
      const bool need = m_run != -CUDART_INF_F && (m_use == -CUDART_INF_F || m_run > m_use + kRescale);
      const float corr = !need ? 1.f : (m_use == -CUDART_INF_F ? 0.f : ex2(m_use - m_run));
      if (need) {
        l_run *= corr;
        m_use = m_run;
      }
      // P = 2^(s - mref) as bf16 pairs, written over the scores already consumed
      // (pair j lands in v[j] after v[2 j], v[2 j + 1] were read), 16 words per store
      const float mref = m_use == -CUDART_INF_F ? 0.f : m_use;
      const uint64_t mref2 = ptx::f2(mref, mref);
      uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int j = 0; j < BN / 2; ++j) {
        const uint64_t d2 = ptx::sub2(ptx::f2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), mref2);
        float dl, dh;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(dl), "=f"(dh) : "l"(d2));
        const uint64_t p2 = ptx::f2(ex2(dl), ex2(dh));  // 2^-inf = 0 for masked keys
        ls[j & 3] = ptx::add2(ls[j & 3], p2);
        v[j] = ptx::f2_to_bf2(p2);
        if ((j & 15) == 15) umma::tmem_st16(t_s + (j & ~15), *reinterpret_cast<const uint32_t(*)[16]>(v + (j & ~15)));
      }
      const uint64_t lsum2 = ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3]));
      float sl, sh;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(sl), "=f"(sh) : "l"(lsum2));
      l_run += sl + sh;
      // lazy O rescale before P_i releases the next products
      if (t > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int part = 0; part < D / 32; ++part) {
          uint32_t o[32];
          umma::tmem_ld32(t_o + part * 32, o);
          umma::tmem_wait_ld();
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            w0[j] = __float_as_uint(__uint_as_float(o[j]) * corr);
            w1[j] = __float_as_uint(__uint_as_float(o[16 + j]) * corr);
          }
          umma::tmem_st16(t_o + part * 32, w0);
          umma::tmem_st16(t_o + part * 32 + 16, w1);
        }
      }
      umma::tmem_wait_st();
      umma::fence_before_sync();
      ptx::mbar_arrive(bar(G_::B_P + i));
    }
    // ---- epilogue: O / l -> global (TMEM loads by the whole warp, stores by valid rows)
    bool have = n_kt > 0 && !failed;
    if (have && !__all_sync(0xffffffffu, ptx::mbar_wait(bar(G_::B_ODONE), 0))) {
      have = false;
      failed = true;
    }
    if (failed && lane == 0) atomicOr(a.err, kErrTimeout);
    umma::fence_after_sync();
    const int hq = hk * G + rh;
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(q0 + tq) * a.Hq + hq) * D;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int part = 0; part < D / 32; ++part) {
      uint32_t v[32];
      if (have) {
        umma::tmem_ld32(t_o + part * 32, v);
        umma::tmem_wait_ld();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0u;
      }
      if (row_ok) {
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint4 o;
          o.x = ptx::pack_bf16(__uint_as_float(v[j]) * inv, __uint_as_float(v[j + 1]) * inv);
          o.y = ptx::pack_bf16(__uint_as_float(v[j + 2]) * inv, __uint_as_float(v[j + 3]) * inv);
          o.z = ptx::pack_bf16(__uint_as_float(v[j + 4]) * inv, __uint_as_float(v[j + 5]) * inv);
          o.w = ptx::pack_bf16(__uint_as_float(v[j + 6]) * inv, __uint_as_float(v[j + 7]) * inv);
          *reinterpret_cast<uint4*>(op + part * 32 + j) = o;
        }
      }
    }
    if (row_ok && a.lse)
      a.lse[(size_t)(q0 + tq) * a.Hq + hq] = l_run > 0.f ? (m_use + log2f(l_run)) * kLn2 : -CUDART_INF_F;
  }

  umma::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) umma::tmem_dealloc(tmem, G_::TCOLS);
}

}  // namespace prefill2_impl
}  // namespace minipic
