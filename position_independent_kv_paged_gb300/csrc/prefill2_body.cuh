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
//   warps 8-11  query preparation, then rotation of every staged key tile
//   warp 12     TMA producer (K~ tiles + block-start cos/sin rows, V tiles)
//   warp 13     TMEM allocation and tcgen05 MMA issue
// K and V are double buffered.  Per 128-key tile t the MMA warp issues
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
constexpr int kRotBase = 256;                     // first thread of the rotation warpgroup
constexpr int kTmaWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int BN = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;

// barriers
enum {
  kBarQ = 0,        // rotation warpgroup -> MMA: both query tiles in shared memory
  kBarKFull = 1,    // [2] TMA -> rotation: K~ stage and its start rows landed
  kBarKRot = 3,     // [2] rotation -> MMA: K stage rotated
  kBarKFree = 5,    // [2] MMA -> TMA: K stage consumed
  kBarVFull = 7,    // [2] TMA -> MMA
  kBarVFree = 9,    // [2] MMA -> TMA
  kBarS = 11,       // [2] MMA -> softmax i: S_i ready
  kBarP = 13,       // [2] softmax i -> MMA: P_i in TMEM
  kBarODone = 15,   // MMA -> softmax: last products finished
  kBarMask = 16,    // [4] rotation -> softmax: key-valid bits of tile t (index t & 3)
  kNumBars = 20
};

template <int D>
struct PG2 {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE = HALVES * BN * 128;      // one Q, K or V tile
  static constexpr int ROWB = 4 * D;                  // one cos|sin table row
  static constexpr int OFF_Q = 0;                     // [2] query tiles
  static constexpr int OFF_K = OFF_Q + 2 * TILE;      // [2] K stages
  static constexpr int OFF_V = OFF_K + 2 * TILE;      // [2] V stages
  static constexpr int OFF_RS = OFF_V + 2 * TILE;     // [2 stages][8] block-start rows
  static constexpr int OFF_META = OFF_RS + 16 * ROWB; // [2 stages] int start[8], int flag[8]
  static constexpr int OFF_MASK = OFF_META + 2 * 64;  // [4 tiles][8] uint16 key-valid bits per block
  static constexpr int OFF_BAR = OFF_MASK + 4 * 16;
  static constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
  static constexpr int TOTAL = OFF_TSLOT + 16;
  static constexpr int NFG = D / 16;                  // rotation work split: frequency groups of 8
  static constexpr int SPT = 16 * NFG / 32;           // slots per rotation thread
  static constexpr uint32_t TCOLS = 512;              // S0 [0,128) S1 [128,256) O0 [256,..) O1 [384,..)
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

template <int D, bool ROPE>
__device__ __forceinline__ void prefill2_cta(const CUtensorMap* kmap_p, const CUtensorMap* vmap_p,
                                             const PrefillLaunch2& L, const int pair, const int n_pairs,
                                             const int hk, const int r, uint8_t* smem_raw) {
  using G_ = PG2<D>;
  const PrefillArgs& a = L.a;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const uint32_t sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sbase - ptx::smem_addr(smem_raw));
  int* meta = reinterpret_cast<int*>(sg + G_::OFF_META);  // [stage][16]: start[8], flag[8]
  uint16_t* mask16 = reinterpret_cast<uint16_t*>(sg + G_::OFF_MASK);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sg + G_::OFF_TSLOT);
  const uint32_t bar0 = sbase + G_::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, TQ = L.tq, mb = a.max_blocks;
  const int q0 = a.cu_q_lens[r];
  const int ql = a.cu_q_lens[r + 1] - q0;
  const int tok0 = 2 * pair * TQ;  // first token of query tile 0
  if (tid == 0 && pair == n_pairs - 1 && ql > n_pairs * 2 * TQ) atomicOr(a.err, kErrSeqLen);
  if (ql <= 0 || tok0 >= ql) return;
  int kvl = a.kv_lens[r];
  if (kvl < ql || kvl > mb * 16) {
    if (tid == 0 && pair == 0) atomicOr(a.err, kErrSeqLen);
    kvl = min(kvl, mb * 16);
  }
  const int nblk = (kvl + 15) >> 4;
  const int ntok_all = min(2 * TQ, ql - tok0);
  const int lim_last = kvl - ql + tok0 + ntok_all - 1;  // largest key any row of the pair sees
  const int n_kt = lim_last >= 0 ? lim_last / BN + 1 : 0;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    ptx::mbar_init(bar(kBarQ), 128);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar(kBarKFull + s), 1);
      ptx::mbar_init(bar(kBarKRot + s), 128);
      ptx::mbar_init(bar(kBarKFree + s), 1);
      ptx::mbar_init(bar(kBarVFull + s), 1);
      ptx::mbar_init(bar(kBarVFree + s), 1);
      ptx::mbar_init(bar(kBarS + s), 1);
      ptx::mbar_init(bar(kBarP + s), 128);
    }
    ptx::mbar_init(bar(kBarODone), 1);
    for (int k = 0; k < 4; ++k) ptx::mbar_init(bar(kBarMask + k), 128);
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    umma::tmem_alloc(ptx::smem_addr(tslot), G_::TCOLS);
    umma::tmem_relinquish();
  }
  // zero K and V stages once so that never-loaded blocks hold finite values
  for (int i = tid; i < 4 * G_::TILE / 16; i += kThreads)
    reinterpret_cast<uint4*>(sg + G_::OFF_K)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  if (warp == kTmaWarp) {
    // ======================================================== TMA producer
    if (lane == 0 && n_kt > 0) {
      const int* bt = a.block_tables + (size_t)r * mb;
      const int* bs = a.block_starts + (size_t)r * mb;
      int nph[8], nst[8], vph[8][2];
      auto load_meta = [&](int t) {
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          const int b = 8 * t + blk;
          nph[blk] = b < nblk ? __ldg(bt + b) : -1;
          nst[blk] = b < nblk ? __ldg(bs + b) : 0;
        }
      };
      bool ok = true;
      load_meta(0);
      for (int t = 0; t < n_kt && ok; ++t) {
        const int s = t & 1;
        if (t >= 2 && !ptx::mbar_wait(bar(kBarKFree + s), ((t >> 1) - 1) & 1)) { ok = false; break; }
        int* m = meta + 16 * s;
        int nvalid = 0, nrows = 0;
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          const int b = 8 * t + blk;
          int flag = 0;
          if (b < nblk) {
            if (nph[blk] >= 0 && nph[blk] < a.num_blocks) flag |= 1;
            else atomicOr(a.err, kErrBlockId);
            if (!ROPE || (nst[blk] >= 0 && nst[blk] < a.max_pos)) flag |= 2;
          }
          m[blk] = nst[blk];
          m[8 + blk] = flag;
          vph[blk][s] = (flag & 1) ? nph[blk] : -1;
          nvalid += flag & 1;
          nrows += (ROPE && (flag & 3) == 3) ? 1 : 0;
        }
        ptx::mbar_arrive_expect_tx(bar(kBarKFull + s), nvalid * G_::HALVES * 2048 + nrows * G_::ROWB);
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          if (vph[blk][s] < 0) continue;
          const int y = (vph[blk][s] * a.Hkv + hk) * 16;
          for (int hh = 0; hh < G_::HALVES; ++hh)
            ptx::tma_load_2d(sbase + G_::OFF_K + s * G_::TILE + hh * (BN * 128) + blk * 2048, &kmap, 64 * hh, y,
                             bar(kBarKFull + s));
          if (ROPE && (m[8 + blk] & 3) == 3)
            ptx::bulk_load(sbase + G_::OFF_RS + (s * 8 + blk) * G_::ROWB, a.cos_sin + (size_t)nst[blk] * D,
                           G_::ROWB, bar(kBarKFull + s));
        }
        if (t + 1 < n_kt) load_meta(t + 1);
        if (t >= 2 && !ptx::mbar_wait(bar(kBarVFree + s), ((t >> 1) - 1) & 1)) { ok = false; break; }
        int vvalid = 0;
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) vvalid += vph[blk][s] >= 0 ? 1 : 0;
        ptx::mbar_arrive_expect_tx(bar(kBarVFull + s), vvalid * G_::HALVES * 2048);
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          if (vph[blk][s] < 0) continue;
          const int y = (vph[blk][s] * a.Hkv + hk) * 16;
          for (int hh = 0; hh < G_::HALVES; ++hh)
            ptx::tma_load_2d(sbase + G_::OFF_V + s * G_::TILE + hh * (BN * 128) + blk * 2048, &vmap, 64 * hh, y,
                             bar(kBarVFull + s));
        }
      }
      if (!ok) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ======================================================== MMA issue
    if (lane == 0 && n_kt > 0) {
      const uint32_t id_qk = ROPE ? umma::idesc_f16_f32(128, BN, false, false)
                                  : umma::idesc_bf16_f32(128, BN, false, false);
      const uint32_t id_pv = umma::idesc_bf16_f32(128, D, false, true);
      auto qk = [&](int i, int t) {
        const uint32_t kb = sbase + G_::OFF_K + (t & 1) * G_::TILE;
        const uint32_t qb = sbase + G_::OFF_Q + i * G_::TILE;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (BN * 128) + (ks & 3) * 32;
          umma::mma_ss(tmem + 128 * i, umma::smem_desc_sw128(qb + off, 16, 1024),
                       umma::smem_desc_sw128(kb + off, 16, 1024), id_qk, ks > 0);
        }
        umma::commit(bar(kBarS + i));
      };
      auto pv = [&](int i, int t) {
        const uint32_t vb = sbase + G_::OFF_V + (t & 1) * G_::TILE;
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks)
          umma::mma_ts(tmem + 256 + 128 * i, tmem + 128 * i + 8 * ks,
                       umma::smem_desc_sw128(vb + ks * 2048, BN * 128, 1024), id_pv, (t > 0 || ks > 0) ? 1u : 0u);
      };
      bool ok = ptx::mbar_wait(bar(kBarQ), 0) && ptx::mbar_wait(bar(kBarKRot), 0);
      if (ok) {
        umma::fence_after_sync();
        qk(0, 0);
        qk(1, 0);
        umma::commit(bar(kBarKFree + 0));
      }
      for (int t = 0; t < n_kt && ok; ++t) {
        const int s = t & 1;
        const bool more = t + 1 < n_kt;
        if (!ptx::mbar_wait(bar(kBarP + 0), t & 1) || !ptx::mbar_wait(bar(kBarVFull + s), (t >> 1) & 1)) {
          ok = false;
          break;
        }
        umma::fence_after_sync();
        pv(0, t);
        if (more) {
          if (!ptx::mbar_wait(bar(kBarKRot + ((t + 1) & 1)), ((t + 1) >> 1) & 1)) { ok = false; break; }
          umma::fence_after_sync();
          qk(0, t + 1);
        }
        if (!ptx::mbar_wait(bar(kBarP + 1), t & 1)) { ok = false; break; }
        umma::fence_after_sync();
        pv(1, t);
        umma::commit(bar(kBarVFree + s));
        if (more) {
          qk(1, t + 1);
          umma::commit(bar(kBarKFree + ((t + 1) & 1)));
        }
      }
      umma::commit(bar(kBarODone));
      if (!ok) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (tid >= kRotBase) {
    // ======================================================== query preparation + key rotation
    const int rt = tid - kRotBase;  // 0..127
    const int rw = rt >> 5;         // warp within the group
    const float qs = a.scale * kLog2e;
    // ---- query tiles: row rt of tile 0 and of tile 1
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      const int row = rt;
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
        sts128(sbase + G_::OFF_Q + i * G_::TILE + (c >> 3) * (BN * 128) + swz(row, c & 7), qc[c]);
    }
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive(bar(kBarQ));

    // ---- key rotation: thread -> (frequency group fg, slot group sgp, blocks rw and rw + 4)
    const int fg = rt % G_::NFG;
    const int sgp = (rt / G_::NFG) % (32 / G_::NFG);
    uint64_t rsc[G_::SPT][4], rss[G_::SPT][4];  // cos/sin(slot theta_f), f = 8 fg .. 8 fg + 7
#pragma unroll
    for (int u = 0; u < (ROPE ? G_::SPT : 0); ++u) {
      const float* tr = a.cos_sin + (size_t)min(sgp * G_::SPT + u, a.max_pos - 1) * D;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = __ldg(reinterpret_cast<const float2*>(tr + 8 * fg + 2 * e));
        const float2 sn = __ldg(reinterpret_cast<const float2*>(tr + D / 2 + 8 * fg + 2 * e));
        rsc[u][e] = ptx::f2(c.x, c.y);
        rss[u][e] = ptx::f2(sn.x, sn.y);
      }
    }
    for (int t = 0; t < n_kt; ++t) {
      const int s = t & 1;
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarKFull + s), (t >> 1) & 1))) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        break;
      }
      const int* m = meta + 16 * s;
      uint8_t* sk = sg + G_::OFF_K + s * G_::TILE;
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int blk = rw + 4 * bb;
        const int flag = m[8 + blk];
        const int start = m[blk];
        uint64_t ac[4], as[4];
        if (ROPE && (flag & 2)) {
          const uint8_t* rb = sg + G_::OFF_RS + (s * 8 + blk) * G_::ROWB;
          const U4 c0 = *reinterpret_cast<const U4*>(rb + 32 * fg);
          const U4 c1 = *reinterpret_cast<const U4*>(rb + 32 * fg + 16);
          const U4 s0 = *reinterpret_cast<const U4*>(rb + 2 * D + 32 * fg);
          const U4 s1 = *reinterpret_cast<const U4*>(rb + 2 * D + 32 * fg + 16);
          ac[0] = ((uint64_t)c0.y << 32) | c0.x; ac[1] = ((uint64_t)c0.w << 32) | c0.z;
          ac[2] = ((uint64_t)c1.y << 32) | c1.x; ac[3] = ((uint64_t)c1.w << 32) | c1.z;
          as[0] = ((uint64_t)s0.y << 32) | s0.x; as[1] = ((uint64_t)s0.w << 32) | s0.z;
          as[2] = ((uint64_t)s1.y << 32) | s1.x; as[3] = ((uint64_t)s1.w << 32) | s1.z;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) ac[e] = as[e] = 0ull;
        }
        uint32_t bits = 0;
#pragma unroll
        for (int u = 0; u < G_::SPT; ++u) {
          const int slot = sgp * G_::SPT + u;
          const int key = blk * 16 + slot;
          const bool v = (flag & 3) == 3 && t * BN + key < kvl && (!ROPE || start + slot < a.max_pos);
          bits |= v ? (1u << slot) : 0u;
          if (!ROPE || !v) continue;
          uint64_t c2[4], s2[4];  // cos/sin((start + slot) theta) by angle addition
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            c2[e] = ptx::sub2(ptx::mul2(ac[e], rsc[u][e]), ptx::mul2(as[e], rss[u][e]));
            s2[e] = ptx::fma2(as[e], rsc[u][e], ptx::mul2(ac[e], rss[u][e]));
          }
          // plain shared-memory accesses (not volatile asm) so that independent keys overlap
          U4* px = reinterpret_cast<U4*>(sk + swz(key, fg));
          U4* py = reinterpret_cast<U4*>(sk + ((D == 128) ? BN * 128 + swz(key, fg) : swz(key, fg + 4)));
          U4 x = *px, y = *py;
          rot_pack(x, y, c2, s2);
          *px = x;
          *py = y;
        }
        bits = __reduce_or_sync(0xffffffffu, bits);
        if (lane == 0) mask16[(t & 3) * 8 + blk] = (uint16_t)bits;
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(kBarMask + (t & 3)));
      ptx::mbar_arrive(bar(kBarKRot + s));
    }
  } else {
    // ======================================================== softmax of query tile i
    const int i = tid >> 7;       // 0 or 1
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
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarS + i), t & 1))) {
        failed = true;
        break;
      }
      umma::fence_after_sync();
      // the mask of tile t is rewritten only for tile t + 4, after this group finished tile t + 1
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarMask + (t & 3)), (t >> 2) & 1))) {
        failed = true;
        break;
      }
      const uint16_t* mk = mask16 + (t & 3) * 8;
      uint32_t mw[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) mw[w] = (uint32_t)mk[2 * w] | ((uint32_t)mk[2 * w + 1] << 16);
      const bool full = (mw[0] & mw[1] & mw[2] & mw[3]) == 0xffffffffu && t * BN + BN - 1 <= lim_first;
      // pass 1: row max
      float mx = -CUDART_INF_F;
      if (full) {
#pragma unroll
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = -CUDART_INF_F;
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32], u[32];
          umma::tmem_ld32(t_s + half * 64, v);
          umma::tmem_ld32(t_s + half * 64 + 32, u);
          umma::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            pm[j & 7] = fmaxf(pm[j & 7], fmaxf(__uint_as_float(v[j]), __uint_as_float(u[j])));
        }
        mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])), fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
      } else {
#pragma unroll 1
        for (int part = 0; part < 4; ++part) {
          uint32_t v[32];
          umma::tmem_ld32(t_s + part * 32, v);
          umma::tmem_wait_ld();
          const int kb0 = t * BN + part * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const bool ok = row_ok && ((mw[part] >> j) & 1u) && kb0 + j <= lim;
            mx = ok ? fmaxf(mx, __uint_as_float(v[j])) : mx;
          }
        }
      }
      m_run = fmaxf(m_run, mx);
      const bool need = m_run != -CUDART_INF_F && (m_use == -CUDART_INF_F || m_run > m_use + kRescale);
      const float corr = !need ? 1.f : (m_use == -CUDART_INF_F ? 0.f : ex2(m_use - m_run));
      if (need) {
        l_run *= corr;
        m_use = m_run;
      }
      if (t > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int part = 0; part < D / 32; ++part) {
          uint32_t v[32];
          umma::tmem_ld32(t_o + part * 32, v);
          umma::tmem_wait_ld();
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            w0[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
            w1[j] = __float_as_uint(__uint_as_float(v[16 + j]) * corr);
          }
          umma::tmem_st16(t_o + part * 32, w0);
          umma::tmem_st16(t_o + part * 32 + 16, w1);
        }
      }
      const float mref = m_use == -CUDART_INF_F ? 0.f : m_use;
      const uint64_t mref2 = ptx::f2(mref, mref);
      // pass 2: P = 2^(s - mref), row sum, bf16 pairs over the S columns
      uint64_t lsum2 = ptx::f2(0.f, 0.f);
      uint64_t ls[4] = {lsum2, lsum2, lsum2, lsum2};
      if (full) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[64];
          umma::tmem_ld32(t_s + half * 64, *reinterpret_cast<uint32_t(*)[32]>(v));
          umma::tmem_ld32(t_s + half * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          umma::tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint64_t d2 =
                  ptx::sub2(ptx::f2(__uint_as_float(v[32 * q + 2 * j]), __uint_as_float(v[32 * q + 2 * j + 1])), mref2);
              float dl, dh;
              asm("mov.b64 {%0, %1}, %2;" : "=f"(dl), "=f"(dh) : "l"(d2));
              const uint64_t p2 = ptx::f2(ex2(dl), ex2(dh));
              ls[j & 3] = ptx::add2(ls[j & 3], p2);
              w[j] = ptx::f2_to_bf2(p2);
            }
            umma::tmem_st16(t_s + (2 * half + q) * 16, w);
          }
        }
      } else {
#pragma unroll 1
        for (int part = 0; part < 4; ++part) {
          uint32_t v[32];
          umma::tmem_ld32(t_s + part * 32, v);
          umma::tmem_wait_ld();
          const int kb0 = t * BN + part * 32;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int j0 = 2 * j, j1 = 2 * j + 1;
            const bool ok0 = row_ok && ((mw[part] >> j0) & 1u) && kb0 + j0 <= lim;
            const bool ok1 = row_ok && ((mw[part] >> j1) & 1u) && kb0 + j1 <= lim;
            const float p0 = ok0 ? ex2(__uint_as_float(v[j0]) - mref) : 0.f;
            const float p1 = ok1 ? ex2(__uint_as_float(v[j1]) - mref) : 0.f;
            const uint64_t p2 = ptx::f2(p0, p1);
            asm("add.rn.f32x2 %0, %0, %1;" : "+l"(lsum2) : "l"(p2));
            w[j] = ptx::pack_bf16(p0, p1);
          }
          umma::tmem_st16(t_s + part * 16, w);
        }
      }
      lsum2 = ptx::add2(lsum2, ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3])));
      float sl, sh;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(sl), "=f"(sh) : "l"(lsum2));
      l_run += sl + sh;
      umma::tmem_wait_st();
      umma::fence_before_sync();
      ptx::mbar_arrive(bar(kBarP + i));
    }
    // ---- epilogue: O / l -> global (TMEM loads by the whole warp, stores by valid rows)
    bool have = n_kt > 0 && !failed;
    if (have && !__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarODone), 0))) {
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
