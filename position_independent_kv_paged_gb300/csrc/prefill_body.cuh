// Chunked prefill over the position-free paged cache on the tcgen05 tensor cores
// (CTA body shared by the prefill kernel and the mixed prefill + decode kernel).
//
// Method (MiniPIC summary, gist.science 2606.13126, section 2.1): stored keys
// are unrotated; the kernel rotates each key at its logical position
// pi(j) = start[r][j / 16] + j % 16 with cos/sin values and multiply-adds per
// key element, then runs softmax attention.  A request's query chunk (the
// last q_len of its kv_len keys) attends causally: chunk query i sees keys
// j <= kv_len - q_len + i.
//
// One CTA = 128 query rows of one (request, kv head): TQ = 128 / G tokens x
// the G query heads of the kv head, so every K/V tile serves the whole GQA
// group.  Warps 0-3 ("compute", thread t = query row t) rotate keys and run the
// softmax; warp 4 lane 0 issues TMA copies and tcgen05 MMAs.  Per 128-key tile:
//   1. TMA: the 8 (block, head) K~ tiles into a [half][128 keys][128 B]
//      128-byte-swizzled buffer (the tensor core's K-major B layout), the V tiles
//      into the same layout (read as an MN-major B operand), and the 8 cos/sin
//      table rows of the blocks' start positions.
//   2. compute warps rotate K~ in place: cos/sin of start + slot come from the
//      staged start row and the slot row (angle addition; slot rows 0..15 are
//      CTA constants in registers).
//   3. S = Q K'^T  (M 128, N 128, fp32 in TMEM columns [0, 128)).
//   4. each thread loads its S row, masks, updates its running max (O is
//      rescaled only when the max grew by more than 2^8) and writes P (bf16)
//      over the S columns.
//   5. O += P V with P read from TMEM (TMEM columns [128, 128 + d)).
// The next tile's K is loaded as soon as step 3 finishes with the buffer, and
// its V as soon as step 5 does; a second CTA on the SM overlaps the phases.
#pragma once

#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace minipic {
namespace prefill_impl {

using ptx::U4;

constexpr int kCompute = 128;           // compute threads (4 warps)
constexpr int kThreads = kCompute + 32; // + the TMA / MMA warp
constexpr int BN = 128;                 // keys per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;         // log2 growth of the row max that forces an O rescale

enum Bar { kBarQ = 0, kBarKFull, kBarKRot, kBarS, kBarP, kBarVFull, kBarPV, kNumBars };

template <int D>
struct PG {
  static constexpr int HALVES = D / 64;
  static constexpr int TILE = HALVES * BN * 128;      // Q, K or V tile bytes
  static constexpr int ROWB = 4 * D;                  // one cos|sin table row
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE;
  static constexpr int OFF_V = OFF_K + TILE;
  static constexpr int OFF_RS = OFF_V + TILE;         // 8 block-start rows
  static constexpr int OFF_META = OFF_RS + 8 * ROWB;  // int start[8], int flag[8], int phys[8], uint mask[2][4]
  static constexpr int OFF_BAR = OFF_META + 128;
  static constexpr int OFF_TSLOT = OFF_BAR + kNumBars * 8;
  static constexpr int TOTAL = OFF_TSLOT + 16;
  static constexpr int NFG = D / 16;                  // frequency groups of 8 (rotation work split)
  static constexpr int SPT = 16 * NFG / 32;           // slots per thread (4 for d 128, 2 for d 64)
  static constexpr uint32_t TCOLS = 256;              // S/P [0,128), O [128, 128 + D)
};

struct PrefillLaunch {
  PrefillArgs a;
  int tq;  // query tokens per 128-row tile (= 128 / G)
};

__device__ __forceinline__ uint32_t swz(int key, int chunk) {
  return (uint32_t)(key * 128 + ((chunk ^ (key & 7)) << 4));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One prefill CTA: query tile mt (of n_qt) of kv head hk of request r.
template <int D, bool ROPE>
__device__ __forceinline__ void prefill_cta(const CUtensorMap* kmap_p, const CUtensorMap* vmap_p,
                                            const PrefillLaunch& L, const int mt, const int n_qt, const int hk,
                                            const int r, uint8_t* smem_raw) {
  using G_ = PG<D>;
  const PrefillArgs& a = L.a;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const uint32_t sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sbase - ptx::smem_addr(smem_raw));
  int* meta_start = reinterpret_cast<int*>(sg + G_::OFF_META);
  int* meta_flag = meta_start + 8;
  uint32_t* meta_mask = reinterpret_cast<uint32_t*>(meta_start + 24);  // [2][4]
  const uint32_t bar0 = sbase + G_::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sg + G_::OFF_TSLOT);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.G, TQ = L.tq, mb = a.max_blocks;

  const int q0 = a.cu_q_lens[r];
  const int ql = a.cu_q_lens[r + 1] - q0;
  const int tok0 = mt * TQ;
  if (tid == 0 && mt == n_qt - 1 && ql > n_qt * TQ) atomicOr(a.err, kErrSeqLen);  // q_len > max_q_len
  if (ql <= 0 || tok0 >= ql) return;
  const int ntok = min(TQ, ql - tok0);
  int kvl = a.kv_lens[r];
  if (kvl < ql || kvl > mb * 16) {
    if (tid == 0 && mt == 0) atomicOr(a.err, kErrSeqLen);
    kvl = min(kvl, mb * 16);
  }
  const int nblk = (kvl + 15) >> 4;
  const int lim_last = kvl - ql + tok0 + ntok - 1;  // largest key index any row of the tile sees
  const int lim_first = kvl - ql + tok0;            // ... the first row sees
  const int n_kt = lim_last >= 0 ? lim_last / BN + 1 : 0;

  // ------------------------------------------------------------ setup
  if (tid == kCompute) {
    ptx::mbar_init(bar(kBarQ), kCompute);
    ptx::mbar_init(bar(kBarKFull), 1);
    ptx::mbar_init(bar(kBarKRot), kCompute);
    ptx::mbar_init(bar(kBarS), 1);
    ptx::mbar_init(bar(kBarP), kCompute);
    ptx::mbar_init(bar(kBarVFull), 1);
    ptx::mbar_init(bar(kBarPV), 1);
    ptx::fence_barrier_init();
  }
  if (warp == 0) {
    umma::tmem_alloc(ptx::smem_addr(tslot), G_::TCOLS);
    umma::tmem_relinquish();
  }
  if (tid < 8) meta_mask[tid] = 0u;
  // zero K and V buffers once so that never-loaded blocks hold finite values
  for (int i = tid; i < 2 * G_::TILE / 16; i += kThreads)
    reinterpret_cast<uint4*>(sg + G_::OFF_K)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;
  const uint32_t t_s = tmem;        // S / P columns
  const uint32_t t_o = tmem + 128;  // O columns

  bool failed = false;

  if (warp == kCompute / 32) {
    // ======================================================== TMA / MMA warp
    if (lane == 0) {
      const int* bt = a.block_tables + (size_t)r * mb;
      const int* bs = a.block_starts + (size_t)r * mb;
      // block ids / starts of the next tile to issue, loaded one tile ahead so that
      // their global-memory latency overlaps the MMA waits
      int nph[8], nst[8];
      int vph[8];  // block ids of the tile whose V is issued next
      auto load_meta = [&](int t) {
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          const int b = 8 * t + blk;
          nph[blk] = b < nblk ? __ldg(bt + b) : -1;
          nst[blk] = b < nblk ? __ldg(bs + b) : 0;
        }
      };
      auto issue_k = [&](int t) {
        // every compute thread has finished tile t - 2 (it arrived on the rotation
        // barrier of tile t - 1 before this issue), so this parity's words are free
#pragma unroll
        for (int w = 0; w < 4; ++w) meta_mask[(t & 1) * 4 + w] = 0u;
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
          meta_start[blk] = nst[blk];
          meta_flag[blk] = flag;
          vph[blk] = (flag & 1) ? nph[blk] : -1;
          nvalid += flag & 1;
          nrows += (ROPE && (flag & 3) == 3) ? 1 : 0;
        }
        ptx::mbar_arrive_expect_tx(bar(kBarKFull), nvalid * G_::HALVES * 2048 + nrows * G_::ROWB);
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          if (vph[blk] < 0) continue;
          const int y = (vph[blk] * a.Hkv + hk) * 16;
          for (int hh = 0; hh < G_::HALVES; ++hh)
            ptx::tma_load_2d(sbase + G_::OFF_K + hh * (BN * 128) + blk * 2048, &kmap, 64 * hh, y, bar(kBarKFull));
          if (ROPE && (meta_flag[blk] & 3) == 3)
            ptx::bulk_load(sbase + G_::OFF_RS + blk * G_::ROWB, a.cos_sin + (size_t)nst[blk] * D, G_::ROWB,
                           bar(kBarKFull));
        }
      };
      auto issue_v = [&]() {
        int nvalid = 0;
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) nvalid += vph[blk] >= 0 ? 1 : 0;
        ptx::mbar_arrive_expect_tx(bar(kBarVFull), nvalid * G_::HALVES * 2048);
#pragma unroll
        for (int blk = 0; blk < 8; ++blk) {
          if (vph[blk] < 0) continue;
          const int y = (vph[blk] * a.Hkv + hk) * 16;
          for (int hh = 0; hh < G_::HALVES; ++hh)
            ptx::tma_load_2d(sbase + G_::OFF_V + hh * (BN * 128) + blk * 2048, &vmap, 64 * hh, y, bar(kBarVFull));
        }
      };
      if (n_kt > 0) {
        load_meta(0);
        issue_k(0);
        issue_v();
        if (n_kt > 1) load_meta(1);
      }
      // rotated operands are f16 (10-bit mantissa); the rotation-free variant feeds bf16 as stored
      const uint32_t id_qk = ROPE ? umma::idesc_f16_f32(128, BN, false, false) : umma::idesc_bf16_f32(128, BN, false, false);
      const uint32_t id_pv = umma::idesc_bf16_f32(128, D, false, true);
      if (!ptx::mbar_wait(bar(kBarQ), 0)) failed = true;
      for (int t = 0; t < n_kt && !failed; ++t) {
        const uint32_t par = t & 1;
        if (!ptx::mbar_wait(bar(kBarKRot), par)) { failed = true; break; }
        umma::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t off = (ks >> 2) * (BN * 128) + (ks & 3) * 32;
          umma::mma_ss(t_s, umma::smem_desc_sw128(sbase + G_::OFF_Q + off, 16, 1024),
                       umma::smem_desc_sw128(sbase + G_::OFF_K + off, 16, 1024), id_qk, ks > 0);
        }
        umma::commit(bar(kBarS));
        if (!ptx::mbar_wait(bar(kBarS), par)) { failed = true; break; }
        if (t + 1 < n_kt) {
          issue_k(t + 1);  // also records the tile's block ids for its V issue
          if (t + 2 < n_kt) load_meta(t + 2);
        }
        if (!ptx::mbar_wait(bar(kBarP), par)) { failed = true; break; }
        if (!ptx::mbar_wait(bar(kBarVFull), par)) { failed = true; break; }
        umma::fence_after_sync();
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t vd = umma::smem_desc_sw128(sbase + G_::OFF_V + ks * 2048, BN * 128, 1024);
          umma::mma_ts(t_o, t_s + 8 * ks, vd, id_pv, (t > 0 || ks > 0) ? 1u : 0u);
        }
        umma::commit(bar(kBarPV));
        if (!ptx::mbar_wait(bar(kBarPV), par)) { failed = true; break; }
        if (t + 1 < n_kt) issue_v();
      }
      if (failed) atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ======================================================== compute warps
    const int row = tid;
    const int rtok = row / G, rh = row - rtok * G;
    const bool row_ok = rtok < ntok;
    const int tq = tok0 + rtok;                  // token index inside the chunk
    const int lim = kvl - ql + tq;               // last key this row attends
    const float qs = a.scale * kLog2e;

    // ---- Q: load, rotate at its position, scale, store in the K-major SW128 layout
    {
      U4 qc[D / 8];
      const __nv_bfloat16* qp = static_cast<const __nv_bfloat16*>(a.q) +
                                ((size_t)(q0 + tq) * a.Hq + (size_t)hk * G + rh) * D;
      int pos = 0;
      if (row_ok) {
        pos = ROPE ? a.q_pos[q0 + tq] : 0;
        if (ROPE && (pos < 0 || pos >= a.max_pos)) {
          atomicOr(a.err, kErrPosition);
          pos = 0;
        }
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(qp) + c);
          qc[c] = U4{v.x, v.y, v.z, v.w};
        }
      } else {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) qc[c] = U4{0u, 0u, 0u, 0u};
      }
      if constexpr (!ROPE) {
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          U4& x = qc[c];
          x = U4{ptx::pack_bf16(ptx::bf_lo(x.x) * qs, ptx::bf_hi(x.x) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.y) * qs, ptx::bf_hi(x.y) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.z) * qs, ptx::bf_hi(x.z) * qs),
                 ptx::pack_bf16(ptx::bf_lo(x.w) * qs, ptx::bf_hi(x.w) * qs)};
        }
      }
      const float* trow = ROPE ? a.cos_sin + (size_t)pos * D : nullptr;
#pragma unroll
      for (int c = 0; c < (ROPE ? D / 16 : 0); ++c) {  // chunk c pairs with chunk c + D/16
        uint64_t c2[4], s2[4];
        const float4 ca = __ldg(reinterpret_cast<const float4*>(trow + 8 * c));
        const float4 cb = __ldg(reinterpret_cast<const float4*>(trow + 8 * c + 4));
        const float4 sa = __ldg(reinterpret_cast<const float4*>(trow + D / 2 + 8 * c));
        const float4 sb = __ldg(reinterpret_cast<const float4*>(trow + D / 2 + 8 * c + 4));
        c2[0] = ptx::f2(ca.x * qs, ca.y * qs); c2[1] = ptx::f2(ca.z * qs, ca.w * qs);
        c2[2] = ptx::f2(cb.x * qs, cb.y * qs); c2[3] = ptx::f2(cb.z * qs, cb.w * qs);
        s2[0] = ptx::f2(sa.x * qs, sa.y * qs); s2[1] = ptx::f2(sa.z * qs, sa.w * qs);
        s2[2] = ptx::f2(sb.x * qs, sb.y * qs); s2[3] = ptx::f2(sb.z * qs, sb.w * qs);
        U4& x = qc[c];
        U4& y = qc[c + D / 16];
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
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint32_t addr = sbase + G_::OFF_Q + (c >> 3) * (BN * 128) + swz(row, c & 7);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(qc[c].x), "r"(qc[c].y),
                     "r"(qc[c].z), "r"(qc[c].w)
                     : "memory");
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(kBarQ));
    }

    // ---- rotation work split: thread -> (frequency group fg, slot group sgp, blocks w and w + 4)
    const int fg = tid % G_::NFG;
    const int sgp = (tid / G_::NFG) % (32 / G_::NFG);
    const int bsel = warp;  // blocks bsel and bsel + 4
    // slot rotation constants cos/sin(s theta_f), f = 8 fg .. 8 fg + 7, for this thread's slots
    uint64_t rsc[G_::SPT][4], rss[G_::SPT][4];
#pragma unroll
    for (int u = 0; u < (ROPE ? G_::SPT : 0); ++u) {
      const int slot = sgp * G_::SPT + u;
      const float* t = a.cos_sin + (size_t)min(slot, a.max_pos - 1) * D;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 c = __ldg(reinterpret_cast<const float2*>(t + 8 * fg + 2 * e));
        const float2 s = __ldg(reinterpret_cast<const float2*>(t + D / 2 + 8 * fg + 2 * e));
        rsc[u][e] = ptx::f2(c.x, c.y);
        rss[u][e] = ptx::f2(s.x, s.y);
      }
    }

    float m_run = -CUDART_INF_F;  // running max (log2 units)
    float m_use = -CUDART_INF_F;  // max the accumulators are scaled to
    float l_run = 0.f;

    for (int t = 0; t < n_kt; ++t) {
      const uint32_t par = t & 1;
      // tcgen05.ld/st below are warp-collective: every decision that skips them is warp-uniform
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarKFull), par))) { failed = true; break; }

      // ---- rotate this thread's keys of the tile in place
      bool kvalid[2][G_::SPT];
#pragma unroll
      for (int bb = 0; bb < 2; ++bb) {
        const int blk = bsel + 4 * bb;
        const int flag = meta_flag[blk];
        const int start = meta_start[blk];
        uint64_t ac[4], as[4];  // cos/sin(start theta_f)
        if (ROPE && (flag & 2)) {
          const uint32_t rb = sbase + G_::OFF_RS + blk * G_::ROWB;
          const U4 c0 = ptx::lds128(rb + 32 * fg), c1 = ptx::lds128(rb + 32 * fg + 16);
          const U4 s0 = ptx::lds128(rb + 2 * D + 32 * fg), s1 = ptx::lds128(rb + 2 * D + 32 * fg + 16);
          ac[0] = ((uint64_t)c0.y << 32) | c0.x; ac[1] = ((uint64_t)c0.w << 32) | c0.z;
          ac[2] = ((uint64_t)c1.y << 32) | c1.x; ac[3] = ((uint64_t)c1.w << 32) | c1.z;
          as[0] = ((uint64_t)s0.y << 32) | s0.x; as[1] = ((uint64_t)s0.w << 32) | s0.z;
          as[2] = ((uint64_t)s1.y << 32) | s1.x; as[3] = ((uint64_t)s1.w << 32) | s1.z;
        }
#pragma unroll
        for (int u = 0; u < G_::SPT; ++u) {
          const int slot = sgp * G_::SPT + u;
          const int key = blk * 16 + slot;
          const int pos = start + slot;
          const bool v = (flag & 3) == 3 && 8 * t * 16 + key < kvl && (!ROPE || pos < a.max_pos);
          kvalid[bb][u] = v;
          if (!ROPE || !v) continue;
          // cos/sin((start + slot) theta) by angle addition
          uint64_t c2[4], s2[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            c2[e] = ptx::sub2(ptx::mul2(ac[e], rsc[u][e]), ptx::mul2(as[e], rss[u][e]));
            s2[e] = ptx::fma2(as[e], rsc[u][e], ptx::mul2(ac[e], rss[u][e]));
          }
          uint32_t ax, ay;
          if constexpr (D == 128) {
            ax = sbase + G_::OFF_K + swz(key, fg);
            ay = ax + BN * 128;
          } else {
            ax = sbase + G_::OFF_K + swz(key, fg);
            ay = sbase + G_::OFF_K + swz(key, fg + 4);
          }
          const U4 x = ptx::lds128(ax), y = ptx::lds128(ay);
          uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t xv = ptx::bf2_to_f2(xw[k]), yv = ptx::bf2_to_f2(yw[k]);
            xw[k] = ptx::f2_to_h2(ptx::sub2(ptx::mul2(xv, c2[k]), ptx::mul2(yv, s2[k])));
            yw[k] = ptx::f2_to_h2(ptx::fma2(xv, s2[k], ptx::mul2(yv, c2[k])));
          }
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ax), "r"(xw[0]), "r"(xw[1]), "r"(xw[2]),
                       "r"(xw[3])
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(ay), "r"(yw[0]), "r"(yw[1]), "r"(yw[2]),
                       "r"(yw[3])
                       : "memory");
        }
      }
      // key validity of the tile as a 128-bit mask, one word per 32 keys
      if (fg == 0) {
        // one thread per (block, slot group) records validity bits
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          uint32_t bits = 0;
          const int blk = bsel + 4 * bb;
#pragma unroll
          for (int u = 0; u < G_::SPT; ++u)
            if (kvalid[bb][u]) bits |= 1u << ((blk & 1) * 16 + sgp * G_::SPT + u);
          atomicOr(&meta_mask[par * 4 + (blk >> 1)], bits);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(kBarKRot));

      // ---- softmax of this thread's S row
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarS), par))) { failed = true; break; }
      umma::fence_after_sync();
      const uint32_t lane_base = ((uint32_t)(warp * 32) << 16);
      const uint32_t mw[4] = {meta_mask[par * 4 + 0], meta_mask[par * 4 + 1], meta_mask[par * 4 + 2],
                              meta_mask[par * 4 + 3]};
      const bool full = (mw[0] & mw[1] & mw[2] & mw[3]) == 0xffffffffu && t * BN + BN - 1 <= lim_first;
      // pass 1: row max of the allowed scores
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int part = 0; part < BN / 32; ++part) {
        uint32_t v[32];
        umma::tmem_ld32(t_s + lane_base + part * 32, v);
        umma::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const bool ok = full || (row_ok && ((mw[part] >> j) & 1u) && (t * BN + part * 32 + j <= lim));
          mx = ok ? fmaxf(mx, __uint_as_float(v[j])) : mx;
        }
      }
      m_run = fmaxf(m_run, mx);
      // move the accumulators to a new reference max when this row's max grew by more than 2^8;
      // the TMEM pass is warp-collective, so lanes without a change scale by 1
      const bool need = m_run != -CUDART_INF_F && (m_use == -CUDART_INF_F || m_run > m_use + kRescale);
      const float corr = !need ? 1.f : (m_use == -CUDART_INF_F ? 0.f : ex2(m_use - m_run));
      if (need) {
        l_run *= corr;
        m_use = m_run;
      }
      if (t > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int part = 0; part < D / 32; ++part) {
          uint32_t v[32];
          umma::tmem_ld32(t_o + lane_base + part * 32, v);
          umma::tmem_wait_ld();
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            w0[j] = __float_as_uint(__uint_as_float(v[j]) * corr);
            w1[j] = __float_as_uint(__uint_as_float(v[16 + j]) * corr);
          }
          umma::tmem_st16(t_o + lane_base + part * 32, w0);
          umma::tmem_st16(t_o + lane_base + part * 32 + 16, w1);
        }
      }
      const float mref = m_use == -CUDART_INF_F ? 0.f : m_use;
      // pass 2: P = 2^(s - mref) (0 where masked), row sum, bf16 pairs over the S columns
      float lsum = 0.f;
#pragma unroll
      for (int part = 0; part < BN / 32; ++part) {
        uint32_t v[32];
        umma::tmem_ld32(t_s + lane_base + part * 32, v);
        umma::tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int j0 = 2 * j, j1 = 2 * j + 1;
          const bool ok0 = full || (row_ok && ((mw[part] >> j0) & 1u) && (t * BN + part * 32 + j0 <= lim));
          const bool ok1 = full || (row_ok && ((mw[part] >> j1) & 1u) && (t * BN + part * 32 + j1 <= lim));
          const float p0 = ok0 ? ex2(__uint_as_float(v[j0]) - mref) : 0.f;
          const float p1 = ok1 ? ex2(__uint_as_float(v[j1]) - mref) : 0.f;
          lsum += p0 + p1;
          w[j] = ptx::pack_bf16(p0, p1);
        }
        umma::tmem_st16(t_s + lane_base + part * 16, w);
      }
      l_run += lsum;
      umma::tmem_wait_st();
      umma::fence_before_sync();
      ptx::mbar_arrive(bar(kBarP));
    }

    // ---- epilogue: O / l -> global (TMEM loads by the whole warp, stores by valid rows)
    bool have = n_kt > 0 && !failed;
    if (have && !__all_sync(0xffffffffu, ptx::mbar_wait(bar(kBarPV), (n_kt - 1) & 1))) {
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
        umma::tmem_ld32(t_o + ((uint32_t)(warp * 32) << 16) + part * 32, v);
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
  if (warp == 0) umma::tmem_dealloc(tmem, G_::TCOLS);
}

}  // namespace prefill_impl
}  // namespace minipic
