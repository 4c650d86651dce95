// Decode attention over the position-free paged cache, bf16 tensor-core form
// (CTA body shared by the decode kernel and the mixed prefill + decode kernel).
//
// Method (MiniPIC summary, gist.science 2606.13126, section 2.1): keys are
// stored unrotated; the kernel rotates them at their logical position
// pi(j) = start[r][block] + slot with a cos/sin table lookup and multiply-adds
// per key element, then runs ordinary softmax attention.
//
// Layout of the work.  One CTA = (split, kv head, request); each of its warps
// owns every NW-th block of the split and runs its own TMA ring of NS stages
// (the standalone kernel: 4 warps, 2 stages with 3 CTAs per SM or 3 stages with
// 2): the (block, head) K and V tiles (16 keys x d, contiguous in the pool)
// arrive by cp.async.bulk.tensor with 128-byte swizzle (at head dim 128 one box
// per tile over a 3-D view of the pool), in a [half][key][64] shared layout
// that makes both the 16-byte key-row reads and the transposing ldmatrix reads
// of V free of bank conflicts.
//
// Per 16-key block and GQA group (up to 8 query heads per n-tile):
//   S^T[key][head] = K'[key][:] . Q'[head][:]  (mma m16n8k16, M = the 16 keys)
//   O^T[dim][head] += V^T[dim][key] P^T[key][head]
// K' is formed in registers: rows are read from shared memory and rotated in
// packed bf16 arithmetic (two bf16x2 multiply / multiply-adds per pair of
// elements) straight into the MMA's bf16 A operand; Q' likewise.  The
// contraction order of the head dimension is a per-thread permutation chosen
// so that each rotary pair (i, i + d/2) is thread-local; Q' uses the same
// permutation.
//
// Rotation is factored per block: with s = slot and b = block start,
//   (R_t q)^T (R_{b+s} k~) = (R_{t-b} q)^T (R_s k~),
// so q is re-rotated once per block by the rotation of the signed angle t - b
// and each key row by the constant R_s (s < 16) held in registers.
// This is the same algebra as rotating k~ by R_{pi(j)}; it reads one table
// row per block instead of sixteen.  The rows are the bf16 form of the table
// over signed angles (cos | sin | -sin of t - b, 384 bytes at d 128): the
// rotation reads its bf16 operands directly, whatever the sign of t - b.
#pragma once

#include <math_constants.h>

#include "internal.h"
#include "ptx.cuh"

namespace minipic {
namespace decode_impl {

using ptx::U4;

constexpr int kWarps = 4;
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Geo {
  static constexpr int TILE = 16 * D * 2;     // bytes of one (block, head) tile of K or V
  static constexpr int NCH = D / 32;          // 16-byte chunks of a key row read by one thread
  static constexpr int NPAIR = NCH / 2;       // rotary chunk pairs per row and thread
  static constexpr int MT = D / 16;           // m-tiles of O^T
  static constexpr int HALVES = D / 64;       // 128-byte halves of a key row
  static constexpr int STAGE = 2 * TILE;
};

// Which 16-byte chunk (0..7 within a 128-byte half) and which half thread
// `tig` reads as its i-th chunk of a key row, and the rotary pairing: thread
// tig owns chunks tig and tig + 4 of every half, so each rotary pair
// (i, i + d/2) is thread-local and every shared read below is conflict-free.
template <int D>
struct Chunks {
  int c[Geo<D>::NCH];
  int h[Geo<D>::NCH];
  int first[Geo<D>::NPAIR], second[Geo<D>::NPAIR];
  int fbase[Geo<D>::NPAIR];  // first frequency index of the pair's 8 elements
  __device__ __forceinline__ explicit Chunks(int tig) {
    if constexpr (D == 128) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        h[i] = i >> 1;
        c[i] = tig + 4 * (i & 1);
      }
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        first[p] = p;
        second[p] = p + 2;
        fbase[p] = 8 * (tig + 4 * p);
      }
    } else {
      c[0] = tig;
      c[1] = tig + 4;
      h[0] = h[1] = 0;
      first[0] = 0;
      second[0] = 1;
      fbase[0] = 8 * tig;
    }
  }
};

// Physical key (slot) held by MMA fragment row g (g < 8; row g + 8 holds
// slot + 8).  Rows read together by a quarter warp then differ in bit 2 of the
// slot, which keeps the swizzled key-row reads conflict-free.
__device__ __forceinline__ int frag_slot(int g) { return (g >> 1) | ((g & 1) << 2); }

// Byte offset of (half, key, chunk) in a swizzled [half][16 keys][128 B] tile.
__device__ __forceinline__ uint32_t swz(int half, int key, int chunk) {
  return (uint32_t)((half * 16 + key) * 128 + ((chunk ^ (key & 7)) << 4));
}

// Rotate one pair of 8-element bf16 chunks (rotary halves x, y) in packed bf16
// arithmetic: x' = bf16(y (-s) + bf16(x c)),  y' = bf16(x s + bf16(y c)), with
// c, s, -s as bf16 pairs.  Keys and queries feed a bf16 product, so they are
// rounded to bf16 anyway; the two extra roundings change the outputs by far
// less than the tolerance (checked against the oracle) and skip the fp32
// unpack / repack.
__device__ __forceinline__ void rotate_pair_bf16(U4& x, U4& y, const uint32_t (&c)[4], const uint32_t (&s)[4],
                                                 const uint32_t (&ns)[4]) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
  const uint32_t yw[4] = {y.x, y.y, y.z, y.w};
  uint32_t xo[4], yo[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    xo[k] = ptx::fma_bf2(yw[k], ns[k], ptx::mul_bf2(xw[k], c[k]));
    yo[k] = ptx::fma_bf2(xw[k], s[k], ptx::mul_bf2(yw[k], c[k]));
  }
  x = U4{xo[0], xo[1], xo[2], xo[3]};
  y = U4{yo[0], yo[1], yo[2], yo[3]};
}

__device__ __forceinline__ uint32_t w_of(const U4& v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Shared-memory plan of one CTA (offsets from a 1024-byte aligned base).
template <int D, int NW = kWarps, int NS = kStages>
struct Smem {
  static constexpr int STAGES = NW * NS * Geo<D>::STAGE;  // K|V tiles
  static constexpr int ROWB = 3 * D;                               // one bf16 cos|sin|-sin table row
  static constexpr int ROWS = STAGES;                              // [warp][stage] table rows
  static constexpr int META = ROWS + NW * NS * ROWB;      // [split block][phys, start]
  static constexpr int kMaxSplit = 512;                            // split_blocks cap (planner)
  static constexpr int BARS = META + kMaxSplit * 8;
  static constexpr int TOTAL = BARS + NW * NS * 8;
};

// One decode CTA: (split, kv head hk, request r) with NW working warps of NS
// stages each.  With BAR = 0 every thread of the block takes part in the CTA
// barriers (__syncthreads) and threads beyond the working warps only do that;
// with BAR > 0 only the first NW warps call this function and their barriers
// are the named barrier BAR over NW * 32 threads (the other warps of the block
// may have left).  With BLOCKMAP the tensor maps are 3-D views of the pools
// (64 columns x rows x 64-column halves) and one box brings a whole K or V tile
// of a block in the [half][key][64] layout: one copy instead of two.
template <int D, int NT, bool ROPE, int NW = kWarps, int NS = kStages, int BAR = 0, bool BLOCKMAP = false>
__device__ __forceinline__ void decode_cta(const CUtensorMap* kmap_p, const CUtensorMap* vmap_p,
                                           const DecodeArgs& a, const int split, const int hk, const int r,
                                           uint8_t* smem_raw) {
  using GE = Geo<D>;
  using SM = Smem<D, NW, NS>;
  const CUtensorMap& kmap = *kmap_p;
  const CUtensorMap& vmap = *vmap_p;
  const uint32_t sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - ptx::smem_addr(smem_raw));
  const uint32_t bar_base = sbase + SM::BARS;
  int* meta = reinterpret_cast<int*>(sgen + SM::META);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g8 = lane >> 2, tig = lane & 3;
  const int nthr = BAR > 0 ? NW * 32 : (int)blockDim.x;  // threads in the CTA barriers
  auto cta_sync = [&]() {
    if constexpr (BAR > 0) ptx::named_sync(BAR, NW * 32);
    else __syncthreads();
  };
  const int G = a.G;
  const bool worker = warp < NW;
  const int mb = a.max_blocks;

  int L = a.seq_lens[r];
  const int Lmax = mb * 16;
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && split == 0) atomicOr(a.err, kErrSeqLen);
    L = L < 0 ? 0 : Lmax;
  }
  const int nblk = (L + 15) >> 4;
  const int n_valid = max(1, (nblk + a.split_blocks - 1) / a.split_blocks);
  if (split >= n_valid) return;
  const int b_begin = split * a.split_blocks;
  const int b_end = min(nblk, b_begin + a.split_blocks);
  const int span = b_end - b_begin;
  const int nmine = (worker && span > warp) ? (span - warp + NW - 1) / NW : 0;

  // lane 0: issue the k-th block of this warp (physical block phys, start
  // position start, query position tqv) into its stage: K and V tiles by TMA,
  // plus the bf16 table row of the angle tqv - start (row |tqv - start|, sign
  // part 1 when negative) the block's query rotation needs
  auto issue_blk = [&](int k, int phys, int start, int tqv) {
    const int stg = k % NS;
    const uint32_t bar = bar_base + (warp * NS + stg) * 8;
    const uint32_t kdst = sbase + (warp * NS + stg) * GE::STAGE;
    if (phys < 0 || phys >= a.num_blocks) {
      ptx::mbar_arrive(bar);  // nothing to load; the consumer masks the block
      return;
    }
    int ad = 0, neg = 0;
    bool row_ok = false;
    if constexpr (ROPE) {
      const int delta = tqv - start;
      ad = delta < 0 ? -delta : delta;
      neg = delta < 0 ? 1 : 0;
      row_ok = ad < a.max_pos;
    }
    ptx::mbar_arrive_expect_tx(bar, 2 * GE::TILE + (row_ok ? SM::ROWB : 0));
    const int y = (phys * a.Hkv + hk) * 16;
    if constexpr (BLOCKMAP) {
      ptx::tma_load_3d(kdst, &kmap, 0, y, 0, bar);
      ptx::tma_load_3d(kdst + GE::TILE, &vmap, 0, y, 0, bar);
    } else {
#pragma unroll
      for (int hh = 0; hh < GE::HALVES; ++hh) {
        ptx::tma_load_2d(kdst + hh * 2048, &kmap, 64 * hh, y, bar);
        ptx::tma_load_2d(kdst + GE::TILE + hh * 2048, &vmap, 64 * hh, y, bar);
      }
    }
    if (row_ok)
      ptx::bulk_load(sbase + SM::ROWS + (warp * NS + stg) * SM::ROWB,
                     a.cs_bf16 + ((size_t)ad * 2 + neg) * (3 * D / 2), SM::ROWB, bar);
  };

  // Each worker warp's lane 0 initialises its stage barriers.  With 3 stages
  // or more (the standalone layout for HBM-bound long contexts) it also starts
  // the copies of its first blocks at once, from the table entries in global
  // memory, so that they overlap the staging and the query setup below (the
  // staged entries serve the later blocks).  Measured: long contexts 0.563 ->
  // 0.544 ms; with 2 stages (L2-served batches, the mixed grid) it was slower.
  constexpr bool kEarly = NS >= 3 && BAR == 0;
  {
    const int* bt = a.block_tables + (size_t)r * mb + b_begin;
    const int* bs_ = a.block_starts + (size_t)r * mb + b_begin;
    if (worker && lane == 0) {
#pragma unroll
      for (int st = 0; st < NS; ++st) ptx::mbar_init(bar_base + (warp * NS + st) * 8, 1);
      ptx::fence_barrier_init();
      ptx::fence_proxy_async_smem();
    }
    if (kEarly && worker && lane == 0) {
      int tq0 = 0;
      if constexpr (ROPE) {
        tq0 = a.q_pos[r];
        if (tq0 < 0 || tq0 >= a.max_pos) tq0 = 0;  // flagged below; the same value the loop uses
      }
      const int pre = nmine < NS ? nmine : NS;
      for (int k = 0; k < pre; ++k) {
        const int i = warp + NW * k;
        issue_blk(k, __ldg(bt + i), ROPE ? __ldg(bs_ + i) : 0, tq0);
      }
    }
    // block ids and start positions of the whole split, staged once
    for (int i = threadIdx.x; i < span; i += nthr) {
      meta[2 * i] = __ldg(bt + i);
      meta[2 * i + 1] = ROPE ? __ldg(bs_ + i) : 0;
    }
  }

  const Chunks<D> ch(tig);
  const int ks0 = frag_slot(g8);  // this thread's key rows: slots ks0 and ks0 + 8

  // unrotated queries of this thread's heads (g8 + 8 nt), in the thread's chunk order
  U4 qraw[NT][GE::NCH];
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int head = 8 * nt + g8;
#pragma unroll
    for (int i = 0; i < GE::NCH; ++i) {
      if (head < G) {
        const __nv_bfloat16* p = qg + ((size_t)r * a.Hq + (size_t)hk * G + head) * D + 64 * ch.h[i] + 8 * ch.c[i];
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
        qraw[nt][i] = U4{v.x, v.y, v.z, v.w};
      } else {
        qraw[nt][i] = U4{0u, 0u, 0u, 0u};
      }
    }
  }
  const float qs = a.scale * kLog2e;  // applied to the scores; softmax runs in base 2

  // R_s for the two key rows (slots ks0, ks0 + 8) of this thread: cos and sin
  // of the slot angles as bf16 pairs (-sin is formed at use: holding it too
  // would make the three-CTA build spill)
  uint32_t rcb[2][GE::NPAIR][4], rsb[2][GE::NPAIR][4];
  int tq = 0;
  if constexpr (ROPE) {
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const int srow = min(ks0 + 8 * row, a.max_pos - 1);
      const float* t = a.cos_sin + (size_t)srow * D;
#pragma unroll
      for (int p = 0; p < GE::NPAIR; ++p) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 c = __ldg(reinterpret_cast<const float2*>(t + ch.fbase[p] + 2 * e));
          const float2 sn = __ldg(reinterpret_cast<const float2*>(t + D / 2 + ch.fbase[p] + 2 * e));
          rcb[row][p][e] = ptx::pack_bf16(c.x, c.y);
          rsb[row][p][e] = ptx::pack_bf16(sn.x, sn.y);
        }
      }
    }
    tq = a.q_pos[r];
    if (tq < 0 || tq >= a.max_pos) {
      if (threadIdx.x == 0 && split == 0) atomicOr(a.err, kErrPosition);
      tq = 0;
    }
  }
  U4 qw[NT][GE::NCH];
  if constexpr (!ROPE) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < GE::NCH; ++i) qw[nt][i] = qraw[nt][i];
  }

  float mrun[NT][2], lrun[NT][2];
  float oacc[GE::MT][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    mrun[nt][0] = mrun[nt][1] = -CUDART_INF_F;
    lrun[nt][0] = lrun[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < GE::MT; ++mt)
#pragma unroll
      for (int k = 0; k < 4; ++k) oacc[mt][nt][k] = 0.f;
  }

  cta_sync();  // meta visible

  // lane 0: issue the k-th block of this warp (from the staged entries)
  auto issue = [&](int k) {
    const int i = warp + NW * k;
    issue_blk(k, meta[2 * i], meta[2 * i + 1], tq);
  };
  if (!kEarly && lane == 0) {
    const int pre = nmine < NS ? nmine : NS;
    for (int k = 0; k < pre; ++k) issue(k);
  }

  bool timed_out = false;
  int k_stop = nmine;
  for (int k = 0; k < nmine; ++k) {
    const int i = warp + NW * k;
    const int b = b_begin + i;
    const int stg = k % NS;
    const uint32_t bar = bar_base + (warp * NS + stg) * 8;
    const uint32_t kbase = sbase + (warp * NS + stg) * GE::STAGE;
    const uint32_t vbase = kbase + GE::TILE;
    const uint32_t rowb = sbase + SM::ROWS + (warp * NS + stg) * SM::ROWB;

    const int phys = meta[2 * i];
    const bool ok = phys >= 0 && phys < a.num_blocks;
    const int start = meta[2 * i + 1];
    const int nk = min(16, L - b * 16);
    bool v0 = ok && ks0 < nk, v1 = ok && ks0 + 8 < nk;
    if (!ok && lane == 0) atomicOr(a.err, kErrBlockId);
    int delta = 0;
    if constexpr (ROPE) {
      delta = tq - start;
      const int ad = delta < 0 ? -delta : delta;
      if (ok && !(ad < a.max_pos && start >= 0 && start + nk - 1 < a.max_pos)) {
        // keys whose position falls outside the table are masked
        const bool p0 = start + ks0 >= 0 && start + ks0 < a.max_pos && ad < a.max_pos;
        const bool p1 = start + ks0 + 8 >= 0 && start + ks0 + 8 < a.max_pos && ad < a.max_pos;
        if (__any_sync(0xffffffffu, (v0 && !p0) || (v1 && !p1)) && lane == 0) atomicOr(a.err, kErrPosition);
        v0 = v0 && p0;
        v1 = v1 && p1;
      }
    }

    // wait for this block's tiles (bounded)
    const bool arrived = ptx::mbar_wait(bar, (uint32_t)((k / NS) & 1));
    if (!__all_sync(0xffffffffu, arrived)) {
      if (lane == 0) atomicOr(a.err, kErrTimeout);
      timed_out = true;
      k_stop = k;
      break;
    }

    // re-rotate q by t - start from the staged bf16 row of that signed angle
    if constexpr (ROPE) {
#pragma unroll
      for (int p = 0; p < GE::NPAIR; ++p) {
        const U4 cw = ptx::lds128(rowb + 2 * ch.fbase[p]);
        const U4 sw = ptx::lds128(rowb + D + 2 * ch.fbase[p]);
        const U4 nw = ptx::lds128(rowb + 2 * D + 2 * ch.fbase[p]);
        const uint32_t cb[4] = {cw.x, cw.y, cw.z, cw.w};
        const uint32_t sb[4] = {sw.x, sw.y, sw.z, sw.w};
        const uint32_t nb[4] = {nw.x, nw.y, nw.z, nw.w};
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          U4 x = qraw[nt][ch.first[p]], y = qraw[nt][ch.second[p]];
          rotate_pair_bf16(x, y, cb, sb, nb);
          qw[nt][ch.first[p]] = x;
          qw[nt][ch.second[p]] = y;
        }
      }
    }

    // key rows g8 and g8 + 8 of the block, rotated by R_slot in registers
    U4 kr[2][GE::NCH];
#pragma unroll
    for (int row = 0; row < 2; ++row)
#pragma unroll
      for (int c = 0; c < GE::NCH; ++c) kr[row][c] = ptx::lds128(kbase + swz(ch.h[c], ks0 + 8 * row, ch.c[c]));
    if constexpr (ROPE) {
#pragma unroll
      for (int row = 0; row < 2; ++row)
#pragma unroll
        for (int p = 0; p < GE::NPAIR; ++p)
        {
          const uint32_t nn[4] = {rsb[row][p][0] ^ 0x80008000u, rsb[row][p][1] ^ 0x80008000u,
                                  rsb[row][p][2] ^ 0x80008000u, rsb[row][p][3] ^ 0x80008000u};
          rotate_pair_bf16(kr[row][ch.first[p]], kr[row][ch.second[p]], rcb[row][p], rsb[row][p], nn);
        }
    }

    // S^T = K' Q'^T, two independent accumulation chains (even / odd k-steps)
    float sacc[NT][4], sacc2[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] = sacc2[nt][e] = 0.f;
#pragma unroll
    for (int c = 0; c < GE::NCH; ++c) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t a0 = w_of(kr[0][c], 2 * u), a1 = w_of(kr[1][c], 2 * u);
        const uint32_t a2 = w_of(kr[0][c], 2 * u + 1), a3 = w_of(kr[1][c], 2 * u + 1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (u == 0)
            ptx::mma_bf16_16816(sacc[nt], a0, a1, a2, a3, w_of(qw[nt][c], 0), w_of(qw[nt][c], 1));
          else
            ptx::mma_bf16_16816(sacc2[nt], a0, a1, a2, a3, w_of(qw[nt][c], 2), w_of(qw[nt][c], 3));
        }
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sacc[nt][e] += sacc2[nt][e];

    // online softmax over the 16 keys, per head column (2 tig + j) of each n-tile
    uint32_t pb0[NT], pb1[NT];
    float corr[NT][2];
    bool any_corr = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float pv[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float sa = v0 ? sacc[nt][j] * qs : -CUDART_INF_F;
        const float sb = v1 ? sacc[nt][2 + j] * qs : -CUDART_INF_F;
        float bm = fmaxf(sa, sb);
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
        const float mnew = fmaxf(mrun[nt][j], bm);
        const float muse = mnew == -CUDART_INF_F ? 0.f : mnew;
        corr[nt][j] = exp2f(mrun[nt][j] - muse);
        any_corr |= mnew != mrun[nt][j];
        const float pa = exp2f(sa - muse), pbv = exp2f(sb - muse);
        lrun[nt][j] = fmaf(lrun[nt][j], corr[nt][j], pa + pbv);
        mrun[nt][j] = mnew;
        pv[j] = pa;
        pv[2 + j] = pbv;
      }
      pb0[nt] = ptx::movmatrix_trans(ptx::pack_bf16(pv[0], pv[1]));  // keys 0..7
      pb1[nt] = ptx::movmatrix_trans(ptx::pack_bf16(pv[2], pv[3]));  // keys 8..15
    }
    // rescale the accumulators only when some running max moved
    if (__any_sync(0xffffffffu, any_corr)) {
#pragma unroll
      for (int mt = 0; mt < GE::MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            oacc[mt][nt][j] *= corr[nt][j];
            oacc[mt][nt][2 + j] *= corr[nt][j];
          }
    }

    // O^T += V^T P^T
    {
      const int mi = lane >> 3, rr = lane & 7;
      const int key = frag_slot(rr) + 8 * (mi >> 1);
#pragma unroll
      for (int mt = 0; mt < GE::MT; ++mt) {
        const int cg = 2 * mt + (mi & 1);
        uint32_t a0, a1, a2, a3;
        ptx::ldsm_x4_trans(vbase + swz(cg >> 3, key, cg & 7), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ptx::mma_bf16_16816(oacc[mt][nt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
      }
    }

    __syncwarp();
    if (lane == 0 && k + NS < nmine) issue(k + NS);
  }

  if (timed_out) {
    // blocks k_stop .. k_stop + NS - 1 were issued and not consumed
    if (lane == 0) {
      const int last = min(nmine, k_stop + NS);
      for (int k2 = k_stop; k2 < last; ++k2) {
        const int stg = k2 % NS;
        ptx::mbar_wait(bar_base + (warp * NS + stg) * 8, (uint32_t)((k2 / NS) & 1), 100000000ull);
      }
    }
  }

  // per-warp state -> this warp's own stage region: m[16], l[16], O[16][D + 4]
  constexpr int OST = D + 4;  // padded row stride (conflict-free stores)
  float* wm = reinterpret_cast<float*>(sgen + warp * NS * GE::STAGE);
  float* wl = wm + 16;
  float* wo = wm + 32;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = lrun[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      lrun[nt][j] = l;
    }
  __syncwarp();
  if (worker && g8 == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        wm[8 * nt + 2 * tig + j] = mrun[nt][j];
        wl[8 * nt + 2 * tig + j] = lrun[nt][j];
      }
  }
  if (worker) {
#pragma unroll
    for (int mt = 0; mt < GE::MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int head = 8 * nt + 2 * tig + j;
          wo[head * OST + 16 * mt + g8] = oacc[mt][nt][j];
          wo[head * OST + 16 * mt + g8 + 8] = oacc[mt][nt][2 + j];
        }
  }
  cta_sync();

  const bool direct = (n_valid == 1);
  for (int idx = threadIdx.x; idx < G * D; idx += nthr) {
    const int head = idx / D, dim = idx - head * D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < NW; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(sgen + w * NS * GE::STAGE)[head]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float* base = reinterpret_cast<const float*>(sgen + w * NS * GE::STAGE);
      const float mw = base[head];
      const float f = mw == -CUDART_INF_F ? 0.f : exp2f(mw - M);
      Ls = fmaf(base[16 + head], f, Ls);
      O = fmaf(base[32 + head * OST + dim], f, O);
    }
    const int hq = hk * G + head;
    if (direct) {
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((size_t)r * a.Hq + hq) * D + dim;
      *out = __float2bfloat16_rn(Ls > 0.f ? O / Ls : 0.f);
      if (dim == 0 && a.lse) a.lse[(size_t)r * a.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
    } else {
      const size_t pi = ((size_t)r * a.Hq + hq) * a.n_split + split;
      a.part_o[pi * D + dim] = O;
      if (dim == 0) {
        a.part_ml[pi * 2] = M;
        a.part_ml[pi * 2 + 1] = Ls;
      }
    }
  }
  if (direct) return;

  // the last split of this (request, kv head) to finish merges all of them
  // (log-sum-exp across splits) and resets the counter for the next call
  __shared__ int s_last;
  cta_sync();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(a.counters + (size_t)r * a.Hkv + hk, 1);
    s_last = old == n_valid - 1;
  }
  cta_sync();
  if (!s_last) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < G * D; idx += nthr) {
    const int head = idx / D, dim = idx - head * D;
    const int hq = hk * G + head;
    const size_t base = ((size_t)r * a.Hq + hq) * a.n_split;
    float M = -CUDART_INF_F;
    for (int s = 0; s < n_valid; ++s) M = fmaxf(M, __ldcg(a.part_ml + (base + s) * 2));
    float Ls = 0.f, O = 0.f;
    for (int s = 0; s < n_valid; ++s) {
      const float ms = __ldcg(a.part_ml + (base + s) * 2);
      const float f = ms == -CUDART_INF_F ? 0.f : exp2f(ms - M);
      Ls = fmaf(__ldcg(a.part_ml + (base + s) * 2 + 1), f, Ls);
      O = fmaf(__ldcg(a.part_o + (base + s) * D + dim), f, O);
    }
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((size_t)r * a.Hq + hq) * D + dim;
    *out = __float2bfloat16_rn(Ls > 0.f ? O / Ls : 0.f);
    if (dim == 0 && a.lse) a.lse[(size_t)r * a.Hq + hq] = Ls > 0.f ? (M + log2f(Ls)) * kLn2 : -CUDART_INF_F;
  }
  if (threadIdx.x == 0) a.counters[(size_t)r * a.Hkv + hk] = 0;
}

}  // namespace decode_impl
}  // namespace minipic
