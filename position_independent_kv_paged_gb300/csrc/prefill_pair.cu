// Chunked prefill over the position-free paged cache, CTA-pair tcgen05 form
// (head dim 128).
//
// Method (MiniPIC summary, gist.science 2606.13126, section 2.1): stored keys
// are unrotated; each key is rotated at its logical position
// pi(j) = start[r][j / 16] + j % 16 with cos/sin values and multiply-adds per
// element, then softmax attention runs.  A request's query chunk (the last
// q_len of its kv_len keys) attends causally: chunk query i sees keys
// j <= kv_len - q_len + i.
//
// A cluster of two CTAs = (request r, kv head hk, query-tile pair): CTA c holds
// query tile 2 pair + c, i.e. TQ = 128 / G consecutive tokens x the G query
// heads of kv head hk (128 rows), and the pair issues every product as one
// tcgen05 MMA of M = 256 rows (cta_group::2):
//   S = Q K_t^T   A = Q from TMEM (each CTA its 128 rows), B = K~_t rotated;
//                 key tile t = 160 keys, keys 0-79 (blocks 0-4) held and
//                 rotated by CTA 0, keys 80-159 by CTA 1
//   O += P V_t    A = P from TMEM (bf16 over S), B = V_t; head dims 0-63
//                 held by CTA 0, 64-127 by CTA 1, all 160 keys
// so each key is fetched and rotated once per pair and every operand is half
// the size a single CTA would hold.  With A in TMEM an MMA costs about
// max(93, 9.5 + N / 2) SM cycles (measured), so a 160-wide QK^T product runs
// near the tensor core's peak, where the shared-memory form at 96 keys ran at
// two thirds of it.  Every stage and barrier lives in both CTAs at the same
// offsets; CTA 0's barriers gather what its tensor core waits for.
//
// Roles in each CTA (16 warps; at the top of its branch each warpgroup sets
// its register budget with setmaxnreg: softmax 176, rotation 96, the rest 64,
// so that the softmax keeps its 80 scores per thread in registers):
//   warps 0-7   softmax: warp w covers TMEM lanes 32 (w % 4).. (query rows)
//               and keys 80 (w / 4) .. +79 of the tile; the two warps of a
//               lane quarter combine their row maxima through shared memory;
//               warps 0-3 first write the rotated, scaled query tile to TMEM
//   warps 8-11  rotation of this CTA's 80 keys of every staged tile in
//               packed fp16 arithmetic, each thread reading the fp16 cos|sin
//               values of its keys' positions from the (L2-resident) table
//   warp 12     K~ producer: this CTA's K~ blocks by TMA, and the tile's key
//               masks, V block ids and block starts
//   warp 13     TMEM allocation; in CTA 0 the MMA issue, in CTA 1 a relay
//               that tells CTA 0 when its rotated keys are ready (one
//               cluster-scope release per tile, covering what it observed)
//   warp 14     V producer: this CTA's 64 head dims of every V block by TMA;
//               both CTAs' copies complete on CTA 0's V barrier
//   warp 15     idle (completes warpgroup 3 for the register split)
// (K~ and V have producers of their own, so that K~ tiles run NSK tiles ahead
// of the products whatever the V stages wait for.)
// S is double-buffered in TMEM, so QK^T of tile t+1 runs while the softmax
// works on tile t; the MMA order is QK(0), QK(1), then per t: PV(t), QK(t+2).
// O is rescaled only when a row maximum grows by more than 2^8.
#include <math_constants.h>

#include "decode_body.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tmap.cuh"
#include "umma.cuh"

namespace minipic {
namespace {

using ptx::U4;

constexpr int D = 128;
constexpr int kHalfBlocks = 5;                 // blocks of a key tile held by one CTA
constexpr int kTileBlocks = 2 * kHalfBlocks;   // blocks of a key tile
constexpr int BN = 16 * kTileBlocks;           // 160 keys per tile
constexpr int BH = 16 * kHalfBlocks;           // 80 keys per CTA
constexpr int kMaskRing = 8;
constexpr int kThreads = 16 * 32;
// registers per thread after the split (the launch gives 128 x 512 = 65536)
constexpr int kRegSoft = 176, kRegRot = 96, kRegAux = 64;
static_assert(2 * 128 * kRegSoft + 128 * kRegRot + 128 * kRegAux <= 128 * kThreads, "register split");
constexpr int kSoftWarps = 8;
constexpr int kRotBase = 256;  // first thread of the four rotation warps
constexpr int kTmaWarp = 12, kMmaWarp = 13, kVWarp = 14;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.f;
constexpr uint16_t kPair = 3;

// TMEM columns (512 allocated): S0, S1 (fp32 scores, P as bf16 pairs over
// their first 80 columns), O (fp32), Q (f16/bf16 pairs).
constexpr uint32_t kColS = 0, kColO = 2 * BN, kColQ = 2 * BN + D, kTCols = 512;
static_assert(kColQ + D / 2 == kTCols, "TMEM plan");

template <int NSK, int NSV>
struct PP {
  static_assert(NSK >= NSV && NSV >= 2 && kMaskRing >= NSK + 2, "stage plan");
  static constexpr int KTILE = 2 * BH * 128;          // [half][80 keys][64] per CTA
  static constexpr int VTILE = kTileBlocks * 2048;    // [block][16 keys][64 dims of this CTA]
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + NSK * KTILE;
  static constexpr int META = 2 * kHalfBlocks;                 // start[5], flag[5]
  static constexpr int OFF_META = OFF_V + NSV * VTILE;
  static constexpr int OFF_VBLK = OFF_META + NSK * META * 4;       // [ring][10] int V block ids
  static constexpr int OFF_MASK = OFF_VBLK + kMaskRing * kTileBlocks * 4;  // [ring][10] uint16
  static constexpr int OFF_RED = (OFF_MASK + kMaskRing * kTileBlocks * 2 + 15) / 16 * 16;  // [2][2][128] f32
  static constexpr int OFF_FLAG = OFF_RED + 2 * 2 * 128 * 4;      // [2][2][4] int
  static constexpr int B_KFULL = 0, B_VFULL = B_KFULL + NSK, B_KFREE = B_VFULL + NSV, B_VFREE = B_KFREE + NSK;
  static constexpr int B_S = B_VFREE + NSV, B_PV = B_S + 2, B_MASK = B_PV + 1;
  // B_KROTL: this CTA's rotation warps; B_KROT: CTA 1's relay (in CTA 0);
  // B_QRDY, B_P: both CTAs' warps; B_VFULL: both CTAs' V copies (used in CTA 0)
  static constexpr int B_QRDY = B_MASK + kMaskRing, B_KROT = B_QRDY + 1;
  static constexpr int B_P = B_KROT + NSK, B_KROTL = B_P + 2, NBARS = B_KROTL + NSK;
  static constexpr int OFF_BAR = (OFF_FLAG + 2 * 2 * 4 * 4 + 15) / 16 * 16;
  static constexpr int OFF_TSLOT = OFF_BAR + NBARS * 8;
  static constexpr int TOTAL = OFF_TSLOT + 16;
  static_assert(KTILE % 1024 == 0 && VTILE % 1024 == 0 && (OFF_META % 16) == 0, "alignment");
  static_assert(TOTAL + 1024 <= 232448, "shared memory");
};

constexpr int kNSK = 4, kNSV = 2;

struct PairLaunch {
  PrefillArgs a;
  int tq;       // tokens per 128-row query tile (= 128 / G)
  int n_pairs;  // query-tile pairs per (request, kv head)
};

// x' = x c - y s, y' = x s + y c on 8 + 8 elements: bf16 keys converted to fp16
// (exact for |x| < 65504 down to 2^-14, then rounded to fp16 subnormals), fp16
// cos/sin, packed fp16 multiply and multiply-add, fp16 result (the QK^T operand)
__device__ __forceinline__ void rot_pack16(U4& x, U4& y, const U4& c, const U4& sn) {
  const uint32_t xw[4] = {x.x, x.y, x.z, x.w}, yw[4] = {y.x, y.y, y.z, y.w};
  const uint32_t cw[4] = {c.x, c.y, c.z, c.w}, sw[4] = {sn.x, sn.y, sn.z, sn.w};
  uint32_t xo[4], yo[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t xh = ptx::f2_to_h2(ptx::bf2_to_f2(xw[k])), yh = ptx::f2_to_h2(ptx::bf2_to_f2(yw[k]));
    xo[k] = ptx::fma_h2(xh, cw[k], ptx::mul_h2(yh, sw[k]) ^ 0x80008000u);
    yo[k] = ptx::fma_h2(xh, sw[k], ptx::mul_h2(yh, cw[k]));
  }
  x = U4{xo[0], xo[1], xo[2], xo[3]};
  y = U4{yo[0], yo[1], yo[2], yo[3]};
}

__device__ __forceinline__ uint32_t swz(int key, int chunk) {
  return (uint32_t)(key * 128 + ((chunk ^ (key & 7)) << 4));
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

// Arrive on barrier `bar` of CTA 0 of the pair (locally in CTA 0) for TMEM
// stores already waited on (tcgen05.wait::st and tcgen05.fence before the
// arrival), which CTA 0's tensor-core operations read.
__device__ __forceinline__ void arrive_leader(uint32_t bar, uint32_t crank) {
  if (crank == 0) ptx::mbar_arrive(bar);
  else ptx::mbar_arrive_peer(bar, 0);
}

template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// One CTA of the pair that computes query-tile pair `pair` of request r and kv
// head hk (both CTAs of a cluster call it with the same item).
template <bool ROPE, int NSK, int NSV>
__device__ __forceinline__ void pair_cta(const CUtensorMap& kmap, const CUtensorMap& vmap, const PairLaunch& L,
                                         const int pair, const int hk, const int r, uint8_t* smem_raw) {
  using P_ = PP<NSK, NSV>;
  const PrefillArgs& a = L.a;
  const uint32_t sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  uint8_t* sg = smem_raw + (sbase - ptx::smem_addr(smem_raw));
  int* meta = reinterpret_cast<int*>(sg + P_::OFF_META);                // [stage][META]
  uint16_t* mask16 = reinterpret_cast<uint16_t*>(sg + P_::OFF_MASK);    // [ring][10] key-valid bits
  int* vblk = reinterpret_cast<int*>(sg + P_::OFF_VBLK);                // [ring][10] V block ids (-1: none)
  float* red = reinterpret_cast<float*>(sg + P_::OFF_RED);              // [parity][half][row]
  int* flg = reinterpret_cast<int*>(sg + P_::OFF_FLAG);                 // [parity][half][quarter]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sg + P_::OFF_TSLOT);
  const uint32_t bar0 = sbase + P_::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  constexpr unsigned FULL = 0xffffffffu;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = ptx::cluster_rank();
  const int G = a.G, TQ = L.tq, mb = a.max_blocks;
  const int q0 = a.cu_q_lens[r];
  const int ql = a.cu_q_lens[r + 1] - q0;
  const int tok0 = (2 * pair + (int)crank) * TQ;  // first token of this CTA's query tile
  if (tid == 0 && crank == 0 && pair == L.n_pairs - 1 && ql > L.n_pairs * 2 * TQ) atomicOr(a.err, kErrSeqLen);

  // Loads whose latency the setup below hides: warps 0-3's query row and its
  // position, and the K~ producer's table entries of the first tile.
  U4 qc[D / 8];
  int qpos = 0;
  if (tid < 128) {  // query row tid of this CTA's tile
    const int rtok = tid / G, rh = tid - rtok * G;
    const int tq = tok0 + rtok;
    if (rtok < TQ && tq < ql) {
      const __nv_bfloat16* qp =
          static_cast<const __nv_bfloat16*>(a.q) + ((size_t)(q0 + tq) * a.Hq + (size_t)hk * G + rh) * D;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(qp) + c);
        qc[c] = U4{v.x, v.y, v.z, v.w};
      }
      if (ROPE) qpos = a.q_pos[q0 + tq];
    } else {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) qc[c] = U4{0u, 0u, 0u, 0u};
    }
  }
  int pre_ph = -1, pre_st = 0;
  if (warp == kTmaWarp && lane < kTileBlocks && lane < mb) {
    pre_ph = __ldg(a.block_tables + (size_t)r * mb + lane);
    pre_st = __ldg(a.block_starts + (size_t)r * mb + lane);
  }
  if (ql <= 0 || 2 * pair * TQ >= ql) return;  // decided alike in both CTAs of the pair
  int kvl = a.kv_lens[r];
  if (kvl < ql || kvl > mb * 16) {
    if (tid == 0 && crank == 0 && pair == 0) atomicOr(a.err, kErrSeqLen);
    kvl = min(kvl, mb * 16);
  }
  const int nblk = (kvl + 15) >> 4;
  // key tiles reached by the pair's last row
  const int lim_last = kvl - ql + min(2 * (pair + 1) * TQ, ql) - 1;
  const int n_kt = lim_last >= 0 ? lim_last / BN + 1 : 0;

  // ------------------------------------------------------------ setup
  if (tid == 0) {
    for (int s = 0; s < NSK; ++s) {
      ptx::mbar_init(bar(P_::B_KFULL + s), 1);
      ptx::mbar_init(bar(P_::B_KFREE + s), 1);
      ptx::mbar_init(bar(P_::B_KROT + s), 1);   // CTA 1's relay
      ptx::mbar_init(bar(P_::B_KROTL + s), 4);  // this CTA's four rotation warps
    }
    for (int s = 0; s < NSV; ++s) {
      ptx::mbar_init(bar(P_::B_VFULL + s), 2);  // one producer arrival from each CTA
      ptx::mbar_init(bar(P_::B_VFREE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(P_::B_S + i), 1);
      ptx::mbar_init(bar(P_::B_P + i), 2 * kSoftWarps);
    }
    ptx::mbar_init(bar(P_::B_PV), 1);
    ptx::mbar_init(bar(P_::B_QRDY), 8);
    for (int k = 0; k < kMaskRing; ++k) ptx::mbar_init(bar(P_::B_MASK + k), 1);
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    umma2::tmem_alloc(ptx::smem_addr(tslot), kTCols);
    umma2::tmem_relinquish();
  }
  // zero the V stages once so that never-loaded blocks hold finite values (a
  // masked key's P is 0, which must not meet an Inf or NaN in V; masked scores
  // are replaced, so K~ stages need no clearing)
  for (int i = tid; i < NSV * P_::VTILE / 16; i += kThreads)
    reinterpret_cast<uint4*>(sg + P_::OFF_V)[i] = make_uint4(0u, 0u, 0u, 0u);
  ptx::fence_proxy_async_smem();
  umma::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers, stages and TMEM exist
  umma::fence_after_sync();
  const uint32_t tmem = *tslot;

  // each warpgroup sets its register budget at the top of its own branch, so
  // that the compiler allocates every role's code within that role's budget
  if (warp >= kTmaWarp) {
    regs_dec<kRegAux>();
    if (warp == kTmaWarp) {
      // ======================================================== K~ producer
      // Step u loads K~ tile u (this CTA's five blocks, once QK(u - NSK) freed
      // the stage) and publishes the key-valid bits and V block ids of tile u
      // in ring slot u % 8.  Lanes 0-9 hold the table entries of the tile's
      // blocks.  The slot is rewritten for tile u + 8 only after QK(u + 4),
      // which follows PV(u + 2): every reader is past tile u by then.
      if (n_kt > 0) {
        const int* bt = a.block_tables + (size_t)r * mb;
        const int* bs = a.block_starts + (size_t)r * mb;
        const int kb = lane % kHalfBlocks, hh = lane / kHalfBlocks;   // copy lanes: block, 64-column half
        const int src = kHalfBlocks * (int)crank + kb;               // lane holding that block's entries
        const int own = lane - kHalfBlocks * (int)crank;             // 0..4 on this CTA's block lanes
        const bool mine = own >= 0 && own < kHalfBlocks;
        int my_ph = -1, my_st = 0;
        auto fetch = [&](int u) {
          const int b = kTileBlocks * u + lane;
          const bool in = lane < kTileBlocks && b < nblk;
          my_ph = in ? __ldg(bt + b) : -1;
          my_st = in ? __ldg(bs + b) : 0;
        };
        bool ok = true;
        my_ph = lane < kTileBlocks && lane < nblk ? pre_ph : -1;  // tile 0, loaded before the setup
        my_st = lane < kTileBlocks && lane < nblk ? pre_st : 0;
        for (int u = 0; u < n_kt; ++u) {
          {
            const int s = u % NSK;
            bool w = true;
            if (lane == 0 && u >= NSK) w = ptx::mbar_wait(bar(P_::B_KFREE + s), ((u / NSK) - 1) & 1);
            if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
            const int b = kTileBlocks * u + lane;
            int flag = 0;  // bit 0: usable block id, bit 1: usable start
            if (lane < kTileBlocks && b < nblk) {
              if (my_ph >= 0 && my_ph < a.num_blocks) flag |= 1;
              else if (mine) atomicOr(a.err, kErrBlockId);
              if (!ROPE || (my_st >= 0 && my_st < a.max_pos)) flag |= 2;
            }
            if (lane < kTileBlocks) {
              // key-valid bits of block b: below kv_len, usable id and start, start + slot in the table
              uint32_t bits = 0;
              if ((flag & 3) == 3) {
                const int nk = min(16, kvl - 16 * b);
                bits = nk >= 16 ? 0xffffu : (1u << nk) - 1u;
                if (ROPE) {
                  const int room = a.max_pos - my_st;
                  bits &= room >= 16 ? 0xffffu : (1u << room) - 1u;
                }
              }
              mask16[(u % kMaskRing) * kTileBlocks + lane] = (uint16_t)bits;
            }
            int* m = meta + P_::META * s;
            if (mine) {
              m[own] = my_st;
              m[kHalfBlocks + own] = flag;
            }
            if (lane < kTileBlocks) vblk[(u % kMaskRing) * kTileBlocks + lane] = (flag & 1) ? my_ph : -1;
            const unsigned kv = __ballot_sync(FULL, mine && (flag & 1));
            const int ph_l = __shfl_sync(FULL, my_ph, src);
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive(bar(P_::B_MASK + u % kMaskRing));
              ptx::mbar_arrive_expect_tx(bar(P_::B_KFULL + s), __popc(kv) * 2 * 2048);
            }
            __syncwarp();
            if (lane < 2 * kHalfBlocks) {
              if ((kv >> src) & 1u)
                ptx::tma_load_2d(sbase + P_::OFF_K + s * P_::KTILE + hh * (BH * 128) + kb * 2048, &kmap, 64 * hh,
                                 (ph_l * a.Hkv + hk) * 16, bar(P_::B_KFULL + s));
            }
            if (u + 1 < n_kt) fetch(u + 1);
          }
        }
        if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
      }
      __syncwarp();
    } else if (warp == kVWarp) {
      // ======================================================== V producer
      // V tile t (this CTA's 64 head dims of all ten blocks) once PV(t - NSV)
      // freed the stage and the K~ producer published the tile's block ids.  The
      // copies complete on CTA 0's barrier (CTA 1's through the cta_group::2 form),
      // so the tensor core that reads both halves waits on one barrier.
      const uint32_t vfull0 = ptx::mapa(bar(P_::B_VFULL), 0);  // CTA 0's barrier, cluster address
      bool ok = true;
      for (int t = 0; t < n_kt; ++t) {
        const int sv = t % NSV;
        bool w = true;
        if (lane == 0) {
          if (t >= NSV) w = ptx::mbar_wait(bar(P_::B_VFREE + sv), ((t / NSV) - 1) & 1);
          w = w && ptx::mbar_wait(bar(P_::B_MASK + t % kMaskRing), (t / kMaskRing) & 1);
        }
        if (!__shfl_sync(FULL, w, 0)) { ok = false; break; }
        const int ph = lane < kTileBlocks ? vblk[(t % kMaskRing) * kTileBlocks + lane] : -1;
        const unsigned vv = __ballot_sync(FULL, ph >= 0);
        const uint32_t vbar = vfull0 + 8u * (uint32_t)sv;
        if (lane == 0) ptx::mbar_arrive_expect_tx_cl(vbar, __popc(vv) * 2048);
        __syncwarp();
        if (ph >= 0)
          ptx::tma_load_2d_pair(sbase + P_::OFF_V + sv * P_::VTILE + lane * 2048, &vmap, 64 * (int)crank,
                                (ph * a.Hkv + hk) * 16, vbar);
      }
      if (!ok && lane == 0) atomicOr(a.err, kErrTimeout);
      __syncwarp();
    } else if (warp == kMmaWarp && crank != 0) {
      // ======================================================== relay (CTA 1)
      // CTA 0 issues the products, which read the keys this CTA's threads rotated
      // in place.  The relay observes each tile's rotation with an acquire and
      // forwards it with a release at cluster scope.
      if (lane == 0) {
        for (int u = 0; u < n_kt; ++u) {
          if (!ptx::mbar_wait(bar(P_::B_KROTL + u % NSK), (u / NSK) & 1)) {
            atomicOr(a.err, kErrTimeout);
            break;
          }
          ptx::mbar_arrive_remote(bar(P_::B_KROT + u % NSK), 0);
        }
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // ======================================================== MMA issue (CTA 0)
      if (lane == 0 && n_kt > 0) {
        const uint32_t id_qk = ROPE ? umma::idesc_f16_f32(256, BN, false, false)
                                    : umma::idesc_bf16_f32(256, BN, false, false);
        const uint32_t id_pv = umma::idesc_bf16_f32(256, D, false, true);
        // S_(t & 1) = Q K_t^T once both CTAs rotated their halves of tile t; the
        // stage is released to both producers while a later tile refills it
        auto qk = [&](int t) -> bool {
          const int s = t % NSK;
          if (!ptx::mbar_wait(bar(P_::B_KROTL + s), (t / NSK) & 1) ||
              !ptx::mbar_wait_cl(bar(P_::B_KROT + s), (t / NSK) & 1))
            return false;
          umma::fence_after_sync();
          const uint32_t kb = sbase + P_::OFF_K + s * P_::KTILE;
  #pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            umma2::mma_ts(tmem + kColS + BN * (t & 1), tmem + kColQ + 8 * ks,
                          umma::smem_desc_sw128(kb + (ks >> 2) * (BH * 128) + (ks & 3) * 32, 16, 1024), id_qk,
                          ks > 0 ? 1u : 0u);
          umma2::commit_mc(bar(P_::B_S + (t & 1)), kPair);
          if (t + NSK < n_kt) umma2::commit_mc(bar(P_::B_KFREE + s), kPair);
          return true;
        };
        bool ok = ptx::mbar_wait(bar(P_::B_QRDY), 0);
        if (ok) ok = qk(0);
        if (ok && n_kt > 1) ok = qk(1);
        for (int t = 0; t < n_kt && ok; ++t) {
          const int sv = t % NSV;
          if (!ptx::mbar_wait(bar(P_::B_P + (t & 1)), (t >> 1) & 1) ||
              !ptx::mbar_wait(bar(P_::B_VFULL + sv), (t / NSV) & 1)) {
            ok = false;
            break;
          }
          umma::fence_after_sync();
          // O += P_t V_t, one 16-key block per MMA; V stage: [block][16 keys][64 dims]
          const uint32_t vb = sbase + P_::OFF_V + sv * P_::VTILE;
  #pragma unroll
          for (int ks = 0; ks < kTileBlocks; ++ks)
            umma2::mma_ts(tmem + kColO, tmem + kColS + BN * (t & 1) + 8 * ks,
                          umma::smem_desc_sw128(vb + ks * 2048, 2048, 1024), id_pv, (t > 0 || ks > 0) ? 1u : 0u);
          umma2::commit_mc(bar(P_::B_PV), kPair);
          if (t + NSV < n_kt) umma2::commit_mc(bar(P_::B_VFREE + sv), kPair);
          if (t + 2 < n_kt) ok = qk(t + 2);  // S_(t & 1) is free once PV(t) has read P_t
        }
        if (!ok) atomicOr(a.err, kErrTimeout);
      }
      __syncwarp();
    }
  } else if (tid >= kRotBase) {
    regs_dec<kRegRot>();
    // ======================================================== key rotation
    const int rt = tid - kRotBase;  // 0..127
    // ---- key rotation: thread -> (frequency group fg of 8, slot sl): slot sl
    // of this CTA's five blocks; cos/sin((start + sl) theta_f), f = 8 fg ..
    // 8 fg + 7, are one 16-byte load each from row start + sl of the fp16 table
    const int fg = rt & 7, sl = rt >> 3;
    const int key0 = (int)crank * BH;  // this CTA's first key of a tile
    for (int t = 0; t < n_kt; ++t) {
      const int s = t % NSK;
      if (!__all_sync(FULL, ptx::mbar_wait(bar(P_::B_KFULL + s), (t / NSK) & 1))) {
        if (lane == 0) atomicOr(a.err, kErrTimeout);
        break;
      }
      if constexpr (ROPE) {
        const int* m = meta + P_::META * s;
        uint8_t* sk = sg + P_::OFF_K + s * P_::KTILE;
        // every load first (an unusable key reads table row 0), stores only for
        // valid keys: no branch between blocks, so their loads overlap
        U4 cvs[kHalfBlocks], svs[kHalfBlocks];
        bool vs[kHalfBlocks];
#pragma unroll
        for (int blk = 0; blk < kHalfBlocks; ++blk) {
          const int flag = m[kHalfBlocks + blk];
          const int start = m[blk];
          const int key = blk * 16 + sl;
          vs[blk] = (flag & 3) == 3 && t * BN + key0 + key < kvl && start + sl < a.max_pos;
          // row start + sl of the fp16 table: cos (64) | sin (64); this thread's 8 frequencies
          const uint16_t* rg = a.cos_sin16 + (size_t)(vs[blk] ? start + sl : 0) * D;
          const uint4 c4 = __ldg(reinterpret_cast<const uint4*>(rg + 8 * fg));
          const uint4 s4 = __ldg(reinterpret_cast<const uint4*>(rg + D / 2 + 8 * fg));
          cvs[blk] = U4{c4.x, c4.y, c4.z, c4.w};
          svs[blk] = U4{s4.x, s4.y, s4.z, s4.w};
        }
        uint32_t wa = 0u, wb = 0u;  // fp16 range watch over the stored keys
#pragma unroll
        for (int blk = 0; blk < kHalfBlocks; ++blk) {
          const U4 cv = cvs[blk], sv = svs[blk];
          const int key = blk * 16 + sl;
          const bool v = vs[blk];
          U4* px = reinterpret_cast<U4*>(sk + swz(key, fg));
          U4* py = reinterpret_cast<U4*>(sk + BH * 128 + swz(key, fg));
          U4 x = *px, y = *py;
          rot_pack16(x, y, cv, sv);
          if (v) {
            *px = x;
            *py = y;
            wa = ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(wa, x.x), x.y), x.z), x.w);
            wb = ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(ptx::watch_h2(wb, y.x), y.y), y.z), y.w);
          }
        }
        if ((wa | wb) != 0u) atomicOr(a.err, kErrRange);
        ptx::fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(P_::B_KROTL + s));
    }
  } else {
    regs_inc<kRegSoft>();
    // ======================================================== softmax
    // Warp w: query rows 32 (w % 4) + lane (TMEM lanes), keys 80 h .. 80 h + 79
    // of each tile (h = w / 4).  The two warps of a lane quarter share the
    // row maximum through shared memory; each keeps its own part of the row
    // sum and rescales its 64 columns of O.
    constexpr int NPW = BH / 2;  // P words of one half
    const int qd = warp & 3, h = warp >> 2;
    const int row = 32 * qd + lane;
    const int rtok = row / G, rh = row - rtok * G;
    const int tq = tok0 + rtok;
    const bool row_ok = rtok < TQ && tq < ql;
    const int lim = kvl - ql + tq;         // last key this row attends
    const int lim_first = kvl - ql + tok0;  // ... the tile's first row attends
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const uint32_t t_o = tmem + kColO + lane_base + 64 * h;
    const uint32_t nb_id = 1 + qd;  // named barrier of warps qd, qd + 4
    float m_run = -CUDART_INF_F, m_use = -CUDART_INF_F, l_run = 0.f;
    bool failed = false, pv_late = false;
    if (h == 0) {
      const float qs = a.scale * kLog2e;
      // ---- query row `row` (warps 0-3, while the rotation warps start on the
      // first key tile): rotated at its position, scaled by scale * log2(e),
      // packed (f16 with rotation, bf16 without) into TMEM columns as the A operand
      
      // qc and qpos (row tid = row) were loaded before the setup
      int pos = qpos;
      if (ROPE && row_ok && (pos < 0 || pos >= a.max_pos)) {
        atomicOr(a.err, kErrPosition);
        pos = 0;
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
      // column j holds head dims 2 j, 2 j + 1
      const uint32_t tq_addr = tmem + kColQ + lane_base;
#pragma unroll
      for (int part = 0; part < D / 32; ++part) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const U4& x = qc[4 * part + c];
          w[4 * c] = x.x;
          w[4 * c + 1] = x.y;
          w[4 * c + 2] = x.z;
          w[4 * c + 3] = x.w;
        }
        umma::tmem_st16(tq_addr + 16 * part, w);
      }
      umma::tmem_wait_st();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_leader(bar(P_::B_QRDY), crank);
    }

    int rounds = 0;
    auto exchange = [&](float mine, bool ok, float& other, bool& other_ok) {
      const int p = rounds & 1;
      red[(p * 2 + h) * 128 + row] = mine;
      if (lane == 0) flg[(p * 2 + h) * 4 + qd] = ok ? 1 : 0;
      umma::fence_before_sync();
      ptx::named_sync(nb_id, 64);
      umma::fence_after_sync();
      other = red[(p * 2 + (h ^ 1)) * 128 + row];
      other_ok = flg[(p * 2 + (h ^ 1)) * 4 + qd] != 0;
      ++rounds;
    };
    for (int t = 0; t < n_kt; ++t) {
      const int b = t & 1;
      const uint32_t t_s = tmem + kColS + BN * b + lane_base;
      bool ok = !pv_late && __all_sync(FULL, ptx::mbar_wait(bar(P_::B_S + b), (t >> 1) & 1));
      // the mask slot of tile t is rewritten for tile t + 8, which needs this warp past tile t + 1
      ok = ok && __all_sync(FULL, ptx::mbar_wait(bar(P_::B_MASK + t % kMaskRing), (t / kMaskRing) & 1));
      umma::fence_after_sync();
      uint32_t v[BH];
      if (ok) {
        umma::tmem_ld32(t_s + BH * h, *reinterpret_cast<uint32_t(*)[32]>(v));
        umma::tmem_ld32(t_s + BH * h + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
        umma::tmem_ld16(t_s + BH * h + 64, *reinterpret_cast<uint32_t(*)[16]>(v + 64));
      }
      const uint16_t* mk = mask16 + (t % kMaskRing) * kTileBlocks + kHalfBlocks * h;
      uint32_t mw[kHalfBlocks];
      uint32_t mall = 0xffffu;
#pragma unroll
      for (int k = 0; k < kHalfBlocks; ++k) {
        mw[k] = mk[k];
        mall &= mw[k];
      }
      const int kb0 = t * BN + BH * h;
      const bool full = mall == 0xffffu && kb0 + BH - 1 <= lim_first;
      umma::tmem_wait_ld();
      float mx = -CUDART_INF_F;
      if (ok && full) {
        float pm[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int j = 0; j < BH; j += 2)
          pm[(j >> 1) & 3] = ptx::fmax3(pm[(j >> 1) & 3], __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
        mx = fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3]));
      } else if (ok && mall == 0xffffu) {
        // every block usable: the valid keys are the causal prefix j < nv
        const int nv = row_ok ? lim - kb0 + 1 : 0;
#pragma unroll
        for (int j = 0; j < BH; ++j) {
          v[j] = j < nv ? v[j] : __float_as_uint(-CUDART_INF_F);
          mx = fmaxf(mx, __uint_as_float(v[j]));
        }
      } else if (ok) {
        // invalid keys become -inf in place, so that both passes treat them alike
#pragma unroll
        for (int j = 0; j < BH; ++j) {
          const bool kv_ok = row_ok && ((mw[j >> 4] >> (j & 15)) & 1u) && kb0 + j <= lim;
          v[j] = kv_ok ? v[j] : __float_as_uint(-CUDART_INF_F);
          mx = fmaxf(mx, __uint_as_float(v[j]));
        }
      }
      float mo;
      bool ok_o;
      exchange(mx, ok, mo, ok_o);  // after this both warps have read their scores
      if (!ok || !ok_o) {
        failed = true;
        break;
      }
      m_run = fmaxf(m_run, fmaxf(mx, mo));
      const bool need = m_run != -CUDART_INF_F && (m_use == -CUDART_INF_F || m_run > m_use + kRescale);
      const float corr = !need ? 1.f : (m_use == -CUDART_INF_F ? 0.f : ex2(m_use - m_run));
      if (need) {
        l_run *= corr;
        m_use = m_run;
      }
      // P = 2^(s - mref) as bf16 pairs over columns 40 h .. 40 h + 39 of S_b
      // (the other warp's scores there were read before the exchange)
      const float mref = m_use == -CUDART_INF_F ? 0.f : m_use;
      const uint64_t mref2 = ptx::f2(mref, mref);
      uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
      const uint32_t t_p = t_s + NPW * h;
#pragma unroll
      for (int j = 0; j < NPW; ++j) {
        const uint64_t d2 = ptx::sub2(ptx::f2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1])), mref2);
        float dl, dh;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(dl), "=f"(dh) : "l"(d2));
        const uint64_t p2 = ptx::f2(ex2(dl), ex2(dh));  // 2^-inf = 0 for masked keys
        ls[j & 3] = ptx::add2(ls[j & 3], p2);
        v[j] = ptx::f2_to_bf2(p2);
        if ((j & 15) == 15) umma::tmem_st16(t_p + (j & ~15), *reinterpret_cast<const uint32_t(*)[16]>(v + (j & ~15)));
      }
      umma::tmem_st8(t_p + 32, *reinterpret_cast<const uint32_t(*)[8]>(v + 32));
      const uint64_t lsum2 = ptx::add2(ptx::add2(ls[0], ls[1]), ptx::add2(ls[2], ls[3]));
      float sl, sh;
      asm("mov.b64 {%0, %1}, %2;" : "=f"(sl), "=f"(sh) : "l"(lsum2));
      l_run += sl + sh;
      // lazy O rescale, once PV(t - 1) has landed (it is still running while
      // this warp works on tile t)
      if (t > 0 && __any_sync(FULL, need)) {
        if (!__all_sync(FULL, ptx::mbar_wait(bar(P_::B_PV), (t - 1) & 1))) {
          pv_late = true;  // reported at the next exchange
        } else {
          umma::fence_after_sync();
#pragma unroll 1
          for (int part = 0; part < 2; ++part) {
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
      }
      umma::tmem_wait_st();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) arrive_leader(bar(P_::B_P + b), crank);
    }
    // ---- epilogue: O / l -> global; this warp writes head dims 64 h .. 64 h + 63
    failed = failed || pv_late;
    bool have = n_kt > 0 && !failed;
    // wait for the last two P V products in order: a parity wait is only
    // meaningful for the barrier's current phase or the one before it, and
    // PV(n_kt - 2) may still be running here (PV(n_kt - 3) is known complete)
    if (have && n_kt > 1 && !__all_sync(FULL, ptx::mbar_wait(bar(P_::B_PV), (n_kt - 2) & 1))) {
      have = false;
      failed = true;
    }
    if (have && !__all_sync(FULL, ptx::mbar_wait(bar(P_::B_PV), (n_kt - 1) & 1))) {
      have = false;
      failed = true;
    }
    if (failed && lane == 0) atomicOr(a.err, kErrTimeout);
    float l_o;
    bool unused;
    exchange(l_run, true, l_o, unused);
    const float l_tot = l_run + l_o;
    umma::fence_after_sync();
    const int hq = hk * G + rh;
    __nv_bfloat16* op = static_cast<__nv_bfloat16*>(a.out) + ((size_t)(q0 + tq) * a.Hq + hq) * D + 64 * h;
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
#pragma unroll
    for (int part = 0; part < 2; ++part) {
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
    if (row_ok && h == 0 && a.lse)
      a.lse[(size_t)(q0 + tq) * a.Hq + hq] = l_tot > 0.f ? (m_use + log2f(l_tot)) * kLn2 : -CUDART_INF_F;
  }

  // teardown: execution barriers only (nothing left to publish)
  umma::fence_before_sync();
  __syncthreads();
  ptx::cluster_sync_relaxed();  // every product of the pair has completed and been read
  umma::fence_after_sync();
  if (warp == kMmaWarp) umma2::tmem_dealloc(tmem, kTCols);
  ptx::cluster_sync_relaxed();  // neither CTA leaves while the pair's TMEM is being released
}

template <bool ROPE, int NSK, int NSV>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const PairLaunch L) {
  extern __shared__ uint8_t smem_raw[];
  // heaviest (latest) query-tile pairs first
  pair_cta<ROPE, NSK, NSV>(kmap, vmap, L, L.n_pairs - 1 - (int)(blockIdx.x >> 1), blockIdx.y, blockIdx.z, smem_raw);
}

// Mixed continuous batch in one launch (the device side of interleaved
// span-prefill scheduling, MiniPIC summary section 2.2 "Scheduling": span
// prefills pipelined with ongoing decodes).  Every cluster of the grid is
// either a prefill cluster (one query-tile pair, the CTA-pair body above) or a
// decode cluster (each of its two CTAs one decode split, the decode kernel's
// CTA body with two stages per warp: for groups of up to 8 heads on warps 0-11
// with 160 registers each while warps 12-15 give their registers up and leave,
// for larger groups, whose body needs more registers, on warps 0-7 with 232;
// register budgets change per warpgroup, as setmaxnreg requires).  The decode
// clusters come first in the grid
// and the prefill clusters (heaviest first) follow, so that the long prefill
// clusters fill the SMs as the short decode CTAs drain (measured against
// prefill first and against decode clusters spread evenly through the grid,
// this order was the fastest).
template <int NT>
struct MixDec {
  static constexpr int kWarps = NT == 1 ? 12 : 8, kStages = 2, kBar = 8;
  static constexpr int kReg = NT == 1 ? 160 : 232, kRegIdle = NT == 1 ? 32 : 24;
  static_assert(kWarps % 4 == 0, "setmaxnreg acts on whole warpgroups");
  static_assert(kWarps * 32 * kReg + (16 - kWarps) * 32 * kRegIdle <= 128 * kThreads, "decode register split");
};

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    mixed_pair_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap kblk, const __grid_constant__ CUtensorMap vblk,
                      const PairLaunch L, const DecodeArgs Dd, const int n_pre, const int n_dec) {
  extern __shared__ uint8_t smem_raw[];
  const long long c = blockIdx.x >> 1;
  const long long d0 = c < n_dec ? c : n_dec;  // decode clusters before cluster c
  if (c < n_dec) {
    using MD = MixDec<NT>;
    if ((threadIdx.x >> 5) >= MD::kWarps) {
      regs_dec<MD::kRegIdle>();
      return;
    }
    regs_inc<MD::kReg>();
    const int u = 2 * (int)d0 + (int)ptx::cluster_rank();  // decode unit: (split, kv head, request)
    if (u >= Dd.n_split * Dd.Hkv * Dd.batch) return;
    const int split = u % Dd.n_split, rest = u / Dd.n_split;
    decode_impl::decode_cta<D, NT, true, MD::kWarps, MD::kStages, MD::kBar, true>(&kblk, &vblk, Dd, split,
                                                                                 rest % Dd.Hkv, rest / Dd.Hkv,
                                                                                 smem_raw);
  } else {
    const int i = (int)(c - d0);  // prefill item: (request, kv head) groups, heaviest pairs first
    const int grp = i / L.n_pairs;
    pair_cta<true, kNSK, kNSV>(kmap, vmap, L, L.n_pairs - 1 - (i - grp * L.n_pairs), grp % L.a.Hkv, grp / L.a.Hkv,
                               smem_raw);
  }
}

template <int NT>
cudaError_t launch_mixed_t(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s) {
  constexpr int sa = PP<kNSK, kNSV>::TOTAL, sb = decode_impl::Smem<D, MixDec<NT>::kWarps, MixDec<NT>::kStages>::TOTAL;
  const int smem = (sa > sb ? sa : sb) + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(mixed_pair_kernel<NT>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm, kb, vb;  // 2-D views for the prefill tiles, 3-D block views for the decode tiles
  const long long rows = (long long)p.num_blocks * p.Hkv * 16;
  if (!make_pool_map(&km, p.k_pool, rows, D) || !make_pool_map(&vm, p.v_pool, rows, D) ||
      !make_pool_block_map(&kb, p.k_pool, rows, D) || !make_pool_block_map(&vb, p.v_pool, rows, D))
    return cudaErrorInvalidValue;
  PairLaunch L{p, 128 / p.G, 0};
  L.n_pairs = (p.max_q_len + 2 * L.tq - 1) / (2 * L.tq);
  const long long n_pre = (long long)L.n_pairs * p.Hkv * p.batch;
  const long long n_dec = ((long long)d.n_split * d.Hkv * d.batch + 1) / 2;
  if (n_pre + n_dec > 0x3fffffffLL) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * (n_pre + n_dec)), 1, 1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mixed_pair_kernel<NT>, km, vm, kb, vb, L, d, (int)n_pre, (int)n_dec);
}

template <bool ROPE>
cudaError_t launch_t(const PrefillArgs& a, cudaStream_t s) {
  using P_ = PP<kNSK, kNSV>;
  const int smem = P_::TOTAL + 1024;
  static bool done[64] = {false};
  cudaError_t e = set_smem_once(prefill_pair_kernel<ROPE, kNSK, kNSV>, smem, done);
  if (e != cudaSuccess) return e;
  CUtensorMap km, vm;
  const long long rows = (long long)a.num_blocks * a.Hkv * 16;
  if (!make_pool_map(&km, a.k_pool, rows, D) || !make_pool_map(&vm, a.v_pool, rows, D)) return cudaErrorInvalidValue;
  PairLaunch L{a, 128 / a.G, 0};
  L.n_pairs = (a.max_q_len + 2 * L.tq - 1) / (2 * L.tq);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * L.n_pairs), (unsigned)a.Hkv, (unsigned)a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_pair_kernel<ROPE, kNSK, kNSV>, km, vm, L);
}

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, bool rotate, cudaStream_t s) {
  if (a.D != D) return cudaErrorInvalidValue;
  return rotate ? launch_t<true>(a, s) : launch_t<false>(a, s);
}

cudaError_t launch_mixed_pair(const PrefillArgs& p, const DecodeArgs& d, cudaStream_t s) {
  if (p.D != D || d.D != D) return cudaErrorInvalidValue;
  return d.G <= 8 ? launch_mixed_t<1>(p, d, s) : launch_mixed_t<2>(p, d, s);
}

}  // namespace minipic
