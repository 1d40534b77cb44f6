// FlashAttention backward for sm_103a: the gradients of sum(dO * O) with
// respect to Q, K and V, recomputing S and P from the stored log-sum-exp
// ("FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
// section "Training: recompute instead of store"; "Flash Attention, tiled",
// section "More arithmetic can still be faster").  With P = exp(S - LSE) and
// D_t = sum_c dO_tc O_tc:
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
//
// Two kernels, no atomics and no T x T matrix in memory:
//   fa_bwd_kernel<d, 0> (dQ)  per (head, 128-row query tile): D and LSE * log2 e of the
//                             tile's rows into a workspace whose rows are padded per head
//                             to a multiple of 128 (D = 0 and LSE * log2 e = +inf there,
//                             so P = 0 without a mask); stream the key tiles,
//                             S = Q K^T and dP = dO V^T on the tensor core, dS in the
//                             row warps, dQ += dS K (dS read from Tensor Memory; at
//                             d = 128 dO is kept in Tensor Memory too);
//   fa_bwd_kernel<d, 1>       per (head, 128-key tile): stream the query tiles and their
//     (dK, dV)                LSE / D vectors, S^T = K Q^T and dP^T = V dO^T, P^T and dS^T
//                             in the row warps, dV += P^T dO and dK += dS^T Q (P^T and
//                             dS^T read from Tensor Memory).
// Each recomputes S and dP (seven matrix products per tile pair instead of
// five) so that every gradient product takes its A operand from Tensor Memory
// with the rows it needs on the lanes, and no partial sum crosses CTAs.  The
// gradients leave through shared memory and TMA stores (32 x 32 boxes), except
// dQ at d = 128, whose shared memory holds a sixth ring stage instead.
//
// Roles (448 threads, one CTA per SM, persistent over work units):
//   warps 0-7    row warps: one TMEM lane (one row of the unit's 128-row tile) per
//                thread, warps w and w + 4 splitting the row's 128 columns
//   warp 8       TMA producer: the unit's resident tiles, then the streamed tiles
//                (and the dK/dV kernel's per-step vectors) through a ring
//   warp 9       Tensor Memory allocator and tcgen05.mma issuer (whole warp,
//                elect.sync picks the issuing lane)
//   warps 10-13  output warps, one per TMEM lane quarter: the finished unit's
//                gradients out of Tensor Memory to global memory while the row warps
//                start on the next unit; in the dQ kernel also the next unit's D and
//                LSE * log2 e rows (and at d = 128 its dO into Tensor Memory)
// Every mbarrier wait is bounded; on expiry the kernel records it in its
// status word and unwinds, as the forward kernel does.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_kernel.h"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int BT = 128;  // rows per tile (queries or keys)
constexpr int BWD_THREADS = 448;
constexpr int BWD_PRODUCER = 8;
constexpr int BWD_MMA = 9;
constexpr int ROW_WARPS = 8;  // two per TMEM lane quarter, each taking half of the 128 columns
constexpr int OUT_WARP0 = 10, OUT_WARPS = 4;  // one per TMEM lane quarter
constexpr int BOX = 128 * 128;  // one TMA box: 128 rows x 64 bf16, 128-byte swizzle
constexpr float LOG2E = 1.4426950408889634074f;

__device__ unsigned int g_bwd_status;  // bit 0: a bounded wait ran out

template <int D, int KIND>
struct BwdLayout {
  static constexpr int TILE = BT * D * 2;
  static constexpr int BOXES = D / 64;
  // The dQ kernel at d = 128 keeps dO in Tensor Memory (the A operand of dP = dO V^T, in the
  // 64 columns its schedule leaves free) and stores dQ rows directly, so that its shared
  // memory holds six ring stages: its key tile K_j stays in the ring until dQ += dS K_j, and
  // with four stages the loads of the next tiles could not keep up.
  static constexpr bool DO_TMEM = (D == 128 && KIND == 0);
  static constexpr bool DIRECT_OUT = DO_TMEM;
  static constexpr int STAGES = (D == 128) ? (DO_TMEM ? 6 : 4) : 6;  // streamed tiles in flight
  static constexpr int RES_TILES = DO_TMEM ? 1 : 2;  // resident tiles in shared memory
  static constexpr int RES_OFF = 0;
  static constexpr int RING_OFF = RES_TILES * TILE;
  static constexpr int VEC_OFF = RING_OFF + STAGES * TILE;  // dK/dV: [2 buffers][LSE*log2e, D][128] fp32
  static constexpr int VEC_BYTES = KIND == 1 ? 2 * 2 * BT * 4 : 0;
  // gradient staging: per output warp two 32-row x 32-column bf16 boxes (2 KB each, rows of 64 bytes)
  static constexpr int STG_OFF = VEC_OFF + VEC_BYTES;
  static constexpr int STG_BOX_BYTES = 32 * 64;
  static constexpr int BAR_OFF = STG_OFF + (DIRECT_OUT ? 0 : OUT_WARPS * 2 * STG_BOX_BYTES);
  // res_full, res_empty, ring_full[S], ring_empty[S], s_full, p_full, o_full, o_empty, done, vec_full[2],
  // s_free, dp_full, dp_free, pv_done, vec_empty[2], do_full, p_half, rv_full[2]
  static constexpr int NUM_BARS = 2 + 2 * STAGES + 5 + 2 + 4 + 2 + 1 + 1 + 2;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;
};
static_assert(BwdLayout<128, 0>::SMEM <= 232448 && BwdLayout<128, 1>::SMEM <= 232448 &&
                  BwdLayout<64, 0>::SMEM <= 232448 && BwdLayout<64, 1>::SMEM <= 232448,
              "shared memory over the limit");

// Tensor Memory columns (512 allocated):
//   dQ kernel:         S [0,128)    dP [128,256)    dQ [256,256+d)  dS [384,448)  (d = 128: dO [448,512))
//   dK/dV kernel d=64: S^T [0,128)  dP^T [128,256)  dV [256,320)  dK [320,384)  P^T [384,448)  dS^T [448,512)
//   dK/dV kernel d=128: S^T, dP^T as above, dV [256,384), dK [384,512); P^T is written over
//     S^T and dS^T over dP^T (each row warp over the first 32 of the 64 columns it has read).
// With P / dS in columns of their own (SPLIT), the next step's S and dP are issued as soon
// as the row warps have read this step's, so the products overlap the row-warp work.
constexpr uint32_t COL_S = 0, COL_DP = 128, COL_ACC = 256, COL_BUF = 384;
constexpr uint32_t COL_DO = 448;  // d = 128 dQ kernel: dO as bf16 pairs (after dS [384, 448))
template <int D, int KIND>
struct BwdSched {
  static constexpr bool SPLIT = (KIND == 0) || (D == 64);
  // Packed (bf16-pair) column of the 16-wide K step kk of P / dS, relative to COL_P / COL_DS.
  // The row warps of column half h write pairs for columns [64h, 64h + 64): contiguous in their
  // own buffers (SPLIT), or over the S / dP columns they read themselves.
  static __device__ __forceinline__ constexpr uint32_t a_col(int kk) {
    return SPLIT ? uint32_t(kk) * 8u : uint32_t(kk / 4) * 64u + uint32_t(kk % 4) * 8u;
  }
  static __device__ __forceinline__ constexpr uint32_t half_col(int h) { return SPLIT ? 32u * h : 64u * h; }
  // where the row warps put P (dK/dV kernel) and dS (both kernels); without SPLIT the row
  // warps of half h write P over S columns [64h, 64h + 32) and dS over dP columns [64h, 64h + 32)
  static constexpr uint32_t COL_P = SPLIT ? COL_BUF : COL_S;
  static constexpr uint32_t COL_DS = SPLIT ? (KIND == 0 ? COL_BUF : COL_BUF + 64) : COL_DP;
};

struct Bars {
  uint32_t res_full, res_empty, ring_full, ring_empty, s_full, p_full, o_full, o_empty, done;
  uint32_t vec_full;  // [2]: the per-step LSE / D vectors of the dK/dV kernel are in shared memory
  uint32_t s_free, dp_full, dp_free, pv_done;  // SPLIT schedule
  uint32_t vec_empty;  // [2]: every row warp is done with that vector buffer
  uint32_t do_full;    // the unit's dO is in Tensor Memory (d = 128 dQ kernel)
  uint32_t p_half;     // P^T is written (d = 128 dK/dV kernel)
  uint32_t rv_full;    // [2]: a unit's D and LSE * log2 e rows are in the workspace (dQ kernel)
};

template <int D, int KIND>
__device__ __forceinline__ Bars make_bars(uint32_t base) {
  using L = BwdLayout<D, KIND>;
  Bars b;
  b.res_full = base;
  b.res_empty = base + 8;
  b.ring_full = base + 16;
  b.ring_empty = base + 16 + 8 * L::STAGES;
  const uint32_t x = base + 16 + 16 * L::STAGES;
  b.s_full = x;
  b.p_full = x + 8;
  b.o_full = x + 16;
  b.o_empty = x + 24;
  b.done = x + 32;
  b.vec_full = x + 40;
  b.s_free = x + 56;
  b.dp_full = x + 64;
  b.dp_free = x + 72;
  b.pv_done = x + 80;
  b.vec_empty = x + 88;
  b.do_full = x + 104;
  b.p_half = x + 112;
  b.rv_full = x + 120;
  return b;
}

// The k-th unit of CTA b in a grid of G (snake over a heavy-first list).
__device__ __forceinline__ int bwd_unit_of(int k, int b, int G) { return k * G + ((k & 1) ? (G - 1 - b) : b); }

// ---------------------------------------------------------------- D = rowsum(dO * O)

// D_t = sum_c dO_tc O_tc and LSE_t * log2 e for the 32 workspace rows [r0, r0 + 32) of head bh
// (the workspace's rows are padded per head to Tp): D = 0 and LSE * log2 e = +inf past T, so
// P = 0 there without a mask.  D / 8 lanes cover a row with 16 bytes of O and of dO each, a
// warp pass covers 256 / D rows, and four passes' loads are issued together.  The stores are
// plain: the dQ kernel's row warps read the rows after an mbarrier hand-over within the CTA,
// the dK/dV kernel after this kernel has finished.
template <int D>
__device__ __forceinline__ void bwd_row_vectors(const BwdParams& p, int bh, int r0, int lane) {
  constexpr int LPR = D / 8;           // lanes per row
  constexpr int RPW = 32 / LPR;        // rows per warp pass
  constexpr int PASSES = 32 / RPW, U = 4;  // (eight spill registers)
  const int sub = lane / LPR, part = lane % LPR;
  const size_t ws = static_cast<size_t>(bh) * p.Tp;
#pragma unroll
  for (int g0 = 0; g0 < PASSES; g0 += U) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = r0 + (g0 + u) * RPW + sub;
      a[u] = b[u] = make_uint4(0, 0, 0, 0);
      if (t < p.T) {
        const size_t src = static_cast<size_t>(bh) * p.T + t;
        a[u] = __ldg(reinterpret_cast<const uint4*>(p.o + src * D) + part);
        b[u] = __ldg(reinterpret_cast<const uint4*>(p.dout + src * D) + part);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
      float acc = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 xf = __bfloat1622float2(x[c]), yf = __bfloat1622float2(y[c]);
        acc = fmaf(xf.x, yf.x, acc);
        acc = fmaf(xf.y, yf.y, acc);
      }
#pragma unroll
      for (int sh = LPR / 2; sh >= 1; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
      const int t = r0 + (g0 + u) * RPW + sub;
      if (part == 0) {
        p.drow[ws + t] = acc;  // 0 past T (both rows were read as zeros)
        p.lse2[ws + t] = t < p.T ? p.lse[static_cast<size_t>(bh) * p.T + t] * LOG2E : INFINITY;
      }
    }
  }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// Common prologue: barriers, Tensor Memory, abort flag.  Returns the TMEM base.
template <int D, int KIND>
__device__ __forceinline__ uint32_t bwd_setup(uint8_t* smem, const Bars& B, uint32_t* tmem_slot,
                                              volatile int* abort_flag, int warp) {
  using L = BwdLayout<D, KIND>;
  if (threadIdx.x == 0) {
    mbar_init(B.res_full, 1);
    mbar_init(B.res_empty, 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(B.ring_full + 8 * s, 1);
      mbar_init(B.ring_empty + 8 * s, 1);
    }
    mbar_init(B.s_full, 1);
    mbar_init(B.p_full, ROW_WARPS);
    mbar_init(B.o_full, 1);
    mbar_init(B.o_empty, OUT_WARPS);
    mbar_init(B.done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(B.vec_full + 8 * b, 1);
      mbar_init(B.vec_empty + 8 * b, ROW_WARPS);
    }
    mbar_init(B.s_free, ROW_WARPS);
    mbar_init(B.dp_full, 1);
    mbar_init(B.dp_free, ROW_WARPS);
    mbar_init(B.pv_done, 1);
    mbar_init(B.do_full, OUT_WARPS);
    mbar_init(B.p_half, ROW_WARPS);
    mbar_init(B.rv_full, OUT_WARPS);
    mbar_init(B.rv_full + 8, OUT_WARPS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BWD_MMA) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return *tmem_slot;
}

template <int D>
__device__ __forceinline__ void bwd_teardown(uint32_t tmem, int warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == BWD_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Unit w -> (head, resident tile, first streamed tile, number of streamed tiles).
// KIND 0 (dQ): resident = the query tile (Q, dO), streamed = key tiles (K, V);
//   causal units are listed longest first (query tile nt-1 first).
// KIND 1 (dK, dV): resident = the key tile (K, V), streamed = query tiles (Q, dO);
//   causal units are listed longest first (key tile 0 first).
template <int KIND>
__device__ __forceinline__ void bwd_decode(const BwdParams& p, int w, int& bh, int& rt, int& first, int& n) {
  const int band = w / p.BH;
  bh = w - band * p.BH;
  if (KIND == 0) {
    rt = p.causal ? p.nt - 1 - band : band;
    first = 0;
    n = p.causal ? rt + 1 : p.nt;
  } else {
    rt = band;
    first = p.causal ? rt : 0;
    n = p.nt - first;
  }
}

// TMA producer (whole warp, one lane issues).  Per unit: the two resident tiles
// from (mapA, mapB) at tile rt, then the streamed tiles from (mapC, mapD) at tiles
// first .. first+n-1 in the order C_0 D_0 C_1 D_1 ...
template <int D, int KIND>
__device__ __forceinline__ void bwd_producer(const BwdParams& p, const Waiter& W, const Bars& B, uint32_t sbase,
                                             const CUtensorMap* mapA, const CUtensorMap* mapB,
                                             const CUtensorMap* mapC, const CUtensorMap* mapD) {
  using L = BwdLayout<D, KIND>;
  const int G = gridDim.x;
  int stage = 0, nu = 0;
  uint32_t phase = 0, issued = 0, issued_parity = 0;
  bool res_issued = false, ok = true;
  uint32_t res_parity = 0;
  int vi = 0;  // dK/dV kernel: steps whose LSE / D vectors have been requested
  uint32_t vec_issued = 0, vec_parity = 0;
  for (int k = 0; ok && k * G < p.num_units; ++k) {
    const int w = bwd_unit_of(k, blockIdx.x, G);
    if (w >= p.num_units) continue;
    int bh, rt, first, n;
    bwd_decode<KIND>(p, w, bh, rt, first, n);
    if (!(ok = wait_all(W, B.res_empty, (nu & 1) ^ 1))) break;
    mbar_arrive_expect_tx_elect(B.res_full, L::RES_TILES * L::TILE);
#pragma unroll
    for (int b = 0; b < L::BOXES; ++b) {
      tma_load_3d_elect(sbase + L::RES_OFF + b * BOX, mapA, b * 64, rt * BT, bh, B.res_full);
      if (L::RES_TILES == 2)
        tma_load_3d_elect(sbase + L::RES_OFF + L::TILE + b * BOX, mapB, b * 64, rt * BT, bh, B.res_full);
    }
    res_issued = true;
    res_parity = nu & 1;
    ++nu;
    for (int t = 0; ok && t < 2 * n; ++t) {
      if (KIND == 1 && !(t & 1)) {  // the step's LSE * log2 e and D vectors (512 bytes each)
        const int vb = vi & 1;
        if (!(ok = wait_all(W, B.vec_empty + 8 * vb, ((vi >> 1) & 1) ^ 1))) break;
        const uint32_t dst = sbase + L::VEC_OFF + vb * 2 * BT * 4;
        const size_t off = static_cast<size_t>(bh) * p.Tp + static_cast<size_t>(first + (t >> 1)) * BT;
        mbar_arrive_expect_tx_elect(B.vec_full + 8 * vb, 2 * BT * 4);
        bulk_load_elect(dst, p.lse2 + off, BT * 4, B.vec_full + 8 * vb);
        bulk_load_elect(dst + BT * 4, p.drow + off, BT * 4, B.vec_full + 8 * vb);
        vec_issued |= 1u << vb;
        vec_parity = (vec_parity & ~(1u << vb)) | (uint32_t((vi >> 1) & 1) << vb);
        ++vi;
      }
      if (!(ok = wait_all(W, B.ring_empty + 8 * stage, phase ^ 1))) break;
      mbar_arrive_expect_tx_elect(B.ring_full + 8 * stage, L::TILE);
#pragma unroll
      for (int b = 0; b < L::BOXES; ++b)
        tma_load_3d_elect(sbase + L::RING_OFF + stage * L::TILE + b * BOX, (t & 1) ? mapD : mapC, b * 64,
                          (first + (t >> 1)) * BT, bh, B.ring_full + 8 * stage);
      // the same tensor's tile two steps on into L2: the ring can hold only two steps, and a
      // stage is free only once the step that holds it has finished
      if ((t >> 1) + 2 < n) {
#pragma unroll
        for (int b = 0; b < L::BOXES; ++b)
          tma_prefetch_l2_3d_elect((t & 1) ? mapD : mapC, b * 64, (first + (t >> 1) + 2) * BT, bh);
      }
      issued |= 1u << stage;
      issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
      if (++stage == L::STAGES) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  if (!ok) {  // let every copy already issued land before the CTA exits
    if (res_issued) drain_all(W, B.res_full, res_parity);
    for (int s = 0; s < L::STAGES; ++s)
      if (issued & (1u << s)) drain_all(W, B.ring_full + 8 * s, (issued_parity >> s) & 1u);
    for (int b = 0; b < 2; ++b)
      if (vec_issued & (1u << b)) drain_all(W, B.vec_full + 8 * b, (vec_parity >> b) & 1u);
  }
}

// MMA issuer (whole warp, one lane issues).
//   KIND 0: S = Q K^T, dP = dO V^T; after the row warps wrote dS: dQ += dS K.
//   KIND 1: S^T = K Q^T, dP^T = V dO^T; after P^T, dS^T: dV += P^T dO, dK += dS^T Q.
// SPLIT schedule (P / dS in columns of their own): per step t the warp issues
//   S(t+1) once the row warps have read S(t) (s_free), dP(t+1) once they have read
//   dP(t) (dp_free), and the gradient products of step t once P / dS are written
//   (p_full), committing pv_done, which the row warps wait on before they overwrite
//   P / dS.  Otherwise (the d = 128 dK/dV kernel, whose accumulators fill half of Tensor
//   Memory) P^T is written over S^T and dS^T over dP^T, and the row warps signal P^T on its
//   own (p_half): per step the warp issues dV(t) once P^T(t) is written, S^T(t+1) behind it
//   (it overwrites P^T), dK(t) once dS^T(t) is written, and dP^T(t+1) behind that, so dV and
//   the next S^T run while the row warps form dS, and dK and the next dP^T while they form
//   the next P.
template <int D, int KIND>
__device__ __forceinline__ void bwd_mma(const BwdParams& p, const Waiter& W, const Bars& B, uint32_t sbase,
                                        uint32_t tmem) {
  using L = BwdLayout<D, KIND>;
  using SC = BwdSched<D, KIND>;
  constexpr uint32_t IDESC_S = make_idesc_bf16(BT, BT, 0);  // both operands K-major (d contiguous)
  constexpr uint32_t IDESC_G = make_idesc_bf16(BT, D, 1);   // B MN-major: rows of d contiguous elements
  const uint64_t dk = make_sdesc_sw128(sbase, 16, 1024);
  const uint64_t dm = make_sdesc_sw128(sbase, BOX, 1024);  // the second 64-column chunk is one box further
  const uint32_t dk_lo = uint32_t(dk), dk_hi = uint32_t(dk >> 32);
  const uint32_t dm_lo = uint32_t(dm), dm_hi = uint32_t(dm >> 32);
  const int G = gridDim.x;
  int stage = 0, nu = 0;
  uint32_t phase = 0, pf = 0, oe = 0, sfr = 0, dpf = 0, dof = 0, phf = 0;
  bool ok = true;
#define BWD_TAKE(slot)                                                   \
  {                                                                      \
    slot = stage;                                                        \
    if (!(ok = wait_all(W, B.ring_full + 8 * stage, phase))) break;      \
    if (++stage == L::STAGES) {                                          \
      stage = 0;                                                         \
      phase ^= 1;                                                        \
    }                                                                    \
    tc_fence_after();                                                    \
  }
#define BWD_WAIT(bar, par)                                  \
  {                                                         \
    if (!(ok = wait_all(W, bar, par))) break;               \
    par ^= 1;                                               \
    tc_fence_after();                                       \
  }
// [resident tile r] x [streamed tile in stage st]^T into Tensor Memory column col
#define BWD_SCORE(col, r, st)                                                                              \
  {                                                                                                        \
    _Pragma("unroll") for (int kk = 0; kk < D / 16; ++kk) {                                                \
      const uint32_t off = ((kk / 4) * BOX + (kk % 4) * 32) >> 4;                                          \
      mma_ss_elect(tmem + (col), dk_lo + ((L::RES_OFF + (r) * L::TILE) >> 4) + off, dk_hi,                  \
                   dk_lo + ((L::RING_OFF + (st) * L::TILE) >> 4) + off, dk_hi, IDESC_S, kk > 0 ? 1u : 0u);   \
    }                                                                                                      \
  }
// dP (or dP^T) = [resident tile 1] x [streamed tile in stage st]^T; the d = 128 dQ kernel
// takes dO from Tensor Memory instead (A operand as bf16 pairs, B the V tile K-major)
#define BWD_DP(st)                                                                                        \
  {                                                                                                       \
    if (L::DO_TMEM) {                                                                                     \
      _Pragma("unroll") for (int kk = 0; kk < D / 16; ++kk) {                                             \
        const uint32_t off = ((kk / 4) * BOX + (kk % 4) * 32) >> 4;                                       \
        mma_ts_elect(tmem + COL_DP, tmem + COL_DO + kk * 8, dk_lo + ((L::RING_OFF + (st) * L::TILE) >> 4) + off, \
                     dk_hi, IDESC_S, kk > 0 ? 1u : 0u);                                                   \
      }                                                                                                   \
    } else                                                                                                \
      BWD_SCORE(COL_DP, 1, st);                                                                           \
  }
// accumulator col += (bf16 pairs at column a) x [streamed tile in stage st] (MN-major)
#define BWD_GRAD(col, a, st, acc0)                                                                         \
  {                                                                                                        \
    _Pragma("unroll") for (int kk = 0; kk < BT / 16; ++kk)                                                 \
      mma_ts_elect(tmem + (col), tmem + (a) + SC::a_col(kk), dm_lo + ((L::RING_OFF + (st) * L::TILE + kk * 2048) >> 4), \
                   dm_hi, IDESC_G, (acc0) | (kk > 0 ? 1u : 0u));                                           \
  }
  for (int k = 0; ok && k * G < p.num_units; ++k) {
    const int w = bwd_unit_of(k, blockIdx.x, G);
    if (w >= p.num_units) continue;
    int bh, rt, first, n;
    bwd_decode<KIND>(p, w, bh, rt, first, n);
    if (!(ok = wait_all(W, B.res_full, nu & 1))) break;
    ++nu;
    tc_fence_after();
    int s0 = 0, s1 = 0;  // ring stages of the current step's two streamed tiles
    if (!SC::SPLIT) {
      do {  // step 0's two products (they follow the previous unit's gradient products in issue order)
        BWD_TAKE(s0);
        BWD_SCORE(COL_S, 0, s0);
        mma_commit_elect(B.s_full);
        BWD_TAKE(s1);
        BWD_SCORE(COL_DP, 1, s1);
        mma_commit_elect(B.dp_full);
      } while (0);
      if (!ok) break;
    } else {
      do {  // step 0's two products
        BWD_TAKE(s0);
        {
          uint32_t par = sfr ^ 1;
          BWD_WAIT(B.s_free, par);
          sfr ^= 1;
        }
        BWD_SCORE(COL_S, 0, s0);
        mma_commit_elect(B.s_full);
        BWD_TAKE(s1);
        {
          uint32_t par = dpf ^ 1;
          BWD_WAIT(B.dp_free, par);
          dpf ^= 1;
        }
        if (L::DO_TMEM) BWD_WAIT(B.do_full, dof);  // the row warps have put the unit's dO in place
        BWD_DP(s1);
        mma_commit_elect(B.dp_full);
      } while (0);
      if (!ok) break;
    }
    for (int t = 0; t < n; ++t) {
      int n0 = -1, n1 = -1;
      if (SC::SPLIT && t + 1 < n) {  // the next step's products, as soon as this step's have been read
        BWD_TAKE(n0);
        {
          uint32_t par = sfr ^ 1;
          BWD_WAIT(B.s_free, par);
          sfr ^= 1;
        }
        BWD_SCORE(COL_S, 0, n0);
        mma_commit_elect(B.s_full);
        BWD_TAKE(n1);
        {
          uint32_t par = dpf ^ 1;
          BWD_WAIT(B.dp_free, par);
          dpf ^= 1;
        }
        BWD_DP(n1);
        mma_commit_elect(B.dp_full);
      }
      if (t == 0) {
        uint32_t par = oe ^ 1;
        BWD_WAIT(B.o_empty, par);
        oe ^= 1;
      }
      const uint32_t acc0 = t > 0 ? 1u : 0u;
      if (!SC::SPLIT) {  // dV(t) once P^T(t) is written, then the next S^T over it
        BWD_WAIT(B.p_half, phf);
        BWD_GRAD(COL_ACC, SC::COL_P, s1, acc0);  // dV += P^T dO_i
        mma_commit_elect(B.ring_empty + 8 * s1);
        if (t + 1 < n) {
          BWD_TAKE(n0);
          BWD_SCORE(COL_S, 0, n0);
          mma_commit_elect(B.s_full);
        }
      }
      BWD_WAIT(B.p_full, pf);
      if (KIND == 0) {
        BWD_GRAD(COL_ACC, SC::COL_DS, s0, acc0);  // dQ += dS K_j
      } else if (SC::SPLIT) {
        BWD_GRAD(COL_ACC, SC::COL_P, s1, acc0);       // dV += P^T dO_i
        BWD_GRAD(COL_ACC + D, SC::COL_DS, s0, acc0);  // dK += dS^T Q_i
      } else {  // dS^T sits over dP^T
        BWD_GRAD(COL_ACC + D, SC::COL_DS, s0, acc0);  // dK += dS^T Q_i
      }
      if (SC::SPLIT) {
        mma_commit_elect(B.pv_done);
        mma_commit_elect(B.ring_empty + 8 * s1);
      }
      mma_commit_elect(B.ring_empty + 8 * s0);
      if (!SC::SPLIT && t + 1 < n) {
        BWD_TAKE(n1);
        BWD_SCORE(COL_DP, 1, n1);
        mma_commit_elect(B.dp_full);
      }
      if (t + 1 == n) {
        mma_commit_elect(B.res_empty);
        mma_commit_elect(B.o_full);
      }
      s0 = n0;
      s1 = n1;
    }
  }
#undef BWD_TAKE
#undef BWD_WAIT
#undef BWD_SCORE
#undef BWD_DP
#undef BWD_GRAD
  // every MMA and commit arrival has landed before Tensor Memory is freed
  mma_commit_elect(B.done);
  drain_all(W, B.done, 0);
}

// Row warps: eight, two per TMEM lane quarter; warp w holds row 32 (w % 4) + lane of
// the unit's 128-row tile and columns [64h, 64h + 64) with h = w / 4.  Each step:
//   P = exp(S - LSE) with masked entries 0, packed to bf16 pairs;
//   dS = P (dP - D), packed to bf16 pairs;
// and the pairs go to Tensor Memory for the gradient products.  With the SPLIT
// schedule S and dP are read whole before anything is written (s_free and dp_free
// let the MMA warp overwrite them with the next step's), and P / dS go to their own
// columns once the previous step's gradient products are done (pv_done); otherwise P
// goes over the S columns the warp has read and is signalled on its own (p_half), and
// dS over the dP columns it has read.
// KIND 0 (dQ): the row is a query; LSE and D are per row, the mask runs along keys.
// KIND 1 (dK, dV): the row is a key; LSE and D are per column (query), read from the
// step's vectors in shared memory (every lane reads the same word), and P^T is
// stored as well as dS^T.
template <int D, int KIND>
__device__ __forceinline__ void bwd_rows(const BwdParams& p, const Waiter& W, const Bars& B, uint32_t tmem,
                                         uint32_t vec) {
  using L = BwdLayout<D, KIND>;
  using SC = BwdSched<D, KIND>;
  constexpr int HC = BT / 2;  // columns per half
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q4 = warp % 4, h = warp / 4;
  const int r = q4 * 32 + lane;
  const uint32_t lane_off = uint32_t(q4 * 32) << 16;
  const uint32_t t_s = tmem + lane_off + COL_S + HC * h, t_dp = tmem + lane_off + COL_DP + HC * h;
  const uint32_t t_p = tmem + lane_off + SC::COL_P + SC::half_col(h);
  const uint32_t t_ds = tmem + lane_off + SC::COL_DS + SC::half_col(h);
  const float sl2 = p.scale_log2;
  const int G = gridDim.x;
  uint32_t sf = 0, dpf = 0, pvd = 0;
  int it = 0;  // steps so far (vector buffer, first pv_done wait)
  int ku = 0;  // dQ kernel: units so far (row-vector hand-over)
  bool ok = true;
  for (int k = 0; ok && k * G < p.num_units; ++k) {
    const int w = bwd_unit_of(k, blockIdx.x, G);
    if (w >= p.num_units) continue;
    int bh, rt, first, n;
    bwd_decode<KIND>(p, w, bh, rt, first, n);
    const int r0 = rt * BT, row = r0 + r;  // this thread's query (KIND 0) or key (KIND 1)
    const size_t rp = static_cast<size_t>(bh) * p.Tp + row;  // the row in the padded workspace
    // KIND 0: LSE * log2 e of the row (+inf past T: P = 0 there); D from the output warps,
    // read once step 0's P has been formed
    const float lse2_row =
        KIND == 0 ? (row < p.T ? __ldg(p.lse + static_cast<size_t>(bh) * p.T + row) * LOG2E : INFINITY) : 0.f;
    float d_row = 0.f;
    for (int t = 0; t < n; ++t, ++it) {
      const int c0 = (first + t) * BT;  // first column of the step: a key (KIND 0) or query (KIND 1)
      const uint32_t lv = vec + ((it & 1) * 2 * BT + HC * h) * 4;  // KIND 1: this half's LSE * log2 e; + 4 BT: D
      if (KIND == 1) {  // the producer has copied the step's LSE * log2 e and D vectors
        if (!(ok = W.wait(B.vec_full + 8 * (it & 1), (it >> 1) & 1))) break;
      }
      // columns valid for this row: KIND 0 keys < min(T, row + 1) (causal); KIND 1 queries >= row
      int lim = BT, lo = 0;
      if (KIND == 0) {
        if ((p.causal && c0 + BT - 1 > r0) || c0 + BT > p.T) {
          lim = p.T - c0;
          if (p.causal) lim = min(lim, row - c0 + 1);
        }
      } else if (p.causal && c0 == r0) {
        lo = r;  // the diagonal tile: query q sees key `row` only if q >= row
      }
      lim -= HC * h;  // in this half's column numbering
      lo -= HC * h;
      if (!(ok = W.wait(B.s_full, sf))) break;
      sf ^= 1;
      tc_fence_after();
      uint32_t pp[HC / 2];  // P as bf16 pairs
#pragma unroll
      for (int c = 0; c < HC / 32; ++c) {
        float4 l4[8];  // KIND 1: the chunk's LSE * log2 e, read before the Tensor Memory load
        if (KIND == 1) {
#pragma unroll
          for (int f = 0; f < 8; ++f) l4[f] = ld_shared_v4f(lv + (32 * c + 4 * f) * 4);
        }
        uint32_t sv[32];
        tmem_ld32_wait(t_s + 32 * c, sv);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float l0 = lse2_row, l1 = lse2_row;
          if (KIND == 1) {
            l0 = (e & 1) ? l4[e / 2].z : l4[e / 2].x;
            l1 = (e & 1) ? l4[e / 2].w : l4[e / 2].y;
          }
          float x0, x1;
          ffma2v(x0, x1, u2f(sv[2 * e]), u2f(sv[2 * e + 1]), sl2, -l0, -l1);
          pp[16 * c + e] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
        }
      }
      if (lim < HC || lo > 0) {  // a diagonal or ragged tile: masked entries of P become +0
#pragma unroll
        for (int e = 0; e < HC / 2; ++e) {
          if (2 * e >= lim || 2 * e < lo) pp[e] &= 0xFFFF0000u;
          if (2 * e + 1 >= lim || 2 * e + 1 < lo) pp[e] &= 0x0000FFFFu;
        }
      }
      if (SC::SPLIT) {  // S may now be overwritten by the next step's
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.s_free);
      } else {  // P^T over the first half of this warp's S^T columns, read above; then dV may start
#pragma unroll
        for (int c = 0; c < HC / 32; ++c)
          tmem_st16(t_p + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(pp + 16 * c));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.p_half);
      }
      if (SC::SPLIT && KIND == 1) {  // P waits for the previous products
        if (it > 0) {
          if (!(ok = W.wait(B.pv_done, pvd))) break;
          pvd ^= 1;
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < HC / 32; ++c)
          tmem_st16(t_p + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(pp + 16 * c));
      }
      if (KIND == 0 && t == 0) {  // the output warps have written the unit's D rows
        if (!(ok = W.wait(B.rv_full + 8 * (ku & 1), (ku >> 1) & 1))) break;
        ++ku;
        d_row = __ldcg(p.drow + rp);
      }
      if (!(ok = W.wait(B.dp_full, dpf))) break;
      dpf ^= 1;
      tc_fence_after();
      // dS, 32 columns at a time: stored as it is formed (without SPLIT over the dP columns this
      // warp has read, chunk c's 16 pairs over the first half of chunk c's 32 columns read so
      // far; with SPLIT into the dS^T columns once the previous step's products are done), or,
      // in the dQ kernel, kept until dP is released and the previous dQ product has read the dS
      // columns
      uint32_t pdk[KIND == 0 ? HC / 2 : 1];
#pragma unroll
      for (int c = 0; c < HC / 32; ++c) {
        float4 d4[8];  // KIND 1: the chunk's D, read before the Tensor Memory load
        if (KIND == 1) {
#pragma unroll
          for (int f = 0; f < 8; ++f) d4[f] = ld_shared_v4f(lv + (BT + 32 * c + 4 * f) * 4);
        }
        uint32_t dv[32];
        tmem_ld32_wait(t_dp + 32 * c, dv);
        uint32_t pd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float d0 = d_row, d1 = d_row;
          if (KIND == 1) {
            d0 = (e & 1) ? d4[e / 2].z : d4[e / 2].x;
            d1 = (e & 1) ? d4[e / 2].w : d4[e / 2].y;
          }
          const uint32_t pw = pp[16 * c + e];
          float s0, s1;
          fmulsub2(s0, s1, u2f(pw << 16), u2f(pw & 0xFFFF0000u), u2f(dv[2 * e]), u2f(dv[2 * e + 1]), d0, d1);
          pd[e] = pack_bf16x2(s0, s1);
          if (KIND == 0) pdk[16 * c + e] = pd[e];
        }
        if (KIND == 1) tmem_st16(t_ds + 16 * c, pd);
      }
      if (KIND == 1) {  // this warp is done with the step's vectors
        __syncwarp();
        if (lane == 0) mbar_arrive(B.vec_empty + 8 * (it & 1));
      }
      if (SC::SPLIT) {  // dP may now be overwritten by the next step's
        if (KIND == 1) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(B.dp_free);
      }
      if (KIND == 0) {  // the previous dQ product has read the dS columns: store this step's
        if (it > 0) {
          if (!(ok = W.wait(B.pv_done, pvd))) break;
          pvd ^= 1;
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < HC / 32; ++c) tmem_st16(t_ds + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(pdk + 16 * c));
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.p_full);
    }
    if (!ok) break;
  }
}

// This lane's row of dO (d = 128, bf16) into Tensor Memory columns [t_do, t_do + 64) as
// bf16 pairs: the A operand of the dQ kernel's dP = dO V^T.  Rows past T are zeros.
__device__ __forceinline__ void bwd_load_do(const BwdParams& p, int bh, int row, uint32_t t_do) {
  const uint4* src = reinterpret_cast<const uint4*>(p.dout + (static_cast<size_t>(bh) * p.T + row) * 128);
#pragma unroll
  for (int c2 = 0; c2 < 2; ++c2) {  // 64 elements (32 pairs) at a time
    uint32_t dw[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = row < p.T ? __ldg(src + 8 * c2 + c) : make_uint4(0, 0, 0, 0);
      dw[4 * c] = x.x;
      dw[4 * c + 1] = x.y;
      dw[4 * c + 2] = x.z;
      dw[4 * c + 3] = x.w;
    }
    tmem_st32(t_do + 32 * c2, dw);
  }
  tmem_wait_st();
}

// Output warps: four, warp w holding rows 32 (w % 4) + lane of the unit's tile and all of
// the accumulator's columns.  Once a unit's last gradient product is done (o_full) the d = 128
// dQ kernel first puts the next unit's dO into Tensor Memory (do_full; the first unit's at
// the start); then the accumulator is read 32 columns at a time, scaled, packed to bf16 and
// stored -- 32 x 32 boxes through two staging boxes per warp and TMA stores (rows past T lie
// outside the output map and are not written), or at d = 128 in the dQ kernel, whose shared
// memory holds no staging, by each thread for its own row -- and o_empty releases the
// accumulator to the next unit.  The row warps meanwhile start on the next unit.
template <int D, int KIND>
__device__ __forceinline__ void bwd_out(const BwdParams& p, const Waiter& W, const Bars& B, uint32_t tmem,
                                        uint32_t stg, const CUtensorMap* g1, const CUtensorMap* g2) {
  using L = BwdLayout<D, KIND>;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int q4 = warp % 4;
  const uint32_t lane_off = uint32_t(q4 * 32) << 16;
  const uint32_t t_acc = tmem + lane_off + COL_ACC;
  const int G = gridDim.x;
  // the first unit index >= k this CTA works on, or -1
  auto next_unit = [&](int k) -> int {
    for (; k * G < p.num_units; ++k)
      if (bwd_unit_of(k, blockIdx.x, G) < p.num_units) return k;
    return -1;
  };
  auto put_do = [&](int k) {  // unit k's dO for this warp's rows, then do_full
    int bh, rt, first, n;
    bwd_decode<KIND>(p, bwd_unit_of(k, blockIdx.x, G), bh, rt, first, n);
    bwd_load_do(p, bh, rt * BT + q4 * 32 + lane, tmem + lane_off + COL_DO);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.do_full);
  };
  auto put_rv = [&](int k, int b) {  // dQ kernel: unit k's D and LSE * log2 e rows, then rv_full[b]
    // (the row warps wait for D only once step 0's P is formed; the dK/dV kernel reads both)
    int bh, rt, first, n;
    bwd_decode<KIND>(p, bwd_unit_of(k, blockIdx.x, G), bh, rt, first, n);
    bwd_row_vectors<D>(p, bh, rt * BT + q4 * 32, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(B.rv_full + 8 * b);
  };
  uint32_t of = 0;
  bool ok = true;
  int nb = 0;             // boxes staged so far: the next goes to staging box nb & 1
  bool stg_busy = false;  // a TMA store may still be reading a staging box
  int ku = 0;             // units so far
  {
    const int k0 = next_unit(0);
    if (KIND == 0 && k0 >= 0) put_rv(k0, 0);
    if (L::DO_TMEM && k0 >= 0) put_do(k0);
  }
  for (int k = 0; ok && k * G < p.num_units; ++k) {
    const int w = bwd_unit_of(k, blockIdx.x, G);
    if (w >= p.num_units) continue;
    int bh, rt, first, n;
    bwd_decode<KIND>(p, w, bh, rt, first, n);
    if (KIND == 0) {  // the next unit's vectors while this one runs
      const int k2 = next_unit(k + 1);
      if (k2 >= 0) put_rv(k2, (ku + 1) & 1);
    }
    ++ku;
    if (!(ok = W.wait(B.o_full, of))) break;
    of ^= 1;
    tc_fence_after();
    if (L::DO_TMEM) {  // every product of this unit has finished reading the dO columns
      const int k2 = next_unit(k + 1);
      if (k2 >= 0) put_do(k2);
    }
    const int y0 = rt * BT + q4 * 32, row = y0 + lane;
    if (L::DIRECT_OUT) {
      __nv_bfloat16* out = p.dq + (static_cast<size_t>(bh) * p.T + row) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32_wait(t_acc + 32 * c, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(u2f(v[2 * e]) * p.scale, u2f(v[2 * e + 1]) * p.scale);
        if (row < p.T) {
          uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        }
      }
    }
#pragma unroll
    for (int part = 0; !L::DIRECT_OUT && part < (KIND == 0 ? 1 : 2); ++part) {  // KIND 0: dQ; KIND 1: dV, then dK
      const CUtensorMap* gm = part ? g2 : g1;
      const float f = (KIND == 0 || part) ? p.scale : 1.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32_wait(t_acc + part * D + 32 * c, v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(u2f(v[2 * e]) * f, u2f(v[2 * e + 1]) * f);
        const uint32_t box = stg + (nb & 1) * L::STG_BOX_BYTES;
        if (stg_busy) {  // the store two boxes back, which used this staging box, has read it
          if (lane == 0) bulk_wait_group_read1();
          __syncwarp();
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) st_shared_v4(box + lane * 64 + e * 16, pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (y0 < p.T) {
          if (lane == 0) {
            tma_store_3d(gm, box, 32 * c, y0, bh);
            bulk_commit_group();
          }
          stg_busy = true;
        }
        ++nb;
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.o_empty);
  }
  if (stg_busy && lane == 0) bulk_wait_group0();  // this warp's gradient stores have completed
  __syncwarp();
}

template <int D, int KIND>
__global__ void __launch_bounds__(BWD_THREADS, 1)
fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmG1, const __grid_constant__ CUtensorMap tmG2, const BwdParams p) {
  using L = BwdLayout<D, KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const Bars B = make_bars<D, KIND>(sbase + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  const int warp = threadIdx.x / 32;
  const uint32_t tmem = bwd_setup<D, KIND>(smem, B, tmem_slot, abort_flag, warp);
  const Waiter W{abort_flag, p.timeout_ns, &g_bwd_status};
  // the set-up above overlaps the previous kernel's tail; memory is read only after it has
  // finished (the tensor maps are kernel parameters, so fetching them may start earlier).
  // Before that, the first unit's resident tiles and first two streamed tiles are pulled
  // into L2: a prefetch only warms the cache that every write of the previous kernel goes
  // through, so it cannot return stale data.
  if (warp == BWD_PRODUCER && threadIdx.x % 32 == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    const int w = bwd_unit_of(0, blockIdx.x, gridDim.x);
    if (w < p.num_units) {
      int bh, rt, first, n;
      bwd_decode<KIND>(p, w, bh, rt, first, n);
      const CUtensorMap* res[2] = {KIND == 0 ? &tmQ : &tmK, KIND == 0 ? &tmDO : &tmV};
      const CUtensorMap* str[2] = {KIND == 0 ? &tmK : &tmQ, KIND == 0 ? &tmV : &tmDO};
      for (int b = 0; b < L::BOXES; ++b)
        for (int m = 0; m < 2; ++m) {
          tma_prefetch_l2_3d(res[m], b * 64, rt * BT, bh);
          for (int j = 0; j < min(n, 2); ++j) tma_prefetch_l2_3d(str[m], b * 64, (first + j) * BT, bh);
        }
    }
  }
  if (warp == OUT_WARP0 && threadIdx.x % 32 == 0) {
    tma_prefetch_desc(&tmG1);
    if (KIND == 1) tma_prefetch_desc(&tmG2);
  }
  pdl_launch_dependents();
  pdl_wait();
  if (warp == BWD_PRODUCER) {
    if (KIND == 0)
      bwd_producer<D, 0>(p, W, B, sbase, &tmQ, &tmDO, &tmK, &tmV);  // resident Q, dO; streamed K, V
    else
      bwd_producer<D, 1>(p, W, B, sbase, &tmK, &tmV, &tmQ, &tmDO);  // resident K, V; streamed Q, dO
    __syncwarp();
  } else if (warp == BWD_MMA) {
    bwd_mma<D, KIND>(p, W, B, sbase, tmem);
    __syncwarp();
  } else if (warp >= OUT_WARP0) {
    bwd_out<D, KIND>(p, W, B, tmem, sbase + L::STG_OFF + (warp - OUT_WARP0) * 2 * L::STG_BOX_BYTES, &tmG1, &tmG2);
  } else {
    bwd_rows<D, KIND>(p, W, B, tmem, sbase + L::VEC_OFF);
  }
  bwd_teardown<D>(tmem, warp);
}

template <int D, int KIND>
cudaError_t launch_bwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& dout,
                       const CUtensorMap& g1, const CUtensorMap& g2, const BwdParams& p, int grid,
                       cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_bwd_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdLayout<D, KIND>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(BWD_THREADS);
  cfg.dynamicSmemBytes = BwdLayout<D, KIND>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_bwd_kernel<D, KIND>, q, k, v, dout, g1, g2, p);
}

}  // namespace

cudaError_t launch_bwd_dq(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, const CUtensorMap& g1, const CUtensorMap& g2, const BwdParams& p,
                          int grid, cudaStream_t stream) {
  return d == 64 ? launch_bwd<64, 0>(q, k, v, dout, g1, g2, p, grid, stream)
                 : launch_bwd<128, 0>(q, k, v, dout, g1, g2, p, grid, stream);
}

cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& g1, const CUtensorMap& g2,
                            const BwdParams& p, int grid, cudaStream_t stream) {
  return d == 64 ? launch_bwd<64, 1>(q, k, v, dout, g1, g2, p, grid, stream)
                 : launch_bwd<128, 1>(q, k, v, dout, g1, g2, p, grid, stream);
}

int fa_bwd_smem_bytes(int d) {
  return d == 64 ? max(BwdLayout<64, 0>::SMEM, BwdLayout<64, 1>::SMEM) : max(BwdLayout<128, 0>::SMEM, BwdLayout<128, 1>::SMEM);
}

cudaError_t read_and_clear_bwd_status(cudaStream_t stream, unsigned int* out) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
