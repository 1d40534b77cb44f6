// FlashAttention forward for sm_103a: a warp-specialised persistent kernel.
//
// What it computes ("Flash Attention, tiled: exact attention without the T x T
// HBM matrix", section "From the example to tiled GPU work", the per-tile
// procedure; "FlashAttention: the IO-aware Attention Kernel", section 3.2):
// for every query tile Q_i and every visible key/value tile K_j, V_j
//   S_ij = Q_i K_j^T, masked; per row m' = max(m, max s), r = e^(m - m'),
//   l = r l + sum p, o = r o + p^T V_j with p = e^(s - m'); at the end O = o / l
// and the row's log-sum-exp.  Scores are kept in base-2 units of the scaled
// score (s * scale * log2 e), so every exponential is one ex2.
//
// Lazy rescale ("FlashAttention and Fused Kernels", section "Four generations
// of FlashAttention", FlashAttention-4): a row's reference max m is moved, and
// l and o rescaled, only when the tile max exceeds m by more than log2(256) = 8;
// otherwise the stale m is kept, so p <= 2^8, and the final o / l and the LSE
// use that same m, which keeps the result exact up to rounding.
//
// Two row sums are kept: lr sums the rounded weights p~ that the P V MMA
// multiplies by, and O = sum p~ v / lr is a convex combination of the value
// rows under exactly the weights used (a row dominated by one key returns that
// key's value row unchanged, whatever the stale m); l sums the fp32 weights and
// gives the LSE without the rounding of the weights.  At d = 64 and for e4m3
// the tensor core forms lr itself: as 16 extra columns of O_i += P_i [V_j | 1]
// (d = 64), or as L_i += P_i x ones, a product of its own (e4m3).
//
// Roles (one CTA per SM, persistent over work units):
//   warps 0-3  softmax for query tile 0 of the unit (one TMEM lane = one row per thread)
//   warps 4-7  softmax for query tile 1 (d = 64, e4m3: the tiles of a causal unit may be
//              handed to the two slots the other way round, see balance_slots)
//   warp 8     TMA producer: Q tiles once per unit, then K_j, V_j through a ring
//   warp 9     Tensor Memory allocator; tcgen05.mma issuer (bf16 d = 128: both tiles;
//              d = 64 and e4m3: tile 0)
//   warp 10    d = 64 and e4m3: tcgen05.mma issuer for tile 1 (warp 11 only joins the
//              final barrier; 384 threads there, 320 at bf16 d = 128)
// The issuing warps run their schedules on all 32 lanes (every operand stays
// warp-uniform); elect.sync inside each TMA, MMA and commit picks the lane that
// issues it.
// A work unit is (batch*head, 256 query rows) = two 128-row query tiles that
// share every K/V tile loaded.  Tensor Memory (512 columns, fp32), bf16 d = 128:
//   S_0 [0,128)  S_1 [128,256)  O_0 [256,384)  O_1 [384,512)
// with P_i (bf16 pairs) written over the first 64 columns of S_i once S_i has
// been read, so S_i(j+1) waits for P_i(j) V_j.  d = 64 and e4m3: one S buffer
// [0,128) that the two tiles' products take in turn, then O_0, O_1 and P_0, P_1
// in columns of their own, so the next S is computed while the softmax of S_i(j)
// runs, and each tile's MMAs are issued by a warp of its own.
// O leaves through shared memory: each softmax warp writes its 32 rows x 64
// columns in the 128-byte swizzled layout of the output tensor map and one lane
// stores them with a TMA tensor store, so every store moves whole rows.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fa_kernel.h"
#include "ptx.cuh"


namespace fa {

constexpr int BM = 128;          // query rows per tile
constexpr int BN = 128;          // keys per tile
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP0 = 9;   // MMA issuer for query tile 0; also allocates Tensor Memory
constexpr int MMA_WARP1 = 10;  // MMA issuer for query tile 1 (warp 11 only joins the final barrier)
constexpr uint32_t TMEM_COLS = 512;
constexpr int BOX_BYTES = 128 * 128;  // one TMA box: 128 rows x 64 bf16, 128-byte swizzle
constexpr float LN2 = 0.693147180559945309f;

__device__ unsigned int g_status;  // bit 0: a bounded wait ran out

// F8: Q, K and V are e4m3 bytes (d = 128 only), V read from a transposed copy (d rows of
// keys), P packed to e4m3 for the P V product.
template <int D, bool F8 = false>
struct Layout {
  static constexpr int TILE_BYTES = BM * D * (F8 ? 1 : 2);
  static constexpr int BOXES = F8 ? 1 : D / 64;        // TMA boxes of 128-byte rows per tile
  // d = 64 and e4m3: two units' Q tiles resident (the next unit's load overlaps the
  // current unit); bf16 d = 128: one unit's Q tiles, the next unit's prefetched into L2.
  static constexpr int QBUF = (D == 128 && !F8) ? 1 : 2;
  static constexpr int STAGES = (D == 128 && !F8) ? 4 : (F8 ? 5 : 6);  // K/V ring depth (tiles)
  static constexpr int Q_OFF = 0;                      // [QBUF units][2 query tiles]
  static constexpr int KV_OFF = QBUF * 2 * TILE_BYTES;
  // d = 64 and e4m3: P_i has Tensor Memory columns of its own and the two query tiles' S
  // products share one buffer, so the next S may be computed while the softmax of S_i(j) runs
  // (see the MMA issuers); bf16 d = 128: P_i overwrites S_i, each tile has its own S buffer.
  static constexpr bool SEP_P = D == 64 || F8;
  // d = 64: O_i += P_i [V_j | 1]: the P V product also forms the sum of the rounded weights
  // (16 columns of ones after V, read from a constant block in shared memory), which divides O.
  static constexpr bool ONES = SEP_P && D == 64 && !F8;
  static constexpr int ON = D;                          // O columns per query tile in TMEM
  static constexpr int ON_MMA = ONES ? D + 16 : D;      // columns the P V product writes
  // e4m3: L_i += P_i x ones (16 columns of one), a product of its own that forms the sum of the
  // rounded weights; its B operand is a constant K-major block of e4m3 ones (16 rows x 128 keys)
  static constexpr bool LSUM = F8;
  // d = 64 and e4m3: one MMA-issuing warp per query tile (warps 9, 10; warp 11 idle);
  // bf16 d = 128: warp 9 alone
  static constexpr int THREADS = SEP_P ? 384 : 320;
  static constexpr int MMA_WARPS = SEP_P ? 2 : 1;
  // bf16 O staging per softmax warp: 32 rows x 64 columns (4 KB, 128-byte swizzle), and for
  // e4m3 (d = 128, where the ring's tiles are half as large) a second one, so that the two
  // 64-column halves of a row need not wait for each other's store
  static constexpr int STG_OFF = KV_OFF + STAGES * TILE_BYTES;
  static constexpr bool STG2 = F8;
  static constexpr int STG_WARP_BYTES = (STG2 ? 2 : 1) * 32 * 128;
  // d = 64: the ones block, laid out as one more 64-column V atom (128 rows of 128 bytes, 1 KB aligned)
  static constexpr int ONES_OFF = STG_OFF + 8 * STG_WARP_BYTES;
  static constexpr int ONES_BYTES = ONES ? 128 * 128 : (LSUM ? 16 * 128 : 0);
  static constexpr int BAR_OFF = ONES_OFF + ONES_BYTES;
  // q_full[2], q_empty[2], kv_full[S], kv_empty[S], s_full[2], p_full[2], o_full[2], o_empty[2],
  // s_free[2], done, unit_full[4], unit_empty[4]
  static constexpr int NUM_BARS = 4 + 2 * STAGES + 10 + 1 + 8;
  // TMEM base slot, abort flag, S-read counters [2], claimed work items [4]
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 32 + 1024;  // + slack to align the base to 1 KB
  // Tensor Memory columns.  bf16 d = 128: S_0 [0,128), S_1 [128,256), O_0, O_1 after them, P_i
  // over S_i.  d = 64: one S buffer [0,128) that the two query tiles' products take in turn,
  // O_0 [128,208) and O_1 [224,304) (64 columns of O and 16 of the weight sum each),
  // P_0 [320,384) and P_1 [384,448).  e4m3: S [0,128), O_0 [128,256), O_1 [256,384),
  // P_0 [384,416), P_1 [416,448) (four e4m3 weights per column), L_0 [448,464), L_1 [464,480).
  static constexpr uint32_t OSTRIDE = ONES ? 96u : uint32_t(D);  // Tensor Memory columns per O_i
  static constexpr uint32_t PCOLS = F8 ? 32u : 64u;                // columns of P_i (4 e4m3 or 2 bf16 each)
  static __device__ __forceinline__ constexpr uint32_t s_col(int i) { return SEP_P ? 0u : uint32_t(i) * 128u; }
  static __device__ __forceinline__ constexpr uint32_t o_col(int i) {
    return SEP_P ? 128u + uint32_t(i) * OSTRIDE : 256u + uint32_t(i) * ON;
  }
  static __device__ __forceinline__ constexpr uint32_t p_col(int i) {
    return SEP_P ? 128u + 2u * OSTRIDE + uint32_t(i) * PCOLS : s_col(i);
  }
  static __device__ __forceinline__ constexpr uint32_t l_col(int i) { return 448u + uint32_t(i) * 16u; }
};
static_assert(Layout<64>::p_col(1) + 64 <= 512 && Layout<128>::p_col(1) + 64 <= 512 &&
              Layout<128, true>::p_col(1) + 32 <= 512, "Tensor Memory columns exceed 512");
static_assert(Layout<64>::ONES_OFF % 1024 == 0 && Layout<128, true>::ONES_OFF % 1024 == 0,
              "the ones block must be 1 KB aligned like the tiles");

constexpr int MAX_SMEM_PER_CTA = 232448;  // 227 KB opt-in dynamic shared memory per block on sm_103
static_assert(Layout<64>::SMEM_BYTES <= MAX_SMEM_PER_CTA && Layout<128>::SMEM_BYTES <= MAX_SMEM_PER_CTA,
              "shared-memory layout exceeds the per-CTA limit");

struct Unit {
  int bh, qb;
  int jb;      // first K/V tile of the unit (0 unless the key range is split)
  int n0, n1;  // K/V tiles slot 0 / slot 1 visits from jb (0 = nothing to do for that slot)
  int sw;      // slot i holds query tile i ^ sw of the unit (see balance_slots)
};

// Work item w -> (batch*head, 256-row query block[, key split]).  Causal
// launches list the longest query blocks first (all heads' longest blocks, then
// the next longest, ...), which balances the persistent CTAs.  Non-causal units
// all cost the same, so they are listed head by head: the CTAs running at one
// time then share a few heads' K and V, which stay in L2.  With split keys,
// split s of a unit covers key tiles [s * split_tiles, (s + 1) * split_tiles)
// of what each query tile may see.
template <bool PARTIAL, bool GROUPED, bool HALVES>
__device__ __forceinline__ Unit decode_unit(const Params& p, int w) {
  Unit u;
  int band, s = 0;
  int half = -1;  // a one-tile item: which query tile of its unit
  if (HALVES && !PARTIAL && p.halves > 0 && w >= p.num_units - p.halves) {
    const int t = w - (p.num_units - p.halves);
    half = t & 1;
    w = p.num_units - p.halves + (t >> 1);
  }
  if (PARTIAL) {
    const int per_band = p.BH * p.num_splits;
    band = w / per_band;
    const int rem = w - band * per_band;
    s = rem / p.BH;
    u.bh = rem - s * p.BH;
  } else if (GROUPED && p.head_group > 0) {  // causal: band by band within each group of head_group heads,
    const int main_bands = p.nqb - p.tail_bands;  // then the lightest bands band by band over all heads
    const int main_units = p.BH * main_bands;
    if (w < main_units) {
      const int per_group = p.head_group * main_bands;
      const int g = w / per_group, r = w - g * per_group;
      band = r / p.head_group;
      u.bh = g * p.head_group + (r - band * p.head_group);
    } else {
      const int t = w - main_units, b2 = t / p.BH;
      band = main_bands + b2;
      u.bh = t - b2 * p.BH;
    }
  } else {  // one division: w = first * unit_div + second
    const int first = w / p.unit_div, second = w - first * p.unit_div;
    band = p.causal ? first : second;
    u.bh = p.causal ? second : first;
  }
  u.qb = p.causal ? (p.nqb - 1 - band) : band;
  const int q0 = u.qb * 2 * BM, q1 = q0 + BM;
  const int e0 = (q0 >= p.T) ? 0 : (p.causal ? min(p.nk, q0 / BN + 1) : p.nk);  // tiles visible to tile 0
  const int e1 = (q1 >= p.T) ? 0 : (p.causal ? min(p.nk, q1 / BN + 1) : p.nk);
  u.sw = 0;
  if (PARTIAL) {
    u.jb = s * p.split_tiles;
    const int end = u.jb + p.split_tiles;
    u.n0 = max(0, min(e0, end) - u.jb);
    u.n1 = max(0, min(e1, end) - u.jb);
  } else {
    u.jb = 0;
    u.n0 = e0;
    u.n1 = e1;
    if (half >= 0) {  // slot 0 takes query tile `half` of the unit, slot 1 nothing
      u.n0 = half ? e1 : e0;
      u.n1 = 0;
      u.sw = half;
    }
  }
  return u;
}

// d = 64, where each query tile has an MMA warp and a softmax warpgroup of its own: the two
// tiles of a causal unit see different numbers of K/V tiles, so the longer one goes to the
// slot that has had less work so far in this CTA (bal = K/V steps of slot 0 minus slot 1).
// Every role walks the same list of units and reaches the same assignment.
__device__ __forceinline__ void balance_slots(Unit& u, int& bal) {
  if (u.n0 != u.n1 && bal != 0 && ((u.n1 > u.n0) == (bal < 0))) {
    const int t = u.n0;
    u.n0 = u.n1;
    u.n1 = t;
    u.sw ^= 1;
  }
  bal += u.n0 - u.n1;
}

// The k-th work item of CTA b in a grid of G: a snake over the heavy-first list
// (b, 2G-1-b, 2G+b, ...), which pairs long causal units with short ones.
__device__ __forceinline__ int unit_of(int k, int b, int G) { return k * G + ((k & 1) ? (G - 1 - b) : b); }

// Claimed work items (p.sched != nullptr): a CTA's first item is blockIdx.x; every later one is
// claimed by the producer warp from the counter pair (item G + the counter's previous value,
// so that the list is worked through in order, each CTA taking the next item whenever it is
// ready for one) and handed to the other warps through a ring of four shared-memory slots:
// item k (k >= 1) goes through slot (k - 1) % 4, whose unit_full barrier the producer
// completes after writing it and whose unit_empty barrier the readers (softmax and MMA warps)
// complete after reading it.  Returns item k for a reading warp, or -1 when the producer has
// handed out an index past the last unit (or a wait ran out: ok = false).
__device__ __forceinline__ int claimed_item(const Params& p, const Waiter& W, uint32_t slots, uint32_t full,
                                            uint32_t empty, int k, bool& ok) {
  if (k == 0) return blockIdx.x;
  const int j = k - 1, s = j & 3;
  if (!(ok = wait_all(W, full + 8 * s, (j >> 2) & 1))) return -1;
  int w;
  asm volatile("ld.shared.s32 %0, [%1];" : "=r"(w) : "r"(slots + 4 * s) : "memory");
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty + 8 * s);
  return w < p.num_units ? w : -1;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Split-KV hand-off ("FlashAttention and Fused Kernels", section "Flash-Decoding": each split
// yields a partial output and one log-sum-exp scalar per row; the partials are weighted by their
// LSE).  Called by a whole warp after it has written the partials of its 32 rows [r0, r0 + 32)
// of head bh for one split: the warp counts itself in that row group's counter, and the warp
// that completes the count (the last split of the group to finish, in whatever CTA) merges the
// group: with M = max_s LSE_s and w_s = e^(LSE_s - M),
//   O = sum_s w_s O_s / sum_s w_s,   LSE = M + ln sum_s w_s,
// over the n_run splits that hold a key these rows can see.  Lane l takes the LSE of row
// r0 + l (M, the weight sum, and each split's weight, handed to the other lanes by shuffle);
// the rows' outputs are formed eight rows at a time with every lane holding D / 32 columns,
// so that eight rows of a split (and two splits) are loaded at once rather than one row after
// another.
template <int D>
__device__ __noinline__ void split_handoff(const Params& p, int bh, int r0, int n_run, int lane) {
  __threadfence();  // this warp's partials are visible device-wide before it is counted
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(p.counters + static_cast<size_t>(bh) * p.ngroups + r0 / 32, 1) == n_run - 1;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();  // the other splits' partials, counted before this warp, are read after their fences
  constexpr int CPL = D / 32;
  constexpr int RB = 8;  // rows per block of the output pass
  const size_t rows = static_cast<size_t>(p.BH) * p.T;
  const size_t g0 = static_cast<size_t>(bh) * p.T + r0;  // first row of the group
  const int nrows = min(32, p.T - r0);
  const bool live = lane < nrows;
  const float* lse_l = p.lsepart + g0 + lane;  // this lane's row in split 0's LSE
  // M and the weight sum in one pass (the sum rescaled whenever the maximum grows), loads four
  // splits at a time
  float M = -INFINITY, wsum = 0.f;
  if (live) {
#pragma unroll 4
    for (int s = 0; s < n_run; ++s) {
      const float x = __ldcg(lse_l + s * rows);
      if (x > M) {
        wsum = wsum * expf(M - x) + 1.f;  // M = -inf at first: 0 * 0 + 1
        M = x;
      } else {
        wsum += expf(x - M);
      }
    }
    p.lse[g0 + lane] = M + logf(wsum);
  }
  const float inv = live ? 1.f / wsum : 0.f;
  for (int t0 = 0; t0 < nrows; t0 += RB) {
    float acc[RB][CPL];
#pragma unroll
    for (int t = 0; t < RB; ++t)
#pragma unroll
      for (int c = 0; c < CPL; ++c) acc[t][c] = 0.f;
#pragma unroll 2
    for (int s = 0; s < n_run; ++s) {
      const float wl = live ? expf(__ldcg(lse_l + s * rows) - M) * inv : 0.f;  // row r0 + lane's weight
      const float* src = p.opart + (s * rows + g0 + t0) * D + lane * CPL;
      float v[RB][CPL];
#pragma unroll
      for (int t = 0; t < RB; ++t) {
        if (t0 + t < nrows) {
          if (CPL == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + t * D));
            v[t][0] = x.x;
            v[t][1] = x.y;
            v[t][2 % CPL] = x.z;
            v[t][3 % CPL] = x.w;
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src + t * D));
            v[t][0] = x.x;
            v[t][1] = x.y;
          }
        } else {
#pragma unroll
          for (int c = 0; c < CPL; ++c) v[t][c] = 0.f;
        }
      }
#pragma unroll
      for (int t = 0; t < RB; ++t) {
        const float w = __shfl_sync(0xffffffffu, wl, t0 + t);
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[t][c] += w * v[t][c];
      }
    }
#pragma unroll
    for (int t = 0; t < RB; ++t) {
      if (t0 + t >= nrows) break;
      __nv_bfloat16* dst = p.o + (g0 + t0 + t) * D + lane * CPL;
      if (CPL == 4) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(acc[t][0], acc[t][1]),
                                                    pack_bf16x2(acc[t][2 % CPL], acc[t][3 % CPL]));
      } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[t][0], acc[t][1]);
      }
    }
  }
}

// CLAIM: the work items are claimed at run time in head-group order (p.sched, p.head_group set;
// unsplit bf16 d = 128 only); every other launch takes the static order, in an instantiation
// that compiles none of the claiming code.
template <int D, bool PARTIAL, bool F8 = false, bool CLAIM = false>
__global__ void __launch_bounds__(Layout<D, F8>::THREADS, 1)
fa_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, const Params p) {
  using L = Layout<D, F8>;
  static_assert(!F8 || (D == 128 && !PARTIAL), "the e4m3 path is d = 128, unsplit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t q_smem = sbase + L::Q_OFF;   // [unit buffer][query tile]
  const uint32_t kv_smem = sbase + L::KV_OFF;
  const uint32_t bar0 = sbase + L::BAR_OFF;
  // barrier addresses (8 bytes each)
  const uint32_t bar_q_full = bar0;                          // [2]
  const uint32_t bar_q_empty = bar0 + 16;                    // [2]
  const uint32_t bar_kv_full = bar0 + 32;                    // [STAGES]
  const uint32_t bar_kv_empty = bar0 + 32 + 8 * L::STAGES;   // [STAGES]
  const uint32_t barx = bar0 + 32 + 16 * L::STAGES;
  const uint32_t bar_s_full = barx;        // [2]
  const uint32_t bar_p_full = barx + 16;   // [2]
  const uint32_t bar_o_full = barx + 32;   // [2]
  const uint32_t bar_o_empty = barx + 48;  // [2]
  const uint32_t bar_s_free = barx + 64;   // [2] (SEP_P: one phase per S_i read, 4 arrivals)
  const uint32_t bar_done = barx + 80;
  const uint32_t bar_unit_full = barx + 88;    // [4] claimed work items (see claimed_item)
  const uint32_t bar_unit_empty = barx + 120;  // [4]
  const uint32_t unit_slots = sbase + L::MISC_OFF + 16;  // [4] s32
  static_assert(!CLAIM || (D == 128 && !F8 && !PARTIAL), "claimed items: unsplit bf16 d = 128 only");
  constexpr bool claimed = CLAIM;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  // SEP_P: S reads of query tile i whose softmax step has ended, 4 per S (one per softmax warp of
  // the tile); they guard the MMA warps' waits on s_free (see the MMA issuers)
  const uint32_t s_reads = sbase + L::MISC_OFF + 8;  // [2] u32

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_q_full + 8 * b, 1);
      mbar_init(bar_q_empty + 8 * b, L::MMA_WARPS);  // one release per MMA-issuing warp
    }
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar_kv_full + 8 * s, 1);
      mbar_init(bar_kv_empty + 8 * s, L::MMA_WARPS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s_full + 8 * i, 1);
      mbar_init(bar_p_full + 8 * i, 4);
      mbar_init(bar_o_full + 8 * i, 1);
      mbar_init(bar_o_empty + 8 * i, 4);
      mbar_init(bar_s_free + 8 * i, 4);
    }
    mbar_init(bar_done, L::MMA_WARPS);
    for (int s = 0; s < 4; ++s) {
      mbar_init(bar_unit_full + 8 * s, 1);
      mbar_init(bar_unit_empty + 8 * s, 8 + L::MMA_WARPS);  // every softmax and MMA warp reads each item
    }
    *abort_flag = 0;
    reinterpret_cast<uint32_t*>(smem + L::MISC_OFF + 8)[0] = 0;
    reinterpret_cast<uint32_t*>(smem + L::MISC_OFF + 8)[1] = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP0) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  if (L::ONES || L::LSUM) {  // 1.0 everywhere in the block; the tensor core reads it through the async proxy
    const uint32_t one = L::LSUM ? 0x38383838u : 0x3F803F80u;  // e4m3 or bf16 ones
    for (int t = threadIdx.x; t < L::ONES_BYTES / 16; t += L::THREADS)
      st_shared_v4(sbase + L::ONES_OFF + 16 * t, one, one, one, one);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Waiter W{abort_flag, p.timeout_ns, &g_status};
  // the set-up above overlaps the previous kernel's tail; inputs are read only after it has
  // finished (the tensor maps are kernel parameters, so fetching them may start earlier).
  // Before that, the first unit's query tiles and first key / value tiles are pulled into
  // L2: a prefetch only warms the cache that every write of the previous kernel goes
  // through, so it cannot return stale data (the block table of paged K/V is input data,
  // so paged K/V tiles are not prefetched here).
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    const int w = unit_of(0, blockIdx.x, G);
    if (w < p.num_units) {
      const Unit u = decode_unit<PARTIAL, CLAIM, F8>(p, w);
      const int nmax = max(u.n0, u.n1);
      if (nmax > 0) {
        for (int i = 0; i < 2; ++i)
          for (int b = 0; b < L::BOXES; ++b) tma_prefetch_l2_3d(&tmQ, b * 64, u.qb * 2 * BM + (i ^ u.sw) * BM, u.bh);
        if (!p.block_table) {
          const int kvh = p.group == 1 ? u.bh : (u.bh / p.H) * (p.H / p.group) + (u.bh % p.H) / p.group;
          for (int j = 0; j < min(nmax, 2); ++j)
            for (int b = 0; b < L::BOXES; ++b) {
              tma_prefetch_l2_3d(&tmK, b * 64, (u.jb + j) * BN, kvh);
              if (F8)
                tma_prefetch_l2_3d(&tmV, (u.jb + j) * BN, 0, kvh);
              else
                tma_prefetch_l2_3d(&tmV, b * 64, (u.jb + j) * BN, kvh);
            }
        }
      }
    }
  }
  if (!PARTIAL && warp == 0 && lane == 0) tma_prefetch_desc(&tmO);
  pdl_launch_dependents();
  pdl_wait();

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer (whole warp, one lane issues)
    {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0, q_issued = 0, q_parity = 0;  // for draining after a timeout
      bool ok = true;
      int nu = 0;  // units this CTA has started
      int bal = 0;
      for (int k = 0; ok; ++k) {
        int w;
        if (claimed) {
          if (k == 0) {
            w = int(blockIdx.x);
          } else {  // claimed when this warp is ready to load it (claiming a unit ahead was 2 % slower)
            int c = 0;
            if (lane == 0) c = atomicAdd(p.sched, 1);
            w = G + __shfl_sync(0xffffffffu, c, 0);
          }
          if (k > 0) {  // hand item k to the other warps (see claimed_item)
            const int j = k - 1, s = j & 3;
            if (!(ok = wait_all(W, bar_unit_empty + 8 * s, ((j >> 2) & 1) ^ 1))) break;
            if (lane == 0) {
              asm volatile("st.shared.s32 [%0], %1;" ::"r"(unit_slots + 4 * s), "r"(w) : "memory");
              mbar_arrive(bar_unit_full + 8 * s);
            }
            __syncwarp();
          }
          if (w >= p.num_units) break;
        } else {
          if (k * G >= p.num_units) break;
          w = unit_of(k, blockIdx.x, G);
          if (w >= p.num_units) continue;
        }
        Unit u = decode_unit<PARTIAL, CLAIM, F8>(p, w);
        if (L::SEP_P) balance_slots(u, bal);
        const int nmax = max(u.n0, u.n1);
        if (nmax == 0) continue;  // an empty key split: no role touches it
        // the K/V head this query head reads (query heads share K/V heads in groups)
        const int kvh = p.group == 1 ? u.bh : (u.bh / p.H) * (p.H / p.group) + (u.bh % p.H) / p.group;
        // paged K/V: the batch entry's block table row (logical 128-key page -> physical page)
        const int* pages = p.block_table ? p.block_table + static_cast<size_t>(u.bh / p.H) * p.max_pages : nullptr;
        const int qb = nu % L::QBUF;
        const uint32_t qpar = (nu / L::QBUF) & 1;
        if (!(ok = wait_all(W, bar_q_empty + 8 * qb, qpar ^ 1))) break;
        mbar_arrive_expect_tx_elect(bar_q_full + 8 * qb, ((u.n0 > 0) + (u.n1 > 0)) * L::TILE_BYTES);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if ((i ? u.n1 : u.n0) == 0) continue;
#pragma unroll
          for (int b = 0; b < L::BOXES; ++b) {
            const uint32_t dst = q_smem + (2 * qb + i) * L::TILE_BYTES + b * BOX_BYTES;
            const int y = u.qb * 2 * BM + (i ^ u.sw) * BM;
            if (claimed)  // query tiles are read once (output tiles written once): in L2 they go before K, V
              tma_load_3d_elect_hint(dst, &tmQ, b * 64, y, u.bh, bar_q_full + 8 * qb, l2_policy_evict_first());
            else
              tma_load_3d_elect(dst, &tmQ, b * 64, y, u.bh, bar_q_full + 8 * qb);
          }
        }
        q_issued |= 1u << qb;
        q_parity = (q_parity & ~(1u << qb)) | (qpar << qb);
        ++nu;
        // warm L2 with the next unit's query tiles (not with claimed items, whose next unit is not
        // known yet)
        if (L::QBUF == 1 && !claimed) {
          int k2 = k + 1, w2 = unit_of(k2, blockIdx.x, G);
          if (w2 >= p.num_units && (k2 + 1) * G < p.num_units) w2 = unit_of(++k2, blockIdx.x, G);
          if (w2 < p.num_units) {
            const Unit u2 = decode_unit<PARTIAL, CLAIM, F8>(p, w2);
            for (int i = 0; i < 2; ++i)
              if ((i ? u2.n1 : u2.n0) > 0)
                for (int b = 0; b < L::BOXES; ++b)
                  tma_prefetch_l2_3d_elect(&tmQ, b * 64, u2.qb * 2 * BM + (i ^ u2.sw) * BM, u2.bh);
          }
        }
        // ring order = the order the MMA warps take tiles in: K_0 V_0 K_1 V_1 ..., or with
        // separate P buffers K_0 K_1 V_0 K_2 V_1 K_3 ... V_(n-2) V_(n-1) (S runs a step ahead)
#define FA_LOAD(kv, j)                                                                                    \
  {                                                                                                       \
    if (!(ok = wait_all(W, bar_kv_empty + 8 * stage, phase ^ 1))) break;                                  \
    /* paged: the tile is one whole page, row 0 of (page, K/V head) in the page pool */                   \
    int row0 = (u.jb + (j)) * BN, head = kvh;                                                             \
    if (pages) {                                                                                          \
      int pg = pages[u.jb + (j)];                                                                         \
      if (pg < 0 || pg >= p.num_pages) { /* out of the pool: read zeros and report it */                  \
        if ((threadIdx.x & 31) == 0) atomicOr(&g_status, 2u);                                             \
        pg = p.num_pages;                                                                                 \
      }                                                                                                   \
      row0 = 0;                                                                                           \
      head = pg * p.Hkv + kvh % p.Hkv;                                                                    \
    }                                                                                                     \
    mbar_arrive_expect_tx_elect(bar_kv_full + 8 * stage, L::TILE_BYTES);                                  \
    _Pragma("unroll") for (int b = 0; b < L::BOXES; ++b)                                                  \
      tma_load_3d_elect(kv_smem + stage * L::TILE_BYTES + b * BOX_BYTES, (kv) == 0 ? &tmK : &tmV,            \
                        (F8 && (kv) == 1) ? (u.jb + (j)) * BN : b * 64,                                   \
                        (F8 && (kv) == 1) ? 0 : row0, head, bar_kv_full + 8 * stage);                   \
    issued |= 1u << stage;                                                                                \
    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);                                  \
    if (++stage == L::STAGES) {                                                                           \
      stage = 0;                                                                                          \
      phase ^= 1;                                                                                         \
    }                                                                                                     \
  }
        if (L::SEP_P) {
          do {
            FA_LOAD(0, 0);
            if (nmax > 1) FA_LOAD(0, 1);
          } while (0);
          for (int j = 0; ok && j < nmax; ++j) {
            FA_LOAD(1, j);
            if (j + 2 < nmax) FA_LOAD(0, j + 2);
          }
        } else {
          for (int j = 0; ok && j < nmax; ++j) {
            FA_LOAD(0, j);
            FA_LOAD(1, j);
          }
        }
#undef FA_LOAD
      }
      if (!ok) {  // let every copy already issued land before the CTA exits
        for (int b = 0; b < 2; ++b)
          if (q_issued & (1u << b)) drain_all(W, bar_q_full + 8 * b, (q_parity >> b) & 1u);
        for (int s = 0; s < L::STAGES; ++s)
          if (issued & (1u << s)) drain_all(W, bar_kv_full + 8 * s, (issued_parity >> s) & 1u);
      }
    }
    __syncwarp();
  } else if (L::SEP_P && (warp == MMA_WARP0 || warp == MMA_WARP1)) {
    // ------------------------------------------------------------ MMA issuers, one warp per query tile (SEP_P)
    // Each warp runs its tile's schedule on all 32 lanes and elects one lane per MMA.  Both
    // warps walk the whole K/V ring in the producer's order and release every stage (and
    // the unit's Q buffer) whether or not their tile used it, so kv_empty and q_empty
    // complete after two arrivals.
    //
    // The two tiles' S products share one Tensor Memory buffer and take it in turn: per K/V
    // step S_0(x), then S_1(x) (a tile past its last step drops out), unit after unit.  A
    // product is issued once the softmax has read the one before it in that order.  Each read
    // of S_t is recorded twice: the four softmax warps of tile t arrive on s_free[t] (one phase
    // per read) right after it, and add one each to the counter s_reads[t] (release) at the
    // end of that step.  A warp may come to wait
    // for a read two or more reads ahead of tile t's progress (for instance the first S of its
    // next unit while the other tile still has two products to go), and an mbarrier's phase
    // parity cannot tell that apart from a completed phase; so the MMA warp first waits
    // (acquire) until the counter shows every earlier read of tile t, and only then waits on
    // the phase of the read it needs, which is then the barrier's current or completed one.
    {
      const int i = warp - MMA_WARP0;  // query tile of this warp
      constexpr uint32_t IDESC_S = F8 ? make_idesc_e4m3(BM, BN) : make_idesc_bf16(BM, BN, 0);  // both K-major
      // O += P [V | 1] (d = 64), O += P V (V MN-major), or e4m3 O += P (V^T)^T (both K-major)
      constexpr uint32_t IDESC_PV = F8 ? make_idesc_e4m3(BM, L::ON) : make_idesc_bf16(BM, L::ON_MMA, 1);
      constexpr int KSTEP = F8 ? 32 : 16;  // reduction depth of one MMA
      // Descriptor halves: the address field (low 14 bits, in 16-byte units) and, for V, the
      // leading byte offset (bits 16-29: from the V tile to the ones block, the second 64-column
      // atom of B) are the parts that change; every offset added below stays inside its field.
      const uint64_t dqk = make_sdesc_sw128(sbase, 16, 1024);        // K-major tiles (Q, K)
      const uint64_t dvv = make_sdesc_sw128(sbase, BOX_BYTES, 1024);  // MN-major V tiles
      const uint32_t dqk_lo = uint32_t(dqk), dqk_hi = uint32_t(dqk >> 32);
      const uint32_t dv_lo = uint32_t(dvv), dv_hi = uint32_t(dvv >> 32);
      const uint32_t ones_addr = sbase + L::ONES_OFF;
      const uint32_t my_p_full = bar_p_full + 8 * i;
      const uint32_t my_o_full = bar_o_full + 8 * i, my_o_empty = bar_o_empty + 8 * i;
      const uint32_t d_s = tmem + L::s_col(i), d_o = tmem + L::o_col(i), a_p = tmem + L::p_col(i);
      const uint32_t d_l = tmem + L::l_col(i);
      constexpr uint32_t IDESC_L = make_idesc_e4m3(BM, 16);
      const uint32_t ones_lo = uint32_t(make_sdesc_sw128(ones_addr, 16, 1024));
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pf = 0, oe = 0;
      int cnt0 = 0, cnt1 = 0;  // S products of tile 0 / tile 1 in the units before this one
      int last_t = -1;         // tile of the last S product of those units (-1: none yet)
      bool ok = true;
      int nu = 0;
      int bal = 0;
      for (int k = 0; ok; ++k) {
        const int w = claimed ? claimed_item(p, W, unit_slots, bar_unit_full, bar_unit_empty, k, ok)
                              : (k * G < p.num_units ? unit_of(k, blockIdx.x, G) : -1);
        if (w < 0) break;
        if (w >= p.num_units) continue;
        Unit u = decode_unit<PARTIAL, CLAIM, F8>(p, w);
        balance_slots(u, bal);
        const int n = i ? u.n1 : u.n0, nmax = max(u.n0, u.n1);
        if (nmax == 0) continue;
        const int qb = nu % L::QBUF;
        if (!(ok = wait_all(W, bar_q_full + 8 * qb, (nu / L::QBUF) & 1))) break;
        ++nu;
        tc_fence_after();
        const uint32_t a_q = dqk_lo + ((L::Q_OFF + (2 * qb + i) * L::TILE_BYTES) >> 4);
        // S_i(x) over d in steps of 16 (stage ks of the ring), after the S product before it has been
        // read; after the tile's last S the Q buffer is released
#define FA_ISSUE_S(ks, x)                                                                               \
  {                                                                                                     \
    int pt = -1, pk = 0; /* tile and per-tile index of the S product before S_i(x) */                   \
    if (i == 1 && (x) < u.n0) {                                                                         \
      pt = 0, pk = cnt0 + (x);                                                                          \
    } else if ((x) > 0) {                                                                               \
      if (i == 0 && (x) - 1 < u.n1) pt = 1, pk = cnt1 + (x) - 1;                                        \
      else pt = i, pk = (i ? cnt1 : cnt0) + (x) - 1;                                                    \
    } else if (last_t >= 0) {                                                                           \
      pt = last_t, pk = (last_t ? cnt1 : cnt0) - 1;                                                     \
    }                                                                                                   \
    if (pt >= 0) {                                                                                      \
      if (!(ok = wait_count_all(W, s_reads + 4 * pt, 4u * uint32_t(pk)))) break;                         \
      if (!(ok = wait_all(W, bar_s_free + 8 * pt, uint32_t(pk) & 1u))) break;                           \
      tc_fence_after();                                                                                 \
    }                                                                                                   \
    const uint32_t b0 = dqk_lo + ((L::KV_OFF + (ks) * L::TILE_BYTES) >> 4);                             \
    _Pragma("unroll") for (int kk = 0; kk < D / KSTEP; ++kk) {                                          \
      const uint32_t off = (((kk / 4) * BOX_BYTES + (kk % 4) * 32) >> 4);                               \
      if (F8)                                                                                           \
        mma_f8_ss_elect(d_s, a_q + off, dqk_hi, b0 + off, dqk_hi, IDESC_S, kk > 0 ? 1u : 0u);           \
      else                                                                                              \
        mma_ss_elect(d_s, a_q + off, dqk_hi, b0 + off, dqk_hi, IDESC_S, kk > 0 ? 1u : 0u);              \
    }                                                                                                   \
    mma_commit_elect(bar_s_full + 8 * i);                                                               \
    if ((x) + 1 == n) mma_commit_elect(bar_q_empty + 8 * qb);                                           \
  }
        // O_i (+)= P_i [V | 1] over keys in steps of 16 (stage vs of the ring)
#define FA_ISSUE_PV(vs, acc)                                                                            \
  {                                                                                                     \
    const uint32_t v_addr = sbase + L::KV_OFF + (vs) * L::TILE_BYTES;                                    \
    if (F8) {                                                                                           \
      const uint32_t b0 = dqk_lo + ((L::KV_OFF + (vs) * L::TILE_BYTES) >> 4);                           \
      _Pragma("unroll") for (int kk = 0; kk < BN / KSTEP; ++kk)                                         \
        mma_f8_ts_elect(d_o, a_p + kk * 8, b0 + ((kk * 32) >> 4), dqk_hi, IDESC_PV, ((acc) || kk > 0) ? 1u : 0u); \
      if (L::LSUM)                                                                                      \
        _Pragma("unroll") for (int kk = 0; kk < BN / KSTEP; ++kk)                                       \
          mma_f8_ts_elect(d_l, a_p + kk * 8, ones_lo + ((kk * 32) >> 4), dqk_hi, IDESC_L,                \
                          ((acc) || kk > 0) ? 1u : 0u);                                                 \
    } else {                                                                                            \
      const uint32_t b0 = L::ONES ? (((v_addr >> 4) & 0x3FFFu) | (((ones_addr - v_addr) >> 4) << 16))  \
                                  : dv_lo + ((L::KV_OFF + (vs) * L::TILE_BYTES) >> 4);                  \
      _Pragma("unroll") for (int kk = 0; kk < BN / 16; ++kk)                                            \
        mma_ts_elect(d_o, a_p + kk * 8, b0 + ((kk * 2048) >> 4), dv_hi, IDESC_PV, ((acc) || kk > 0) ? 1u : 0u); \
    }                                                                                                   \
  }
#define FA_TAKE(slot)                                                      \
  {                                                                        \
    slot = stage;                                                          \
    if (!(ok = wait_all(W, bar_kv_full + 8 * stage, phase))) break;        \
    if (++stage == L::STAGES) {                                            \
      stage = 0;                                                           \
      phase ^= 1;                                                          \
    }                                                                      \
    tc_fence_after();                                                      \
  }
#define FA_WAIT(bar, par)                                       \
  {                                                             \
    if (!(ok = wait_all(W, bar, par))) break;                   \
    par ^= 1;                                                   \
    tc_fence_after();                                           \
  }
        {
          // S runs one K/V step ahead of the softmax; P_i(j) V_j once P_i(j) is written (p_full),
          // with a commit to o_full that the softmax waits on before it overwrites P_i or rescales
          // O_i, and at the end of the unit.  Ring order: K_0 K_1 V_0 K_2 V_1 ...
          do {
            int ks = 0;
            FA_TAKE(ks);
            if (n > 0) FA_ISSUE_S(ks, 0);
            mma_commit_elect(bar_kv_empty + 8 * ks);
            if (nmax > 1) {
              FA_TAKE(ks);
              if (n > 1) FA_ISSUE_S(ks, 1);
              mma_commit_elect(bar_kv_empty + 8 * ks);
            }
          } while (0);
          if (!ok) break;
          for (int j = 0; j < nmax; ++j) {
            int vs = 0;
            FA_TAKE(vs);
            if (j < n) {
              if (j == 0) {
                uint32_t par = oe ^ 1;
                FA_WAIT(my_o_empty, par);
                oe ^= 1;
              }
              FA_WAIT(my_p_full, pf);
              FA_ISSUE_PV(vs, j > 0);
              mma_commit_elect(my_o_full);
            }
            mma_commit_elect(bar_kv_empty + 8 * vs);
            if (j + 2 < nmax) {
              int ks = 0;
              FA_TAKE(ks);
              if (j + 2 < n) FA_ISSUE_S(ks, j + 2);
              mma_commit_elect(bar_kv_empty + 8 * ks);
            }
          }
        }
        if (!ok) break;
        if (n == 0) mma_commit_elect(bar_q_empty + 8 * qb);  // this tile had nothing to do in the unit
        cnt0 += u.n0;
        cnt1 += u.n1;
        last_t = u.n1 >= u.n0 ? 1 : 0;
#undef FA_ISSUE_S
#undef FA_ISSUE_PV
#undef FA_TAKE
#undef FA_WAIT
      }
      // every MMA and every commit arrival of both warps has landed before TMEM is freed
      mma_commit_elect(bar_done);
      drain_all(W, bar_done, 0);
    }
    __syncwarp();
  } else if (!L::SEP_P && warp == MMA_WARP0) {
    // ------------------------------------------------------------ MMA issuer, both query tiles (whole warp, one lane issues)
    {
      constexpr uint32_t IDESC_S = make_idesc_bf16(BM, BN, 0);   // S = Q K^T: both K-major
      constexpr uint32_t IDESC_PV = make_idesc_bf16(BM, L::ON, 1);  // O += P V: V is MN-major
      constexpr uint32_t IDESC_S8 = make_idesc_e4m3(BM, BN);     // e4m3: S = Q K^T
      constexpr uint32_t IDESC_PV8 = make_idesc_e4m3(BM, L::ON);  // e4m3: O += P (V^T)^T, both K-major
      constexpr int KSTEP = F8 ? 32 : 16;                        // reduction depth of one MMA
      // Descriptor halves: the address field (low 14 bits, in 16-byte units) is the
      // only part that changes, and every offset added below stays inside it.
      const uint64_t dqk = make_sdesc_sw128(sbase, 16, 1024);        // K-major tiles (Q, K)
      const uint64_t dvv = make_sdesc_sw128(sbase, BOX_BYTES, 1024);  // MN-major V tiles
      const uint32_t dqk_lo = uint32_t(dqk), dqk_hi = uint32_t(dqk >> 32);
      const uint32_t dv_lo = uint32_t(dvv), dv_hi = uint32_t(dvv >> 32);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pf0 = 0, pf1 = 0, oe0 = 0, oe1 = 0;
      bool ok = true;
      int nu = 0;
      for (int k = 0; ok; ++k) {
        const int w = claimed ? claimed_item(p, W, unit_slots, bar_unit_full, bar_unit_empty, k, ok)
                              : (k * G < p.num_units ? unit_of(k, blockIdx.x, G) : -1);
        if (w < 0) break;
        if (w >= p.num_units) continue;
        const Unit u = decode_unit<PARTIAL, CLAIM, F8>(p, w);
        const int n0 = u.n0, n1 = u.n1, nmax = max(n0, n1);
        if (nmax == 0) continue;
        const int last_i = n1 > 0 ? 1 : 0;
        const int qb = nu % L::QBUF;
        if (!(ok = wait_all(W, bar_q_full + 8 * qb, (nu / L::QBUF) & 1))) break;
        ++nu;
        tc_fence_after();
        const uint32_t q_lo0 = dqk_lo + ((L::Q_OFF + 2 * qb * L::TILE_BYTES) >> 4);
        // S_i = Q_i K^T over d in steps of 16 (stage ks of the ring)
#define FA_ISSUE_S(i, ks)                                                                                 \
  {                                                                                                       \
    const uint32_t a0 = q_lo0 + (((i) * L::TILE_BYTES) >> 4);                                             \
    const uint32_t b0 = dqk_lo + ((L::KV_OFF + (ks) * L::TILE_BYTES) >> 4);                               \
    _Pragma("unroll") for (int kk = 0; kk < D / KSTEP; ++kk) {                                            \
      const uint32_t off = (((kk / 4) * BOX_BYTES + (kk % 4) * 32) >> 4);                                 \
      if (F8)                                                                                             \
        mma_f8_ss_elect(tmem + L::s_col(i), a0 + off, dqk_hi, b0 + off, dqk_hi, IDESC_S8, kk > 0 ? 1u : 0u); \
      else                                                                                                \
        mma_ss_elect(tmem + L::s_col(i), a0 + off, dqk_hi, b0 + off, dqk_hi, IDESC_S, kk > 0 ? 1u : 0u);   \
    }                                                                                                     \
  }
        // O_i (+)= P_i V over keys in steps of 16 (bf16; V MN-major) or 32 (e4m3; V^T K-major),
        // stage vs of the ring
#define FA_ISSUE_PV(i, vs, acc)                                                                           \
  {                                                                                                       \
    const uint32_t s16 = ((vs) * L::TILE_BYTES) >> 4;                                                     \
    const uint32_t b0 = (F8 ? dqk_lo : dv_lo) + (L::KV_OFF >> 4) + s16;                                   \
    _Pragma("unroll") for (int kk = 0; kk < BN / KSTEP; ++kk) {                                           \
      if (F8)                                                                                             \
        mma_f8_ts_elect(tmem + L::o_col(i), tmem + L::p_col(i) + kk * 8, b0 + ((kk * 32) >> 4), dqk_hi,    \
                        IDESC_PV8, ((acc) || kk > 0) ? 1u : 0u);                                           \
      else                                                                                                \
        mma_ts_elect(tmem + L::o_col(i), tmem + L::p_col(i) + kk * 8, b0 + ((kk * 2048) >> 4), dv_hi,      \
                     IDESC_PV, ((acc) || kk > 0) ? 1u : 0u);                                               \
    }                                                                                                     \
  }
#define FA_TAKE(slot)                                                  \
  {                                                                    \
    slot = stage;                                                      \
    if (!(ok = wait_all(W, bar_kv_full + 8 * stage, phase))) break;         \
    if (++stage == L::STAGES) {                                        \
      stage = 0;                                                       \
      phase ^= 1;                                                      \
    }                                                                  \
    tc_fence_after();                                                  \
  }
        int ks = 0;
        do {
          FA_TAKE(ks);
        } while (0);
        if (!ok) break;
        if (n0 > 0) {
          FA_ISSUE_S(0, ks);
          mma_commit_elect(bar_s_full);
          if (last_i == 0 && n0 == 1) mma_commit_elect(bar_q_empty + 8 * qb);
        }
        if (n1 > 0) {
          FA_ISSUE_S(1, ks);
          mma_commit_elect(bar_s_full + 8);
          if (n1 == 1) mma_commit_elect(bar_q_empty + 8 * qb);
        }
        mma_commit_elect(bar_kv_empty + 8 * ks);
        for (int j = 0; j < nmax; ++j) {
          int vs = 0, ks1 = -1;
          FA_TAKE(vs);
          if (j < n0) {
            if (j == 0) {
              if (!(ok = wait_all(W, bar_o_empty, oe0 ^ 1))) break;
              oe0 ^= 1;
            }
            if (!(ok = wait_all(W, bar_p_full, pf0))) break;
            pf0 ^= 1;
            tc_fence_after();
            FA_ISSUE_PV(0, vs, j > 0);
            if (j + 1 == n0) mma_commit_elect(bar_o_full);
            if (j + 1 < n0) {
              FA_TAKE(ks1);
              FA_ISSUE_S(0, ks1);
              mma_commit_elect(bar_s_full);
              if (last_i == 0 && j + 2 == n0) mma_commit_elect(bar_q_empty + 8 * qb);
            }
          }
          if (j < n1) {
            if (j == 0) {
              if (!(ok = wait_all(W, bar_o_empty + 8, oe1 ^ 1))) break;
              oe1 ^= 1;
            }
            if (!(ok = wait_all(W, bar_p_full + 8, pf1))) break;
            pf1 ^= 1;
            tc_fence_after();
            FA_ISSUE_PV(1, vs, j > 0);
            if (j + 1 == n1) mma_commit_elect(bar_o_full + 8);
          }
          mma_commit_elect(bar_kv_empty + 8 * vs);
          if (j + 1 < n1) {
            if (ks1 < 0) FA_TAKE(ks1);
            FA_ISSUE_S(1, ks1);
            mma_commit_elect(bar_s_full + 8);
            if (j + 2 == n1) mma_commit_elect(bar_q_empty + 8 * qb);
          }
          if (ks1 >= 0) mma_commit_elect(bar_kv_empty + 8 * ks1);
        }
#undef FA_ISSUE_S
#undef FA_ISSUE_PV
#undef FA_TAKE
      }
      // every MMA and every commit arrival has landed before TMEM is freed
      mma_commit_elect(bar_done);
      drain_all(W, bar_done, 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax warpgroups
    const int i = warp / 4;         // query tile of this warpgroup
    const int wq = warp % 4;        // TMEM lane quarter this warp may access
    const int rt = wq * 32 + lane;  // row within the query tile
    const uint32_t lane_off = uint32_t(wq * 32) << 16;
    const uint32_t t_s = tmem + lane_off + L::s_col(i);
    const uint32_t t_o = tmem + lane_off + L::o_col(i);
    const uint32_t t_p = tmem + lane_off + L::p_col(i);
    const uint32_t my_s_full = bar_s_full + 8 * i, my_p_full = bar_p_full + 8 * i, my_s_reads = s_reads + 4 * i;
    const uint32_t my_s_free = bar_s_free + 8 * i;
    const uint32_t my_o_full = bar_o_full + 8 * i, my_o_empty = bar_o_empty + 8 * i;
    const float sl2 = p.scale_log2;
    const uint32_t stg = sbase + L::STG_OFF + warp * L::STG_WARP_BYTES;  // this warp's O staging
    bool stg_busy = false;  // a TMA store from the staging buffer may still be reading it
    uint32_t sf_phase = 0, of_phase = 0;
    bool ok = true;
    int bal = 0;
    for (int k = 0; ok; ++k) {
      const int w = claimed ? claimed_item(p, W, unit_slots, bar_unit_full, bar_unit_empty, k, ok)
                            : (k * G < p.num_units ? unit_of(k, blockIdx.x, G) : -1);
      if (w < 0) break;
      if (w >= p.num_units) continue;
      Unit u = decode_unit<PARTIAL, CLAIM, F8>(p, w);
      if (L::SEP_P) balance_slots(u, bal);
      const int n = i ? u.n1 : u.n0;
      if (n == 0) continue;
      const int q0 = u.qb * 2 * BM + (i ^ u.sw) * BM;
      const int row = q0 + rt;
      float m_run = -INFINITY;  // reference max, base-2 units of the scaled score
      float l = 0.f;            // sum of the fp32 weights: the softmax denominator of the LSE
      float lr = 0.f;           // sum of the bf16 weights the P V product used: divides O
      for (int j = 0; j < n; ++j) {
        if (!(ok = W.wait(my_s_full, sf_phase))) break;
        sf_phase ^= 1;
        tc_fence_after();
        uint32_t sr[BN];
        tmem_ld128_wait(t_s, sr);
        if (L::SEP_P) {  // S_i may now be overwritten by S_i(j+1)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(my_s_free);
        }
        const int k0 = (u.jb + j) * BN;
        if ((p.causal && k0 + BN - 1 > q0) || k0 + BN > p.T) {  // diagonal or ragged tail tile
          int lim = p.T - k0;
          if (p.causal) lim = min(lim, row - k0 + 1);
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= lim) sr[c] = f2u(-INFINITY);
        }
        float m8[8];  // eight independent chains of 2-input max (full rate; 3-input max is half rate)
#pragma unroll
        for (int e = 0; e < 8; ++e) m8[e] = u2f(sr[e]);
#pragma unroll
        for (int c = 8; c < BN; c += 8)
#pragma unroll
          for (int e = 0; e < 8; ++e) m8[e] = fmaxf(m8[e], u2f(sr[c + e]));
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int e = 0; e < w; ++e) m8[e] = fmaxf(m8[e], m8[e + w]);
        float mx = m8[0];
        mx *= sl2;
        // lazy rescale decision (warp-uniform: TMEM access below is warp-collective)
        float r = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_run = mx;
        } else if (__any_sync(0xffffffffu, mx > m_run + 8.f)) {
          const float m_new = (mx > m_run + 8.f) ? mx : m_run;
          r = ex2_approx(m_run - m_new);
          m_run = m_new;
          l *= r;
          lr *= r;
          rescale = true;
        }
        const float nm = -m_run;
        float la0 = 0.f, la1 = 0.f, lb0 = 0.f, lb1 = 0.f;  // fp32 weights, two packed chains
        float lr0 = 0.f, lr1 = 0.f;                         // bf16 weights
        uint32_t pk[BN / 2];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t h8 = 0;  // e4m3: this chunk's weights summed as f16 pairs (exact inputs, 16 terms)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float x0, x1;
            ffma2(x0, x1, u2f(sr[32 * c + 2 * e]), u2f(sr[32 * c + 2 * e + 1]), sl2, nm);
            const float p0 = ex2_approx(x0);
            const float p1 = ex2_approx(x1);
            if (e & 1)
              fadd2(lb0, lb1, p0, p1);
            else
              fadd2(la0, la1, p0, p1);
            if (F8) {  // four e4m3 weights per Tensor Memory column
              const uint32_t b2 = pack_e4m3x2(p0, p1);
              if (e & 1)
                pk[8 * c + e / 2] |= b2 << 16;
              else
                pk[8 * c + e / 2] = b2;
              if (!L::LSUM) h8 = add_f16x2(h8, e4m3x2_to_f16x2(b2));
              continue;
            }
            pk[16 * c + e] = pack_bf16x2(p0, p1);
            if (!L::ONES) add_bf16x2_f32(pk[16 * c + e], lr0, lr1);  // sum of the bf16 weights
          }
          if (F8) {
            if (!L::LSUM) {
              float h0, h1;
              f16x2_to_f32(h8, h0, h1);
              lr0 += h0;
              lr1 += h1;
            }
            if (!L::SEP_P && (c & 1))
              tmem_st16(t_p + (c / 2) * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16 * (c / 2)));
          } else if (!L::SEP_P) {
            tmem_st16(t_p + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16 * c));
          }
        }
        if (L::SEP_P) {  // P_i(j-1) V_(j-1) must be done before P_i is overwritten and before O_i is rescaled
          if (j > 0) {
            if (!(ok = W.wait(my_o_full, of_phase))) break;
            of_phase ^= 1;
            tc_fence_after();
          }
#pragma unroll
          for (int c = 0; c < int(L::PCOLS) / 16; ++c)
            tmem_st16(t_p + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(pk + 16 * c));
        }
        l += (la0 + la1) + (lb0 + lb1);
        if (!L::ONES && !L::LSUM) lr += lr0 + lr1;
        if (rescale) {  // o *= r; PV_i(j-1) has completed (it was issued before S_i(j), or waited for above)
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32_wait(t_o + c * 32, ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = f2u(u2f(ov[e]) * r);
            tmem_st32(t_o + c * 32, ov);
          }
          if (L::LSUM) {
            const uint32_t t_l = tmem + lane_off + L::l_col(i);
            tmem_st1(t_l, f2u(u2f(tmem_ld1_wait(t_l)) * r));
          }
          if (L::ONES) {  // the weight sum the tensor core keeps beside O
            uint32_t sv[16];
            tmem_ld16_wait(t_o + D, sv);
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[e] = f2u(u2f(sv[e]) * r);
            tmem_st16(t_o + D, sv);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // counted at the end of the step (release: after this read's s_free arrival), off the path
          // from the S read to the next S product; the count guards the MMA warps' s_free waits
          if (L::SEP_P) smem_count_add_release(my_s_reads, 1u);
          mbar_arrive(my_p_full);
        }
      }
      if (!ok) break;
      // epilogue: O = o / lr in bf16, LSE = ln(2) (m + log2 l)
      if (!(ok = W.wait(my_o_full, of_phase))) break;
      of_phase ^= 1;
      tc_fence_after();
      if (L::ONES) lr = u2f(tmem_ld1_wait(t_o + D));  // sum of the rounded weights, from the P [V | 1] product
      if (L::LSUM) lr = u2f(tmem_ld1_wait(tmem + lane_off + L::l_col(i)));  // from the P x ones product
      const float inv_l = p.v_descale / lr;  // v_descale: 1, or the e4m3 V's scale
      if (PARTIAL) {  // this split's normalised output (fp32) and its LSE
        const int s = u.jb / p.split_tiles;
        const size_t prow = static_cast<size_t>(s) * p.BH * p.T + static_cast<size_t>(u.bh) * p.T + row;
        float* orow = p.opart + prow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32_wait(t_o + c * 32, ov);
          if (row < p.T) {
            float4* dst = reinterpret_cast<float4*>(orow + c * 32);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(u2f(ov[4 * e]) * inv_l, u2f(ov[4 * e + 1]) * inv_l, u2f(ov[4 * e + 2]) * inv_l,
                                   u2f(ov[4 * e + 3]) * inv_l);
          }
        }
        if (row < p.T) p.lsepart[prow] = (m_run + log2f(l)) * LN2;
        const int r0 = q0 + wq * 32;
        if (r0 < p.T)  // splits that hold a key of this query tile: every one before its last visible key tile
          split_handoff<D>(p, u.bh, r0, p.causal ? min(p.num_splits, (q0 / BN) / p.split_tiles + 1) : p.num_splits,
                           lane);
      } else {
        // O in bf16 through shared memory: the warp's 32 rows x 64 columns in the 128-byte
        // swizzled layout of the output map (16-byte chunk c of row r at chunk c ^ (r % 8), so
        // every group of eight lanes hits eight different banks), then one TMA store per 64
        // columns.  Rows past T lie outside the map and are not written.
        const int y0 = q0 + wq * 32;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          uint32_t pk[2][16];
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t ov[32];
            tmem_ld32_wait(t_o + h * 64 + c2 * 32, ov);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[c2][e] = pack_bf16x2(u2f(ov[2 * e]) * inv_l, u2f(ov[2 * e + 1]) * inv_l);
          }
          const uint32_t buf = stg + (L::STG2 ? h * 32 * 128 : 0);
          if (stg_busy && (!L::STG2 || h == 0)) {  // earlier boxes must have been read out of it
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
          }
#pragma unroll
          for (int c2 = 0; c2 < 2; ++c2)
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(buf + lane * 128 + ((uint32_t(c2 * 4 + q) ^ uint32_t(lane & 7)) << 4), pk[c2][4 * q],
                           pk[c2][4 * q + 1], pk[c2][4 * q + 2], pk[c2][4 * q + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (y0 < p.T) {
            if (lane == 0) {
              if (claimed)
                tma_store_3d_hint(&tmO, buf, h * 64, y0, u.bh, l2_policy_evict_first());
              else
                tma_store_3d(&tmO, buf, h * 64, y0, u.bh);
              bulk_commit_group();
            }
            stg_busy = true;
          }
        }
        if (row < p.T) p.lse[static_cast<size_t>(u.bh) * p.T + row] = (m_run + log2f(l)) * LN2;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(my_o_empty);
    }
    if (stg_busy && lane == 0) bulk_wait_group0();  // this warp's O stores have completed
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  // claimed items: every warp of this CTA is past its last claim; the launch's last CTA to get
  // here zeroes the counter pair for the next launch that takes this slot (a dependent launch
  // reads it only after griddepcontrol.wait, i.e. after this grid has completed)
  if (claimed && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sched + 1, 1) == int(gridDim.x) - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// ever arrives on, so the wait runs out after `timeout_ns` and records the
// timeout in the status word, exactly as a stalled attention launch would.
__global__ void fa_wait_selftest_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const Waiter W{&abort_flag, timeout_ns, &g_status};
  if (threadIdx.x == 0) W.wait(smem_u32(&bar), 0);
}

// Throughput probe of the exponential unit: every thread runs eight independent chains of
// x <- 2^(-x) (one ex2.approx and one FMA each), so the unit, not latency, sets the rate.
__device__ float g_ex2_sink;
__global__ void __launch_bounds__(256) fa_ex2_rate_kernel(int iters) {
  float x[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) x[i] = 0.125f * i + 1e-3f * (threadIdx.x % 32);
  for (int it = 0; it < iters; ++it)
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = ex2_approx(fmaf(x[i], -1.f, 0.f));
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += x[i];
  if (s == 12345.f) g_ex2_sink = s;  // never true (x stays in [0.5, 1]); keeps the chains live
}

cudaError_t measure_ex2_rate(int num_sms, double* ops_per_second, cudaStream_t stream) {
  constexpr int kIters = 4096, kThreads = 256;
  const int grid = num_sms * 4;
  cudaEvent_t a = nullptr, b = nullptr;
  cudaError_t e = cudaEventCreate(&a);
  if (e == cudaSuccess) e = cudaEventCreate(&b);
  if (e == cudaSuccess) {
    fa_ex2_rate_kernel<<<grid, kThreads, 0, stream>>>(kIters);  // warm-up
    cudaEventRecord(a, stream);
    fa_ex2_rate_kernel<<<grid, kThreads, 0, stream>>>(kIters);
    cudaEventRecord(b, stream);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaEventSynchronize(b);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, a, b);
  if (e == cudaSuccess)
    *ops_per_second = static_cast<double>(grid) * kThreads * 8.0 * kIters / (static_cast<double>(ms) * 1e-3);
  if (a) cudaEventDestroy(a);
  if (b) cudaEventDestroy(b);
  return e;
}

// ---------------------------------------------------------------- host side

template <int D, bool PARTIAL, bool F8 = false, bool CLAIM = false>
static cudaError_t launch(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& o,
                          const Params& p, int grid, cudaStream_t stream) {
  using L = Layout<D, F8>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && !attr_set[dev]) {
    e = cudaFuncSetAttribute(fa_fwd_kernel<D, PARTIAL, F8, CLAIM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(L::THREADS);
  cfg.dynamicSmemBytes = L::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, PARTIAL, F8, CLAIM>, q, k, v, o, p);
}

static_assert(Layout<128, true>::SMEM_BYTES <= MAX_SMEM_PER_CTA, "e4m3 layout exceeds the per-CTA limit");

cudaError_t launch_fa_fwd_e4m3(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& vt,
                               const CUtensorMap& o, const Params& p, int grid, cudaStream_t stream) {
  return launch<128, false, true>(q, k, vt, o, p, grid, stream);
}

int fa_fwd_e4m3_smem_bytes() { return Layout<128, true>::SMEM_BYTES; }

// V (rows of 128 e4m3 bytes per key) -> V^T (rows of Tp bytes per channel), keys past T zero.
// A block moves 64 keys x 128 channels through shared memory.  In the load phase thread
// (kg, cg) = (warp, lane) reads keys 8 kg .. 8 kg + 7 at channels 4 cg .. 4 cg + 3, one 4-byte
// word per key (each warp instruction reads one whole 128-byte row of V), turns the 8 x 4
// bytes into 4 channels x 8 keys with byte permutes, and stores one 8-byte word per channel;
// in the store phase thread (c, h) writes channel c's keys 32 h .. 32 h + 31 as two 16-byte
// words.  In shared memory row c holds channel c's 64 keys as eight 8-byte chunks, chunk k at
// position k ^ ((c / 4) % 8), so that each phase's accesses spread over the banks.
__global__ void __launch_bounds__(256) fa_transpose_e4m3_kernel(const uint8_t* __restrict__ v,
                                                                uint8_t* __restrict__ vt, int T, int Tp) {
  __shared__ __align__(16) uint8_t tile[128 * 64];
  // the attention kernel that reads V^T may start its set-up; its griddepcontrol.wait still
  // waits for this whole grid
  pdl_launch_dependents();
  const int bh = blockIdx.y, t0 = blockIdx.x * 64;
  const uint8_t* src = v + static_cast<size_t>(bh) * T * 128;
  uint8_t* dst = vt + static_cast<size_t>(bh) * 128 * Tp;
  {
    const int cg = threadIdx.x % 32, kg = threadIdx.x / 32;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int t = t0 + 8 * kg + i;
      w[i] = t < T ? __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(t) * 128) + cg) : 0u;
    }
    uint32_t ch[4][2];  // [channel 4 cg + j][keys 0-3 | 4-7 of the eight]
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t a01 = __byte_perm(w[4 * h], w[4 * h + 1], 0x5140);  // bytes 0, 1 of both, interleaved
      const uint32_t a23 = __byte_perm(w[4 * h + 2], w[4 * h + 3], 0x5140);
      const uint32_t b01 = __byte_perm(w[4 * h], w[4 * h + 1], 0x7362);  // bytes 2, 3 of both, interleaved
      const uint32_t b23 = __byte_perm(w[4 * h + 2], w[4 * h + 3], 0x7362);
      ch[0][h] = __byte_perm(a01, a23, 0x5410);
      ch[1][h] = __byte_perm(a01, a23, 0x7632);
      ch[2][h] = __byte_perm(b01, b23, 0x5410);
      ch[3][h] = __byte_perm(b01, b23, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint2*>(tile + (4 * cg + j) * 64 + 8 * (kg ^ (cg % 8))) = make_uint2(ch[j][0], ch[j][1]);
  }
  __syncthreads();
  {
    const int c = threadIdx.x / 2, h = threadIdx.x % 2;
    const int sw = (c / 4) % 8;
    uint32_t o[8];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const uint2 x = *reinterpret_cast<const uint2*>(tile + c * 64 + 8 * ((4 * h + m) ^ sw));
      o[2 * m] = x.x;
      o[2 * m + 1] = x.y;
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int tt = t0 + 32 * h + 16 * q;
      if (tt < Tp)  // Tp is a multiple of 16, so the whole 16-byte word is inside
        *reinterpret_cast<uint4*>(dst + static_cast<size_t>(c) * Tp + tt) =
            make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
  }
}

cudaError_t launch_transpose_e4m3(const void* v, void* vt, int BH, int T, int Tp, cudaStream_t stream) {
  const dim3 grid((Tp + 63) / 64, BH);
  fa_transpose_e4m3_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t*>(v), static_cast<uint8_t*>(vt),
                                                      T, Tp);
  return cudaGetLastError();
}

cudaError_t launch_fa_fwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const Params& p, int grid, cudaStream_t stream) {
  if (d == 64) return launch<64, false>(q, k, v, o, p, grid, stream);
  if (p.sched) return launch<128, false, false, true>(q, k, v, o, p, grid, stream);
  return launch<128, false>(q, k, v, o, p, grid, stream);
}

// (the partial form writes fp32 rows directly and never uses the output map; q stands in for it)
cudaError_t launch_fa_fwd_partial(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const Params& p, int grid, cudaStream_t stream) {
  if (d == 64) return launch<64, true>(q, k, v, q, p, grid, stream);
  return launch<128, true>(q, k, v, q, p, grid, stream);
}

// ---------------------------------------------------------------- fixed scratch (no allocation)
// Scratch for fa_fwd_splitkv_noalloc: a device global, so the library never
// allocates for that entry point.  Every device that loads the library holds
// one copy of it until the process exits.  In host code `g_noalloc_scratch`
// names a host-side stand-in, not device memory: its device address comes from
// cudaGetSymbolAddress, looked up with the device current.  The address belongs
// to a CUDA context (a cudaDeviceReset ends the primary context; a driver-API
// caller may make another context current), so the cache is keyed on the
// context's process-unique id and the address is looked up again in a context
// not seen before.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Counter pairs of the launches whose work items are claimed at run time (see claimed_item):
// one pair every kSchedStride ints (a 128-byte line each), zero at load time, and zeroed again
// by the last CTA of every launch that used the pair.
static __device__ __align__(128) int g_sched[kSchedSlots * kSchedStride];

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Device address of the __device__ variable whose host shadow is `symbol`, in the current CUDA
// context: looked up with cudaGetSymbolAddress on the first call in each context, then cached
// by the context's process-unique id (up to 64 contexts, the oldest replaced after that).  One
// cache per Tag.
template <int Tag>
cudaError_t context_symbol_address(const void* symbol, void** out) {
  struct Entry {
    unsigned long long ctx_id;
    void* addr;
  };
  static Entry cache[64] = {};
  static int used = 0, next = 0;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!get_current || !get_id) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return cudaErrorNotSupported;
    get_id = reinterpret_cast<CtxGetIdFn>(f);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) {
    // no context current yet: the symbol lookup below makes the device's primary context current
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess) return e;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  }
  for (int i = 0; i < used; ++i)
    if (cache[i].ctx_id == id) {
      *out = cache[i].addr;
      return cudaSuccess;
    }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, symbol);  // in the current context
  if (e != cudaSuccess) return e;
  Entry& slot = used < 64 ? cache[used++] : cache[next++ % 64];
  slot.ctx_id = id;
  slot.addr = p;
  *out = p;
  return cudaSuccess;
}
}  // namespace

cudaError_t noalloc_scratch_address(void** out) {
  return context_symbol_address<0>(static_cast<const void*>(g_noalloc_scratch), out);
}

cudaError_t sched_counters_address(int** out) {
  void* p = nullptr;
  const cudaError_t e = context_symbol_address<1>(static_cast<const void*>(g_sched), &p);
  *out = static_cast<int*>(p);
  return e;
}

cudaError_t launch_wait_selftest(unsigned long long timeout_ns, cudaStream_t stream) {
  fa_wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

int fa_fwd_smem_bytes(int d) { return d == 64 ? Layout<64>::SMEM_BYTES : Layout<128>::SMEM_BYTES; }
int fa_fwd_threads(int d) { return d == 64 ? Layout<64>::THREADS : Layout<128>::THREADS; }
int fa_fwd_rows_per_unit() { return 2 * BM; }

cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* out) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace fa
