// Internal interface between the C-ABI layer (fa_api.cu) and the kernel (fa_kernel.cu).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fa {

struct Params {
  __nv_bfloat16* o;           // (B*H, T, d) bf16 output
  float* lse;                 // (B*H, T) fp32 output
  int BH;                     // batch * query heads
  int H;                      // query heads per batch entry
  int group;                  // query heads per K/V head (1 = multi-head; H / H_kv with grouped K/V)
  int Hkv;                    // K/V heads per batch entry (H / group)
  // paged K/V (block_table != nullptr): K and V are pools of 128-key pages, (num_pages, Hkv, 128, d);
  // key tile j of batch entry b is page block_table[b * max_pages + j]
  const int* block_table;
  int max_pages;
  int num_pages;
  int T;                      // sequence length
  int causal;                 // 0 or 1
  int nqb;                    // 256-row query blocks per head: ceil(T / 256)
  int nk;                     // 128-key tiles per head: ceil(T / 128)
  int num_units;              // BH * nqb
  int unit_div;               // causal: BH (units listed band by band); otherwise nqb (head by head)
  float scale_log2;           // scale * log2(e) (e4m3: times the Q and K scales)
  float v_descale;            // 1, or the scale of e4m3 V (the real value is the byte's value times it)
  unsigned long long timeout_ns;  // bound on every in-kernel wait
  // split-KV (partial) launches only: each row's key tiles are cut into
  // num_splits ranges of split_tiles tiles; unit w -> (band, split, bh)
  int num_splits;             // 1 for a plain launch
  int split_tiles;            // key tiles per split (>= 1)
  float* opart;               // [num_splits][BH*T][d] fp32 partial outputs (normalised)
  float* lsepart;             // [num_splits][BH*T] fp32 partial LSE (natural log)
  int* counters;              // [BH][ngroups] splits finished per 32-row group (zero at launch)
  int ngroups;                // ceil(T / 32)
  // order of the work items (unsplit causal launches): head_group > 0 lists the units band by
  // band within groups of head_group heads (head_group divides BH), so that the CTAs running
  // at one time read the K / V of a few heads, except the lightest tail_bands bands, which
  // follow band by band over all heads (short units last, whatever their head); sched !=
  // nullptr hands the items out in that order from a device-wide counter pair (sched[0]: items
  // claimed after each CTA's first, sched[1]: CTAs finished; both zero at launch, and the
  // launch's last CTA zeroes them again)
  // non-causal unsplit e4m3 launches: the last `halves` work items are the two query tiles of
  // the units of a part-empty last round of the grid, one tile per item (0: none)
  int halves;
  int head_group;
  int tail_bands;             // head_group > 0: the lightest tail_bands bands of every head come last, band by band
  int* sched;
};

// Rows per box of the output tensor map `o` (bf16 (d, T, B*H), 128-byte swizzle): each
// softmax warp writes its 32 rows of a query tile with one TMA store per 64 columns.
constexpr int kOutBoxRows = 32;
cudaError_t launch_fa_fwd(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o, const Params& p, int grid, cudaStream_t stream);
// e4m3 Q, K and a transposed e4m3 V ((B*H, d, Tp) bytes), d = 128; bf16 O as above.
cudaError_t launch_fa_fwd_e4m3(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& vt,
                               const CUtensorMap& o, const Params& p, int grid, cudaStream_t stream);
// V (B*H, T, 128) e4m3 -> V^T (B*H, 128, Tp) with keys Tp > T zero (Tp = T rounded up to 16).
cudaError_t launch_transpose_e4m3(const void* v, void* vt, int BH, int T, int Tp, cudaStream_t stream);
int fa_fwd_e4m3_smem_bytes();
// The same kernel over (query block, key split) units: each split writes its partials
// (p.opart, p.lsepart), and the last split of every 32-row group to finish merges the group
// into O and LSE (p.counters must be zero at launch).
cudaError_t launch_fa_fwd_partial(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                  const Params& p, int grid, cudaStream_t stream);
int fa_fwd_smem_bytes(int d);
int fa_fwd_threads(int d);
int fa_fwd_rows_per_unit();
cudaError_t read_and_clear_status(cudaStream_t stream, unsigned int* out);
cudaError_t launch_wait_selftest(unsigned long long timeout_ns, cudaStream_t stream);
// ex2.approx operations per second of the whole device (two launches of a probe kernel;
// waits for the second).
cudaError_t measure_ex2_rate(int num_sms, double* ops_per_second, cudaStream_t stream);

// Size of the fixed device scratch behind fa_fwd_splitkv_noalloc (32 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
// Device address of that scratch in the current CUDA context; looked up on the first
// call in each context (cudaGetSymbolAddress), then cached by the context's unique id.
cudaError_t noalloc_scratch_address(void** out);

// Counter pairs for launches whose work items are claimed at run time: kSchedSlots pairs, one
// every kSchedStride ints; a launch takes the next slot in turn.  Returns the device address of
// the first pair in the current CUDA context (looked up once per context, like the scratch).
constexpr int kSchedSlots = 64;
constexpr int kSchedStride = 32;
cudaError_t sched_counters_address(int** out);

// ---------------------------------------------------------------- backward pass (fa_bwd.cu)

struct BwdParams {
  const __nv_bfloat16* o;     // (B*H, T, d) forward output
  const __nv_bfloat16* dout;  // (B*H, T, d) upstream gradient
  const float* lse;           // (B*H, T) forward log-sum-exp (natural log)
  // workspace, rows padded to Tp per head: D_t = sum_c dO_tc O_tc (0 past T) and
  // LSE_t * log2 e (+inf past T, so that P = 0 there)
  float* drow;                // (B*H, Tp)
  float* lse2;                // (B*H, Tp)
  __nv_bfloat16* dq;          // (B*H, T, d) outputs
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int BH, T, causal;
  int nt;                     // 128-row tiles per head: ceil(T / 128)
  int Tp;                     // nt * 128
  int num_units;              // BH * nt
  float scale;                // softmax scale
  float scale_log2;           // scale * log2(e) (e4m3: times the Q and K scales)
  float v_descale;            // 1, or the scale of e4m3 V (the real value is the byte's value times it)
  unsigned long long timeout_ns;
};

// D_t = sum_c dO_tc O_tc and LSE_t * log2 e for every row of the padded workspace.
// dQ: one CTA per SM, units (head, 128-row query tile), key tiles streamed.
// Gradient outputs (dQ, dK, dV: bf16 (d, T, B*H), no swizzle) are written in boxes of
// kGradBoxRows rows x kGradBoxCols columns: a row warp's 32 rows and 32 of its columns.
constexpr int kGradBoxRows = 32;
constexpr int kGradBoxCols = 32;
// g1, g2: the output maps (dQ kernel: dQ, and g2 unused; dK/dV kernel: dV, dK).
cudaError_t launch_bwd_dq(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& dout, const CUtensorMap& g1, const CUtensorMap& g2, const BwdParams& p,
                          int grid, cudaStream_t stream);
// dK, dV: one CTA per SM, units (head, 128-key tile), query tiles streamed.
cudaError_t launch_bwd_dkdv(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const CUtensorMap& dout, const CUtensorMap& g1, const CUtensorMap& g2,
                            const BwdParams& p, int grid, cudaStream_t stream);
int fa_bwd_smem_bytes(int d);
// Reads and clears the backward kernels' device status word (bit 0: a wait ran out).
cudaError_t read_and_clear_bwd_status(cudaStream_t stream, unsigned int* out);

}  // namespace fa
