/*
 * fa.h - FlashAttention forward pass for one GB300 (sm_103), C ABI.
 *
 * The operation (exact attention, tiled, with the online softmax):
 *   for every batch b, head h and query row i,
 *     s_ij  = scale * sum_c Q[b,h,i,c] * K[b,h,j,c]      for visible keys j
 *     O[b,h,i,:] = sum_j softmax_j(s_i.) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(s_ij)                      (natural log)
 *   where key j is visible to query i when causal == 0, or when j <= i if
 *   causal == 1.
 * Sources: "Flash Attention, tiled: exact attention without the T x T HBM
 * matrix", sections "Ordinary causal attention" (S = Q K^T / sqrt(d), causal
 * mask, softmax, Y = P V) and "From the example to tiled GPU work" (the
 * per-tile procedure and its outputs: the output and limited softmax state);
 * "FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
 * section "Step 3: FlashAttention, one fused kernel"; "FlashAttention: the
 * IO-aware Attention Kernel", section 3.2 (the online-softmax recurrence).
 * The LSE is not defined on the pages; this library writes the natural log of
 * the softmax denominator of the scaled, masked scores.
 *
 * Memory layout: Q, K, V and O are dense, contiguous, row-major bf16 tensors
 * of shape (B, H, T, d) (d fastest).  LSE is a dense fp32 tensor (B, H, T).
 *
 * Ownership: the caller owns every buffer; all five pointers are device
 * memory of the current CUDA device.  The library allocates no memory.  O
 * and LSE must not overlap Q, K, V or each other.
 *
 * Shared state: a causal d = 128 fa_fwd whose K and V exceed 96 MB over all
 * heads hands its work units out at run time from one of 64 counter pairs
 * that the library holds in device memory (a launch takes the next pair in
 * turn; its last block zeroes the pair again).  Such launches may run
 * concurrently on unordered streams as long as fewer than 64 of them are in
 * flight at once; a CUDA graph that contains one must not be replayed on two
 * streams at the same time (both replays would share its pair).  The first
 * such call in a CUDA context looks the pairs' address up (make it before a
 * stream capture).  Every other call keeps no state between calls.
 *
 * Execution: fa_fwd only validates its arguments and enqueues one kernel on
 * `stream`; it does not synchronise.  O and LSE are complete once the stream
 * has reached that point.
 *
 * Errors: validation happens before anything is enqueued and returns a status
 * code other than FA_OK; nothing is written in that case.  Every wait inside
 * the kernel is bounded in time: if one runs out, the kernel stops early,
 * records FA_ERR_DEVICE_TIMEOUT in a device status word and returns, leaving
 * O and LSE incomplete; fa_device_status() reads (and clears) that word.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <cuda_runtime.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL_PTR = 1,              /* a required pointer is NULL */
  FA_ERR_MISALIGNED = 2,            /* a pointer is not 16-byte aligned */
  FA_ERR_BAD_SHAPE = 3,             /* B, H or T < 1, or a size too large to index */
  FA_ERR_UNSUPPORTED_HEAD_DIM = 4,  /* d is not 64 or 128 */
  FA_ERR_BAD_SCALE = 5,             /* scale is not finite and > 0 */
  FA_ERR_NO_DEVICE_SUPPORT = 6,     /* the current device is not sm_103 */
  FA_ERR_LAUNCH = 7,                /* the CUDA runtime refused the launch */
  FA_ERR_DEVICE_TIMEOUT = 8,        /* a bounded in-kernel wait ran out */
  FA_ERR_BAD_ARG = 9,               /* an argument is out of range (causal not 0 or 1, a self-test timeout) */
  FA_ERR_BAD_POINTER = 10,          /* a pointer is not device memory, or its allocation is too small */
  FA_ERR_ALIAS = 11,                /* O or LSE overlaps an input or each other */
  FA_ERR_CUDA = 12,                 /* a CUDA runtime or driver query failed */
  FA_ERR_WORKSPACE = 13,            /* a workspace is missing or smaller than its *_workspace_bytes() */
  FA_ERR_BAD_PAGE = 14              /* (device) a block-table entry was outside the page pool */
} fa_status;

/* Largest number of key splits fa_fwd_splitkv accepts. */
#define FA_MAX_SPLITS 256

/*
 * Attention forward.
 *   q, k, v : bf16 (B, H, T, d), contiguous, read only.
 *   o       : bf16 (B, H, T, d), contiguous, written: O = softmax(scale Q K^T [+ mask]) V.
 *   lse     : fp32 (B, H, T), written: natural-log LSE of each row's scaled scores.
 *   B, H, T : batch, heads, sequence length; each >= 1; B*H <= 2^31-1, T <= 2^30.
 *   d       : head size, 64 or 128.
 *   causal  : 1 = query i sees keys j <= i; 0 = every key.
 *   scale   : score multiplier, finite and > 0 (usually 1/sqrt(d)).
 *   stream  : CUDA stream the kernel is enqueued on (0 = legacy default).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int T, int d, int causal, float scale,
                 cudaStream_t stream);

/*
 * Attention forward with grouped keys and values: H query heads share Hkv K/V
 * heads, query head h reading K/V head h / (H / Hkv) of the same batch entry
 * ("FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
 * section "Step 4: decoding is a different problem": Llama 3.1 8B shares each
 * K/V head among 4 query heads).  Per query head the result is exactly the
 * attention fa_fwd computes with that head's K and V.
 *   q, o   : (B, H, T, d) bf16, as for fa_fwd.
 *   k, v   : (B, Hkv, T, d) bf16, contiguous, d fastest.
 *   lse    : (B, H, T) fp32.
 *   Hkv    : 1 <= Hkv <= H with H % Hkv == 0 (Hkv == H is fa_fwd).
 *   the rest as for fa_fwd.
 * Errors: as fa_fwd; FA_ERR_BAD_SHAPE also when Hkv does not divide H; the
 * pointer range checks use the K/V size B * Hkv * T * d.
 */
fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Hkv, int T, int d, int causal, float scale,
                     cudaStream_t stream);

/*
 * Attention forward with the keys of every row split into ranges that run as
 * separate work units (Flash-Decoding: "FlashAttention and Fused Kernels:
 * Attention Without the n x n Matrix", section "Flash-Decoding: split the
 * cache, not the queries").  Each unit writes its range's normalised output
 * (fp32) and log-sum-exp into `workspace`; in the same launch, the last split
 * of every group of 32 query rows to finish merges that group, weighting each
 * split by its log-sum-exp (a counter per group in the workspace, cleared by
 * an asynchronous memset on `stream` before the launch).  O and LSE are the
 * same quantities fa_fwd computes (up to rounding).
 *   q .. scale, stream : as for fa_fwd.
 *   num_splits : 1 .. FA_MAX_SPLITS; the keys (ceil(T / 128) tiles of 128) are
 *                cut into ceil(tiles / ceil(tiles / num_splits)) ranges of
 *                equal tile count.  0 chooses the count: the library replays
 *                the persistent grid's static schedule on the host for 1 .. 16
 *                splits (costs counted in 128-key steps, with a fixed cost per
 *                unit and per merge) and takes the count with the shortest
 *                busiest SM, if it beats one split by at least 10 %.  When the
 *                count comes to one range, the call is fa_fwd (no partials,
 *                no merge, the workspace untouched; the result is bit-identical
 *                to fa_fwd's).
 *   workspace  : caller-owned device memory of at least
 *                fa_fwd_splitkv_workspace_bytes(B, H, T, d, num_splits) bytes,
 *                16-byte aligned, not overlapping any tensor argument.  Its
 *                contents are scratch: overwritten, never read before written
 *                (the counters are cleared by the call itself).
 * Errors: as fa_fwd, plus FA_ERR_BAD_ARG (num_splits out of range) and
 * FA_ERR_WORKSPACE (NULL or too small a workspace).
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int T, int d, int causal, float scale, int num_splits,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Forward pass with K and V in a pool of fixed-size pages ("FlashAttention and
 * Fused Kernels: Attention Without the n x n Matrix", section "Paged caches":
 * the key/value cache is kept in fixed-size blocks found through a block
 * table).  Pages hold 128 keys.  Key t of batch entry b (and K/V head g) is row
 * t % 128 of page block_table[b * max_pages + t / 128] of head g.  The result is
 * exactly fa_fwd_gqa's on the K and V those pages hold.
 *   q, o, lse   : as for fa_fwd_gqa ((B, H, T, d) bf16, (B, H, T) fp32).
 *   k_pages,
 *   v_pages     : (num_pages, Hkv, 128, d) bf16, contiguous, d fastest.  Rows of
 *                 the last page past T must hold finite values (they are masked
 *                 out, but V's rows are still multiplied by zero weights).
 *   block_table : (B, max_pages) int32, device memory; entries 0 .. ceil(T/128)-1
 *                 of each row are read.  An entry outside [0, num_pages) makes
 *                 that page read as zeros and sets FA_ERR_BAD_PAGE in the device
 *                 status word (fa_device_status).
 *   Hkv, the rest as for fa_fwd_gqa; max_pages >= ceil(T / 128), num_pages >= 1.
 * Errors: as fa_fwd_gqa; FA_ERR_NULL_PTR for a NULL block table,
 * FA_ERR_BAD_SHAPE for max_pages < ceil(T / 128) or num_pages < 1.
 */
fa_status fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table,
                       void* o, float* lse, int B, int H, int Hkv, int T, int d, int causal, float scale,
                       int num_pages, int max_pages, cudaStream_t stream);

/*
 * Forward pass with 8-bit inputs (FlashAttention-3's FP8 mode, "FlashAttention
 * and Fused Kernels: Attention Without the n x n Matrix", section "Four
 * generations of FlashAttention").  Q, K and V are e4m3 bytes (OCP FP8: sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448, 0x7F / 0xFF
 * NaN) with one scale per tensor: the real value of a byte is its e4m3 value
 * times q_descale, k_descale or v_descale.  Both matrix products run in e4m3
 * (tcgen05.mma kind::f8f6f4, fp32 accumulation): P is rounded to e4m3 for the
 * P V product and O is divided by the sum of those rounded weights, so each
 * output row is still a convex combination of value rows; LSE uses the fp32
 * weights.  O is bf16, LSE fp32, as for fa_fwd.
 *   q, k, v    : (B, H, T, 128) e4m3 bytes, contiguous; d must be 128.
 *   o, lse     : as for fa_fwd.
 *   workspace  : device memory of at least fa_fwd_fp8_workspace_bytes(B, H, T, d)
 *                bytes, 16-byte aligned; it receives V transposed to (B, H, 128,
 *                T rounded up to 16), keys past T zero.  Nothing in it needs to be
 *                set beforehand.
 * Two kernels run in order on `stream`: the transpose of V, then attention.
 * Errors: as fa_fwd; FA_ERR_UNSUPPORTED_HEAD_DIM for d != 128, FA_ERR_BAD_SCALE
 * for a descale that is not finite and > 0, FA_ERR_WORKSPACE, FA_ERR_ALIAS when
 * O, LSE or the workspace overlaps an input or each other, FA_ERR_BAD_SHAPE when
 * B * H > 65535.
 */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int T, int d, int causal, float scale,
                     float q_descale, float k_descale, float v_descale,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace fa_fwd_fp8 needs: B * H * 128 * (T rounded up to 16) bytes, rounded up to 256; 0 if d != 128. */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int T, int d);

/*
 * Backward pass: the gradients of sum(dO * O) with respect to Q, K and V
 * ("FlashAttention and Fused Kernels: Attention Without the n x n Matrix",
 * section "Training: recompute instead of store": only O and the per-row
 * log-sum-exp are kept from the forward pass; S and P are recomputed tile by
 * tile).  With P = exp(scale Q K^T - LSE) (masked when causal) and
 * D_t = sum_c dO_tc O_tc:
 *   dV = P^T dO,   dS = P * (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q.
 *   q, k, v, o, dout : (B, H, T, d) bf16, contiguous, d fastest; o and lse are
 *                      what fa_fwd returned for q, k, v, causal and scale.
 *   lse              : (B, H, T) fp32, natural log.
 *   dq, dk, dv       : (B, H, T, d) bf16 outputs, overwritten.
 *   workspace        : device memory of at least fa_bwd_workspace_bytes(B, H, T)
 *                      bytes, 16-byte aligned (it receives D and LSE * log2 e per
 *                      row; nothing in it needs to be set beforehand).
 * Two kernels run in order on `stream`: dQ (one unit per 128-row query tile,
 * which also writes D and LSE * log2 e into the workspace), then dK and dV (one
 * unit per 128-key tile, reading them); no output is accumulated across units,
 * so the result does not depend on scheduling.
 * Errors: as fa_fwd for the shared arguments; FA_ERR_NULL_PTR / FA_ERR_MISALIGNED
 * / FA_ERR_BAD_POINTER for dout, dq, dk, dv; FA_ERR_WORKSPACE for a NULL or too
 * small workspace; FA_ERR_ALIAS when an output or the workspace overlaps an input
 * or another output; FA_ERR_BAD_SHAPE when B * H * (T rounded up to 128) exceeds
 * 2^31 - 1.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const void* dout, void* dq, void* dk, void* dv,
                 int B, int H, int T, int d, int causal, float scale,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace fa_bwd needs: 2 * B * H * Tp * 4 bytes (Tp = T rounded up to 128), rounded up
 * to 256; 0 for sizes out of range. */
size_t fa_bwd_workspace_bytes(int B, int H, int T);

/* Size of the fixed device scratch fa_fwd_splitkv_noalloc uses (32 MiB). */
#define FA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * fa_fwd_splitkv without a workspace argument and without any allocation.
 * (Not part of the method described on the pages; an interface addition.)
 *
 * For callers that cannot allocate device memory while they run: code whose
 * device memory is owned by a framework's pool or a fixed budget, plugins
 * that must not call the CUDA allocator, or hosts where an allocation at that
 * point would block or fail.  The split partials go to a fixed scratch array
 * of FA_NOALLOC_SCRATCH_BYTES that the library holds on every device it is
 * loaded on (for the life of the process); nothing calls cudaMalloc, cudaFree
 * or any other allocating routine.
 *
 * Arguments and results are those of fa_fwd_splitkv minus the workspace.
 * Limits and behaviour:
 *   - the scratch that the call needs (fa_fwd_splitkv_workspace_bytes for the
 *     split count it uses; num_splits = 0 chooses it as fa_fwd_splitkv does)
 *     must not exceed FA_NOALLOC_SCRATCH_BYTES, else FA_ERR_WORKSPACE and
 *     nothing runs;
 *   - the first call on each device looks up the scratch's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture on that device.  The
 *     address belongs to the CUDA context that was current: after a
 *     cudaDeviceReset, or when a driver-API caller makes another context
 *     current, the next call looks it up again (the cache is keyed on the
 *     context's unique id), and that call too should precede any capture;
 *   - every call on a device shares the one scratch array, which keeps what
 *     the last call left there.  The only part that must start at zero, the
 *     merge counters, is cleared by each call (an asynchronous memset on
 *     `stream`); every partial is written before the merge reads it.  Calls whose
 *     kernels overlap on the GPU (different streams without ordering between
 *     them) race on the scratch and give wrong results; order them.
 */
fa_status fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int T, int d, int causal, float scale, int num_splits,
                                 cudaStream_t stream);

/*
 * Workspace bytes fa_fwd_splitkv needs (0 for invalid sizes):
 * num_splits * B*H*T * (d + 1) * 4 + B*H*ceil(T / 32) * 4, rounded up to 256.
 * num_splits = 0: the size for the count the call would choose on the current
 * device (the larger of the causal and non-causal choices).
 */
size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int T, int d, int num_splits);

/*
 * Number of key ranges fa_fwd_splitkv (and fa_fwd_splitkv_noalloc) would use
 * for these arguments on the current device: num_splits = 0 resolved as
 * described at fa_fwd_splitkv, then ceil(tiles / ceil(tiles / num_splits))
 * with tiles = ceil(T / 128).  1 means the call runs fa_fwd.  Returns -1 for
 * invalid sizes or num_splits, or when no CUDA device is current (num_splits
 * = 0 only).  No device work.
 */
int fa_fwd_splitkv_count(int B, int H, int T, int d, int causal, int num_splits);

/* A static, human-readable name for a status code. */
const char* fa_status_string(fa_status s);

/*
 * Reads and clears the device status word that kernels of this library set
 * when a bounded wait runs out.  Synchronises `stream` first.  *out receives
 * FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_BAD_PAGE (fa_fwd_paged met a page
 * outside its pool; reported first).  Returns FA_ERR_CUDA if the copy fails.
 */
fa_status fa_device_status(cudaStream_t stream, int* out);

/*
 * The launch the library would make for these sizes: persistent CTAs, threads
 * per CTA and dynamic shared memory bytes.  For tools and tests; it validates
 * d and the sizes like fa_fwd but needs no device pointers.
 */
fa_status fa_fwd_launch_shape(int B, int H, int T, int d, int causal, int num_sms,
                              int* grid, int* threads, int* smem_bytes);

/*
 * Self-test of the in-kernel wait bound (no attention involved): enqueues a
 * one-block kernel whose single waiting thread waits on a barrier that nothing
 * ever completes, so the wait runs out after `timeout_us` microseconds
 * (1 .. 2,000,000) and the kernel returns, recording FA_ERR_DEVICE_TIMEOUT in
 * the device status word that fa_device_status() reads.  Nothing faults or
 * hangs; the context stays usable.  Returns FA_ERR_BAD_ARG for an
 * out-of-range timeout, FA_ERR_NO_DEVICE_SUPPORT off sm_103, FA_ERR_LAUNCH if
 * the launch is refused.
 */
fa_status fa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream);

/*
 * Throughput of the exponential unit the softmax uses (ex2.approx.ftz.f32),
 * measured on the current device: the whole-device rate in operations per
 * second, for the SFU-limited attention rate (one exponential per unmasked
 * score against 4 d tensor FLOPs; "Flash Attention, tiled", the GPU cost
 * model of exp vs matmul).  Enqueues two short probe launches on `stream` and
 * waits for them (the call is synchronous).  FA_ERR_NULL_PTR for a NULL
 * `ops_per_second`, FA_ERR_NO_DEVICE_SUPPORT off sm_103, FA_ERR_LAUNCH if a
 * launch or the timing fails.
 */
fa_status fa_ex2_rate(double* ops_per_second, cudaStream_t stream);

/* Library version, e.g. "0.1.0". */
const char* fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
