// C ABI of the attention library: argument validation, TMA descriptors and the launch.
// The operation and its contract are documented in include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <vector>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_kernel.h"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
using PointerAttrsFn = CUresult (*)(unsigned int, CUpointer_attribute*, void**, CUdeviceptr);

struct DriverFns {
  EncodeTiledFn encode_tiled = nullptr;
  PointerAttrsFn pointer_attrs = nullptr;
};

// Driver entry points, resolved through the runtime so the library needs no link to libcuda.
const DriverFns& driver_fns() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.encode_tiled = reinterpret_cast<EncodeTiledFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttributes", &f, 7000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.pointer_attrs = reinterpret_cast<PointerAttrsFn>(f);
  });
  return fns;
}

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s bound on any in-kernel wait
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  int checked = 0;  // 0 unknown, 1 supported, -1 unsupported
  int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// The current device must be an sm_103 part; caches its SM count.
fa_status current_device(int* dev_out, int* num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE_SUPPORT;
  }
  if (dev >= kMaxDevices) return FA_ERR_NO_DEVICE_SUPPORT;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo& info = g_devices[dev];
  if (info.checked == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    if (major == 10 && minor == 3) {
      if (cudaSetDevice(dev) != cudaSuccess) {  // makes the primary context current
        cudaGetLastError();
        return FA_ERR_CUDA;
      }
      info.num_sms = sms;
      info.checked = 1;
    } else {
      info.checked = -1;
    }
  }
  if (info.checked < 0) return FA_ERR_NO_DEVICE_SUPPORT;
  *dev_out = dev;
  *num_sms = info.num_sms;
  return FA_OK;
}

// `p` must be device memory of device `dev`, and [p, p + bytes) must lie in one
// allocation.  One driver query per pointer (memory type, ordinal, range).
fa_status check_device_range(const void* p, size_t bytes, int dev) {
  const DriverFns& fns = driver_fns();
  if (!fns.pointer_attrs) return FA_ERR_CUDA;
  const CUdeviceptr dp = reinterpret_cast<CUdeviceptr>(p);
  unsigned int mem_type = 0;
  int ordinal = -1;
  CUdeviceptr base = 0;
  size_t size = 0;
  CUpointer_attribute attrs[4] = {CU_POINTER_ATTRIBUTE_MEMORY_TYPE, CU_POINTER_ATTRIBUTE_DEVICE_ORDINAL,
                                  CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, CU_POINTER_ATTRIBUTE_RANGE_SIZE};
  void* data[4] = {&mem_type, &ordinal, &base, &size};
  // an address the driver does not know leaves the values untouched (type 0) or fails
  if (fns.pointer_attrs(4, attrs, data, dp) != CUDA_SUCCESS) return FA_ERR_BAD_POINTER;
  if (mem_type != CU_MEMORYTYPE_DEVICE || ordinal != dev || size == 0) return FA_ERR_BAD_POINTER;
  if (dp < base || dp - base > size || bytes > size - (dp - base)) return FA_ERR_BAD_POINTER;
  return FA_OK;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Checks that need no device: pointers, sizes, head size, scale, mask flag, alignment.
fa_status validate_host(const void* q, const void* k, const void* v, const void* o, const void* lse, int B, int H,
                        int T, int d, int causal, float scale) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL_PTR;
  if (B < 1 || H < 1 || T < 1) return FA_ERR_BAD_SHAPE;
  if (static_cast<long long>(B) * H > INT_MAX || T > (1 << 30)) return FA_ERR_BAD_SHAPE;
  const long long bh = static_cast<long long>(B) * H;
  const long long nqb = (T + 255) / 256;
  if (bh * nqb > INT_MAX) return FA_ERR_BAD_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_HEAD_DIM;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_SCALE;
  if (causal != 0 && causal != 1) return FA_ERR_BAD_ARG;
  for (const void* p : {q, k, v, o, lse})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return FA_ERR_MISALIGNED;
  return FA_OK;
}

// 3-D view (inner, rows, B*H) of a contiguous tensor: a box (box_bytes of the inner
// dimension x box_rows rows x 1) never crosses from one head into the next, rows past
// `rows` read as zeros and are not written.  bf16 (d, T, B*H) views, or byte views for
// e4m3 tensors.  128-byte boxes use the 128-byte swizzle, narrower ones none.
bool encode_tensor_map(CUtensorMap* map, const void* base, int BH, int rows, int inner, bool bytes, int box_rows,
                       int box_bytes) {
  const DriverFns& fns = driver_fns();
  if (!fns.encode_tiled) return false;
  const cuuint64_t es = bytes ? 1 : 2;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * es, static_cast<cuuint64_t>(rows) * inner * es};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_bytes / es), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  return fns.encode_tiled(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded descriptors, reused when the same tensor comes back (encoding reads no
// memory, so a cached descriptor is exactly what encoding again would give).
struct MapCacheEntry {
  const void* base = nullptr;
  int BH = 0, T = 0, d = 0, box_rows = 0, box_bytes = 0;
  bool bytes = false;
  CUtensorMap map;
};
constexpr int kMapCache = 16;
MapCacheEntry g_map_cache[kMapCache];
std::mutex g_map_mu;

bool make_tensor_map(CUtensorMap* map, const void* base, int BH, int T, int d, bool bytes = false,
                     int box_rows = 128, int box_bytes = 128) {
  const size_t slot = ((reinterpret_cast<uintptr_t>(base) >> 8) + (box_rows == 128 ? 0 : 1)) % kMapCache;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapCacheEntry& e = g_map_cache[slot];
  if (e.base == base && e.BH == BH && e.T == T && e.d == d && e.bytes == bytes && e.box_rows == box_rows &&
      e.box_bytes == box_bytes) {
    *map = e.map;
    return true;
  }
  if (!encode_tensor_map(map, base, BH, T, d, bytes, box_rows, box_bytes)) return false;
  e.base = base;
  e.BH = BH;
  e.T = T;
  e.d = d;
  e.box_rows = box_rows;
  e.box_bytes = box_bytes;
  e.bytes = bytes;
  e.map = *map;
  return true;
}

struct Prepared {
  fa::Params p{};
  CUtensorMap tq, tk, tv, to;  // to: the bf16 output O, written in boxes of 32 rows
  int dev = 0, num_sms = 0;
};

// Work items of an unsplit e4m3 launch of `units` units (256 query rows each) on num_sms
// persistent CTAs.  Non-causal units all cost the same, so a last round that leaves SMs idle
// (units not a multiple of the SMs) is worked in single query tiles, one per item, when twice its
// units still fit on the SMs and the units are at least 8 K/V steps long.  In the e4m3 kernel,
// where each query tile has an MMA warp of its own, a one-tile item takes about half a unit's
// time (+5.6 % on 32 heads at T = 4096); in the bf16 d = 128 kernel, whose one MMA warp overlaps
// the two tiles' products with each other's softmax, a one-tile item took nearly a unit's time
// (+0.6 %), and decoding one-tile items cost the d = 64 kernel registers (-0.7 %), so those
// kernels keep whole units.  Causal units are balanced by the longest-first order instead.
// Returns the item count; *halves = the one-tile items at its end.
long long work_items_e4m3(long long units, int nk, int causal, int num_sms, int* halves) {
  *halves = 0;
  if (causal || nk < 8 || num_sms < 1) return units;
  const long long full = units / num_sms * num_sms, tail = units - full;
  if (tail == 0 || 2 * tail > num_sms) return units;
  *halves = static_cast<int>(2 * tail);
  return full + 2 * tail;
}

// Validation shared by the entry points, then the TMA descriptors and the
// launch parameters of a plain (unsplit) launch.  K and V hold Hkv heads per
// batch entry; H query heads share them in groups of H / Hkv (Hkv == H: one K/V
// head per query head).
fa_status prepare(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int T,
                  int d, int causal, float scale, Prepared* pr) {
  fa_status st = validate_host(q, k, v, o, lse, B, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_BAD_SHAPE;
  if ((st = current_device(&pr->dev, &pr->num_sms)) != FA_OK) return st;
  const int BH = B * H, BHkv = B * Hkv;
  const size_t q_bytes = static_cast<size_t>(BH) * T * d * 2;
  const size_t kv_bytes = static_cast<size_t>(BHkv) * T * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * T * 4;
  for (const void* x : {q, static_cast<const void*>(o)})
    if ((st = check_device_range(x, q_bytes, pr->dev)) != FA_OK) return st;
  for (const void* x : {k, v})
    if ((st = check_device_range(x, kv_bytes, pr->dev)) != FA_OK) return st;
  if ((st = check_device_range(lse, lse_bytes, pr->dev)) != FA_OK) return st;
  const struct {
    const void* p;
    size_t n;
  } inputs[3] = {{q, q_bytes}, {k, kv_bytes}, {v, kv_bytes}};
  for (const auto& in : inputs)
    if (overlaps(o, q_bytes, in.p, in.n) || overlaps(lse, lse_bytes, in.p, in.n)) return FA_ERR_ALIAS;
  if (overlaps(o, q_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;
  if (!make_tensor_map(&pr->tq, q, BH, T, d) || !make_tensor_map(&pr->tk, k, BHkv, T, d) ||
      !make_tensor_map(&pr->tv, v, BHkv, T, d) || !make_tensor_map(&pr->to, o, BH, T, d, false, fa::kOutBoxRows))
    return FA_ERR_CUDA;
  fa::Params& p = pr->p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = BH;
  p.H = H;
  p.group = H / Hkv;
  p.Hkv = Hkv;
  p.block_table = nullptr;
  p.max_pages = 0;
  p.num_pages = 0;
  p.T = T;
  p.causal = causal;
  p.nqb = (T + 255) / 256;
  p.nk = (T + 127) / 128;
  p.num_units = BH * p.nqb;
  p.unit_div = causal ? BH : p.nqb;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.v_descale = 1.f;
  p.timeout_ns = kWaitLimitNs;
  p.num_splits = 1;
  p.split_tiles = p.nk;
  p.opart = nullptr;
  p.lsepart = nullptr;
  return FA_OK;
}

// Key splits chosen for num_splits == 0.  The persistent grid's static schedule is replayed on
// the host for 1 .. 16 splits (the kernel's unit list and its snake assignment of units to
// CTAs; a unit costs the K/V steps of its longer query tile plus kUnitSteps for its start and
// epilogue, plus kMergeSteps when it holds the last key tile of its rows and so may merge
// them; a split launch adds kLaunchSteps), and the count with the least busiest-CTA total wins
// if it beats the unsplit launch by at least 10 %.  The costs are in 128-key steps and were
// fitted to split and unsplit timings on GB300 (B = 1-2, H = 1-32, T = 256-32768, d = 64 and
// 128, causal and not).  Larger problems (more than 16 K units) are not split: their units
// already spread over the SMs.  Results are cached per shape, so that only the first call of a
// shape pays for the replay.
int auto_splits_uncached(int B, int H, int T, int causal, int num_sms) {
  constexpr double kUnitSteps = 2.0, kMergeSteps = 10.0, kLaunchSteps = 2.0;
  const long long BH = static_cast<long long>(B) * H;
  const int nk = (T + 127) / 128, nqb = (T + 255) / 256;
  if (BH * nqb > 16384) return 1;
  std::vector<double> load;
  auto makespan = [&](int want) -> double {
    const int st = (nk + want - 1) / want, ns = (nk + st - 1) / st;
    const long long units = BH * nqb * ns;
    const long long G = std::min<long long>(units, num_sms);
    load.assign(static_cast<size_t>(G), 0.0);
    for (long long w = 0; w < units; ++w) {
      const long long k = w / G, pos = w - k * G;
      const long long b = (k & 1) ? G - 1 - pos : pos;
      int band, sp = 0;
      if (ns > 1) {  // (band, split, head), as the kernel's split form lists them
        band = static_cast<int>(w / (BH * ns));
        sp = static_cast<int>((w - band * BH * ns) / BH);
      } else {  // causal: band by band; otherwise head by head
        band = static_cast<int>(causal ? w / BH : w % nqb);
      }
      const int qb = causal ? nqb - 1 - band : band;
      const int q0 = qb * 256, q1 = q0 + 128;
      const int e0 = q0 >= T ? 0 : (causal ? std::min(nk, q0 / 128 + 1) : nk);
      const int e1 = q1 >= T ? 0 : (causal ? std::min(nk, q1 / 128 + 1) : nk);
      const int lo = sp * st, hi = lo + st;
      const int n = std::max(std::max(0, std::min(e0, hi) - lo), std::max(0, std::min(e1, hi) - lo));
      if (n == 0) continue;
      double c = n + kUnitSteps;
      if (ns > 1 && std::max(e0, e1) <= hi) c += kMergeSteps;
      load[static_cast<size_t>(b)] += c;
    }
    return *std::max_element(load.begin(), load.end()) + (ns > 1 ? kLaunchSteps : 0.0);
  };
  const double t1 = makespan(1);
  double best = t1;
  int best_s = 1;
  for (int sp = 2; sp <= std::min(nk, 16); ++sp) {
    const double t = makespan(sp);
    if (t < best) {
      best = t;
      best_s = sp;
    }
  }
  return best <= 0.9 * t1 ? best_s : 1;
}

int auto_splits(int B, int H, int T, int causal, int num_sms) {
  struct Entry {
    int B, H, T, causal, sms, splits;
  };
  static Entry cache[64] = {};
  static int used = 0, next = 0;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i) {
      const Entry& e = cache[i];
      if (e.B == B && e.H == H && e.T == T && e.causal == causal && e.sms == num_sms) return e.splits;
    }
  }
  const int s = auto_splits_uncached(B, H, T, causal, num_sms);
  std::lock_guard<std::mutex> lock(mu);
  Entry& e = used < 64 ? cache[used++] : cache[next++ % 64];
  e = Entry{B, H, T, causal, num_sms, s};
  return s;
}

// Order of the work items of an unsplit launch.  Causal bf16 d = 128 launches whose K and V
// (one K/V head per query head) exceed 96 MB over all heads, so that L2 cannot hold what the
// CTAs running at one time stream when every head is in flight: the units are listed band by
// band within groups of heads whose K and V fit in 48 MB, except the lightest eighth of the
// bands, which come last band by band over all heads; the CTAs claim the units at run time,
// in list order, from one of the library's counter pairs (taken in turn).  The CTAs running
// at one time then work on one or two groups' heads, and claiming a longest-first list that
// ends in short units keeps the SMs evenly loaded.  Every other launch keeps the static
// band-by-band (causal) or head-by-head order.  If the counters cannot be found the static
// order is kept.
void choose_order(fa::Params& p, int d, int group) {
  constexpr double kGroupBytes = 48e6;
  p.head_group = 0;
  p.sched = nullptr;
  if (!p.causal || d != 128 || group != 1) return;
  const double head_kv = static_cast<double>(p.T) * d * 2 * 2;  // bytes of K and V of one head
  if (head_kv * p.BH <= 96e6) return;
  int g = std::max(1, std::min(p.BH, static_cast<int>(kGroupBytes / head_kv)));
  while (p.BH % g != 0) --g;
  p.tail_bands = std::max(1, p.nqb / 8);
  int* base = nullptr;
  if (fa::sched_counters_address(&base) != cudaSuccess || !base) {
    cudaGetLastError();
    return;
  }
  static std::atomic<unsigned> seq{0};
  p.sched = base + static_cast<size_t>(seq.fetch_add(1) % fa::kSchedSlots) * fa::kSchedStride;
  p.head_group = g;
}

// Workspace layout of the split form: [splits][B*H*T][d] fp32 partial outputs, [splits][B*H*T]
// fp32 partial LSE, then one int counter per 32 query rows of every head.
size_t splitkv_bytes(int B, int H, int T, int d, int num_splits) {
  const size_t rows = static_cast<size_t>(B) * H * T;
  const size_t counters = static_cast<size_t>(B) * H * ((T + 31) / 32);
  const size_t bytes = static_cast<size_t>(num_splits) * rows * (static_cast<size_t>(d) + 1) * 4 + counters * 4;
  return (bytes + 255) / 256 * 256;
}

// Split-KV launch: one kernel over (query block, key split) units.  The counters are cleared
// first (an asynchronous memset on the stream; nothing is allocated); each split writes its
// partials and the last split of every 32-row group merges the group into O and LSE.
fa_status launch_splitkv(Prepared& pr, int d, int num_splits, float* ws, cudaStream_t stream) {
  fa::Params& p = pr.p;
  p.split_tiles = (p.nk + num_splits - 1) / num_splits;
  p.num_splits = (p.nk + p.split_tiles - 1) / p.split_tiles;  // every split holds at least one key tile
  if (p.num_splits == 1) {  // one split is the plain launch: no partials, nothing to merge
    const int grid = p.num_units < pr.num_sms ? p.num_units : pr.num_sms;
    if (fa::launch_fa_fwd(d, pr.tq, pr.tk, pr.tv, pr.to, p, grid, stream) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
    return FA_OK;
  }
  const size_t rows = static_cast<size_t>(p.BH) * p.T;
  p.opart = ws;
  p.lsepart = ws + static_cast<size_t>(p.num_splits) * rows * d;
  p.counters = reinterpret_cast<int*>(p.lsepart + static_cast<size_t>(p.num_splits) * rows);
  p.ngroups = (p.T + 31) / 32;
  const long long units = static_cast<long long>(p.BH) * p.nqb * p.num_splits;
  if (units > INT_MAX) return FA_ERR_BAD_SHAPE;
  p.num_units = static_cast<int>(units);
  p.halves = 0;  // split units are never cut into single tiles
  const int grid = p.num_units < pr.num_sms ? p.num_units : pr.num_sms;
  if (cudaMemsetAsync(p.counters, 0, static_cast<size_t>(p.BH) * p.ngroups * sizeof(int), stream) != cudaSuccess ||
      fa::launch_fa_fwd_partial(d, pr.tq, pr.tk, pr.tv, p, grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T, int d,
                 int causal, float scale, cudaStream_t stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, T, d, causal, scale, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int T,
                     int d, int causal, float scale, cudaStream_t stream) {
  Prepared pr;
  fa_status st = prepare(q, k, v, o, lse, B, H, Hkv, T, d, causal, scale, &pr);
  if (st != FA_OK) return st;
  choose_order(pr.p, d, H / Hkv);
  const int grid = pr.p.num_units < pr.num_sms ? pr.p.num_units : pr.num_sms;
  if (fa::launch_fa_fwd(d, pr.tq, pr.tk, pr.tv, pr.to, pr.p, grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

fa_status fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages, const int* block_table, void* o,
                       float* lse, int B, int H, int Hkv, int T, int d, int causal, float scale, int num_pages,
                       int max_pages, cudaStream_t stream) {
  fa_status st = validate_host(q, k_pages, v_pages, o, lse, B, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (!block_table) return FA_ERR_NULL_PTR;
  if (reinterpret_cast<uintptr_t>(block_table) % 4 != 0) return FA_ERR_MISALIGNED;
  if (Hkv < 1 || Hkv > H || H % Hkv != 0) return FA_ERR_BAD_SHAPE;
  const int nk = (T + 127) / 128;
  if (num_pages < 1 || max_pages < nk || static_cast<long long>(num_pages) * Hkv >= INT_MAX ||
      static_cast<long long>(B) * max_pages > INT_MAX)
    return FA_ERR_BAD_SHAPE;
  int dev = 0, num_sms = 0;
  if ((st = current_device(&dev, &num_sms)) != FA_OK) return st;
  const int BH = B * H;
  const size_t q_bytes = static_cast<size_t>(BH) * T * d * 2, lse_bytes = static_cast<size_t>(BH) * T * 4;
  const size_t pool_bytes = static_cast<size_t>(num_pages) * Hkv * 128 * d * 2;
  const size_t table_bytes = static_cast<size_t>(B) * max_pages * 4;
  const struct {
    const void* p;
    size_t n;
  } ins[4] = {{q, q_bytes}, {k_pages, pool_bytes}, {v_pages, pool_bytes}, {block_table, table_bytes}},
    outs[2] = {{o, q_bytes}, {lse, lse_bytes}};
  for (const auto& x : ins)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (const auto& x : outs)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (const auto& x : ins)
    if (overlaps(o, q_bytes, x.p, x.n) || overlaps(lse, lse_bytes, x.p, x.n)) return FA_ERR_ALIAS;
  if (overlaps(o, q_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;
  Prepared pr;
  pr.dev = dev;
  pr.num_sms = num_sms;
  // page pools as (d, 128 rows, num_pages * Hkv): one TMA box is one page of one head
  if (!make_tensor_map(&pr.tq, q, BH, T, d) || !make_tensor_map(&pr.tk, k_pages, num_pages * Hkv, 128, d) ||
      !make_tensor_map(&pr.tv, v_pages, num_pages * Hkv, 128, d) ||
      !make_tensor_map(&pr.to, o, BH, T, d, false, fa::kOutBoxRows))
    return FA_ERR_CUDA;
  fa::Params& p = pr.p;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = BH;
  p.H = H;
  p.group = H / Hkv;
  p.Hkv = Hkv;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.T = T;
  p.causal = causal;
  p.nqb = (T + 255) / 256;
  p.nk = nk;
  p.num_units = BH * p.nqb;
  p.unit_div = causal ? BH : p.nqb;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.v_descale = 1.f;
  p.timeout_ns = kWaitLimitNs;
  p.num_splits = 1;
  p.split_tiles = p.nk;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  if (fa::launch_fa_fwd(d, pr.tq, pr.tk, pr.tv, pr.to, p, grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

fa_status fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                 int T, int d, int causal, float scale, int num_splits, cudaStream_t stream) {
  if (num_splits < 0 || num_splits > FA_MAX_SPLITS) return FA_ERR_BAD_ARG;
  Prepared pr;
  fa_status st = prepare(q, k, v, o, lse, B, H, H, T, d, causal, scale, &pr);
  if (st != FA_OK) return st;
  if (num_splits == 0) num_splits = auto_splits(B, H, T, causal, pr.num_sms);
  if (splitkv_bytes(B, H, T, d, num_splits) > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (fa::noalloc_scratch_address(&scratch) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return launch_splitkv(pr, d, num_splits, static_cast<float*>(scratch), stream);
}

size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int T, int d, int num_splits) {
  if (B < 1 || H < 1 || T < 1 || (d != 64 && d != 128) || num_splits < 0 || num_splits > FA_MAX_SPLITS) return 0;
  if (num_splits == 0) {  // the automatic choice, for either mask, on the current device
    int dev = 0, sms = 0;
    if (current_device(&dev, &sms) != FA_OK) return 0;
    num_splits = std::max(auto_splits(B, H, T, 0, sms), auto_splits(B, H, T, 1, sms));
  }
  return splitkv_bytes(B, H, T, d, num_splits);
}

int fa_fwd_splitkv_count(int B, int H, int T, int d, int causal, int num_splits) {
  if (B < 1 || H < 1 || T < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1) || num_splits < 0 ||
      num_splits > FA_MAX_SPLITS)
    return -1;
  if (num_splits == 0) {
    int dev = 0, sms = 0;
    if (current_device(&dev, &sms) != FA_OK) return -1;
    num_splits = auto_splits(B, H, T, causal, sms);
  }
  const int nk = (T + 127) / 128, st = (nk + num_splits - 1) / num_splits;
  return (nk + st - 1) / st;
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T,
                         int d, int causal, float scale, int num_splits, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  if (num_splits < 0 || num_splits > FA_MAX_SPLITS) return FA_ERR_BAD_ARG;
  Prepared pr;
  fa_status st = prepare(q, k, v, o, lse, B, H, H, T, d, causal, scale, &pr);
  if (st != FA_OK) return st;
  if (num_splits == 0) num_splits = auto_splits(B, H, T, causal, pr.num_sms);
  const size_t need = splitkv_bytes(B, H, T, d, num_splits);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return FA_ERR_MISALIGNED;
  if ((st = check_device_range(workspace, need, pr.dev)) != FA_OK) return st;
  const size_t qkv_bytes = static_cast<size_t>(B) * H * T * d * 2, lse_bytes = static_cast<size_t>(B) * H * T * 4;
  for (const void* x : {q, k, v, static_cast<const void*>(o)})
    if (overlaps(workspace, need, x, qkv_bytes)) return FA_ERR_ALIAS;
  if (overlaps(workspace, need, lse, lse_bytes)) return FA_ERR_ALIAS;
  return launch_splitkv(pr, d, num_splits, static_cast<float*>(workspace), stream);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int T, int d) {
  if (B < 1 || H < 1 || T < 1 || d != 128) return 0;
  const size_t Tp = (static_cast<size_t>(T) + 15) / 16 * 16;
  const size_t bytes = static_cast<size_t>(B) * H * 128 * Tp;
  return (bytes + 255) / 256 * 256;
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int T, int d,
                     int causal, float scale, float q_descale, float k_descale, float v_descale, void* workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
  fa_status st = validate_host(q, k, v, o, lse, B, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (d != 128) return FA_ERR_UNSUPPORTED_HEAD_DIM;
  for (float x : {q_descale, k_descale, v_descale})
    if (!std::isfinite(x) || !(x > 0.f)) return FA_ERR_BAD_SCALE;
  const size_t need = fa_fwd_fp8_workspace_bytes(B, H, T, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return FA_ERR_MISALIGNED;
  const int BH = B * H;
  if (BH > 65535) return FA_ERR_BAD_SHAPE;  // one grid row of the V transpose per head
  int dev = 0, num_sms = 0;
  if ((st = current_device(&dev, &num_sms)) != FA_OK) return st;
  const int Tp = (T + 15) / 16 * 16;
  const size_t in_bytes = static_cast<size_t>(BH) * T * 128, o_bytes = static_cast<size_t>(BH) * T * 128 * 2,
               lse_bytes = static_cast<size_t>(BH) * T * 4;
  const struct {
    const void* p;
    size_t n;
  } ins[3] = {{q, in_bytes}, {k, in_bytes}, {v, in_bytes}},
    outs[3] = {{o, o_bytes}, {lse, lse_bytes}, {workspace, need}};
  for (const auto& x : ins)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (const auto& x : outs)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (int a = 0; a < 3; ++a) {
    for (const auto& x : ins)
      if (overlaps(outs[a].p, outs[a].n, x.p, x.n)) return FA_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(outs[a].p, outs[a].n, outs[b].p, outs[b].n)) return FA_ERR_ALIAS;
  }
  CUtensorMap tq, tk, tvt, to;
  if (!make_tensor_map(&tq, q, BH, T, 128, true) || !make_tensor_map(&tk, k, BH, T, 128, true) ||
      !make_tensor_map(&tvt, workspace, BH, 128, Tp, true) ||
      !make_tensor_map(&to, o, BH, T, 128, false, fa::kOutBoxRows))
    return FA_ERR_CUDA;
  fa::Params p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = BH;
  p.H = H;
  p.group = 1;
  p.Hkv = H;
  p.block_table = nullptr;
  p.T = T;
  p.causal = causal;
  p.nqb = (T + 255) / 256;
  p.nk = (T + 127) / 128;
  p.num_units = BH * p.nqb;
  p.unit_div = causal ? BH : p.nqb;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * q_descale * k_descale * 1.4426950408889634074);
  p.v_descale = v_descale;
  p.timeout_ns = kWaitLimitNs;
  p.num_splits = 1;
  p.split_tiles = p.nk;
  const long long items = work_items_e4m3(p.num_units, p.nk, causal, num_sms, &p.halves);
  if (items > INT_MAX) return FA_ERR_BAD_SHAPE;
  p.num_units = static_cast<int>(items);
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  if (fa::launch_transpose_e4m3(v, workspace, BH, T, Tp, stream) != cudaSuccess ||
      fa::launch_fa_fwd_e4m3(tq, tk, tvt, to, p, grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

size_t fa_bwd_workspace_bytes(int B, int H, int T) {
  if (B < 1 || H < 1 || T < 1) return 0;
  const size_t Tp = (static_cast<size_t>(T) + 127) / 128 * 128;
  const size_t bytes = 2 * static_cast<size_t>(B) * H * Tp * 4;  // D and LSE * log2 e, rows padded to 128
  return (bytes + 255) / 256 * 256;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                 void* dq, void* dk, void* dv, int B, int H, int T, int d, int causal, float scale, void* workspace,
                 size_t workspace_bytes, cudaStream_t stream) {
  fa_status st = validate_host(q, k, v, o, lse, B, H, T, d, causal, scale);
  if (st != FA_OK) return st;
  if (!dout || !dq || !dk || !dv) return FA_ERR_NULL_PTR;
  for (const void* x : {dout, static_cast<const void*>(dq), static_cast<const void*>(dk), static_cast<const void*>(dv)})
    if (reinterpret_cast<uintptr_t>(x) % 16 != 0) return FA_ERR_MISALIGNED;
  const size_t need = fa_bwd_workspace_bytes(B, H, T);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return FA_ERR_MISALIGNED;
  int dev = 0, num_sms = 0;
  if ((st = current_device(&dev, &num_sms)) != FA_OK) return st;
  const int BH = B * H;
  const size_t t_bytes = static_cast<size_t>(BH) * T * d * 2, r_bytes = static_cast<size_t>(BH) * T * 4;
  const struct {
    const void* p;
    size_t n;
  } ins[6] = {{q, t_bytes}, {k, t_bytes}, {v, t_bytes}, {o, t_bytes}, {dout, t_bytes}, {lse, r_bytes}},
    outs[4] = {{dq, t_bytes}, {dk, t_bytes}, {dv, t_bytes}, {workspace, need}};
  for (const auto& x : ins)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (const auto& x : outs)
    if ((st = check_device_range(x.p, x.n, dev)) != FA_OK) return st;
  for (int a = 0; a < 4; ++a) {
    for (const auto& x : ins)
      if (overlaps(outs[a].p, outs[a].n, x.p, x.n)) return FA_ERR_ALIAS;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a].p, outs[a].n, outs[b].p, outs[b].n)) return FA_ERR_ALIAS;
  }
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;  // outputs: 32-row x 32-column boxes, no swizzle
  if (!make_tensor_map(&tq, q, BH, T, d) || !make_tensor_map(&tk, k, BH, T, d) ||
      !make_tensor_map(&tv, v, BH, T, d) || !make_tensor_map(&tdo, dout, BH, T, d) ||
      !make_tensor_map(&tdq, dq, BH, T, d, false, fa::kGradBoxRows, fa::kGradBoxCols * 2) ||
      !make_tensor_map(&tdk, dk, BH, T, d, false, fa::kGradBoxRows, fa::kGradBoxCols * 2) ||
      !make_tensor_map(&tdv, dv, BH, T, d, false, fa::kGradBoxRows, fa::kGradBoxCols * 2))
    return FA_ERR_CUDA;
  fa::BwdParams p{};
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.drow = static_cast<float*>(workspace);
  p.Tp = (T + 127) / 128 * 128;
  p.lse2 = p.drow + static_cast<size_t>(BH) * p.Tp;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.BH = BH;
  p.T = T;
  p.causal = causal;
  p.nt = (T + 127) / 128;
  const long long units = static_cast<long long>(BH) * p.nt;
  if (units * 128 > INT_MAX) return FA_ERR_BAD_SHAPE;  // padded rows are indexed in 32 bits
  p.num_units = static_cast<int>(units);
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
  p.timeout_ns = kWaitLimitNs;
  const int grid = p.num_units < num_sms ? p.num_units : num_sms;
  if (fa::launch_bwd_dq(d, tq, tk, tv, tdo, tdq, tdq, p, grid, stream) != cudaSuccess ||
      fa::launch_bwd_dkdv(d, tq, tk, tv, tdo, tdv, tdk, p, grid, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

static_assert(FA_NOALLOC_SCRATCH_BYTES == fa::kNoAllocScratchBytes, "fa.h and the kernel disagree on the scratch size");

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_NULL_PTR: return "a required pointer is NULL";
    case FA_ERR_MISALIGNED: return "a pointer is not 16-byte aligned";
    case FA_ERR_BAD_SHAPE: return "B, H or T out of range";
    case FA_ERR_UNSUPPORTED_HEAD_DIM: return "head size d must be 64 or 128";
    case FA_ERR_BAD_SCALE: return "scale must be finite and > 0";
    case FA_ERR_NO_DEVICE_SUPPORT: return "the current device is not an sm_103 GPU";
    case FA_ERR_LAUNCH: return "kernel launch failed";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded in-kernel wait ran out";
    case FA_ERR_BAD_ARG: return "causal must be 0 or 1";
    case FA_ERR_BAD_POINTER: return "a pointer is not device memory of the current device, or its allocation is too small";
    case FA_ERR_ALIAS: return "an output overlaps an input or the other output";
    case FA_ERR_CUDA: return "a CUDA runtime or driver call failed";
    case FA_ERR_BAD_PAGE: return "a block-table entry named a page outside the pool (its keys read as zeros)";
    case FA_ERR_WORKSPACE: return "the workspace is missing or smaller than the size its *_workspace_bytes() gives";
  }
  return "unknown status";
}

fa_status fa_device_status(cudaStream_t stream, int* out) {
  if (!out) return FA_ERR_NULL_PTR;
  unsigned int word = 0, bwd = 0;
  if (fa::read_and_clear_status(stream, &word) != cudaSuccess ||
      fa::read_and_clear_bwd_status(stream, &bwd) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  word |= bwd;
  *out = (word & 2u) ? FA_ERR_BAD_PAGE : (word & 1u) ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
  return FA_OK;
}

fa_status fa_fwd_launch_shape(int B, int H, int T, int d, int causal, int num_sms, int* grid, int* threads,
                              int* smem_bytes) {
  if (!grid || !threads || !smem_bytes) return FA_ERR_NULL_PTR;
  static const char dummy[16] __attribute__((aligned(16))) = {};
  fa_status st = validate_host(dummy, dummy, dummy, dummy, dummy, B, H, T, d, causal, 1.0f);
  if (st != FA_OK) return st;
  if (num_sms < 1) return FA_ERR_BAD_ARG;
  const long long units = static_cast<long long>(B) * H * ((T + 255) / 256);
  *grid = static_cast<int>(units < num_sms ? units : num_sms);
  *threads = fa::fa_fwd_threads(d);
  *smem_bytes = fa::fa_fwd_smem_bytes(d);
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(unsigned int timeout_us, cudaStream_t stream) {
  if (timeout_us < 1 || timeout_us > 2000000) return FA_ERR_BAD_ARG;
  int dev = 0, num_sms = 0;
  fa_status st = current_device(&dev, &num_sms);
  if (st != FA_OK) return st;
  if (fa::launch_wait_selftest(static_cast<unsigned long long>(timeout_us) * 1000ull, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

fa_status fa_ex2_rate(double* ops_per_second, cudaStream_t stream) {
  if (!ops_per_second) return FA_ERR_NULL_PTR;
  int dev = 0, num_sms = 0;
  fa_status st = current_device(&dev, &num_sms);
  if (st != FA_OK) return st;
  if (fa::measure_ex2_rate(num_sms, ops_per_second, stream) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

const char* fa_version(void) { return "0.1.0"; }

}  // extern "C"
