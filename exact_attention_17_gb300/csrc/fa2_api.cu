// Host side of libfa2.so: argument validation, TMA tensor maps, launches.
// The C ABI is declared (and documented) in include/fa2.h.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fa2.h"
#include "fa2_launch.h"

namespace {

// Kernels of this library OR their error bits here (one word per device).
__device__ int g_device_status = 0;

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per barrier wait
constexpr int kMaxSplits = 64;
constexpr int kMaxDevices = 64;

struct DriverFns {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  PFN_cuMemGetAddressRange_v3020 range = nullptr;
  bool ok = false;
};

const DriverFns& driver() {
  static DriverFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
    cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f2, 3020, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
      fns.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
      fns.range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(f2);
      fns.ok = true;
    }
  });
  return fns;
}

// Per device: is it an sm_103 part, and have the kernels' shared-memory limits been raised.
struct DeviceState {
  std::once_flag once;
  bool usable = false;
  int sms = 0;
};
DeviceState g_devices[kMaxDevices];

int device_ready() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_DEVICE;
  DeviceState& st = g_devices[dev];
  std::call_once(st.once, [&] {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return;
    if (major != 10 || minor != 3) return;
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return;
    if (fa2host::prepare_tc_d64_bf16() != cudaSuccess || fa2host::prepare_tc_d128_bf16() != cudaSuccess ||
        fa2host::prepare_tc_d64_f16() != cudaSuccess || fa2host::prepare_tc_d128_f16() != cudaSuccess ||
        fa2host::prepare_tc_d256_bf16() != cudaSuccess || fa2host::prepare_tc_d256_f16() != cudaSuccess ||
        fa2host::prepare_tc_pair_d128() != cudaSuccess || fa2host::prepare_simt() != cudaSuccess ||
        fa2host::prepare_bwd() != cudaSuccess || fa2host::prepare_bwd2() != cudaSuccess)
      return;
    st.usable = true;
  });
  if (!st.usable) return FA2_ERR_DEVICE;
  if (!driver().ok) return FA2_ERR_DEVICE;
  return FA2_OK;
}

// Streaming multiprocessors of the current device (after device_ready succeeded).
int sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  return g_devices[dev].sms > 0 ? g_devices[dev].sms : 148;
}

// Allocations (base address, size) already found to be device or managed
// memory.  The range query below runs on every call and returns the live
// allocation holding a pointer; only the memory-type query is skipped for an
// allocation seen before.  An allocation freed and replaced by another at
// the same base with the same size is looked up again only if the range
// query fails for it (memory that is not a device allocation).
struct AllocCache {
  static constexpr int kEntries = 32;
  std::mutex mu;
  CUdeviceptr base[kEntries] = {};
  size_t size[kEntries] = {};
  int next = 0;

  bool hit(CUdeviceptr b, size_t n) {
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < kEntries; ++i)
      if (base[i] == b && size[i] == n && n != 0) return true;
    return false;
  }
  void add(CUdeviceptr b, size_t n) {
    std::lock_guard<std::mutex> lock(mu);
    base[next] = b;
    size[next] = n;
    next = (next + 1) % kEntries;
  }
};
AllocCache g_alloc_cache;

// The whole byte range [p, p + bytes) must be device memory of one allocation.
// The cheap range query comes first; when it fails (it also fails before the
// runtime has made the device's context current on this thread), the memory
// type query, which makes it current, runs and the range query is repeated.
bool device_range_ok(const void* p, size_t bytes) {
  const uintptr_t begin = reinterpret_cast<uintptr_t>(p);
  CUdeviceptr base = 0;
  size_t size = 0;
  bool have_range = driver().range(&base, &size, static_cast<CUdeviceptr>(begin)) == CUDA_SUCCESS;
  if (have_range && !(begin >= base && bytes <= size && begin - base <= size - bytes)) return false;
  if (have_range && g_alloc_cache.hit(base, size)) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) return false;
  if (!have_range) {
    if (driver().range(&base, &size, static_cast<CUdeviceptr>(begin)) != CUDA_SUCCESS) return false;
    if (!(begin >= base && bytes <= size && begin - base <= size - bytes)) return false;
  }
  g_alloc_cache.add(base, size);
  return true;
}

// Device address of the status word on the current device (looked up once
// per device; a failed lookup is retried by the next call).
int* status_word() {
  static std::mutex mu;
  static int* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

// 3-D map over [BH][N][d] 16-bit elements (bf16 or fp16): box = 64 columns
// (128 B, one swizzle atom) x `rows` rows x 1 (128 by default; 64 for the
// K halves of the two-SM kernel).  Rows past N read as zero instead of
// running into the next head.
bool encode_map(CUtensorMap* map, const void* base, int d, int N, int BH, bool f16, unsigned rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = driver().encode(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                               3, const_cast<void*>(base), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over an fp32 [BH][N][d] array: box = 32 columns (128 B) x `rows`
// rows x 1 (128 by default; 32 for the two-tile backward kernel), 128-byte
// swizzle; the backward pass adds its dQ partials through it.
bool encode_map_f32(CUtensorMap* map, const void* base, int d, int N, int BH, unsigned rows = 128) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4, static_cast<cuuint64_t>(N) * d * 4};
  cuuint32_t box[3] = {32, rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = driver().encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the forward's output [Z][Nq][d] (Z = B*H, or splits * B*H for
// the split-KV partials): fp32 with 32-column boxes, or 16-bit (bf16/fp16)
// with 64-column boxes; 128 rows, 128-byte swizzle.  The epilogue stores O
// through it; rows past Nq fall outside the map.
bool encode_map_out(CUtensorMap* map, const void* base, int d, int Nq, long long Z, int elem_bytes,
                    bool f16) {
  if (Z > 0x7fffffffLL) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(Nq),
                        static_cast<cuuint64_t>(Z)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                           static_cast<cuuint64_t>(Nq) * d * elem_bytes};
  cuuint32_t box[3] = {elem_bytes == 4 ? 32u : 64u, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType type = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : f16           ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = driver().encode(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Multiplier and shift of fa2dev::fast_div for a divisor d >= 1.
fa2dev::FastDiv make_fast_div(int d) {
  int l = 0;
  while ((1LL << l) < d) ++l;
  const unsigned long long two = 1ULL << (31 + l);
  fa2dev::FastDiv f;
  f.m = static_cast<uint32_t>((two + static_cast<unsigned long long>(d) - 1) / static_cast<unsigned long long>(d));
  f.s = 31 + l;
  return f;
}

// Head dimensions of the tensor-core forward kernels (and of the merge).
bool forward_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

struct Problem {
  int B, H, Nq, Nk, d;
  long long BH;
  bool empty;
};

int validate(const void* Q, const void* K, const void* V, const void* O, const float* LSE, int B,
             int H, int Nq, int Nk, int d, float scale, Problem* pr, size_t o_elem_bytes = 4) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA2_ERR_SHAPE;
  pr->B = B; pr->H = H; pr->Nq = Nq; pr->Nk = Nk; pr->d = d;
  pr->BH = static_cast<long long>(B) * H;
  pr->empty = pr->BH == 0 || Nq == 0;
  if (pr->empty) return FA2_OK;
  if (Nk < 1) return FA2_ERR_SHAPE;
  if (pr->BH > 0x7fffffffLL) return FA2_ERR_SHAPE;
  if (!forward_head_dim(d)) return FA2_ERR_HEADDIM;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  if (!Q || !K || !V || !O || !LSE) return FA2_ERR_NULL;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0) return FA2_ERR_ALIGN;
  int rc = device_ready();
  if (rc != FA2_OK) return rc;
  const size_t bh = static_cast<size_t>(pr->BH);
  const size_t q_elems = bh * Nq * d, kv_elems = bh * Nk * d;
  if (!device_range_ok(Q, q_elems * 2) || !device_range_ok(K, kv_elems * 2) ||
      !device_range_ok(V, kv_elems * 2) || !device_range_ok(O, q_elems * o_elem_bytes) ||
      !device_range_ok(LSE, bh * Nq * 4))
    return FA2_ERR_MEMORY;
  return FA2_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

// The two-SM kernel is the default for the shapes where the one-CTA kernel
// takes two query sub-tiles per CTA.
constexpr bool kPairByDefault = false;

// Query sub-tiles of 128 rows per CTA.  Two (one CTA per SM, the sub-tiles
// ping-pong on the tensor core) is faster for long query blocks; one (two
// CTAs per SM) when a second sub-tile would have no rows (Nq <= 128) or when
// two-sub-tile CTAs would not fill two waves of the GPU.
int subtiles_per_cta(const Problem& pr, int splits) {
  if (pr.Nq <= 128 || pr.d == 256) return 1;
  const long long ctas2 = (static_cast<long long>(pr.Nq) + 255) / 256 * pr.BH * splits;
  return ctas2 < 2LL * sm_count() ? 1 : 2;
}

// Items (b*H + h, key range) per scheduling group: as many as have their
// K and V tiles fit in kL2GroupBytes together (at least one).
constexpr long long kL2GroupBytes = 64LL << 20;

int item_group(const Problem& pr, int splits) {
  const long long items = pr.BH * splits;
  const long long kv_bytes = 2LL * ((pr.Nk + splits - 1) / splits) * pr.d * 2;
  long long g = kL2GroupBytes / (kv_bytes > 0 ? kv_bytes : 1);
  if (g < 1) g = 1;
  if (g > items) g = items;
  return static_cast<int>(g);
}

// Which forward kernel runs a head-dimension-128 problem: the two-SM kernel
// (a CTA pair per 512 query rows) or the one-CTA kernel.  FA2_FORWARD_KERNEL
// = "pair" or "single" in the environment overrides the choice (for
// comparing the two); by default the pair kernel runs where the one-CTA
// kernel would take two query sub-tiles per CTA.
bool use_pair_kernel(const Problem& pr, int subs) {
  if (pr.d != 128) return false;
  const char* v = std::getenv("FA2_FORWARD_KERNEL");
  if (v != nullptr && std::strcmp(v, "pair") == 0) return true;
  if (v != nullptr && std::strcmp(v, "single") == 0) return false;
  return kPairByDefault && subs == 2;
}

// Launch of the tensor-core kernel over `splits` key ranges of `tiles_per_split`
// tiles each (splits == 1: the whole key range, outputs O and LSE directly).
int launch_forward(const void* Q, const void* K, const void* V, float* O, float* LSE,
                   const Problem& pr, int causal, float scale, int splits, int tiles_per_split,
                   float* O_part, float* LSE_part, cudaStream_t s, bool f16 = false,
                   bool o_half = false) {
  const int Nq = pr.Nq, Nk = pr.Nk, d = pr.d;
  const int subs = subtiles_per_cta(pr, splits);
  const bool pair = use_pair_kernel(pr, subs);
  // query blocks: 512 rows per CTA pair, else 128 x subs rows per CTA
  const long long rows_per_block = pair ? 512 : 128 * subs;
  const long long blocks = (static_cast<long long>(Nq) + rows_per_block - 1) / rows_per_block;
  if (blocks * pr.BH * splits * (pair ? 2 : 1) > 0x7fffffffLL) return FA2_ERR_SHAPE;

  CUtensorMap mq, mk, mv, mo;
  const bool split_out = splits > 1;
  if (!encode_map(&mq, Q, d, Nq, static_cast<int>(pr.BH), f16) ||
      !encode_map(&mk, K, d, Nk, static_cast<int>(pr.BH), f16, pair ? 64 : 128) ||
      !encode_map(&mv, V, d, Nk, static_cast<int>(pr.BH), f16) ||
      !encode_map_out(&mo, split_out ? static_cast<const void*>(O_part) : static_cast<const void*>(O), d, Nq,
                      split_out ? pr.BH * splits : pr.BH, (o_half && !split_out) ? 2 : 4, f16))
    return FA2_ERR_SHAPE;

  fa2dev::FwdParams p;
  p.O = O;
  p.LSE = LSE;
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = static_cast<int>(pr.BH);
  p.q_blocks = static_cast<int>(blocks);
  p.scale_log2 = scale * kLog2e;
  p.timeout_ns = kWaitTimeoutNs;
  p.num_splits = splits;
  p.tiles_per_split = tiles_per_split;
  p.O_part = O_part;
  p.LSE_part = LSE_part;
  p.o_half = o_half ? 1 : 0;
  p.item_group = item_group(pr, splits);
  p.div_per_group = make_fast_div(static_cast<int>(p.item_group * blocks));
  p.div_group = make_fast_div(p.item_group);
  p.div_splits = make_fast_div(splits);
  p.wave = sm_count() * (pair || subs == 2 || d == 256 ? 1 : 2);
  p.status = status_word();
  if (p.status == nullptr) return FA2_ERR_LAUNCH;

  const unsigned grid = static_cast<unsigned>(blocks * pr.BH * splits * (pair ? 2 : 1));
  const bool c = causal != 0;
  cudaError_t e;
  if (pair)
    e = fa2host::launch_tc_pair_d128(c, f16, mq, mk, mv, mo, p, grid, s);
  else if (d == 64)
    e = f16 ? fa2host::launch_tc_d64_f16(subs, c, mq, mk, mv, mo, p, grid, s)
            : fa2host::launch_tc_d64_bf16(subs, c, mq, mk, mv, mo, p, grid, s);
  else if (d == 128)
    e = f16 ? fa2host::launch_tc_d128_f16(subs, c, mq, mk, mv, mo, p, grid, s)
            : fa2host::launch_tc_d128_bf16(subs, c, mq, mk, mv, mo, p, grid, s);
  else
    e = f16 ? fa2host::launch_tc_d256_f16(subs, c, mq, mk, mv, mo, p, grid, s)
            : fa2host::launch_tc_d256_bf16(subs, c, mq, mk, mv, mo, p, grid, s);
  return e == cudaSuccess ? FA2_OK : FA2_ERR_LAUNCH;
}

int key_tiles(int Nk) { return (Nk + 127) / 128; }

// Key ranges actually used for a requested split count: ranges of
// ceil(tiles / requested) tiles, as many as that takes.
void split_plan(int Nk, int requested, int* splits, int* tiles_per_split) {
  const int tiles = key_tiles(Nk);
  const int want = requested < 1 ? 1 : (requested > tiles ? tiles : requested);
  *tiles_per_split = (tiles + want - 1) / want;
  *splits = (tiles + *tiles_per_split - 1) / *tiles_per_split;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Workspace layout for `splits` ranges: O_part, then LSE_part (256-byte aligned).
size_t workspace_bytes(long long BH, int Nq, int d, int splits) {
  const size_t rows = static_cast<size_t>(BH) * Nq;
  return align256(static_cast<size_t>(splits) * rows * d * 4) + align256(static_cast<size_t>(splits) * rows * 4);
}

// Backward workspace: LSE log2(e), then D, each [BH][Nq rounded up to 128] fp32.
size_t bwd_workspace_bytes(long long BH, int Nq) {
  const size_t pad = (static_cast<size_t>(Nq) + 127) / 128 * 128;
  return 2 * align256(static_cast<size_t>(BH) * pad * 4);
}

}  // namespace

extern "C" int fa2_forward(const void* Q, const void* K, const void* V, float* O, float* LSE, int B,
                           int H, int Nq, int Nk, int d, int causal, float scale,
                           fa2_stream_t stream) {
  Problem pr;
  int rc = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, &pr);
  if (rc != FA2_OK || pr.empty) return rc;
  return launch_forward(Q, K, V, O, LSE, pr, causal, scale, 1, key_tiles(Nk), nullptr, nullptr,
                        reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int fa2_forward_typed(const void* Q, const void* K, const void* V, void* O, float* LSE,
                                 int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                 int qkv_dtype, int o_dtype, fa2_stream_t stream) {
  if (qkv_dtype != FA2_DTYPE_BF16 && qkv_dtype != FA2_DTYPE_FP16) return FA2_ERR_DTYPE;
  if (o_dtype != FA2_DTYPE_FP32 && o_dtype != qkv_dtype) return FA2_ERR_DTYPE;
  const bool o_half = o_dtype != FA2_DTYPE_FP32;
  Problem pr;
  int rc = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, &pr, o_half ? 2 : 4);
  if (rc != FA2_OK || pr.empty) return rc;
  return launch_forward(Q, K, V, static_cast<float*>(O), LSE, pr, causal, scale, 1, key_tiles(Nk),
                        nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream),
                        qkv_dtype == FA2_DTYPE_FP16, o_half);
}

extern "C" size_t fa2_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 0 || H < 0 || Nq < 0 || num_splits < 1 || !forward_head_dim(d)) return 0;
  return workspace_bytes(static_cast<long long>(B) * H, Nq, d, num_splits);
}

namespace {

// Split count for fa2_forward_splitkv on a machine with `sms` SMs.  Without a
// split every (b*H + h, query block) is one CTA of one 128-row sub-tile, two
// of which run on each SM; with S key ranges there are S times as many CTAs,
// each visiting about 1/S of the key tiles, and a second kernel merges the
// ranges.  The estimate of the time, in units of one key tile of one CTA,
// is (waves of CTAs) x (key tiles per CTA + kCtaFixedTiles) plus, for S > 1,
// kMergeTiles: measured, a CTA's start and end cost about four tiles' time
// (a 1000-length, 16-head problem ran slower in two ranges than in one) and
// the merge launch about five.  The smallest S with the least estimate wins.
// Only grids that leave CTA slots empty are split: a grid of a wave or more
// keeps S = 1.
constexpr long long kCtaFixedTiles = 4;
constexpr long long kMergeTiles = 5;

int recommended_splits(long long BH, int Nq, int Nk, int sms) {
  if (BH <= 0 || Nq <= 0 || Nk <= 0 || sms <= 0) return 1;
  const long long ctas = (static_cast<long long>(Nq) + 127) / 128 * BH;
  const long long slots = 2LL * sms;
  if (ctas >= slots) return 1;
  const int tiles = key_tiles(Nk);
  int best = 1;
  long long best_cost = -1;
  for (int want = 1; want <= kMaxSplits && want <= tiles; ++want) {
    int splits = 1, tps = 1;
    split_plan(Nk, want, &splits, &tps);
    if (splits != want) continue;   // the same plan as a smaller count
    const long long waves = (ctas * splits + slots - 1) / slots;
    const long long cost = waves * (tps + kCtaFixedTiles) + (splits > 1 ? kMergeTiles : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = splits;
    }
  }
  return best;
}

}  // namespace

extern "C" int fa2_splitkv_recommended_splits(int B, int H, int Nq, int Nk, int sm_count) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return 1;
  int sms = sm_count;
  if (sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 1;
    }
  }
  return recommended_splits(static_cast<long long>(B) * H, Nq, Nk, sms);
}

extern "C" int fa2_forward_splitkv(const void* Q, const void* K, const void* V, float* O, float* LSE,
                                   int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                   int num_splits, void* workspace, size_t workspace_size,
                                   fa2_stream_t stream) {
  if (num_splits < 1 || num_splits > kMaxSplits) return FA2_ERR_SHAPE;
  Problem pr;
  int rc = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, &pr);
  if (rc != FA2_OK || pr.empty) return rc;
  int splits = 1, tps = 1;
  split_plan(Nk, num_splits, &splits, &tps);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (splits == 1)
    return launch_forward(Q, K, V, O, LSE, pr, causal, scale, 1, tps, nullptr, nullptr, s);
  const size_t need = workspace_bytes(pr.BH, Nq, d, splits);
  if (!workspace) return FA2_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA2_ERR_ALIGN;
  if (workspace_size < need || !device_range_ok(workspace, need)) return FA2_ERR_MEMORY;
  const size_t rows = static_cast<size_t>(pr.BH) * Nq;
  float* O_part = static_cast<float*>(workspace);
  float* LSE_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             align256(static_cast<size_t>(splits) * rows * d * 4));
  rc = launch_forward(Q, K, V, O, LSE, pr, causal, scale, splits, tps, O_part, LSE_part, s);
  if (rc != FA2_OK) return rc;
  return fa2host::launch_combine(d, O_part, LSE_part, splits, static_cast<long long>(rows), O, LSE, s) ==
                 cudaSuccess
             ? FA2_OK
             : FA2_ERR_LAUNCH;
}

extern "C" int fa2_merge(const float* O_parts, const float* LSE_parts, int num_parts, long long rows,
                         int d, float* O, float* LSE, fa2_stream_t stream) {
  if (rows < 0 || num_parts < 0) return FA2_ERR_SHAPE;
  if (rows == 0) return FA2_OK;
  if (num_parts < 1 || num_parts > kMaxSplits) return FA2_ERR_SHAPE;
  if (!forward_head_dim(d)) return FA2_ERR_HEADDIM;
  if (!O_parts || !LSE_parts || !O || !LSE) return FA2_ERR_NULL;
  if (((reinterpret_cast<uintptr_t>(O_parts) | reinterpret_cast<uintptr_t>(O)) & 15u) != 0 ||
      ((reinterpret_cast<uintptr_t>(LSE_parts) | reinterpret_cast<uintptr_t>(LSE)) & 3u) != 0)
    return FA2_ERR_ALIGN;
  int rc = device_ready();
  if (rc != FA2_OK) return rc;
  const size_t r = static_cast<size_t>(rows);
  if (!device_range_ok(O_parts, r * num_parts * d * 4) || !device_range_ok(LSE_parts, r * num_parts * 4) ||
      !device_range_ok(O, r * d * 4) || !device_range_ok(LSE, r * 4))
    return FA2_ERR_MEMORY;
  return fa2host::launch_combine(d, O_parts, LSE_parts, num_parts, rows, O, LSE,
                                 reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FA2_OK
             : FA2_ERR_LAUNCH;
}

extern "C" int fa2_forward_simt(const void* Q, const void* K, const void* V, float* O, float* LSE,
                                int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                fa2_stream_t stream) {
  Problem pr;
  int rc = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, &pr);
  if (rc != FA2_OK || pr.empty) return rc;
  if (d == 256) return FA2_ERR_HEADDIM;   // the SIMT kernels cover 64 and 128
  if (pr.BH > 65535) return FA2_ERR_SHAPE;
  fa2dev::SimtParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.V = static_cast<const __nv_bfloat16*>(V);
  p.O = O;
  p.LSE = LSE;
  p.Nq = Nq;
  p.Nk = Nk;
  p.scale_log2 = scale * kLog2e;
  dim3 grid((Nq + fa2dev::kSimtRows - 1) / fa2dev::kSimtRows, static_cast<unsigned>(pr.BH));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = fa2host::launch_simt(d, causal != 0, p, grid, s);
  return e == cudaSuccess ? FA2_OK : FA2_ERR_LAUNCH;
}

extern "C" size_t fa2_backward_workspace_bytes(int B, int H, int Nq) {
  if (B < 0 || H < 0 || Nq < 0) return 0;
  return bwd_workspace_bytes(static_cast<long long>(B) * H, Nq);
}

namespace {

// The two-tile backward kernel (two 64-row query tiles in flight) runs head
// dimension 128 by default; FA2_BACKWARD_KERNEL = "one_tile" or "two_tile"
// in the environment overrides the choice (for comparing the two).
constexpr bool kTwoTileByDefault = false;

bool use_two_tile_backward(int d) {
  if (d != 128) return false;
  const char* v = std::getenv("FA2_BACKWARD_KERNEL");
  if (v != nullptr && std::strcmp(v, "two_tile") == 0) return true;
  if (v != nullptr && std::strcmp(v, "one_tile") == 0) return false;
  return kTwoTileByDefault;
}

// The backward pass for bf16 (f16 = false) or fp16 Q, K, V and dO.
int backward_impl(const void* Q, const void* K, const void* V, const float* O, const void* dO,
                  const float* LSE, float* dQ, float* dK, float* dV, int B, int H, int Nq, int Nk,
                  int d, int causal, float scale, void* workspace, size_t workspace_size,
                  fa2_stream_t stream, bool f16) {
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0) return FA2_ERR_SHAPE;
  const long long BH = static_cast<long long>(B) * H;
  if (BH == 0 || (Nq == 0 && Nk == 0)) return FA2_OK;
  if (BH > 0x7fffffffLL) return FA2_ERR_SHAPE;
  if (Nq > 0 && Nk == 0) return FA2_ERR_SHAPE;
  if (d != 64 && d != 128) return FA2_ERR_HEADDIM;
  if (!(scale > 0.f) || !std::isfinite(scale)) return FA2_ERR_SCALE;
  if (!dK || !dV) return FA2_ERR_NULL;
  if (Nq > 0 && (!Q || !K || !V || !O || !dO || !LSE || !dQ || !workspace)) return FA2_ERR_NULL;
  const uintptr_t a16 = reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
                        reinterpret_cast<uintptr_t>(V) | reinterpret_cast<uintptr_t>(O) |
                        reinterpret_cast<uintptr_t>(dO) | reinterpret_cast<uintptr_t>(dQ) |
                        reinterpret_cast<uintptr_t>(dK) | reinterpret_cast<uintptr_t>(dV);
  if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(LSE) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return FA2_ERR_ALIGN;
  int rc = device_ready();
  if (rc != FA2_OK) return rc;
  const size_t bh = static_cast<size_t>(BH);
  const size_t q_elems = bh * Nq * d, kv_elems = bh * Nk * d;
  if (!device_range_ok(dK, kv_elems * 4) || !device_range_ok(dV, kv_elems * 4)) return FA2_ERR_MEMORY;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (Nq == 0) {
    // no query sees any key: the gradients of K and V are zero
    if (fa2host::launch_zero(dK, static_cast<long long>(kv_elems), s) != cudaSuccess ||
        fa2host::launch_zero(dV, static_cast<long long>(kv_elems), s) != cudaSuccess)
      return FA2_ERR_LAUNCH;
    return FA2_OK;
  }
  const size_t need = bwd_workspace_bytes(BH, Nq);
  if (!device_range_ok(Q, q_elems * 2) || !device_range_ok(K, kv_elems * 2) ||
      !device_range_ok(V, kv_elems * 2) || !device_range_ok(O, q_elems * 4) ||
      !device_range_ok(dO, q_elems * 2) || !device_range_ok(LSE, bh * Nq * 4) ||
      !device_range_ok(dQ, q_elems * 4) || workspace_size < need ||
      !device_range_ok(workspace, need))
    return FA2_ERR_MEMORY;

  // the two-tile kernel (64-row query tiles) for head dimension 128
  const bool two_tile = use_two_tile_backward(d);
  const unsigned qrows = two_tile ? 64 : 128;
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!encode_map(&mq, Q, d, Nq, static_cast<int>(BH), f16, qrows) ||
      !encode_map(&mk, K, d, Nk, static_cast<int>(BH), f16) ||
      !encode_map(&mv, V, d, Nk, static_cast<int>(BH), f16) ||
      !encode_map(&mdo, dO, d, Nq, static_cast<int>(BH), f16, qrows) ||
      !encode_map_f32(&mdq, dQ, d, Nq, static_cast<int>(BH), two_tile ? 32 : 128))
    return FA2_ERR_SHAPE;

  const int Nq_pad = (Nq + 127) / 128 * 128;
  float* L2 = static_cast<float*>(workspace);
  float* Dr = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(bh * Nq_pad * 4));
  if (fa2host::launch_bwd_pre(d, f16, O, dO, LSE, dQ, L2, Dr, static_cast<long long>(bh) * Nq, Nq, Nq_pad,
                              s) != cudaSuccess)
    return FA2_ERR_LAUNCH;

  fa2dev::BwdParams p;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.L2 = L2;
  p.Dr = Dr;
  p.Nq = Nq;
  p.Nk = Nk;
  p.Nq_pad = Nq_pad;
  p.BH = static_cast<int>(BH);
  p.key_blocks = key_tiles(Nk);
  // heads per scheduling group: their Q and dO tiles fit in kL2GroupBytes together
  const long long qd_bytes = 2LL * Nq * d * 2;
  long long g = kL2GroupBytes / (qd_bytes > 0 ? qd_bytes : 1);
  p.item_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.timeout_ns = kWaitTimeoutNs;
  p.status = status_word();
  if (p.status == nullptr) return FA2_ERR_LAUNCH;
  const long long grid = BH * p.key_blocks;
  if (grid > 0x7fffffffLL) return FA2_ERR_SHAPE;
  const cudaError_t e =
      two_tile ? fa2host::launch_bwd2(causal != 0, f16, mq, mk, mv, mdo, mdq, p, static_cast<unsigned>(grid), s)
               : fa2host::launch_bwd(d, causal != 0, f16, mq, mk, mv, mdo, mdq, p, static_cast<unsigned>(grid), s);
  return e == cudaSuccess ? FA2_OK : FA2_ERR_LAUNCH;
}

}  // namespace

extern "C" int fa2_backward(const void* Q, const void* K, const void* V, const float* O,
                            const void* dO, const float* LSE, float* dQ, float* dK, float* dV,
                            int B, int H, int Nq, int Nk, int d, int causal, float scale,
                            void* workspace, size_t workspace_size, fa2_stream_t stream) {
  return backward_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, workspace,
                       workspace_size, stream, false);
}

extern "C" int fa2_backward_typed(const void* Q, const void* K, const void* V, const float* O,
                                  const void* dO, const float* LSE, float* dQ, float* dK, float* dV,
                                  int B, int H, int Nq, int Nk, int d, int causal, float scale,
                                  int qkv_dtype, void* workspace, size_t workspace_size,
                                  fa2_stream_t stream) {
  if (qkv_dtype != FA2_DTYPE_BF16 && qkv_dtype != FA2_DTYPE_FP16) return FA2_ERR_DTYPE;
  return backward_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, Nq, Nk, d, causal, scale, workspace,
                       workspace_size, stream, qkv_dtype == FA2_DTYPE_FP16);
}

extern "C" const char* fa2_status_string(int status) {
  switch (status) {
    case FA2_OK: return "ok";
    case FA2_ERR_NULL: return "a required pointer is NULL";
    case FA2_ERR_ALIGN: return "Q/K/V/O must be 16-byte aligned and LSE 4-byte aligned";
    case FA2_ERR_SHAPE: return "invalid or unsupported sizes";
    case FA2_ERR_HEADDIM: return "unsupported head dimension (forward 64, 128 or 256; backward and SIMT 64 or 128)";
    case FA2_ERR_LAUNCH: return "CUDA launch or call failed";
    case FA2_ERR_TIMEOUT: return "a kernel gave up waiting on an internal barrier";
    case FA2_ERR_SCALE: return "scale must be finite and > 0";
    case FA2_ERR_MEMORY: return "a pointer is not device memory or its buffer is too small";
    case FA2_ERR_DEVICE: return "no usable sm_103 device is current";
    case FA2_ERR_SCRATCH: return "the problem needs more split-KV scratch than the library's 32 MiB static buffer";
    case FA2_ERR_DTYPE: return "unsupported element types (Q/K/V bf16 or fp16; O fp32 or the Q/K/V type)";
    default: return "unknown status";
  }
}

namespace fa2dev {

// One thread waits on an mbarrier that nothing completes, with the bounded
// wait of the pipeline kernels, and records the timeout as they do.
__global__ void fa2_wait_check_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    bar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
    if (!wait_bar(&bar, 0, &abort_flag, timeout_ns)) atomicOr(status, kDevErrTimeout);
  }
}

}  // namespace fa2dev

extern "C" int fa2_check_wait_timeout(unsigned long long timeout_ns, fa2_stream_t stream) {
  if (timeout_ns < 1000ull || timeout_ns > 10000000000ull) return FA2_ERR_SHAPE;
  const int rc = device_ready();
  if (rc != FA2_OK) return rc;
  int* status = status_word();
  if (status == nullptr) return FA2_ERR_LAUNCH;
  fa2dev::fa2_wait_check_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? FA2_OK : FA2_ERR_LAUNCH;
}

extern "C" int fa2_device_status(fa2_stream_t stream, int reset) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA2_ERR_LAUNCH;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return FA2_ERR_LAUNCH;
  if (reset) {
    const int z = 0;
    if (cudaMemcpyToSymbol(g_device_status, &z, sizeof z) != cudaSuccess) return FA2_ERR_LAUNCH;
  }
  return v ? FA2_ERR_TIMEOUT : FA2_OK;
}

// ---------------------------------------------------------------------------
// Split-KV forward whose scratch lives in the library, for callers that cannot
// allocate device memory themselves (see fa2_forward_splitkv_static in fa2.h).
//
// The scratch is one file-scope device array.  Host code must not pass the
// array's name to a kernel: on the host it is only a stand-in for the symbol.
// Its device address is looked up per device, with that device current, by
// the first call on the device (again by the next call if that lookup failed).  All calls share the array and it keeps
// the last call's contents; nothing in it needs to start at zero, because the
// partial-results kernel writes every entry the merge kernel reads.  Calls
// whose kernels overlap on the GPU (different streams, or different host
// threads) race on it.
namespace {

constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

// Device address of the array on the current device (nullptr on failure).
// Only a successful lookup is kept: a lookup that failed (for example one
// made during a stream capture) is retried by the next call, and its error
// is cleared so that it cannot surface in a later, unrelated check.
struct StaticScratch {
  std::mutex mu;
  void* ptr = nullptr;
};
StaticScratch g_static_scratch[kMaxDevices];

void* static_scratch_address(int dev) {
  StaticScratch& st = g_static_scratch[dev];
  std::lock_guard<std::mutex> lock(st.mu);
  if (st.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    st.ptr = p;
  }
  return st.ptr;
}

}  // namespace

extern "C" int fa2_forward_splitkv_static(const void* Q, const void* K, const void* V, float* O,
                                          float* LSE, int B, int H, int Nq, int Nk, int d,
                                          int causal, float scale, int num_splits,
                                          fa2_stream_t stream) {
  if (num_splits < 1 || num_splits > kMaxSplits) return FA2_ERR_SHAPE;
  Problem pr;
  int rc = validate(Q, K, V, O, LSE, B, H, Nq, Nk, d, scale, &pr);
  if (rc != FA2_OK || pr.empty) return rc;
  int splits = 1, tps = 1;
  split_plan(Nk, num_splits, &splits, &tps);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (splits == 1)
    return launch_forward(Q, K, V, O, LSE, pr, causal, scale, 1, tps, nullptr, nullptr, s);
  const size_t need = workspace_bytes(pr.BH, Nq, d, splits);
  if (need > kStaticScratchBytes) return FA2_ERR_SCRATCH;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_DEVICE;
  void* scratch = static_scratch_address(dev);
  if (scratch == nullptr) return FA2_ERR_LAUNCH;

  const size_t rows = static_cast<size_t>(pr.BH) * Nq;
  float* O_part = static_cast<float*>(scratch);
  float* LSE_part = reinterpret_cast<float*>(static_cast<char*>(scratch) +
                                             align256(static_cast<size_t>(splits) * rows * d * 4));
  rc = launch_forward(Q, K, V, O, LSE, pr, causal, scale, splits, tps, O_part, LSE_part, s);
  if (rc != FA2_OK) return rc;
  return fa2host::launch_combine(d, O_part, LSE_part, splits, static_cast<long long>(rows), O, LSE, s) ==
                 cudaSuccess
             ? FA2_OK
             : FA2_ERR_LAUNCH;
}

// ---------------------------------------------------------------------------
// Forward pass from host memory, pipelined over groups of heads: while one
// group computes, the next one's inputs are copied in and the previous one's
// outputs are copied out.  Three streams per device (copies in, compute,
// copies out) and their events are created by the first call on the device
// and kept; a mutex serialises the enqueueing so that two host threads do
// not interleave their event records.
namespace {

constexpr int kMaxChunks = 16;

struct HostPipe {
  std::mutex mu;
  bool ready = false;
  cudaStream_t in = nullptr, compute = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kMaxChunks] = {};
  cudaEvent_t computed[kMaxChunks] = {};
};
HostPipe g_pipes[kMaxDevices];

bool make_pipe(HostPipe& hp) {
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.compute, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.start, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.done, ef) == cudaSuccess;
  for (int c = 0; ok && c < kMaxChunks; ++c)
    ok = cudaEventCreateWithFlags(&hp.loaded[c], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.computed[c], ef) == cudaSuccess;
  if (!ok) cudaGetLastError();
  return ok;
}

}  // namespace

extern "C" int fa2_forward_host(const void* Qh, const void* Kh, const void* Vh, float* Oh, float* LSEh,
                                void* Qd, void* Kd, void* Vd, float* Od, float* LSEd, int B, int H,
                                int Nq, int Nk, int d, int causal, float scale, int chunks,
                                fa2_stream_t stream) {
  if (chunks < 1 || chunks > kMaxChunks) return FA2_ERR_SHAPE;
  Problem pr;
  int rc = validate(Qd, Kd, Vd, Od, LSEd, B, H, Nq, Nk, d, scale, &pr);
  if (rc != FA2_OK || pr.empty) return rc;
  if (!Qh || !Kh || !Vh || !Oh || !LSEh) return FA2_ERR_NULL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA2_ERR_DEVICE;
  HostPipe& hp = g_pipes[dev];
  std::lock_guard<std::mutex> lock(hp.mu);
  if (!hp.ready) {
    if (!make_pipe(hp)) return FA2_ERR_LAUNCH;
    hp.ready = true;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const long long BH = pr.BH;
  const int n = static_cast<int>(chunks < BH ? chunks : BH);
  // Head groups weighted min(c + 1, n - c): small groups at both ends shorten
  // the copy-in before the first computation and the computation and
  // copy-out after the last copy-in, larger ones in the middle keep each
  // launch big enough to fill the GPU.  Group c covers heads
  // [first(c), first(c + 1)), each at least one head.
  long long wsum = 0;
  for (int c = 0; c < n; ++c) wsum += (c + 1 < n - c ? c + 1 : n - c);
  auto first = [&](int c) -> long long {
    long long w = 0;
    for (int i = 0; i < c; ++i) w += (i + 1 < n - i ? i + 1 : n - i);
    long long h = (BH * w + wsum / 2) / wsum;
    if (h < c) h = c;                         // at least one head per earlier group
    if (h > BH - (n - c)) h = BH - (n - c);   // at least one head per later group
    return h;
  };
  // the pipeline starts after the work already queued on the caller's stream
  bool ok = cudaEventRecord(hp.start, s) == cudaSuccess &&
            cudaStreamWaitEvent(hp.in, hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.compute, hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.out, hp.start, 0) == cudaSuccess;
  const size_t q_head = static_cast<size_t>(Nq) * d, kv_head = static_cast<size_t>(Nk) * d;
  for (int c = 0; c < n && ok; ++c) {
    const long long h0 = first(c), h1 = c + 1 < n ? first(c + 1) : BH;
    const size_t nh = static_cast<size_t>(h1 - h0), off = static_cast<size_t>(h0);
    const char* qh = static_cast<const char*>(Qh) + off * q_head * 2;
    const char* kh = static_cast<const char*>(Kh) + off * kv_head * 2;
    const char* vh = static_cast<const char*>(Vh) + off * kv_head * 2;
    char* qd = static_cast<char*>(Qd) + off * q_head * 2;
    char* kd = static_cast<char*>(Kd) + off * kv_head * 2;
    char* vd = static_cast<char*>(Vd) + off * kv_head * 2;
    ok = cudaMemcpyAsync(qd, qh, nh * q_head * 2, cudaMemcpyDefault, hp.in) == cudaSuccess &&
         cudaMemcpyAsync(kd, kh, nh * kv_head * 2, cudaMemcpyDefault, hp.in) == cudaSuccess &&
         cudaMemcpyAsync(vd, vh, nh * kv_head * 2, cudaMemcpyDefault, hp.in) == cudaSuccess &&
         cudaEventRecord(hp.loaded[c], hp.in) == cudaSuccess &&
         cudaStreamWaitEvent(hp.compute, hp.loaded[c], 0) == cudaSuccess;
    if (!ok) break;
    Problem sub = pr;
    sub.B = 1;
    sub.H = static_cast<int>(nh);
    sub.BH = static_cast<long long>(nh);
    float* od = Od + off * q_head;
    float* ld = LSEd + off * static_cast<size_t>(Nq);
    rc = launch_forward(qd, kd, vd, od, ld, sub, causal, scale, 1, key_tiles(Nk), nullptr, nullptr,
                        hp.compute);
    if (rc != FA2_OK) break;
    ok = cudaEventRecord(hp.computed[c], hp.compute) == cudaSuccess &&
         cudaStreamWaitEvent(hp.out, hp.computed[c], 0) == cudaSuccess &&
         cudaMemcpyAsync(Oh + off * q_head, od, nh * q_head * 4, cudaMemcpyDefault, hp.out) == cudaSuccess &&
         cudaMemcpyAsync(LSEh + off * Nq, ld, nh * static_cast<size_t>(Nq) * 4, cudaMemcpyDefault,
                         hp.out) == cudaSuccess;
  }
  // Join: the caller's stream continues after everything enqueued above
  // (the copies out follow every computation, which follow every copy in).
  const bool joined = cudaEventRecord(hp.done, hp.out) == cudaSuccess &&
                      cudaStreamWaitEvent(s, hp.done, 0) == cudaSuccess;
  if (rc != FA2_OK) return rc;
  if (!ok || !joined) {
    cudaGetLastError();
    return FA2_ERR_LAUNCH;
  }
  return FA2_OK;
}
