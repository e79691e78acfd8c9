// Host side of the C ABI declared in include/fa.h: argument validation, TMA
// descriptor construction and the launch of the fused attention kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_splitkv.cuh"

namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 1000000000ull;
constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_wait_limit_ns{kDefaultWaitLimitNs};
std::atomic<unsigned int> g_inject{0u};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

// Per-device readiness: 0 = unchecked, 1 = supported and configured, -1 = unsupported.
std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices] = {0};
int g_dev_sms[kMaxDevices] = {0};  // multiprocessor count of each configured device

void load_encode() {
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  void* fn = nullptr;
  g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                  cudaEnableDefault, &q);
  if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess && fn != nullptr)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

// Sets the dynamic shared-memory size, and checks that the kernel was built
// with exactly the per-thread register count its setmaxnreg split assumes
// (a different count could leave the softmax warpgroups waiting for
// registers that the pool does not hold).
template <int D, bool kNeg>
cudaError_t configure_kernel() {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, fa::fa_fwd_kernel<D, kNeg>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != static_cast<int>(fa::kLaunchRegs)) return cudaErrorInvalidKernelImage;
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, kNeg>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::Cfg<D>::kSmemAlloc));
}

template <int D>
cudaError_t configure_split_kernel() {
  return cudaFuncSetAttribute(fa::fa_splitkv_partial_kernel<D>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::SplitCfg<D>::kSmemAlloc));
}

// Checks that the current device is sm_103 and configures the kernels for it once.
int prepare_device(int* dev_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_LAUNCH;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_DEVICE;
  *dev_out = dev;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] == 1) {
    *sms_out = g_dev_sms[dev];
    return FA_OK;
  }
  if (g_dev_state[dev] == -1) return FA_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (major != 10 || minor != 3) {
    g_dev_state[dev] = -1;
    return FA_ERR_DEVICE;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return FA_ERR_LAUNCH;
  if (configure_kernel<64, false>() != cudaSuccess || configure_kernel<64, true>() != cudaSuccess ||
      configure_kernel<128, false>() != cudaSuccess || configure_kernel<128, true>() != cudaSuccess ||
      configure_split_kernel<64>() != cudaSuccess || configure_split_kernel<128>() != cudaSuccess)
    return FA_ERR_LAUNCH;
  g_dev_sms[dev] = sms;
  *sms_out = sms;
  g_dev_state[dev] = 1;
  return FA_OK;
}

// [BH][N][d] bf16 viewed as a 3-D tensor (d innermost), boxes of
// 64 columns x `box_rows` rows x 1 slice with the 128-byte swizzle.
bool encode_map(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r =
      g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
               elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

// Persistent launch: one CTA per multiprocessor (at most one per work unit);
// each CTA walks its share of the units inside the kernel.
template <int D, bool kNeg>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
           const fa::FwdParams& prm, int sms, cudaStream_t stream) {
  const unsigned ctas = static_cast<unsigned>(prm.total_units < sms ? prm.total_units : sms);
  fa::fa_fwd_kernel<D, kNeg><<<ctas, fa::kNumThreads, fa::Cfg<D>::kSmemAlloc, stream>>>(
      mq, mk, mv, prm);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int N, int d, int causal, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t num_units = (static_cast<int64_t>(N) + fa::kUnitM - 1) / fa::kUnitM;
  // Work units (B*H x 256-row query units) are counted in int, and so are
  // the row offsets bh*N + row of the LSE store.
  if (BH > INT_MAX || BH * num_units > INT_MAX || BH * N > INT_MAX) return FA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) &
      15u)
    return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  const size_t tensor_bytes = static_cast<size_t>(BH) * N * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * N * 4;
  for (const void* in : {q, k, v}) {
    if (overlaps(o, tensor_bytes, in, tensor_bytes) || overlaps(lse, lse_bytes, in, tensor_bytes))
      return FA_ERR_ALIAS;
  }
  if (overlaps(o, tensor_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;

  CUtensorMap mq, mk, mv;
  if (!encode_map(&mq, q, static_cast<int>(BH), N, d) ||
      !encode_map(&mk, k, static_cast<int>(BH), N, d) ||
      !encode_map(&mv, v, static_cast<int>(BH), N, d))
    return FA_ERR_LAUNCH;

  fa::FwdParams prm;
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  prm.N = N;
  prm.num_bh = static_cast<int>(BH);
  prm.num_units = static_cast<int>(num_units);
  prm.total_units = static_cast<int>(BH * num_units);
  prm.causal = causal;
  // scale * log2(e).  A zero scale is passed as 1e-30: every scaled score is
  // then below 1e-25 in magnitude, so 2^x rounds to exactly 1 in fp32 as for
  // a true zero, while a masked score (-inf) still maps to -inf.
  double c = static_cast<double>(scale) * 1.4426950408889634;
  if (c == 0.0) c = 1e-30;
  prm.scale_log2 = static_cast<float>(c);
  prm.inject = g_inject.load(std::memory_order_relaxed);
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool neg = prm.scale_log2 < 0.0f;
  if (d == 64)
    return neg ? launch<64, true>(mq, mk, mv, prm, sms, s) : launch<64, false>(mq, mk, mv, prm, sms, s);
  return neg ? launch<128, true>(mq, mk, mv, prm, sms, s) : launch<128, false>(mq, mk, mv, prm, sms, s);
}

// ---------------------------------------------------------------- split-KV

namespace {

constexpr size_t kWsAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Effective split count and keys per split: the requested count, or (0) the
// largest count whose CTAs all fit in one wave (kSplitCtasPerSm per
// multiprocessor), at least 1; capped by the number of 64-key tiles and by
// kSplitMaxSplits.  Every split covers a multiple of 64 keys except the last.
void split_geometry(int64_t BH, int Nk, int requested, int sms, int* splits, int* keys_per_split) {
  const int tiles = (Nk + fa::kSplitTileKeys - 1) / fa::kSplitTileKeys;
  int s = requested;
  if (s <= 0) {
    const int64_t slots = static_cast<int64_t>(fa::kSplitCtasPerSm) * sms;
    s = static_cast<int>(slots / BH < fa::kSplitMaxSplits ? slots / BH : fa::kSplitMaxSplits);
  }
  if (s > tiles) s = tiles;
  if (s > fa::kSplitMaxSplits) s = fa::kSplitMaxSplits;
  if (s < 1) s = 1;
  const int tiles_per_split = (tiles + s - 1) / s;
  *keys_per_split = tiles_per_split * fa::kSplitTileKeys;
  *splits = (tiles + tiles_per_split - 1) / tiles_per_split;
}

size_t split_ws_bytes(int splits, int64_t BH, int Nq, int d) {
  const size_t rows = static_cast<size_t>(splits) * BH * Nq;
  return round_up(rows * d * 4, kWsAlign) + round_up(rows * 4, kWsAlign);
}

int split_shape_ok(int B, int H, int Nq, int Nk, int d, int causal, int num_splits) {
  if (B <= 0 || H <= 0 || Nq <= 0 || Nk <= 0) return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
  if (Nq > fa::kSplitMaxQ || num_splits < 0 || num_splits > fa::kSplitMaxSplits)
    return FA_ERR_SHAPE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  if (causal && Nq > Nk) return FA_ERR_SHAPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > 65535 || BH * Nk > INT_MAX || BH * Nq > INT_MAX) return FA_ERR_SHAPE;
  return FA_OK;
}

// Split count the library uses for a request on the current device.
int current_sms() {
  int dev = 0, sms = 0;
  if (prepare_device(&dev, &sms) != FA_OK) return 0;
  return sms;
}

template <int D>
int launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const fa::SplitParams& prm,
                 cudaStream_t stream) {
  const dim3 grid1(static_cast<unsigned>(prm.splits), static_cast<unsigned>(prm.num_bh));
  fa::fa_splitkv_partial_kernel<D>
      <<<grid1, fa::kSplitThreads, fa::SplitCfg<D>::kSmemAlloc, stream>>>(mk, mv, prm);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  const unsigned rows = static_cast<unsigned>(prm.num_bh * prm.Nq);
  fa::fa_splitkv_combine_kernel<D><<<(rows + 7) / 8, 256, 0, stream>>>(prm);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (split_shape_ok(B, H, Nq, Nk, d, 0, num_splits) != FA_OK) return 0;
  const int sms = num_splits > 0 ? 1 : current_sms();
  if (sms <= 0) return 0;
  int splits = 0, kps = 0;
  split_geometry(static_cast<int64_t>(B) * H, Nk, num_splits, sms, &splits, &kps);
  return splits;
}

extern "C" size_t fa_fwd_splitkv_workspace_bytes(int B, int H, int Nq, int Nk, int d,
                                                 int num_splits) {
  const int splits = fa_fwd_splitkv_num_splits(B, H, Nq, Nk, d, num_splits);
  if (splits <= 0) return 0;
  return split_ws_bytes(splits, static_cast<int64_t>(B) * H, Nq, d);
}

extern "C" int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H, int Nq, int Nk, int d, int causal, float scale,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  const int shape = split_shape_ok(B, H, Nq, Nk, d, causal, num_splits);
  if (shape != FA_OK) return shape;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
       reinterpret_cast<uintptr_t>(workspace)) &
      15u)
    return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const size_t q_bytes = static_cast<size_t>(BH) * Nq * d * 2;
  const size_t kv_bytes = static_cast<size_t>(BH) * Nk * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * Nq * 4;
  for (const void* in : {q, k, v}) {
    const size_t n = (in == q) ? q_bytes : kv_bytes;
    if (overlaps(o, q_bytes, in, n) || overlaps(lse, lse_bytes, in, n)) return FA_ERR_ALIAS;
  }
  if (overlaps(o, q_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  int splits = 0, kps = 0;
  split_geometry(BH, Nk, num_splits, sms, &splits, &kps);
  const size_t need = split_ws_bytes(splits, BH, Nq, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  for (const void* other : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse)}) {
    const size_t n = other == q || other == o ? q_bytes : other == lse ? lse_bytes : kv_bytes;
    if (overlaps(workspace, need, other, n)) return FA_ERR_ALIAS;
  }

  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;
  CUtensorMap mk, mv;
  if (!encode_map(&mk, k, static_cast<int>(BH), Nk, d, fa::kSplitTileKeys) ||
      !encode_map(&mv, v, static_cast<int>(BH), Nk, d, fa::kSplitTileKeys))
    return FA_ERR_LAUNCH;

  fa::SplitParams prm;
  prm.q = static_cast<const uint16_t*>(q);
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  const size_t rows = static_cast<size_t>(splits) * BH * Nq;
  prm.ws_o = static_cast<float*>(workspace);
  prm.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        round_up(rows * d * 4, kWsAlign));
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.num_bh = static_cast<int>(BH);
  prm.splits = splits;
  prm.keys_per_split = kps;
  prm.causal = causal;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_split<64>(mk, mv, prm, s) : launch_split<128>(mk, mv, prm, s);
}

// ----------------------------------------------------------------------------
// fa_fwd_splitkv_static: the split-KV path with its scratch in a buffer that
// is part of the library, for callers that cannot allocate device memory
// (code running inside a memory pool or arena that owns all device memory,
// real-time or capture-time callers for which a cudaMalloc's implicit
// synchronisation or failure is not acceptable, plug-ins whose host gives
// them no allocator).
//
// The buffer is a file-scope device array: every GPU that loads this library
// holds kStaticScratchBytes of it until the process exits.  Its name is only
// a host-side handle; the device address comes from cudaGetSymbolAddress,
// taken once per device (with that device current) on the first call there.
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_splitkv_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on `dev` (the current device).
int static_scratch(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_LAUNCH;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return FA_OK;
}

}  // namespace

extern "C" size_t fa_fwd_splitkv_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" int fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int H, int Nq, int Nk, int d, int causal,
                                     float scale, int num_splits, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  const int shape = split_shape_ok(B, H, Nq, Nk, d, causal, num_splits);
  if (shape != FA_OK) return shape;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) &
      15u)
    return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const size_t q_bytes = static_cast<size_t>(BH) * Nq * d * 2;
  const size_t kv_bytes = static_cast<size_t>(BH) * Nk * d * 2;
  const size_t lse_bytes = static_cast<size_t>(BH) * Nq * 4;
  for (const void* in : {q, k, v}) {
    const size_t n = (in == q) ? q_bytes : kv_bytes;
    if (overlaps(o, q_bytes, in, n) || overlaps(lse, lse_bytes, in, n)) return FA_ERR_ALIAS;
  }
  if (overlaps(o, q_bytes, lse, lse_bytes)) return FA_ERR_ALIAS;

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  int splits = 0, kps = 0;
  split_geometry(BH, Nk, num_splits, sms, &splits, &kps);
  if (split_ws_bytes(splits, BH, Nq, d) > kStaticScratchBytes) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int got = static_scratch(dev, &scratch);
  if (got != FA_OK) return got;

  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;
  CUtensorMap mk, mv;
  if (!encode_map(&mk, k, static_cast<int>(BH), Nk, d, fa::kSplitTileKeys) ||
      !encode_map(&mv, v, static_cast<int>(BH), Nk, d, fa::kSplitTileKeys))
    return FA_ERR_LAUNCH;

  // Nothing in the scratch has to start at zero: pass 1 writes every partial
  // output and log-sum-exp that pass 2 reads.
  fa::SplitParams prm;
  prm.q = static_cast<const uint16_t*>(q);
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  const size_t rows = static_cast<size_t>(splits) * BH * Nq;
  prm.ws_o = static_cast<float*>(scratch);
  prm.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                        round_up(rows * d * 4, kWsAlign));
  prm.Nq = Nq;
  prm.Nk = Nk;
  prm.num_bh = static_cast<int>(BH);
  prm.splits = splits;
  prm.keys_per_split = kps;
  prm.causal = causal;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_split<64>(mk, mv, prm, s) : launch_split<128>(mk, mv, prm, s);
}

extern "C" const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid shape (B, H, N must be >= 1 and within index limits; causal 0 or 1)";
    case FA_ERR_HEAD_DIM: return "unsupported head dimension (d must be 64 or 128)";
    case FA_ERR_ALIGN: return "misaligned pointer (q, k, v, o need 16 bytes; lse needs 4)";
    case FA_ERR_SCALE: return "scale is not finite";
    case FA_ERR_ALIAS: return "an output overlaps an input or the other output";
    case FA_ERR_DEVICE: return "current device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "CUDA error while preparing or launching the kernel";
    case FA_ERR_TIMEOUT: return "a kernel wait exceeded its time limit";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_fwd_splitkv_workspace_bytes()";
    case FA_ERR_SCRATCH_LIMIT:
      return "request needs more scratch than fa_fwd_splitkv_static's built-in buffer holds "
             "(see fa_fwd_splitkv_static_scratch_bytes(); use fa_fwd_splitkv with a workspace)";
    default: return "unknown error code";
  }
}

extern "C" int fa_get_device_status(unsigned int* status) {
  if (!status) return FA_ERR_NULL;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, fa::g_fa_status, sizeof v) != cudaSuccess) return FA_ERR_LAUNCH;
  *status = v;
  return FA_OK;
}

extern "C" int fa_clear_device_status(void) {
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof zero) == cudaSuccess ? FA_OK
                                                                               : FA_ERR_LAUNCH;
}

extern "C" int fa_set_wait_limit_ns(unsigned long long ns) {
  g_wait_limit_ns.store(ns == 0 ? kDefaultWaitLimitNs : ns, std::memory_order_relaxed);
  return FA_OK;
}

extern "C" int fa_set_fault_injection(unsigned int flags) {
  g_inject.store(flags, std::memory_order_relaxed);
  return FA_OK;
}

extern "C" int fa_version(void) { return 100; }
