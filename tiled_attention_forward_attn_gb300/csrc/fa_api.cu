// Host side of the C ABI declared in include/fa.h: argument validation, TMA
// descriptor construction and the launch of the fused attention kernel.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_fwd_d256.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_order_ablation.cuh"
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
template <int D, bool kNeg, bool kF16, bool kPartialD>
cudaError_t configure_kernel() {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, fa::fa_fwd_kernel<D, kNeg, kF16, kPartialD>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != static_cast<int>(fa::kLaunchRegs)) return cudaErrorInvalidKernelImage;
  return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, kNeg, kF16, kPartialD>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::Cfg<D>::kSmemAlloc));
}

template <int D, bool kF16, bool kPartialD>
bool configure_both_signs() {
  return configure_kernel<D, false, kF16, kPartialD>() == cudaSuccess &&
         configure_kernel<D, true, kF16, kPartialD>() == cudaSuccess;
}

template <bool kNeg, bool kF16>
cudaError_t configure_d256() {
  return cudaFuncSetAttribute(fa::fa_fwd_d256_kernel<kNeg, kF16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::WideCfg::kSmemAlloc));
}

template <int D>
bool configure_dim() {
  return configure_both_signs<D, false, false>() && configure_both_signs<D, true, false>() &&
         configure_both_signs<D, false, true>() && configure_both_signs<D, true, true>();
}

// As for the forward: the register split (setmaxnreg) assumes the launch
// register count.
template <int D, bool kKV, bool kF16>
cudaError_t configure_bwd_one() {
  cudaFuncAttributes attr;
  cudaError_t e = cudaFuncGetAttributes(&attr, fa::fa_bwd_kernel<D, kKV, kF16>);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != static_cast<int>(fa::kBwdLaunchRegs)) return cudaErrorInvalidKernelImage;
  return cudaFuncSetAttribute(fa::fa_bwd_kernel<D, kKV, kF16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::BwdCfg<D, kKV>::kSmemAlloc));
}

template <int D, bool kKV>
cudaError_t configure_bwd_kernel() {
  const cudaError_t e = configure_bwd_one<D, kKV, false>();
  return e != cudaSuccess ? e : configure_bwd_one<D, kKV, true>();
}

template <int D, bool kV1>
cudaError_t configure_order_kernel() {
  return cudaFuncSetAttribute(fa::fa_order_kernel<D, kV1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(fa::OrdCfg<D, kV1>::kSmemAlloc));
}

template <int D>
cudaError_t configure_split_kernel() {
  cudaError_t e = cudaFuncSetAttribute(fa::fa_splitkv_partial_kernel<D, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(fa::SplitCfg<D>::kSmemAlloc));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa::fa_splitkv_partial_kernel<D, true>,
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
  if (!configure_dim<64>() || !configure_dim<128>() ||
      configure_d256<false, false>() != cudaSuccess || configure_d256<true, false>() != cudaSuccess ||
      configure_d256<false, true>() != cudaSuccess || configure_d256<true, true>() != cudaSuccess ||
      configure_split_kernel<64>() != cudaSuccess || configure_split_kernel<128>() != cudaSuccess ||
      configure_bwd_kernel<64, true>() != cudaSuccess ||
      configure_bwd_kernel<64, false>() != cudaSuccess ||
      configure_bwd_kernel<128, true>() != cudaSuccess ||
      configure_bwd_kernel<128, false>() != cudaSuccess ||
      configure_order_kernel<64, true>() != cudaSuccess ||
      configure_order_kernel<64, false>() != cudaSuccess ||
      configure_order_kernel<128, true>() != cudaSuccess ||
      configure_order_kernel<128, false>() != cudaSuccess)
    return FA_ERR_LAUNCH;
  g_dev_sms[dev] = sms;
  *sms_out = sms;
  g_dev_state[dev] = 1;
  return FA_OK;
}

// Contiguous [BH][N][d] bf16 viewed as a 3-D tensor (d innermost), boxes of
// 64 columns x `box_rows` rows x 1 slice with the 128-byte swizzle (split-KV).
bool encode_map(CUtensorMap* map, const void* ptr, int BH, int N, int d, int box_rows = 128,
                CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t elem_strides[3] = {1, 1, 1};
  const CUresult r =
      g_encode(map, type, 3, const_cast<void*>(ptr), dims, strides, box,
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
template <int D, bool kNeg, bool kF16, bool kPartialD>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
           const fa::FwdParams& prm, int sms, cudaStream_t stream) {
  const unsigned ctas = static_cast<unsigned>(prm.total_units < sms ? prm.total_units : sms);
  fa::fa_fwd_kernel<D, kNeg, kF16, kPartialD>
      <<<ctas, fa::kNumThreads, fa::Cfg<D>::kSmemAlloc, stream>>>(mq, mk, mv, prm);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

template <bool kF16>
int launch_d256(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const fa::FwdParams& prm, int sms, cudaStream_t stream) {
  const unsigned ctas = static_cast<unsigned>(prm.total_units < sms ? prm.total_units : sms);
  if (prm.scale_log2 < 0.0f)
    fa::fa_fwd_d256_kernel<true, kF16><<<ctas, fa::kW_Threads, fa::WideCfg::kSmemAlloc, stream>>>(
        mq, mk, mv, prm);
  else
    fa::fa_fwd_d256_kernel<false, kF16><<<ctas, fa::kW_Threads, fa::WideCfg::kSmemAlloc, stream>>>(
        mq, mk, mv, prm);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

template <int D, bool kF16, bool kPartialD>
int launch_sign(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                const fa::FwdParams& prm, int sms, cudaStream_t stream) {
  return prm.scale_log2 < 0.0f ? launch<D, true, kF16, kPartialD>(mq, mk, mv, prm, sms, stream)
                               : launch<D, false, kF16, kPartialD>(mq, mk, mv, prm, sms, stream);
}

// [B][H][N][d] view with element strides (sb, sh, sn) and unit column stride,
// as a 4-D tensor map {d, N, H, B}: boxes of 64 columns x 128 rows x 1 x 1
// with the 128-byte swizzle; columns past d and rows past N read as zero.
bool encode_map4(CUtensorMap* map, const void* ptr, CUtensorMapDataType type, int B, int H, int N,
                 int d, const int64_t* st, int box_rows = 128) {
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(B)};
  // A dimension of extent 1 is never stepped; give it a harmless stride.
  auto stride = [&](int i, int extent) -> cuuint64_t {
    const int64_t bytes = st[i] * 2;
    return static_cast<cuuint64_t>(extent == 1 && bytes == 0 ? 16 : bytes);
  };
  const cuuint64_t strides[3] = {stride(2, N), stride(1, H), stride(0, B)};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, 1};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  const CUresult r =
      g_encode(map, type, 4, const_cast<void*>(ptr), dims, strides, box, elem_strides,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Whether the element span of a strided [B][H][N][d] tensor stays below
// 2^55 elements (64 PiB of 2-byte elements), so that every later span,
// overlap and kernel address computation is exact in int64.  Each product is
// checked before it is formed.
bool span_in_range(int B, int H, int N, int d, const int64_t* st) {
  constexpr int64_t kLimit = int64_t(1) << 55;
  const int64_t ext[3] = {B, H, N};
  int64_t total = d;
  for (int i = 0; i < 3; ++i) {
    const int64_t n1 = ext[i] - 1;
    if (n1 > 0 && st[i] > (kLimit - total) / n1) return false;
    total += n1 * st[i];
  }
  return true;
}

// Bytes from the first to one past the last element of a strided
// [B][H][N][d] tensor of 2-byte elements (span_in_range must hold).
size_t span_bytes(int B, int H, int N, int d, const int64_t* st) {
  const int64_t last = (B - 1) * st[0] + (H - 1) * st[1] + (N - 1) * st[2] + d;
  return static_cast<size_t>(last) * 2;
}

// Whether distinct (b, h, row, col) of a strided [B][H][N][d] tensor with
// unit column stride map to distinct addresses: with the dimensions of
// extent > 1 sorted by stride, each stride must step over the whole extent
// of the ones below it.
bool strides_disjoint(int B, int H, int N, int d, const int64_t* st) {
  int64_t s[3] = {st[0], st[1], st[2]};
  int64_t n[3] = {B, H, N};
  for (int i = 0; i < 3; ++i)
    for (int j = i + 1; j < 3; ++j)
      if (s[j] < s[i]) {
        const int64_t ts = s[i], tn = n[i];
        s[i] = s[j];
        n[i] = n[j];
        s[j] = ts;
        n[j] = tn;
      }
  int64_t covered = d;  // extent of the dimensions below, in elements
  for (int i = 0; i < 3; ++i) {
    if (n[i] == 1) continue;
    if (s[i] < covered) return false;
    covered = s[i] * (n[i] - 1) + covered;
  }
  return true;
}

int fwd_impl(const void* q, const int64_t* qs_in, const void* k, const int64_t* ks_in,
             const void* v, const int64_t* vs_in, void* o, const int64_t* os_in, float* lse,
             int dtype, int B, int H, int N, int d, int causal, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_SHAPE;
  if (d != 256 && (d < 16 || d > 128 || d % 16 != 0)) return FA_ERR_HEAD_DIM;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_DTYPE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  // Work units: 256-row query units, or single 128-row query tiles at d = 256.
  const int64_t unit_rows = d == 256 ? fa::kW_TileM : fa::kUnitM;
  const int64_t num_units = (static_cast<int64_t>(N) + unit_rows - 1) / unit_rows;
  // Work units (B*H x 256-row query units) are counted in int, and so are
  // the row offsets bh*N + row of the LSE store.
  if (BH > INT_MAX || BH * num_units > INT_MAX || BH * N > INT_MAX) return FA_ERR_SHAPE;
  const int64_t contig[3] = {static_cast<int64_t>(H) * N * d, static_cast<int64_t>(N) * d, d};
  const int64_t* qs = qs_in ? qs_in : contig;
  const int64_t* ks = ks_in ? ks_in : contig;
  const int64_t* vs = vs_in ? vs_in : contig;
  const int64_t* os = os_in ? os_in : contig;
  for (const int64_t* st : {qs, ks, vs, os}) {
    for (int i = 0; i < 3; ++i)
      if (st[i] < 0 || st[i] % 8 != 0 || st[i] >= (int64_t(1) << 38)) return FA_ERR_STRIDE;
    if (!span_in_range(B, H, N, d, st)) return FA_ERR_STRIDE;
  }
  if (!strides_disjoint(B, H, N, d, os)) return FA_ERR_STRIDE;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o)) &
      15u)
    return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  const size_t o_span = span_bytes(B, H, N, d, os);
  const size_t lse_bytes = static_cast<size_t>(BH) * N * 4;
  const void* ins[3] = {q, k, v};
  const int64_t* in_st[3] = {qs, ks, vs};
  for (int i = 0; i < 3; ++i) {
    const size_t n = span_bytes(B, H, N, d, in_st[i]);
    if (overlaps(o, o_span, ins[i], n) || overlaps(lse, lse_bytes, ins[i], n)) return FA_ERR_ALIAS;
  }
  if (overlaps(o, o_span, lse, lse_bytes)) return FA_ERR_ALIAS;

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;

  const CUtensorMapDataType tt =
      dtype == FA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // d = 256 streams 64-key K/V tiles; otherwise 128-key tiles.
  const int kv_rows = d == 256 ? fa::kW_BlockN : 128;
  CUtensorMap mq, mk, mv;
  if (!encode_map4(&mq, q, tt, B, H, N, d, qs) ||
      !encode_map4(&mk, k, tt, B, H, N, d, ks, kv_rows) ||
      !encode_map4(&mv, v, tt, B, H, N, d, vs, kv_rows))
    return FA_ERR_LAUNCH;

  const bool f16 = dtype == FA_DTYPE_FP16;
  fa::FwdParams prm;
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  prm.o_sb = os[0];
  prm.o_sh = os[1];
  prm.o_sn = os[2];
  prm.o_vec32 = (reinterpret_cast<uintptr_t>(o) % 32 == 0 && os[0] % 16 == 0 && os[1] % 16 == 0 &&
                 os[2] % 16 == 0)
                    ? 1
                    : 0;
  prm.N = N;
  prm.H = H;
  prm.d = d;
  prm.k_slices = d / 16;
  prm.idesc_pv = f16 ? fa::idesc_f16_f32(fa::kTileM, static_cast<uint32_t>(d), 0, 1)
                     : fa::idesc_bf16_f32(fa::kTileM, static_cast<uint32_t>(d), 0, 1);
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

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (d == 256)
    return f16 ? launch_d256<true>(mq, mk, mv, prm, sms, st) : launch_d256<false>(mq, mk, mv, prm, sms, st);
  if (d == 128)
    return f16 ? launch_sign<128, true, false>(mq, mk, mv, prm, sms, st)
               : launch_sign<128, false, false>(mq, mk, mv, prm, sms, st);
  if (d == 64)
    return f16 ? launch_sign<64, true, false>(mq, mk, mv, prm, sms, st)
               : launch_sign<64, false, false>(mq, mk, mv, prm, sms, st);
  if (d > 64)
    return f16 ? launch_sign<128, true, true>(mq, mk, mv, prm, sms, st)
               : launch_sign<128, false, true>(mq, mk, mv, prm, sms, st);
  return f16 ? launch_sign<64, true, true>(mq, mk, mv, prm, sms, st)
             : launch_sign<64, false, true>(mq, mk, mv, prm, sms, st);
}

}  // namespace

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                      int N, int d, int causal, float scale, void* stream) {
  return fwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, FA_DTYPE_BF16, B, H, N, d,
                  causal, scale, stream);
}

namespace {

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0) return 0;
  if (d != 256 && (d < 16 || d > 128 || d % 16 != 0)) return 0;
  if (static_cast<int64_t>(B) * H * N > INT_MAX) return 0;  // as fa_fwd_host rejects
  const size_t rows = static_cast<size_t>(B) * H * N;
  return 4 * round256(rows * d * 2) + round256(rows * 4);
}

extern "C" int fa_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                           void* o_host, float* lse_host, int dtype, int B, int H, int N, int d,
                           int causal, float scale, void* workspace, size_t workspace_bytes,
                           void* stream) {
  // Everything fa_fwd would reject is rejected here, before any copy is queued.
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return FA_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_SHAPE;
  if (d != 256 && (d < 16 || d > 128 || d % 16 != 0)) return FA_ERR_HEAD_DIM;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_DTYPE;
  if (causal != 0 && causal != 1) return FA_ERR_SHAPE;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t unit_rows = d == 256 ? fa::kW_TileM : fa::kUnitM;
  const int64_t num_units = (static_cast<int64_t>(N) + unit_rows - 1) / unit_rows;
  if (BH > INT_MAX || BH * num_units > INT_MAX || BH * N > INT_MAX) return FA_ERR_SHAPE;
  const size_t need = fa_fwd_host_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(BH) * N * d * 2;
  const size_t lb = static_cast<size_t>(BH) * N * 4;
  // The outputs overlap neither an input nor each other (host ranges).
  const void* hin[3] = {q_host, k_host, v_host};
  for (int i = 0; i < 3; ++i)
    if (overlaps(o_host, tb, hin[i], tb) || overlaps(lse_host, lb, hin[i], tb)) return FA_ERR_ALIAS;
  if (overlaps(o_host, tb, lse_host, lb)) return FA_ERR_ALIAS;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t t = round256(tb);
  void* qd = ws;
  void* kd = ws + t;
  void* vd = ws + 2 * t;
  void* od = ws + 3 * t;
  float* ld = reinterpret_cast<float*>(ws + 4 * t);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(qd, q_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(kd, k_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(vd, v_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const int rc = fwd_impl(qd, nullptr, kd, nullptr, vd, nullptr, od, nullptr, ld, dtype, B, H, N,
                          d, causal, scale, stream);
  if (rc != FA_OK) return rc;
  if (cudaMemcpyAsync(o_host, od, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, ld, lb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

extern "C" int fa_fwd_strided(const void* q, const int64_t* q_strides, const void* k,
                              const int64_t* k_strides, const void* v, const int64_t* v_strides,
                              void* o, const int64_t* o_strides, float* lse, int dtype, int B,
                              int H, int N, int d, int causal, float scale, void* stream) {
  return fwd_impl(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, dtype, B, H, N, d,
                  causal, scale, stream);
}

// ---------------------------------------------------------------- backward

namespace {

int64_t bwd_npad(int N) { return (static_cast<int64_t>(N) + fa::kBwdTile - 1) / fa::kBwdTile * fa::kBwdTile; }

// Three launches on one stream: D and LSE*log2(e) into the workspace, the
// dK/dV pass (prm_kv: out0 = dK, out1 = dV), the dQ pass (prm_q: out0 = dQ).
// mX: 128-row boxes (stationary tiles); mX64: 64-row boxes (streamed halves).
// Inputs of the D pre-pass: O and dO at their element strides
// (batch, head, row), and the forward's LSE.
struct BwdPrepIn {
  const void* o;
  const int64_t* os;
  const void* dout;
  const int64_t* dos;
  const float* lse;
};

template <int D, bool kF16>
int launch_bwd(const BwdPrepIn& in, const CUtensorMap& mq, const CUtensorMap& mk,
               const CUtensorMap& mv, const CUtensorMap& mdo, const CUtensorMap& mq64,
               const CUtensorMap& mk64, const CUtensorMap& mv64, const CUtensorMap& mdo64,
               const fa::BwdParams& base, const fa::BwdParams& prm_q, int sms,
               cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(base.num_bh) * base.Npad;
  const int64_t threads = rows * (D / 8);  // a multiple of 256: Npad is a multiple of 128
  fa::fa_bwd_prep_kernel<D, kF16><<<static_cast<unsigned>(threads / 256), 256, 0, stream>>>(
      static_cast<const uint16_t*>(in.o), static_cast<const uint16_t*>(in.dout), in.lse,
      const_cast<float*>(base.lse2), const_cast<float*>(base.dvec), base.N, base.Npad, base.d,
      base.H, in.os[0], in.os[1], in.os[2], in.dos[0], in.dos[1], in.dos[2]);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  // Persistent grids: one CTA per SM (at most one per tile) walks the tiles.
  const unsigned ctas = static_cast<unsigned>(
      std::min<int64_t>(static_cast<int64_t>(base.T) * base.num_bh, sms));
  fa::fa_bwd_kernel<D, true, kF16><<<ctas, fa::kBwdThreads, fa::BwdCfg<D, true>::kSmemAlloc, stream>>>(
      mk, mv, mq64, mdo64, base);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  fa::fa_bwd_kernel<D, false, kF16><<<ctas, fa::kBwdThreads, fa::BwdCfg<D, false>::kSmemAlloc, stream>>>(
      mq, mdo, mk64, mv64, prm_q);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

// Head dimensions of the backward: multiples of 16 up to 128, laid out in the
// kernels' D = 64 or D = 128 tiles (columns past d arrive as zeros and are
// never stored).
bool bwd_head_dim_ok(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }

extern "C" size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0 || !bwd_head_dim_ok(d)) return 0;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH * bwd_npad(N) > INT_MAX) return 0;  // as the backward rejects
  return static_cast<size_t>(2 * BH * bwd_npad(N) * 4);
}

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                      const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                      int causal, float scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return fa_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, FA_DTYPE_BF16, B, H, N, d, causal, scale,
                   workspace, workspace_bytes, stream);
}

namespace {

int bwd_impl(const void* q, const int64_t* qs_in, const void* k, const int64_t* ks_in,
             const void* v, const int64_t* vs_in, const void* o, const int64_t* os_in,
             const float* lse, const void* dout, const int64_t* dos_in, void* dq,
             const int64_t* dqs_in, void* dk, const int64_t* dks_in, void* dv,
             const int64_t* dvs_in, int dtype, int B, int H, int N, int d, int causal,
             float scale, void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_NULL;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_DTYPE;
  if (B <= 0 || H <= 0 || N <= 0 || (causal != 0 && causal != 1)) return FA_ERR_SHAPE;
  if (!bwd_head_dim_ok(d)) return FA_ERR_HEAD_DIM;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t Npad = bwd_npad(N);
  const int64_t T = Npad / fa::kBwdTile;
  if (BH > INT_MAX || BH * T > INT_MAX || BH * Npad > INT_MAX) return FA_ERR_SHAPE;
  const int64_t contig[3] = {static_cast<int64_t>(H) * N * d, static_cast<int64_t>(N) * d, d};
  // Order: q, k, v, o, dout, dq, dk, dv.
  const int64_t* st[8] = {qs_in, ks_in, vs_in, os_in, dos_in, dqs_in, dks_in, dvs_in};
  for (auto& s : st) {
    if (!s) s = contig;
    // Multiples of 8 elements keep every row (and every 8-column group the
    // D pre-pass and the gradient stores move as one 16-byte word) aligned.
    for (int i = 0; i < 3; ++i)
      if (s[i] < 0 || s[i] % 8 != 0 || s[i] >= (int64_t(1) << 38)) return FA_ERR_STRIDE;
    if (!span_in_range(B, H, N, d, s)) return FA_ERR_STRIDE;
  }
  for (int i = 5; i < 8; ++i)
    if (!strides_disjoint(B, H, N, d, st[i])) return FA_ERR_STRIDE;
  for (const void* ptr : {q, k, v, o, dout, static_cast<const void*>(dq),
                          static_cast<const void*>(dk), static_cast<const void*>(dv),
                          static_cast<const void*>(workspace)})
    if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const size_t lb = static_cast<size_t>(BH) * N * 4;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  // Outputs (dq, dk, dv, workspace) overlap neither an input nor each other
  // (address spans, first to one past the last element).
  const void* ins[6] = {q, k, v, o, lse, dout};
  const size_t in_bytes[6] = {span_bytes(B, H, N, d, st[0]), span_bytes(B, H, N, d, st[1]),
                              span_bytes(B, H, N, d, st[2]), span_bytes(B, H, N, d, st[3]), lb,
                              span_bytes(B, H, N, d, st[4])};
  const void* outs[4] = {dq, dk, dv, workspace};
  const size_t out_bytes[4] = {span_bytes(B, H, N, d, st[5]), span_bytes(B, H, N, d, st[6]),
                               span_bytes(B, H, N, d, st[7]), need};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return FA_ERR_ALIAS;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return FA_ERR_ALIAS;
  }

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv, mdo, mq64, mk64, mv64, mdo64;
  const bool f16 = dtype == FA_DTYPE_FP16;
  const CUtensorMapDataType tt =
      f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const int rows = 128, half = fa::kBwdSub;
  if (!encode_map4(&mq, q, tt, B, H, N, d, st[0], rows) ||
      !encode_map4(&mk, k, tt, B, H, N, d, st[1], rows) ||
      !encode_map4(&mv, v, tt, B, H, N, d, st[2], rows) ||
      !encode_map4(&mdo, dout, tt, B, H, N, d, st[4], rows) ||
      !encode_map4(&mq64, q, tt, B, H, N, d, st[0], half) ||
      !encode_map4(&mk64, k, tt, B, H, N, d, st[1], half) ||
      !encode_map4(&mv64, v, tt, B, H, N, d, st[2], half) ||
      !encode_map4(&mdo64, dout, tt, B, H, N, d, st[4], half))
    return FA_ERR_LAUNCH;

  fa::BwdParams prm;
  prm.out0 = static_cast<uint16_t*>(dk);
  prm.out0_sb = st[6][0];
  prm.out0_sh = st[6][1];
  prm.out0_sn = st[6][2];
  prm.out1 = static_cast<uint16_t*>(dv);
  prm.out1_sb = st[7][0];
  prm.out1_sh = st[7][1];
  prm.out1_sn = st[7][2];
  float* ws = static_cast<float*>(workspace);
  prm.lse2 = ws;
  prm.dvec = ws + BH * Npad;
  prm.N = N;
  prm.d = d;
  prm.Npad = static_cast<int>(Npad);
  prm.T = static_cast<int>(T);
  prm.num_bh = static_cast<int>(BH);
  prm.H = H;
  prm.causal = causal;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.scale = scale;
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  prm.inject = g_inject.load(std::memory_order_relaxed);
  fa::BwdParams prm_q = prm;
  prm_q.out0 = static_cast<uint16_t*>(dq);
  prm_q.out0_sb = st[5][0];
  prm_q.out0_sh = st[5][1];
  prm_q.out0_sn = st[5][2];
  prm_q.out1 = nullptr;
  const BwdPrepIn pin{o, st[3], dout, st[4], lse};
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const bool narrow = d <= 64;  // the D = 64 layout
  if (f16)
    return narrow ? launch_bwd<64, true>(pin, mq, mk, mv, mdo, mq64, mk64, mv64, mdo64, prm,
                                         prm_q, sms, cs)
                  : launch_bwd<128, true>(pin, mq, mk, mv, mdo, mq64, mk64, mv64, mdo64, prm,
                                          prm_q, sms, cs);
  return narrow ? launch_bwd<64, false>(pin, mq, mk, mv, mdo, mq64, mk64, mv64, mdo64, prm, prm_q,
                                        sms, cs)
                : launch_bwd<128, false>(pin, mq, mk, mv, mdo, mq64, mk64, mv64, mdo64, prm,
                                         prm_q, sms, cs);
}

}  // namespace

extern "C" int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                         int dtype, int B, int H, int N, int d, int causal, float scale,
                         void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, nullptr, k, nullptr, v, nullptr, o, nullptr, lse, dout, nullptr, dq, nullptr,
                  dk, nullptr, dv, nullptr, dtype, B, H, N, d, causal, scale, workspace,
                  workspace_bytes, stream);
}

extern "C" int fa_bwd_strided(const void* q, const int64_t* q_strides, const void* k,
                              const int64_t* k_strides, const void* v, const int64_t* v_strides,
                              const void* o, const int64_t* o_strides, const float* lse,
                              const void* dout, const int64_t* dout_strides, void* dq,
                              const int64_t* dq_strides, void* dk, const int64_t* dk_strides,
                              void* dv, const int64_t* dv_strides, int dtype, int B, int H, int N,
                              int d, int causal, float scale, void* workspace,
                              size_t workspace_bytes, void* stream) {
  return bwd_impl(q, q_strides, k, k_strides, v, v_strides, o, o_strides, lse, dout, dout_strides,
                  dq, dq_strides, dk, dk_strides, dv, dv_strides, dtype, B, H, N, d, causal, scale,
                  workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- host buffers (backward)
// Device staging of fa_bwd_host: Q, K, V, O, dO, dQ, dK, dV, LSE and the
// backward's workspace, each 256-byte aligned, in that order.
extern "C" size_t fa_bwd_host_workspace_bytes(int B, int H, int N, int d) {
  const size_t part = fa_bwd_workspace_bytes(B, H, N, d);
  if (part == 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return 8 * round256(rows * d * 2) + round256(rows * 4) + round256(part);
}

extern "C" int fa_bwd_host(const void* q_host, const void* k_host, const void* v_host,
                           const void* o_host, const float* lse_host, const void* dout_host,
                           void* dq_host, void* dk_host, void* dv_host, int dtype, int B, int H,
                           int N, int d, int causal, float scale, void* workspace,
                           size_t workspace_bytes, void* stream) {
  // Everything fa_bwd_ex would reject is rejected here, before any copy is queued.
  if (!q_host || !k_host || !v_host || !o_host || !lse_host || !dout_host || !dq_host ||
      !dk_host || !dv_host)
    return FA_ERR_NULL;
  if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_FP16) return FA_ERR_DTYPE;
  if (B <= 0 || H <= 0 || N <= 0 || (causal != 0 && causal != 1)) return FA_ERR_SHAPE;
  if (!bwd_head_dim_ok(d)) return FA_ERR_HEAD_DIM;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t Npad = bwd_npad(N);
  if (BH > INT_MAX || BH * (Npad / fa::kBwdTile) > INT_MAX || BH * Npad > INT_MAX)
    return FA_ERR_SHAPE;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const size_t need = fa_bwd_host_workspace_bytes(B, H, N, d);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  const size_t tb = static_cast<size_t>(BH) * N * d * 2;
  const size_t lb = static_cast<size_t>(BH) * N * 4;
  // Host outputs overlap neither a host input nor each other.
  const void* ins[6] = {q_host, k_host, v_host, o_host, lse_host, dout_host};
  const size_t in_bytes[6] = {tb, tb, tb, tb, lb, tb};
  const void* outs[3] = {dq_host, dk_host, dv_host};
  for (int a = 0; a < 3; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], tb, ins[b], in_bytes[b])) return FA_ERR_ALIAS;
    for (int b = a + 1; b < 3; ++b)
      if (overlaps(outs[a], tb, outs[b], tb)) return FA_ERR_ALIAS;
  }
  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t t = round256(tb);
  void* qd = ws;
  void* kd = ws + t;
  void* vd = ws + 2 * t;
  void* od = ws + 3 * t;
  void* dod = ws + 4 * t;
  void* dqd = ws + 5 * t;
  void* dkd = ws + 6 * t;
  void* dvd = ws + 7 * t;
  float* ld = reinterpret_cast<float*>(ws + 8 * t);
  uint8_t* part = ws + 8 * t + round256(lb);
  const size_t part_bytes = need - static_cast<size_t>(part - ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(qd, q_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(kd, k_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(vd, v_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(od, o_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(ld, lse_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(dod, dout_host, tb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const int rc = fa_bwd_ex(qd, kd, vd, od, ld, dod, dqd, dkd, dvd, dtype, B, H, N, d, causal,
                           scale, part, part_bytes, stream);
  if (rc != FA_OK) return rc;
  if (cudaMemcpyAsync(dq_host, dqd, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(dk_host, dkd, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(dv_host, dvd, tb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
}

// ------------------------------------------------------- loop-order ablation

namespace {

int64_t ord_npad(int N) { return (static_cast<int64_t>(N) + fa::kOrdTile - 1) / fa::kOrdTile * fa::kOrdTile; }

template <int D>
int launch_order(int order, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                 const fa::OrderParams& prm, cudaStream_t stream) {
  if (order == 1) {
    fa::fa_order_kernel<D, true><<<static_cast<unsigned>(prm.num_bh), fa::kOrdThreads,
                                   fa::OrdCfg<D, true>::kSmemAlloc, stream>>>(mq, mk, mv, prm);
  } else {
    const unsigned ctas = static_cast<unsigned>(static_cast<int64_t>(prm.T) * prm.num_bh);
    fa::fa_order_kernel<D, false><<<ctas, fa::kOrdThreads, fa::OrdCfg<D, false>::kSmemAlloc,
                                    stream>>>(mq, mk, mv, prm);
  }
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

extern "C" size_t fa_fwd_order_ablation_workspace_bytes(int B, int H, int N, int d, int order) {
  if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128) || (order != 1 && order != 2)) return 0;
  if (order == 2) return 16;  // the v2 order keeps its state on chip
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > 65535) return 0;  // as the call rejects
  const int64_t rows = BH * ord_npad(N);
  if (rows > INT_MAX / 4) return 0;
  return static_cast<size_t>(rows * (static_cast<int64_t>(d) + 2) * 4);
}

extern "C" int fa_fwd_order_ablation(const void* q, const void* k, const void* v, void* o, float* lse,
                                     int B, int H, int N, int d, int causal, float scale, int order,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
  if (B <= 0 || H <= 0 || N <= 0 || (causal != 0 && causal != 1) || (order != 1 && order != 2))
    return FA_ERR_SHAPE;
  if (d != 64 && d != 128) return FA_ERR_HEAD_DIM;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t Npad = ord_npad(N);
  if (BH > 65535 || BH * Npad > INT_MAX / 4) return FA_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
       reinterpret_cast<uintptr_t>(workspace)) &
      15u)
    return FA_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_ALIGN;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  const size_t need = fa_fwd_order_ablation_workspace_bytes(B, H, N, d, order);
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  const size_t tb = static_cast<size_t>(BH) * N * d * 2, lb = static_cast<size_t>(BH) * N * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, tb, in, tb) || overlaps(lse, lb, in, tb) || overlaps(workspace, need, in, tb))
      return FA_ERR_ALIAS;
  if (overlaps(o, tb, lse, lb) || overlaps(workspace, need, o, tb) || overlaps(workspace, need, lse, lb))
    return FA_ERR_ALIAS;

  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  std::call_once(g_encode_once, load_encode);
  if (g_encode == nullptr) return FA_ERR_LAUNCH;
  CUtensorMap mq, mk, mv;
  if (!encode_map(&mq, q, static_cast<int>(BH), N, d, fa::kOrdTile) ||
      !encode_map(&mk, k, static_cast<int>(BH), N, d, fa::kOrdTile) ||
      !encode_map(&mv, v, static_cast<int>(BH), N, d, fa::kOrdTile))
    return FA_ERR_LAUNCH;
  fa::OrderParams prm;
  prm.o = static_cast<uint16_t*>(o);
  prm.lse = lse;
  float* ws = static_cast<float*>(workspace);
  prm.ws_o = ws;
  prm.ws_m = ws + BH * Npad * d;
  prm.ws_l = prm.ws_m + BH * Npad;
  prm.N = N;
  prm.Npad = static_cast<int>(Npad);
  prm.T = static_cast<int>(Npad / fa::kOrdTile);
  prm.num_bh = static_cast<int>(BH);
  prm.causal = causal;
  prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_order<64>(order, mq, mk, mv, prm, st)
                 : launch_order<128>(order, mq, mk, mv, prm, st);
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

// Largest cluster the split pass uses (portable cluster size).
constexpr int kMaxClusterSplits = 8;

// The split pass, then the merge: on chip in one clustered launch when the
// ranges of a batch*head fit in one cluster (and `allow_cluster`), else
// through the workspace and the combine kernel.
template <int D>
int launch_split(const CUtensorMap& mk, const CUtensorMap& mv, const fa::SplitParams& prm,
                 cudaStream_t stream, bool allow_cluster) {
  const dim3 grid1(static_cast<unsigned>(prm.splits), static_cast<unsigned>(prm.num_bh));
  if (allow_cluster && prm.splits <= kMaxClusterSplits) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid1;
    cfg.blockDim = dim3(fa::kSplitThreads);
    cfg.dynamicSmemBytes = fa::SplitCfg<D>::kSmemAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(prm.splits);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fa::fa_splitkv_partial_kernel<D, true>, mk, mv, prm);
    return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
  }
  fa::fa_splitkv_partial_kernel<D, false>
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
  prm.inject = g_inject.load(std::memory_order_relaxed);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return d == 64 ? launch_split<64>(mk, mv, prm, s, true) : launch_split<128>(mk, mv, prm, s, true);
}


// ---------------------------------------------------------------- host buffers (split-KV)
// Device staging of fa_fwd_splitkv_host: Q, K, V, O, LSE and the split
// partials, each 256-byte aligned, in that order.
extern "C" size_t fa_fwd_splitkv_host_workspace_bytes(int B, int H, int Nq, int Nk, int d,
                                                      int num_splits) {
  const size_t part = fa_fwd_splitkv_workspace_bytes(B, H, Nq, Nk, d, num_splits);
  if (part == 0) return 0;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t qb = BH * Nq * d * 2, kvb = BH * Nk * d * 2, lb = BH * Nq * 4;
  return 2 * round256(qb) + 2 * round256(kvb) + round256(lb) + round256(part);
}

extern "C" int fa_fwd_splitkv_host(const void* q_host, const void* k_host, const void* v_host,
                                   void* o_host, float* lse_host, int B, int H, int Nq, int Nk,
                                   int d, int causal, float scale, int num_splits, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  // Everything fa_fwd_splitkv would reject is rejected here, before any copy is queued.
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return FA_ERR_NULL;
  const int shape = split_shape_ok(B, H, Nq, Nk, d, causal, num_splits);
  if (shape != FA_OK) return shape;
  if (!std::isfinite(scale)) return FA_ERR_SCALE;
  int dev = 0, sms = 0;
  const int prep = prepare_device(&dev, &sms);
  if (prep != FA_OK) return prep;
  const size_t need = fa_fwd_splitkv_host_workspace_bytes(B, H, Nq, Nk, d, num_splits);
  if (need == 0) return FA_ERR_LAUNCH;
  if (!workspace || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return FA_ERR_ALIGN;
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t qb = BH * Nq * d * 2, kvb = BH * Nk * d * 2, lb = BH * Nq * 4;
  const void* hin[3] = {q_host, k_host, v_host};
  const size_t hin_bytes[3] = {qb, kvb, kvb};
  for (int i = 0; i < 3; ++i)
    if (overlaps(o_host, qb, hin[i], hin_bytes[i]) || overlaps(lse_host, lb, hin[i], hin_bytes[i]))
      return FA_ERR_ALIAS;
  if (overlaps(o_host, qb, lse_host, lb)) return FA_ERR_ALIAS;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qd = ws;
  void* kd = ws + round256(qb);
  void* vd = static_cast<uint8_t*>(kd) + round256(kvb);
  void* od = static_cast<uint8_t*>(vd) + round256(kvb);
  float* ld = reinterpret_cast<float*>(static_cast<uint8_t*>(od) + round256(qb));
  uint8_t* part = reinterpret_cast<uint8_t*>(ld) + round256(lb);
  const size_t part_bytes = need - static_cast<size_t>(part - ws);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(qd, q_host, qb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(kd, k_host, kvb, cudaMemcpyHostToDevice, st) != cudaSuccess ||
      cudaMemcpyAsync(vd, v_host, kvb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const int rc = fa_fwd_splitkv(qd, kd, vd, od, ld, B, H, Nq, Nk, d, causal, scale, num_splits,
                                part, part_bytes, stream);
  if (rc != FA_OK) return rc;
  if (cudaMemcpyAsync(o_host, od, qb, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, ld, lb, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return FA_OK;
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
// taken once per device (with that device current) on the first call there,
// and again whenever that device's current context is a different one (after
// a cudaDeviceReset the module is loaded anew, possibly at another address).
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) uint8_t g_splitkv_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // context id the address belongs to

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

void load_ctx_queries() {
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  void* fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fn != nullptr)
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  fn = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fn != nullptr)
    g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
}

// Process-unique id of the current context (never reused for another
// context), or 0 when it cannot be queried.
unsigned long long current_context_id() {
  std::call_once(g_ctx_once, load_ctx_queries);
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on `dev` (the current device).
int static_scratch(int dev, void** out) {
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr || ctx == 0 || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || ptr == nullptr)
      return FA_ERR_LAUNCH;
    g_scratch_addr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
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
  prm.inject = g_inject.load(std::memory_order_relaxed);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // Always the two-pass form: this entry point's partials go through its
  // built-in scratch array.
  return d == 64 ? launch_split<64>(mk, mv, prm, s, false) : launch_split<128>(mk, mv, prm, s, false);
}

extern "C" const char* fa_strerror(int code) {
  switch (code) {
    case FA_OK: return "success";
    case FA_ERR_NULL: return "a required pointer is NULL";
    case FA_ERR_SHAPE: return "invalid shape (B, H, N must be >= 1 and within index limits; causal 0 or 1)";
    case FA_ERR_HEAD_DIM:
      return "unsupported head dimension (fa_fwd: a multiple of 16 in 16..128, or 256; split-KV "
             "and backward: 64 or 128)";
    case FA_ERR_ALIGN: return "misaligned pointer (q, k, v, o need 16 bytes; lse needs 4)";
    case FA_ERR_SCALE: return "scale is not finite";
    case FA_ERR_ALIAS: return "an output overlaps an input or the other output";
    case FA_ERR_DEVICE: return "current device is not sm_103 (GB300)";
    case FA_ERR_LAUNCH: return "CUDA error while preparing or launching the kernel";
    case FA_ERR_TIMEOUT: return "a kernel wait exceeded its time limit";
    case FA_ERR_WORKSPACE: return "workspace missing or smaller than fa_fwd_splitkv_workspace_bytes()";
    case FA_ERR_DTYPE: return "unsupported element type (FA_DTYPE_BF16 or FA_DTYPE_FP16)";
    case FA_ERR_STRIDE:
      return "invalid strides (non-negative multiples of 8 elements below 2^38; o's elements "
             "must not overlap)";
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
