// Split-KV attention forward for a short block of queries against a long key
// sequence (decode): O = softmax(scale * Q K^T [+ causal mask]) V, LSE.
//
// The key sequence is cut into `splits` contiguous ranges.  Pass 1 computes,
// for every (split, batch*head), the attention of all Nq queries against that
// range only — a normalised fp32 output O_s and its log-sum-exp LSE_s — into
// a workspace.  Pass 2 merges the ranges with the block-merge identity of
// "Parsing FlashAttention (2): FlashAttention-v1 forward pass" eq. (20) and
// "Online Softmax and FlashAttention" (course unit 12):
//     LSE = ln sum_s e^(LSE_s),    O = sum_s e^(LSE_s - LSE) O_s,
// a range with no visible key (LSE_s = -inf) weighing 0.  Causal masking is
// aligned to the end of the keys: query i sees keys 0 .. Nk - Nq + i.
//
// With a handful of queries the work is bound by reading K and V from HBM
// (about one FLOP per byte), so pass 1 runs on the CUDA cores: a producer warp
// streams 128-key K and V tiles (contiguous rows) into a shared-memory ring
// with 1-D bulk copies, and eight consumer warps each own 16 keys of every
// tile: a lane pair computes one q.k dot product (half of d each), the warp
// keeps a running max / exponent sum / output slice per query (lane l owns
// output columns [D/32*l, D/32*(l+1))), and at the end the eight warp states
// are merged in shared memory.  Shared-memory reads are skewed per lane so
// the 32 lanes of a warp never queue on one bank.
//
// Waits are bounded like those of the main kernel (status word, no hang).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "fa_fwd_kernel.cuh"  // g_fa_status, kStatusTimeout
#include "ptx.cuh"

namespace fa {

constexpr int kSplitMaxQ = 16;          // queries per call
constexpr int kSplitTileKeys = 128;     // keys per streamed tile
constexpr int kSplitConsumerWarps = 8;  // 16 keys of each tile per warp
constexpr int kSplitThreads = (kSplitConsumerWarps + 1) * 32;
constexpr int kSplitStages = 2;
constexpr int kSplitMaxSplits = 256;

struct SplitParams {
  const uint16_t* q;  // [BH][Nq][D] bf16
  const uint16_t* k;  // [BH][Nk][D]
  const uint16_t* v;  // [BH][Nk][D]
  uint16_t* o;        // [BH][Nq][D] bf16 (pass 2)
  float* lse;         // [BH][Nq] (pass 2)
  float* ws_o;        // [splits][BH][Nq][D] fp32 partial outputs
  float* ws_lse;      // [splits][BH][Nq] fp32 partial log-sum-exp (natural log)
  int Nq, Nk, num_bh, splits, keys_per_split, causal;
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
};

template <int D>
struct SplitCfg {
  static constexpr uint32_t kTileBytes = kSplitTileKeys * D * 2;  // K (or V) tile
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kSplitStages * kTileBytes;
  static constexpr uint32_t kOffQ = kOffV + kSplitStages * kTileBytes;  // bf16 [16][D]
  // Per-warp running state of every query: max m and exponent sum l
  // [warps][16] and the unnormalised output O [warps][16][D], fp32.
  static constexpr uint32_t kOffM = kOffQ + kSplitMaxQ * D * 2;
  static constexpr uint32_t kOffL = kOffM + kSplitConsumerWarps * kSplitMaxQ * 4;
  static constexpr uint32_t kOffAcc = kOffL + kSplitConsumerWarps * kSplitMaxQ * 4;
  static constexpr uint32_t kOffBar = kOffAcc + kSplitConsumerWarps * kSplitMaxQ * D * 4;
  static constexpr uint32_t kSmemBytes = kOffBar + 2 * kSplitStages * 8 + 16;
  static_assert(kSmemBytes + 128 <= 232448, "dynamic shared memory per block");
};

__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Bounded wait (same contract as the main kernel's): false on expiry, after
// recording FA_DEVICE_STATUS_TIMEOUT.
__device__ __forceinline__ bool split_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > limit_ns) break;
  }
  atomicOr(&g_fa_status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Pass 1: one CTA per (split, batch*head).
template <int D>
__global__ void __launch_bounds__(kSplitThreads, 1)
    fa_splitkv_partial_kernel(const SplitParams p) {
  using C = SplitCfg<D>;
  constexpr int kCols = D / 32;             // output columns per lane
  constexpr int kChunksHalf = D / 16;       // 16-byte chunks in half a row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~static_cast<uintptr_t>(127));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * kSplitStages;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int Nq = p.Nq;
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.Nk, k_begin + p.keys_per_split);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + kSplitTileKeys - 1) / kSplitTileKeys : 0;

  // Q -> shared memory (bf16), all threads.
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + static_cast<size_t>(bh) * Nq * D);
    uint4* dst = reinterpret_cast<uint4*>(smem + C::kOffQ);
    for (int i = threadIdx.x; i < Nq * D / 8; i += blockDim.x) dst[i] = src[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSplitStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kSplitConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // Consumer state in shared memory: m, l per (warp, query) and this
  // lane's D/32 output columns per (warp, query).
  const float c = p.scale_log2;
  float* m_s = reinterpret_cast<float*>(smem + C::kOffM);
  float* l_s = reinterpret_cast<float*>(smem + C::kOffL);
  float* acc_s = reinterpret_cast<float*>(smem + C::kOffAcc);
  if (warp < kSplitConsumerWarps) {
    if (lane < kSplitMaxQ) {
      m_s[warp * kSplitMaxQ + lane] = -CUDART_INF_F;
      l_s[warp * kSplitMaxQ + lane] = 0.0f;
    }
    for (int i = 0; i < kSplitMaxQ; ++i)
#pragma unroll
      for (int e = 0; e < kCols; ++e) acc_s[(warp * kSplitMaxQ + i) * D + lane * kCols + e] = 0.0f;
    __syncwarp();
  }
  bool ok = true;

  if (warp == kSplitConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint16_t* kb = p.k + static_cast<size_t>(bh) * p.Nk * D;
      const uint16_t* vb = p.v + static_cast<size_t>(bh) * p.Nk * D;
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kSplitStages;
        if (t >= kSplitStages &&
            !split_wait(bar_empty + 8 * s, static_cast<uint32_t>(t / kSplitStages - 1) & 1u,
                        p.wait_limit_ns))
          break;
        const int k0 = k_begin + t * kSplitTileKeys;
        const int rows = min(kSplitTileKeys, k_end - k0);
        const uint32_t bytes = static_cast<uint32_t>(rows) * D * 2;
        mbar_arrive_expect_tx(bar_full + 8 * s, 2 * bytes);
        bulk_copy_g2s(sbase + C::kOffK + s * C::kTileBytes, kb + static_cast<size_t>(k0) * D, bytes,
                      bar_full + 8 * s);
        bulk_copy_g2s(sbase + C::kOffV + s * C::kTileBytes, vb + static_cast<size_t>(k0) * D, bytes,
                      bar_full + 8 * s);
        issued = t + 1;
      }
      // Drain: the last copy into each stage must land before the CTA exits.
      for (int s = 0; s < kSplitStages; ++s) {
        if (issued > s) {
          const int last = issued - 1 - ((issued - 1 - s) % kSplitStages);
          split_wait(bar_full + 8 * s, static_cast<uint32_t>(last / kSplitStages) & 1u,
                     p.wait_limit_ns);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int key_in_tile = 16 * warp + (lane >> 1);
    const int half = lane & 1;
    const uint8_t* q_s = smem + C::kOffQ;
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % kSplitStages;
      const bool got = split_wait(bar_full + 8 * s, static_cast<uint32_t>(t / kSplitStages) & 1u,
                                  p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint8_t* k_s = smem + C::kOffK + s * C::kTileBytes;
      const uint8_t* v_s = smem + C::kOffV + s * C::kTileBytes;
      const int k0 = k_begin + t * kSplitTileKeys;
      const int key = k0 + key_in_tile;
      const bool in_range = key < k_end;
      // This lane's half row of K, read in a lane-skewed chunk order.
      const uint8_t* k_row = k_s + key_in_tile * (D * 2) + half * D;
#pragma unroll 1
      for (int i = 0; i < Nq; ++i) {
        const uint8_t* q_row = q_s + i * (D * 2) + half * D;
        float dot = 0.0f;
#pragma unroll
        for (int cc = 0; cc < kChunksHalf; ++cc) {
          const int ch = (cc + (lane >> 1)) % kChunksHalf;
          const uint4 kv = *reinterpret_cast<const uint4*>(k_row + ch * 16);
          const uint4 qv = *reinterpret_cast<const uint4*>(q_row + ch * 16);
          dot = fmaf(bf16_lo(qv.x), bf16_lo(kv.x), dot);
          dot = fmaf(bf16_hi(qv.x), bf16_hi(kv.x), dot);
          dot = fmaf(bf16_lo(qv.y), bf16_lo(kv.y), dot);
          dot = fmaf(bf16_hi(qv.y), bf16_hi(kv.y), dot);
          dot = fmaf(bf16_lo(qv.z), bf16_lo(kv.z), dot);
          dot = fmaf(bf16_hi(qv.z), bf16_hi(kv.z), dot);
          dot = fmaf(bf16_lo(qv.w), bf16_lo(kv.w), dot);
          dot = fmaf(bf16_hi(qv.w), bf16_hi(kv.w), dot);
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);  // the other half of the row
        const bool visible = in_range && (!p.causal || key <= p.Nk - Nq + i);
        const float x = visible ? dot * c : -CUDART_INF_F;
        // Max over the warp's 16 keys (lane pairs hold the same value).
        float mt = x;
#pragma unroll
        for (int off = 2; off < 32; off <<= 1)
          mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
        const float m_old = m_s[warp * kSplitMaxQ + i];
        const float m_new = fmaxf(m_old, mt);
        if (m_new == -CUDART_INF_F) continue;  // nothing visible to this warp yet (uniform)
        const float alpha = ex2_approx(m_old - m_new);  // 0 when m_old was -inf
        const float pr = ex2_approx(x - m_new);         // 0 for masked keys
        float ps = half == 0 ? pr : 0.0f;               // count each key once
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
        const float l_new = l_s[warp * kSplitMaxQ + i] * alpha + ps;
        __syncwarp();
        if (lane == 0) {
          m_s[warp * kSplitMaxQ + i] = m_new;
          l_s[warp * kSplitMaxQ + i] = l_new;
        }
        float* acc_row = acc_s + (warp * kSplitMaxQ + i) * D + lane * kCols;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = acc_row[e] * alpha;
        // Output slice += sum over the warp's 16 keys of p_key * V[key][lane's columns].
        // Rows past the end of the range were not copied this time (stale or
        // never written), so they are skipped rather than multiplied by 0.
        const int warp_keys = k_end - (k0 + 16 * warp);  // uniform across the warp
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          if (kk >= warp_keys) break;
          const float pk = __shfl_sync(0xffffffffu, pr, 2 * kk);
          const uint8_t* v_row = v_s + (16 * warp + kk) * (D * 2) + lane * (kCols * 2);
          if (kCols == 4) {
            const uint2 vv = *reinterpret_cast<const uint2*>(v_row);
            acc[0] = fmaf(pk, bf16_lo(vv.x), acc[0]);
            acc[1] = fmaf(pk, bf16_hi(vv.x), acc[1]);
            acc[2] = fmaf(pk, bf16_lo(vv.y), acc[2]);
            acc[3] = fmaf(pk, bf16_hi(vv.y), acc[3]);
          } else {
            const uint32_t vv = *reinterpret_cast<const uint32_t*>(v_row);
            acc[0] = fmaf(pk, bf16_lo(vv), acc[0]);
            acc[1] = fmaf(pk, bf16_hi(vv), acc[1]);
          }
        }
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc_row[e] = acc[e];
        __syncwarp();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
  }

  // ------------------------------------------------------------ merge warps
  float* ms = m_s;
  float* ls = l_s;
  float* os = acc_s;
  const bool all_ok = __syncthreads_and(ok);
  // One thread per (query, column): merge the warps, normalise, write.
  for (int idx = threadIdx.x; idx < Nq * D; idx += kSplitThreads) {
    const int i = idx / D;
    const int col = idx % D;
    float m = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kSplitConsumerWarps; ++w) m = fmaxf(m, ms[w * kSplitMaxQ + i]);
    float l = 0.0f, o = 0.0f;
    if (m != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kSplitConsumerWarps; ++w) {
        const float mw = ms[w * kSplitMaxQ + i];
        const float e = mw == -CUDART_INF_F ? 0.0f : ex2_approx(mw - m);
        l += e * ls[w * kSplitMaxQ + i];
        o += e * os[(w * kSplitMaxQ + i) * D + col];
      }
    }
    const size_t row = (static_cast<size_t>(split) * p.num_bh + bh) * Nq + i;
    const bool any = all_ok && l > 0.0f;
    p.ws_o[row * D + col] = any ? o / l : 0.0f;
    if (col == 0) p.ws_lse[row] = any ? (m + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
  }
}

// Pass 2: one warp per (batch*head, query) row; lane l owns D/32 columns.
template <int D>
__global__ void __launch_bounds__(256)
    fa_splitkv_combine_kernel(const SplitParams p) {
  constexpr int kCols = D / 32;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // bh * Nq + i
  const int lane = threadIdx.x & 31;
  if (row >= p.num_bh * p.Nq) return;
  const size_t stride = static_cast<size_t>(p.num_bh) * p.Nq;  // between splits
  float m = -CUDART_INF_F;
  for (int s = lane; s < p.splits; s += 32) m = fmaxf(m, p.ws_lse[s * stride + row]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float total = 0.0f;
  float o[kCols];
#pragma unroll
  for (int e = 0; e < kCols; ++e) o[e] = 0.0f;
  for (int s = 0; s < p.splits; ++s) {
    const float ls = p.ws_lse[s * stride + row];
    if (ls == -CUDART_INF_F) continue;  // no visible key in this range
    const float w = __expf(ls - m);
    total += w;
    const float* src = p.ws_o + (s * stride + row) * D + lane * kCols;
#pragma unroll
    for (int e = 0; e < kCols; ++e) o[e] = fmaf(w, src[e], o[e]);
  }
  const float inv = 1.0f / total;
  uint16_t* dst = p.o + static_cast<size_t>(row) * D + lane * kCols;
#pragma unroll
  for (int e = 0; e < kCols; e += 2) {
    const uint32_t pk = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = pk;
  }
  if (lane == 0) p.lse[row] = m + __logf(total);
}

}  // namespace fa
