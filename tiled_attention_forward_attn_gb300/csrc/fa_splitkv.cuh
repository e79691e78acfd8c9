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
// With at most 16 queries the work is bound by reading K and V from HBM
// (Nq FLOPs per byte of K and V).  Pass 1: a
// producer warp streams 64-key K and V tiles into a shared-memory ring with
// TMA (128-byte swizzle, evict-first L2 hint, zero fill past the end), and
// four consumer warps each take 16 keys of every tile: S = Q K^T with
// warp-level 16x8x16 tensor-core MMAs (the query block is exactly one
// 16-row MMA tile), the online-softmax update in registers, and O += P V
// with P kept in registers as the next MMA's A operand.  At the end of the
// range the four warp states are merged in shared memory.  Two CTAs fit on
// a multiprocessor; the host picks the split count so that all CTAs run in
// one wave when the batch allows.
//
// With at most 8 key ranges (the common decode case) the ranges of one
// (batch, head) are launched as one thread-block cluster (kCluster) and
// merged on chip instead: each CTA leaves its normalised partial output and
// log-sum-exp in its own shared memory, the cluster synchronises, each CTA
// merges a share of the output elements reading the others' partials
// through distributed shared memory, and a second cluster barrier keeps
// every partial alive until all reads are done.  No workspace and no second
// launch.
//
// Waits are bounded like those of the main kernel (status word, no hang);
// every CTA of a cluster reaches both cluster barriers, also after a
// timed-out wait.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "fa_fwd_kernel.cuh"  // g_fa_status, kStatusTimeout
#include "ptx.cuh"

namespace fa {

constexpr int kSplitMaxQ = 16;          // queries per call (one MMA row tile)
constexpr int kSplitTileKeys = 64;      // keys per streamed tile
constexpr int kSplitConsumerWarps = 4;  // 16 keys of each tile per warp
constexpr int kSplitThreads = (kSplitConsumerWarps + 1) * 32;
constexpr int kSplitCtasPerSm = 2;
constexpr int kSplitMaxSplits = 256;

struct SplitParams {
  const uint16_t* q;  // [BH][Nq][D] bf16
  uint16_t* o;        // [BH][Nq][D] bf16 (pass 2)
  float* lse;         // [BH][Nq] (pass 2)
  float* ws_o;        // [splits][BH][Nq][D] fp32 partial outputs
  float* ws_lse;      // [splits][BH][Nq] fp32 partial log-sum-exp (natural log)
  int Nq, Nk, num_bh, splits, keys_per_split, causal;
  float scale_log2;  // scale * log2(e)
  uint64_t wait_limit_ns;
  uint32_t inject = 0;  // test hooks (0 in normal use)
};

template <int D>
struct SplitCfg {
  static constexpr int kStages = D == 64 ? 6 : 3;
  static constexpr uint32_t kBoxBytes = kSplitTileKeys * 128;    // 64 keys x 64 columns
  static constexpr uint32_t kTileBytes = kSplitTileKeys * D * 2;  // K (or V) tile: D/64 boxes
  static constexpr uint32_t kStageBytes = 2 * kTileBytes;         // K then V
  static constexpr uint32_t kOffBar = kStages * kStageBytes;
  // The warp merge reuses the ring: O [warps][16][D], then m and l
  // [warps][16], then the range's partial O [16][D] and LSE [16].
  static constexpr uint32_t kMergeBytes =
      kSplitConsumerWarps * kSplitMaxQ * (D + 2) * 4 + kSplitMaxQ * (D + 1) * 4;
  static_assert(kMergeBytes <= kOffBar, "merge area fits in the ring");
  static constexpr uint32_t kSmemBytes = kOffBar + 2 * kStages * 8;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // 1024-byte alignment for SW128
  static_assert(kSplitCtasPerSm * (kSmemAlloc + 1024) <= 233472, "two CTAs per multiprocessor");
};

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

// Byte offset of 16-byte chunk `chunk` (8 columns) of row `row` in a tile of
// D/64 boxes, each 64 rows x 128 bytes with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
  return static_cast<uint32_t>((chunk >> 3) * (kSplitTileKeys * 128) + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// Pass 1: one CTA per (split, batch*head); with kCluster, the CTAs of one
// batch*head form a cluster and also do pass 2.
template <int D, bool kCluster>
__global__ void __launch_bounds__(kSplitThreads, kSplitCtasPerSm)
    fa_splitkv_partial_kernel(const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const SplitParams p) {
  using C = SplitCfg<D>;
  constexpr int kS = C::kStages;
  constexpr int kKSteps = D / 16;  // MMA k-steps of Q K^T over the head dimension
  constexpr int kNTiles = D / 8;   // 8-column MMA tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::kOffBar;
  const uint32_t bar_empty = bar_full + 8 * kS;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int split = blockIdx.x;
  const int bh = blockIdx.y;
  const int Nq = p.Nq;
  const int k_begin = split * p.keys_per_split;
  const int k_end = min(p.Nk, k_begin + p.keys_per_split);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + kSplitTileKeys - 1) / kSplitTileKeys : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kSplitConsumerWarps);
    }
    fence_barrier_init();
  }
  if (threadIdx.x == 32 * kSplitConsumerWarps) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();

  bool ok = true;
  // Consumer state (rows g and g + 8 of the 16-row query block).
  const int g = lane >> 2, t4 = lane & 3;
  float acc[kNTiles][4];
  float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.0f, l1 = 0.0f;
#pragma unroll
  for (int n = 0; n < kNTiles; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

  if (warp == kSplitConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t policy = make_l2_policy_evict_first();
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % kS;
        if (t >= kS &&
            !split_wait(bar_empty + 8 * s, static_cast<uint32_t>(t / kS - 1) & 1u, p.wait_limit_ns))
          break;
        const int k0 = k_begin + t * kSplitTileKeys;
        const uint32_t stage = sbase + s * C::kStageBytes;
        // Test hook: the first K/V tile is never copied, so its wait must time out.
        if (!(t == 0 && (p.inject & kInjectSkipFirstV))) {
          mbar_arrive_expect_tx(bar_full + 8 * s, C::kStageBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            if (!tma_coord_ok(64 * b, D, k0, p.Nk, bh, p.num_bh) ||
                !smem_range_ok(s * C::kStageBytes + C::kTileBytes + b * C::kBoxBytes, C::kBoxBytes,
                               C::kOffBar))
              continue;
            tma_load_3d_hint(stage + b * C::kBoxBytes, &tm_k, bar_full + 8 * s, 64 * b, k0, bh,
                             policy);
            tma_load_3d_hint(stage + C::kTileBytes + b * C::kBoxBytes, &tm_v, bar_full + 8 * s,
                             64 * b, k0, bh, policy);
          }
        }
        issued = t + 1;
      }
      // Drain: the last copy into each stage must land before the CTA exits
      // or the ring is reused by the merge (the skipped one never lands).
      for (int s = 0; s < kS; ++s) {
        if (issued > s) {
          const int last = issued - 1 - ((issued - 1 - s) % kS);
          if (!(last == 0 && (p.inject & kInjectSkipFirstV)))
            split_wait(bar_full + 8 * s, static_cast<uint32_t>(last / kS) & 1u, p.wait_limit_ns);
        }
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    // Q as MMA A fragments, loaded once; rows past Nq are zero.
    uint32_t qa[kKSteps][4];
    {
      const uint32_t* qg = reinterpret_cast<const uint32_t*>(p.q + static_cast<size_t>(bh) * Nq * D);
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        const int c0 = 16 * ks + 2 * t4;
        qa[ks][0] = g < Nq ? qg[(g * D + c0) >> 1] : 0u;
        qa[ks][1] = g + 8 < Nq ? qg[((g + 8) * D + c0) >> 1] : 0u;
        qa[ks][2] = g < Nq ? qg[(g * D + c0 + 8) >> 1] : 0u;
        qa[ks][3] = g + 8 < Nq ? qg[((g + 8) * D + c0 + 8) >> 1] : 0u;
      }
    }
    const float c = p.scale_log2;
    // Last key each of the two rows may see (end-aligned causal mask).
    const int lim0 = p.causal ? p.Nk - Nq + g : INT_MAX;
    const int lim1 = p.causal ? p.Nk - Nq + g + 8 : INT_MAX;
    // ldmatrix row addresses: lane l feeds row (l & 7) of matrix (l >> 3).
    const int mi = lane >> 3, r8 = lane & 7;
    const int k_row = 16 * warp + ((mi >> 1) << 3) + r8;  // K: matrices (keys 0-7|8-15) x (cols lo|hi)
    const int v_row = 16 * warp + ((mi & 1) << 3) + r8;   // V: matrices (keys lo|hi) x (n | n+1)

    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % kS;
      const bool got = split_wait(bar_full + 8 * s, static_cast<uint32_t>(t / kS) & 1u,
                                  p.wait_limit_ns);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint32_t kt = sbase + s * C::kStageBytes;
      const uint32_t vt = kt + C::kTileBytes;

      // S (16 queries x this warp's 16 keys) = Q K^T.
      float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
      for (int ks = 0; ks < kKSteps; ++ks) {
        uint32_t b[4];
        ldsm_x4(b, kt + sw128_offset(k_row, 2 * ks + (mi & 1)));
        mma_bf16_16816(sc[0], qa[ks], b[0], b[1]);
        mma_bf16_16816(sc[1], qa[ks], b[2], b[3]);
      }

      // Mask, running max, probabilities.  Keys past the range's end are
      // masked (TMA filled them with zeros or the next range's rows).
      const int key0 = k_begin + t * kSplitTileKeys + 16 * warp + 2 * t4;
      float x0[4], x1[4];
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + 8 * j + e;
          const bool in = key < k_end;
          x0[2 * j + e] = (in && key <= lim0) ? sc[j][e] * c : -CUDART_INF_F;
          x1[2 * j + e] = (in && key <= lim1) ? sc[j][2 + e] * c : -CUDART_INF_F;
        }
      float mx0 = fmaxf(fmaxf(x0[0], x0[1]), fmaxf(x0[2], x0[3]));
      float mx1 = fmaxf(fmaxf(x1[0], x1[1]), fmaxf(x1[2], x1[3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // Base 0 while a row has seen no visible key: its probabilities and
      // rescale factors are then exactly 0 (no -inf - -inf).
      const float mu0 = mn0 == -CUDART_INF_F ? 0.0f : mn0;
      const float mu1 = mn1 == -CUDART_INF_F ? 0.0f : mn1;
      const float alpha0 = ex2_approx(m0 - mu0), alpha1 = ex2_approx(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      float p0[4], p1[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p0[e] = ex2_approx(x0[e] - mu0);
        p1[e] = ex2_approx(x1[e] - mu1);
      }
      l0 = l0 * alpha0 + ((p0[0] + p0[1]) + (p0[2] + p0[3]));
      l1 = l1 * alpha1 + ((p1[0] + p1[1]) + (p1[2] + p1[3]));
      // P as the A operand of the 16-key step: the S accumulator layout of
      // key tiles 0 and 1 is the A layout of keys 0-15.
      const uint32_t pa[4] = {pack_bf16x2(p0[0], p0[1]), pack_bf16x2(p1[0], p1[1]),
                              pack_bf16x2(p0[2], p0[3]), pack_bf16x2(p1[2], p1[3])};
#pragma unroll
      for (int n = 0; n < kNTiles; n += 2) {
        uint32_t b[4];
        ldsm_x4_trans(b, vt + sw128_offset(v_row, n + (mi >> 1)));
        acc[n][0] *= alpha0;
        acc[n][1] *= alpha0;
        acc[n][2] *= alpha1;
        acc[n][3] *= alpha1;
        acc[n + 1][0] *= alpha0;
        acc[n + 1][1] *= alpha0;
        acc[n + 1][2] *= alpha1;
        acc[n + 1][3] *= alpha1;
        mma_bf16_16816(acc[n], pa, b[0], b[1]);
        mma_bf16_16816(acc[n + 1], pa, b[2], b[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }
    // Row sums: each lane of a quad summed a quarter of the keys.
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }

  // ------------------------------------------------------------ merge warps
  const bool all_ok = __syncthreads_and(ok);
  const size_t row_base = (static_cast<size_t>(split) * p.num_bh + bh) * Nq;
  // Partial result of this range: normalised O_s and LSE_s (natural log),
  // to the workspace or (kCluster) to this CTA's shared memory after the
  // warp-merge area.
  float* os = reinterpret_cast<float*>(smem);                           // [warp][16][D]
  float* ms = os + kSplitConsumerWarps * kSplitMaxQ * D;                // [warp][16]
  float* ls = ms + kSplitConsumerWarps * kSplitMaxQ;                    // [warp][16]
  float* part_o = ls + kSplitConsumerWarps * kSplitMaxQ;                // [16][D]
  float* part_lse = part_o + kSplitMaxQ * D;                            // [16]
  auto put = [&](int i, int col, float o, float lse) {
    if (kCluster) {
      part_o[i * D + col] = o;
      if (col == 0) part_lse[i] = lse;
    } else if (guard(split < p.splits && bh < p.num_bh && i < Nq && col < D)) {
      p.ws_o[(row_base + i) * D + col] = o;
      if (col == 0) p.ws_lse[row_base + i] = lse;
    }
  };
  if (!all_ok) {
    for (int idx = threadIdx.x; idx < Nq * D; idx += kSplitThreads)
      put(idx / D, idx % D, 0.0f, -CUDART_INF_F);
  } else {
    // Every issued tile was consumed, so no copy is in flight: reuse the ring.
    if (warp < kSplitConsumerWarps) {
#pragma unroll
      for (int n = 0; n < kNTiles; ++n) {
        float* r0 = os + (warp * kSplitMaxQ + g) * D + 8 * n + 2 * t4;
        float* r1 = r0 + 8 * D;
        *reinterpret_cast<float2*>(r0) = make_float2(acc[n][0], acc[n][1]);
        *reinterpret_cast<float2*>(r1) = make_float2(acc[n][2], acc[n][3]);
      }
      if (t4 == 0) {
        ms[warp * kSplitMaxQ + g] = m0;
        ms[warp * kSplitMaxQ + g + 8] = m1;
        ls[warp * kSplitMaxQ + g] = l0;
        ls[warp * kSplitMaxQ + g + 8] = l1;
      }
    }
    __syncthreads();
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
      const bool any = l > 0.0f;
      put(i, col, any ? o / l : 0.0f, any ? (m + __log2f(l)) * 0.6931471805599453f : -CUDART_INF_F);
    }
  }
  if (kCluster) {
    // Pass 2 on chip: CTA `rank` merges output elements rank, rank + S*T, ...
    // of this batch*head from the partials of all S ranges (block merge,
    // as in fa_splitkv_combine_kernel).
    cluster_sync_all();
    const uint32_t rank = cluster_ctarank();
    const uint32_t nr = static_cast<uint32_t>(p.splits);
    const uint32_t po = smem_u32(part_o), pl = smem_u32(part_lse);
    for (int idx = static_cast<int>(rank) * kSplitThreads + threadIdx.x; idx < Nq * D;
         idx += static_cast<int>(nr) * kSplitThreads) {
      const int i = idx / D;
      const int col = idx % D;
      float m = -CUDART_INF_F;
      for (uint32_t s2 = 0; s2 < nr; ++s2)
        m = fmaxf(m, ld_cluster_f32(cluster_map(pl + 4u * i, s2)));
      float total = 0.0f, o = 0.0f;
      if (m != -CUDART_INF_F) {
        for (uint32_t s2 = 0; s2 < nr; ++s2) {
          const float ls2 = ld_cluster_f32(cluster_map(pl + 4u * i, s2));
          if (ls2 == -CUDART_INF_F) continue;  // no visible key in that range
          const float w = __expf(ls2 - m);
          total += w;
          o = fmaf(w, ld_cluster_f32(cluster_map(po + 4u * (i * D + col), s2)), o);
        }
      }
      const size_t orow = static_cast<size_t>(bh) * Nq + i;
      const float inv = total > 0.0f ? 1.0f / total : 0.0f;
      if (guard(bh < p.num_bh && i < Nq && col < D)) {
        reinterpret_cast<__nv_bfloat16*>(p.o)[orow * D + col] = __float2bfloat16_rn(o * inv);
        if (col == 0) p.lse[orow] = m + __logf(total);
      }
    }
    cluster_sync_all();  // the other CTAs' partials stay alive until here
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
  // total is 0 only when every range timed out (each partial LSE is -inf):
  // O is then written as zeros, as the clustered merge does.
  const float inv = total > 0.0f ? 1.0f / total : 0.0f;
  uint16_t* dst = p.o + static_cast<size_t>(row) * D + lane * kCols;
  if (!guard(row < p.num_bh * p.Nq && lane * kCols + kCols <= D)) return;
#pragma unroll
  for (int e = 0; e < kCols; e += 2) {
    const uint32_t pk = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
    *reinterpret_cast<uint32_t*>(dst + e) = pk;
  }
  if (lane == 0) p.lse[row] = m + __logf(total);
}

}  // namespace fa
