// Fused attention forward for sm_103a:  O = softmax(scale * Q K^T [+ causal mask]) V,
// LSE = log-sum-exp of each row of the scaled, masked scores.
//
// Method: the tiled online softmax of "Parsing FlashAttention (2):
// FlashAttention-v1 forward pass" (§2-§3: running max m, running exponent sum
// l, accumulator rescaled by exp(m_old - m_new) when the max grows) in the
// loop order of "Online Softmax and FlashAttention" (course unit 12: one CTA
// keeps its Q tile and output accumulator on chip for the whole K/V sweep;
// fully-future tiles are never loaded; diagonal tiles are masked element by
// element; the unnormalised accumulator is divided by l once at the end).
// No score or probability tile ever leaves the SM.
//
// One CTA = one (batch*head, 128-row query tile).  Six warps:
//   warps 0-3  softmax / rescale / epilogue; thread t owns query row t, which
//              is TMEM lane t, so row max and row sum are in-thread reductions
//   warp 4     TMA producer: Q once, then K_j and V_j into two SMEM rings
//   warp 5     TMEM allocator and tcgen05.mma issuer
// TMEM (512 columns): S double buffer at columns [0,128) and [128,256), the
// fp32 output accumulator at [256, 256+D).  P (bf16) goes through SMEM in the
// same 128-byte-swizzled K-major layout TMA gives Q, and feeds the P.V MMA.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// FA_STATUS_TIMEOUT in a device status word, every role leaves its loop,
// in-flight copies and MMAs are drained (again bounded), TMEM is freed and the
// CTA exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;  // query rows per CTA (= TMEM lanes)
constexpr int kBlockN = 128;  // keys per K/V tile
constexpr int kNumThreads = 192;
constexpr int kNumRowThreads = 128;
constexpr int kLoadWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kSwBlockBytes = 128 * 128;  // [128 rows x 64 bf16] swizzled block

constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kInjectSkipFirstV = 1u;  // test hook: never issue the first V load

__device__ uint32_t g_fa_status;

struct FwdParams {
  float* lse;           // [BH][N] fp32
  int N;                // sequence length
  int num_q_tiles;      // ceil(N / kBlockM)
  int causal;           // 0 / 1
  float scale_log2;     // scale * log2(e)
  uint32_t inject;      // test hooks (0 in normal use)
  uint64_t wait_limit_ns;
};

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  static constexpr int kStages = (D == 64) ? 3 : 2;
  static constexpr uint32_t kQBytes = kBlockM * D * 2;
  static constexpr uint32_t kKVBytes = kBlockN * D * 2;
  static constexpr uint32_t kPBytes = kBlockM * kBlockN * 2;
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKVBytes;
  static constexpr uint32_t kOffP = kOffV + kStages * kKVBytes;
  static constexpr uint32_t kOffBar = kOffP + kPBytes;
  // q_full, k_full[S], k_empty[S], v_full[S], v_empty[S], s_full[2], p_full, o_done, mma_done
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 3;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S buffer b at kColS + 128*b
  static constexpr uint32_t kColO = 256;  // fp32 accumulator, D columns
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(kBlockM, kBlockN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kBlockM, D, 0, 1);
};

struct Barriers {
  uint32_t q_full, s_full0, p_full, o_done, mma_done;
  uint32_t k_full0, k_empty0, v_full0, v_empty0;  // + 8*stage
  __device__ uint32_t k_full(int s) const { return k_full0 + 8u * s; }
  __device__ uint32_t k_empty(int s) const { return k_empty0 + 8u * s; }
  __device__ uint32_t v_full(int s) const { return v_full0 + 8u * s; }
  __device__ uint32_t v_empty(int s) const { return v_empty0 + 8u * s; }
  __device__ uint32_t s_full(int b) const { return s_full0 + 8u * b; }
};

struct WaitCtx {
  volatile uint32_t* abort;
  uint64_t limit_ns;
};

__device__ __forceinline__ void record_timeout(const WaitCtx& w) {
  *w.abort = 1u;
  atomicOr(&g_fa_status, kStatusTimeout);
}

// Slow path of wait_bar: poll until the phase completes, the CTA aborts or
// the time limit expires.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u) {
      if (*w.abort) return false;
      if (global_timer_ns() - t0 > w.limit_ns) break;
    }
  }
  record_timeout(w);
  return false;
}

// Bounded wait for the phase with parity `parity` of barrier `bar`.
// Returns false if the CTA is aborting or the time limit expired.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(bar, parity, w);
}

// Bounded wait used while draining: ignores the abort flag (copies and MMAs
// already issued always complete), bounded by time alone.
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > w.limit_ns) break;
  }
  record_timeout(w);
  return false;
}

// Bounded wait whose result is uniform across the calling warp (every lane
// must call it): tcgen05.ld/st and warp votes that follow need the whole warp.
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = wait_bar(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// AND-reduce a flag over the 128 row threads (named barrier 1).
__device__ __forceinline__ bool row_threads_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// Descriptor of the 16-wide K slice `kk` of a K-major operand stored as
// [rows x 64] swizzled blocks (block b holds K columns [64b, 64b+64)).
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return smem_desc_sw128(base + (kk >> 2) * kSwBlockBytes + (kk & 3) * 32, 16, 1024);
}

// Descriptor of the 16-row K slice `kk` of the MN-major V tile: rows are keys
// (the K dimension), 128-byte rows hold 64 head-dim columns; the next 64
// columns sit one swizzled block further (leading-dimension offset).
__device__ __forceinline__ uint64_t v_desc(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 16 * 128, kSwBlockBytes, 1024);
}

// Byte offset of the 16-byte chunk `chunk` (0..D/8-1) of row `row` in a
// [128 x D] tile stored as 128-byte-swizzled [128 x 64] blocks.
__device__ __forceinline__ uint32_t swizzled_chunk(int row, int chunk) {
  return (chunk >> 3) * kSwBlockBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using C = Cfg<D>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  const uint32_t sP = sbase + C::kOffP;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);

  Barriers bars;
  {
    uint32_t b = sbase + C::kOffBar;
    bars.q_full = b;
    b += 8;
    bars.k_full0 = b;
    b += 8 * S;
    bars.k_empty0 = b;
    b += 8 * S;
    bars.v_full0 = b;
    b += 8 * S;
    bars.v_empty0 = b;
    b += 8 * S;
    bars.s_full0 = b;
    b += 16;
    bars.p_full = b;
    b += 8;
    bars.o_done = b;
    b += 8;
    bars.mma_done = b;
  }
  const WaitCtx wctx{abort_flag, p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int q_tile = p.num_q_tiles - 1 - static_cast<int>(blockIdx.y);  // heaviest first
  const int q0 = q_tile * kBlockM;
  const int q_end = min(q0 + kBlockM, p.N);
  // Causal: key tiles whose first key is at or past the query tile's end are
  // entirely in the future and are skipped (never loaded, never computed).
  const int kv_end = p.causal ? q_end : p.N;
  const int n_tiles = (kv_end + kBlockN - 1) / kBlockN;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full, 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
    mbar_init(bars.s_full(0), 1);
    mbar_init(bars.s_full(1), 1);
    mbar_init(bars.p_full, kNumRowThreads);
    mbar_init(bars.o_done, 1);
    mbar_init(bars.mma_done, 1);
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int last_k[S], last_v[S];
      for (int s = 0; s < S; ++s) last_k[s] = last_v[s] = -1;
      mbar_arrive_expect_tx(bars.q_full, C::kQBytes);
#pragma unroll
      for (int b = 0; b < D / 64; ++b)
        tma_load_3d(sQ + b * kSwBlockBytes, &tm_q, bars.q_full, 64 * b, q0, bh);
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % S;
        const uint32_t ph = static_cast<uint32_t>(j / S) & 1u;
        if (j >= S && !wait_bar(bars.k_empty(s), ph ^ 1u, wctx)) break;
        mbar_arrive_expect_tx(bars.k_full(s), C::kKVBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sK + s * C::kKVBytes + b * kSwBlockBytes, &tm_k, bars.k_full(s), 64 * b,
                      j * kBlockN, bh);
        last_k[s] = j;
        if (j >= S && !wait_bar(bars.v_empty(s), ph ^ 1u, wctx)) break;
        if (j == 0 && (p.inject & kInjectSkipFirstV)) continue;
        mbar_arrive_expect_tx(bars.v_full(s), C::kKVBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sV + s * C::kKVBytes + b * kSwBlockBytes, &tm_v, bars.v_full(s), 64 * b,
                      j * kBlockN, bh);
        last_v[s] = j;
      }
      // Drain: every copy issued must land before the CTA may exit.
      wait_bar_drain(bars.q_full, 0, wctx);
      for (int s = 0; s < S; ++s) {
        if (last_k[s] >= 0) wait_bar_drain(bars.k_full(s), (last_k[s] / S) & 1, wctx);
        if (last_v[s] >= 0) wait_bar_drain(bars.v_full(s), (last_v[s] / S) & 1, wctx);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      auto issue_s = [&](int j) -> bool {
        const int s = j % S;
        if (!wait_bar(bars.k_full(s), static_cast<uint32_t>(j / S) & 1u, wctx)) return false;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + C::kColS + 128u * static_cast<uint32_t>(j & 1);
        const uint32_t kbase = sK + s * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(d_tmem, kmajor_desc(sQ, kk), kmajor_desc(kbase, kk), C::kIdescQK, kk > 0);
        umma_commit(bars.k_empty(s));
        umma_commit(bars.s_full(j & 1));
        return true;
      };
      bool ok = wait_bar(bars.q_full, 0, wctx);
      if (ok) tc_fence_after_sync();
      for (int j = 0; ok && j < n_tiles && j < 2; ++j) ok = issue_s(j);
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % S;
        if (!wait_bar(bars.p_full, static_cast<uint32_t>(j) & 1u, wctx)) break;
        if (!wait_bar(bars.v_full(s), static_cast<uint32_t>(j / S) & 1u, wctx)) break;
        tc_fence_after_sync();
        const uint32_t vbase = sV + s * C::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_ss(tmem + C::kColO, kmajor_desc(sP, kk), v_desc(vbase, kk), C::kIdescPV,
                  (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bars.v_empty(s));
        umma_commit(bars.o_done);
        if (j + 2 < n_tiles) ok = issue_s(j + 2);
      }
      // Drain: wait for every MMA issued by this thread.
      umma_commit(bars.mma_done);
      wait_bar_drain(bars.mma_done, 0, wctx);
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int row = threadIdx.x;  // 0..127 = TMEM lane
    const int q_idx = q0 + row;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    // Last key index this row may see: itself when causal, else N-1.
    const int row_last_key = p.causal ? min(q_idx, p.N - 1) : p.N - 1;
    float m_run = -CUDART_INF_F;  // running max of scale*log2(e)*s
    float l_run = 0.0f;           // running sum of 2^(x - m_run)
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int buf = j & 1;
      if (!warp_wait_bar(bars.s_full(buf), static_cast<uint32_t>(j >> 1) & 1u, wctx)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      uint32_t sr[4][32];
      const uint32_t s_addr = tmem + lane_off + C::kColS + 128u * buf;
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + 32 * c, sr[c]);
      tmem_ld_wait();

      float x[kBlockN];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) x[32 * c + i] = __uint_as_float(sr[c][i]) * p.scale_log2;

      const int k0 = j * kBlockN;
      if (k0 + kBlockN - 1 > row_last_key) {  // diagonal or ragged tile: mask per element
        const int lim = row_last_key - k0;
#pragma unroll
        for (int i = 0; i < kBlockN; ++i)
          if (i > lim) x[i] = -CUDART_INF_F;
      }

      float mx0 = x[0], mx1 = x[1], mx2 = x[2], mx3 = x[3];
#pragma unroll
      for (int i = 4; i < kBlockN; i += 4) {
        mx0 = fmaxf(mx0, x[i]);
        mx1 = fmaxf(mx1, x[i + 1]);
        mx2 = fmaxf(mx2, x[i + 2]);
        mx3 = fmaxf(mx3, x[i + 3]);
      }
      const float m_new = fmaxf(m_run, fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)));
      // alpha = 2^(m_old - m_new): 0 on the first tile (m_old = -inf).
      const float alpha = ex2_approx(m_run - m_new);

      uint32_t pk[kBlockN / 2];
      float ls0 = 0.f, ls1 = 0.f, ls2 = 0.f, ls3 = 0.f;
#pragma unroll
      for (int i = 0; i < kBlockN / 2; i += 2) {
        const float p0 = ex2_approx(x[2 * i] - m_new);
        const float p1 = ex2_approx(x[2 * i + 1] - m_new);
        const float p2 = ex2_approx(x[2 * i + 2] - m_new);
        const float p3 = ex2_approx(x[2 * i + 3] - m_new);
        ls0 += p0;
        ls1 += p1;
        ls2 += p2;
        ls3 += p3;
        pk[i] = pack_bf16x2(p0, p1);
        pk[i + 1] = pack_bf16x2(p2, p3);
      }
      l_run = l_run * alpha + ((ls0 + ls1) + (ls2 + ls3));
      m_run = m_new;

      if (j > 0) {
        // P.V of the previous tile must be complete: it reads the P buffer
        // we are about to overwrite and writes the accumulator we rescale.
        if (!warp_wait_bar(bars.o_done, static_cast<uint32_t>(j - 1) & 1u, wctx)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
          const uint32_t o_addr = tmem + lane_off + C::kColO;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_addr + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(o_addr + 32 * c, o);
          }
          tmem_st_wait();
        }
      }
      // P tile -> SMEM (K-major, 128-byte swizzle: the A operand of P.V).
#pragma unroll
      for (int c = 0; c < kBlockN / 8; ++c)
        st_shared_v4(sP + swizzled_chunk(row, c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                     pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bars.p_full);
    }

    // ---------------------------------------------------------- epilogue
    if (ok && !warp_wait_bar(bars.o_done, static_cast<uint32_t>(n_tiles - 1) & 1u, wctx)) ok = false;
    if (row_threads_all(ok)) {
      tc_fence_after_sync();
      const float inv_l = 1.0f / l_run;
      const uint32_t o_addr = tmem + lane_off + C::kColO;
      // The Q tile is dead (its last MMA completed before the last P.V), so
      // its SMEM stages the bf16 output for the TMA store.
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32 * c, o);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w4[e] = pack_bf16x2(__uint_as_float(o[8 * g + 2 * e]) * inv_l,
                                __uint_as_float(o[8 * g + 2 * e + 1]) * inv_l);
          st_shared_v4(sQ + swizzled_chunk(row, 4 * c + g), w4[0], w4[1], w4[2], w4[3]);
        }
      }
      fence_proxy_async_smem();
      named_barrier_sync(1, kNumRowThreads);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int b = 0; b < D / 64; ++b) tma_store_3d(&tm_o, sQ + b * kSwBlockBytes, 64 * b, q0, bh);
        tma_store_commit();
        tma_store_wait_all();
      }
      if (q_idx < p.N)
        p.lse[static_cast<size_t>(bh) * p.N + q_idx] = (m_run + __log2f(l_run)) * 0.6931471805599453f;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
