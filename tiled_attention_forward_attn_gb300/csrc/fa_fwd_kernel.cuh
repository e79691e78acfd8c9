// Fused attention forward for sm_103a:  O = softmax(scale * Q K^T [+ causal mask]) V,
// LSE = log-sum-exp of each row of the scaled, masked scores.
//
// Method: the tiled online softmax of "Parsing FlashAttention (2):
// FlashAttention-v1 forward pass" (§2-§3: running max m, running exponent sum
// l, accumulator rescaled by exp(m_old - m_new) when the max grows) in the
// loop order of "Online Softmax and FlashAttention" (course unit 12: one CTA
// keeps its Q tiles and output accumulators on chip for the whole K/V sweep;
// fully-future tiles are never loaded; diagonal tiles are masked element by
// element; the unnormalised accumulator is divided by l once at the end).
// No score or probability tile ever leaves the SM.
//
// One CTA = one (batch*head, 256-row query unit) = two 128-row query tiles,
// "A" (rows q0..q0+127) and "B" (rows q0+128..q0+255), that share every K/V
// tile loaded.  Three warpgroups:
//   warps 0-3   softmax of tile A; thread t owns row t of A = TMEM lane t
//   warps 4-7   softmax of tile B; thread t owns row t of B = TMEM lane t
//   warp 8      TMA producer of Q_A, Q_B (once) and the K_j ring
//   warp 9      TMEM allocator and tcgen05.mma issuer
//   warp 10     TMA producer of the V_j ring
//   warp 11     idle (it completes the third warpgroup)
// K and V have separate rings and producers, so neither ring's refill waits
// behind the other's; the rings are as deep as shared memory allows because
// a K/V tile copy takes a few microseconds to land under full load.
// The third warpgroup hands most of its registers to the two softmax
// warpgroups (setmaxnreg): 384 threads launch with 168 registers each
// (64512 in all); afterwards 256 x 232 + 128 x 40 = 64512 are in use.
// The tensor core alternates between the tiles: while the softmax warps of A
// turn S_A(j) into P_A(j), it computes P_B(j-1) V_(j-1) and S_B(j), and vice
// versa, so the exponentials of one tile overlap the MMAs of the other.
//
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A and O_B after them
// (D columns each, fp32).  P_t (bf16 pairs, 64 columns) is written over the
// first half of S_t once S_t is in registers and feeds the P.V MMA straight
// from TMEM; the next S_t MMA is issued after that P.V MMA, and tcgen05.mma
// operations of one thread execute in issue order.  Because the S_t(j) MMA is
// also committed after P_t(j-1) V_(j-1), the softmax warps know O_t is
// complete whenever S_t(j) is, and may rescale it in place.
//
// Rescaling is lazy: the exponent reference m_ref of a row only moves when a
// tile's maximum exceeds it by more than 8 (base-2 exponent units), so P, l
// and O keep sharing one reference and the result is unchanged; most tiles
// then need no O rescale at all.
//
// Every mbarrier wait is bounded: on expiry the kernel records
// FA_DEVICE_STATUS_TIMEOUT in a device status word, every role leaves its
// loop, in-flight copies and MMAs are drained (again bounded), TMEM is freed
// and the CTA exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "ptx.cuh"

namespace fa {

constexpr int kTileM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kTilesPerCta = 2;
constexpr int kUnitM = kTileM * kTilesPerCta;  // query rows per CTA
constexpr int kBlockN = 128;                   // keys per K/V tile
constexpr int kNumThreads = 384;
constexpr uint32_t kLaunchRegs = 168;    // 65536 / (3 warps per sub-partition x 32 x 4)
constexpr uint32_t kSoftmaxRegs = 232;   // after setmaxnreg.inc
constexpr uint32_t kControlRegs = 40;    // after setmaxnreg.dec
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kNumThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(2 * kSoftmaxRegs + kControlRegs <= 512, "per-sub-partition register file");
constexpr int kRowThreadsPerTile = 128;
constexpr int kLoadWarp = 8;    // Q and K producer
constexpr int kMmaWarp = 9;
constexpr int kLoadVWarp = 10;  // V producer
constexpr uint32_t kSwBlockBytes = 128 * 128;  // [128 rows x 64 bf16] swizzled block
constexpr float kRescaleThreshold = 8.0f;      // log2 units: P stays <= 2^8

constexpr uint32_t kStatusTimeout = 1u;
constexpr uint32_t kInjectSkipFirstV = 1u;  // test hook: never issue the first V load

__device__ uint32_t g_fa_status;

struct FwdParams {
  float* lse;        // [BH][N] fp32
  int N;             // sequence length
  int num_units;     // ceil(N / kUnitM)
  int causal;        // 0 / 1
  float scale_log2;  // scale * log2(e); never 0 (scale 0 arrives as a tiny positive value)
  uint32_t inject;   // test hooks (0 in normal use)
  uint64_t wait_limit_ns;
};

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "head dimension");
  // Ring depths: 64 KB of Q plus 3 K and 2 V tiles of 32 KB fill 224 KB at
  // D = 128; at D = 64 the tiles are half as large.
  static constexpr int kStagesK = (D == 64) ? 4 : 3;
  static constexpr int kStagesV = (D == 64) ? 4 : 2;
  static constexpr uint32_t kQBytes = kTileM * D * 2;  // one query tile
  static constexpr uint32_t kKVBytes = kBlockN * D * 2;
  static constexpr uint32_t kOffQ = 0;  // Q_A, Q_B
  static constexpr uint32_t kOffK = kOffQ + kTilesPerCta * kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStagesK * kKVBytes;
  static constexpr uint32_t kOffBar = kOffV + kStagesV * kKVBytes;
  // q_full[2], s_full[2], p_full[2], o_done[2], mma_done,
  // k_full[SK], k_empty[SK], v_full[SV], v_empty[SV]
  static constexpr int kNumBars = 9 + 2 * kStagesK + 2 * kStagesV;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;  // slack for 1024-byte alignment
  static_assert(kSmemAlloc <= 232448, "dynamic shared memory per block");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // S_t at kColS + 128*t, P_t over its first 64 columns
  static constexpr uint32_t kColO = 256;  // O_t at kColO + D*t
  static constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileM, kBlockN, 0, 0);
  static constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileM, D, 0, 1);
};

// Barrier addresses (8 bytes each) in the order of the layout above.
struct Barriers {
  uint32_t base;
  int sk, sv;  // K and V ring depths
  __device__ uint32_t q_full(int t) const { return base + 8u * t; }
  __device__ uint32_t s_full(int t) const { return base + 16u + 8u * t; }
  __device__ uint32_t p_full(int t) const { return base + 32u + 8u * t; }
  __device__ uint32_t o_done(int t) const { return base + 48u + 8u * t; }
  __device__ uint32_t mma_done() const { return base + 64u; }
  __device__ uint32_t k_full(int s) const { return base + 72u + 8u * s; }
  __device__ uint32_t k_empty(int s) const { return base + 72u + 8u * (sk + s); }
  __device__ uint32_t v_full(int s) const { return base + 72u + 8u * (2 * sk + s); }
  __device__ uint32_t v_empty(int s) const { return base + 72u + 8u * (2 * sk + sv + s); }
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
__device__ __forceinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const WaitCtx& w) {
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

// Bounded wait whose result is uniform across the calling warp (every lane
// must call it): tcgen05.ld/st and warp votes that follow need the whole warp.
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const bool ok = wait_bar(bar, parity, w);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used while draining: ignores the abort flag (copies and MMAs
// already issued always complete), bounded by time alone.
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, const WaitCtx& w) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > w.limit_ns) break;
  }
  record_timeout(w);
  return false;
}

// AND-reduce a flag over the 128 threads of one tile (named barrier `id`).
__device__ __forceinline__ bool tile_threads_all(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %2, 0;\n\t"
      "bar.red.and.pred q, %1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// Byte offset of the 16-byte chunk `chunk` (0..D/8-1) of row `row` in a
// [128 x D] tile stored as 128-byte-swizzled [128 x 64] blocks.
__device__ __forceinline__ uint32_t swizzled_chunk(int row, int chunk) {
  return (chunk >> 3) * kSwBlockBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// Number of key tiles a query tile starting at row r0 must visit (0 when the
// tile lies entirely past the end of the sequence).  Causal: key tiles whose
// first key is at or past the tile's end are entirely in the future and are
// skipped (never loaded, never computed).
__device__ __forceinline__ int key_tiles_for(int r0, int N, int causal) {
  if (r0 >= N) return 0;
  const int kv_end = causal ? min(r0 + kTileM, N) : N;
  return (kv_end + kBlockN - 1) / kBlockN;
}

// ----------------------------------------------------------------------------
// Softmax warps of one query tile (128 threads, one row each)
// ----------------------------------------------------------------------------
template <int D, bool kNegScale>
__device__ __forceinline__ void softmax_tile(const int t, const int n_tiles, const int r0,
                                             const uint32_t tmem, const uint32_t sQt,
                                             const Barriers& bars, const WaitCtx& wctx,
                                             const CUtensorMap* tm_o, const FwdParams& p,
                                             const int bh) {
  using C = Cfg<D>;
  const int row = threadIdx.x & 127;  // row within the tile = TMEM lane
  const int warp_in_tile = (threadIdx.x >> 5) & 3;
  const uint32_t lane_off = static_cast<uint32_t>(warp_in_tile * 32) << 16;
  const uint32_t s_addr = tmem + lane_off + C::kColS + 128u * t;
  const uint32_t o_addr = tmem + lane_off + C::kColO + static_cast<uint32_t>(D) * t;
  const int q_idx = r0 + row;
  const float c = p.scale_log2;
  // Last key index this row may see: itself when causal, else N-1.
  const int row_last_key = p.causal ? min(q_idx, p.N - 1) : p.N - 1;
  float m_ref = -CUDART_INF_F;  // exponent reference, scaled log2 units
  float l_run = 0.0f;           // sum of 2^(scaled score - m_ref)
  bool ok = true;

  for (int j = 0; j < n_tiles; ++j) {
    if (!warp_wait_bar(bars.s_full(t), static_cast<uint32_t>(j) & 1u, wctx)) {
      ok = false;
      break;
    }
    tc_fence_after_sync();
    uint32_t sr[kBlockN];
#pragma unroll
    for (int cc = 0; cc < kBlockN / 32; ++cc)
      tmem_ld32(s_addr + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * cc]));
    tmem_ld_wait();
    float s[kBlockN];
#pragma unroll
    for (int i = 0; i < kBlockN; ++i) s[i] = __uint_as_float(sr[i]);

    const int k0 = j * kBlockN;
    if (k0 + kBlockN - 1 > row_last_key) {  // diagonal or ragged tile: mask per element
      const int lim = row_last_key - k0;
      const float masked = kNegScale ? CUDART_INF_F : -CUDART_INF_F;
#pragma unroll
      for (int i = 0; i < kBlockN; ++i)
        if (i > lim) s[i] = masked;
    }

    // Row extreme of the raw scores (max for a positive scale, min for a
    // negative one), four independent 3-input chains.
    float e0 = s[0], e1 = s[1], e2 = s[2], e3 = s[3];
#pragma unroll
    for (int i = 4; i < kBlockN; i += 8) {
      if (kNegScale) {
        e0 = fmin3(e0, s[i], s[i + 1]);
        e1 = fmin3(e1, s[i + 2], s[i + 3]);
        e2 = fmin3(e2, s[i + 4], s[i + 5]);
        e3 = fmin3(e3, s[i + 6], s[i + 7]);
      } else {
        e0 = fmax3(e0, s[i], s[i + 1]);
        e1 = fmax3(e1, s[i + 2], s[i + 3]);
        e2 = fmax3(e2, s[i + 4], s[i + 5]);
        e3 = fmax3(e3, s[i + 6], s[i + 7]);
      }
    }
    const float ext =
        kNegScale ? fminf(fminf(e0, e1), fminf(e2, e3)) : fmaxf(fmaxf(e0, e1), fmaxf(e2, e3));
    const float m_tile = ext * c;  // max of the scaled scores of this tile

    // Lazy rescale: move the reference only when the tile max exceeds it by
    // more than the threshold (always on the first tile, where m_ref = -inf).
    const bool rescale = __any_sync(0xffffffffu, m_tile > m_ref + kRescaleThreshold);
    float alpha = 1.0f;
    if (rescale) {
      const float m_new = fmaxf(m_ref, m_tile);
      alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile
      l_run *= alpha;
      m_ref = m_new;
    }

    // P = 2^(s*c - m_ref) and its row sum; P_t goes, as bf16 pairs, over the
    // first 64 columns of S_t (whose values are already in registers), in
    // two halves so that half of the scores are dead before the second.
    const float neg_m = -m_ref;
    float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 64; i += 4) {
        const int e = 64 * h + i;
        float x0, x1, x2, x3;
        ffma2(x0, x1, s[e], s[e + 1], c, c, neg_m, neg_m);
        ffma2(x2, x3, s[e + 2], s[e + 3], c, c, neg_m, neg_m);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
        fadd2(sa0, sa1, sa0, sa1, p0, p1);
        fadd2(sb0, sb1, sb0, sb1, p2, p3);
        pk[i / 2] = pack_bf16x2(p0, p1);
        pk[i / 2 + 1] = pack_bf16x2(p2, p3);
      }
      tmem_st32(s_addr + 32 * h, pk);
    }
    l_run += (sa0 + sa1) + (sb0 + sb1);

    if (rescale && j > 0) {
      // O_t holds every P.V product up to tile j-1 (the S_t(j) MMA was
      // committed after them) and no MMA touches it until p_full: rescale
      // it in place.
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32 * cc, o);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float a0, a1;
          fmul2(a0, a1, __uint_as_float(o[i]), __uint_as_float(o[i + 1]), alpha, alpha);
          o[i] = __float_as_uint(a0);
          o[i + 1] = __float_as_uint(a1);
        }
        tmem_st32(o_addr + 32 * cc, o);
      }
    }
    tmem_st_wait();
    tc_fence_before_sync();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bars.p_full(t));
  }

  // ---------------------------------------------------------------- epilogue
  if (ok && n_tiles > 0 && !warp_wait_bar(bars.o_done(t), 0u, wctx)) ok = false;
  if (tile_threads_all(1u + t, ok) && n_tiles > 0) {
    tc_fence_after_sync();
    const float inv_l = 1.0f / l_run;
    // Q_t is dead (its last MMA completed before the last P.V), so its SMEM
    // stages the bf16 output for the TMA store.
#pragma unroll
    for (int cc = 0; cc < D / 32; ++cc) {
      uint32_t o[32];
      tmem_ld32(o_addr + 32 * cc, o);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a0, a1;
          fmul2(a0, a1, __uint_as_float(o[8 * g + 2 * e]), __uint_as_float(o[8 * g + 2 * e + 1]),
                inv_l, inv_l);
          w4[e] = pack_bf16x2(a0, a1);
        }
        st_shared_v4(sQt + swizzled_chunk(row, 4 * cc + g), w4[0], w4[1], w4[2], w4[3]);
      }
    }
    fence_proxy_async_smem();
    named_barrier_sync(1u + t, kRowThreadsPerTile);
    if (row == 0) {
#pragma unroll
      for (int b = 0; b < D / 64; ++b) tma_store_3d(tm_o, sQt + b * kSwBlockBytes, 64 * b, r0, bh);
      tma_store_commit();
      tma_store_wait_all();
    }
    if (q_idx < p.N)
      p.lse[static_cast<size_t>(bh) * p.N + q_idx] =
          (m_ref + __log2f(l_run)) * 0.6931471805599453f;
  }
}

template <int D, bool kNegScale>
__global__ void __launch_bounds__(kNumThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using C = Cfg<D>;
  constexpr int SK = C::kStagesK;
  constexpr int SV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ;
  const uint32_t sK = sbase + C::kOffK;
  const uint32_t sV = sbase + C::kOffV;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  const Barriers bars{sbase + C::kOffBar, SK, SV};
  const WaitCtx wctx{abort_flag, p.wait_limit_ns};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int unit = p.num_units - 1 - static_cast<int>(blockIdx.y);  // heaviest first
  const int q0 = unit * kUnitM;
  int n_t[kTilesPerCta];
#pragma unroll
  for (int t = 0; t < kTilesPerCta; ++t) n_t[t] = key_tiles_for(q0 + kTileM * t, p.N, p.causal);
  const int n_max = max(n_t[0], n_t[1]);  // n_t[0] >= 1 always

  if (threadIdx.x == 0) {
    for (int t = 0; t < kTilesPerCta; ++t) {
      mbar_init(bars.q_full(t), 1);
      mbar_init(bars.s_full(t), 1);
      mbar_init(bars.p_full(t), kRowThreadsPerTile / 32);  // one arrival per warp
      mbar_init(bars.o_done(t), 1);
    }
    mbar_init(bars.mma_done(), 1);
    for (int s = 0; s < SK; ++s) {
      mbar_init(bars.k_full(s), 1);
      mbar_init(bars.k_empty(s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      mbar_init(bars.v_full(s), 1);
      mbar_init(bars.v_empty(s), 1);
    }
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

  // Register reallocation: one setmaxnreg per warpgroup, executed by all
  // four of its warps at the same instruction (it is warpgroup-aligned).
  if (warp < kLoadWarp) {
    setmaxnreg_inc<kSoftmaxRegs>();
  } else {
    setmaxnreg_dec<kControlRegs>();
  }

  if (warp < kLoadWarp) {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    softmax_tile<D, kNegScale>(t, n_t[t], q0 + kTileM * t, tmem, sQ + t * C::kQBytes, bars, wctx,
                               &tm_o, p, bh);
  } else if (warp == kLoadWarp) {
    // ------------------------------------------------------------ Q, K producer
    if (lane == 0) {
      int issued = 0;  // K_j copies issued for j < issued
      bool q_issued[kTilesPerCta] = {false, false};
      for (int j = 0; j < n_max; ++j) {
        const int s = j % SK;
        if (j >= SK && !wait_bar(bars.k_empty(s), (static_cast<uint32_t>(j / SK) & 1u) ^ 1u, wctx))
          break;
        if (j == 0) {  // Q_A first: S_A(0) needs only Q_A and K_0
          mbar_arrive_expect_tx(bars.q_full(0), C::kQBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(sQ + b * kSwBlockBytes, &tm_q, bars.q_full(0), 64 * b, q0, bh);
          q_issued[0] = true;
        }
        mbar_arrive_expect_tx(bars.k_full(s), C::kKVBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sK + s * C::kKVBytes + b * kSwBlockBytes, &tm_k, bars.k_full(s), 64 * b,
                      j * kBlockN, bh);
        issued = j + 1;
        if (j == 0 && n_t[1] > 0) {
          mbar_arrive_expect_tx(bars.q_full(1), C::kQBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b)
            tma_load_3d(sQ + C::kQBytes + b * kSwBlockBytes, &tm_q, bars.q_full(1), 64 * b,
                        q0 + kTileM, bh);
          q_issued[1] = true;
        }
      }
      // Drain: every copy issued must land before the CTA may exit.  The last
      // copy into stage s is the largest j < issued with j % SK == s.
#pragma unroll
      for (int t = 0; t < kTilesPerCta; ++t)
        if (q_issued[t]) wait_bar_drain(bars.q_full(t), 0, wctx);
#pragma unroll
      for (int s = 0; s < SK; ++s) {
        if (issued > s) {
          const int jl = issued - 1 - ((issued - 1 - s) % SK);
          wait_bar_drain(bars.k_full(s), static_cast<uint32_t>(jl / SK) & 1u, wctx);
        }
      }
    }
  } else if (warp == kLoadVWarp) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      int issued = 0;  // V_j copies issued (or deliberately skipped) for j < issued
      bool v0_skipped = false;
      for (int j = 0; j < n_max; ++j) {
        const int s = j % SV;
        if (j >= SV && !wait_bar(bars.v_empty(s), (static_cast<uint32_t>(j / SV) & 1u) ^ 1u, wctx))
          break;
        issued = j + 1;
        if (j == 0 && (p.inject & kInjectSkipFirstV)) {
          v0_skipped = true;
          continue;
        }
        mbar_arrive_expect_tx(bars.v_full(s), C::kKVBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_load_3d(sV + s * C::kKVBytes + b * kSwBlockBytes, &tm_v, bars.v_full(s), 64 * b,
                      j * kBlockN, bh);
      }
#pragma unroll
      for (int s = 0; s < SV; ++s) {
        if (issued > s) {
          const int jl = issued - 1 - ((issued - 1 - s) % SV);
          if (!(jl == 0 && v0_skipped))
            wait_bar_drain(bars.v_full(s), static_cast<uint32_t>(jl / SV) & 1u, wctx);
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // Descriptor halves.  Every operand sits at a fixed SMEM address, so
      // the low halves of all descriptors are a base plus compile-time
      // offsets (>> 4) and each MMA issue costs a couple of integer adds.
      constexpr uint32_t kHi = desc_hi_sw128(1024);
      const uint32_t q_lo = desc_lo(sQ, 16);
      const uint32_t k_lo = desc_lo(sK, 16);
      const uint32_t v_lo = desc_lo(sV, kSwBlockBytes);
      // K-major slice kk of a [128 x D] tile: block kk/4, 32 bytes per slice.
      auto kmaj_off = [](int kk) -> uint32_t {
        return ((kk >> 2) * kSwBlockBytes + (kk & 3) * 32) >> 4;
      };
      auto issue_s = [&](int t, int j) {
        const uint32_t a_lo = q_lo + ((t * C::kQBytes) >> 4);
        const uint32_t b_lo = k_lo + (((j % SK) * C::kKVBytes) >> 4);
        const uint32_t d_tmem = tmem + C::kColS + 128u * t;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_lohi(d_tmem, a_lo + kmaj_off(kk), kHi, b_lo + kmaj_off(kk), kHi, C::kIdescQK,
                       kk > 0 ? 1u : 0u);
        umma_commit(bars.s_full(t));
      };
      auto issue_pv = [&](int t, int j) {
        // V slice kk: 16 key rows of 128 bytes.
        const uint32_t b_lo = v_lo + (((j % SV) * C::kKVBytes) >> 4);
        const uint32_t p_tmem = tmem + C::kColS + 128u * t;
        const uint32_t d_tmem = tmem + C::kColO + static_cast<uint32_t>(D) * t;
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_ts_lohi(d_tmem, p_tmem + 8u * kk, b_lo + ((kk * 16 * 128) >> 4), kHi, C::kIdescPV,
                       kk > 0 ? 1u : acc0);
      };
      auto wait_k = [&](int j) {
        return wait_bar(bars.k_full(j % SK), static_cast<uint32_t>(j / SK) & 1u, wctx);
      };

      bool ok = wait_k(0) && wait_bar(bars.q_full(0), 0, wctx);
      if (ok) {
        tc_fence_after_sync();
        issue_s(0, 0);
        if (n_t[1] > 0) {
          ok = wait_bar(bars.q_full(1), 0, wctx);
          if (ok) {
            tc_fence_after_sync();
            issue_s(1, 0);
          }
        }
        if (ok) umma_commit(bars.k_empty(0));
      }
      // Issuing a tcgen05.mma waits for room in the tensor core's queue, so
      // this thread runs only a little ahead of the MMAs: every wait, fence
      // or commit between two MMA groups is tensor-core idle time.  All
      // waits of an iteration therefore come first (the TMA waits are
      // normally already satisfied), and commits are batched after groups.
      for (int j = 0; ok && j < n_max; ++j) {
        const int s = j % SV;
        const bool more = j + 1 < n_max;
        if (!wait_bar(bars.v_full(s), static_cast<uint32_t>(j / SV) & 1u, wctx)) break;
        if (more && !wait_k(j + 1)) break;
#pragma unroll
        for (int t = 0; t < kTilesPerCta; ++t) {
          if (j >= n_t[t]) continue;
          if (!wait_bar(bars.p_full(t), static_cast<uint32_t>(j) & 1u, wctx)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_pv(t, j);
          if (j + 1 < n_t[t]) {
            issue_s(t, j + 1);  // commits s_full(t), which also covers P_t(j) V_j
          } else {
            umma_commit(bars.o_done(t));
          }
        }
        if (!ok) break;
        umma_commit(bars.v_empty(s));                 // V_j: both P.V products issued
        if (more) umma_commit(bars.k_empty((j + 1) % SK));  // K_j+1: both S MMAs issued
      }
      // Drain: wait for every MMA issued by this thread.
      umma_commit(bars.mma_done());
      wait_bar_drain(bars.mma_done(), 0, wctx);
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
