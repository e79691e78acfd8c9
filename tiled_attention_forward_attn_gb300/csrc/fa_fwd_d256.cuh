// Fused attention forward for head dimension 256 on sm_103a: the method of
// fa_fwd_kernel.cuh (tiled online softmax, "Q/O stay, K/V move", causal
// tiles past the diagonal skipped, lazy rescale, one division at the end),
// laid out for a 256-column accumulator.
//
// Two query tiles per CTA would need 2 x (128 + 256) TMEM columns, more than
// the 512 there are, so a work unit is one 128-row query tile and the
// tensor core is kept busy by double-buffering S instead: keys come in
// 64-key tiles, S(j) lives in one of two 64-column TMEM buffers, and while
// the softmax warps turn S(j) into P(j) the tensor core computes S(j+1) and
// then P(j-1) V(j-1).  TMEM: S buffers [0,64) and [64,128), O [256,512).
// SMEM: Q 64 KB, a 3-stage K ring and a 2-stage V ring of 32 KB tiles.
//
// pv_done completes one phase per P.V.  A parity wait is only meaningful
// while the waiter is at most one phase behind, so the softmax warps
// confirm the previous tile's P.V on every tile (at the rescale point, or
// just before handing over P; the P.V after that cannot start earlier).
//
// Warps: 0-3 softmax and epilogue (thread = row = TMEM lane), 4 TMA producer
// of Q and K, 5 TMEM allocator and MMA issuer, 6 TMA producer of V, 7 idle.
// The persistent grid walks (batch*head, query tile) units heaviest first in
// a serpentine, like the main kernel.  O is rescaled in place only when the
// reference max moves (rare); before that the softmax warps wait for the
// previous P.V to complete (pv_done).  Every wait is bounded (status word,
// drain, TMEM freed).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "fa_fwd_kernel.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kW_TileM = 128;   // query rows per unit
constexpr int kW_BlockN = 64;   // keys per K/V tile
constexpr int kW_D = 256;
constexpr int kW_Threads = 256;
constexpr int kW_LoadWarp = 4, kW_MmaWarp = 5, kW_LoadVWarp = 6;
constexpr int kW_StagesK = 3, kW_StagesV = 2;

struct WideCfg {
  static constexpr uint32_t kQBlock = kW_TileM * 128;   // 64 columns x 128 rows
  static constexpr uint32_t kKVBlock = kW_BlockN * 128;  // 64 columns x 64 rows
  static constexpr uint32_t kQBytes = kW_TileM * kW_D * 2;   // 64 KB
  static constexpr uint32_t kKVBytes = kW_BlockN * kW_D * 2;  // 32 KB
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + kQBytes;
  static constexpr uint32_t kOffV = kOffK + kW_StagesK * kKVBytes;
  static constexpr uint32_t kOffBar = kOffV + kW_StagesV * kKVBytes;
  // q_full, q_empty, s_full[2], p_full[2], pv_done, mma_done, k_full/empty[SK], v_full/empty[SV]
  static constexpr int kNumBars = 8 + 2 * kW_StagesK + 2 * kW_StagesV;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "dynamic shared memory per block");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // buffer b at 64 b; P as 16-bit pairs over its first 32 columns
  static constexpr uint32_t kColO = 256;
};

struct WideBars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t q_empty() const { return base + 8u; }
  __device__ uint32_t s_full(int b) const { return base + 16u + 8u * b; }
  __device__ uint32_t p_full(int b) const { return base + 32u + 8u * b; }
  __device__ uint32_t pv_done() const { return base + 48u; }
  __device__ uint32_t mma_done() const { return base + 56u; }
  __device__ uint32_t k_full(int s) const { return base + 64u + 8u * s; }
  __device__ uint32_t k_empty(int s) const { return base + 64u + 8u * (kW_StagesK + s); }
  __device__ uint32_t v_full(int s) const { return base + 64u + 8u * (2 * kW_StagesK + s); }
  __device__ uint32_t v_empty(int s) const {
    return base + 64u + 8u * (2 * kW_StagesK + kW_StagesV + s);
  }
};

struct WideUnit {
  int bh, b, h, q0, n;  // n: 64-key tiles this query tile visits
};

__device__ __forceinline__ WideUnit wide_unit_at(int idx, const FwdParams& p) {
  WideUnit u;
  const int qt = p.num_units - 1 - idx / p.num_bh;  // heaviest (last) query tile first
  u.bh = idx % p.num_bh;
  u.b = u.bh / p.H;
  u.h = u.bh - u.b * p.H;
  u.q0 = qt * kW_TileM;
  const int kv_end = p.causal ? min(u.q0 + kW_TileM, p.N) : p.N;
  u.n = (kv_end + kW_BlockN - 1) / kW_BlockN;
  return u;
}

template <bool kNegScale, bool kF16>
__global__ void __launch_bounds__(kW_Threads, 1)
    fa_fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = WideCfg;
  constexpr int SK = kW_StagesK, SV = kW_StagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ, sK = sbase + C::kOffK, sV = sbase + C::kOffV;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  const WideBars bars{sbase + C::kOffBar};
  const WaitCtx wctx{abort_flag, p.wait_limit_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.s_full(b), 1);
      mbar_init(bars.p_full(b), 4);  // one arrival per softmax warp
    }
    mbar_init(bars.pv_done(), 1);
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
  if (warp == kW_MmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kW_LoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t o_addr = tmem + lane_off + C::kColO;
    const float c = p.scale_log2;
    uint32_t su[2] = {0u, 0u};  // s_full phases consumed per buffer
    uint32_t pv_seen = 0;       // P.V products issued before the current tile (global count)
    uint32_t gt = 0;            // key tiles processed so far (buffer of tile = gt & 1)
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int idx = unit_index(r);
      if (idx >= p.total_units) break;
      const WideUnit u = wide_unit_at(idx, p);
      const int q_idx = u.q0 + row;
      const int row_last_key = p.causal ? min(q_idx, p.N - 1) : p.N - 1;
      float m_ref = -CUDART_INF_F, l_run = 0.0f;
      for (int j = 0; j < u.n; ++j, ++gt) {
        const int b = static_cast<int>(gt & 1u);
        if (!warp_wait_bar(bars.s_full(b), parity_of(su[b]), wctx)) {
          ok = false;
          break;
        }
        ++su[b];
        tc_fence_after_sync();
        const uint32_t s_addr = tmem + lane_off + C::kColS + 64u * b;
        uint32_t sr[64];
        tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld_wait();
        tmem_ld_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        float s[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(sr[i]);
        const int k0 = j * kW_BlockN;
        if (k0 + kW_BlockN - 1 > row_last_key) {
          const int lim = row_last_key - k0;
          const float masked = kNegScale ? CUDART_INF_F : -CUDART_INF_F;
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (i > lim) s[i] = masked;
        }
        float ev[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) ev[k] = s[k];
#pragma unroll
        for (int i = 8; i < 64; i += 8)
#pragma unroll
          for (int k = 0; k < 8; ++k)
            ev[k] = kNegScale ? fminf(ev[k], s[i + k]) : fmaxf(ev[k], s[i + k]);
#pragma unroll
        for (int w = 4; w > 0; w >>= 1)
#pragma unroll
          for (int k = 0; k < w; ++k)
            ev[k] = kNegScale ? fminf(ev[k], ev[k + w]) : fmaxf(ev[k], ev[k + w]);
        const float m_tile = ev[0] * c;
        const bool rescale = __any_sync(0xffffffffu, m_tile > m_ref + kRescaleThreshold);
        // The previous P.V: within the unit, confirmed on this tile; at a
        // unit's first tile it was confirmed by the previous epilogue.
        bool prev_pv_seen = j == 0;
        if (rescale) {
          const float m_new = fmaxf(m_ref, m_tile);
          const float alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile
          l_run *= alpha;
          m_ref = m_new;
          if (j > 0) {
            // O holds P.V products up to tile j-1 once the last of them is
            // complete (at most one P.V is in flight: the next is issued
            // only after this tile's p_full).
            if (!warp_wait_bar(bars.pv_done(), parity_of(pv_seen - 1), wctx)) {
              ok = false;
              break;
            }
            prev_pv_seen = true;
            tc_fence_after_sync();
#pragma unroll 1
            for (int cc = 0; cc < kW_D / 32; ++cc) {
              uint32_t o[32];
              tmem_ld32(o_addr + 32 * cc, o);
              tmem_ld_wait();
              tmem_ld_fence(o);
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
        }
        const float neg_m = -m_ref;
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          float x0, x1, x2, x3;
          ffma2(x0, x1, s[i], s[i + 1], c, c, neg_m, neg_m);
          ffma2(x2, x3, s[i + 2], s[i + 3], c, c, neg_m, neg_m);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          const float p2 = ex2_approx(x2), p3 = ex2_approx(x3);
          fadd2(sa0, sa1, sa0, sa1, p0, p1);
          fadd2(sb0, sb1, sb0, sb1, p2, p3);
          pk[i / 2] = pack_x2<kF16>(p0, p1);
          pk[i / 2 + 1] = pack_x2<kF16>(p2, p3);
        }
        tmem_st32(s_addr, pk);
        l_run += (sa0 + sa1) + (sb0 + sb1);
        if (!prev_pv_seen && !warp_wait_bar(bars.pv_done(), parity_of(pv_seen - 1), wctx)) {
          ok = false;
          break;
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.p_full(b));
        ++pv_seen;  // the P.V of this tile is issued after p_full
      }
      if (!ok) break;
      // ------------------------------------------------------------ epilogue
      if (!warp_wait_bar(bars.pv_done(), parity_of(pv_seen - 1), wctx)) break;
      tc_fence_after_sync();
      const float inv_l = 1.0f / l_run;
      const bool in_range = q_idx < p.N;
      uint4* dst = reinterpret_cast<uint4*>(p.o + u.b * p.o_sb + u.h * p.o_sh + q_idx * p.o_sn);
#pragma unroll 1
      for (int cc = 0; cc < kW_D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(o_addr + 32 * cc, o);
        tmem_ld_wait();
        tmem_ld_fence(o);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float a0, a1;
            fmul2(a0, a1, __uint_as_float(o[8 * g + 2 * e]), __uint_as_float(o[8 * g + 2 * e + 1]),
                  inv_l, inv_l);
            w4[e] = pack_x2<kF16>(a0, a1);
          }
          if (in_range) dst[4 * cc + g] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
      if (in_range)
        p.lse[static_cast<size_t>(u.bh) * p.N + q_idx] = (m_ref + __log2f(l_run)) * 0.6931471805599453f;
      // O is read: the next unit's first P.V (which overwrites O) waits for
      // that unit's first p_full, after this point.
      tc_fence_before_sync();
    }
  } else if (warp == kW_LoadWarp) {
    // ------------------------------------------------------------ Q, K producer
    if (lane == 0) {
      const uint64_t keep = make_l2_policy_evict_last();
      const uint64_t once = make_l2_policy_evict_first();
      uint32_t kc = 0, qc = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = unit_index(r);
        if (idx >= p.total_units) break;
        const WideUnit u = wide_unit_at(idx, p);
        if (qc > 0 && !wait_bar(bars.q_empty(), parity_of(qc - 1), wctx)) break;
        mbar_arrive_expect_tx(bars.q_full(), C::kQBytes);
#pragma unroll
        for (int b = 0; b < kW_D / 64; ++b)
          tma_load_4d_hint(sQ + b * C::kQBlock, &tm_q, bars.q_full(), 64 * b, u.q0, u.h, u.b, once);
        ++qc;
        for (int j = 0; j < u.n; ++j) {
          const int s = static_cast<int>(kc % SK);
          if (kc >= static_cast<uint32_t>(SK) &&
              !wait_bar(bars.k_empty(s), parity_of(kc / SK - 1), wctx)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.k_full(s), C::kKVBytes);
#pragma unroll
          for (int b = 0; b < kW_D / 64; ++b)
            tma_load_4d_hint(sK + s * C::kKVBytes + b * C::kKVBlock, &tm_k, bars.k_full(s), 64 * b,
                             j * kW_BlockN, u.h, u.b, keep);
          ++kc;
        }
      }
      if (qc > 0) wait_bar_drain(bars.q_full(), parity_of(qc - 1), wctx);
      for (int s = 0; s < SK; ++s) {
        if (kc > static_cast<uint32_t>(s)) {
          const uint32_t last = kc - 1 - ((kc - 1 - s) % SK);
          wait_bar_drain(bars.k_full(s), parity_of(last / SK), wctx);
        }
      }
    }
  } else if (warp == kW_LoadVWarp) {
    // ------------------------------------------------------------ V producer
    if (lane == 0) {
      const uint64_t keep = make_l2_policy_evict_last();
      uint32_t vc = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int idx = unit_index(r);
        if (idx >= p.total_units) break;
        const WideUnit u = wide_unit_at(idx, p);
        for (int j = 0; j < u.n; ++j) {
          const int s = static_cast<int>(vc % SV);
          if (vc >= static_cast<uint32_t>(SV) &&
              !wait_bar(bars.v_empty(s), parity_of(vc / SV - 1), wctx)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bars.v_full(s), C::kKVBytes);
#pragma unroll
          for (int b = 0; b < kW_D / 64; ++b)
            tma_load_4d_hint(sV + s * C::kKVBytes + b * C::kKVBlock, &tm_v, bars.v_full(s), 64 * b,
                             j * kW_BlockN, u.h, u.b, keep);
          ++vc;
        }
      }
      for (int s = 0; s < SV; ++s) {
        if (vc > static_cast<uint32_t>(s)) {
          const uint32_t last = vc - 1 - ((vc - 1 - s) % SV);
          wait_bar_drain(bars.v_full(s), parity_of(last / SV), wctx);
        }
      }
    }
  } else if (warp == kW_MmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one_sync();
    constexpr uint32_t kHi = desc_hi_sw128(1024);
    constexpr uint32_t kIdescS = kF16 ? idesc_f16_f32(kW_TileM, kW_BlockN, 0, 0)
                                      : idesc_bf16_f32(kW_TileM, kW_BlockN, 0, 0);
    constexpr uint32_t kIdescPV = kF16 ? idesc_f16_f32(kW_TileM, kW_D, 0, 1)
                                       : idesc_bf16_f32(kW_TileM, kW_D, 0, 1);
    const uint32_t q_lo = desc_lo(sQ, 16);
    const uint32_t k_lo = desc_lo(sK, 16);
    const uint32_t v_lo = desc_lo(sV, C::kKVBlock);  // MN-major: 64-column blocks 8 KB apart
    auto commit = [&](uint32_t bar) {
      if (leader) umma_commit(bar);
      __syncwarp();
    };
    auto issue_s = [&](int b, uint32_t k_stage) {  // S_b = Q K^T, 16 K-slices of 16 columns
      const uint32_t kb = k_lo + ((k_stage * C::kKVBytes) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kW_D / 16; ++kk)
          umma_ss_lohi(tmem + C::kColS + 64u * b,
                       q_lo + (((kk >> 2) * C::kQBlock + (kk & 3) * 32) >> 4), kHi,
                       kb + (((kk >> 2) * C::kKVBlock + (kk & 3) * 32) >> 4), kHi, kIdescS,
                       kk > 0 ? 1u : 0u);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int b, uint32_t v_stage, bool first) {  // O (+)= P_b V, 4 slices of 16 keys
      const uint32_t vb = v_lo + ((v_stage * C::kKVBytes) >> 4);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < kW_BlockN / 16; ++kk)
          umma_ts_lohi(tmem + C::kColO, tmem + C::kColS + 64u * b + 8u * kk,
                       vb + ((kk * 16 * 128) >> 4), kHi, kIdescPV, (kk > 0 || !first) ? 1u : 0u);
      }
      __syncwarp();
    };
    uint32_t kc = 0, vc = 0, qc = 0, gt = 0;
    uint32_t pu[2] = {0u, 0u};  // p_full phases consumed per buffer
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int idx = unit_index(r);
      if (idx >= p.total_units) break;
      const WideUnit u = wide_unit_at(idx, p);
      if (!warp_wait_bar(bars.q_full(), parity_of(qc), wctx)) break;
      ++qc;
      // S(0) and S(1) ahead of the softmax.
      for (int j = 0; ok && j < 2 && j < u.n; ++j) {
        if (!warp_wait_bar(bars.k_full(kc % SK), parity_of(kc / SK), wctx)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_s(static_cast<int>((gt + j) & 1u), kc % SK);
        commit(bars.s_full(static_cast<int>((gt + j) & 1u)));
        commit(bars.k_empty(kc % SK));
        if (j == u.n - 1) commit(bars.q_empty());  // last S of the unit
        ++kc;
      }
      for (int j = 0; ok && j < u.n; ++j) {
        const int b = static_cast<int>((gt + j) & 1u);
        if (!warp_wait_bar(bars.v_full(vc % SV), parity_of(vc / SV), wctx) ||
            !warp_wait_bar(bars.p_full(b), parity_of(pu[b]), wctx)) {
          ok = false;
          break;
        }
        ++pu[b];
        tc_fence_after_sync();
        issue_pv(b, vc % SV, j == 0);
        commit(bars.v_empty(vc % SV));
        commit(bars.pv_done());
        ++vc;
        if (j + 2 < u.n) {
          // S(j+2) overwrites P(j) in buffer b after the P.V that reads it.
          if (!warp_wait_bar(bars.k_full(kc % SK), parity_of(kc / SK), wctx)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(b, kc % SK);
          commit(bars.s_full(b));
          commit(bars.k_empty(kc % SK));
          if (j + 2 == u.n - 1) commit(bars.q_empty());
          ++kc;
        }
      }
      gt += static_cast<uint32_t>(u.n);
    }
    commit(bars.mma_done());
    wait_bar_drain(bars.mma_done(), 0, wctx);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kW_MmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
