// Fused attention forward for head dimension 256 on sm_103a: the method of
// fa_fwd_kernel.cuh (the tiled online softmax of "Parsing FlashAttention (2):
// FlashAttention-v1 forward pass" §2-§3 in the loop order of "Online Softmax
// and FlashAttention", course unit 12: "Q/O stay, K/V move", causal tiles
// past the diagonal skipped, lazy exponent reference, one division at the
// end), laid out for a 256-column accumulator.
//
// Two query tiles per CTA would need 2 x (128 + 256) TMEM columns, more than
// the 512 there are, so a work unit is one 128-row query tile and the
// tensor core is kept busy by double-buffering S instead: keys come in
// 64-key tiles, S(j) lives in one of two 64-column TMEM buffers, and while
// the softmax warps turn S(j) into P(j) the tensor core computes P(j-1) V
// and S(j+1).
//
// Q lives in TMEM too, as 16-bit pairs (128 columns): S = Q K^T is then a
// TS-form MMA that reads only K (2 KB per 128x64x16 step) from shared
// memory, at the tensor core's full rate; with Q in shared memory too the
// 64-key product is bound by shared-memory bandwidth (6 KB per step, 48
// instead of 32 cycles).  The softmax warps copy each unit's Q from the
// swizzled shared-memory tile into TMEM once its last S MMA of the previous
// unit has completed, before that unit's epilogue, so the next unit's first
// S MMAs overlap the epilogue.
//
// TMEM: S buffers [0,64) and [64,128) (P as 16-bit pairs over the first 32
// columns of its buffer), Q [128,256), O [256,512).  SMEM: the Q staging
// tile (64 KB) and one ring of five 32 KB K/V tiles filled in the order the
// MMAs read them (K_0, K_1, then V_j, K_j+2).
//
// pv_done completes one phase per P.V.  A parity wait is only meaningful
// while the waiter is at most one phase behind, so the softmax warps
// confirm the previous tile's P.V on every tile (when the reference moves,
// or just before handing over P; the P.V after that cannot start earlier).
//
// Warps: 0-3 softmax, Q copy and epilogue (thread = row = TMEM lane), 4 TMA
// producer of Q and the K/V ring, 5 TMEM allocator and MMA issuer, 6-7
// idle.  The persistent grid walks (batch*head, query tile) units heaviest
// first in a serpentine, like the main kernel.  Every wait is bounded
// (status word, drain, TMEM freed).
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
constexpr int kW_LoadWarp = 4, kW_MmaWarp = 5;
constexpr int kW_Slots = 5;     // K/V ring depth

struct WideCfg {
  static constexpr uint32_t kQBlock = kW_TileM * 128;   // 64 columns x 128 rows
  static constexpr uint32_t kKVBlock = kW_BlockN * 128;  // 64 columns x 64 rows
  static constexpr uint32_t kQBytes = kW_TileM * kW_D * 2;   // 64 KB
  static constexpr uint32_t kKVBytes = kW_BlockN * kW_D * 2;  // 32 KB
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffRing = kOffQ + kQBytes;
  static constexpr uint32_t kOffBar = kOffRing + kW_Slots * kKVBytes;
  // q_full, q_empty, q_tmem, s_full[2], p_full[2], pv_done, mma_done, kv_full[R], kv_empty[R]
  static constexpr int kNumBars = 9 + 2 * kW_Slots;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "dynamic shared memory per block");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;    // buffer b at 64 b
  static constexpr uint32_t kColQ = 128;  // Q as 16-bit pairs, 128 columns
  static constexpr uint32_t kColO = 256;
};

struct WideBars {
  uint32_t base;
  __device__ uint32_t q_full() const { return base; }
  __device__ uint32_t q_empty() const { return base + 8u; }
  __device__ uint32_t q_tmem() const { return base + 16u; }
  __device__ uint32_t s_full(int b) const { return base + 24u + 8u * b; }
  __device__ uint32_t p_full(int b) const { return base + 40u + 8u * b; }
  __device__ uint32_t pv_done() const { return base + 56u; }
  __device__ uint32_t mma_done() const { return base + 64u; }
  __device__ uint32_t kv_full(int s) const { return base + 72u + 8u * s; }
  __device__ uint32_t kv_empty(int s) const { return base + 72u + 8u * (kW_Slots + s); }
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
  constexpr int R = kW_Slots;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::kOffQ, sRing = sbase + C::kOffRing;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  const WideBars bars{sbase + C::kOffBar};
  const WaitCtx wctx{abort_flag, p.wait_limit_ns};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(bars.q_full(), 1);
    mbar_init(bars.q_empty(), 4);  // one arrival per softmax warp, after its copy
    mbar_init(bars.q_tmem(), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.s_full(b), 1);
      mbar_init(bars.p_full(b), 4);  // one arrival per softmax warp
    }
    mbar_init(bars.pv_done(), 1);
    mbar_init(bars.mma_done(), 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(bars.kv_full(s), 1);
      mbar_init(bars.kv_empty(s), 1);
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
    uint32_t qc = 0;            // Q tiles copied into TMEM so far
    // This row of the staged Q tile into TMEM as 16-bit pairs: 16-byte chunk
    // c of the row sits in 64-column block c / 8 at row * 128 + ((c % 8) ^
    // (row % 8)) * 16 (the 128-byte swizzle of the TMA copy).
    auto copy_q = [&]() -> bool {
      if (!warp_wait_bar(bars.q_full(), parity_of(qc), wctx)) return false;
      ++qc;
#pragma unroll
      for (int h = 0; h < kW_D / 64; ++h) {
        uint32_t wv[32];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const uint4 v4 = *reinterpret_cast<const uint4*>(
              smem + C::kOffQ + h * C::kQBlock + row * 128 + ((c8 ^ (row & 7)) << 4));
          wv[4 * c8] = v4.x;
          wv[4 * c8 + 1] = v4.y;
          wv[4 * c8 + 2] = v4.z;
          wv[4 * c8 + 3] = v4.w;
        }
        tmem_st32(tmem + lane_off + C::kColQ + 32 * h, wv);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.q_empty());  // the staging tile may be refilled
        mbar_arrive(bars.q_tmem());   // the S MMAs may read Q
      }
      return true;
    };
    bool ok = unit_index(0) >= p.total_units || copy_q();
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
        float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
        uint32_t pk[32];
        auto exps = [&](float neg_m) {
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
        };
        // Lazy reference, as in the main kernel: P against the current m_ref
        // with no row extreme; the reference moves to the true maximum only
        // on the unit's first tile or when the tile's P sum exceeds 2^15.
        // The previous P.V: within the unit, confirmed on this tile; at a
        // unit's first tile it was confirmed by the previous epilogue.
        bool prev_pv_seen = j == 0;
        bool moved = j == 0;
        if (!moved) {
          exps(-m_ref);
          moved = __any_sync(0xffffffffu, !((sa0 + sa1) + (sb0 + sb1) <= kPSumLimit));
        }
        if (moved) {
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
          const float m_new = fmaxf(m_ref, ev[0] * c);
          const float alpha = ex2_approx(m_ref - m_new);  // 0 on the first tile
          l_run *= alpha;
          m_ref = m_new;
          sa0 = sa1 = sb0 = sb1 = 0.f;
          exps(-m_ref);
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
      // The next unit's Q into TMEM: every S MMA of this unit has completed
      // (the last one was waited for above), so the Q columns are free, and
      // the next unit's first S MMAs then run during this epilogue.
      if (unit_index(r + 1) < p.total_units && !copy_q()) break;
      // ------------------------------------------------------------ epilogue
      // O = O / l in the element type, in two halves of 128 columns (each read
      // from TMEM with one wait), straight to global memory: each thread
      // writes its own row, 32-byte stores where O's alignment allows.
      if (!warp_wait_bar(bars.pv_done(), parity_of(pv_seen - 1), wctx)) break;
      tc_fence_after_sync();
      const float inv_l = 1.0f / l_run;
      const bool in_range = q_idx < p.N;
      uint16_t* orow = p.o + u.b * p.o_sb + u.h * p.o_sh + q_idx * p.o_sn;
#pragma unroll 1
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t ov[128];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(o_addr + 128 * hh + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&ov[32 * cc]));
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld_fence(*reinterpret_cast<uint32_t(*)[32]>(&ov[32 * cc]));
        uint32_t w[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float a0, a1;
          fmul2(a0, a1, __uint_as_float(ov[2 * i]), __uint_as_float(ov[2 * i + 1]), inv_l, inv_l);
          w[i] = pack_x2<kF16>(a0, a1);
        }
        if (in_range && guard(u.bh < p.num_bh && u.h < p.H && q_idx >= 0)) {
          if (p.o_vec32) {
#pragma unroll
            for (int g = 0; g < 8; ++g) st_global_v8(orow + 128 * hh + 16 * g, &w[8 * g]);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + 128 * hh);
#pragma unroll
            for (int g = 0; g < 16; ++g)
              dst[g] = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
          }
        }
      }
      if (in_range && guard(u.bh < p.num_bh && q_idx >= 0))
        p.lse[static_cast<size_t>(u.bh) * p.N + q_idx] = (m_ref + __log2f(l_run)) * 0.6931471805599453f;
      // O is read: the next unit's first P.V (which overwrites O) waits for
      // that unit's first p_full, after this point.
      tc_fence_before_sync();
    }
  } else if (warp == kW_LoadWarp) {
    // ------------------------------------------------------------ Q, K, V producer
    if (lane == 0) {
      const uint64_t keep = make_l2_policy_evict_last();
      const uint64_t once = make_l2_policy_evict_first();
      uint32_t ic = 0, qc = 0;  // K/V items and Q tiles issued (or skipped) so far
      int64_t skipped = -1;     // test hook: the item never issued
      bool v_seen = false;
      int cur_h = 0, cur_b = 0;
      // One K or V tile into the next ring slot, once that slot is free.
      auto issue = [&](const CUtensorMap* map, int row0, bool skip) -> bool {
        const int s = static_cast<int>(ic % R);
        if (ic >= static_cast<uint32_t>(R) &&
            !wait_bar(bars.kv_empty(s), parity_of(ic / R - 1), wctx))
          return false;
        if (skip) {
          skipped = ic;
        } else {
          mbar_arrive_expect_tx(bars.kv_full(s), C::kKVBytes);
#pragma unroll
          for (int b = 0; b < kW_D / 64; ++b)
            if (tma_coord_ok(64 * b, kW_D, row0, p.N, cur_b * p.H + cur_h, p.num_bh) &&
                smem_range_ok(C::kOffRing + s * C::kKVBytes + b * C::kKVBlock, C::kKVBlock,
                              C::kOffBar))
              tma_load_4d_hint(sRing + s * C::kKVBytes + b * C::kKVBlock, map, bars.kv_full(s),
                               64 * b, row0, cur_h, cur_b, keep);
        }
        ++ic;
        return true;
      };
      for (int r = 0;; ++r) {
        const int idx = unit_index(r);
        if (idx >= p.total_units) break;
        const WideUnit u = wide_unit_at(idx, p);
        cur_h = u.h;
        cur_b = u.b;
        // Q of this unit replaces the previous one in the staging tile once
        // the softmax warps have copied that one into TMEM (q_empty).
        if (qc > 0 && !wait_bar(bars.q_empty(), parity_of(qc - 1), wctx)) break;
        mbar_arrive_expect_tx(bars.q_full(), C::kQBytes);
#pragma unroll
        for (int b = 0; b < kW_D / 64; ++b)
          if (tma_coord_ok(64 * b, kW_D, u.q0, p.N, u.bh, p.num_bh) &&
              smem_range_ok(C::kOffQ + b * C::kQBlock, C::kQBlock, C::kOffRing))
            tma_load_4d_hint(sQ + b * C::kQBlock, &tm_q, bars.q_full(), 64 * b, u.q0, u.h, u.b, once);
        ++qc;
        // Items in the order the MMAs read them: K_0, K_1, then V_j, K_j+2.
        bool ok = issue(&tm_k, 0, false) && (u.n < 2 || issue(&tm_k, kW_BlockN, false));
        for (int j = 0; ok && j < u.n; ++j) {
          const bool skip = !v_seen && (p.inject & kInjectSkipFirstV);
          v_seen = true;
          ok = issue(&tm_v, j * kW_BlockN, skip) &&
               (j + 2 >= u.n || issue(&tm_k, (j + 2) * kW_BlockN, false));
        }
        if (!ok) break;
      }
      // Drain: every copy issued must land before the CTA may exit.  The last
      // item in slot s is the largest count < ic congruent to s mod R.
      if (qc > 0) wait_bar_drain(bars.q_full(), parity_of(qc - 1), wctx);
      for (int s = 0; s < R; ++s) {
        if (ic > static_cast<uint32_t>(s)) {
          const uint32_t last = ic - 1 - ((ic - 1 - s) % R);
          if (static_cast<int64_t>(last) != skipped)
            wait_bar_drain(bars.kv_full(s), parity_of(last / R), wctx);
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
    const uint32_t k_lo = desc_lo(sRing, 16);             // K slots, K-major
    const uint32_t v_lo = desc_lo(sRing, C::kKVBlock);    // V slots, MN-major: 64-column blocks 8 KB apart
    auto commit = [&](uint32_t bar) {
      if (leader) umma_commit(bar);
      __syncwarp();
    };
    // S_b = Q K^T: Q (16-bit pairs) from TMEM, 16 K-slices of 16 columns of
    // the K tile in ring slot `slot`.
    auto issue_s = [&](int b, uint32_t slot) {
      const uint32_t kb = k_lo + ((slot * C::kKVBytes) >> 4);
      if (leader && tmem_range_ok(tmem + C::kColS + 64u * b, kW_BlockN) &&
          tmem_range_ok(tmem + C::kColQ, kW_D / 2) && guard(slot < static_cast<uint32_t>(R))) {
#pragma unroll
        for (int kk = 0; kk < kW_D / 16; ++kk)
          umma_ts_lohi(tmem + C::kColS + 64u * b, tmem + C::kColQ + 8u * kk,
                       kb + (((kk >> 2) * C::kKVBlock + (kk & 3) * 32) >> 4), kHi, kIdescS,
                       kk > 0 ? 1u : 0u);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int b, uint32_t slot, bool first) {  // O (+)= P_b V, 4 slices of 16 keys
      const uint32_t vb = v_lo + ((slot * C::kKVBytes) >> 4);
      if (leader && tmem_range_ok(tmem + C::kColO, kW_D) &&
          tmem_range_ok(tmem + C::kColS + 64u * b, kW_BlockN / 2) &&
          guard(slot < static_cast<uint32_t>(R))) {
#pragma unroll
        for (int kk = 0; kk < kW_BlockN / 16; ++kk)
          umma_ts_lohi(tmem + C::kColO, tmem + C::kColS + 64u * b + 8u * kk,
                       vb + ((kk * 16 * 128) >> 4), kHi, kIdescPV, (kk > 0 || !first) ? 1u : 0u);
      }
      __syncwarp();
    };
    uint32_t ic = 0, qt = 0, gt = 0;  // ring items consumed, Q copies consumed, key tiles
    uint32_t pu[2] = {0u, 0u};        // p_full phases consumed per buffer
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int idx = unit_index(r);
      if (idx >= p.total_units) break;
      const WideUnit u = wide_unit_at(idx, p);
      if (!warp_wait_bar(bars.q_tmem(), parity_of(qt), wctx)) break;
      ++qt;
      tc_fence_after_sync();
      // S(0) and S(1) ahead of the softmax.
      for (int j = 0; ok && j < 2 && j < u.n; ++j) {
        if (!warp_wait_bar(bars.kv_full(ic % R), parity_of(ic / R), wctx)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_s(static_cast<int>((gt + j) & 1u), ic % R);
        commit(bars.s_full(static_cast<int>((gt + j) & 1u)));
        commit(bars.kv_empty(ic % R));
        ++ic;
      }
      for (int j = 0; ok && j < u.n; ++j) {
        const int b = static_cast<int>((gt + j) & 1u);
        if (!warp_wait_bar(bars.kv_full(ic % R), parity_of(ic / R), wctx) ||
            !warp_wait_bar(bars.p_full(b), parity_of(pu[b]), wctx)) {
          ok = false;
          break;
        }
        ++pu[b];
        tc_fence_after_sync();
        issue_pv(b, ic % R, j == 0);
        commit(bars.kv_empty(ic % R));
        commit(bars.pv_done());
        ++ic;
        if (j + 2 < u.n) {
          // S(j+2) overwrites P(j) in buffer b after the P.V that reads it.
          if (!warp_wait_bar(bars.kv_full(ic % R), parity_of(ic / R), wctx)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_s(b, ic % R);
          commit(bars.s_full(b));
          commit(bars.kv_empty(ic % R));
          ++ic;
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
