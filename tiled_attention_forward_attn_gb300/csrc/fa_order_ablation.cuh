// Loop-order ablation of the attention forward: the same tile computation in
// the two loop orders the pages compare, so that their HBM traffic and time
// can be measured side by side.
//
//   kV1 = true  — "Parsing FlashAttention (2): FlashAttention-v1 forward
//                 pass" §4 (Algorithm 1): per (batch, head), K/V tiles in the
//                 outer loop (loaded once, kept in shared memory), query
//                 tiles in the inner loop; every (i, j) step reads Q_i and the
//                 running O_i, m_i, l_i from HBM and writes O_i, m_i, l_i back,
//                 with the normalised update of eq. (37):
//                   m_new = max(m, m~),  l_new = e^(m - m_new) l + e^(m~ - m_new) l~,
//                   O_i  <- (l e^(m - m_new) O_i + e^(m~ - m_new) P~ V_j) / l_new.
//                 One CTA per (batch, head), as in that algorithm.
//   kV1 = false — the order of "Online Softmax and FlashAttention" (course
//                 unit 12, "Q/O stay, K/V move"): one CTA per (batch, head,
//                 query tile); Q_i and the unnormalised accumulator stay on
//                 chip for the whole K/V sweep; O is written once.
//
// Both use 64-row query and key tiles, four warps (16 query rows each),
// warp-level 16x8x16 bf16 tensor-core MMAs fed by ldmatrix from
// TMA-loaded, 128-byte-swizzled tiles, fp32 statistics, causal tiles past
// the diagonal skipped.  The running O of the v1 order is kept in fp32 in a
// workspace (one round trip per step), so both orders compute the same
// result to fp32 rounding.  This is a measurement instrument, not the
// production path (fa_fwd).
#pragma once

#include <climits>
#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "fa_fwd_kernel.cuh"  // g_fa_status, kStatusTimeout
#include "ptx.cuh"

namespace fa {

constexpr int kOrdTile = 64;     // query rows and keys per tile
constexpr int kOrdThreads = 128;  // four warps x 16 query rows

struct OrderParams {
  uint16_t* o;     // [BH][N][D] bf16, written
  float* lse;      // [BH][N], written
  float* ws_o;     // v1: [BH][Npad][D] fp32 running output
  float* ws_m;     // v1: [BH][Npad] running max (scaled, log2 units)
  float* ws_l;     // v1: [BH][Npad] running exponent sum
  int N, Npad, T;  // T = Npad / 64 tiles
  int num_bh, causal;
  float scale_log2;
  uint64_t wait_limit_ns;
};

template <int D, bool kV1>
struct OrdCfg {
  static constexpr uint32_t kTileBytes = kOrdTile * D * 2;
  // v2: Q, then 2 stages of (K, V).  v1: K, V, then 2 Q stages.
  static constexpr uint32_t kOffQ = kV1 ? 2 * kTileBytes : 0;
  static constexpr uint32_t kOffKV = kV1 ? 0 : kTileBytes;
  static constexpr uint32_t kOffBar = kV1 ? 4 * kTileBytes : 5 * kTileBytes;
  static constexpr uint32_t kSmemBytes = kOffBar + 64;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
};

__device__ __forceinline__ uint32_t ord_sw(int row, int chunk) {
  // 16-byte chunk of a row in a tile of D/64 boxes of 64 rows x 128 bytes,
  // 128-byte swizzle.
  return static_cast<uint32_t>((chunk >> 3) * (kOrdTile * 128) + row * 128 +
                               (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ bool ord_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 30); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 15u && global_timer_ns() - t0 > limit_ns) break;
  }
  atomicOr(&g_fa_status, kStatusTimeout);
  return false;
}

// Loads a 64-row tile (rows r0.., slice bh) of a [BH][N][D] tensor.
// rows, nbh: the tensor's row count and slice count (for the guarded build).
template <int D>
__device__ __forceinline__ void ord_load(uint32_t dst, const CUtensorMap* map, uint32_t bar, int r0,
                                         int bh, int rows, int nbh) {
#pragma unroll
  for (int b = 0; b < D / 64; ++b)
    if (tma_coord_ok(64 * b, D, r0, rows, bh, nbh))
      tma_load_3d(dst + b * kOrdTile * 128, map, bar, 64 * b, r0, bh);
}

// S = Q K^T for this warp's 16 query rows against the 64 keys of a tile,
// scaled to log2 units and masked; sc[nt][e]: key 8nt + 2t4 + (e & 1), row
// g + 8 (e >> 1).
template <int D>
__device__ __forceinline__ void ord_scores(float (&sc)[8][4], const uint32_t (&qa)[D / 16][4],
                                          uint32_t sK, int lane, int q_row0, int k0,
                                          const OrderParams& p) {
  const int mi = lane >> 3, r8 = lane & 7, g = lane >> 2, t4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
#pragma unroll
  for (int np = 0; np < 4; ++np) {
    const int k_row = 16 * np + ((mi >> 1) << 3) + r8;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t b[4];
      ldsm_x4(b, sK + ord_sw(k_row, 2 * ks + (mi & 1)));
      mma_bf16_16816(sc[2 * np], qa[ks], b[0], b[1]);
      mma_bf16_16816(sc[2 * np + 1], qa[ks], b[2], b[3]);
    }
  }
  const int r0 = q_row0 + g, r1 = r0 + 8;
  const bool edge = k0 + kOrdTile > p.N || (p.causal && k0 + kOrdTile - 1 > q_row0);
#pragma unroll
  for (int nt = 0; nt < 8; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float x = sc[nt][e] * p.scale_log2;
      if (edge) {
        const int key = k0 + 8 * nt + 2 * t4 + (e & 1);
        const int row = (e >> 1) ? r1 : r0;
        if (key >= p.N || (p.causal && key > row)) x = -CUDART_INF_F;
      }
      sc[nt][e] = x;
    }
}

// acc (16 rows x D) += P (16 x 64, bf16 A fragments) V (64 x D).
template <int D>
__device__ __forceinline__ void ord_pv(float (&acc)[D / 8][4], const float (&pr)[8][4], uint32_t sV,
                                      int lane) {
  const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t pa[4] = {pack_bf16x2(pr[2 * kk][0], pr[2 * kk][1]),
                            pack_bf16x2(pr[2 * kk][2], pr[2 * kk][3]),
                            pack_bf16x2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]),
                            pack_bf16x2(pr[2 * kk + 1][2], pr[2 * kk + 1][3])};
    const int v_row = 16 * kk + ((mi & 1) << 3) + r8;
#pragma unroll
    for (int n = 0; n < D / 8; n += 2) {
      uint32_t b[4];
      ldsm_x4_trans(b, sV + ord_sw(v_row, n + (mi >> 1)));
      mma_bf16_16816(acc[n], pa, b[0], b[1]);
      mma_bf16_16816(acc[n + 1], pa, b[2], b[3]);
    }
  }
}

// Row maximum of a tile (rows g and g + 8; the quad holds one row).
__device__ __forceinline__ void ord_rowmax(const float (&sc)[8][4], float& m0, float& m1) {
  m0 = -CUDART_INF_F;
  m1 = -CUDART_INF_F;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    m0 = fmaxf(m0, fmaxf(sc[nt][0], sc[nt][1]));
    m1 = fmaxf(m1, fmaxf(sc[nt][2], sc[nt][3]));
  }
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, off));
    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, off));
  }
}

template <int D, bool kV1>
__global__ void __launch_bounds__(kOrdThreads)
    fa_order_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const OrderParams p) {
  using C = OrdCfg<D, kV1>;
  constexpr int kN = D / 8;  // 8-column MMA tiles of the output
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;  // v2: q, kv[0], kv[1];  v1: kv, q[0], q[1]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t4 = lane & 3, mi = lane >> 3, r8 = lane & 7;
  if (threadIdx.x == 0) {
    for (int b = 0; b < 3; ++b) mbar_init(bar0 + 8 * b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // Phases started (thread 0, which issues every copy) and completed (every
  // thread waits on every phase, in order) per barrier; a timed-out wait is
  // not counted, so the drain at the end waits for it again.
  uint32_t started[3] = {0u, 0u, 0u}, waited[3] = {0u, 0u, 0u};
  auto expect = [&](int b, uint32_t bytes) {
    mbar_arrive_expect_tx(bar0 + 8 * b, bytes);
    ++started[b];
  };
  auto wait = [&](int b) -> bool {
    const bool r = ord_wait(bar0 + 8 * b, waited[b] & 1u, p.wait_limit_ns);
    if (r) ++waited[b];
    return r;
  };
  auto drain = [&]() {
    if (threadIdx.x == 0)
      for (int b = 0; b < 3; ++b)
        while (waited[b] < started[b] && wait(b)) {
        }
  };

  if (!kV1) {
    // ---------------------------------------------------------------- v2 order
    // Barriers: 0 = Q, 1 + s = K/V stage s.
    const int band = static_cast<int>(blockIdx.x) / p.num_bh;
    const int bh = static_cast<int>(blockIdx.x) - band * p.num_bh;
    const int it = p.T - 1 - band;  // query tile, heaviest first when causal
    const int q0 = it * kOrdTile;
    const int nj = p.causal ? it + 1 : p.T;
    const uint32_t sQ = sbase + C::kOffQ;
    auto kv_stage = [&](int s) { return sbase + C::kOffKV + s * 2 * C::kTileBytes; };
    if (threadIdx.x == 0) {
      expect(0, C::kTileBytes);
      ord_load<D>(sQ, &tm_q, bar0, q0, bh, p.N, p.num_bh);
      for (int j = 0; j < 2 && j < nj; ++j) {
        expect(1 + j, 2 * C::kTileBytes);
        ord_load<D>(kv_stage(j), &tm_k, bar0 + 8 * (1 + j), j * kOrdTile, bh, p.N, p.num_bh);
        ord_load<D>(kv_stage(j) + C::kTileBytes, &tm_v, bar0 + 8 * (1 + j), j * kOrdTile, bh, p.N, p.num_bh);
      }
    }
    bool ok = __syncthreads_and(wait(0));
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      ldsm_x4(qa[ks], sQ + ord_sw(16 * warp + ((mi & 1) << 3) + r8, 2 * ks + (mi >> 1)));
    float acc[kN][4];
#pragma unroll
    for (int n = 0; n < kN; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.0f, l1 = 0.0f;
    const int q_row0 = q0 + 16 * warp;
    for (int j = 0; ok && j < nj; ++j) {
      const int s = j & 1;
      ok = __syncthreads_and(wait(1 + s));
      if (!ok) break;
      const uint32_t sK = kv_stage(s), sV = sK + C::kTileBytes;
      float sc[8][4];
      ord_scores<D>(sc, qa, sK, lane, q_row0, j * kOrdTile, p);
      float mx0, mx1;
      ord_rowmax(sc, mx0, mx1);
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float mu0 = mn0 == -CUDART_INF_F ? 0.0f : mn0, mu1 = mn1 == -CUDART_INF_F ? 0.0f : mn1;
      const float a0 = ex2_approx(m0 - mu0), a1 = ex2_approx(m1 - mu1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = ex2_approx(sc[nt][0] - mu0);
        sc[nt][1] = ex2_approx(sc[nt][1] - mu0);
        sc[nt][2] = ex2_approx(sc[nt][2] - mu1);
        sc[nt][3] = ex2_approx(sc[nt][3] - mu1);
        ps0 += sc[nt][0] + sc[nt][1];
        ps1 += sc[nt][2] + sc[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int n = 0; n < kN; ++n) {
        acc[n][0] *= a0;
        acc[n][1] *= a0;
        acc[n][2] *= a1;
        acc[n][3] *= a1;
      }
      ord_pv<D>(acc, sc, sV, lane);
      __syncthreads();  // every warp is done with stage s
      if (threadIdx.x == 0 && j + 2 < nj) {
        expect(1 + s, 2 * C::kTileBytes);
        ord_load<D>(sK, &tm_k, bar0 + 8 * (1 + s), (j + 2) * kOrdTile, bh, p.N, p.num_bh);
        ord_load<D>(sV, &tm_v, bar0 + 8 * (1 + s), (j + 2) * kOrdTile, bh, p.N, p.num_bh);
      }
    }
    if (!ok) {
      drain();
      return;
    }
    // Row sums over the quad, then O = acc / l and LSE.
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int r0 = q_row0 + g, r1 = r0 + 8;
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
#pragma unroll
    for (int n = 0; n < kN; ++n) {
      const int col = 8 * n + 2 * t4;
      if (r0 < p.N && guard(bh < p.num_bh && col + 2 <= D))
        *reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bh) * p.N + r0) * D + col) =
            pack_bf16x2(acc[n][0] * i0, acc[n][1] * i0);
      if (r1 < p.N && guard(bh < p.num_bh && col + 2 <= D))
        *reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bh) * p.N + r1) * D + col) =
            pack_bf16x2(acc[n][2] * i1, acc[n][3] * i1);
    }
    if (t4 == 0) {
      if (r0 < p.N) p.lse[static_cast<size_t>(bh) * p.N + r0] = (m0 + __log2f(l0)) * 0.6931471805599453f;
      if (r1 < p.N) p.lse[static_cast<size_t>(bh) * p.N + r1] = (m1 + __log2f(l1)) * 0.6931471805599453f;
    }
    return;
  }

  // ------------------------------------------------------------------ v1 order
  // Barriers: 0 = K/V, 1 + s = Q stage s.  Q loads are numbered in issue
  // order; load n goes to stage n & 1.
  const int bh = blockIdx.x;
  const uint32_t sK = sbase + C::kOffKV, sV = sK + C::kTileBytes;
  auto q_stage = [&](uint32_t s) { return sbase + C::kOffQ + s * C::kTileBytes; };
  uint32_t q_loads = 0;  // Q tiles loaded (or being loaded) so far
  bool ok = true;
  for (int j = 0; ok && j < p.T; ++j) {
    const int i_first = p.causal ? j : 0;  // query tiles that see key tile j
    const int ni = p.T - i_first;
    if (threadIdx.x == 0) {
      expect(0, 2 * C::kTileBytes);
      ord_load<D>(sK, &tm_k, bar0, j * kOrdTile, bh, p.N, p.num_bh);
      ord_load<D>(sV, &tm_v, bar0, j * kOrdTile, bh, p.N, p.num_bh);
      const uint32_t s = q_loads & 1u;
      expect(1 + s, C::kTileBytes);
      ord_load<D>(q_stage(s), &tm_q, bar0 + 8 * (1 + s), i_first * kOrdTile, bh, p.N, p.num_bh);
    }
    ok = __syncthreads_and(wait(0));
    for (int ii = 0; ok && ii < ni; ++ii) {
      const int i = i_first + ii;
      const uint32_t s = (q_loads + ii) & 1u;
      if (threadIdx.x == 0 && ii + 1 < ni) {  // prefetch the next Q tile
        expect(1 + (s ^ 1u), C::kTileBytes);
        ord_load<D>(q_stage(s ^ 1u), &tm_q, bar0 + 8 * (1 + (s ^ 1u)), (i + 1) * kOrdTile, bh, p.N, p.num_bh);
      }
      ok = __syncthreads_and(wait(1 + s));
      if (!ok) break;
      uint32_t qa[D / 16][4];
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks)
        ldsm_x4(qa[ks], q_stage(s) + ord_sw(16 * warp + ((mi & 1) << 3) + r8, 2 * ks + (mi >> 1)));
      const int q_row0 = i * kOrdTile + 16 * warp;
      float sc[8][4];
      ord_scores<D>(sc, qa, sK, lane, q_row0, j * kOrdTile, p);
      // Tile statistics m~, P~ = 2^(s - m~), l~ (eq. (37)'s tilde terms).
      float mt0, mt1;
      ord_rowmax(sc, mt0, mt1);
      const float mu0 = mt0 == -CUDART_INF_F ? 0.0f : mt0, mu1 = mt1 == -CUDART_INF_F ? 0.0f : mt1;
      float lt0 = 0.0f, lt1 = 0.0f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        sc[nt][0] = ex2_approx(sc[nt][0] - mu0);
        sc[nt][1] = ex2_approx(sc[nt][1] - mu0);
        sc[nt][2] = ex2_approx(sc[nt][2] - mu1);
        sc[nt][3] = ex2_approx(sc[nt][3] - mu1);
        lt0 += sc[nt][0] + sc[nt][1];
        lt1 += sc[nt][2] + sc[nt][3];
      }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, off);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, off);
      }
      float pv[kN][4];
#pragma unroll
      for (int n = 0; n < kN; ++n) pv[n][0] = pv[n][1] = pv[n][2] = pv[n][3] = 0.0f;
      ord_pv<D>(pv, sc, sV, lane);
      // Running state of rows r0, r1 from HBM (none before the first key tile).
      const int r0 = q_row0 + g, r1 = r0 + 8;
      const size_t w0 = static_cast<size_t>(bh) * p.Npad + r0, w1 = w0 + 8;
      const bool first = j == 0;
      const float m_0 = first ? -CUDART_INF_F : p.ws_m[w0];
      const float m_1 = first ? -CUDART_INF_F : p.ws_m[w1];
      const float l_0 = first ? 0.0f : p.ws_l[w0];
      const float l_1 = first ? 0.0f : p.ws_l[w1];
      const float mn0 = fmaxf(m_0, mt0), mn1 = fmaxf(m_1, mt1);
      const float e_old0 = m_0 == -CUDART_INF_F ? 0.0f : ex2_approx(m_0 - mn0);
      const float e_old1 = m_1 == -CUDART_INF_F ? 0.0f : ex2_approx(m_1 - mn1);
      const float e_new0 = mt0 == -CUDART_INF_F ? 0.0f : ex2_approx(mt0 - mn0);
      const float e_new1 = mt1 == -CUDART_INF_F ? 0.0f : ex2_approx(mt1 - mn1);
      const float ln0 = e_old0 * l_0 + e_new0 * lt0, ln1 = e_old1 * l_1 + e_new1 * lt1;
      const float ia0 = ln0 > 0.0f ? 1.0f / ln0 : 0.0f, ia1 = ln1 > 0.0f ? 1.0f / ln1 : 0.0f;
      const bool last = p.causal ? j == i : j == p.T - 1;
      const float c00 = l_0 * e_old0 * ia0, c01 = e_new0 * ia0;
      const float c10 = l_1 * e_old1 * ia1, c11 = e_new1 * ia1;
#pragma unroll
      for (int n = 0; n < kN; ++n) {
        const int col = 8 * n + 2 * t4;
        float2 o0 = make_float2(0.0f, 0.0f), o1 = make_float2(0.0f, 0.0f);
        if (!first) {
          o0 = *reinterpret_cast<const float2*>(p.ws_o + w0 * D + col);
          o1 = *reinterpret_cast<const float2*>(p.ws_o + w1 * D + col);
        }
        o0.x = o0.x * c00 + pv[n][0] * c01;
        o0.y = o0.y * c00 + pv[n][1] * c01;
        o1.x = o1.x * c10 + pv[n][2] * c11;
        o1.y = o1.y * c10 + pv[n][3] * c11;
        if (last) {
          if (r0 < p.N && guard(bh < p.num_bh && col + 2 <= D))
            *reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bh) * p.N + r0) * D + col) =
                pack_bf16x2(o0.x, o0.y);
          if (r1 < p.N && guard(bh < p.num_bh && col + 2 <= D))
            *reinterpret_cast<uint32_t*>(p.o + (static_cast<size_t>(bh) * p.N + r1) * D + col) =
                pack_bf16x2(o1.x, o1.y);
        } else if (guard(bh < p.num_bh && r1 < p.Npad && col + 2 <= D)) {
          *reinterpret_cast<float2*>(p.ws_o + w0 * D + col) = o0;
          *reinterpret_cast<float2*>(p.ws_o + w1 * D + col) = o1;
        }
      }
      if (t4 == 0) {
        if (last) {
          if (r0 < p.N) p.lse[static_cast<size_t>(bh) * p.N + r0] = (mn0 + __log2f(ln0)) * 0.6931471805599453f;
          if (r1 < p.N) p.lse[static_cast<size_t>(bh) * p.N + r1] = (mn1 + __log2f(ln1)) * 0.6931471805599453f;
        } else if (guard(bh < p.num_bh && r1 < p.Npad)) {
          p.ws_m[w0] = mn0;
          p.ws_m[w1] = mn1;
          p.ws_l[w0] = ln0;
          p.ws_l[w1] = ln1;
        }
      }
      __syncthreads();  // Q stage s is free for the prefetch after next
    }
    q_loads += ni;
    __syncthreads();  // K_j, V_j are free for the next key tile
  }
  if (!ok) drain();
}

}  // namespace fa
