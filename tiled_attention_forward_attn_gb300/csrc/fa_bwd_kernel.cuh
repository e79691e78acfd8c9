// Attention backward by recomputation for sm_103a.
//
// Given Q, K, V, the forward's O and LSE and the output gradient dO, the
// gradients of sum(dO * O) are, with s = scale * Q K^T (+ causal mask),
// P = exp(s - LSE) (the forward's probabilities, recomputed from the saved
// row statistic as "Parsing FlashAttention (2)" §1 and "Online Softmax and
// FlashAttention" keep it for), D_i = rowsum(dO_i * O_i):
//     dV = P^T dO,   dP = dO V^T,   dS = P * (dP - D),
//     dQ = scale * dS K,   dK = scale * dS^T Q.
// (D_i equals sum_j P_ij dP_ij, the softmax Jacobian's correction term,
// because O = P V.)
//
// Q, K, V, O, dO and the gradients are (batch, head, row, column) tensors at
// caller strides (columns unit-stride), read through 4-D tensor maps {d, N,
// H, B}; LSE and the workspace are contiguous.
//
// Three launches, no atomics:
//   fa_bwd_prep_kernel    D and LSE * log2(e) per query row, into a
//                         workspace padded to whole 128-row tiles;
//   fa_bwd_kernel<D,true> one CTA per (batch*head, 128-key tile j): K_j and
//                         V_j stay in shared memory, Q_i, dO_i and the
//                         tile's D, LSE stream through a TMA ring; per query
//                         tile i the tensor core computes S^T = K_j Q_i^T
//                         and dP^T = V_j dO_i^T into TMEM, four warps (one
//                         key row = one TMEM lane each) turn them into P^T
//                         and dS^T (16-bit pairs written back over them), and
//                         dV_j += P^T dO_i, dK_j += dS^T Q_i accumulate in
//                         TMEM with P^T / dS^T read straight from TMEM;
//   fa_bwd_kernel<D,false> one CTA per (batch*head, 128-query tile i): Q_i
//                         and dO_i stay, K_j and V_j stream; S, dP into
//                         TMEM, dS written back over S, dQ_i += dS K_j.
// Causal: the key tile j only meets query tiles i >= j, the query tile i
// only key tiles j <= i; the diagonal tile is masked element by element.
//
// Each streamed 128-row tile is processed in two 64-row sub-steps whose S
// and dP live in alternating TMEM buffers, so the tensor core computes the
// next sub-step's S and dP (and the previous one's accumulation) while the
// elementwise warps work on the current one.  Four elementwise warpgroups
// all work on every sub-step, warpgroup g on its 16 columns (the latency of
// a sub-step's elementwise work is on the critical path), and each writes
// its P/dS pairs into the first half of its own column range, which is
// exactly the TMEM A operand of one 16-row accumulation MMA.  TMEM (512 columns): S
// buffers [0,64) and [64,128), dP buffers [128,192) and [192,256), then the
// accumulators (dK and dV, or dQ), D columns each.  Warps: 0-15 elementwise
// and epilogue, 16 the TMA producer, 17 the TMEM allocator and MMA issuer,
// 18-19 idle.  Every wait is bounded like the forward's (status word, drain,
// TMEM freed).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <math_constants.h>

#include "fa_fwd_kernel.cuh"  // wait helpers, status word, kSwBlockBytes
#include "ptx.cuh"

namespace fa {

// Five warpgroups: four elementwise, one with the producer, the MMA issuer
// and two idle warps.  Launched with 96 registers a thread (five warps per
// sub-partition); setmaxnreg then moves registers from the control
// warpgroup to the elementwise ones.
constexpr int kBwdEwGroups = 4;
constexpr int kBwdThreads = (kBwdEwGroups + 1) * 128;
constexpr int kBwdLoadWarp = 4 * kBwdEwGroups;
constexpr int kBwdMmaWarp = kBwdLoadWarp + 1;
constexpr uint32_t kBwdLaunchRegs = 96;
constexpr uint32_t kBwdEwRegs = 104;
constexpr uint32_t kBwdControlRegs = 56;
static_assert(kBwdEwGroups * 128 * kBwdEwRegs + 128 * kBwdControlRegs <=
                  kBwdThreads * kBwdLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kBwdTile = 128;  // rows of every tile (keys or queries)
constexpr int kBwdSub = 64;    // streamed rows per sub-step
constexpr int kBwdEwCols = kBwdSub / 4;  // columns of a sub-step per elementwise warpgroup

struct BwdParams {
  uint16_t* out0;     // key-tile pass: dK; query-tile pass: dQ   (b, h, row, col) bf16 or fp16
  uint16_t* out1;     // key-tile pass: dV; unused otherwise
  int64_t out0_sb, out0_sh, out0_sn;  // element strides of out0 (batch, head, row; columns unit)
  int64_t out1_sb, out1_sh, out1_sn;  // and of out1
  const float* lse2;  // [BH][Npad] -LSE * log2(e) per query (0 past N)
  const float* dvec;  // [BH][Npad] -rowsum(dO * O) per query (0 past N)
  int N;              // sequence length
  int d;              // head dimension (<= D, a multiple of 16; columns past it are zeros)
  int Npad;           // N rounded up to whole tiles
  int T;              // tiles per (batch, head) = Npad / 128
  int num_bh;         // B * H
  int H;              // heads (bh = b * H + h)
  int causal;
  float scale_log2;   // scale * log2(e)
  float scale;        // the softmax scale
  uint64_t wait_limit_ns;
  uint32_t inject = 0;  // test hooks (0 in normal use)
};

template <int D, bool kKV>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dimension");
  // The streamed tiles arrive in 64-row halves (one sub-step each), so a
  // stage is released as soon as its sub-step's MMAs complete.
  static constexpr int kStages = (D == 64) ? 8 : 4;
  static constexpr uint32_t kTileBytes = kBwdTile * D * 2;  // a stationary 128-row tile
  static constexpr uint32_t kHalfBytes = kBwdSub * D * 2;   // a streamed 64-row half tile
  static constexpr uint32_t kHalfBlock = kBwdSub * 128;     // 64 columns x 64 rows
  static constexpr uint32_t kStageBytes = 2 * kHalfBytes;   // Y0 half, Y1 half
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned for the swizzle");
  static constexpr uint32_t kVecBytes = kKV ? 2 * kBwdSub * 4 : 0;  // -LSE2[64], -D[64] per stage
  static constexpr uint32_t kOffX = 0;                // stationary tiles X0, X1
  static constexpr uint32_t kOffY = 2 * kTileBytes;   // ring of (Y0, Y1) halves
  static constexpr uint32_t kOffVec = kOffY + kStages * kStageBytes;
  static constexpr uint32_t kOffBar = kOffVec + kStages * kVecBytes;
  // x_full, st_full[2], p_full[2], acc_done, y_full[S], y_empty[S], x_tmem
  // (query-tile pass: X copied into TMEM), x_empty, acc_free, mma_done
  static constexpr int kNumBars = 10 + 2 * kStages;
  static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kSmemAlloc = kSmemBytes + 1024;
  static_assert(kSmemAlloc <= 232448, "dynamic shared memory per block");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;      // S buffer b at 64b; then P^T or dS as 16-bit pairs
  static constexpr uint32_t kColDP = 128;   // dP buffer b at 128 + 64b; then dS^T (key-tile pass)
  static constexpr uint32_t kColAcc0 = 256;      // dK (key-tile pass) or dQ
  static constexpr uint32_t kColAcc1 = 256 + D;  // dV (key-tile pass)
  // Query-tile pass: Q_i and dO_i as 16-bit pairs in the spare columns, so
  // the S and dP MMAs read their A operand from TMEM and only K/V from SMEM.
  static constexpr uint32_t kColXT = 384;
  static_assert(kKV || kColXT + D <= kTmemCols, "Q and dO pairs fit in TMEM");
};

struct BwdBars {
  uint32_t base;
  int stages;
  __device__ uint32_t x_full() const { return base; }
  __device__ uint32_t st_full(int b) const { return base + 8u + 8u * b; }
  __device__ uint32_t p_full(int b) const { return base + 24u + 8u * b; }
  __device__ uint32_t acc_done() const { return base + 40u; }
  __device__ uint32_t y_full(int s) const { return base + 48u + 8u * s; }
  __device__ uint32_t y_empty(int s) const { return base + 48u + 8u * (stages + s); }
  __device__ uint32_t x_tmem() const { return base + 48u + 16u * stages; }
  // The stationary tile's shared memory may be refilled (key-tile pass: its
  // last S/dP MMAs are complete; query-tile pass: it is copied into TMEM).
  __device__ uint32_t x_empty() const { return base + 56u + 16u * stages; }
  // The accumulators of a tile have been read by its epilogue.
  __device__ uint32_t acc_free() const { return base + 64u + 16u * stages; }
  __device__ uint32_t mma_done() const { return base + 72u + 16u * stages; }
};

// -D_i = -rowsum(dO_i * O_i) and -LSE_i * log2(e) for every row of the
// padded [BH][Npad] layout (0 past N), negated for the elementwise pass's
// fused multiply-adds.  D/8 threads per row, 16 bytes each; O and dO at
// their element strides.  Row indices stay in 32 bits (the host rejects
// BH * Npad above INT_MAX), so no thread pays for a 64-bit division.
template <int D, bool kF16>
__global__ void __launch_bounds__(256)
    fa_bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dout,
                       const float* __restrict__ lse, float* __restrict__ lse2,
                       float* __restrict__ dvec, int N, int Npad, int d, int H,
                       int64_t o_sb, int64_t o_sh, int64_t o_sn, int64_t do_sb, int64_t do_sh,
                       int64_t do_sn) {
  constexpr int kTpr = D / 8;             // threads per row
  constexpr int kRowsPerCta = 256 / kTpr;
  const int row = static_cast<int>(blockIdx.x) * kRowsPerCta +
                  static_cast<int>(threadIdx.x) / kTpr;  // padded row index bh * Npad + n
  const int part = static_cast<int>(threadIdx.x) % kTpr;
  const int bh = row / Npad;
  const int n = row - bh * Npad;
  float acc = 0.0f;
  if (n < N && part * 8 < d) {
    const int bb = bh / H, hh = bh - bb * H;
    const int64_t off_o = bb * o_sb + hh * o_sh + n * o_sn + part * 8;
    const int64_t off_do = bb * do_sb + hh * do_sh + n * do_sn + part * 8;
    // Read once: streamed past L1.
    const uint4 a = __ldcs(reinterpret_cast<const uint4*>(o + off_o));
    const uint4 b = __ldcs(reinterpret_cast<const uint4*>(dout + off_do));
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc = fmaf(elem_to_f32<kF16>(aw[e], false), elem_to_f32<kF16>(bw[e], false), acc);
      acc = fmaf(elem_to_f32<kF16>(aw[e], true), elem_to_f32<kF16>(bw[e], true), acc);
    }
  }
#pragma unroll
  for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0 && guard(bh >= 0 && n >= 0 && n < Npad)) {
    dvec[row] = n < N ? -acc : 0.0f;
    lse2[row] = n < N ? -lse[static_cast<size_t>(bh) * N + n] * 1.4426950408889634f : 0.0f;
  }
}

// kKV = true: X = (K, V) of key tile xt, Y = (Q, dO) of query tiles.
// kKV = false: X = (Q, dO) of query tile xt, Y = (K, V) of key tiles.
template <int D, bool kKV, bool kF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_x0, const __grid_constant__ CUtensorMap tm_x1,
                  const __grid_constant__ CUtensorMap tm_y0, const __grid_constant__ CUtensorMap tm_y1,
                  const BwdParams p) {
  using C = BwdCfg<D, kKV>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sX = sbase + C::kOffX;
  const uint32_t sY = sbase + C::kOffY;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kOffMisc + 4);
  const BwdBars bars{sbase + C::kOffBar, S};
  const WaitCtx wctx{abort_flag, p.wait_limit_ns};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // The grid is persistent: CTA c takes the tiles unit_index(0), (1), ...
  // of the order below, dealt in a serpentine like the forward's units.
  // Tile t, heaviest first under the causal mask: key tile 0 meets every
  // query tile; query tile T-1 meets every key tile.
  struct Tile {
    int bh, xt, y_first, steps;
  };
  const int total = p.num_bh * p.T;
  auto tile_at = [&](int t) -> Tile {
    const int band = t / p.num_bh;
    Tile u;
    u.bh = t - band * p.num_bh;
    u.xt = kKV ? band : p.T - 1 - band;
    u.y_first = (kKV && p.causal) ? u.xt : 0;
    const int y_last = (!kKV && p.causal) ? u.xt : p.T - 1;
    u.steps = y_last - u.y_first + 1;
    return u;
  };

  if (threadIdx.x == 0) {
    mbar_init(bars.x_full(), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bars.st_full(b), 1);
      mbar_init(bars.p_full(b), 4 * kBwdEwGroups);  // one arrival per elementwise warp
    }
    mbar_init(bars.acc_done(), 1);
    mbar_init(bars.x_tmem(), 4 * kBwdEwGroups);  // one arrival per elementwise warp
    // Key-tile pass: a commit after a tile's last S/dP MMAs; query-tile
    // pass: one arrival per elementwise warp after the copy into TMEM.
    mbar_init(bars.x_empty(), kKV ? 1 : 4 * kBwdEwGroups);
    mbar_init(bars.acc_free(), 4 * kBwdEwGroups);
    mbar_init(bars.mma_done(), 1);
    for (int s = 0; s < S; ++s) {
      mbar_init(bars.y_full(s), 1);
      mbar_init(bars.y_empty(s), 1);
    }
    *abort_flag = 0u;
    fence_barrier_init();
  }
  if (warp == kBwdMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  if (warp == kBwdLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_x0);
    tma_prefetch_desc(&tm_x1);
    tma_prefetch_desc(&tm_y0);
    tma_prefetch_desc(&tm_y1);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // One setmaxnreg per warpgroup, executed by all four of its warps.
  if (warp < 4 * kBwdEwGroups) {
    setmaxnreg_inc<kBwdEwRegs>();
  } else {
    setmaxnreg_dec<kBwdControlRegs>();
  }

  if (warp < 4 * kBwdEwGroups) {
    // ------------------------------------------------------------ elementwise
    const int g = warp >> 2;            // warpgroup: its 16 columns of every sub-step
    const int row = threadIdx.x & 127;  // = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float cs = p.scale_log2;
    uint32_t gsub = 0;  // sub-steps of earlier tiles (always even)
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int t = unit_index(r);
      if (t >= total) break;
      const Tile u = tile_at(t);
      const int bh = u.bh, xt = u.xt, y_first = u.y_first, steps = u.steps;
      const int x_idx = xt * kBwdTile + row;  // key (kKV) or query index of this row
      if (!kKV) {
        // Warpgroups 0 and 1 copy this row of X_g (g = 0: Q_i, 1: dO_i) from the swizzled SMEM
        // tile into TMEM as 16-bit pairs: 16-byte chunk c of the row sits in
        // 64-column block c / 8 at row * 128 + ((c % 8) ^ (row % 8)) * 16.  The
        // previous tile's S/dP MMAs, the only readers of these columns, are
        // complete: its last st_full was consumed.
        if (g < 2) {
          if (!warp_wait_bar(bars.x_full(), parity_of(r), wctx)) {
            ok = false;
            break;
          }
          const uint8_t* xt_s = smem + C::kOffX + g * C::kTileBytes;
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            uint32_t wv[32];
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              const uint4 v4 = *reinterpret_cast<const uint4*>(
                  xt_s + h * kSwBlockBytes + row * 128 + (((c8 ^ (row & 7))) << 4));
              wv[4 * c8] = v4.x;
              wv[4 * c8 + 1] = v4.y;
              wv[4 * c8 + 2] = v4.z;
              wv[4 * c8 + 3] = v4.w;
            }
            tmem_st32(tmem + lane_off + C::kColXT + g * (D / 2) + 32 * h, wv);
          }
          tmem_st_wait();
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bars.x_tmem());
          mbar_arrive(bars.x_empty());
        }
      }
      float nlse_r = 0.0f, nd_r = 0.0f;
      if (!kKV) {
        nlse_r = p.lse2[static_cast<size_t>(bh) * p.Npad + x_idx];
        nd_r = p.dvec[static_cast<size_t>(bh) * p.Npad + x_idx];
      }
      for (int m = 0; m < 2 * steps; ++m) {
        const int b = m & 1;  // TMEM buffer
        const int n = m >> 1;
        const uint32_t gm = gsub + static_cast<uint32_t>(m);  // sub-step over all tiles
        if (!warp_wait_bar(bars.st_full(b), parity_of(gm >> 1), wctx)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int yt = y_first + n;
        const int y0 = yt * kBwdTile + kBwdSub * b + kBwdEwCols * g;  // first streamed row here
        const bool need_mask = (p.causal && yt == xt) || (y0 + kBwdEwCols > p.N);
        const float4* vec = reinterpret_cast<const float4*>(smem + C::kOffVec + (gm % S) * C::kVecBytes) +
                            (kBwdEwCols / 4) * g;
        const uint32_t col_s = C::kColS + kBwdSub * b + kBwdEwCols * g;
        const uint32_t col_dp = C::kColDP + kBwdSub * b + kBwdEwCols * g;
        uint32_t sr[kBwdEwCols], dr[kBwdEwCols];
        tmem_ld16(tmem + lane_off + col_s, sr);
        tmem_ld16(tmem + lane_off + col_dp, dr);
        tmem_ld_wait();
        tmem_ld_fence16(sr);
        tmem_ld_fence16(dr);
        uint32_t pp[kBwdEwCols / 2], pd[kBwdEwCols / 2];
#pragma unroll
        for (int e = 0; e < kBwdEwCols; e += 4) {
          // -LSE2 and -D of the four columns (kKV: per column, from shared
          // memory; otherwise this row's).
          float nl[4], nd[4];
          if (kKV) {
            const float4 a = vec[e / 4];
            const float4 c4 = vec[(kBwdSub + e) / 4];
            nl[0] = a.x; nl[1] = a.y; nl[2] = a.z; nl[3] = a.w;
            nd[0] = c4.x; nd[1] = c4.y; nd[2] = c4.z; nd[3] = c4.w;
          } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              nl[h] = nlse_r;
              nd[h] = nd_r;
            }
          }
#pragma unroll
          for (int h = 0; h < 4; h += 2) {
            float x0, x1, p0, p1, t0, t1, d0, d1;
            ffma2(x0, x1, __uint_as_float(sr[e + h]), __uint_as_float(sr[e + h + 1]), cs, cs, nl[h],
                  nl[h + 1]);
            p0 = ex2_approx(x0);
            p1 = ex2_approx(x1);
            if (need_mask) {
              // key <= query when causal; padding rows past N see nothing.
              const int ya = y0 + e + h;
              const bool va = ya < p.N && (!p.causal || (kKV ? x_idx <= ya : ya <= x_idx));
              const bool vb = ya + 1 < p.N &&
                              (!p.causal || (kKV ? x_idx <= ya + 1 : ya + 1 <= x_idx));
              if (!va) p0 = 0.0f;
              if (!vb) p1 = 0.0f;
            }
            fadd2(t0, t1, __uint_as_float(dr[e + h]), __uint_as_float(dr[e + h + 1]), nd[h],
                  nd[h + 1]);
            fmul2(d0, d1, p0, p1, t0, t1);
            pp[(e + h) / 2] = pack_x2<kF16>(p0, p1);
            pd[(e + h) / 2] = pack_x2<kF16>(d0, d1);
          }
        }
        // The pairs go into the first 8 of this warpgroup's 16 columns, which
        // it has already read: the A operand of accumulation slice g.
        if (kKV) {
          tmem_st8(tmem + lane_off + col_s, pp);
          tmem_st8(tmem + lane_off + col_dp, pd);
        } else {
          tmem_st8(tmem + lane_off + col_s, pd);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars.p_full(b));
      }
      if (!ok) break;
      gsub += static_cast<uint32_t>(2 * steps);
      // -------------------------------------------------------------- epilogue
      // kKV: warpgroups 0 and 1 store the two column halves of dK (scaled), 2
      // and 3 those of dV; otherwise each warpgroup stores a quarter of dQ's
      // columns (scaled).  The accumulators are read with one wait and
      // released (acc_free) before the stores, so the next tile's first
      // accumulation does not wait for them.
      if (!warp_wait_bar(bars.acc_done(), parity_of(r), wctx)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      constexpr int kCols = kKV ? D / 2 : D / 4;
      const int part = kKV ? (g & 1) : g;
      const bool is_dv = kKV && g >= 2;
      const uint32_t col = (is_dv ? C::kColAcc1 : C::kColAcc0) + kCols * part;
      const float mul = is_dv ? 1.0f : p.scale;
      uint16_t* out = is_dv ? p.out1 : p.out0;
      uint32_t racc[kCols];
#pragma unroll
      for (int cc = 0; cc < kCols / 16; ++cc)
        tmem_ld16(tmem + lane_off + col + 16 * cc, *reinterpret_cast<uint32_t(*)[16]>(&racc[16 * cc]));
      tmem_ld_wait();
#pragma unroll
      for (int cc = 0; cc < kCols / 16; ++cc)
        tmem_ld_fence16(*reinterpret_cast<uint32_t(*)[16]>(&racc[16 * cc]));
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.acc_free());
      // Packed to 16 bits first: half the registers live across the stores.
      uint32_t w[kCols / 2];
#pragma unroll
      for (int e = 0; e < kCols / 2; ++e)
        w[e] = pack_x2<kF16>(__uint_as_float(racc[2 * e]) * mul, __uint_as_float(racc[2 * e + 1]) * mul);
      // 16-byte groups of this thread's part that exist: none past the last
      // row, and none past column d (d may be below the layout's D).
      const int live8 = (x_idx < p.N && guard(bh < p.num_bh && x_idx >= 0 && p.d <= D))
                            ? (p.d - kCols * part) / 8
                            : 0;
      const int ob = bh / p.H, oh = bh - ob * p.H;
      const int64_t row_off = is_dv ? ob * p.out1_sb + oh * p.out1_sh + x_idx * p.out1_sn
                                    : ob * p.out0_sb + oh * p.out0_sh + x_idx * p.out0_sn;
      uint4* dst = reinterpret_cast<uint4*>(out + row_off + kCols * part);
#pragma unroll
      for (int q8 = 0; q8 < kCols / 8; ++q8)
        if (q8 < live8) dst[q8] = make_uint4(w[4 * q8], w[4 * q8 + 1], w[4 * q8 + 2], w[4 * q8 + 3]);
    }
  } else if (warp == kBwdLoadWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // Y tiles are read by every X tile of the same head: keep them in L2.
      const uint64_t keep = make_l2_policy_evict_last();
      const uint64_t once = make_l2_policy_evict_first();
      uint32_t yc = 0;  // Y stages issued over all tiles
      int nx = 0;       // X tiles issued
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const int t = unit_index(r);
        if (t >= total) break;
        const Tile u = tile_at(t);
        // X of this tile replaces the previous one once that one is no longer
        // read from shared memory (x_empty).
        if (r > 0 && !wait_bar(bars.x_empty(), parity_of(r - 1), wctx)) break;
        mbar_arrive_expect_tx(bars.x_full(), 2 * C::kTileBytes);
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
          if (!tma_coord_ok(64 * b, p.d, u.xt * kBwdTile, p.N, u.bh, p.num_bh) ||
              !smem_range_ok(C::kOffX + C::kTileBytes + b * kSwBlockBytes, kSwBlockBytes, C::kOffY))
            continue;
          tma_load_4d_hint(sX + b * kSwBlockBytes, &tm_x0, bars.x_full(), 64 * b,
                           u.xt * kBwdTile, u.bh % p.H, u.bh / p.H, once);
          tma_load_4d_hint(sX + C::kTileBytes + b * kSwBlockBytes, &tm_x1, bars.x_full(), 64 * b,
                           u.xt * kBwdTile, u.bh % p.H, u.bh / p.H, once);
        }
        ++nx;
        for (int m = 0; m < 2 * u.steps; ++m, ++yc) {
          const int s = static_cast<int>(yc % S);
          if (yc >= static_cast<uint32_t>(S) &&
              !wait_bar(bars.y_empty(s), parity_of(yc / S - 1), wctx)) {
            ok = false;
            break;
          }
          const int row0 = (u.y_first + (m >> 1)) * kBwdTile + kBwdSub * (m & 1);
          const uint32_t stage = sY + s * C::kStageBytes;
          // Test hook: the first streamed stage is never copied, so its wait
          // must time out.
          if (yc == 0 && (p.inject & kInjectSkipFirstV)) continue;
          mbar_arrive_expect_tx(bars.y_full(s), C::kStageBytes + C::kVecBytes);
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            // A streamed half may start past N (the last tile's second half
            // when N is ragged): TMA reads it as zeros; it must start inside
            // the padded extent.
            if (!tma_coord_ok(64 * b, p.d, row0, p.Npad, u.bh, p.num_bh) ||
                !smem_range_ok(C::kOffY + s * C::kStageBytes + C::kHalfBytes + b * C::kHalfBlock,
                               C::kHalfBlock, C::kOffVec))
              continue;
            tma_load_4d_hint(stage + b * C::kHalfBlock, &tm_y0, bars.y_full(s), 64 * b, row0,
                             u.bh % p.H, u.bh / p.H, keep);
            tma_load_4d_hint(stage + C::kHalfBytes + b * C::kHalfBlock, &tm_y1, bars.y_full(s),
                             64 * b, row0, u.bh % p.H, u.bh / p.H, keep);
          }
          if (kKV && guard(row0 >= 0 && row0 + kBwdSub <= p.Npad && u.bh < p.num_bh) &&
              smem_range_ok(C::kOffVec + s * C::kVecBytes, C::kVecBytes, C::kOffBar)) {
            const size_t v0 = static_cast<size_t>(u.bh) * p.Npad + row0;
            const uint32_t vec = sbase + C::kOffVec + s * C::kVecBytes;
            bulk_load(vec, p.lse2 + v0, kBwdSub * 4, bars.y_full(s));
            bulk_load(vec + kBwdSub * 4, p.dvec + v0, kBwdSub * 4, bars.y_full(s));
          }
        }
      }
      // Drain: every copy issued must land before the CTA exits.  The last
      // stage count in slot s is the largest one < yc congruent to s mod S.
      if (nx > 0) wait_bar_drain(bars.x_full(), parity_of(nx - 1), wctx);
      for (int s = 0; s < S; ++s) {
        if (yc > static_cast<uint32_t>(s)) {
          const uint32_t last = yc - 1 - ((yc - 1 - s) % S);
          if (!(last == 0 && (p.inject & kInjectSkipFirstV)))
            wait_bar_drain(bars.y_full(s), parity_of(last / S), wctx);
        }
      }
    }
  } else if (warp == kBwdMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = elect_one_sync();
    constexpr uint32_t kHi = desc_hi_sw128(1024);
    // Both operands of every MMA share the element type (P, dS included).
    constexpr uint32_t kIdescSS = kF16 ? idesc_f16_f32(kBwdTile, kBwdSub, 0, 0)
                                       : idesc_bf16_f32(kBwdTile, kBwdSub, 0, 0);
    constexpr uint32_t kIdescAcc = kF16 ? idesc_f16_f32(kBwdTile, D, 0, 1)
                                        : idesc_bf16_f32(kBwdTile, D, 0, 1);
    const uint32_t x_lo = desc_lo(sX, 16);               // X tiles, K-major A
    const uint32_t yk_lo = desc_lo(sY, 16);              // Y tiles, K-major B
    const uint32_t ymn_lo = desc_lo(sY, C::kHalfBlock);  // Y halves, MN-major B
    // K-major slice kk of a stationary 128-row tile (16 KB blocks) and of a
    // streamed 64-row half tile (8 KB blocks).
    auto kmaj_off = [](int kk) -> uint32_t {
      return ((kk >> 2) * kSwBlockBytes + (kk & 3) * 32) >> 4;
    };
    auto kmaj_off_half = [](int kk) -> uint32_t {
      return ((kk >> 2) * C::kHalfBlock + (kk & 3) * 32) >> 4;
    };
    auto commit = [&](uint32_t bar) {
      if (leader) umma_commit(bar);
      __syncwarp();
    };
    // S and dP into TMEM buffer b: X0 and X1 against the 64 streamed rows of
    // Y0 and Y1 in ring slot `stage`.
    auto issue_sdp = [&](int b, uint32_t stage) {
      const uint32_t st = stage * C::kStageBytes;
      const uint32_t y0 = yk_lo + (st >> 4);
      const uint32_t y1 = yk_lo + ((st + C::kHalfBytes) >> 4);
      constexpr uint32_t x1 = C::kTileBytes >> 4;
      if (leader && tmem_range_ok(tmem + C::kColS + kBwdSub * b, kBwdSub) &&
          tmem_range_ok(tmem + C::kColDP + kBwdSub * b, kBwdSub) &&
          (kKV || tmem_range_ok(tmem + C::kColXT, D)) && guard(stage < static_cast<uint32_t>(S))) {
        if (kKV) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss_lohi(tmem + C::kColS + kBwdSub * b, x_lo + kmaj_off(kk), kHi,
                         y0 + kmaj_off_half(kk), kHi, kIdescSS, kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ss_lohi(tmem + C::kColDP + kBwdSub * b, x_lo + x1 + kmaj_off(kk), kHi,
                         y1 + kmaj_off_half(kk), kHi, kIdescSS, kk > 0 ? 1u : 0u);
        } else {
          // A (Q_i, dO_i) from TMEM: 16 columns of the head dimension = 8
          // TMEM columns of pairs.
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ts_lohi(tmem + C::kColS + kBwdSub * b, tmem + C::kColXT + 8u * kk,
                         y0 + kmaj_off_half(kk), kHi, kIdescSS, kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_ts_lohi(tmem + C::kColDP + kBwdSub * b, tmem + C::kColXT + D / 2 + 8u * kk,
                         y1 + kmaj_off_half(kk), kHi, kIdescSS, kk > 0 ? 1u : 0u);
        }
      }
      __syncwarp();
    };
    // Accumulation over the 64 streamed rows of ring slot `stage`, 16 per
    // MMA; the A operand (P^T / dS^T / dS as 16-bit pairs) comes from TMEM
    // buffer b.  `first`: the tile's first sub-step overwrites the accumulators.
    auto issue_acc = [&](int b, uint32_t stage, bool first) {
      const uint32_t st = stage * C::kStageBytes;
      if (leader && tmem_range_ok(tmem + C::kColAcc0, D) &&
          (!kKV || tmem_range_ok(tmem + C::kColAcc1, D)) &&
          tmem_range_ok(tmem + C::kColS + kBwdSub * b, kBwdSub) &&
          tmem_range_ok(tmem + C::kColDP + kBwdSub * b, kBwdSub) &&
          guard(stage < static_cast<uint32_t>(S))) {
#pragma unroll
        for (int kk = 0; kk < kBwdSub / 16; ++kk) {
          const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
          const uint32_t r0 = (st + kk * 16 * 128) >> 4;
          const uint32_t r1 = (st + C::kHalfBytes + kk * 16 * 128) >> 4;
          // Slice kk (16 streamed rows) was packed by warpgroup kk into the
          // first 8 of its 16 columns.
          const uint32_t a_off = kBwdSub * b + kBwdEwCols * kk;
          if (kKV) {
            umma_ts_lohi(tmem + C::kColAcc1, tmem + C::kColS + a_off, ymn_lo + r1, kHi, kIdescAcc,
                         acc);  // dV += P^T dO
            umma_ts_lohi(tmem + C::kColAcc0, tmem + C::kColDP + a_off, ymn_lo + r0, kHi,
                         kIdescAcc, acc);  // dK += dS^T Q
          } else {
            umma_ts_lohi(tmem + C::kColAcc0, tmem + C::kColS + a_off, ymn_lo + r0, kHi, kIdescAcc,
                         acc);  // dQ += dS K
          }
        }
      }
      __syncwarp();
    };
    uint32_t gsub = 0;  // sub-steps (= Y stages) of earlier tiles
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const int t = unit_index(r);
      if (t >= total) break;
      const Tile u = tile_at(t);
      const int M = 2 * u.steps;
      // The key-tile pass reads X from SMEM; the query-tile pass from TMEM,
      // once the elementwise warps have copied it there.
      if (!warp_wait_bar(kKV ? bars.x_full() : bars.x_tmem(), parity_of(r), wctx)) break;
      tc_fence_after_sync();
      // S, dP of sub-steps 0 and 1 overwrite buffers whose previous contents
      // (the last tile's) are read by accumulations issued before them.
      for (int m = 0; ok && m < 2 && m < M; ++m) {
        const uint32_t gm = gsub + static_cast<uint32_t>(m);
        if (!warp_wait_bar(bars.y_full(gm % S), parity_of(gm / S), wctx)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_sdp(m, gm % S);
        commit(bars.st_full(m));
        if (kKV && m == M - 1) commit(bars.x_empty());  // X's last reader issued
      }
      for (int m = 0; ok && m < M; ++m) {
        const int b = m & 1;
        const uint32_t gm = gsub + static_cast<uint32_t>(m);
        if (!warp_wait_bar(bars.p_full(b), parity_of(gm >> 1), wctx) ||
            (m == 0 && r > 0 && !warp_wait_bar(bars.acc_free(), parity_of(r - 1), wctx))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        issue_acc(b, gm % S, m == 0);
        commit(bars.y_empty(gm % S));  // this sub-step's half tiles are consumed
        const int m2 = m + 2;
        if (m2 < M) {
          // S, dP of sub-step m + 2 overwrite buffer b after the accumulation
          // that reads it (MMAs of one thread run in issue order).
          const uint32_t gm2 = gsub + static_cast<uint32_t>(m2);
          if (!warp_wait_bar(bars.y_full(gm2 % S), parity_of(gm2 / S), wctx)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          issue_sdp(b, gm2 % S);
          commit(bars.st_full(b));
          if (kKV && m2 == M - 1) commit(bars.x_empty());
        }
      }
      if (!ok) break;
      commit(bars.acc_done());  // the tile's accumulators are complete
      gsub += static_cast<uint32_t>(M);
    }
    // Every MMA issued has completed once mma_done fires.
    commit(bars.mma_done());
    wait_bar_drain(bars.mma_done(), 0, wctx);
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kBwdMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace fa
