// One row of step a0 (M <- M + G, and the row's l1 norm and sum of squares of
// the new M), shared by the accumulation kernels of mem_kernels.cu and by the
// streaming warps of the tensor-core GEMM (gemm_tcgen05.cu), so every path
// produces the same bits.
//
// Method source: "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of
// the paper), third-level paragraph: the momentum of every row accumulates its
// gradient, and rows are then chosen by their l1 norm.
//
// One warp per row.  The vector path moves 8 elements per lane per iteration
// (two float4 of M, one 16-byte bf16 or two float4 fp32 gradient loads) and
// keeps U iterations of loads in flight before the first dependent store.
// Lane `lane` visits columns lane*8 + 256 t for t = 0, 1, 2, ... in that order
// whatever U is, so the per-lane sums, and after the fixed shuffle tree the
// row's l1 and sum of squares, do not depend on U.
#pragma once

#include "internal.h"

namespace dion3 {

__device__ __forceinline__ float accum_warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void accum_bf16x8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
  }
}

__device__ __forceinline__ float accum_load_grad(const void* g, size_t i, int gd) {
  if (gd == kBF16) {
    const uint16_t h = reinterpret_cast<const uint16_t*>(g)[i];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  return reinterpret_cast<const float*>(g)[i];
}

// Row `r` of an n x cols matrix: Mrow = M + r cols, Grow = G + r cols (or null
// with GD = -1: norms only).  rs is the row's pending lazy-decay factor (1: none):
// the accumulation is then M <- fp32(fp32(rs M) + G).  Returns l1 and sum of
// squares in lane 0 (every lane holds the warp's sums).  EVICT_M: M is read and
// written with the evict-first policy (the gradient always is), for rows moved
// beside a GEMM whose operands should keep L2.
template <bool VEC, int GD, int U, bool EVICT_M = false>
__device__ __forceinline__ void accum_row(float* __restrict__ Mrow, const void* Grow, int cols, float rs,
                                          float& l1_out, float& sq_out) {
  const int lane = threadIdx.x % 32;
  float l1 = 0.f, sq = 0.f;
  const bool scaled = rs != 1.0f;
  if constexpr (VEC) {
    constexpr int step = 32 * 8;
    for (int c0 = lane * 8; c0 < cols; c0 += step * U) {
      float m[U][8];
      // Gradients as loaded: bf16 stays packed (four registers per eight
      // values) until it is used, so more iterations fit in registers.
      uint4 gb[GD == kBF16 ? U : 1];
      float gf[GD == kF32 ? U : 1][8];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * step;
        if (c < cols) {
          float4 x0, x1;
          if constexpr (EVICT_M) {
            x0 = __ldcs(reinterpret_cast<const float4*>(Mrow + c));
            x1 = __ldcs(reinterpret_cast<const float4*>(Mrow + c + 4));
          } else {
            x0 = *reinterpret_cast<const float4*>(Mrow + c);
            x1 = *reinterpret_cast<const float4*>(Mrow + c + 4);
          }
          m[u][0] = x0.x; m[u][1] = x0.y; m[u][2] = x0.z; m[u][3] = x0.w;
          m[u][4] = x1.x; m[u][5] = x1.y; m[u][6] = x1.z; m[u][7] = x1.w;
          if constexpr (GD == kBF16) {
            gb[u] = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(Grow) + c));
          } else if constexpr (GD == kF32) {
            const float* G = reinterpret_cast<const float*>(Grow);
            const float4 y0 = __ldcs(reinterpret_cast<const float4*>(G + c));
            const float4 y1 = __ldcs(reinterpret_cast<const float4*>(G + c + 4));
            gf[u][0] = y0.x; gf[u][1] = y0.y; gf[u][2] = y0.z; gf[u][3] = y0.w;
            gf[u][4] = y1.x; gf[u][5] = y1.y; gf[u][6] = y1.z; gf[u][7] = y1.w;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * step;
        if (c < cols) {
          if constexpr (GD >= 0) {
            float g[8];
            if constexpr (GD == kBF16) {
              accum_bf16x8(gb[u], g);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) g[j] = gf[u][j];
            }
            if (scaled) {
#pragma unroll
              for (int j = 0; j < 8; ++j) m[u][j] = __fmul_rn(rs, m[u][j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) m[u][j] = __fadd_rn(m[u][j], g[j]);
            const float4 y0 = make_float4(m[u][0], m[u][1], m[u][2], m[u][3]);
            const float4 y1 = make_float4(m[u][4], m[u][5], m[u][6], m[u][7]);
            if constexpr (EVICT_M) {
              __stcs(reinterpret_cast<float4*>(Mrow + c), y0);
              __stcs(reinterpret_cast<float4*>(Mrow + c + 4), y1);
            } else {
              *reinterpret_cast<float4*>(Mrow + c) = y0;
              *reinterpret_cast<float4*>(Mrow + c + 4) = y1;
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            l1 += fabsf(m[u][j]);
            sq = fmaf(m[u][j], m[u][j], sq);
          }
        }
      }
    }
  } else {
    for (int c = lane; c < cols; c += 32) {
      float m = Mrow[c];
      if constexpr (GD >= 0) {
        if (scaled) m = __fmul_rn(rs, m);
        m = __fadd_rn(m, accum_load_grad(Grow, static_cast<size_t>(c), GD));
        Mrow[c] = m;
      }
      l1 += fabsf(m);
      sq = fmaf(m, m, sq);
    }
  }
  l1_out = accum_warp_sum(l1);
  sq_out = accum_warp_sum(sq);
}

// Row `row` (= matrix b x rows + r) of an accumulation pool, processed by the
// calling warp: the pool's bookkeeping around accum_row.
template <int GD, int U, bool EVICT_M = false>
__device__ __forceinline__ void accum_pool_row(const AccumPool& pool, long long row) {
  const int b = static_cast<int>(row / pool.rows);
  const int r = static_cast<int>(row - static_cast<long long>(b) * pool.rows);
  float* Mrow = pool.M[b] + static_cast<size_t>(r) * pool.cols;
  const size_t goff = static_cast<size_t>(r) * pool.cols;
  const float rs = pool.scale != nullptr ? pool.scale[row] : 1.0f;
  float l1, sq;
  if constexpr (GD == kBF16)
    accum_row<true, kBF16, U, EVICT_M>(Mrow, reinterpret_cast<const uint16_t*>(pool.G[b]) + goff, pool.cols, rs,
                                       l1, sq);
  else
    accum_row<true, kF32, U, EVICT_M>(Mrow, reinterpret_cast<const float*>(pool.G[b]) + goff, pool.cols, rs, l1,
                                      sq);
  if (threadIdx.x % 32 == 0) {
    pool.l1[row] = l1;
    pool.sq[row] = sq;
    if (pool.scale != nullptr && rs != 1.0f) pool.scale[row] = 1.0f;
  }
}

// Hands out the pool's next row to the calling warp (every lane gets it); a
// value >= pool.total means the pool is exhausted.
__device__ __forceinline__ long long accum_pool_next(const AccumPool& pool) {
  unsigned long long v = 0;
  if (threadIdx.x % 32 == 0) v = atomicAdd(pool.next, 1ull);
  return static_cast<long long>(__shfl_sync(0xffffffffu, v, 0));
}

}  // namespace dion3
