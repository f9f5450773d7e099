// One row of step a7 (W[S_i] <- round_p(W[S_i] - lr O[i])), shared by the
// scatter kernel of mem_kernels.cu and by the streaming warps of the
// tensor-core GEMM (gemm_tcgen05.cu) when a shape group's update is deferred
// into another group's Newton-Schulz launches, so every path writes the same
// bits.
//
// Method source: "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of
// the paper), third-level paragraph: only the weight rows that were selected
// are updated, each from its row of the orthogonalised sub-matrix.
//
// One warp per row, 8 columns per lane per iteration (cols a multiple of 8,
// W and O rows 16-byte aligned): W' = round_p(fma(-lr, O, W)).
#pragma once

#include "internal.h"

#include <cuda_bf16.h>

namespace dion3 {

// 16-bit O elements: fp16, or bf16 when O_BF16.
template <bool O_BF16>
__device__ __forceinline__ float2 scatter_o2(uint32_t w) {
  if constexpr (O_BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// nlr = -lr (times the row's factor when the rows are normalised).  U
// iterations of loads (8 columns per lane each) are in flight before the first
// dependent store; the arithmetic of every element is the same whatever U is.
template <int PD, bool O_BF16, int U = 1>
__device__ __forceinline__ void scatter_row(void* Wrow, const __half* Orow, int cols, float nlr) {
  const int lane = threadIdx.x % 32;
  constexpr int step = 32 * 8;
  for (int c0 = lane * 8; c0 < cols; c0 += step * U) {
    uint4 o[U];
    uint4 w[PD == kBF16 ? U : 2 * U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * step;
      if (c < cols) {
        o[u] = *reinterpret_cast<const uint4*>(Orow + c);
        if constexpr (PD == kBF16) {
          w[u] = *reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(Wrow) + c);
        } else {
          w[2 * u] = *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(Wrow) + c);
          w[2 * u + 1] = *reinterpret_cast<const uint4*>(reinterpret_cast<const float*>(Wrow) + c + 4);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u * step;
      if (c >= cols) break;
      const uint32_t ow[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
      if constexpr (PD == kBF16) {
        const uint32_t ww[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
        uint32_t outw[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float w0 = __uint_as_float(ww[j] << 16), w1 = __uint_as_float(ww[j] & 0xffff0000u);
          const float2 of = scatter_o2<O_BF16>(ow[j]);
          const __nv_bfloat162 r = __floats2bfloat162_rn(fmaf(nlr, of.x, w0), fmaf(nlr, of.y, w1));
          outw[j] = *reinterpret_cast<const uint32_t*>(&r);
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(Wrow) + c) =
            make_uint4(outw[0], outw[1], outw[2], outw[3]);
      } else {
        const uint32_t wv[8] = {w[2 * u].x, w[2 * u].y, w[2 * u].z, w[2 * u].w,
                                w[2 * u + 1].x, w[2 * u + 1].y, w[2 * u + 1].z, w[2 * u + 1].w};
        float r[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 of = scatter_o2<O_BF16>(ow[j]);
          r[2 * j] = fmaf(nlr, of.x, __uint_as_float(wv[2 * j]));
          r[2 * j + 1] = fmaf(nlr, of.y, __uint_as_float(wv[2 * j + 1]));
        }
        float* W = reinterpret_cast<float*>(Wrow) + c;
        *reinterpret_cast<float4*>(W) = make_float4(r[0], r[1], r[2], r[3]);
        *reinterpret_cast<float4*>(W + 4) = make_float4(r[4], r[5], r[6], r[7]);
      }
    }
  }
}

// Row `row` of a scatter pool (segments of deferred shape groups, rows
// numbered segment by segment, matrix by matrix, selected row by selected
// row), written by the calling warp with U iterations of loads in flight.  An
// index outside the matrix records kDevCheck and touches nothing.
template <int U>
__device__ __forceinline__ void scatter_pool_row(const ScatterPool& p, long long row) {
  int s = 0;
  while (s + 1 < p.nseg && row >= p.seg[s + 1].start) ++s;
  const ScatterSeg& g = p.seg[s];
  const long long local = row - g.start;
  const int b = static_cast<int>(local / g.k);
  const int i = static_cast<int>(local - static_cast<long long>(b) * g.k);
  const int r = g.idx[static_cast<size_t>(b) * g.k + i];
  if (r < 0 || r >= g.rows) {
    if (threadIdx.x % 32 == 0) atomicOr(p.status, kDevCheck);
    return;
  }
  const __half* O = g.O + static_cast<long long>(b) * g.o_bstride + static_cast<size_t>(i) * g.ld_o;
  // The scatter kernel's expression, so a deferred normalised row gets the same bits.
  const float nlr = g.row_factor != nullptr ? -(g.lr * g.row_factor[static_cast<size_t>(b) * g.k + i]) : -g.lr;
  if (g.param_dtype == kBF16) {
    void* W = reinterpret_cast<__nv_bfloat16*>(g.W[b]) + static_cast<size_t>(r) * g.cols;
    if (g.o_bf16) scatter_row<kBF16, true, U>(W, O, g.cols, nlr);
    else scatter_row<kBF16, false, U>(W, O, g.cols, nlr);
  } else {
    void* W = reinterpret_cast<float*>(g.W[b]) + static_cast<size_t>(r) * g.cols;
    if (g.o_bf16) scatter_row<kF32, true, (U + 1) / 2>(W, O, g.cols, nlr);
    else scatter_row<kF32, false, (U + 1) / 2>(W, O, g.cols, nlr);
  }
}

// Hands out the scatter pool's next row to the calling warp (every lane gets
// it); a value >= p.total means the pool is exhausted.
__device__ __forceinline__ long long scatter_pool_next(const ScatterPool& p) {
  unsigned long long v = 0;
  if (threadIdx.x % 32 == 0) v = atomicAdd(p.next, 1ull);
  return static_cast<long long>(__shfl_sync(0xffffffffu, v, 0));
}

}  // namespace dion3
