// Memory-bound kernels of the Dion3 step: momentum accumulation with row
// norms, l1 top-k selection, gather/normalise/transpose into fp16, the sum of
// squares used for normalisation, and the row-scatter parameter update.
//
// Method source: "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of
// the paper), third-level paragraph: rows are chosen by l1 norm, k = ceil(f n),
// only the chosen sub-matrix is orthogonalised and only the matching weight
// rows are updated; error feedback decays only the chosen momentum rows by mu.
#include "accum_row.cuh"
#include "internal.h"
#include "scatter_row.cuh"

#include <cuda_bf16.h>

#include <algorithm>

namespace dion3 {
namespace {

constexpr int kWarp = 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 16-bit operand elements of the Gram-NS path: fp16, or bf16 when BF16.
template <bool BF16>
__device__ __forceinline__ float e16_to_f32(uint16_t h) {
  if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
  else return __half2float(__ushort_as_half(h));
}
template <bool BF16>
__device__ __forceinline__ float2 e16x2_to_f32(uint32_t w) {
  if constexpr (BF16) return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  else return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <bool BF16>
__device__ __forceinline__ __half f32_to_e16(float f) {
  if constexpr (BF16) return __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(f)));
  else return __float2half_rn(f);
}

// ---------------------------------------------------------------------------
// a0: M <- M + G and per-row l1 / sum of squares.  One warp per row; the
// vector path moves 8 elements per lane per iteration (two float4 of M, one
// 16-byte bf16 or two float4 fp32 gradient loads) and keeps UNROLL iterations
// of loads in flight before the first dependent store.
// ---------------------------------------------------------------------------
template <bool VEC, int GD>  // GD: kF32, kBF16, or -1 (no gradient: norms only)
__global__ void __launch_bounds__(256) accum_rownorm_kernel(const __grid_constant__ AccumArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const long long total = static_cast<long long>(a.batch) * a.rows;
  if (gw >= total) return;
  const int b = static_cast<int>(gw / a.rows);
  const int r = static_cast<int>(gw % a.rows);
  const int cols = a.cols;
  float* __restrict__ Mrow = a.M[b] + static_cast<size_t>(r) * cols;
  const void* Grow = nullptr;
  if constexpr (GD == kBF16) Grow = reinterpret_cast<const uint16_t*>(a.G[b]) + static_cast<size_t>(r) * cols;
  if constexpr (GD == kF32) Grow = reinterpret_cast<const float*>(a.G[b]) + static_cast<size_t>(r) * cols;
  // Pending lazy decay of this row (warp-uniform); only with a gradient.
  const float rs = (GD >= 0 && a.scale != nullptr) ? a.scale[gw] : 1.0f;
  float l1, sq;
  // 2 iterations of loads in flight measured fastest here (more resident warps).
  accum_row<VEC, GD, 2>(Mrow, Grow, cols, rs, l1, sq);
  if (lane == 0) {
    a.l1[gw] = l1;
    a.sq[gw] = sq;
    if (GD >= 0 && a.scale != nullptr && rs != 1.0f) a.scale[gw] = 1.0f;
  }
}

// The rows of an accumulation pool that nobody has taken yet: each warp takes
// rows from the pool's counter until it is exhausted.
template <int GD>
__global__ void __launch_bounds__(256) accum_pool_kernel(const __grid_constant__ AccumPool pool) {
  pdl_trigger();
  pdl_wait();
  for (;;) {
    const long long row = accum_pool_next(pool);
    if (row >= pool.total) break;
    accum_pool_row<GD, 2>(pool, row);
  }
}

// ---------------------------------------------------------------------------
// a1: top-k by l1.  One CTA per matrix.  l1 >= 0, so its fp32 bit pattern
// orders like its value: a 4-pass 8-bit radix select finds the k-th largest
// key t and how many of the keys equal to t are still needed; a single pass in
// index order then keeps every key > t and the first `need` keys == t (ties go
// to the lower index) and compacts the kept indices in ascending order.
// ---------------------------------------------------------------------------
constexpr int kTopkThreads = 1024;

// Exclusive block-wide scan of one 0/1 flag per thread; returns the rank and
// stores the block total in *total.
__device__ __forceinline__ int block_excl_scan_flag(bool flag, int* warp_tot, int* total) {
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;
  const unsigned ball = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(ball & ((1u << lane) - 1u));
  if (lane == 0) warp_tot[warp] = __popc(ball);
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x / kWarp;
    int v = lane < nw ? warp_tot[lane] : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < nw) warp_tot[lane] = incl - v;  // exclusive
    if (lane == nw - 1) *total = incl;
  }
  __syncthreads();
  const int r = warp_tot[warp] + in_warp;
  __syncthreads();  // warp_tot is reused by the next call
  return r;
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const TopkArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ unsigned hist[256];
  __shared__ unsigned s_prefix;
  __shared__ int s_need;
  __shared__ int warp_tot[32];
  __shared__ int tot_a, tot_b;
  __shared__ float red[32];

  const int b = blockIdx.x;
  const int n = a.rows;
  const unsigned* keys = reinterpret_cast<const unsigned*>(a.l1 + static_cast<size_t>(b) * n);
  const float* sq = a.sq + static_cast<size_t>(b) * n;
  const int tid = threadIdx.x;

  unsigned prefix = 0u, mask = 0u;
  int need = a.k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += blockDim.x) {
      const unsigned u = keys[i];
      if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid == 0) {
      unsigned above = 0u;
      int d = 255;
      for (; d > 0; --d) {
        if (above + hist[d] >= static_cast<unsigned>(need)) break;
        above += hist[d];
      }
      s_prefix = prefix | (static_cast<unsigned>(d) << shift);
      s_need = need - static_cast<int>(above);
    }
    __syncthreads();
    prefix = s_prefix;
    need = s_need;
    mask |= 255u << shift;
    __syncthreads();
  }

  // Compaction in index order.
  int run_eq = 0, run_sel = 0;
  float fsum = 0.f;
  int32_t* out = a.idx + static_cast<size_t>(b) * a.k;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const bool valid = i < n;
    const unsigned u = valid ? keys[i] : 0u;
    const bool gt = valid && u > prefix;
    const bool eq = valid && u == prefix;
    const int eq_rank = run_eq + block_excl_scan_flag(eq, warp_tot, &tot_a);
    const bool sel = gt || (eq && eq_rank < need);
    const int pos = run_sel + block_excl_scan_flag(sel, warp_tot, &tot_b);
    if (sel && pos < a.k) {
      out[pos] = i;
      fsum += sq[i];
    }
    run_eq += tot_a;
    run_sel += tot_b;
  }
  if (a.fro2 != nullptr) {
    fsum = warp_sum(fsum);
    if (tid % kWarp == 0) red[tid / kWarp] = fsum;
    __syncthreads();
    if (tid < kWarp) {
      float v = tid < static_cast<int>(blockDim.x / kWarp) ? red[tid] : 0.f;
      v = warp_sum(v);
      if (tid == 0) a.fro2[b] = v;
    }
  }
}

// ---------------------------------------------------------------------------
// a2: gather + normalise into fp16, in the rows orientation and (if out_cols
// is set) also the columns orientation, with the error-feedback decay of the
// source momentum rows fused in (the undecayed values are the ones
// normalised).  Tile: 32 selected rows x 128 columns per CTA; each warp reads
// one 512-byte row segment per pass; the column-major copy is staged through
// shared memory so both outputs are written in contiguous runs.
// ---------------------------------------------------------------------------
constexpr int kGRows = 32, kGCols = 128;

template <bool SRC_F32, bool VEC, bool BF16>
__global__ void __launch_bounds__(256) gather_kernel(const __grid_constant__ GatherArgs a) {
  pdl_trigger();
  pdl_wait();
  // Column-major staging: a pitch of 34 halves (17 words) spreads the 2-byte
  // writes of a warp over 8 banks (4-way conflicts; a 16-byte-aligned pitch of
  // 40 gave 16-way conflicts and cost a quarter of the kernel's time).
  __shared__ __align__(16) __half tile[kGCols][kGRows + 2];
  const int b = blockIdx.z;
  const int i0 = blockIdx.y * kGRows;
  const int c0 = blockIdx.x * kGCols;
  const int lane = threadIdx.x % kWarp, warp = threadIdx.x / kWarp;

  if constexpr (SRC_F32) {
    // Lazy decay: record the pending factor of each selected row once (by the
    // CTAs of the first column tile) instead of writing mu M back.
    if (a.scale_out != nullptr && blockIdx.x == 0 && threadIdx.x < kGRows && i0 + threadIdx.x < a.k) {
      const int row = a.idx[static_cast<size_t>(b) * a.k + i0 + threadIdx.x];
      if (row >= 0 && row < a.n) a.scale_out[static_cast<size_t>(b) * a.n + row] = a.mu;
    }
  }
  float f2 = 0.f;
  for (int p = 0; p < a.fro2_parts; ++p) f2 += a.fro2[static_cast<size_t>(b) * a.fro2_parts + p];
  const float inv = 1.0f / (sqrtf(f2) + a.eps);

  for (int rr = warp; rr < kGRows; rr += 256 / kWarp) {
    const int i = i0 + rr;
    const int c = c0 + lane * 4;
    __half h[4] = {__float2half_rn(0.f), __float2half_rn(0.f), __float2half_rn(0.f), __float2half_rn(0.f)};
    bool live = i < a.k && c < a.m;
    int row = 0;
    if constexpr (SRC_F32) {
      if (i < a.k) {
        row = a.idx[static_cast<size_t>(b) * a.k + i];
        if (row < 0 || row >= a.n) {  // never expected: record it and skip the access
          if (lane == 0) atomicOr(a.status, kDevCheck);
          live = false;
        }
      }
    }
    if (live) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      const bool full = VEC && (c + 4 <= a.m);
      if constexpr (SRC_F32) {
        float* src = a.M[b] + static_cast<size_t>(row) * a.m;
        if (full) {
          const float4 x = *reinterpret_cast<const float4*>(src + c);
          v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
          if (a.decay)
            *reinterpret_cast<float4*>(src + c) =
                make_float4(__fmul_rn(a.mu, x.x), __fmul_rn(a.mu, x.y), __fmul_rn(a.mu, x.z), __fmul_rn(a.mu, x.w));
        } else {
          for (int j = 0; j < 4; ++j)
            if (c + j < a.m) {
              v[j] = src[c + j];
              if (a.decay) src[c + j] = __fmul_rn(a.mu, v[j]);
            }
        }
      } else {
        const __half* src = a.X + (static_cast<size_t>(b) * a.k + i) * a.m;
        if (full) {
          const uint2 x = *reinterpret_cast<const uint2*>(src + c);
          const float2 p0 = e16x2_to_f32<BF16>(x.x), p1 = e16x2_to_f32<BF16>(x.y);
          v[0] = p0.x; v[1] = p0.y;
          v[2] = p1.x; v[3] = p1.y;
        } else {
          for (int j = 0; j < 4; ++j)
            if (c + j < a.m) v[j] = e16_to_f32<BF16>(__half_as_ushort(src[c + j]));
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = f32_to_e16<BF16>(v[j] * inv);
      __half* dst = a.out_rows + static_cast<long long>(b) * a.rows_bstride + static_cast<size_t>(i) * a.ld_rows + c;
      if (full && (a.ld_rows % 4 == 0)) {
        uint2 w;
        __half2 q0 = __halves2half2(h[0], h[1]);
        __half2 q1 = __halves2half2(h[2], h[3]);
        w.x = *reinterpret_cast<uint32_t*>(&q0);
        w.y = *reinterpret_cast<uint32_t*>(&q1);
        *reinterpret_cast<uint2*>(dst) = w;
      } else {
        for (int j = 0; j < 4; ++j)
          if (c + j < a.m) dst[j] = h[j];
      }
    }
    if (a.out_cols != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j) tile[lane * 4 + j][rr] = h[j];
    }
  }
  if (a.out_cols == nullptr) return;  // CTA-uniform
  __syncthreads();

  // Column-major copy: out_cols[c][i0 .. i0+32), 16 bytes per thread.  Rows
  // in [k, ld_cols) are pitch padding and receive zeros.
  for (int pass = 0; pass < 2; ++pass) {
    const int cc = pass * 64 + threadIdx.x / 4;
    const int seg = (threadIdx.x % 4) * 8;
    const int c = c0 + cc;
    const int i = i0 + seg;
    if (c >= a.m || i >= a.ld_cols) continue;
    __half* dst = a.out_cols + static_cast<long long>(b) * a.cols_bstride + static_cast<size_t>(c) * a.ld_cols + i;
    if (i + 8 <= a.ld_cols && (a.ld_cols % 8 == 0)) {
      const uint32_t* t32 = reinterpret_cast<const uint32_t*>(&tile[cc][seg]);  // 4-byte aligned rows
      *reinterpret_cast<uint4*>(dst) = make_uint4(t32[0], t32[1], t32[2], t32[3]);
    } else {
      for (int j = 0; j < 8 && i + j < a.ld_cols; ++j) dst[j] = tile[cc][seg + j];
    }
  }
}

// a2, rows orientation only (the Gram path): one warp per selected row and
// column span of kGSpan (grid.y), 8 elements per lane per step, so each warp
// streams 8 KB row pieces (the tiled kernel above reads 512-byte pieces).  Same arithmetic as the tiled
// kernel: inv = 1 / (sqrt(sum of the fro2 parts) + eps), X = e16(v * inv), and
// the decay mu v written back in fp32.
constexpr int kGSpan = 2048;

template <bool SRC_F32, bool VEC, bool BF16>
__global__ void __launch_bounds__(256) gather_rows_kernel(const __grid_constant__ GatherArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const long long total = static_cast<long long>(a.batch) * a.k;
  if (gw >= total) return;
  const int b = static_cast<int>(gw / a.k);
  const int i = static_cast<int>(gw % a.k);
  float f2 = 0.f;
  for (int p = 0; p < a.fro2_parts; ++p) f2 += a.fro2[static_cast<size_t>(b) * a.fro2_parts + p];
  const float inv = 1.0f / (sqrtf(f2) + a.eps);
  __half* dst = a.out_rows + static_cast<long long>(b) * a.rows_bstride + static_cast<size_t>(i) * a.ld_rows;
  const int cbeg = blockIdx.y * kGSpan;
  const int m = a.m - cbeg < kGSpan ? a.m : cbeg + kGSpan;  // end of this warp's columns
  if constexpr (SRC_F32) {
    const int row = a.idx[static_cast<size_t>(b) * a.k + i];
    if (row < 0 || row >= a.n) {  // never expected: record it and skip the access
      if (lane == 0) atomicOr(a.status, kDevCheck);
      return;
    }
    if (a.scale_out != nullptr && lane == 0 && blockIdx.y == 0)
      a.scale_out[static_cast<size_t>(b) * a.n + row] = a.mu;
    float* src = a.M[b] + static_cast<size_t>(row) * a.m;
    if constexpr (VEC) {
      constexpr int U = 4;  // steps of loads in flight per lane
      const int step = kWarp * 8;
      for (int c0 = cbeg + lane * 8; c0 < m; c0 += step * U) {
        float4 x[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * step;
          if (c < m) {
            x[u][0] = *reinterpret_cast<const float4*>(src + c);
            x[u][1] = *reinterpret_cast<const float4*>(src + c + 4);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * step;
          if (c >= m) continue;
          const float4 x0 = x[u][0], x1 = x[u][1];
          const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __half2 q = __halves2half2(f32_to_e16<BF16>(v[2 * j] * inv), f32_to_e16<BF16>(v[2 * j + 1] * inv));
            w[j] = *reinterpret_cast<uint32_t*>(&q);
          }
          *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
          if (a.decay) {
            *reinterpret_cast<float4*>(src + c) =
                make_float4(__fmul_rn(a.mu, x0.x), __fmul_rn(a.mu, x0.y), __fmul_rn(a.mu, x0.z), __fmul_rn(a.mu, x0.w));
            *reinterpret_cast<float4*>(src + c + 4) =
                make_float4(__fmul_rn(a.mu, x1.x), __fmul_rn(a.mu, x1.y), __fmul_rn(a.mu, x1.z), __fmul_rn(a.mu, x1.w));
          }
        }
      }
    } else {
      for (int c = cbeg + lane; c < m; c += kWarp) {
        const float v = src[c];
        dst[c] = f32_to_e16<BF16>(v * inv);
        if (a.decay) src[c] = __fmul_rn(a.mu, v);
      }
    }
  } else {
    const __half* src = a.X + (static_cast<size_t>(b) * a.k + i) * a.m;
    if constexpr (VEC) {
      for (int c = cbeg + lane * 8; c < m; c += kWarp * 8) {
        const uint4 x = *reinterpret_cast<const uint4*>(src + c);
        const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = e16x2_to_f32<BF16>(xw[j]);
          __half2 q = __halves2half2(f32_to_e16<BF16>(f.x * inv), f32_to_e16<BF16>(f.y * inv));
          w[j] = *reinterpret_cast<uint32_t*>(&q);
        }
        *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      for (int c = cbeg + lane; c < m; c += kWarp)
        dst[c] = f32_to_e16<BF16>(e16_to_f32<BF16>(__half_as_ushort(src[c])) * inv);
    }
  }
}

// Sum of squares of fp16 X: grid (nparts, batch); part p covers a contiguous
// chunk of matrix b.
template <bool BF16>
__global__ void __launch_bounds__(256) sumsq_f16_kernel(const __half* X, long long n, float* parts, int nparts) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8];
  const int b = blockIdx.y, p = blockIdx.x;
  const long long chunk = ((n + nparts - 1) / nparts + 7) / 8 * 8;
  const long long lo = p * chunk;
  const long long hi = lo + chunk < n ? lo + chunk : n;
  const __half* x = X + static_cast<long long>(b) * n;
  float s = 0.f;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & 15u) == 0) && (n % 8 == 0);
  if (vec) {
    for (long long i = lo + threadIdx.x * 8LL; i < hi; i += 256LL * 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(x + i);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = e16x2_to_f32<BF16>(w[j]);
        s = fmaf(f.x, f.x, s);
        s = fmaf(f.y, f.y, s);
      }
    }
  } else {
    for (long long i = lo + threadIdx.x; i < hi; i += 256) {
      const float f = e16_to_f32<BF16>(__half_as_ushort(x[i]));
      s = fmaf(f, f, s);
    }
  }
  s = warp_sum(s);
  if (threadIdx.x % kWarp == 0) red[threadIdx.x / kWarp] = s;
  __syncthreads();
  if (threadIdx.x < kWarp) {
    float v = threadIdx.x < 8 ? red[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) parts[static_cast<size_t>(b) * nparts + p] = v;
  }
}

// ---------------------------------------------------------------------------
// a7: W[S_i] <- round_p(W[S_i] - lr O[i]).  One warp per selected row.
// ---------------------------------------------------------------------------
template <int PD, bool VEC, bool BF16, bool NORM = false>
__global__ void __launch_bounds__(256) scatter_kernel(const __grid_constant__ ScatterArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const long long total = static_cast<long long>(a.batch) * a.k;
  if (gw >= total) return;
  const int b = static_cast<int>(gw / a.k);
  const int i = static_cast<int>(gw % a.k);
  const int row = a.idx[static_cast<size_t>(b) * a.k + i];
  if (row < 0 || row >= a.rows) {  // never expected: record and skip the access
    if (lane == 0) atomicOr(a.status, kDevCheck);
    return;
  }
  const __half* O = a.O + static_cast<long long>(b) * a.o_bstride + static_cast<size_t>(i) * a.ld_o;
  const int cols = a.cols;
  const float nlr = NORM ? -(a.lr * a.row_factor[static_cast<size_t>(b) * a.k + i]) : -a.lr;
  if constexpr (VEC) {
    void* W = PD == kBF16 ? static_cast<void*>(reinterpret_cast<__nv_bfloat16*>(a.W[b]) + static_cast<size_t>(row) * cols)
                          : static_cast<void*>(reinterpret_cast<float*>(a.W[b]) + static_cast<size_t>(row) * cols);
    scatter_row<PD, BF16>(W, O, cols, nlr);
  } else if constexpr (PD == kBF16) {
    __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(a.W[b]) + static_cast<size_t>(row) * cols;
    for (int c = lane; c < cols; c += kWarp)
      W[c] = __float2bfloat16_rn(fmaf(nlr, e16_to_f32<BF16>(__half_as_ushort(O[c])), __bfloat162float(W[c])));
  } else {
    float* W = reinterpret_cast<float*>(a.W[b]) + static_cast<size_t>(row) * cols;
    for (int c = lane; c < cols; c += kWarp) W[c] = fmaf(nlr, e16_to_f32<BF16>(__half_as_ushort(O[c])), W[c]);
  }
}

// The rest of a scatter pool: warps take rows from the pool's counter until
// it is exhausted.
__global__ void __launch_bounds__(256) scatter_pool_kernel(const __grid_constant__ ScatterPool p) {
  pdl_trigger();
  pdl_wait();
  for (;;) {
    const long long row = scatter_pool_next(p);
    if (row >= p.total) break;
    scatter_pool_row<1>(p, row);
  }
}

// M[b][r] <- fp32(s M[b][r]) for rows whose pending factor s is not 1; s <- 1.
// One warp per row; rows with s = 1 cost one load.
__global__ void __launch_bounds__(256) flush_scale_kernel(const __grid_constant__ FlushArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  if (gw >= static_cast<long long>(a.batch) * a.rows) return;
  const float s = a.scale[gw];
  if (s == 1.0f) return;
  const int b = static_cast<int>(gw / a.rows), r = static_cast<int>(gw % a.rows);
  float* row = a.M[b] + static_cast<size_t>(r) * a.cols;
  for (int c = lane; c < a.cols; c += kWarp) row[c] = __fmul_rn(s, row[c]);
  __syncwarp();
  if (lane == 0) a.scale[gw] = 1.0f;
}

inline unsigned ceil_div(long long a, long long b) { return static_cast<unsigned>((a + b - 1) / b); }

}  // namespace

// ---------------------------------------------------------------------------
// Per-neuron normalisation (NorMuon reading; "Dion3 Cuts Muon Optimizer Time
// by Up to 6x ...", section "Dion3's fastest path is a combined systems stack",
// names it; "Dion3: Full-Stack Orthogonal Updates", limitations paragraph: in
// float32).  One warp per selected row: the row's sum of squares of O, the
// running second moment of the row's parameter row, and its factor
// 1 / (sqrt(v) + eps); then one CTA per matrix sums d^2 q over the rows in a
// fixed order and scales the factors so that the written block has RMS rms.
// ---------------------------------------------------------------------------
template <bool VEC, bool BF16>
__global__ void __launch_bounds__(256) normuon_rows_kernel(const __grid_constant__ NormRowsArgs a) {
  pdl_trigger();
  pdl_wait();
  const int lane = threadIdx.x % kWarp;
  const long long gw = static_cast<long long>(blockIdx.x) * (blockDim.x / kWarp) + threadIdx.x / kWarp;
  const long long total = static_cast<long long>(a.batch) * a.k;
  if (gw >= total) return;
  const int b = static_cast<int>(gw / a.k);
  const int i = static_cast<int>(gw % a.k);
  const int row = a.idx[gw];
  if (row < 0 || row >= a.rows) {  // never expected: record and skip the access
    if (lane == 0) atomicOr(a.status, kDevCheck);
    return;
  }
  const __half* O = a.O + static_cast<long long>(b) * a.o_bstride + static_cast<size_t>(i) * a.ld_o;
  float q = 0.f;
  if constexpr (VEC) {
    for (int c = lane * 8; c < a.m; c += kWarp * 8) {
      const uint4 o = *reinterpret_cast<const uint4*>(O + c);
      const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = e16x2_to_f32<BF16>(w[j]);
        q = fmaf(f.x, f.x, q);
        q = fmaf(f.y, f.y, q);
      }
    }
  } else {
    for (int c = lane; c < a.m; c += kWarp) {
      const float f = e16_to_f32<BF16>(__half_as_ushort(O[c]));
      q = fmaf(f, f, q);
    }
  }
  q = warp_sum(q);
  if (lane == 0) {
    float* v = a.v + static_cast<size_t>(b) * a.rows + row;
    const float vn = __fadd_rn(__fmul_rn(a.beta2, *v), __fmul_rn(1.0f - a.beta2, q / static_cast<float>(a.m)));
    *v = vn;
    const float d = 1.0f / (sqrtf(vn) + a.eps);
    a.d[gw] = d;
    a.rowc[gw] = d * d * q;
  }
}

constexpr int kNormScaleThreads = 256;

__global__ void __launch_bounds__(kNormScaleThreads) normuon_scale_kernel(const __grid_constant__ NormScaleArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float part[kNormScaleThreads / kWarp];
  __shared__ float g_sh;
  const int b = blockIdx.x;
  const float* rc = a.rowc + static_cast<size_t>(b) * a.k;
  float acc = 0.f;
  for (int i = threadIdx.x; i < a.k; i += kNormScaleThreads) acc += rc[i];
  acc = warp_sum(acc);
  if (threadIdx.x % kWarp == 0) part[threadIdx.x / kWarp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float f2 = 0.f;
    for (int w = 0; w < kNormScaleThreads / kWarp; ++w) f2 += part[w];
    g_sh = f2 > 0.f ? a.rms * sqrtf(static_cast<float>(a.k) * static_cast<float>(a.m)) / sqrtf(f2) : 0.f;
  }
  __syncthreads();
  const float g = g_sh;
  float* d = a.d + static_cast<size_t>(b) * a.k;
  for (int i = threadIdx.x; i < a.k; i += kNormScaleThreads) d[i] *= g;
}

cudaError_t launch_accum_rownorm(const AccumArgs& a, bool vec, cudaStream_t s) {
  const long long total = static_cast<long long>(a.batch) * a.rows;
  const bool has_grad = a.G[0] != nullptr;
  void (*k)(AccumArgs);
  if (vec)
    k = !has_grad ? accum_rownorm_kernel<true, -1>
                  : (a.grad_dtype == kBF16 ? accum_rownorm_kernel<true, kBF16> : accum_rownorm_kernel<true, kF32>);
  else
    k = !has_grad ? accum_rownorm_kernel<false, -1>
                  : (a.grad_dtype == kBF16 ? accum_rownorm_kernel<false, kBF16> : accum_rownorm_kernel<false, kF32>);
  return launch_kernel(false, k, dim3(ceil_div(total, 8)), dim3(256), 0, s, a);
}

cudaError_t launch_accum_pool(const AccumPool& p, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Enough warps to keep HBM busy (8 CTAs of 8 warps per SM), no more than rows.
  const long long want = std::min<long long>(static_cast<long long>(sms) * 8, ceil_div(p.total, 8));
  return launch_kernel(false, p.grad_dtype == kBF16 ? accum_pool_kernel<kBF16> : accum_pool_kernel<kF32>,
                       dim3(static_cast<unsigned>(std::max<long long>(want, 1))), dim3(256), 0, s, p);
}

cudaError_t launch_flush_scale(const FlushArgs& a, cudaStream_t s) {
  const long long total = static_cast<long long>(a.batch) * a.rows;
  return launch_kernel(false, flush_scale_kernel, dim3(ceil_div(total, 8)), dim3(256), 0, s, a);
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s) {
  return launch_kernel(false, topk_kernel, dim3(a.batch), dim3(kTopkThreads), 0, s, a);
}

cudaError_t launch_gather(const GatherArgs& a, bool vec, cudaStream_t s) {
  if (a.out_cols == nullptr) {
    // Rows only: whole-row warps; 16-byte accesses need m and the pitch in
    // multiples of 8 (and 16-byte aligned bases, which the callers keep).
    const bool v8 = vec && a.m % 8 == 0 && a.ld_rows % 8 == 0;
    void (*k)(GatherArgs);
    if (a.bf16) {
      if (a.src_f32) k = v8 ? gather_rows_kernel<true, true, true> : gather_rows_kernel<true, false, true>;
      else k = v8 ? gather_rows_kernel<false, true, true> : gather_rows_kernel<false, false, true>;
    } else {
      if (a.src_f32) k = v8 ? gather_rows_kernel<true, true, false> : gather_rows_kernel<true, false, false>;
      else k = v8 ? gather_rows_kernel<false, true, false> : gather_rows_kernel<false, false, false>;
    }
    const long long total = static_cast<long long>(a.batch) * a.k;
    return launch_kernel(false, k, dim3(ceil_div(total, 8), ceil_div(a.m, kGSpan)), dim3(256), 0, s, a);
  }
  const dim3 grid(ceil_div(a.m, kGCols), ceil_div(a.k, kGRows), a.batch), block(256);
  void (*k)(GatherArgs);
  if (a.bf16) {
    if (a.src_f32) k = vec ? gather_kernel<true, true, true> : gather_kernel<true, false, true>;
    else k = vec ? gather_kernel<false, true, true> : gather_kernel<false, false, true>;
  } else {
    if (a.src_f32) k = vec ? gather_kernel<true, true, false> : gather_kernel<true, false, false>;
    else k = vec ? gather_kernel<false, true, false> : gather_kernel<false, false, false>;
  }
  return launch_kernel(false, k, grid, block, 0, s, a);
}

cudaError_t launch_sumsq_f16(const __half* X, long long n, int batch, float* parts, int nparts, bool bf16,
                             cudaStream_t s) {
  return launch_kernel(false, bf16 ? sumsq_f16_kernel<true> : sumsq_f16_kernel<false>, dim3(nparts, batch), dim3(256), 0,
                       s, X, n, parts, nparts);
}

cudaError_t launch_scatter(const ScatterArgs& a, bool vec, cudaStream_t s) {
  const long long total = static_cast<long long>(a.batch) * a.k;
  void (*k)(ScatterArgs);
  const bool norm = a.row_factor != nullptr;
  if (a.param_dtype == kBF16) {
    if (a.o_bf16)
      k = vec ? (norm ? scatter_kernel<kBF16, true, true, true> : scatter_kernel<kBF16, true, true>)
              : (norm ? scatter_kernel<kBF16, false, true, true> : scatter_kernel<kBF16, false, true>);
    else
      k = vec ? (norm ? scatter_kernel<kBF16, true, false, true> : scatter_kernel<kBF16, true, false>)
              : (norm ? scatter_kernel<kBF16, false, false, true> : scatter_kernel<kBF16, false, false>);
  } else {
    if (a.o_bf16)
      k = vec ? (norm ? scatter_kernel<kF32, true, true, true> : scatter_kernel<kF32, true, true>)
              : (norm ? scatter_kernel<kF32, false, true, true> : scatter_kernel<kF32, false, true>);
    else
      k = vec ? (norm ? scatter_kernel<kF32, true, false, true> : scatter_kernel<kF32, true, false>)
              : (norm ? scatter_kernel<kF32, false, false, true> : scatter_kernel<kF32, false, false>);
  }
  return launch_kernel(false, k, dim3(ceil_div(total, 8)), dim3(256), 0, s, a);
}

cudaError_t launch_scatter_pool(const ScatterPool& p, cudaStream_t s) {
  int sms = 0, dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long want = std::max<long long>(1, ceil_div(p.total, 8));
  const int grid = static_cast<int>(std::min<long long>(static_cast<long long>(sms) * 8, want));
  return launch_kernel(false, scatter_pool_kernel, dim3(grid), dim3(256), 0, s, p);
}

cudaError_t launch_normuon_rows(const NormRowsArgs& a, bool vec, cudaStream_t s) {
  const long long total = static_cast<long long>(a.batch) * a.k;
  void (*k)(NormRowsArgs);
  if (a.o_bf16)
    k = vec ? normuon_rows_kernel<true, true> : normuon_rows_kernel<false, true>;
  else
    k = vec ? normuon_rows_kernel<true, false> : normuon_rows_kernel<false, false>;
  return launch_kernel(false, k, dim3(ceil_div(total, 8)), dim3(256), 0, s, a);
}

cudaError_t launch_normuon_scale(const NormScaleArgs& a, cudaStream_t s) {
  return launch_kernel(false, normuon_scale_kernel, dim3(a.batch), dim3(kNormScaleThreads), 0, s, a);
}

}  // namespace dion3
