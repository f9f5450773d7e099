// Internal launcher interface shared by the library's translation units.
// Nothing here crosses the C ABI (include/dion3.h is the public surface).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace dion3 {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The tensor-core GEMMs are launched with
// programmatic stream serialization: their CTAs may be scheduled while the
// previous kernel on the stream is finishing, run their set-up (barriers,
// tensor memory), and then wait in pdl_wait() until that kernel has completed
// and its memory is visible; no global memory is touched before the wait.
// Every kernel calls pdl_trigger() first, so a following GEMM may be scheduled
// as soon as all of its CTAs have started.  The memory-bound kernels are
// launched without the attribute (their early CTAs would sit beside a running
// GEMM: measured slower), so for them both instructions do nothing.
// DION3_PDL=0 turns the attribute off everywhere.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Whether GEMM launches carry the attribute (DION3_PDL, read once; default on).
bool pdl_enabled();

// Launch with or without the programmatic-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (pdl) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Device status word bits (written by bounded device-side waits and checks).
enum : unsigned { kDevTimeout = 1u, kDevCheck = 2u };

// Matrices per launch of the pointer-table kernels (keeps parameters < 4 KB).
constexpr int kMaxBatchPerLaunch = 96;

enum DType : int { kF32 = 0, kBF16 = 1, kF16 = 2 };

// ---------------------------------------------------------------------------
// Memory-bound kernels (mem_kernels.cu)
// ---------------------------------------------------------------------------

// a0: M <- M + G (if G given) and per-row l1 / sum of squares of the new M.
struct AccumArgs {
  int rows, cols, batch;             // batch <= kMaxBatchPerLaunch
  int grad_dtype;                    // kF32 or kBF16
  float* M[kMaxBatchPerLaunch];
  const void* G[kMaxBatchPerLaunch]; // all null: norms only
  float* l1;                         // [batch][rows]
  float* sq;                         // [batch][rows]
  // Lazy decay: pending per-row factor s ([batch][rows]); the accumulation
  // becomes M <- fp32(fp32(s M) + G) and s is reset to 1.  Null: s = 1.
  float* scale = nullptr;
};
cudaError_t launch_accum_rownorm(const AccumArgs& a, bool vec, cudaStream_t s);

// Step a0 of one shape group as a pool of rows (row id = matrix x rows + row)
// handed out one at a time by a device counter to whichever warps ask first:
// the streaming warps of the tensor-core GEMM launches that run meanwhile (see
// GemmDesc::pool), then launch_accum_pool for whatever is left.  Every row is
// accumulated exactly once, with the arithmetic of accum_rownorm.
constexpr int kPoolMax = 128;  // matrices per pool
struct AccumPool {
  long long total = 0;                 // batch x rows; 0: no pool
  int rows = 0, cols = 0;              // cols a multiple of 8 (vector path)
  int grad_dtype = kBF16;              // kBF16 or kF32
  unsigned long long* next = nullptr;  // rows handed out so far; zero before the pool's first user
  float* l1 = nullptr;                 // [batch][rows]
  float* sq = nullptr;                 // [batch][rows]
  float* scale = nullptr;              // lazy decay factors [batch][rows], or null
  float* M[kPoolMax];
  const void* G[kPoolMax];
};
// The rest of a pool: every row the counter has not handed out yet.
cudaError_t launch_accum_pool(const AccumPool& p, cudaStream_t s);

// Step a7 of shape groups whose update is deferred (their O and selected
// indices stay in the workspace) as one pool of rows, one segment per group,
// handed out by a device counter: to the streaming warps of the GEMM launches
// that run meanwhile (GemmDesc::spool), then to launch_scatter_pool for what is
// left.  Every row is written exactly once, with the arithmetic of the scatter
// kernel (vector path: cols a multiple of 8).
constexpr int kScatterSegMax = 2;  // deferred groups per pool
struct ScatterSeg {
  long long start = 0;               // the segment's first row of the pool
  int rows = 0, cols = 0, k = 0, batch = 0;
  int param_dtype = kBF16;           // kF32 or kBF16
  bool o_bf16 = false;               // O holds bf16 (else fp16)
  const int32_t* idx = nullptr;      // [batch][k]
  const __half* O = nullptr; long long o_bstride = 0; int ld_o = 0;   // [batch][k][ld_o]
  float lr = 0.f;
  const float* row_factor = nullptr; // [batch][k]: row i's lr is lr * row_factor[b][i] (null: lr)
  void* W[kPoolMax];
};
struct ScatterPool {
  long long total = 0;                 // rows over all segments; 0: no pool
  int nseg = 0;
  unsigned long long* next = nullptr;  // rows handed out so far; zero before the pool's first user
  unsigned* status = nullptr;          // device status word (kDevCheck on a bad index)
  ScatterSeg seg[kScatterSegMax];
};
cudaError_t launch_scatter_pool(const ScatterPool& p, cudaStream_t s);

// a1: top-k rows by l1 (ties to the lower index), indices ascending, and
// fro2 = sum of sq over the selected rows.
struct TopkArgs {
  int rows, k, batch;
  const float* l1;   // [batch][rows]
  const float* sq;   // [batch][rows]
  int32_t* idx;      // [batch][k]
  float* fro2;       // [batch] (may be null)
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t s);

// a2: gather + normalise (+ optional decay of the source rows) into fp16,
// rows-major [k][ld_rows] and, if out_cols is set, also columns-major
// [m][ld_cols] (the standard-NS comparison path; the Gram path reads the
// other orientation through transposed GEMM operands).
struct GatherArgs {
  int n;                           // rows of each source matrix (bounds check of idx)
  int k, m, batch;                 // batch <= kMaxBatchPerLaunch when src_f32
  bool src_f32;                    // true: rows of fp32 M picked by idx; false: 16-bit X
  bool bf16;                       // 16-bit type of X and of the outputs: bf16 (else fp16)
  float* M[kMaxBatchPerLaunch];    // src_f32: momentum pointers
  const int32_t* idx;              // src_f32: [batch][k]
  const __half* X;                 // !src_f32: [batch][k][m] contiguous
  const float* fro2;               // [batch][fro2_parts]
  int fro2_parts;
  float eps;
  float mu;                        // decay applied to the source rows (src_f32)
  bool decay;
  float* scale_out = nullptr;      // lazy decay: scale_out[b][row] = mu for the selected rows
  unsigned* status;                // device status word (kDevCheck on a bad index)
  __half* out_rows; long long rows_bstride; int ld_rows;   // [k][ld_rows]
  __half* out_cols; long long cols_bstride; int ld_cols;   // [m][ld_cols], or null: rows only
};
cudaError_t launch_gather(const GatherArgs& a, bool vec, cudaStream_t s);

// Lazy decay made explicit: M[b][r] <- fp32(scale[b][r] M[b][r]) where the
// factor is not 1, then the factor is reset to 1.
struct FlushArgs {
  int rows, cols, batch;             // batch <= kMaxBatchPerLaunch
  float* M[kMaxBatchPerLaunch];
  float* scale;                      // [batch][rows]
};
cudaError_t launch_flush_scale(const FlushArgs& a, cudaStream_t s);

// Sum of squares of fp16 X [batch][n] into parts [batch][parts].
cudaError_t launch_sumsq_f16(const __half* X, long long n, int batch, float* parts,
                             int nparts, bool bf16, cudaStream_t s);

// a7: W[S_i] <- round(W[S_i] - lr O[i]) for the selected rows.
struct ScatterArgs {
  int rows, cols, k, batch;        // batch <= kMaxBatchPerLaunch
  int param_dtype;                 // kF32 or kBF16
  void* W[kMaxBatchPerLaunch];
  const int32_t* idx;              // [batch][k]
  const __half* O; long long o_bstride; int ld_o;   // [k][ld_o]
  float lr;
  bool o_bf16;                     // O holds bf16 (else fp16)
  unsigned* status;                // device status word (kDevCheck on a bad index)
  const float* row_factor = nullptr;  // [batch][k]: row i's lr is lr * row_factor[b][i] (null: lr)
};
cudaError_t launch_scatter(const ScatterArgs& a, bool vec, cudaStream_t s);

// Per-neuron normalisation of the orthogonalised rows (the NorMuon reading):
// per selected row i of matrix b, with q_i = sum_j O_ij^2,
//   v[b][S_i] <- beta2 v[b][S_i] + (1 - beta2) q_i / m,
//   d[b][i] = 1 / (sqrt(v[b][S_i]) + eps),  rowc[b][i] = d^2 q_i.
struct NormRowsArgs {
  int rows, k, m, batch;
  const int32_t* idx;              // [batch][k]
  const __half* O; long long o_bstride; int ld_o;   // [batch][k][ld_o]
  bool o_bf16;
  float* v;                        // [batch][rows] fp32 state
  float beta2, eps;
  float* d;                        // [batch][k]
  float* rowc;                     // [batch][k]
  unsigned* status;
};
cudaError_t launch_normuon_rows(const NormRowsArgs& a, bool vec, cudaStream_t s);
// Per matrix: F^2 = sum_i rowc[b][i] (fixed order), g = rms sqrt(k m) / F
// (0 when F = 0), then d[b][i] <- g d[b][i].
struct NormScaleArgs {
  int k, m, batch;
  const float* rowc;
  float* d;
  float rms;
};
cudaError_t launch_normuon_scale(const NormScaleArgs& a, cudaStream_t s);

// ---------------------------------------------------------------------------
// Tensor-core GEMM (gemm_tcgen05.cu): D = A B^T with A [batch][M][K] and
// B [batch][N][K] fp16 (K contiguous), fp32 accumulation in TMEM, and the
// epilogue  v = alpha D + beta C + gamma I  written as fp16.
// ---------------------------------------------------------------------------
enum GemmMode : int {
  kRect = 0,      // every tile; write `out` (normal) and/or `outT` (transposed)
  kSymLower = 1,  // M == N, lower-triangle tiles only; `out` gets the tile and its mirror
                  // (with out_half, the mirror on the diagonal super-tiles only)
};

struct GemmDesc {
  const __half* A; long long a_bstride; int lda;
  const __half* B; long long b_bstride; int ldb;
  int M, N, K, batch;
  int mode;
  float alpha, beta, gamma;
  const __half* C; long long c_bstride; int ldc;     // may be null (beta ignored)
  __half* out; long long out_bstride; int ld_out;    // may be null in kRect
  __half* outT; long long outT_bstride; int ld_outT; // may be null
  // Visit the batch from the last matrix to the first.  Consecutive launches
  // of a chain alternate the order, so each starts on the matrices the
  // previous one wrote last (still in L2).
  bool reverse = false;
  int elem = kF16;  // operand / output element type: kF16 or kBF16 (16-bit storage either way)
  // Half-stored symmetric matrices (s x s): only the 256 x 256 blocks below the
  // diagonal and the full diagonal blocks are valid.  a_half / b_half: the
  // operand is one (M == K / N == K); out_half (kSymLower): write the result
  // as one (no mirror outside the diagonal super-tiles).
  bool a_half = false, b_half = false, out_half = false;
  // The operand is given as its transpose: A stored [batch][K][M] (lda >= M),
  // B stored [batch][K][N] (ldb >= N); read as MN-major tiles.
  bool a_tr = false, b_tr = false;
  // Optional: rows of another shape group's step a0 for the launch's
  // streaming warps to take while the tensor cores work (null: none), and
  // rows of deferred step a7 updates, taken once `pool` is exhausted.
  const AccumPool* pool = nullptr;
  const ScatterPool* spool = nullptr;
};

// Host-side checks of a descriptor (alignment and pitch rules of the TMA
// tensor maps); returns false with a message if the GEMM cannot be launched.
bool gemm_check(const GemmDesc& g, const char** why);
cudaError_t launch_gemm(const GemmDesc& g, unsigned* dev_status, cudaStream_t s);

// One thread waits on an mbarrier with the GEMM's bounded wait and the given
// limit; without `arrive` nothing completes the barrier and the wait runs out
// (kDevTimeout in *status).  A diagnostic of the timeout path.
cudaError_t launch_wait_probe(bool arrive, unsigned long long limit_ns, unsigned* status, cudaStream_t s);

// Status word address on the current device (set up by the API unit).
unsigned* device_status_ptr();

// Sets the message dion3_last_error() returns on this host thread.
void set_last_error_message(const char* msg);

}  // namespace dion3
