// C ABI of the Dion3 step (include/dion3.h): argument validation, workspace
// planning, and the launch schedule of steps (a)-(c) on one stream.
//
// Method source: "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of the
// paper): first-level paragraph (Gram Newton-Schulz with a restart at
// iteration 3, float16) and third-level paragraph (l1 selection of
// k = ceil(f n) rows, update of those rows only, lr ~ 1/sqrt(f), decay of the
// selected momentum rows by mu).  Megabatching (fourth-level paragraph) becomes
// shape-grouped batched launches on one GPU.
#include "../../include/dion3.h"
#include "internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

namespace dion3 {

__device__ unsigned g_device_status = 0u;

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("DION3_PDL");
    return v == nullptr || atoi(v) != 0;
  }();
  return on;
}

unsigned* device_status_ptr() {
  static std::mutex mu;
  static std::vector<unsigned*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, nullptr);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned*>(p);
  }
  return cache[dev];
}

namespace {

thread_local std::string t_last_error;

dion3_status fail(dion3_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
dion3_status fail(dion3_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

dion3_status ok() {
  t_last_error.clear();
  return DION3_OK;
}

// ---------------------------------------------------------------------------
// Optional launch trace: when enabled, every launch of a memory-bound kernel,
// and every chain of GEMM launches of one Newton-Schulz run, is bracketed by
// two CUDA events on its stream and recorded with its algorithmic work (useful
// FLOPs for the GEMM, bytes for the memory-bound kernels) and launch count.
// Events between the GEMMs of a chain would keep each GEMM from overlapping
// its set-up with the end of the previous one (programmatic dependent
// launch), so a chain gets one pair; DION3_TRACE_DETAIL=1|2 records every
// GEMM launch on its own instead, labelled by role.
// ---------------------------------------------------------------------------
struct TraceRec {
  std::string name;
  cudaEvent_t a, b;
  double flops, bytes;
  int launches;
};
std::mutex g_trace_mu;
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

void trace_clear_locked() {
  for (auto& r : g_trace) {
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  g_trace.clear();
}

int trace_detail() {
  static const int detail = [] {
    const char* v = getenv("DION3_TRACE_DETAIL");
    return v != nullptr ? atoi(v) : 0;
  }();
  return detail;
}

// The open chain of this host thread (launches of kernel `name` on stream s).
struct TraceSpan {
  std::string name;
  cudaStream_t s = nullptr;
  cudaEvent_t a = nullptr;
  double flops = 0.0, bytes = 0.0;
  int launches = 0;
};
thread_local TraceSpan* t_span = nullptr;

// Opens a chain for the launches of `name` on `s` made while it lives (if the
// trace is on, per-launch detail is off and no chain is open yet).
class TraceChain {
 public:
  TraceChain(const char* name, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_trace_mu);
    if (!g_trace_on || trace_detail() > 0 || t_span != nullptr) return;
    span_.name = name;
    span_.s = s;
    span_.a = pooled_event();
    if (span_.a == nullptr) return;
    cudaEventRecord(span_.a, s);
    open_ = true;
    t_span = &span_;
  }
  ~TraceChain() {
    if (!open_) return;
    t_span = nullptr;
    std::lock_guard<std::mutex> lock(g_trace_mu);
    cudaEvent_t b = (g_trace_on && span_.launches > 0) ? pooled_event() : nullptr;
    if (b == nullptr) {
      g_event_pool.push_back(span_.a);
      return;
    }
    cudaEventRecord(b, span_.s);
    g_trace.push_back({span_.name, span_.a, b, span_.flops, span_.bytes, span_.launches});
  }
  TraceChain(const TraceChain&) = delete;
  TraceChain& operator=(const TraceChain&) = delete;

 private:
  TraceSpan span_;
  bool open_ = false;
};

template <class Launch>
cudaError_t traced(const std::string& name, double flops, double bytes, cudaStream_t s, Launch&& launch) {
  std::unique_lock<std::mutex> lock(g_trace_mu);
  if (!g_trace_on) {
    lock.unlock();
    return launch();
  }
  if (t_span != nullptr && t_span->name == name && t_span->s == s) {
    t_span->flops += flops;
    t_span->bytes += bytes;
    ++t_span->launches;
    lock.unlock();
    return launch();
  }
  cudaEvent_t a = pooled_event(), b = pooled_event();
  if (a == nullptr || b == nullptr) return cudaErrorMemoryAllocation;
  cudaEventRecord(a, s);
  const cudaError_t e = launch();
  cudaEventRecord(b, s);
  g_trace.push_back({name, a, b, flops, bytes, 1});
  return e;
}

inline long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dion3_status cuda_fail(cudaError_t e, const char* what) {
  return fail(DION3_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Host-side fault injection for tests of error propagation: DION3_INJECT=
// launch_fail makes the first launch of a call report a CUDA error without
// launching anything.
bool inject_launch_fail() {
  const char* v = getenv("DION3_INJECT");
  return v != nullptr && strcmp(v, "launch_fail") == 0;
}

dion3_status check_hparams(const dion3_hparams* hp, bool need_step_fields) {
  if (hp == nullptr) return fail(DION3_ERR_INVALID_ARG, "hparams is NULL");
  if (hp->ns_steps < 1 || hp->ns_steps > 64) return fail(DION3_ERR_INVALID_ARG, "ns_steps must lie in [1, 64]");
  if (hp->restart_iter != 0 && (hp->restart_iter < 2 || hp->restart_iter > hp->ns_steps))
    return fail(DION3_ERR_INVALID_ARG, "restart_iter must be 0 or lie in [2, ns_steps]");
  if (!std::isfinite(hp->a) || !std::isfinite(hp->b) || !std::isfinite(hp->c))
    return fail(DION3_ERR_INVALID_ARG, "NS coefficients must be finite");
  if (!(hp->eps >= 0.0f) || !std::isfinite(hp->eps)) return fail(DION3_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (hp->ns_dtype != DION3_F16 && hp->ns_dtype != DION3_BF16)
    return fail(DION3_ERR_UNSUPPORTED, "ns_dtype must be DION3_F16 or DION3_BF16");
  if (need_step_fields) {
    if (!(hp->f > 0.0f && hp->f <= 1.0f)) return fail(DION3_ERR_INVALID_ARG, "f must lie in (0, 1]");
    if (!std::isfinite(hp->mu)) return fail(DION3_ERR_INVALID_ARG, "mu must be finite");
    if (!std::isfinite(hp->lr)) return fail(DION3_ERR_INVALID_ARG, "lr must be finite");
  }
  return DION3_OK;
}

int32_t num_selected(float f, int32_t rows) {
  if (!(f > 0.0f && f <= 1.0f) || rows < 1) return 0;
  const double k = std::ceil(static_cast<double>(f) * static_cast<double>(rows));
  if (k < 1.0) return 1;
  if (k > rows) return rows;
  return static_cast<int32_t>(k);
}

// ---------------------------------------------------------------------------
// Workspace planning
// ---------------------------------------------------------------------------
struct Carver {
  char* base;  // may be null (size query)
  size_t off = 0;
  template <class T>
  T* take(long long count) {
    off = static_cast<size_t>(round_up(static_cast<long long>(off), 256));
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += static_cast<size_t>(count) * sizeof(T);
    return p;
  }
};

// Gram-NS buffers for `batch` k x m problems.  Y is the s x L operand (s =
// min(k, m)); Yt0/Yt1 hold L x s transposes; S[0..3] are s x s buffers.
// The Gram-NS workspace of one shape group.  The normalised rows are kept in
// one orientation only, X itself ([batch][k][mp], mp = round_up(m, 8)): when
// k <= m (wide) that is Y, when k > m it is Y^T.  Products that need the other
// orientation read it through the GEMM's transposed-operand tiles.
struct NsPlan {
  int k, m, batch, s, L, sp, mp;
  bool wide;      // k <= m: Y = X (s x L); else Y = X^T and X is Y^T (L x s)
  __half* X[2];   // ping-pong for the restart (Y <- Q Y reads one, writes the other)
  __half* S[4];   // s x s matrices, half-stored symmetric
  long long x_bs, s_bs;
};

void plan_ns(Carver& c, int k, int m, int batch, NsPlan& p) {
  p.k = k;
  p.m = m;
  p.batch = batch;
  p.wide = k <= m;
  p.s = p.wide ? k : m;
  p.L = p.wide ? m : k;
  p.sp = static_cast<int>(round_up(p.s, 8));
  p.mp = static_cast<int>(round_up(m, 8));
  p.x_bs = static_cast<long long>(k) * p.mp;
  p.s_bs = static_cast<long long>(p.s) * p.sp;
  p.X[0] = c.take<__half>(p.x_bs * batch);
  p.X[1] = c.take<__half>(p.x_bs * batch);
  for (int i = 0; i < 4; ++i) p.S[i] = c.take<__half>(p.s_bs * batch);
}

// Where the gather kernel writes the normalised rows: X[0], rows only.
void gather_targets(const NsPlan& p, GatherArgs& g) {
  g.out_rows = p.X[0];
  g.rows_bstride = p.x_bs;
  g.ld_rows = p.mp;
  g.out_cols = nullptr;
}

// Traced launch helpers: the algorithmic work of one launch.
// With DION3_TRACE_DETAIL=1 in the environment the GEMM launches are
// labelled by role (SYRK, symmetric square product, rectangular) instead of
// under the kernel's name.
cudaError_t traced_gemm(const GemmDesc& g, unsigned* st, cudaStream_t s) {
  const double flops = g.mode == kSymLower ? static_cast<double>(g.M) * g.M * g.K * g.batch
                                           : 2.0 * g.M * g.N * g.K * g.batch;
  const double bytes = 2.0 * g.batch * (static_cast<double>(g.M) * g.K + static_cast<double>(g.N) * g.K);
  const int detail = trace_detail();
  std::string name = "gemm_tcgen05";
  if (detail >= 1) name = g.mode == kRect ? "gemm:rect" : (g.K == g.M ? "gemm:sym_square" : "gemm:syrk");
  if (detail >= 2) name += ":" + std::to_string(g.mode == kRect ? std::min(g.M, g.N) : g.M);
  return traced(name, flops, bytes, s, [&] { return launch_gemm(g, st, s); });
}
cudaError_t traced_accum(const AccumArgs& a, bool vec, cudaStream_t s) {
  const double gb = a.G[0] == nullptr ? 0.0 : (a.grad_dtype == kBF16 ? 2.0 : 4.0);
  const double wb = a.G[0] == nullptr ? 0.0 : 4.0;
  const double bytes = static_cast<double>(a.batch) * a.rows * (a.cols * (4.0 + gb + wb) + 8.0);
  return traced("accum_rownorm", 0.0, bytes, s, [&] { return launch_accum_rownorm(a, vec, s); });
}
// The rest of a pooled accumulation.  Its trace entry carries the algorithmic
// bytes of the whole group's accumulation, part of which the streaming warps of
// the GEMM launches before it have moved.
cudaError_t traced_accum_pool(const AccumPool& p, cudaStream_t s) {
  const double gb = p.grad_dtype == kBF16 ? 2.0 : 4.0;
  const double bytes = static_cast<double>(p.total) * (p.cols * (4.0 + gb + 4.0) + 8.0);
  return traced("accum_pool", 0.0, bytes, s, [&] { return launch_accum_pool(p, s); });
}
cudaError_t traced_topk(const TopkArgs& t, cudaStream_t s) {
  const double bytes = static_cast<double>(t.batch) * (t.rows * 8.0 + t.k * 4.0 + 4.0);
  return traced("topk_select", 0.0, bytes, s, [&] { return launch_topk(t, s); });
}
cudaError_t traced_gather(const GatherArgs& g, bool vec, cudaStream_t s) {
  const double per = g.src_f32 ? (4.0 + (g.decay ? 4.0 : 0.0)) : 2.0;
  const double bytes = static_cast<double>(g.batch) * g.k * g.m * (per + (g.out_cols != nullptr ? 4.0 : 2.0));
  return traced("gather_normalize", 0.0, bytes, s, [&] { return launch_gather(g, vec, s); });
}
cudaError_t traced_sumsq(const __half* X, long long n, int batch, float* parts, int nparts, bool bf16,
                         cudaStream_t s) {
  return traced("sumsq_f16", 0.0, 2.0 * n * batch, s,
                [&] { return launch_sumsq_f16(X, n, batch, parts, nparts, bf16, s); });
}
cudaError_t traced_scatter(const ScatterArgs& a, bool vec, cudaStream_t s) {
  const double pb = a.param_dtype == kBF16 ? 2.0 : 4.0;
  const double bytes = static_cast<double>(a.batch) * a.k * a.cols * (2.0 + 2.0 * pb);
  return traced("scatter_update", 0.0, bytes, s, [&] { return launch_scatter(a, vec, s); });
}
// The rest of a scatter pool.  Its trace entry carries the algorithmic bytes
// of every deferred update in the pool, part of which the streaming warps of
// the GEMM launches before it have written.
cudaError_t traced_scatter_pool(const ScatterPool& p, cudaStream_t s) {
  double bytes = 0.0;
  for (int i = 0; i < p.nseg; ++i) {
    const ScatterSeg& g = p.seg[i];
    const double pb = g.param_dtype == kBF16 ? 2.0 : 4.0;
    bytes += static_cast<double>(g.batch) * g.k * g.cols * (2.0 + 2.0 * pb);
  }
  return traced("scatter_pool", 0.0, bytes, s, [&] { return launch_scatter_pool(p, s); });
}
cudaError_t traced_normuon_rows(const NormRowsArgs& a, bool vec, cudaStream_t s) {
  // O read once; per row: the index, v read and written, d and rowc written.
  const double bytes = static_cast<double>(a.batch) * a.k * (2.0 * a.m + 4.0 + 8.0 + 8.0);
  return traced("normuon_rows", 0.0, bytes, s, [&] { return launch_normuon_rows(a, vec, s); });
}
cudaError_t traced_normuon_scale(const NormScaleArgs& a, cudaStream_t s) {
  const double bytes = static_cast<double>(a.batch) * a.k * 12.0;
  return traced("normuon_scale", 0.0, bytes, s, [&] { return launch_normuon_scale(a, s); });
}

// Useful FLOPs of the schedule run_gram_ns() launches (triangle = half).
double schedule_flops(int k, int m, const dion3_hparams& hp) {
  const double s = std::min(k, m), L = std::max(k, m);
  const double syrk = s * s * L, sym = s * s * s, rect = 2.0 * s * s * L;
  double f = syrk;
  bool q_identity = true;
  const int T = hp.ns_steps, rs = hp.restart_iter;
  for (int t = 1; t <= T; ++t) {
    if (rs > 1 && t == rs) {
      f += rect + syrk;
      q_identity = true;
    }
    f += sym;  // Z
    if (!q_identity) f += sym;
    q_identity = false;
    if (t < T && t + 1 != rs) f += 2.0 * sym;
  }
  return f + rect;
}

// ---------------------------------------------------------------------------
// Gram Newton-Schulz schedule (first-level paragraph of the summary page):
//   R = Y Y^T;  for t = 1..T:
//     [t == restart] Y <- Q Y (written as Y^T Q and its transpose), R = Y Y^T, Q <- I
//     Z = aI + bR + cR^2;  Q <- Z (Q = I) or Q <- Z Q;
//     [t < T and t + 1 != restart] R <- Z (R Z)
//   O = Q Y  (written in the k x m orientation of X).
// ---------------------------------------------------------------------------
struct NsOut {
  __half* O;
  long long o_bs;
  int ld_o;
};

dion3_status run_gram_ns(const NsPlan& p, const dion3_hparams& hp, const NsOut& out, unsigned* st,
                         cudaStream_t stream, bool dense = false, const AccumPool* pool = nullptr,
                         const ScatterPool* spool = nullptr) {
  TraceChain chain("gemm_tcgen05", stream);
  // Symmetric product of two s x s matrices (or, with xi >= 0, the SYRK
  // R = Y Y^T from X[xi]: Y itself when wide, given as its transpose X = Y^T
  // otherwise).
  auto sym = [&](const __half* A, const __half* B, __half* D, const __half* C, float alpha, float beta,
                 float gamma, int xi = -1) -> GemmDesc {
    GemmDesc g{};
    const bool from_y = xi >= 0;
    if (from_y) {
      g.A = g.B = p.X[xi];
      g.a_bstride = g.b_bstride = p.x_bs;
      g.lda = g.ldb = p.mp;
      g.a_tr = g.b_tr = !p.wide;
    } else {
      g.A = A; g.a_bstride = p.s_bs; g.lda = p.sp;
      g.B = B; g.b_bstride = p.s_bs; g.ldb = p.sp;
    }
    g.M = p.s; g.N = p.s; g.K = from_y ? p.L : p.s; g.batch = p.batch;
    // dense: every tile of the product (the comparison path without the
    // symmetric savings); otherwise lower-triangle tiles.  Every s x s matrix
    // of the chain is then half-stored (the 256 x 256 blocks below the block
    // diagonal and the full diagonal blocks): written without the mirror
    // outside the diagonal blocks, and read back with the K ranges above the
    // diagonal taken from the transpose.
    g.mode = dense ? kRect : kSymLower;
    g.out_half = !dense;
    g.a_half = g.b_half = !dense && !from_y;
    g.alpha = alpha; g.beta = beta; g.gamma = gamma;
    g.C = C; g.c_bstride = p.s_bs; g.ldc = p.sp;
    g.out = D; g.out_bstride = p.s_bs; g.ld_out = p.sp;
    return g;
  };
  bool reverse = false;  // serpentine batch order across the chain
  auto launch = [&](const GemmDesc& g0) -> dion3_status {
    GemmDesc g = g0;
    g.elem = hp.ns_dtype == DION3_BF16 ? kBF16 : kF16;
    // Every launch of the run lends its streaming warps to the pools (limiting
    // that to the launches with a long K, whose epilogue warps are idle more
    // of the time, measured no better).
    g.pool = pool;
    g.spool = spool;
    g.reverse = reverse;
    reverse = !reverse;
    const char* why = nullptr;
    if (!gemm_check(g, &why)) return fail(DION3_ERR_INVALID_ARG, "internal GEMM rejected: %s", why);
    const cudaError_t e = traced_gemm(g, st, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tcgen05 GEMM launch");
    return DION3_OK;
  };
  dion3_status rc;

  // s x s buffer roles: indices into p.S.
  int R = 0, Z = -1, Q = -1;
  auto free_buf = [&](int a, int b, int c) {
    for (int i = 0; i < 4; ++i)
      if (i != a && i != b && i != c) return i;
    return -1;
  };
  int xcur = 0;  // X[xcur] holds the current Y (wide) or Y^T
  // The product with Q in X's own orientation, written as is (no transposed
  // store): wide, D = Q Y (s x L) with A = Q half-stored and B = Y^T given as
  // its transpose, which is X[xi] itself; otherwise D = Y^T Q (L x s) with
  // A = X[xi] = Y^T and B = Q half-stored.
  auto rect_q = [&](int xi) -> GemmDesc {
    GemmDesc g{};
    if (p.wide) {
      g.A = p.S[Q]; g.a_bstride = p.s_bs; g.lda = p.sp;
      g.a_half = !dense;
      g.B = p.X[xi]; g.b_bstride = p.x_bs; g.ldb = p.mp;
      g.b_tr = true;
      g.M = p.s; g.N = p.L;
    } else {
      g.A = p.X[xi]; g.a_bstride = p.x_bs; g.lda = p.mp;
      g.B = p.S[Q]; g.b_bstride = p.s_bs; g.ldb = p.sp;
      g.b_half = !dense;
      g.M = p.L; g.N = p.s;
    }
    g.K = p.s; g.batch = p.batch;
    g.mode = kRect; g.alpha = 1.f;
    return g;
  };

  // R = Y Y^T
  if ((rc = launch(sym(nullptr, nullptr, p.S[R], nullptr, 1.f, 0.f, 0.f, xcur))) != DION3_OK) return rc;
  const int T = hp.ns_steps, rs = hp.restart_iter;
  for (int t = 1; t <= T; ++t) {
    if (rs > 1 && t == rs) {
      // Y <- Q Y, in X's orientation.
      GemmDesc g = rect_q(xcur);
      g.out = p.X[xcur ^ 1]; g.out_bstride = p.x_bs; g.ld_out = p.mp;
      if ((rc = launch(g)) != DION3_OK) return rc;
      xcur ^= 1;
      if ((rc = launch(sym(nullptr, nullptr, p.S[R], nullptr, 1.f, 0.f, 0.f, xcur))) != DION3_OK) return rc;
      Q = -1;
    }
    // Z = c R.R + b R + a I
    Z = free_buf(R, Q, -1);
    if ((rc = launch(sym(p.S[R], p.S[R], p.S[Z], p.S[R], hp.c, hp.b, hp.a))) != DION3_OK) return rc;
    if (Q < 0) {
      Q = Z;  // Q <- Z
    } else {
      const int nq = free_buf(R, Q, Z);
      if ((rc = launch(sym(p.S[Z], p.S[Q], p.S[nq], nullptr, 1.f, 0.f, 0.f))) != DION3_OK) return rc;
      Q = nq;
    }
    if (t < T && t + 1 != rs) {
      // R <- Z (R Z); Z may be the buffer Q now points at, which is only read.
      const int tm = free_buf(R, Q, Z);
      if ((rc = launch(sym(p.S[R], p.S[Z], p.S[tm], nullptr, 1.f, 0.f, 0.f))) != DION3_OK) return rc;
      if ((rc = launch(sym(p.S[Z], p.S[tm], p.S[R], nullptr, 1.f, 0.f, 0.f))) != DION3_OK) return rc;
    }
  }
  // O = Q Y, written in X's k x m orientation.
  GemmDesc g = rect_q(xcur);
  g.out = out.O; g.out_bstride = out.o_bs; g.ld_out = out.ld_o;
  return launch(g);
}

// ---------------------------------------------------------------------------
// Standard Newton-Schulz on the same kernels (the comparison path of the
// first-level paragraph of the summary page: the common implementation that
// iterates on X itself).  Per iteration on Y (s x L, s <= L):
//   A = Y Y^T;  B = c A.A + b A;  Y <- a Y + B Y
// with Y and Y^T ping-ponged so every operand is K-major; the last iteration
// writes O in X's orientation.
// ---------------------------------------------------------------------------
struct StdPlan {
  int k, m, batch, s, L, sp, Lp;
  bool wide;
  __half* Y[2];
  __half* Yt[2];
  __half* S[2];
  long long y_bs, yt_bs, s_bs;
};

void plan_std(Carver& c, int k, int m, int batch, StdPlan& p) {
  p.k = k;
  p.m = m;
  p.batch = batch;
  p.wide = k <= m;
  p.s = p.wide ? k : m;
  p.L = p.wide ? m : k;
  p.sp = static_cast<int>(round_up(p.s, 8));
  p.Lp = static_cast<int>(round_up(p.L, 8));
  p.y_bs = static_cast<long long>(p.s) * p.Lp;
  p.yt_bs = static_cast<long long>(p.L) * p.sp;
  p.s_bs = static_cast<long long>(p.s) * p.sp;
  for (int i = 0; i < 2; ++i) p.Y[i] = c.take<__half>(p.y_bs * batch);
  for (int i = 0; i < 2; ++i) p.Yt[i] = c.take<__half>(p.yt_bs * batch);
  for (int i = 0; i < 2; ++i) p.S[i] = c.take<__half>(p.s_bs * batch);
}

void gather_targets_std(const StdPlan& p, GatherArgs& g) {
  if (p.wide) {
    g.out_rows = p.Y[0];   g.rows_bstride = p.y_bs;  g.ld_rows = p.Lp;
    g.out_cols = p.Yt[0];  g.cols_bstride = p.yt_bs; g.ld_cols = p.sp;
  } else {
    g.out_rows = p.Yt[0];  g.rows_bstride = p.yt_bs; g.ld_rows = p.sp;
    g.out_cols = p.Y[0];   g.cols_bstride = p.y_bs;  g.ld_cols = p.Lp;
  }
}

dion3_status run_standard_ns(const StdPlan& p, const dion3_hparams& hp, const NsOut& out, unsigned* st,
                             cudaStream_t stream, bool dense) {
  TraceChain chain("gemm_tcgen05", stream);
  auto launch = [&](const GemmDesc& g0) -> dion3_status {
    GemmDesc g = g0;
    g.elem = hp.ns_dtype == DION3_BF16 ? kBF16 : kF16;
    const char* why = nullptr;
    if (!gemm_check(g, &why)) return fail(DION3_ERR_INVALID_ARG, "internal GEMM rejected: %s", why);
    const cudaError_t e = traced_gemm(g, st, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tcgen05 GEMM launch");
    return DION3_OK;
  };
  const int mode_sym = dense ? kRect : kSymLower;
  dion3_status rc;
  for (int t = 0; t < hp.ns_steps; ++t) {
    const int cur = t & 1, nxt = cur ^ 1;
    const bool last = t + 1 == hp.ns_steps;
    // A = Y Y^T
    GemmDesc g1{};
    g1.A = p.Y[cur]; g1.a_bstride = p.y_bs; g1.lda = p.Lp;
    g1.B = p.Y[cur]; g1.b_bstride = p.y_bs; g1.ldb = p.Lp;
    g1.M = p.s; g1.N = p.s; g1.K = p.L; g1.batch = p.batch;
    g1.mode = mode_sym; g1.alpha = 1.f;
    // The symmetric s x s matrices are half-stored, as in the Gram schedule.
    g1.out_half = !dense;
    g1.out = p.S[0]; g1.out_bstride = p.s_bs; g1.ld_out = p.sp;
    if ((rc = launch(g1)) != DION3_OK) return rc;
    // B = c A.A + b A
    GemmDesc g2{};
    g2.A = p.S[0]; g2.a_bstride = p.s_bs; g2.lda = p.sp;
    g2.B = p.S[0]; g2.b_bstride = p.s_bs; g2.ldb = p.sp;
    g2.M = p.s; g2.N = p.s; g2.K = p.s; g2.batch = p.batch;
    g2.mode = mode_sym; g2.alpha = hp.c; g2.beta = hp.b;
    g2.a_half = g2.b_half = g2.out_half = !dense;
    g2.C = p.S[0]; g2.c_bstride = p.s_bs; g2.ldc = p.sp;
    g2.out = p.S[1]; g2.out_bstride = p.s_bs; g2.ld_out = p.sp;
    if ((rc = launch(g2)) != DION3_OK) return rc;
    // Y <- a Y + B Y:  D = B (Y^T)^T, C = Y
    GemmDesc g3{};
    g3.A = p.S[1]; g3.a_bstride = p.s_bs; g3.lda = p.sp;
    g3.B = p.Yt[cur]; g3.b_bstride = p.yt_bs; g3.ldb = p.sp;
    g3.M = p.s; g3.N = p.L; g3.K = p.s; g3.batch = p.batch;
    g3.mode = kRect; g3.alpha = 1.f; g3.beta = hp.a;
    g3.a_half = !dense;
    g3.C = p.Y[cur]; g3.c_bstride = p.y_bs; g3.ldc = p.Lp;
    if (!last) {
      g3.out = p.Y[nxt]; g3.out_bstride = p.y_bs; g3.ld_out = p.Lp;
      g3.outT = p.Yt[nxt]; g3.outT_bstride = p.yt_bs; g3.ld_outT = p.sp;
    } else if (p.wide) {
      g3.out = out.O; g3.out_bstride = out.o_bs; g3.ld_out = out.ld_o;
    } else {
      g3.outT = out.O; g3.outT_bstride = out.o_bs; g3.ld_outT = out.ld_o;
    }
    if ((rc = launch(g3)) != DION3_OK) return rc;
  }
  return DION3_OK;
}

// Useful FLOPs of each variant (a computed triangle counts half; the dense
// variants compute every tile, so their products count in full).
double variant_flops(int variant, int k, int m, const dion3_hparams& hp) {
  const double s = std::min(k, m), L = std::max(k, m), T = hp.ns_steps;
  switch (variant) {
    case DION3_NS_GRAM: return schedule_flops(k, m, hp);
    case DION3_NS_GRAM_DENSE: {
      // every product of the Gram schedule in full: SYRK 2 s^2 L, square 2 s^3
      const double sym = schedule_flops(k, m, hp);
      const int restarts = (hp.restart_iter > 1) ? 1 : 0;
      const double syrk = s * s * L * (1 + restarts), rect = 2.0 * s * s * L * (1 + restarts);
      return 2.0 * (sym - syrk - rect) + 2.0 * syrk + rect;
    }
    case DION3_NS_STANDARD: return T * (3.0 * s * s * L + s * s * s);
    case DION3_NS_STANDARD_DENSE: return T * (4.0 * s * s * L + 2.0 * s * s * s);
    default: return -1.0;
  }
}

// Step workspace layout for one group.
struct GroupPlan {
  int n, m, batch, k;
  float* l1;
  float* sq;
  int32_t* idx;
  float* fro2;
  __half* O;
  long long o_bs;
  int ld_o;
  float* nm_d;     // per-neuron normalisation: row factors [batch][k]
  float* nm_rowc;  // and the rows' d^2 q [batch][k]
  unsigned long long* pool_next;  // row counter when this group's accumulation is pooled
  unsigned long long* spool_next; // row counter of the scatter pool riding on this group's launches
  NsPlan ns;
};

void plan_group(Carver& c, const dion3_group& g, float f, GroupPlan& gp) {
  gp.n = g.rows;
  gp.m = g.cols;
  gp.batch = g.batch;
  gp.k = num_selected(f, g.rows);
  gp.l1 = c.take<float>(static_cast<long long>(g.batch) * g.rows);
  gp.sq = c.take<float>(static_cast<long long>(g.batch) * g.rows);
  gp.idx = c.take<int32_t>(static_cast<long long>(g.batch) * gp.k);
  gp.fro2 = c.take<float>(g.batch);
  gp.ld_o = static_cast<int>(round_up(g.cols, 8));
  gp.o_bs = static_cast<long long>(gp.k) * gp.ld_o;
  gp.O = c.take<__half>(gp.o_bs * g.batch);
  gp.nm_d = c.take<float>(static_cast<long long>(g.batch) * gp.k);
  gp.nm_rowc = c.take<float>(static_cast<long long>(g.batch) * gp.k);
  gp.pool_next = c.take<unsigned long long>(1);
  gp.spool_next = c.take<unsigned long long>(1);
  plan_ns(c, gp.k, gp.m, gp.batch, gp.ns);
}

dion3_status check_group(const dion3_group& g, int gi) {
  if (g.rows < 1 || g.cols < 1 || g.batch < 1)
    return fail(DION3_ERR_INVALID_ARG, "group %d: rows, cols and batch must be >= 1", gi);
  if (g.batch > 65535) return fail(DION3_ERR_INVALID_ARG, "group %d: batch > 65535", gi);
  if (static_cast<long long>(g.rows) * g.cols > (1LL << 40))
    return fail(DION3_ERR_INVALID_ARG, "group %d: matrix too large", gi);
  if (g.param_dtype != DION3_F32 && g.param_dtype != DION3_BF16)
    return fail(DION3_ERR_INVALID_ARG, "group %d: param_dtype must be DION3_F32 or DION3_BF16", gi);
  if (g.grad_dtype != DION3_F32 && g.grad_dtype != DION3_BF16)
    return fail(DION3_ERR_INVALID_ARG, "group %d: grad_dtype must be DION3_F32 or DION3_BF16", gi);
  if (g.params == nullptr || g.grads == nullptr || g.momentum == nullptr)
    return fail(DION3_ERR_INVALID_ARG, "group %d: pointer arrays must not be NULL", gi);
  for (int b = 0; b < g.batch; ++b) {
    if (g.params[b] == nullptr || g.grads[b] == nullptr || g.momentum[b] == nullptr)
      return fail(DION3_ERR_INVALID_ARG, "group %d matrix %d: NULL tensor pointer", gi, b);
    if (!aligned16(g.params[b]) || !aligned16(g.grads[b]) || !aligned16(g.momentum[b]))
      return fail(DION3_ERR_INVALID_ARG, "group %d matrix %d: tensor pointers must be 16-byte aligned", gi, b);
  }
  return DION3_OK;
}

dion3_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need > 0 && ws == nullptr) return fail(DION3_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (ws != nullptr && (reinterpret_cast<uintptr_t>(ws) & 255u))
    return fail(DION3_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < need) return fail(DION3_ERR_WORKSPACE, "workspace too small: %zu < %zu bytes", ws_bytes, need);
  return DION3_OK;
}

}  // namespace

void set_last_error_message(const char* msg) { t_last_error = msg != nullptr ? msg : ""; }

}  // namespace dion3

using namespace dion3;

extern "C" {

size_t dion3_abi_version(void) { return DION3_ABI_VERSION; }

const char* dion3_status_string(int status) {
  switch (status) {
    case DION3_OK: return "DION3_OK";
    case DION3_ERR_INVALID_ARG: return "DION3_ERR_INVALID_ARG";
    case DION3_ERR_UNSUPPORTED: return "DION3_ERR_UNSUPPORTED";
    case DION3_ERR_WORKSPACE: return "DION3_ERR_WORKSPACE";
    case DION3_ERR_CUDA: return "DION3_ERR_CUDA";
    case DION3_ERR_TIMEOUT: return "DION3_ERR_TIMEOUT";
    case DION3_ERR_DEVICE_CHECK: return "DION3_ERR_DEVICE_CHECK";
    default: return "unknown dion3 status";
  }
}

const char* dion3_last_error(void) { return t_last_error.c_str(); }

int32_t dion3_num_selected(float f, int32_t rows) { return dion3::num_selected(f, rows); }

double dion3_useful_flops(int32_t k, int32_t m, const dion3_hparams* hp) {
  if (k < 1 || m < 1 || check_hparams(hp, false) != DION3_OK) return -1.0;
  return schedule_flops(k, m, *hp);
}

dion3_status dion3_select_workspace_size(int32_t rows, int32_t cols, int32_t batch, int32_t k, size_t* bytes) {
  if (bytes == nullptr) return fail(DION3_ERR_INVALID_ARG, "bytes is NULL");
  if (rows < 1 || cols < 1 || batch < 1 || k < 1 || k > rows)
    return fail(DION3_ERR_INVALID_ARG, "need rows, cols, batch >= 1 and 1 <= k <= rows");
  Carver c{nullptr};
  c.take<float>(static_cast<long long>(batch) * rows);
  c.take<float>(static_cast<long long>(batch) * rows);
  *bytes = round_up(static_cast<long long>(c.off), 256);
  return ok();
}

dion3_status dion3_select_rows(int32_t rows, int32_t cols, int32_t batch, float* const* momentum,
                               const void* const* grads, int32_t grad_dtype, int32_t k, int32_t* idx_out,
                               float* fro2_out, void* ws, size_t ws_bytes, dion3_stream_t stream) {
  size_t need = 0;
  dion3_status rc = dion3_select_workspace_size(rows, cols, batch, k, &need);
  if (rc != DION3_OK) return rc;
  if (batch > 65535) return fail(DION3_ERR_INVALID_ARG, "batch > 65535");
  if (momentum == nullptr || idx_out == nullptr) return fail(DION3_ERR_INVALID_ARG, "momentum and idx_out must not be NULL");
  if (grads != nullptr && grad_dtype != DION3_F32 && grad_dtype != DION3_BF16)
    return fail(DION3_ERR_INVALID_ARG, "grad_dtype must be DION3_F32 or DION3_BF16");
  for (int b = 0; b < batch; ++b) {
    if (momentum[b] == nullptr || !aligned16(momentum[b]))
      return fail(DION3_ERR_INVALID_ARG, "momentum[%d] NULL or not 16-byte aligned", b);
    if (grads != nullptr && (grads[b] == nullptr || !aligned16(grads[b])))
      return fail(DION3_ERR_INVALID_ARG, "grads[%d] NULL or not 16-byte aligned", b);
  }
  if ((rc = check_ws(ws, ws_bytes, need)) != DION3_OK) return rc;
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carver c{static_cast<char*>(ws)};
  float* l1 = c.take<float>(static_cast<long long>(batch) * rows);
  float* sq = c.take<float>(static_cast<long long>(batch) * rows);
  const bool vec = cols % 8 == 0;
  for (int b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
    const int nb = std::min(kMaxBatchPerLaunch, batch - b0);
    AccumArgs a{};
    a.rows = rows; a.cols = cols; a.batch = nb; a.grad_dtype = grad_dtype;
    for (int i = 0; i < nb; ++i) {
      a.M[i] = momentum[b0 + i];
      a.G[i] = grads ? grads[b0 + i] : nullptr;
    }
    a.l1 = l1 + static_cast<size_t>(b0) * rows;
    a.sq = sq + static_cast<size_t>(b0) * rows;
    const cudaError_t e = traced_accum(a, vec, s);
    if (e != cudaSuccess) return cuda_fail(e, "accum_rownorm launch");
  }
  TopkArgs t{};
  t.rows = rows; t.k = k; t.batch = batch; t.l1 = l1; t.sq = sq; t.idx = idx_out; t.fro2 = fro2_out;
  const cudaError_t e = traced_topk(t, s);
  if (e != cudaSuccess) return cuda_fail(e, "topk launch");
  return ok();
}

dion3_status dion3_gram_ns_workspace_size(int32_t k, int32_t m, int32_t batch, const dion3_hparams* hp,
                                          size_t* bytes) {
  if (bytes == nullptr) return fail(DION3_ERR_INVALID_ARG, "bytes is NULL");
  if (k < 1 || m < 1 || batch < 1 || batch > 65535)
    return fail(DION3_ERR_INVALID_ARG, "need k, m >= 1 and 1 <= batch <= 65535");
  dion3_status rc = check_hparams(hp, false);
  if (rc != DION3_OK) return rc;
  Carver c{nullptr};
  NsPlan p;
  plan_ns(c, k, m, batch, p);
  c.take<float>(static_cast<long long>(batch) * 64);
  *bytes = round_up(static_cast<long long>(c.off), 256);
  return ok();
}

dion3_status dion3_gram_ns_batched(int32_t k, int32_t m, int32_t batch, const void* X, void* O,
                                   const dion3_hparams* hp, void* ws, size_t ws_bytes, dion3_stream_t stream) {
  size_t need = 0;
  dion3_status rc = dion3_gram_ns_workspace_size(k, m, batch, hp, &need);
  if (rc != DION3_OK) return rc;
  if (X == nullptr || O == nullptr) return fail(DION3_ERR_INVALID_ARG, "X and O must not be NULL");
  if (!aligned16(X) || !aligned16(O)) return fail(DION3_ERR_INVALID_ARG, "X and O must be 16-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, need)) != DION3_OK) return rc;
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carver c{static_cast<char*>(ws)};
  NsPlan p;
  plan_ns(c, k, m, batch, p);
  constexpr int kParts = 64;
  float* parts = c.take<float>(static_cast<long long>(batch) * kParts);
  const long long n = static_cast<long long>(k) * m;
  cudaError_t e = traced_sumsq(static_cast<const __half*>(X), n, batch, parts, kParts, hp->ns_dtype == DION3_BF16, s);
  if (e != cudaSuccess) return cuda_fail(e, "sumsq launch");
  GatherArgs g{};
  g.k = k; g.m = m; g.batch = batch; g.src_f32 = false;
  g.X = static_cast<const __half*>(X);
  g.fro2 = parts; g.fro2_parts = kParts; g.eps = hp->eps; g.decay = false;
  g.bf16 = hp->ns_dtype == DION3_BF16;
  g.n = k; g.status = st;
  gather_targets(p, g);
  e = traced_gather(g, m % 4 == 0, s);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  NsOut out{static_cast<__half*>(O), static_cast<long long>(k) * m, m};
  if ((rc = run_gram_ns(p, *hp, out, st, s)) != DION3_OK) return rc;
  return ok();
}

double dion3_ns_useful_flops(int32_t variant, int32_t k, int32_t m, const dion3_hparams* hp) {
  if (k < 1 || m < 1 || check_hparams(hp, false) != DION3_OK) return -1.0;
  return variant_flops(variant, k, m, *hp);
}

dion3_status dion3_ns_workspace_size(int32_t variant, int32_t k, int32_t m, int32_t batch,
                                     const dion3_hparams* hp, size_t* bytes) {
  if (variant == DION3_NS_GRAM || variant == DION3_NS_GRAM_DENSE)
    return dion3_gram_ns_workspace_size(k, m, batch, hp, bytes);
  if (variant != DION3_NS_STANDARD && variant != DION3_NS_STANDARD_DENSE)
    return fail(DION3_ERR_INVALID_ARG, "unknown Newton-Schulz variant %d", variant);
  if (bytes == nullptr) return fail(DION3_ERR_INVALID_ARG, "bytes is NULL");
  if (k < 1 || m < 1 || batch < 1 || batch > 65535)
    return fail(DION3_ERR_INVALID_ARG, "need k, m >= 1 and 1 <= batch <= 65535");
  dion3_status rc = check_hparams(hp, false);
  if (rc != DION3_OK) return rc;
  Carver c{nullptr};
  StdPlan p;
  plan_std(c, k, m, batch, p);
  c.take<float>(static_cast<long long>(batch) * 64);
  *bytes = round_up(static_cast<long long>(c.off), 256);
  return ok();
}

dion3_status dion3_ns_batched(int32_t variant, int32_t k, int32_t m, int32_t batch, const void* X, void* O,
                              const dion3_hparams* hp, void* ws, size_t ws_bytes, dion3_stream_t stream) {
  size_t need = 0;
  dion3_status rc = dion3_ns_workspace_size(variant, k, m, batch, hp, &need);
  if (rc != DION3_OK) return rc;
  if (X == nullptr || O == nullptr) return fail(DION3_ERR_INVALID_ARG, "X and O must not be NULL");
  if (!aligned16(X) || !aligned16(O)) return fail(DION3_ERR_INVALID_ARG, "X and O must be 16-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, need)) != DION3_OK) return rc;
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carver c{static_cast<char*>(ws)};
  GatherArgs g{};
  NsPlan gp;
  StdPlan sp;
  const bool gram = variant == DION3_NS_GRAM || variant == DION3_NS_GRAM_DENSE;
  if (gram) {
    plan_ns(c, k, m, batch, gp);
    gather_targets(gp, g);
  } else {
    plan_std(c, k, m, batch, sp);
    gather_targets_std(sp, g);
  }
  constexpr int kParts = 64;
  float* parts = c.take<float>(static_cast<long long>(batch) * kParts);
  const long long n = static_cast<long long>(k) * m;
  cudaError_t e = traced_sumsq(static_cast<const __half*>(X), n, batch, parts, kParts, hp->ns_dtype == DION3_BF16, s);
  if (e != cudaSuccess) return cuda_fail(e, "sumsq launch");
  g.k = k; g.m = m; g.batch = batch; g.src_f32 = false;
  g.X = static_cast<const __half*>(X);
  g.fro2 = parts; g.fro2_parts = kParts; g.eps = hp->eps; g.decay = false;
  g.bf16 = hp->ns_dtype == DION3_BF16;
  g.n = k; g.status = st;
  e = traced_gather(g, m % 4 == 0, s);
  if (e != cudaSuccess) return cuda_fail(e, "gather launch");
  NsOut out{static_cast<__half*>(O), static_cast<long long>(k) * m, m};
  rc = gram ? run_gram_ns(gp, *hp, out, st, s, variant == DION3_NS_GRAM_DENSE)
            : run_standard_ns(sp, *hp, out, st, s, variant == DION3_NS_STANDARD_DENSE);
  if (rc != DION3_OK) return rc;
  return ok();
}

dion3_status dion3_workspace_size(const dion3_group* groups, int32_t ngroups, const dion3_hparams* hp,
                                  size_t* bytes) {
  if (bytes == nullptr) return fail(DION3_ERR_INVALID_ARG, "bytes is NULL");
  if (groups == nullptr || ngroups < 1) return fail(DION3_ERR_INVALID_ARG, "need ngroups >= 1 groups");
  dion3_status rc = check_hparams(hp, true);
  if (rc != DION3_OK) return rc;
  Carver c{nullptr};
  for (int i = 0; i < ngroups; ++i) {
    if (groups[i].rows < 1 || groups[i].cols < 1 || groups[i].batch < 1 || groups[i].batch > 65535)
      return fail(DION3_ERR_INVALID_ARG, "group %d: rows, cols >= 1 and 1 <= batch <= 65535 required", i);
    GroupPlan gp;
    plan_group(c, groups[i], hp->f, gp);
  }
  *bytes = round_up(static_cast<long long>(c.off), 256);
  return ok();
}

}  // extern "C"

namespace {
// Streams (one per group, up to kGroupStreams, reused round-robin) and events
// for running the shape groups of one step concurrently.  The per-device pool
// is created on first use; a call holds the pool's lock from the fork to the
// join, so the events are never re-recorded by another host thread in
// between.  The streams and events live until the process exits.  DION3_GROUP_STREAMS=0 runs every group on the caller's stream, and
// so does the launch trace, whose per-launch events would otherwise time
// overlapping kernels.
constexpr int kGroupStreams = 4;
struct StreamPool {
  std::mutex mu;
  bool ready = false;
  cudaStream_t streams[kGroupStreams] = {};
  cudaEvent_t fork = nullptr;
  cudaEvent_t done[kGroupStreams] = {};
};
StreamPool g_pools[64];

bool group_streams_enabled() {
  static const bool on = [] {
    const char* v = getenv("DION3_GROUP_STREAMS");
    return v == nullptr || atoi(v) != 0;
  }();
  if (!on) return false;
  std::lock_guard<std::mutex> lock(g_trace_mu);
  return !g_trace_on;
}

// Whether dion3_step overlaps the accumulation of one shape group with the
// Newton-Schulz GEMMs of another: dion3_set_overlap, initially DION3_OVERLAP
// (default on).
std::atomic<int> g_overlap{-1};
bool overlap_enabled() {
  int v = g_overlap.load();
  if (v < 0) {
    const char* e = getenv("DION3_OVERLAP");
    v = (e == nullptr || atoi(e) != 0) ? 1 : 0;
    int expected = -1;
    g_overlap.compare_exchange_strong(expected, v);
    v = g_overlap.load();
  }
  return v != 0;
}

class GroupStreams {
 public:
  cudaError_t begin(cudaStream_t caller, int ngroups) {
    caller_ = caller;
    n_ = (ngroups > 1 && group_streams_enabled()) ? std::min(ngroups, kGroupStreams) : 0;
    if (n_ == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    pool_ = &g_pools[dev & 63];
    lock_ = std::unique_lock<std::mutex>(pool_->mu);
    if (!pool_->ready) {
      // Handles made by an earlier, failed attempt are kept, not made again.
      for (int i = 0; i < kGroupStreams; ++i) {
        if (pool_->streams[i] == nullptr &&
            (e = cudaStreamCreateWithFlags(&pool_->streams[i], cudaStreamNonBlocking)) != cudaSuccess)
          return e;
        if (pool_->done[i] == nullptr &&
            (e = cudaEventCreateWithFlags(&pool_->done[i], cudaEventDisableTiming)) != cudaSuccess)
          return e;
      }
      if (pool_->fork == nullptr && (e = cudaEventCreateWithFlags(&pool_->fork, cudaEventDisableTiming)) != cudaSuccess)
        return e;
      pool_->ready = true;
    }
    if ((e = cudaEventRecord(pool_->fork, caller_)) != cudaSuccess) return e;
    for (int i = 0; i < n_; ++i)
      if ((e = cudaStreamWaitEvent(pool_->streams[i], pool_->fork, 0)) != cudaSuccess) return e;
    return cudaSuccess;
  }
  cudaStream_t stream(int gi) const { return n_ == 0 ? caller_ : pool_->streams[gi % n_]; }
  cudaError_t end() {
    if (n_ == 0) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_ && e == cudaSuccess; ++i) {
      e = cudaEventRecord(pool_->done[i], pool_->streams[i]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(caller_, pool_->done[i], 0);
    }
    n_ = 0;
    if (lock_.owns_lock()) lock_.unlock();
    return e;
  }
  ~GroupStreams() { end(); }

 private:
  cudaStream_t caller_ = nullptr;
  int n_ = 0;
  StreamPool* pool_ = nullptr;
  std::unique_lock<std::mutex> lock_;
};

// The step of dion3_step; with row_scale (one [batch][rows] fp32 buffer per
// group) the decay of the selected momentum rows is left pending in row_scale
// instead of being written back (dion3_step_lazy).
dion3_status step_impl(const dion3_group* groups, int32_t ngroups, const dion3_hparams* hp, void* ws,
                       size_t ws_bytes, int32_t* const* sel_idx_out, float* const* row_scale,
                       dion3_stream_t stream, const dion3_normuon_params* nm = nullptr,
                       float* const* nm_v = nullptr) {
  size_t need = 0;
  dion3_status rc = dion3_workspace_size(groups, ngroups, hp, &need);
  if (rc != DION3_OK) return rc;
  for (int i = 0; i < ngroups; ++i)
    if ((rc = check_group(groups[i], i)) != DION3_OK) return rc;
  if (sel_idx_out != nullptr)
    for (int i = 0; i < ngroups; ++i)
      if (sel_idx_out[i] != nullptr && (reinterpret_cast<uintptr_t>(sel_idx_out[i]) & 3u))
        return fail(DION3_ERR_INVALID_ARG, "sel_idx_out[%d] must be 4-byte aligned", i);
  if (row_scale != nullptr)
    for (int i = 0; i < ngroups; ++i)
      if (row_scale[i] == nullptr || (reinterpret_cast<uintptr_t>(row_scale[i]) & 3u))
        return fail(DION3_ERR_INVALID_ARG, "row_scale[%d] must be a 4-byte aligned device pointer", i);
  if (nm != nullptr) {
    // eps > 0 keeps d = 1 / (sqrt(v) + eps) finite for a selected row whose
    // orthogonalised values are all zero (v = 0 there).
    if (!(nm->beta2 >= 0.f && nm->beta2 < 1.f) || !(nm->eps > 0.f) || !(nm->rms > 0.f) ||
        !std::isfinite(nm->rms) || !std::isfinite(nm->eps))
      return fail(DION3_ERR_INVALID_ARG, "normuon: need 0 <= beta2 < 1, finite eps > 0, finite rms > 0");
    if (nm_v == nullptr) return fail(DION3_ERR_INVALID_ARG, "normuon: v must not be NULL");
    for (int i = 0; i < ngroups; ++i)
      if (nm_v[i] == nullptr || (reinterpret_cast<uintptr_t>(nm_v[i]) & 3u))
        return fail(DION3_ERR_INVALID_ARG, "v[%d] must be a 4-byte aligned device pointer", i);
  }
  if ((rc = check_ws(ws, ws_bytes, need)) != DION3_OK) return rc;
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");

  cudaStream_t s0 = reinterpret_cast<cudaStream_t>(stream);
  const float lr_eff = static_cast<float>(static_cast<double>(hp->lr) / std::sqrt(static_cast<double>(hp->f)));
  std::vector<GroupPlan> plans(ngroups);
  {
    Carver c{static_cast<char*>(ws)};
    for (int gi = 0; gi < ngroups; ++gi) plan_group(c, groups[gi], hp->f, plans[gi]);
  }
  auto sel_of = [&](int gi) -> int32_t* {
    return (sel_idx_out != nullptr && sel_idx_out[gi] != nullptr) ? sel_idx_out[gi] : plans[gi].idx;
  };
  // (a) accumulate + norms of group gi, standalone launches.
  auto accumulate = [&](int gi, cudaStream_t s) -> dion3_status {
    const dion3_group& g = groups[gi];
    const GroupPlan& gp = plans[gi];
    for (int b0 = 0; b0 < g.batch; b0 += kMaxBatchPerLaunch) {
      const int nb = std::min(kMaxBatchPerLaunch, g.batch - b0);
      AccumArgs a{};
      a.rows = g.rows; a.cols = g.cols; a.batch = nb; a.grad_dtype = g.grad_dtype;
      for (int i = 0; i < nb; ++i) {
        a.M[i] = g.momentum[b0 + i];
        a.G[i] = g.grads[b0 + i];
      }
      a.l1 = gp.l1 + static_cast<size_t>(b0) * g.rows;
      a.sq = gp.sq + static_cast<size_t>(b0) * g.rows;
      if (row_scale != nullptr) a.scale = row_scale[gi] + static_cast<size_t>(b0) * g.rows;
      const cudaError_t e = traced_accum(a, g.cols % 8 == 0, s);
      if (e != cudaSuccess) return cuda_fail(e, "accum_rownorm launch");
    }
    return DION3_OK;
  };
  // The same accumulation as a pool of rows (for the streaming warps of the
  // GEMM launches that run meanwhile): only for groups of <= kPoolMax matrices
  // whose rows take the vector path.
  auto poolable = [&](int gi) { return groups[gi].batch <= kPoolMax && groups[gi].cols % 8 == 0; };
  auto make_pool = [&](int gi, AccumPool& pool) {
    const dion3_group& g = groups[gi];
    const GroupPlan& gp = plans[gi];
    pool.total = static_cast<long long>(g.batch) * g.rows;
    pool.rows = g.rows;
    pool.cols = g.cols;
    pool.grad_dtype = g.grad_dtype == DION3_BF16 ? kBF16 : kF32;
    pool.next = gp.pool_next;
    pool.l1 = gp.l1;
    pool.sq = gp.sq;
    pool.scale = row_scale != nullptr ? row_scale[gi] : nullptr;
    for (int b = 0; b < g.batch; ++b) {
      pool.M[b] = g.momentum[b];
      pool.G[b] = g.grads[b];
    }
  };
  // Top-k, gather/normalise (+ decay of the selected momentum rows), Gram-NS
  // (its GEMM launches lending their streaming warps to `pool`, then to
  // `spool`), the per-neuron normalisation if asked, and the scatter update of
  // group gi unless it is deferred into a later group's scatter pool.
  auto select_orthogonalise_update = [&](int gi, cudaStream_t s, const AccumPool* pool, int pool_gi,
                                         const ScatterPool* spool, bool defer) -> dion3_status {
    const dion3_group& g = groups[gi];
    const GroupPlan& gp = plans[gi];
    int32_t* idx = sel_of(gi);
    const bool vec = g.cols % 8 == 0;
    cudaError_t e;
    TopkArgs t{};
    t.rows = g.rows; t.k = gp.k; t.batch = g.batch; t.l1 = gp.l1; t.sq = gp.sq; t.idx = idx; t.fro2 = gp.fro2;
    if ((e = traced_topk(t, s)) != cudaSuccess) return cuda_fail(e, "topk launch");
    for (int b0 = 0; b0 < g.batch; b0 += kMaxBatchPerLaunch) {
      const int nb = std::min(kMaxBatchPerLaunch, g.batch - b0);
      GatherArgs ga{};
      ga.k = gp.k; ga.m = g.cols; ga.batch = nb; ga.src_f32 = true;
      for (int i = 0; i < nb; ++i) ga.M[i] = g.momentum[b0 + i];
      ga.idx = idx + static_cast<size_t>(b0) * gp.k;
      ga.fro2 = gp.fro2 + b0; ga.fro2_parts = 1; ga.eps = hp->eps; ga.mu = hp->mu;
      ga.decay = row_scale == nullptr;
      if (row_scale != nullptr) ga.scale_out = row_scale[gi] + static_cast<size_t>(b0) * g.rows;
      ga.bf16 = hp->ns_dtype == DION3_BF16;
      ga.n = g.rows; ga.status = st;
      gather_targets(gp.ns, ga);
      ga.out_rows += ga.rows_bstride * b0;
      if (ga.out_cols != nullptr) ga.out_cols += ga.cols_bstride * b0;
      if ((e = traced_gather(ga, vec, s)) != cudaSuccess) return cuda_fail(e, "gather launch");
    }
    if (pool != nullptr) {
      e = cudaMemsetAsync(pool->next, 0, sizeof(unsigned long long), s);
      if (e != cudaSuccess) return cuda_fail(e, "pool counter reset");
    }
    if (spool != nullptr) {
      e = cudaMemsetAsync(spool->next, 0, sizeof(unsigned long long), s);
      if (e != cudaSuccess) return cuda_fail(e, "scatter pool counter reset");
    }
    NsOut out{gp.O, gp.o_bs, gp.ld_o};
    dion3_status rc2 = run_gram_ns(gp.ns, *hp, out, st, s, false, pool, spool);
    if (rc2 != DION3_OK) return rc2;
    if (pool != nullptr) {
      // Rows of the pool the streaming warps did not reach.
      if ((e = traced_accum_pool(*pool, s)) != cudaSuccess) return cuda_fail(e, "accum_pool launch");
    } else if (pool_gi >= 0) {
      if ((rc2 = accumulate(pool_gi, s)) != DION3_OK) return rc2;
    }
    if (spool != nullptr) {
      // Deferred updates the streaming warps did not reach.
      if ((e = traced_scatter_pool(*spool, s)) != cudaSuccess) return cuda_fail(e, "scatter_pool launch");
    }
    if (nm != nullptr) {
      // Per-neuron normalisation of the k orthogonalised rows (v of the
      // selected parameter rows, the row factors, scaled to RMS rms).
      NormRowsArgs na{};
      na.rows = g.rows; na.k = gp.k; na.m = g.cols; na.batch = g.batch;
      na.idx = idx; na.O = gp.O; na.o_bstride = gp.o_bs; na.ld_o = gp.ld_o;
      na.o_bf16 = hp->ns_dtype == DION3_BF16;
      na.v = nm_v[gi]; na.beta2 = nm->beta2; na.eps = nm->eps;
      na.d = gp.nm_d; na.rowc = gp.nm_rowc; na.status = st;
      if ((e = traced_normuon_rows(na, g.cols % 8 == 0 && gp.ld_o % 8 == 0, s)) != cudaSuccess)
        return cuda_fail(e, "normuon rows launch");
      NormScaleArgs sc{};
      sc.k = gp.k; sc.m = g.cols; sc.batch = g.batch; sc.rowc = gp.nm_rowc; sc.d = gp.nm_d; sc.rms = nm->rms;
      if ((e = traced_normuon_scale(sc, s)) != cudaSuccess) return cuda_fail(e, "normuon scale launch");
    }
    // (c) scatter update of the selected parameter rows.
    for (int b0 = 0; b0 < g.batch && !defer; b0 += kMaxBatchPerLaunch) {
      const int nb = std::min(kMaxBatchPerLaunch, g.batch - b0);
      ScatterArgs sa{};
      sa.rows = g.rows; sa.cols = g.cols; sa.k = gp.k; sa.batch = nb; sa.param_dtype = g.param_dtype;
      for (int i = 0; i < nb; ++i) sa.W[i] = g.params[b0 + i];
      sa.idx = idx + static_cast<size_t>(b0) * gp.k;
      sa.O = gp.O + gp.o_bs * b0; sa.o_bstride = gp.o_bs; sa.ld_o = gp.ld_o;
      sa.lr = lr_eff;
      sa.status = st;
      sa.o_bf16 = hp->ns_dtype == DION3_BF16;
      if (nm != nullptr) sa.row_factor = gp.nm_d + static_cast<size_t>(b0) * gp.k;
      if ((e = traced_scatter(sa, vec, s)) != cudaSuccess) return cuda_fail(e, "scatter launch");
    }
    return DION3_OK;
  };

  if (ngroups > 1 && overlap_enabled()) {
    // Accumulation overlapped with Newton-Schulz: the groups run in order on
    // the caller's stream, the one with the most Newton-Schulz work first.
    // Only the first group's accumulation stands alone; each later group's is
    // a pool of rows that the streaming warps of the previous group's GEMM
    // launches work through while the tensor cores run, and a pool kernel
    // finishes (its top-k comes after both, in stream order).
    std::vector<int> order(ngroups);
    std::vector<double> work(ngroups);
    for (int gi = 0; gi < ngroups; ++gi) {
      order[gi] = gi;
      work[gi] = schedule_flops(plans[gi].k, groups[gi].cols, *hp) * groups[gi].batch;
    }
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return work[x] > work[y]; });
    // The last group's GEMM launches have no accumulation to carry; they carry
    // the scatter updates of up to kScatterSegMax earlier groups instead (the
    // ones nearest to it; groups with ragged rows or more than kPoolMax
    // matrices keep their own scatter launches).  Each such group's O,
    // selected indices and per-neuron row factors stay in its part of the
    // workspace until then.
    std::vector<char> deferred(ngroups, 0);
    ScatterPool spool;
    {
      int nd = 0;
      for (int i = ngroups - 2; i >= 0 && nd < kScatterSegMax; --i) {
        const int gi = order[i];
        if (groups[gi].cols % 8 == 0 && groups[gi].batch <= kPoolMax) {
          deferred[gi] = 1;
          ++nd;
        }
      }
      for (int i = 0; i + 1 < ngroups; ++i) {
        const int gi = order[i];
        if (!deferred[gi]) continue;
        const dion3_group& g = groups[gi];
        const GroupPlan& gp = plans[gi];
        ScatterSeg& sg = spool.seg[spool.nseg++];
        sg.start = spool.total;
        sg.rows = g.rows; sg.cols = g.cols; sg.k = gp.k; sg.batch = g.batch;
        sg.param_dtype = g.param_dtype == DION3_BF16 ? kBF16 : kF32;
        sg.o_bf16 = hp->ns_dtype == DION3_BF16;
        sg.idx = sel_of(gi);
        sg.O = gp.O; sg.o_bstride = gp.o_bs; sg.ld_o = gp.ld_o;
        sg.lr = lr_eff;
        sg.row_factor = nm != nullptr ? gp.nm_d : nullptr;
        for (int b = 0; b < g.batch; ++b) sg.W[b] = g.params[b];
        spool.total += static_cast<long long>(g.batch) * gp.k;
      }
      spool.next = plans[order[ngroups - 1]].spool_next;
      spool.status = st;
    }
    if ((rc = accumulate(order[0], s0)) != DION3_OK) return rc;
    for (int i = 0; i < ngroups; ++i) {
      const int gi = order[i];
      const int nx = i + 1 < ngroups ? order[i + 1] : -1;
      AccumPool pool;
      const bool pooled = nx >= 0 && poolable(nx);
      if (pooled) make_pool(nx, pool);
      const bool carries = nx < 0 && spool.total > 0;
      if ((rc = select_orthogonalise_update(gi, s0, pooled ? &pool : nullptr, nx, carries ? &spool : nullptr,
                                            deferred[gi] != 0)) != DION3_OK)
        return rc;
    }
    return ok();
  }

  // Otherwise every group has its own part of the workspace, so the groups are
  // independent: with more than one, each runs on a stream of its own, forked
  // from and joined back into the caller's stream (capturable in a graph).
  GroupStreams fork;
  cudaError_t fe = fork.begin(s0, ngroups);
  if (fe != cudaSuccess) return cuda_fail(fe, "group stream fork");
  for (int gi = 0; gi < ngroups; ++gi) {
    cudaStream_t s = fork.stream(gi);
    if ((rc = accumulate(gi, s)) != DION3_OK) return rc;
    if ((rc = select_orthogonalise_update(gi, s, nullptr, -1, nullptr, false)) != DION3_OK) return rc;
  }
  if ((fe = fork.end()) != cudaSuccess) return cuda_fail(fe, "group stream join");
  return ok();
}
}  // namespace

extern "C" {

dion3_status dion3_step(const dion3_group* groups, int32_t ngroups, const dion3_hparams* hp, void* ws,
                        size_t ws_bytes, int32_t* const* sel_idx_out, dion3_stream_t stream) {
  return step_impl(groups, ngroups, hp, ws, ws_bytes, sel_idx_out, nullptr, stream);
}

dion3_status dion3_step_lazy(const dion3_group* groups, int32_t ngroups, const dion3_hparams* hp,
                             float* const* row_scale, void* ws, size_t ws_bytes, int32_t* const* sel_idx_out,
                             dion3_stream_t stream) {
  if (row_scale == nullptr) return fail(DION3_ERR_INVALID_ARG, "row_scale must not be NULL");
  return step_impl(groups, ngroups, hp, ws, ws_bytes, sel_idx_out, row_scale, stream);
}

dion3_status dion3_step_normuon(const dion3_group* groups, int32_t ngroups, const dion3_hparams* hp,
                               const dion3_normuon_params* nm, float* const* v, void* ws, size_t ws_bytes,
                               int32_t* const* sel_idx_out, dion3_stream_t stream) {
  if (nm == nullptr) return fail(DION3_ERR_INVALID_ARG, "normuon parameters must not be NULL");
  return step_impl(groups, ngroups, hp, ws, ws_bytes, sel_idx_out, nullptr, stream, nm, v);
}

dion3_status dion3_flush_row_scale(int32_t rows, int32_t cols, int32_t batch, float* const* momentum,
                                   float* row_scale, dion3_stream_t stream) {
  if (rows < 1 || cols < 1 || batch < 1) return fail(DION3_ERR_INVALID_ARG, "need rows, cols, batch >= 1");
  if (momentum == nullptr || row_scale == nullptr || (reinterpret_cast<uintptr_t>(row_scale) & 3u))
    return fail(DION3_ERR_INVALID_ARG, "momentum and a 4-byte aligned row_scale are required");
  for (int b = 0; b < batch; ++b)
    if (momentum[b] == nullptr || (reinterpret_cast<uintptr_t>(momentum[b]) & 3u))
      return fail(DION3_ERR_INVALID_ARG, "momentum[%d] NULL or misaligned", b);
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
    const int nb = std::min(kMaxBatchPerLaunch, batch - b0);
    FlushArgs a{};
    a.rows = rows; a.cols = cols; a.batch = nb;
    for (int i = 0; i < nb; ++i) a.M[i] = momentum[b0 + i];
    a.scale = row_scale + static_cast<size_t>(b0) * rows;
    const cudaError_t e = launch_flush_scale(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "flush launch");
  }
  return ok();
}

dion3_status dion3_gemm_f16(int32_t mode, int32_t M, int32_t N, int32_t K, int32_t batch, const void* A,
                            int32_t lda, int64_t a_bstride, const void* B, int32_t ldb, int64_t b_bstride,
                            const void* C, int32_t ldc, int64_t c_bstride, void* D, int32_t ldd,
                            int64_t d_bstride, void* DT, int32_t lddt, int64_t dt_bstride, float alpha,
                            float beta, float gamma, dion3_stream_t stream) {
  const int32_t flags = mode & ~0xF;
  mode &= 0xF;
  if (mode != DION3_GEMM_RECT && mode != DION3_GEMM_SYM_LOWER) return fail(DION3_ERR_INVALID_ARG, "bad GEMM mode");
  if ((flags & ~(DION3_GEMM_OUT_HALF | DION3_GEMM_A_HALF | DION3_GEMM_B_HALF | DION3_GEMM_A_TRANS |
                 DION3_GEMM_B_TRANS)) != 0)
    return fail(DION3_ERR_INVALID_ARG, "unknown GEMM mode flag");
  const bool a_tr = (flags & DION3_GEMM_A_TRANS) != 0, b_tr = (flags & DION3_GEMM_B_TRANS) != 0;
  if (M < 1 || N < 1 || K < 1 || batch < 1 || batch > 65535)
    return fail(DION3_ERR_INVALID_ARG, "need M, N, K >= 1 and 1 <= batch <= 65535");
  if (mode == DION3_GEMM_SYM_LOWER && (M != N || D == nullptr || DT != nullptr))
    return fail(DION3_ERR_INVALID_ARG, "symmetric mode needs M == N, D set and DT NULL");
  if (D == nullptr && DT == nullptr) return fail(DION3_ERR_INVALID_ARG, "no output given");
  if (D != nullptr && ldd < N) return fail(DION3_ERR_INVALID_ARG, "ldd < N");
  if (DT != nullptr && lddt < M) return fail(DION3_ERR_INVALID_ARG, "lddt < M");
  if (C != nullptr && ldc < N) return fail(DION3_ERR_INVALID_ARG, "ldc < N");
  if (((reinterpret_cast<uintptr_t>(D) | reinterpret_cast<uintptr_t>(DT) | reinterpret_cast<uintptr_t>(C)) & 1u) != 0)
    return fail(DION3_ERR_INVALID_ARG, "C, D and DT must be 2-byte aligned");
  if (batch > 1 && (a_bstride < static_cast<int64_t>(lda) * (a_tr ? K : M) ||
                    b_bstride < static_cast<int64_t>(ldb) * (b_tr ? K : N)))
    return fail(DION3_ERR_INVALID_ARG, "operand batch stride smaller than one matrix");
  GemmDesc g{};
  g.A = static_cast<const __half*>(A); g.a_bstride = a_bstride; g.lda = lda;
  g.B = static_cast<const __half*>(B); g.b_bstride = b_bstride; g.ldb = ldb;
  g.M = M; g.N = N; g.K = K; g.batch = batch;
  g.mode = mode == DION3_GEMM_SYM_LOWER ? kSymLower : kRect;
  g.alpha = alpha; g.beta = beta; g.gamma = gamma;
  g.C = static_cast<const __half*>(C); g.c_bstride = c_bstride; g.ldc = ldc;
  g.out = static_cast<__half*>(D); g.out_bstride = d_bstride; g.ld_out = ldd;
  g.outT = static_cast<__half*>(DT); g.outT_bstride = dt_bstride; g.ld_outT = lddt;
  g.out_half = (flags & DION3_GEMM_OUT_HALF) != 0;
  g.a_half = (flags & DION3_GEMM_A_HALF) != 0;
  g.b_half = (flags & DION3_GEMM_B_HALF) != 0;
  g.a_tr = a_tr;
  g.b_tr = b_tr;
  const char* why = nullptr;
  if (!gemm_check(g, &why)) return fail(DION3_ERR_INVALID_ARG, "%s", why);
  if (inject_launch_fail()) return fail(DION3_ERR_CUDA, "injected launch failure (DION3_INJECT=launch_fail)");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");
  const cudaError_t e = traced_gemm(g, st, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "tcgen05 GEMM launch");
  return ok();
}

dion3_status dion3_trace_enable(int32_t on) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  trace_clear_locked();
  g_trace_on = on != 0;
  return ok();
}

dion3_status dion3_trace_collect(dion3_trace_entry* out, int32_t capacity, int32_t* count) {
  if (count == nullptr || (out == nullptr && capacity > 0) || capacity < 0)
    return fail(DION3_ERR_INVALID_ARG, "count must not be NULL and out must hold capacity entries");
  std::lock_guard<std::mutex> lock(g_trace_mu);
  std::vector<dion3_trace_entry> agg;
  for (const auto& r : g_trace) {
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e != cudaSuccess) return cuda_fail(e, "trace event synchronise");
    float ms = 0.f;
    if ((e = cudaEventElapsedTime(&ms, r.a, r.b)) != cudaSuccess) return cuda_fail(e, "trace elapsed time");
    dion3_trace_entry* slot = nullptr;
    for (auto& x : agg)
      if (strncmp(x.name, r.name.c_str(), sizeof x.name - 1) == 0) slot = &x;
    if (slot == nullptr) {
      agg.push_back(dion3_trace_entry{});
      slot = &agg.back();
      snprintf(slot->name, sizeof slot->name, "%s", r.name.c_str());
    }
    slot->launches += r.launches;
    slot->total_ms += ms;
    slot->useful_flops += r.flops;
    slot->algo_bytes += r.bytes;
  }
  *count = static_cast<int32_t>(agg.size());
  for (int i = 0; i < static_cast<int>(agg.size()) && i < capacity; ++i) out[i] = agg[i];
  trace_clear_locked();
  return ok();
}

dion3_status dion3_set_overlap(int32_t on) {
  g_overlap.store(on != 0 ? 1 : 0);
  return ok();
}

dion3_status dion3_wait_probe(int32_t arrive, int64_t limit_ns, dion3_stream_t stream) {
  if (limit_ns < 1000 || limit_ns > 1000000000LL)
    return fail(DION3_ERR_INVALID_ARG, "limit_ns must lie in [1e3, 1e9]");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");
  const cudaError_t e = launch_wait_probe(arrive != 0, static_cast<unsigned long long>(limit_ns), st,
                                          reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "wait probe launch");
  return ok();
}

dion3_status dion3_device_status(dion3_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  unsigned* st = device_status_ptr();
  if (st == nullptr) return fail(DION3_ERR_CUDA, "cannot resolve the device status word");
  unsigned v = 0;
  if ((e = cudaMemcpy(&v, st, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e, "status read");
  const unsigned zero = 0;
  if ((e = cudaMemcpy(st, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "status clear");
  if (v & kDevTimeout) return fail(DION3_ERR_TIMEOUT, "a bounded device-side wait ran out");
  if (v & kDevCheck) return fail(DION3_ERR_DEVICE_CHECK, "a device-side check failed");
  return ok();
}

}  // extern "C"
