// Tensor-core GEMM for the Gram Newton-Schulz path on sm_103a.
//
// D = A B^T with A [batch][M][K] and B [batch][N][K] in fp16, both K-major,
// fp32 accumulation in tensor memory, and the epilogue
//     v = alpha D + beta C + gamma I
// rounded to fp16.  In kSymLower mode (M == N, symmetric result) only tiles
// that meet the lower triangle are computed; every element on or below the
// diagonal is written in place and mirrored above it, so the stored matrix is
// exactly symmetric.  In kRect mode every tile is computed and written in the
// normal and/or the transposed orientation.
//
// Half-stored symmetric matrices.  A symmetric s x s result may instead be
// written as its lower triangle at 256 x 256 block granularity: the blocks
// below the diagonal and the full diagonal blocks (mirrored inside), nothing
// above (out_half).  Such a matrix is read back as an operand (a_half /
// b_half): a K range of 64 that lies within or left of the operand rows'
// diagonal block is loaded K-major from the rows themselves; a K range right
// of it, where S[m][k] is above the diagonal, is loaded from S[k][m] (below
// it) as an MN-major tile: two 64 x 64 boxes, read by the MMA with the
// MN-major bit of the instruction descriptor set.  Both CTAs of a pair have
// the same 256-row super-row, so they always agree on the orientation.  This
// skips the mirror writes outside the diagonal blocks and never touches the
// upper triangle.  When the product is A A^T (plus beta A, with A half-stored,
// and gamma I), a diagonal super-tile is written whole as computed instead of
// mirrored (diag_full): element (i, j) and (j, i) are the same sum of the same
// products in the same order, so the tile is exactly symmetric either way, and
// every epilogue warp then writes the same number of chunks.  The same MN-major
// tiles read an operand that is given as its
// transpose (a_tr / b_tr: A stored [K][M]), so a matrix kept in one orientation
// serves as A = Y or A = Y^T alike.
//
// Method source: "Dion3: Full-Stack Orthogonal Updates" (agihunt summary of the
// paper).  First-level paragraph: Newton-Schulz iterates on the small
// symmetric Gram matrix X X^T and multiplies back by X at the end.  Second-level
// paragraph: the symmetric products A^T A and A^2 + B only need the lower
// triangle, copied to the upper one.  The products used here:
//   R = Y Y^T          (A = B = Y, kSymLower)
//   Z = cR.R + bR + aI (A = B = R, C = R, kSymLower)
//   Q <- Z Q, T = R Z, R <- Z T  (B symmetric, so B^T = B; kSymLower)
//   Y_new^T = Y^T Q, O = (Y^T Q)^T  (A = Y^T, B = Q, kRect)
//
// Kernel: persistent clusters of two CTAs on two SMs (a CTA pair), one CTA
// per SM.  A cluster owns a 256 x 256 super-tile at a time, handed out
// round-robin over the whole batch, and computes it with the paired-SM MMA
// (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16): CTA rank r holds rows
// 128 r .. 128 r + 127 of A and rows 128 r .. 128 r + 127 of the B panel in its
// own shared memory, and receives rows 128 r .. of the result in its own TMEM.
// A ring slot therefore holds 32 KB per CTA (its A tile and its half of B), so
// the 192 KB ring is 6 slots deep.  12 warps per CTA:
//   warp 0         TMA producer (both CTAs): the whole warp runs the loop and
//                  waits, one elected lane fills the CTA's own slot and
//                  signals the even CTA's "full" barrier (cta_group::2 copy);
//   warp 1         allocates 512 TMEM columns for the pair (both CTAs); in the
//                  even CTA the whole warp runs the MMA loop and one elected
//                  lane issues the paired MMAs into one of two 256-column fp32
//                  accumulators and releases ring slots and accumulators in
//                  both CTAs with multicast commits;
//   warps 2..9     epilogue (both CTAs): two warps per TMEM lane quadrant
//                  (warp % 4), each taking half of the 256 columns, 32 at a
//                  time in a rolled loop (C, when given, loaded one chunk
//                  ahead, the first chunk's before the accumulator is ready):
//                  tcgen05.ld, alpha/beta/gamma, then the 32 x 32 box (and
//                  its transpose) staged in swizzled shared memory and
//                  written with bulk tensor stores (a chunk on the diagonal
//                  of a symmetric result as one symmetric box); then one
//                  CTA-scope arrive per thread tells the even CTA that the
//                  accumulator is free;
//   warps 10, 11   streaming warps (and warp 1 of the odd CTA, which issues
//                  no MMAs): when the launch carries an accumulation pool
//                  (GemmDesc::pool), rows of another shape group's step a0,
//                  then, when it carries a scatter pool (GemmDesc::spool),
//                  rows of deferred step a7 updates, each taken from its
//                  pool's counter until this CTA's producer has issued its
//                  last copy; otherwise they go straight to the final barrier.
// Running the producer and MMA loops on whole warps keeps their loop state
// warp-uniform; a single-lane loop (`if (lane == 0)`) measured 3-18 % slower
// once its body branched between copy shapes.
// Every mbarrier wait is bounded (about one second of %globaltimer); a wait
// that runs out sets a bit in the device status word and the CTA winds down:
// the issuing CTA waits (bounded) for its MMAs, both CTAs meet at a cluster
// barrier before freeing TMEM, and TMEM is freed on every path.
#include "accum_row.cuh"
#include "internal.h"
#include "scatter_row.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

namespace dion3 {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // fp16 elements per 128-byte swizzle row
constexpr int BN = 256;
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;   // two per TMEM lane quadrant, each half of the columns
constexpr int kSideWarps = 2;  // streaming warps: rows of another group's accumulation
// Iterations of loads each streaming warp keeps in flight per row (bf16
// gradients stay packed, so they afford more depth than fp32 ones; deeper
// ones spill at the kernel's register budget).
constexpr int kSideUnrollBF16 = 6;
constexpr int kSideUnrollF32 = 4;
constexpr bool kSideEvict = true;
constexpr int kSideUnrollScatter = 4;  // bf16 parameters; half of it for fp32 ones
constexpr int kThreads = 32 * (2 + kEpiWarps + kSideWarps);
constexpr int kTmemCols = 512; // two 256-column accumulators
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

struct GemmParams {
  int M, N, K, mode;
  int tiles_r, tiles_c;      // row (128) and column (256) tile counts of one matrix
  int pairs_r;               // super-tile rows (256) of one matrix
  int units_per_mat, total_units;  // super-tiles per matrix / in the launch
  float alpha, beta, gamma;
  const __half* C; long long c_bs; int ldc;
  __half* out; long long out_bs; int ld_out;
  __half* outT; long long outT_bs; int ld_outT;
  int tma_out, tma_outT;     // the output has a TMA store map (16-byte pitch rules hold)
  int batch, reverse;        // visit matrices from the last one when reverse
  int a_half, b_half;        // A / B is a half-stored symmetric matrix (M == K / N == K)
  int a_tr, b_tr;            // A / B is given as its transpose ([K][M] / [K][N]): all tiles MN-major
  int out_half;              // kSymLower: no mirror outside the diagonal super-tiles
  int diag_full;             // out_half: diagonal super-tiles written whole, as computed (no mirror)
  unsigned* status;
  AccumPool pool;            // rows for the streaming warps (total 0: none)
  ScatterPool spool;         // then these (total 0: none)
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}

// Bounded wait for the phase of `bar` with the given parity: gives up after
// `limit_ns` of %globaltimer, recording kDevTimeout in the status word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
  return true;
}

// The same wait by a whole warp: true only if every lane saw the phase.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, status));
}

// One lane of a fully active warp (the same lane every time: the lowest).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(pred));
  return pred != 0u;
}

// Paired-SM variant: the box lands in this CTA's shared memory and the
// completed bytes are reported to an mbarrier that may live in the peer CTA
// (`bar` is a shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                                 int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Bulk tensor store of a shared-memory box to global memory (bulk-group
// completion; out-of-range parts of the box are not written).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// None of this thread's bulk groups is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// At most this thread's most recent bulk group may still be reading shared
// memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Generic-proxy shared-memory writes become visible to the async proxy.
__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void ld_shared_v4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in the
// peer CTA).  Its one use hands a TMEM accumulator back to the MMA issuer: the
// epilogue's reads of it are complete (tcgen05.wait::ld) and ordered before
// the arrive by tcgen05.fence::before_thread_sync, and no generic memory write
// depends on it, so the release is at CTA scope.  At cluster scope the arrive
// waited for the thread's bulk stores in flight: 1.3-2.4 k cycles per tile in
// every epilogue warp, measured, and the products with K = 512 7-14 % slower.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster_addr) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster_addr) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the cluster (each warp reconverges first: the
// barrier instructions are .aligned).
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Paired allocation: one warp of each CTA of the pair executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Paired-SM MMA: A and B descriptors name the same shared-memory offsets in
// both CTAs of the pair; D is the same TMEM address in both.
__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at offset `bar` of every CTA in `mask` once this
// thread's earlier paired MMAs have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   bar),
               "h"(mask)
               : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Ties registers written by an earlier tcgen05.ld to a point after the wait,
// so no use of them is scheduled before it (no instruction is emitted).
__device__ __forceinline__ void tmem_regs_ready(uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) asm volatile("" : "+r"(v[j])::"memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row (1024-byte) core groups
// stacked along M/N (stride-dimension byte offset 1024), descriptor version 1
// (bits 46-47), swizzle mode 2 = 128B (bits 61-63).  The leading-dimension
// offset is not used for swizzled K-major layouts whose MMA K extent (32 bytes)
// lies inside one swizzle row; it is set to 1 (16 bytes).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// The same for an MN-major operand tile of 128 rows (M or N) x 64 K written by
// TMA as two 64 x 64 boxes with 128-byte swizzling: each box holds 64 K rows of
// 128 bytes (64 elements along M/N); 8-row K groups 1024 bytes apart
// (stride-dimension offset) and the two 64-element M/N halves 8192 bytes apart
// (leading-dimension offset).  One K = 16 step spans two K groups: 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(8192u >> 4) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}
constexpr uint32_t kIdescATransposed = 1u << 15;  // A is MN-major
constexpr uint32_t kIdescBTransposed = 1u << 16;  // B is MN-major

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B both fp16
// (bits 7-9, 10-12 = 0) or both bf16 (= 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28; M = 256 for the paired MMA (128
// rows per CTA).
template <bool BF16>
__device__ __forceinline__ constexpr uint32_t idesc_f32acc() {
  return (1u << 4) | ((BF16 ? 1u : 0u) << 7) | ((BF16 ? 1u : 0u) << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>((2 * BM) >> 4) << 24);
}

// 16-bit element conversions of the two operand types (storage is 16-bit
// words either way).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
}
template <bool BF16>
__device__ __forceinline__ float unpack1(uint16_t h) {
  if constexpr (BF16) {
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    return __half2float(__ushort_as_half(h));
  }
}
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&t);
  } else {
    const __half2 t = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&t);
  }
}

// Super-tile u of one matrix -> (super-row P, column tile bc); the CTA of
// rank r computes row tile 2 P + r.  kSymLower keeps the super-tiles that meet
// the lower triangle: 256 P + 255 >= 256 bc, i.e. P >= bc, enumerated column by
// column.
__device__ __forceinline__ void unit_coords(const GemmParams& p, int u, int& P, int& bc) {
  if (p.mode == kSymLower) {
    bc = 0;
    for (;;) {
      const int cnt = p.pairs_r - bc;
      if (u < cnt) break;
      u -= cnt;
      ++bc;
    }
    P = bc + u;
  } else {
    P = u / p.tiles_c;
    bc = u % p.tiles_c;
  }
}

struct Smem {
  static constexpr int kABytes = BM * BK * 2;   // 16 KB
  static constexpr int kBBytes = (BN / 2) * BK * 2;   // this CTA's half of B: 16 KB
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  // Epilogue staging: per epilogue warp one 32 x 32 fp16 box and its
  // transpose (2 KB each), laid out with the 64-byte swizzle of the store
  // tensor maps.
  static constexpr int kStageBoxBytes = 32 * 32 * 2;
  static constexpr int kWarpStagingBytes = 2 * kStageBoxBytes;
  static constexpr int kStagingBytes = kEpiWarps * kWarpStagingBytes;
  // barriers: full[S], empty[S], tfull[2], tempty[2], drain
  static constexpr int kBarBytes = (2 * kStages + 5) * 8;
  static constexpr int kDyn = 1024 + kRingBytes + kStagingBytes + kBarBytes + 16;
};

// First K slab (of BK) of an operand whose rows lie in super-row `blk` that is
// read from the transpose as MN-major tiles: 0 for an operand given as its
// transpose; for a half-stored one the slabs right of its diagonal 256 x 256
// block; nkb (never) for a plain operand.
__device__ __forceinline__ int first_transposed_slab(int tr, int half, int blk, int nkb) {
  if (tr) return 0;
  const int t = 4 * (blk + 1);
  return half && t < nkb ? t : nkb;
}

// MMA issue for K slabs [kb0, kb1) of one tile, A / B K-major or MN-major
// (AT / BT), run by a whole warp: wait for each ring slot, then one elected
// lane (always the same, so its commits track all its MMAs) issues four
// K = 16 paired MMAs and releases the slot in both CTAs.  One K = 16 step advances a descriptor's start address
// (16-byte units) by 32 bytes along a K-major row, or by two 1024-byte K
// groups MN-major.  Returns false if a wait ran out.
template <bool BF16, bool AT, bool BT>
__device__ __forceinline__ bool mma_slabs(int kb0, int kb1, uint32_t& kc, uint32_t d, uint32_t sA, uint32_t sB,
                                          uint32_t bar_full, uint32_t bar_empty, unsigned* status) {
  constexpr uint32_t id = idesc_f32acc<BF16>() | (AT ? kIdescATransposed : 0u) | (BT ? kIdescBTransposed : 0u);
  constexpr uint64_t a_step = AT ? 128u : 2u, b_step = BT ? 128u : 2u;
  for (int kb = kb0; kb < kb1; ++kb, ++kc) {
    const uint32_t s = kc % kStages, ph = (kc / kStages) & 1u;
    if (!mbar_wait_warp(bar_full + 8 * s, ph, status)) return false;
    tc_fence_after();
    const uint32_t a_src = sA + s * Smem::kABytes, b_src = sB + s * Smem::kBBytes;
    const uint64_t da = AT ? sdesc_mnmajor_sw128(a_src) : sdesc_kmajor_sw128(a_src);
    const uint64_t db = BT ? sdesc_mnmajor_sw128(b_src) : sdesc_kmajor_sw128(b_src);
    if (elect_one()) {
#pragma unroll
      for (int kk = 0; kk < BK / 16; ++kk)
        mma_f16_pair(d, da + a_step * kk, db + b_step * kk, id, (kb > 0 || kk > 0) ? 1u : 0u);
      mma_commit_pair(bar_empty + 8 * s, 0x3);
    }
    __syncwarp();
  }
  return true;
}

// Values of one 32-row x 32-column chunk held by a warp: thread `lane` owns
// row r; v[j] is column c0 + j of the fp32 accumulator.  hp receives
// alpha D + beta C + gamma I as packed fp16 pairs (rows r >= M give zeros and
// read nothing).
// The C operand of a chunk in 16-byte pieces.  A warp loads the C values of
// all its chunks of a tile before it waits for the accumulator, so the load
// latency overlaps the MMAs (only when the chunk is full and C's pitch allows
// vector loads; otherwise chunk_values reads C element-wise).
__device__ __forceinline__ bool c_vector_ok(const GemmParams& p, int c0) {
  return p.C != nullptr && (c0 + 32 <= p.N) && (p.ldc % 8 == 0);
}
__device__ __forceinline__ void prefetch_c(const GemmParams& p, int bidx, int r, int c0, uint4 (&cv)[4]) {
  if (c_vector_ok(p, c0) && r < p.M) {
    const __half* crow = p.C + static_cast<long long>(bidx) * p.c_bs + static_cast<size_t>(r) * p.ldc + c0;
#pragma unroll
    for (int q = 0; q < 4; ++q) cv[q] = *reinterpret_cast<const uint4*>(crow + 8 * q);
  }
}

// READ_C = false: the caller knows there is no C (the fast path).
template <bool BF16, bool READ_C>
__device__ __forceinline__ void chunk_values(const GemmParams& p, int bidx, int r, int c0, const uint32_t (&v)[32],
                                             const uint4 (&cv)[4], uint32_t (&hp)[16]) {
  float f[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) f[j] = p.alpha * __uint_as_float(v[j]);
  if (READ_C && p.C != nullptr && r < p.M) {
    const __half* crow = p.C + static_cast<long long>(bidx) * p.c_bs + static_cast<size_t>(r) * p.ldc + c0;
    if (c_vector_ok(p, c0)) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {cv[q].x, cv[q].y, cv[q].z, cv[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = unpack2<BF16>(w[e]);
          f[8 * q + 2 * e] = fmaf(p.beta, x.x, f[8 * q + 2 * e]);
          f[8 * q + 2 * e + 1] = fmaf(p.beta, x.y, f[8 * q + 2 * e + 1]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < p.N) f[j] = fmaf(p.beta, unpack1<BF16>(__half_as_ushort(crow[j])), f[j]);
    }
  }
  // gamma I meets only the chunk whose columns are the warp's rows (both
  // start at a multiple of 32).
  if (p.gamma != 0.0f && c0 == (r & ~31)) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (r == c0 + j) f[j] += p.gamma;
  }
  if (r >= p.M) {
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j) hp[j] = pack2<BF16>(f[2 * j], f[2 * j + 1]);
}

__device__ __forceinline__ uint16_t half_bits(const uint32_t (&hp)[16], int j) {
  return static_cast<uint16_t>(hp[j / 2] >> (16 * (j % 2)));
}

// Element-wise stores of one chunk: chunks on the diagonal of a symmetric
// result (an element is kept when r >= c and mirrored when r > c), or outputs
// whose pitch a TMA map cannot describe.  row0 is the warp's first row;
// mirror = false skips the mirror of a symmetric result.
__device__ __forceinline__ void store_chunk_scalar(const GemmParams& p, int bidx, int r, int c0, int row0,
                                                   const uint32_t (&hp)[16], bool mirror) {
  if (r >= p.M) return;
  const bool sym = p.mode == kSymLower && !p.diag_full;
  const bool full = (c0 + 32 <= p.N);
  const bool below = !sym || (row0 > c0 + 31);
  __half* outb = p.out ? p.out + static_cast<long long>(bidx) * p.out_bs : nullptr;
  if (outb != nullptr) {
    __half* dst = outb + static_cast<size_t>(r) * p.ld_out + c0;
    if (below && full && (p.ld_out % 8 == 0)) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(hp[4 * q], hp[4 * q + 1], hp[4 * q + 2], hp[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (c0 + j < p.N && (!sym || r >= c0 + j)) dst[j] = __ushort_as_half(half_bits(hp, j));
    }
  }
  __half* tb = sym ? (mirror ? outb : nullptr)
                    : (p.outT ? p.outT + static_cast<long long>(bidx) * p.outT_bs : nullptr);
  if (tb != nullptr) {
    const int ldt = sym ? p.ld_out : p.ld_outT;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const int c = c0 + j;
      if (c < p.N && (!sym || r > c)) tb[static_cast<size_t>(c) * ldt + r] = __ushort_as_half(half_bits(hp, j));
    }
  }
}

// A chunk on the diagonal of a triangle-only result (its first row and column
// coincide: both are multiples of 32) is written as one symmetric 32 x 32
// box.  The warp stages the chunk's transpose in the second half of its
// staging buffer, then each row keeps its own values on and below the
// diagonal, takes the rest from the transpose, and is staged in the first
// half, ready for one bulk store.
__device__ __forceinline__ void diag_chunk(uint32_t buf, uint32_t sw, int lane, uint32_t staged,
                                           uint32_t (&hp)[16]) {
  const uint32_t tbuf = buf + Smem::kStageBoxBytes;
  if (lane == 0 && staged >= 1) bulk_wait_read_0();
  __syncwarp();
  const uint32_t lo = static_cast<uint32_t>(lane & 7) << 1, hi = static_cast<uint32_t>(lane >> 3);
#pragma unroll
  for (int j = 0; j < 32; ++j) st_shared_u16(tbuf + j * 64 + (((hi ^ ((j >> 1) & 3)) << 4) | lo), half_bits(hp, j));
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t t[4];
    ld_shared_v4(tbuf + lane * 64 + ((static_cast<uint32_t>(q) ^ sw) << 4), t);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int m = 4 * q + e;  // columns 2m and 2m + 1 of this row
      if (2 * m > lane)
        hp[m] = t[e];
      else if (2 * m == lane)
        hp[m] = (hp[m] & 0xFFFFu) | (t[e] & 0xFFFF0000u);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st_shared_v4(buf + lane * 64 + ((static_cast<uint32_t>(q) ^ sw) << 4), hp[4 * q], hp[4 * q + 1], hp[4 * q + 2],
                 hp[4 * q + 3]);
  fence_async_shared();
  __syncwarp();
}

template <bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmAT, const __grid_constant__ CUtensorMap tmBT,
                        const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ CUtensorMap tmOutT,
                        const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + kStages * Smem::kABytes;
  const uint32_t staging = base + Smem::kRingBytes;
  const uint32_t bar_full = staging + Smem::kStagingBytes;
  const uint32_t bar_empty = bar_full + kStages * 8;
  const uint32_t bar_tfull = bar_empty + kStages * 8;
  const uint32_t bar_tempty = bar_tfull + 2 * 8;
  const uint32_t bar_drain = bar_tempty + 2 * 8;
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + Smem::kRingBytes + Smem::kStagingBytes + Smem::kBarBytes);
  // Whether this CTA's TMA producer has issued its last copy: the streaming
  // warps take no new row after that.  The MMAs and epilogues of the last
  // tiles still cover the row being moved, and the CTA's exit (and with it the
  // next launch) waits less for a long row than if they stopped once the
  // epilogue warps had finished (measured 0.1-0.2 ms per step faster).
  uint32_t* prod_done = tmem_slot + 1;

  // The next kernel on the stream may be scheduled once every CTA of this one
  // has started (programmatic dependent launch).
  pdl_trigger();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nkb = (p.K + BK - 1) / BK;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;  // issues the pair's MMAs
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  constexpr uint16_t kPair = 0x3;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8 * s, 1);   // used in the even CTA: its producer + both CTAs' bytes
      mbar_init(bar_empty + 8 * s, 1);  // the pair's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull + 8 * a, 1);
      mbar_init(bar_tempty + 8 * a, 2 * 32 * kEpiWarps);  // used in the even CTA: both CTAs' epilogue threads
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    *prod_done = 0u;
  }
  if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  // Both CTAs' barriers are initialised before any multicast copy or remote
  // arrive can reach them.
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Set-up done (barriers, tensor memory): wait for the previous kernel on the
  // stream before touching global memory.
  pdl_wait();

  if (warp == 0) {
    {
      // ---------------- TMA producer: the whole warp runs the loop, one
      // elected lane issues the copies ----------------
      uint32_t kc = 0;
      bool ok = true;
      for (int u = cluster; u < p.total_units && ok; u += nclusters) {
        const int bidx = p.reverse ? p.batch - 1 - u / p.units_per_mat : u / p.units_per_mat;
        int P, bc;
        unit_coords(p, u % p.units_per_mat, P, bc);
        const int bi = 2 * P + static_cast<int>(rank);
        const int b_row = bc * BN + static_cast<int>(rank) * (BN / 2);
        const int a_t0 = first_transposed_slab(p.a_tr, p.a_half, P, nkb);
        const int b_t0 = first_transposed_slab(p.b_tr, p.b_half, bc, nkb);
        for (int kb = 0; kb < nkb; ++kb, ++kc) {
          const uint32_t s = kc % kStages, ph = (kc / kStages) & 1u;
          if (!mbar_wait_warp(bar_empty + 8 * s, ph ^ 1u, p.status)) {
            ok = false;
            break;
          }
          // An operand tile is one 128-row box of the operand's rows (K-major)
          // or, for a K range above the diagonal of a half-stored operand, two
          // 64 x 64 boxes of its transpose: K rows x M/N columns (MN-major).
          // Coordinates are (column, row, matrix).
          const uint32_t a_dst = sA + s * Smem::kABytes, b_dst = sB + s * Smem::kBBytes;
          const int am = bi * BM, k0 = kb * BK;
          if (elect_one()) {
            if (leader) mbar_arrive_expect_tx(bar_full + 8 * s, 2 * Smem::kStageBytes);
            const uint32_t full_even = map_to_rank(bar_full + 8 * s, 0);
            if (kb >= a_t0) {
              tma_load_3d_pair(a_dst, &tmAT, full_even, am, k0, bidx);
              tma_load_3d_pair(a_dst + Smem::kABytes / 2, &tmAT, full_even, am + BM / 2, k0, bidx);
            } else {
              tma_load_3d_pair(a_dst, &tmA, full_even, k0, am, bidx);
            }
            if (kb >= b_t0) {
              tma_load_3d_pair(b_dst, &tmBT, full_even, b_row, k0, bidx);
              tma_load_3d_pair(b_dst + Smem::kBBytes / 2, &tmBT, full_even, b_row + BN / 4, k0, bidx);
            } else {
              tma_load_3d_pair(b_dst, &tmB, full_even, k0, b_row, bidx);
            }
          }
          __syncwarp();
        }
      }
      if (lane == 0) *reinterpret_cast<volatile uint32_t*>(prod_done) = 1u;
      // Wait (bounded) until every copy issued into the ring has landed, so no
      // copy is in flight when the pair exits (the even CTA's barriers count
      // the bytes of both CTAs).
      for (uint32_t i = 0; leader && i < kStages && i < kc; ++i) {
        const uint32_t last = kc - 1 - i;  // most recent fill of stage last % kStages
        mbar_wait_warp(bar_full + 8 * (last % kStages), (last / kStages) & 1u, p.status);
      }
    }
  } else if (warp == 1 && leader) {
    {
      // ---------------- MMA issuer: the whole warp of the even CTA runs the
      // loop, one elected lane issues ----------------
      uint32_t kc = 0, tc = 0;
      bool ok = true;
      for (int u = cluster; u < p.total_units && ok; u += nclusters, ++tc) {
        const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
        int P, bc;
        unit_coords(p, u % p.units_per_mat, P, bc);
        const int a_t0 = first_transposed_slab(p.a_tr, p.a_half, P, nkb);
        const int b_t0 = first_transposed_slab(p.b_tr, p.b_half, bc, nkb);
        if (!mbar_wait_warp(bar_tempty + 8 * acc, aph ^ 1u, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        // K slabs in up to three ranges of fixed operand orientation.
        const int t1 = a_t0 < b_t0 ? a_t0 : b_t0, t2 = a_t0 < b_t0 ? b_t0 : a_t0;
        ok = mma_slabs<BF16, false, false>(0, t1, kc, d, sA, sB, bar_full, bar_empty, p.status);
        if (ok)
          ok = a_t0 <= b_t0 ? mma_slabs<BF16, true, false>(t1, t2, kc, d, sA, sB, bar_full, bar_empty, p.status)
                            : mma_slabs<BF16, false, true>(t1, t2, kc, d, sA, sB, bar_full, bar_empty, p.status);
        if (ok) ok = mma_slabs<BF16, true, true>(t2, nkb, kc, d, sA, sB, bar_full, bar_empty, p.status);
        if (!ok) break;
        if (elect_one()) mma_commit_pair(bar_tfull + 8 * acc, kPair);
        __syncwarp();
      }
      // All MMAs issued by the elected lane complete before TMEM is freed.
      if (elect_one()) mma_commit_pair(bar_drain, 0x1);
      __syncwarp();
      mbar_wait_warp(bar_drain, 0u, p.status);
    }
  } else if (warp >= 2 + kEpiWarps || warp == 1) {
    // ---------------- streaming warps (and warp 1 of the odd CTA, which
    // issues no MMAs): rows of another shape group's step a0 (M <- M + G and
    // row norms), then rows of deferred step a7 updates, taken from the
    // pools' counters one at a time until this CTA's producer has issued its
    // last copy; the rest is left for the pool kernels that follow the GEMM
    // launches ----------------
    auto producer_done = [&]() {
      uint32_t fin = 0;
      if (lane == 0) fin = *reinterpret_cast<volatile uint32_t*>(prod_done);
      return __shfl_sync(0xffffffffu, fin, 0) != 0u;
    };
    bool stop = false;
    if (p.pool.total > 0) {
      for (;;) {
        if (producer_done()) {
          stop = true;
          break;
        }
        const long long row = accum_pool_next(p.pool);
        if (row >= p.pool.total) break;
        // Evict-first for M too: the GEMM's operand panels keep L2.
        if (p.pool.grad_dtype == kBF16)
          accum_pool_row<kBF16, kSideUnrollBF16, kSideEvict>(p.pool, row);
        else
          accum_pool_row<kF32, kSideUnrollF32, kSideEvict>(p.pool, row);
      }
    }
    if (!stop && p.spool.total > 0) {
      for (;;) {
        if (producer_done()) break;
        const long long row = scatter_pool_next(p.spool);
        if (row >= p.spool.total) break;
        scatter_pool_row<kSideUnrollScatter>(p.spool, row);
      }
    }
  } else {
    // ---------------- epilogue warps 2 .. 2 + kEpiWarps - 1 ----------------
    const int quad = warp % 4;  // TMEM lanes 32 quad .. 32 quad + 31
    const int col_lo = ((warp - 2) / 4) * (BN * 4 / kEpiWarps);  // this warp's columns of the tile
    constexpr int kChunks = BN * 4 / kEpiWarps / 32;  // 32-column chunks per warp and tile
    const uint32_t my_staging = staging + static_cast<uint32_t>(warp - 2) * Smem::kWarpStagingBytes;
    const bool sym = p.mode == kSymLower;
    // Outputs of a staged chunk: the tile itself, and its transpose (the mirror
    // of a symmetric result, or outT).
    const bool want_n = p.out != nullptr;
    const bool want_t_any = sym || p.outT != nullptr;
    const bool tma_ok = (!want_n || p.tma_out) && (!want_t_any || (sym ? p.tma_out : p.tma_outT));
    const CUtensorMap* map_t = sym ? &tmOut : &tmOutT;
    uint32_t staged = 0;    // chunks this warp has staged
    uint32_t fast_run = 0;  // of them, the last ones staged by the fast path (one 2 KB half each)
    uint32_t tc = 0;
    for (int u = cluster; u < p.total_units; u += nclusters, ++tc) {
      const int bidx = p.reverse ? p.batch - 1 - u / p.units_per_mat : u / p.units_per_mat;
      int P, bc;
      unit_coords(p, u % p.units_per_mat, P, bc);
      const int bi = 2 * P + static_cast<int>(rank);
      const uint32_t acc = tc & 1u, aph = (tc >> 1) & 1u;
      // The transposed box of this tile: outT, or the mirror of a symmetric
      // result (a half-stored one is mirrored on the diagonal super-tiles only).
      const bool want_t = sym ? (!p.out_half || (P == bc && !p.diag_full)) : p.outT != nullptr;
      // Chunks above the diagonal are skipped, and chunks on it are written as
      // symmetric boxes, unless the diagonal super-tile is written whole.
      const bool tri = sym && !p.diag_full;
      const int row0 = bi * BM + quad * 32;
      const int r = row0 + lane;
      // Rectangular products without C (Q Y at the restart and at the end):
      // every chunk of this warp is written once as a plain box, so the next
      // chunk's TMEM load can run while the current one is staged and stored,
      // and the warp's two 2 KB staging boxes alternate, a chunk waiting only
      // for the bulk store of the chunk two back.  (Measured per role: these
      // products 8-10 % faster at s = 512.  Taken for the off-diagonal tiles
      // of symmetric products too, it made those 2-4 % slower: switching to
      // and from the mirrored path of their diagonal tiles waits for every
      // store.)  Only the other path loads C, so its registers are never live
      // here.
      const bool fast = p.mode == kRect && p.C == nullptr && tma_ok && !want_t && row0 < p.M;
      const uint32_t tbase = tmem + acc * BN + (static_cast<uint32_t>(quad * 32) << 16);
      if (fast) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * acc, aph, p.status))) break;
        tc_fence_after();
        const int nact = min(kChunks, (p.N - bc * BN - col_lo + 31) / 32);  // chunks with c0 < N
        const uint4 no_c[4] = {};
        uint32_t v[32];
        if (nact > 0) {
          tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(col_lo), v);
          tmem_ld_wait();
          tmem_regs_ready(v);
        }
#pragma unroll 1
        for (int i = 0; i < kChunks; ++i) {
          if (i >= nact) break;
          const int c0 = bc * BN + col_lo + 32 * i;
          uint32_t hp[16];
          chunk_values<BF16, false>(p, bidx, r, c0, v, no_c, hp);
          // The next chunk's TMEM load runs while this one is staged and stored.
          if (i + 1 < nact) tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(col_lo + 32 * (i + 1)), v);
          const uint32_t buf = my_staging + (staged & 1u) * Smem::kStageBoxBytes;
          const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
          // The half written now was read by the store two chunks back; when the
          // previous chunk came from the other path, its group may have read
          // both halves, so every group must be done.
          if (lane == 0) {
            if (fast_run >= 1) {
              if (staged >= 2) bulk_wait_read_1();
            } else if (staged >= 1) {
              bulk_wait_read_0();
            }
          }
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            st_shared_v4(buf + lane * 64 + ((static_cast<uint32_t>(q) ^ sw) << 4), hp[4 * q], hp[4 * q + 1],
                         hp[4 * q + 2], hp[4 * q + 3]);
          fence_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmOut, buf, c0, row0, bidx);
            bulk_commit();
          }
          ++staged;
          ++fast_run;
          if (i + 1 < nact) {
            tmem_ld_wait();
            tmem_regs_ready(v);
          }
        }
      } else {
        // Chunks this warp writes: inside the matrix, rows in range, and not
        // wholly above the diagonal of a triangle-only result.
        auto writes = [&](int i) {
          const int c0 = bc * BN + col_lo + 32 * i;
          return c0 < p.N && !(tri && row0 + 31 < c0) && row0 < p.M;
        };
        // C of the first chunk is loaded before the accumulator is ready, and
        // each chunk loads the next one's while it is processed.  The loop
        // stays rolled: one copy of the chunk code (TMEM load, epilogue
        // values, staging of the box, its transpose or a symmetric diagonal
        // box, bulk stores) instead of four.
        uint4 cv[4] = {}, cv_next[4] = {};
        if (writes(0)) prefetch_c(p, bidx, r, bc * BN + col_lo, cv);
        if (!__all_sync(0xffffffffu, mbar_wait(bar_tfull + 8 * acc, aph, p.status))) break;
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < kChunks; ++i) {
          const int cc = col_lo + 32 * i;
          const int c0 = bc * BN + cc;
          if (c0 >= p.N) break;
          if (i + 1 < kChunks && writes(i + 1)) prefetch_c(p, bidx, r, c0 + 32, cv_next);
          if (writes(i)) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + static_cast<uint32_t>(cc), v);
            tmem_ld_wait();
            uint32_t hp[16];
            chunk_values<BF16, true>(p, bidx, r, c0, v, cv, hp);
            const uint32_t buf = my_staging;
            const uint32_t sw = static_cast<uint32_t>((lane >> 1) & 3);
            if (!tma_ok) {
              store_chunk_scalar(p, bidx, r, c0, row0, hp, want_t);
            } else if (tri && row0 <= c0 + 31) {
              fast_run = 0;
              diag_chunk(buf, sw, lane, staged, hp);
              if (lane == 0) {
                tma_store_3d(&tmOut, buf, c0, row0, bidx);
                bulk_commit();
              }
              ++staged;
            } else {
              fast_run = 0;
              // Stage the box (and its transpose) in swizzled shared memory,
              // then one lane writes them with bulk tensor stores.
              if (lane == 0 && staged >= 1) bulk_wait_read_0();
              __syncwarp();
              if (want_n) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                  st_shared_v4(buf + lane * 64 + ((static_cast<uint32_t>(q) ^ sw) << 4), hp[4 * q], hp[4 * q + 1],
                               hp[4 * q + 2], hp[4 * q + 3]);
              }
              if (want_t) {
                const uint32_t tbuf = buf + Smem::kStageBoxBytes;
                const uint32_t lo = static_cast<uint32_t>(lane & 7) << 1, hi = static_cast<uint32_t>(lane >> 3);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  st_shared_u16(tbuf + j * 64 + (((hi ^ ((j >> 1) & 3)) << 4) | lo), half_bits(hp, j));
              }
              fence_async_shared();
              __syncwarp();
              if (lane == 0) {
                if (want_n) tma_store_3d(&tmOut, buf, c0, row0, bidx);
                if (want_t) tma_store_3d(map_t, buf + Smem::kStageBoxBytes, row0, c0, bidx);
                bulk_commit();
              }
              ++staged;
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) cv[q] = cv_next[q];
        }
      }
      tc_fence_before();
      mbar_arrive_cluster(map_to_rank(bar_tempty + 8 * acc, 0));
    }
    // Every bulk store has finished before the CTA (and its shared memory)
    // goes away.
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }
  tc_fence_before();
  // Neither CTA leaves while its peer may still multicast into its shared
  // memory or arrive on its barriers.
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// The bounded wait on its own: one thread initialises an mbarrier (count 1),
// optionally arrives on it, and waits for its first phase with the GEMM's
// bounded wait and the given limit.  Without the arrival nothing completes the
// phase, so the wait runs out, records kDevTimeout and the kernel returns.  No
// copy or MMA is ever in flight here.
__global__ void __launch_bounds__(32, 1) wait_probe_kernel(unsigned long long limit_ns, int arrive,
                                                           unsigned* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (arrive) mbar_arrive_local(b);
  mbar_wait(b, 0u, status, limit_ns);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* q_fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q_fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(q_fn);
  });
  return fn;
}

// 3-D tensor map over [batch][rows][cols] fp16 for the epilogue's bulk
// stores: box 32 x 32 x 1 with the 64-byte swizzle of the staging buffers.
bool make_store_map(CUtensorMap* map, const __half* ptr, long long bstride, int ld, int rows, int cols,
                    int batch, CUtensorMapDataType dt) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, static_cast<cuuint64_t>(bstride) * 2u};
  cuuint32_t box[3] = {32u, 32u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, dt, 3, const_cast<__half*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An output can take the bulk-store path when its base is 16-byte aligned and
// its row pitch and batch stride are multiples of 8 elements.
bool storable(const __half* ptr, int ld, long long bstride, int rows, int batch) {
  if (ptr == nullptr) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0 || ld % 8 != 0 || bstride % 8 != 0) return false;
  return batch == 1 || bstride >= static_cast<long long>(ld) * rows;
}

// 3-D tensor map over [batch][rows][cols] fp16 with row pitch `ld` elements,
// box = 64 columns x box_rows rows x 1 matrix, 128-byte swizzle, zero fill.
bool make_map(CUtensorMap* map, const __half* ptr, long long bstride, int ld, int rows, int cols, int batch,
              int box_rows, CUtensorMapDataType dt) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(batch)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2u, static_cast<cuuint64_t>(bstride) * 2u};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = fn(map, dt, 3, const_cast<__half*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Whether self-products write their diagonal super-tiles whole
// (DION3_DIAG_FULL, read once; default on).
bool diag_full_enabled() {
  static const bool on = [] {
    const char* v = getenv("DION3_DIAG_FULL");
    return v == nullptr || atoi(v) != 0;
  }();
  return on;
}

// Clusters of this kernel that fit on the device at once (persistent grid).
int max_active_clusters(int dev) {
  static int cached[64] = {0};
  if (cached[dev & 63] == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = Smem::kDyn;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_tcgen05_kernel<false>, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      int sms = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      n = sms > 1 ? sms / 2 : 1;
    }
    cached[dev & 63] = n;
  }
  return cached[dev & 63];
}

}  // namespace

cudaError_t launch_wait_probe(bool arrive, unsigned long long limit_ns, unsigned* status, cudaStream_t s) {
  return launch_kernel(false, wait_probe_kernel, dim3(1), dim3(32), 0, s, limit_ns, arrive ? 1 : 0, status);
}

bool gemm_check(const GemmDesc& g, const char** why) {
  auto fail = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.batch <= 0) return fail("gemm: empty dimension");
  if (g.A == nullptr || g.B == nullptr) return fail("gemm: null operand");
  if ((reinterpret_cast<uintptr_t>(g.A) | reinterpret_cast<uintptr_t>(g.B)) & 15u)
    return fail("gemm: operands must be 16-byte aligned");
  if (g.lda % 8 || g.ldb % 8 || g.a_bstride % 8 || g.b_bstride % 8)
    return fail("gemm: operand pitches must be multiples of 8 elements");
  if (g.lda < (g.a_tr ? g.M : g.K) || g.ldb < (g.b_tr ? g.N : g.K)) return fail("gemm: operand pitch smaller than its row");
  if ((g.a_tr && g.a_half) || (g.b_tr && g.b_half)) return fail("gemm: an operand is either transposed or half-stored");
  if (g.mode == kSymLower && (g.M != g.N || g.out == nullptr)) return fail("gemm: symmetric mode needs M == N and out");
  if (g.mode == kRect && g.out == nullptr && g.outT == nullptr) return fail("gemm: no output");
  if (g.M > (1 << 24) || g.N > (1 << 24)) return fail("gemm: dimension too large");
  if (g.elem != kF16 && g.elem != kBF16) return fail("gemm: element type must be fp16 or bf16");
  if (g.a_half && g.M != g.K) return fail("gemm: a half-stored symmetric A needs M == K");
  if (g.b_half && g.N != g.K) return fail("gemm: a half-stored symmetric B needs N == K");
  if (g.out_half && g.mode != kSymLower) return fail("gemm: a half-stored output needs the symmetric mode");
  return true;
}

cudaError_t launch_gemm(const GemmDesc& g, unsigned* dev_status, cudaStream_t s) {
  const bool bf16 = g.elem == kBF16;
  const bool has_c = g.C != nullptr && g.beta != 0.0f;
  auto kern = bf16 ? gemm_tcgen05_kernel<true> : gemm_tcgen05_kernel<false>;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  static std::once_flag once[64][2];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63][bf16 ? 1 : 0], [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem::kDyn);
  });
  if (attr_err != cudaSuccess) return attr_err;

  // Operand maps: 128-row boxes for K-major tiles, and 64 x 64 boxes of the
  // same matrices for the MN-major tiles of half-stored operands (built for
  // every launch, so the kernel never sees an unset map).
  // An operand given as its transpose is stored [K][M] (or [K][N]): both of
  // its maps describe that storage (only the 64 x 64 one is used).
  CUtensorMap ta, tb, tat, tbt;
  const int a_rows = g.a_tr ? g.K : g.M, a_cols = g.a_tr ? g.M : g.K;
  const int b_rows = g.b_tr ? g.K : g.N, b_cols = g.b_tr ? g.N : g.K;
  if (!make_map(&ta, g.A, g.a_bstride, g.lda, a_rows, a_cols, g.batch, g.a_tr ? BK : BM, dt)) return cudaErrorInvalidValue;
  if (!make_map(&tb, g.B, g.b_bstride, g.ldb, b_rows, b_cols, g.batch, g.b_tr ? BK : BN / 2, dt)) return cudaErrorInvalidValue;
  if (!make_map(&tat, g.A, g.a_bstride, g.lda, a_rows, a_cols, g.batch, BK, dt)) return cudaErrorInvalidValue;
  if (!make_map(&tbt, g.B, g.b_bstride, g.ldb, b_rows, b_cols, g.batch, BK, dt)) return cudaErrorInvalidValue;

  CUtensorMap to, tt;
  memset(&to, 0, sizeof to);
  memset(&tt, 0, sizeof tt);
  int tma_out = 0, tma_outT = 0;
  if (storable(g.out, g.ld_out, g.out_bstride, g.M, g.batch) &&
      make_store_map(&to, g.out, g.out_bstride > 0 ? g.out_bstride : static_cast<long long>(g.ld_out) * g.M,
                     g.ld_out, g.M, g.N, g.batch, dt))
    tma_out = 1;
  if (g.mode == kRect && storable(g.outT, g.ld_outT, g.outT_bstride, g.N, g.batch) &&
      make_store_map(&tt, g.outT, g.outT_bstride > 0 ? g.outT_bstride : static_cast<long long>(g.ld_outT) * g.N,
                     g.ld_outT, g.N, g.M, g.batch, dt))
    tma_outT = 1;

  GemmParams p{};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.mode = g.mode;
  p.tiles_r = (g.M + BM - 1) / BM;
  p.tiles_c = (g.N + BN - 1) / BN;
  p.pairs_r = (p.tiles_r + 1) / 2;
  if (g.mode == kSymLower) {
    // BN == 2 BM: super-tile rows and column tiles have the same 256 extent.
    p.units_per_mat = p.pairs_r * (p.pairs_r + 1) / 2;
  } else {
    p.units_per_mat = p.pairs_r * p.tiles_c;
  }
  const long long total = static_cast<long long>(p.units_per_mat) * g.batch;
  if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  p.total_units = static_cast<int>(total);
  p.alpha = g.alpha;
  p.beta = g.beta;
  p.gamma = g.gamma;
  p.C = has_c ? g.C : nullptr;  // beta = 0: C is not read
  p.c_bs = g.c_bstride;
  p.ldc = g.ldc;
  p.out = g.out;
  p.out_bs = g.out_bstride;
  p.ld_out = g.ld_out;
  p.outT = g.outT;
  p.outT_bs = g.outT_bstride;
  p.ld_outT = g.ld_outT;
  p.tma_out = tma_out;
  p.tma_outT = tma_outT;
  p.batch = g.batch;
  p.reverse = g.reverse ? 1 : 0;
  p.a_half = g.a_half ? 1 : 0;
  p.a_tr = g.a_tr ? 1 : 0;
  p.b_tr = g.b_tr ? 1 : 0;
  p.b_half = g.b_half ? 1 : 0;
  p.out_half = g.out_half ? 1 : 0;
  // A A^T (+ beta C with C = A half-stored, + gamma I): exactly symmetric as
  // computed, so the diagonal super-tiles of a half-stored result need no mirror.
  const bool self = g.A == g.B && g.lda == g.ldb && g.a_bstride == g.b_bstride && g.a_tr == g.b_tr &&
                    g.a_half == g.b_half;
  const bool c_sym = g.C == nullptr || g.beta == 0.0f ||
                     (g.a_half && g.C == g.A && g.ldc == g.lda && g.c_bstride == g.a_bstride);
  p.diag_full = (g.mode == kSymLower && g.out_half && self && c_sym && diag_full_enabled()) ? 1 : 0;
  p.status = dev_status;
  if (g.pool != nullptr) p.pool = *g.pool;
  if (g.spool != nullptr) p.spool = *g.spool;

  const int clusters = static_cast<int>(std::min<long long>(total, max_active_clusters(dev)));
  const int grid = 2 * clusters;
  return launch_kernel(pdl_enabled(), kern, dim3(grid), dim3(kThreads), Smem::kDyn, s, ta, tb, tat, tbt, to, tt, p);
}

}  // namespace dion3
