// nx_score_tc.cu -- fused direct scores + Nexus walk + selection keys on the tensor cores
// (bf16 caches, head_dim 64 or 128, W in {16, 32, 64}, contiguous or paged).
//
// Nexus Sampling paper, §2.1 Eq. (1) (b = 1), §2.2 Eqs. (2)-(5), §2.3 (keys of Eq. (6),
// n = 1). One persistent, cooperatively launched kernel, one CTA per SM, holding one or
// two pipelines ("teams"). A pipeline takes chunks of up to 8 tiles of 128 cached rows of
// one slice (the chunk schedule below) and:
//   1. a TMA producer thread stages each K tile in a ring of shared-memory stages
//      (128-byte swizzle, one box per 64-element column block -- per page when paged);
//   2. an MMA thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32), M = 128 rows,
//      N = W window rows, K = head_dim, against Qbar -- a bf16 tensor, the head average of
//      a bf16 model -- so the logits are the exact products summed in fp32. A chunk's
//      logits fill one of two or three TMEM buffers (tile t -> columns [t*W, (t+1)*W));
//   3. the epilogue warpgroups (one TMEM lane = one row) take per-column maxima over each
//      warp's rows, write e = exp((l - max)/sqrt(d)) back to TMEM, and store the chunk
//      record (chunk maxima, sums, the H x H Gram of the walk rows); a publisher warp
//      makes it visible and counts it into the slice;
//   4. a merge warp waits (bounded) until every chunk of the slice is counted in, merges
//      the slice's records, runs the walk recurrence (gamma_t = 1 + sum_{u<t} gamma_u
//      <P_t, P_u>, the rank-1 form of Eq. (4)) and hands the per-column weights over;
//   5. the epilogue turns the chunk's TMEM e values into a, c~, w and the order key of
//      every row (one chunk behind step 3, so the slice wait overlaps the next chunk).
// K is read from HBM exactly once; nothing but one key (and optional outputs) per row
// goes back to memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "nx_internal.cuh"

namespace nx {
namespace tc {

// A CTA holds one or two teams; each team is a complete pipeline of its own (its own
// chunks, shared-memory region, barriers and half of TMEM) and acts as one "virtual CTA"
// of the chunk schedule. Warp roles of a team whose epilogue has NWG warpgroups: warps
// [0, 4 NWG) run the epilogue, then come the TMA producer, the MMA issuer, the merge warp
// and the publisher. NWG = 4: one team holding all 512 TMEM columns. NWG = 2: two teams of
// 256 columns each, whose epilogues fill one another's waits (a kernel that allocates
// TMEM runs one CTA per SM, so the overlap has to come from inside the CTA).
template <int NWG>
struct Roles {
  static constexpr int kEpiWarps = 4 * NWG;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kProducerWarp = kEpiWarps;
  static constexpr int kMmaWarp = kEpiWarps + 1;
  static constexpr int kMergeWarp = kEpiWarps + 2;
  static constexpr int kPublishWarp = kEpiWarps + 3;
  static constexpr int kThreads = kEpiThreads + 128;          // one team
  static constexpr int kTeams = NWG == 2 ? 2 : 1;
  static constexpr int kBlockThreads = kTeams * kThreads;
  static constexpr uint32_t kTmemCols = 512u / kTeams;      // one team's share
  static constexpr int kMaxChunkTiles = 8;         // the pass-2 partials are sized for it
  static constexpr int kGroup = 32;                // records per bulk copy of the merge
};
constexpr int kTileRows = 128;
// Who folds a chunk's max shift into the per-column weights: the merge warp (off the
// epilogue's path) for windows of up to 32 rows; the epilogue for W = 64, whose merge warp
// is already the slower side (measured).
template <int W>
constexpr bool kFoldInMerge = W <= 32;
constexpr long long kWaitLimit = 1LL << 22;   // mbarrier polls before giving up
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
  nx_cache c;
  nx_params p;
  const unsigned char* qimg;   // [slices] shared-memory images of the bf16 window queries
  uint32_t tmem_cols;      // columns the CTA allocates (all 512; split between its teams)
  int nbuf;                // TMEM buffers (2: the next chunk's MMAs overlap this epilogue)
  long long* trace;        // optional phase trace: [grid][kTraceEvents][2] (null: off)
  float* partial;          // [slices][maxc][stride]
  int* arrive;             // [slices] chunks whose records are published
  const int32_t* newlen;   // [slices]
  ScoreOut out;
  int32_t* dev_status;
  int tiles_per_chunk;
  int maxc;                // chunk ids per slice
  int stride;              // floats per partial record
  long long total_ids;     // slices * maxc
  int slices;
  // 0: one pass (chunk records merged across CTAs through the slice barrier);
  // 1: records only (each TMEM buffer is freed once its chunk's record is stored);
  // 2: the pass after 1: the records are complete, nothing waits on another CTA
  int pass;
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase; false (and NX_DEV_TIMEOUT) when it gives up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* dev_status) {
  for (long long i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(dev_status, NX_DEV_TIMEOUT);
  return false;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row core groups
// 1024 bytes apart (SBO), version 1 (bits 46-47), layout type 2 = SWIZZLE_128B.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major.
template <int N>
__device__ __forceinline__ constexpr uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(kTileRows >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 16 columns of 32-bit TMEM words into registers (and back).
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  uint32_t r[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[i]);
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// N (4, 8 or 16) consecutive TMEM columns of this thread's lane, issued without a wait
// (tmem_ld_wait() makes them usable).
template <int N>
__device__ __forceinline__ void tmem_ld_issue(uint32_t taddr, uint32_t* r) {
  if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else {
    tmem_ld16_nowait(taddr, r);
  }
}

// N (4, 8 or 16) consecutive TMEM columns of this thread's lane, loaded and awaited.
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, float* v) {
  uint32_t r[N];
  if constexpr (N == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
  } else {
    tmem_ld16_nowait(taddr, r);
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = __uint_as_float(r[i]);
}

template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const float* v) {
  uint32_t r[N];
#pragma unroll
  for (int i = 0; i < N; ++i) r[i] = __float_as_uint(v[i]);
  if constexpr (N == 4) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
  } else if constexpr (N == 8) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(
                     taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                 "r"(r[7])
                 : "memory");
  } else {
    tmem_st16(taddr, v);
  }
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier of a team's epilogue warps (barrier 1 + team; __syncthreads uses 0).
template <int NWG>
__device__ __forceinline__ void epi_sync(int bar_id) {
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(Roles<NWG>::kEpiThreads) : "memory");
}

// Warp maximum of a float through its monotone integer image (one redux instruction).
__device__ __forceinline__ float warp_max_redux(float x) {
  uint32_t b = __float_as_uint(x);
  uint32_t k = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  uint32_t r;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(k));
  return __uint_as_float((r & 0x80000000u) ? (r & 0x7FFFFFFFu) : ~r);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// Merging chunk statistics
// ---------------------------------------------------------------------------
constexpr int kMaxChunksPerSlice = 256;   // grid choice

// A record holds, for the rows it covers: per window row w the maximum raw logit m_w and
// sum_j exp((l_wj - m_w)/sqrt(d)) (natural-log units), and per walk-row pair (p, q) the
// Gram sum_j exp((l_pj - m_p)/sqrt(d)) exp((l_qj - m_q)/sqrt(d)). Records of one slice sit
// contiguously in global memory, `stride` floats apart, in chunk order; the merge warp
// below combines them in that fixed order.

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int W, int D, int NWG>
struct Smem {
  using R = Roles<NWG>;
  // K tiles in flight: 128-160 KB of them per SM
  static constexpr int kStages =
      NWG == 4 ? (D == 128 ? (W == 64 ? 4 : 5) : 8) : (D == 128 ? 2 : 4);
  static constexpr int KB = D / 64;                       // 128-byte column blocks per row
  static constexpr int kRegionA = kTileRows * 128;        // one column block of a K tile
  static constexpr int kTileBytes = KB * kRegionA;
  static constexpr int kRegionB = W * 128;                // one column block of Qbar
  static constexpr int kQBytes = KB * kRegionB;           // bf16 query image
  static constexpr int kRec = 2 * W + kMaxPairs;          // floats of one chunk record
  static constexpr int kRedStride = W + kMaxPairs;        // one warp's partial reductions
  static constexpr int kOffK = 0;
  static constexpr int kOffQ = kStages * kTileBytes;
  static constexpr int kOffBar = kOffQ + kQBytes;         // up to 32 mbarriers
  static constexpr int kOffMisc = kOffBar + 256;          // tmem slot + control words
  static constexpr int kOffRed = kOffMisc + 64;           // [kEpiWarps][kRedStride]
  static constexpr int kOffMc = kOffRed + R::kEpiWarps * kRedStride * 4;   // [3][W] chunk maxima
  static constexpr int kOffCa = kOffMc + 3 * W * 4;       // [3][W] a coefficients
  static constexpr int kOffCc = kOffCa + 3 * W * 4;       // [3][kMaxWalk] walk coefficients
  // [3][4][W] per TMEM buffer, lane quarter and column: the maximum over that quarter's
  // rows of the chunk (the shift of its e values)
  static constexpr int kOffMw = kOffCc + 3 * kMaxWalk * 4;
  // [kEpiWarps][CW + kMaxWalk] each warp's pass-2 weights for its columns and walk rows
  static constexpr int kWca = W / NWG + kMaxWalk;
  static constexpr int kOffWca = kOffMw + 3 * 4 * W * 4;
  static constexpr int kMrec = 2 * W + kMaxWalk;          // merged: max, normaliser, walk
  static constexpr int kOffMrec = kOffWca + R::kEpiWarps * kWca * 4;   // [3][kMrec]
  static constexpr int kOffMs = kOffMrec + 3 * kMrec * 4; // merge warp scratch [2][W]
  static constexpr int kOffPart = kOffMs + 2 * W * 4;
  // pass-2 partial a per tile, warpgroup and row; the walk term per tile and row
  static constexpr int kOffCt = kOffPart + R::kMaxChunkTiles * NWG * kTileRows * 4;
  // merge staging: kGroup chunk records as laid out in global memory
  static constexpr int kRecStride = (kRec + 3) / 4 * 4;
  static constexpr int kOffStage = kOffCt + R::kMaxChunkTiles * kTileRows * 4;
  static constexpr int kBytes = kOffStage + R::kGroup * kRecStride * 4;
  static constexpr int kTeamBytes = (kBytes + 1023) / 1024 * 1024;   // one team's region
  static constexpr int kAlloc = R::kTeams * kTeamBytes + 1024;     // + 1024-byte alignment
};

// The chunk schedule. The chunks of all slices are numbered in slice order (a slice that
// is empty or was rejected has none), and chunk number x goes to CTA x mod grid. In the
// one-pass mode a slice has at most grid chunks, so a CTA holds at most one chunk of any
// slice, and it takes its chunks in increasing slice order: that keeps the slice barrier
// deadlock-free (the earliest unfinished slice never waits on a later one), and however
// ragged the lengths, the CTAs' chunk counts differ by at most one. (The two-pass mode,
// which waits on no other CTA, allows more chunks per slice than CTAs.) Every warp of every role walks the same
// sequence itself, warp-collectively: 32 slices at a time, one per lane, with a warp
// scan of their chunk counts.
struct Sched {
  int cta, ncta;     // this (virtual) CTA and how many there are
  long long first;   // chunk number of the first chunk of slice `base`
  int base;          // first slice of the current batch
  uint32_t mask;     // lanes whose slice has a chunk left for this CTA
  int k, T, n;       // this lane's slice: the next chunk index for this CTA, its length,
                     // its chunk count
};

__device__ __forceinline__ void sched_init(Sched& S, int cta, int ncta) {
  S.cta = cta;
  S.ncta = ncta;
  S.first = 0;
  S.base = -32;
  S.mask = 0;
  S.k = 0;
  S.T = 0;
  S.n = 0;
}

// Warp-collective: the next chunk of this CTA; false once there is none.
__device__ __forceinline__ bool sched_next(const Args& A, Sched& S, int chunk_rows,
                                           int& slice, int& k, int& T) {
  const int lane = threadIdx.x & 31;
  while (S.mask == 0) {
    S.base += 32;
    if (S.base >= A.slices) return false;
    const int sl = S.base + lane;
    int nl = -1, t = 0, n = 0;
    if (sl < A.slices) {
      nl = __ldg(&A.newlen[sl]);
      t = __ldg(&A.c.lens[sl]);
    }
    if (sl < A.slices && nl >= 0) n = (t + chunk_rows - 1) / chunk_rows;
    else t = 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long f = S.first + (incl - n);
    int kk = S.cta - (int)(f % S.ncta);
    if (kk < 0) kk += S.ncta;
    S.k = kk;
    S.T = t;
    S.n = n;
    S.mask = __ballot_sync(0xffffffffu, kk < n);
    S.first += __shfl_sync(0xffffffffu, incl, 31);
  }
  const int j = __ffs(S.mask) - 1;
  slice = S.base + j;
  k = __shfl_sync(0xffffffffu, S.k, j);
  T = __shfl_sync(0xffffffffu, S.T, j);
  // a slice with more chunks than CTAs gives this CTA chunks k, k + ncta, ... (only in
  // the two-pass mode, which has no slice barrier)
  const int n_j = __shfl_sync(0xffffffffu, S.n, j);
  if ((threadIdx.x & 31) == j) S.k += S.ncta;
  if (k + S.ncta >= n_j) S.mask &= S.mask - 1;
  return true;
}

// A flag that any thread may set, read by lane 0 and broadcast (warp-uniform).
__device__ __forceinline__ int warp_flag(volatile int* f) {
  int v = 0;
  if ((threadIdx.x & 31) == 0) v = *f;
  return __shfl_sync(0xffffffffu, v, 0);
}

constexpr int kTraceEvents = 1024;

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Phase trace (diagnostics, off unless a buffer is installed): event e of this CTA gets
// (tag, globaltimer ns); the last three slots hold kernel-level marks.
__device__ __forceinline__ void trace_ev(const Args& A, int cta, int& n, int tag) {
  if (A.trace && n < kTraceEvents - 3) {
    long long* t = A.trace + ((long long)cta * kTraceEvents + n) * 2;
    t[0] = tag;
    t[1] = global_ns();
    ++n;
  }
}

// the same for the MMA issuer (slots from 512) and the TMA producer (slots from 768)
__device__ __forceinline__ void trace_role(const Args& A, int cta, int base, int& n, int tag) {
  if (A.trace && base + n < kTraceEvents - 3 && n < 256) {
    long long* t = A.trace + ((long long)cta * kTraceEvents + base + n) * 2;
    t[0] = tag;
    t[1] = global_ns();
    ++n;
  }
}

// kernel-level marks in the last three trace slots of the CTA: entry, setup done, exit
__device__ __forceinline__ void trace_mark(const Args& A, int cta, int slot, int tag) {
  if (A.trace) {
    long long* t = A.trace + ((long long)cta * kTraceEvents + kTraceEvents - 3 + slot) * 2;
    t[0] = tag;
    t[1] = global_ns();
  }
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One chunk as the epilogue sees it.
struct Chunk {
  int slice, k, T, nchunks, j0, ntiles, l, s, h;
  uint32_t b;          // TMEM buffer
  uint32_t use;        // how many times this buffer was used before
  uint32_t cnt;        // this pipeline's chunk number
};

__device__ __forceinline__ Chunk make_chunk(const Args& A, int slice, int k, int T,
                                            int chunk_rows, uint32_t cc, int nbuf) {
  Chunk ch;
  ch.slice = slice;
  ch.k = k;
  ch.T = T;
  ch.nchunks = (ch.T + chunk_rows - 1) / chunk_rows;
  ch.j0 = ch.k * chunk_rows;
  ch.ntiles = min(A.tiles_per_chunk, (ch.T - ch.j0 + kTileRows - 1) / kTileRows);
  slice_coords(A.c, ch.slice, ch.l, ch.s, ch.h);
  ch.b = cc % nbuf;
  ch.use = cc / nbuf;
  ch.cnt = cc;
  return ch;
}

// Epilogue state shared by the passes. The W query columns are split over the NWG
// warpgroups (warpgroup g owns columns [g W/NWG, (g+1) W/NWG)); the four warps of a
// warpgroup own the 128 rows of a tile (TMEM lanes). The walk rows, the last H <= W/NWG
// columns, belong to the last warpgroup.
template <int W, int D, int NWG>
struct Epi {
  static constexpr int CW = W / NWG;
  static constexpr int kWalkWg = NWG - 1;
  // tiles whose TMEM loads share one wait, per pass (two measured slower than one: the
  // passes are bound by arithmetic and barriers, not by the load latency)
  static constexpr int P1a = 1, P1b = 1, P2 = 1;
  // per-column coefficients kept in registers across the tiles (when few enough)
  static constexpr bool kHoist = CW <= 8;
  const Args& A;
  uint8_t* sm;
  uint32_t tmem;
  uint32_t buf_cols;
  float cl2;
  int H;
  int tid;              // thread index within the team
  int vcta, vgrid;      // this team's place in the chunk schedule
  int bar_id;           // the team epilogue's named barrier
  int warp, lane, wg, lg, col0;
  int nev = 0;          // trace events written (thread 0)
  __device__ Epi(const Args& a, uint8_t* s, uint32_t t, uint32_t bc, float c2, int h, int ti,
                 int vc, int vg, int bid)
      : A(a), sm(s), tmem(t), buf_cols(bc), cl2(c2), H(h), tid(ti), vcta(vc), vgrid(vg),
        bar_id(bid) {
    warp = tid >> 5;
    lane = tid & 31;
    wg = warp >> 2;
    lg = warp & 3;
    col0 = wg * CW;
  }
  __device__ float* red() { return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffRed); }
  __device__ float* mc(uint32_t b) {
    return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffMc) + b * W;
  }
  __device__ float* ca(uint32_t b) {
    return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffCa) + b * W;
  }
  __device__ float* cc(uint32_t b) {
    return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffCc) + b * kMaxWalk;
  }
  __device__ float* mw(uint32_t b) {   // [4][W] lane-quarter maxima of buffer b
    return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffMw) + b * 4 * W;
  }
  __device__ float* wca() {            // this warp's pass-2 weights
    return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffWca) + warp * Smem<W, D, NWG>::kWca;
  }
  __device__ float* apart() { return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffPart); }
  __device__ float* ctp() { return reinterpret_cast<float*>(sm + Smem<W, D, NWG>::kOffCt); }
  __device__ uint32_t taddr(const Chunk& ch, int t) {
    return tmem + ((uint32_t)(lg * 32) << 16) + ch.b * buf_cols + (uint32_t)(t * W + col0);
  }
  __device__ bool row_valid(const Chunk& ch, int t) {
    return ch.j0 + t * kTileRows + lg * 32 + lane < ch.T;
  }
  __device__ bool tile_full(const Chunk& ch, int t) {
    return ch.j0 + (t + 1) * kTileRows <= ch.T;
  }

  // Passes 1a/1b: per-column maxima over this warp's rows, e = exp((l - max)/sqrt(d))
  // written back to TMEM, sums and the walk-row Gram; the chunk's record (the four lane
  // quarters rescaled to the chunk maxima) goes to global memory.
  template <int HT>
  __device__ void stats(const Chunk& ch) {
    constexpr int RS = Smem<W, D, NWG>::kRedStride;
    const bool blocks = A.p.block_size > 1;
    float* m = mc(ch.b);
    float mx[CW];
#pragma unroll
    for (int i = 0; i < CW; ++i) mx[i] = -INFINITY;
    for (int t0 = 0; t0 < ch.ntiles; t0 += P1a) {
      uint32_t r[P1a][CW];
#pragma unroll
      for (int u = 0; u < P1a; ++u)
        if (t0 + u < ch.ntiles) tmem_ld_issue<CW>(taddr(ch, t0 + u), r[u]);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < P1a; ++u) {
        if (t0 + u >= ch.ntiles) break;
        if (kHoist && tile_full(ch, t0 + u)) {   // warp-uniform: no per-row test
#pragma unroll
          for (int i = 0; i < CW; ++i) mx[i] = fmaxf(mx[i], __uint_as_float(r[u][i]));
        } else {
          const bool valid = row_valid(ch, t0 + u);
#pragma unroll
          for (int i = 0; i < CW; ++i)
            mx[i] = fmaxf(mx[i], valid ? __uint_as_float(r[u][i]) : -INFINITY);
        }
      }
    }
    if (tid == 0) trace_ev(A, vcta, nev, 10);
    // The publisher warp reads the previous chunk's lane-quarter partials (mw, red) to
    // build its record; they are overwritten only once it has taken them.
    if (ch.cnt > 0 && lane == 0) {
      uint64_t* bar_rec =
          reinterpret_cast<uint64_t*>(sm + Smem<W, D, NWG>::kOffBar) + 2 * Smem<W, D, NWG>::kStages + 15;
      int* ctl = reinterpret_cast<int*>(sm + Smem<W, D, NWG>::kOffMisc + 16);
      if (!mbar_wait(bar_rec, (ch.cnt - 1) & 1, A.dev_status)) ctl[1] = 1;
    }
    __syncwarp();
    // Each warp shifts its own rows by its own column maxima (no barrier here); the
    // publisher warp rescales the four lane quarters to the chunk maximum for the record,
    // and pass 2 folds the same factor into its weights.
    float* mwq = mw(ch.b) + lg * W;
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      mx[i] = warp_max_redux(mx[i]);
      if (lane == 0) mwq[col0 + i] = mx[i];
    }
    if (tid == 0) trace_ev(A, vcta, nev, 11);
    float z[CW], gp[kMaxPairs], snm[kHoist ? CW : 1];
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      z[i] = 0.f;
      if (kHoist) snm[i] = -mx[i] * cl2;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < kMaxPairs; ++i) gp[i] = 0.f;
    const bool walk_wg = (wg == kWalkWg);
    for (int t0 = 0; t0 < ch.ntiles; t0 += P1b) {
      uint32_t r[P1b][CW];
#pragma unroll
      for (int u = 0; u < P1b; ++u)
        if (t0 + u < ch.ntiles) tmem_ld_issue<CW>(taddr(ch, t0 + u), r[u]);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < P1b; ++u) {
        const int t = t0 + u;
        if (t >= ch.ntiles) break;
        const bool valid = (kHoist && tile_full(ch, t)) || row_valid(ch, t);
        float v[CW];
#pragma unroll
        for (int i = 0; i < CW; ++i) {
          const float sh = kHoist ? snm[i] : -mwq[col0 + i] * cl2;
          const float e = valid ? ex2_approx(fmaf(__uint_as_float(r[u][i]), cl2, sh)) : 0.f;
          v[i] = e;
          z[i] += e;
        }
        tmem_stn<CW>(taddr(ch, t), v);
        if (walk_wg) {
          float ew[kMaxWalk];
          constexpr int NW = HT >= 0 ? HT : kMaxWalk;     // walk columns carried
          if (HT >= 0) {
#pragma unroll
            for (int tt = 0; tt < kMaxWalk; ++tt) ew[tt] = (tt < HT) ? v[CW - HT + tt] : 0.f;
          } else {
#pragma unroll
            for (int tt = 0; tt < kMaxWalk; ++tt) {
              float x = 0.f;
#pragma unroll
              for (int i = 0; i < CW; ++i)
                if (tt < H && i == CW - H + tt) x = v[i];
              ew[tt] = x;
            }
          }
          if (blocks) {
            // b = 32: the walk's inner products are between block rows, the sums over the
            // 32 rows of a block -- this warp's rows (chunks start at multiples of 128);
            // lane 0 carries the block's products
#pragma unroll
            for (int tt = 0; tt < NW; ++tt) {
              const float x = warp_sum(ew[tt]);
              ew[tt] = lane == 0 ? x : 0.f;
            }
          }
#pragma unroll
          for (int tt = 1; tt < (NW > 0 ? NW : 1); ++tt)
#pragma unroll
            for (int uu = 0; uu < tt; ++uu) gp[pair_index(uu, tt)] += ew[uu] * ew[tt];
        }
      }
    }
    tmem_st_wait();
    if (tid == 0) trace_ev(A, vcta, nev, 12);
#pragma unroll
    for (int i = 0; i < CW; ++i) {
      const float x = warp_sum(z[i]);
      if (lane == 0) red()[warp * RS + col0 + i] = x;
    }
    if (walk_wg) {
      constexpr int NP = (HT >= 0) ? (HT * (HT - 1) / 2 > 0 ? HT * (HT - 1) / 2 : 0) : kMaxPairs;
#pragma unroll
      for (int i = 0; i < kMaxPairs; ++i) {
        const float x = (i < NP) ? warp_sum(gp[i]) : 0.f;
        if (lane == 0) red()[warp * RS + W + i] = x;
      }
    }
  }

  // Hand the chunk's partials to the publisher warp: each epilogue warp arrives once its
  // shared-memory stores are issued (the arrive releases them to the publisher).
  __device__ void publish(const Chunk& ch, bool ok, uint64_t* bar_pub) {
    using S = Smem<W, D, NWG>;
    int* ctl = reinterpret_cast<int*>(sm + S::kOffMisc + 16);
    if (!ok && tid == 0) ctl[1] = 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_pub[ch.b]);
  }

  // With one TMEM buffer and W = 64 the epilogue would only wait for the merge warp, and
  // every pipeline works on chunks of the same slice at once: the epilogue warps merge the
  // slice's chunk records themselves, several threads per column.
  __device__ bool epi_merges() const { return !kFoldInMerge<W> && A.nbuf == 1; }

  // Merge the slice's chunk records (from memory) into the merged record of buffer ch.b:
  // per window row the maximum M and the normaliser Z, and the walk coefficients
  // gamma_t / (sum gamma * Z_t) of Eq. (4) in rank-1 form.
  __device__ void merge_records(const Chunk& ch) {
    using S = Smem<W, D, NWG>;
    constexpr int kThreads = Roles<NWG>::kEpiThreads;
    constexpr int P = kThreads / W;            // threads per column (consecutive lanes)
    static_assert(P >= 1 && P <= 32 && (P & (P - 1)) == 0, "threads per column");
    const float* rec = A.partial + (long long)ch.slice * A.maxc * A.stride;
    const int n = ch.nchunks;
    float* out = reinterpret_cast<float*>(sm + S::kOffMrec) + ch.b * S::kMrec;
    float* gm = reinterpret_cast<float*>(sm + S::kOffMs);       // [kMaxPairs] merged Gram
    const int col = tid / P, part = tid % P;
    {
      float mx = -INFINITY;
      for (int r = part; r < n; r += P) mx = fmaxf(mx, rec[(long long)r * A.stride + col]);
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float z = 0.f;
      for (int r = part; r < n; r += P) {
        const float* rr = rec + (long long)r * A.stride;
        z += rr[W + col] * ex2_approx((rr[col] - mx) * cl2);
      }
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      if (part == 0) {
        out[col] = mx;
        out[W + col] = z;
      }
    }
    epi_sync<NWG>(bar_id);
    const int np = H * (H - 1) / 2;
    // whole warps take part (the shuffles below need every lane); P threads per pair,
    // lanes past the last pair add nothing
    if (tid < (np * P + 31) / 32 * 32) {
      const int k = tid / P;
      float g = 0.f;
      int cp = 0, cq = 0;
      if (k < np) {
        int u = 0, t = 0;
        pair_of(k, u, t);
        cp = W - H + u;
        cq = W - H + t;
        const float Mp = out[cp], Mq = out[cq];
        for (int r = part; r < n; r += P) {
          const float* rr = rec + (long long)r * A.stride;
          g += rr[2 * W + k] * ex2_approx(((rr[cp] - Mp) + (rr[cq] - Mq)) * cl2);
        }
      }
#pragma unroll
      for (int o = P / 2; o > 0; o >>= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
      if (k < np && part == 0) gm[k] = g / (out[W + cp] * out[W + cq]);   // <P_u, P_t>
    }
    epi_sync<NWG>(bar_id);
    if (tid == 0) {
      // gamma_t = 1 + sum_{u<t} gamma_u <P_t, P_u>; ||C||_1 = sum_t gamma_t
      float gam[kMaxWalk], gsum = 0.f;
      for (int t = 0; t < H; ++t) {
        float g = 1.f;
        for (int u = 0; u < t; ++u) g += gam[u] * gm[pair_index(u, t)];
        gam[t] = g;
        gsum += g;
      }
      for (int t = 0; t < H; ++t) out[2 * W + t] = gam[t] / (gsum * out[W + (W - H + t)]);
    }
    epi_sync<NWG>(bar_id);
  }

  // Wait for the merge warp's slice statistics, then a, c~, w and the order key of every
  // row of the chunk. kDirect (the second pass of the two-pass mode): no statistics ran
  // for this chunk; e = exp((l - M)/sqrt(d)) comes straight from the logits in TMEM against
  // the merged slice maximum M, weighted by 1 / (W Z) and the walk coefficients.
  template <int HT, bool kDirect>
  __device__ bool emit(const Chunk& ch) {
    using S = Smem<W, D, NWG>;
    int* ctl = reinterpret_cast<int*>(sm + S::kOffMisc + 16);
    const nx_cache& c = A.c;
    const nx_params& p = A.p;
    // rows this thread finalizes: tiles t = wg, wg + NWG, ... (R2 of them); positions first
    constexpr int R2 = Roles<NWG>::kMaxChunkTiles / NWG;
    int32_t posv[R2];
#pragma unroll
    for (int r = 0; r < R2; ++r) {
      const int t = wg + NWG * r;
      const int j = ch.j0 + t * kTileRows + lg * 32 + lane;
      posv[r] = (t < ch.ntiles && j < ch.T && (A.out.flags & kEmitKeys))
                    ? __ldg(&c.pos[row_of(c, ch.l, ch.s, ch.h, j)]) : 0;
    }
    const uint32_t head_id = (uint32_t)((p.layer_id_base + ch.l) * c.kv_heads + ch.h);
    const uint32_t seq_id = (uint32_t)(p.seq_id_base + ch.s);
    // the merge warp publishes the slice's merged statistics for this TMEM buffer; thread 0
    // waits (the abort flag may be set by other warps at any time) and everyone acts on
    // its snapshot after the barrier
    uint64_t* bar_mfull = reinterpret_cast<uint64_t*>(sm + S::kOffBar) + 2 * S::kStages + 8;
    const bool self_merge = epi_merges();
    if (tid == 0) {
      if (self_merge) {
        // every chunk record of the slice must be in memory (after a records-only pass
        // they all are)
        if (!ctl[1] && A.pass != 2 &&
            !wait_at_least(&A.arrive[ch.slice], ch.nchunks, A.dev_status))
          ctl[1] = 1;
        __threadfence();
      } else if (!ctl[1] && !mbar_wait(&bar_mfull[ch.b], ch.use & 1, A.dev_status)) {
        ctl[1] = 1;
      }
      ctl[2] = ctl[1];
    }
    epi_sync<NWG>(bar_id);
    if (ctl[2]) return false;
    if (self_merge) merge_records(ch);
    if (tid == 0) trace_ev(A, vcta, nev, 5 + 1000 * (ch.slice + 1));
    if (kDirect) {
      // the chunk slot's weights straight from the merged record: M / sqrt(d) in log2
      // units (in the chunk-maximum slot, unused here), 1 / (W Z), the walk coefficients
      const float* mr = reinterpret_cast<const float*>(sm + S::kOffMrec) + ch.b * S::kMrec;
      if (tid < W) {
        const int w = tid;
        mc(ch.b)[w] = mr[w] * cl2;
        ca(ch.b)[w] = 1.f / ((float)W * mr[W + w]);
        if (w >= W - H) cc(ch.b)[w - (W - H)] = mr[2 * W + (w - (W - H))];
        if (ch.k == 0 && (A.out.flags & kEmitStats)) {
          A.out.row_stats[((long long)ch.slice * W + w) * 2] = mr[w] * rsqrtf((float)D);
          A.out.row_stats[((long long)ch.slice * W + w) * 2 + 1] = mr[W + w];
        }
      }
      epi_sync<NWG>(bar_id);
    } else if (!kFoldInMerge<W>) {
      const float* mr = reinterpret_cast<const float*>(sm + S::kOffMrec) + ch.b * S::kMrec;
      const float* m = mc(ch.b);
      if (tid < W) {
        const int w = tid;
        // fold this chunk's max shift into the slice's per-column weights
        const float shift = ex2_approx((m[w] - mr[w]) * cl2);
        ca(ch.b)[w] = shift / ((float)W * mr[W + w]);
        if (w >= W - H) cc(ch.b)[w - (W - H)] = mr[2 * W + (w - (W - H))] * shift;
        if (ch.k == 0 && (A.out.flags & kEmitStats)) {
          A.out.row_stats[((long long)ch.slice * W + w) * 2] = mr[w] * rsqrtf((float)D);
          A.out.row_stats[((long long)ch.slice * W + w) * 2 + 1] = mr[W + w];
        }
      }
      epi_sync<NWG>(bar_id);
    }
    if (tid == 0) trace_ev(A, vcta, nev, 6);
    // partial sums over this warpgroup's columns for every tile, one barrier, then each
    // warpgroup finalizes a quarter of the tiles
    // this warp's weights: the slice weights times the shift from its lane quarter's
    // maxima (its e values' reference) to the chunk maxima
    float* wc = wca();
    if (kDirect) {
      if (lane < CW) {
        wc[lane] = ca(ch.b)[col0 + lane];
      } else if (lane < CW + kMaxWalk) {
        const int tt = lane - CW;
        wc[lane] = tt < H ? cc(ch.b)[tt] : 0.f;
      }
      __syncwarp();
    } else {
      const float* mwq = mw(ch.b) + lg * W;
      const float* mcb = mc(ch.b);
      if (lane < CW) {
        const int col = col0 + lane;
        wc[lane] = ca(ch.b)[col] * ex2_approx((mwq[col] - mcb[col]) * cl2);
      } else if (lane < CW + kMaxWalk) {
        const int tt = lane - CW;
        float x = 0.f;
        if (tt < H) {
          const int col = W - H + tt;
          x = cc(ch.b)[tt] * ex2_approx((mwq[col] - mcb[col]) * cl2);
        }
        wc[lane] = x;
      }
      __syncwarp();
    }
    float scc[kMaxWalk], sca[kHoist ? CW : 1];
#pragma unroll
    for (int tt = 0; tt < kMaxWalk; ++tt) scc[tt] = wc[CW + tt];
#pragma unroll
    for (int i = 0; i < (kHoist ? CW : 0); ++i) sca[i] = wc[i];
    const int row = lg * 32 + lane;
    for (int t0 = 0; t0 < ch.ntiles; t0 += P2) {
      uint32_t r[P2][CW];
#pragma unroll
      for (int u = 0; u < P2; ++u)
        if (t0 + u < ch.ntiles) tmem_ld_issue<CW>(taddr(ch, t0 + u), r[u]);
      tmem_ld_wait();
#pragma unroll
      for (int u = 0; u < P2; ++u) {
        const int t = t0 + u;
        if (t >= ch.ntiles) break;
        float v[CW];
        if (kDirect) {
          const float* shc = mc(ch.b) + col0;
#pragma unroll
          for (int q = 0; q < CW / 4; ++q) {
            const float4 sh = reinterpret_cast<const float4*>(shc)[q];
            v[4 * q] = ex2_approx(fmaf(__uint_as_float(r[u][4 * q]), cl2, -sh.x));
            v[4 * q + 1] = ex2_approx(fmaf(__uint_as_float(r[u][4 * q + 1]), cl2, -sh.y));
            v[4 * q + 2] = ex2_approx(fmaf(__uint_as_float(r[u][4 * q + 2]), cl2, -sh.z));
            v[4 * q + 3] = ex2_approx(fmaf(__uint_as_float(r[u][4 * q + 3]), cl2, -sh.w));
          }
        } else {
#pragma unroll
          for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[u][i]);
        }
        float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < CW; ++i)
          a4[i & 3] = fmaf(v[i], kHoist ? sca[i] : wc[i], a4[i & 3]);
        apart()[(t * NWG + wg) * kTileRows + row] = (a4[0] + a4[1]) + (a4[2] + a4[3]);
        if (wg == kWalkWg) {
          float ct = 0.f;
          if (HT >= 0) {
#pragma unroll
            for (int tt = 0; tt < (HT > 0 ? HT : 0); ++tt)
              ct = fmaf(v[CW - HT + tt], scc[tt], ct);
          } else {
#pragma unroll
            for (int i = 0; i < CW; ++i)
              if (i >= CW - H) ct = fmaf(v[i], scc[(i - (CW - H)) & (kMaxWalk - 1)], ct);
          }
          ctp()[t * kTileRows + row] = ct;
        }
      }
    }
    // Pass 2 was the last read of the chunk's TMEM buffer: hand it back to the MMA issuer
    // now, so that a later chunk's MMAs refill it while the keys are finalized.
    tc_fence_before();
    epi_sync<NWG>(bar_id);
    if (tid == 0) {
      uint64_t* bar_tempty = reinterpret_cast<uint64_t*>(sm + S::kOffBar) + 2 * S::kStages + 3;
      mbar_arrive(&bar_tempty[ch.b]);
    }
    const int bs = p.block_size;
    const int N = units_of(ch.T, bs);
#pragma unroll
    for (int r = 0; r < R2; ++r) {
      const int t = wg + NWG * r;
      if (t >= ch.ntiles) break;
      const int j = ch.j0 + t * kTileRows + row;
      if (bs == 1 && j >= ch.T) continue;
      const float* ap = apart() + t * NWG * kTileRows + row;
      float a;
      if (NWG == 4)
        a = (ap[0] + ap[kTileRows]) + (ap[2 * kTileRows] + ap[3 * kTileRows]);
      else
        a = ap[0] + ap[kTileRows];
      float ct = ctp()[t * kTileRows + row];
      int u = j;                 // the decision unit: this row, or its 32-row block
      if (bs > 1) {
        // Eq. (1) BlockSum: a block's a and c~ are the sums over its rows, which are this
        // warp's 32 rows; lane 0 (the block's first row) finalizes it
        a = warp_sum(j < ch.T ? a : 0.f);
        ct = warp_sum(j < ch.T ? ct : 0.f);
        if (lane != 0 || j >= ch.T) continue;
        u = j / bs;
      }
      const float sj = a + p.lambda * ct;
      const float ramp = (N > 1) ? (float)u / (float)(N - 1) : 0.f;
      const float wj = sj + p.eps_tie * ramp;
      const long long o = (long long)ch.slice * c.capacity + u;
      if (A.out.flags & kEmitA) A.out.a[o] = a;
      if (A.out.flags & kEmitC) A.out.ctilde[o] = ct;
      if (A.out.flags & kEmitW) A.out.w[o] = wj;
      if (A.out.flags & kEmitKeys) {
        uint32_t key = kForcedKey;
        if (p.n_avg > 1)
          key = __float_as_uint(wj);   // the averaged keys are drawn by a pass of their own
        else if (!(u < p.n_sink || u >= N - p.n_recent))
          key = candidate_key1(wj, posv[r], p, head_id, seq_id);
        A.out.keys[o] = key;
      }
    }
    return true;
  }

  // The epilogue loop, software-pipelined when TMEM holds two or more chunks: chunk c+1's
  // statistics are computed and published before chunk c waits for its slice.
  template <int HT>
  __device__ void run(uint64_t* bar_tfull, uint64_t* bar_tempty, uint64_t* bar_pub,
                      int chunk_rows, int nbuf) {
    using S = Smem<W, D, NWG>;
    int* ctl = reinterpret_cast<int*>(sm + S::kOffMisc + 16);
    Chunk prev;
    bool have_prev = false;
    uint32_t cnt = 0;
    auto finish = [&](const Chunk& ch) -> bool {
      if (tid == 0) trace_ev(A, vcta, nev, 3 + 1000 * (ch.slice + 1));
      const bool ok = emit<HT, false>(ch);   // true: emit handed the buffer back after pass 2
      tc_fence_before();
      epi_sync<NWG>(bar_id);
      if (tid == 0) {
        trace_ev(A, vcta, nev, 4);
        if (!ok) {
          mbar_arrive(&bar_tempty[ch.b]);
          ctl[1] = 1;
        }
      }
      return ok;
    };
    Sched sc;
    sched_init(sc, vcta, vgrid);
    int sl, kq, Tq;
    if (A.pass == 2) {
      // the second pass of the two-pass mode: the slice statistics are complete, so every
      // chunk goes straight to its emit (the next chunk's MMAs fill the other buffer)
      for (; sched_next(A, sc, chunk_rows, sl, kq, Tq); ++cnt) {
        const Chunk ch = make_chunk(A, sl, kq, Tq, chunk_rows, cnt, nbuf);
        if (tid == 0) {
          ctl[3] = ctl[1];
          ctl[2] = (!ctl[3] && mbar_wait(&bar_tfull[ch.b], ch.use & 1, A.dev_status)) ? 1 : 0;
        }
        epi_sync<NWG>(bar_id);
        if (ctl[3]) break;
        if (!ctl[2]) {
          if (tid == 0) ctl[1] = 1;
          break;
        }
        tc_fence_after();
        const bool ok = emit<HT, true>(ch);
        tc_fence_before();
        epi_sync<NWG>(bar_id);
        if (!ok) {
          if (tid == 0) {
            mbar_arrive(&bar_tempty[ch.b]);
            ctl[1] = 1;
          }
          break;
        }
      }
      return;
    }
    for (; sched_next(A, sc, chunk_rows, sl, kq, Tq); ++cnt) {
      const Chunk ch = make_chunk(A, sl, kq, Tq, chunk_rows, cnt, nbuf);
      // thread 0 takes one snapshot of the abort flag and waits for the chunk's logits;
      // everyone acts on both after the barrier
      if (tid == 0) {
        trace_ev(A, vcta, nev, 100 + ch.k);
        ctl[3] = ctl[1];
        ctl[2] = (!ctl[3] && mbar_wait(&bar_tfull[ch.b], ch.use & 1, A.dev_status)) ? 1 : 0;
      }
      epi_sync<NWG>(bar_id);
      if (ctl[3]) break;
      const bool ok = ctl[2] != 0;
      tc_fence_after();
      if (tid == 0) trace_ev(A, vcta, nev, 1);
      if (ok) stats<HT>(ch);
      if (tid == 0) trace_ev(A, vcta, nev, 2 + 1000 * (ch.slice + 1));
      publish(ch, ok, bar_pub);
      if (!ok) break;
      if (A.pass == 1) {
        // records only: the chunk's TMEM buffer is free as soon as its record is stored
        tc_fence_before();
        epi_sync<NWG>(bar_id);
        if (tid == 0) mbar_arrive(&bar_tempty[ch.b]);
        continue;
      }
      if (nbuf == 1) {
        if (!finish(ch)) break;
      } else {
        if (have_prev && !finish(prev)) break;
        prev = ch;
        have_prev = true;
      }
    }
    if (tid == 0) ctl[3] = ctl[1];
    epi_sync<NWG>(bar_id);
    if (nbuf != 1 && have_prev && !ctl[3]) finish(prev);
  }
};

// The merge warp: for every chunk of this CTA (in the epilogue's order), once its TMEM
// buffer's previous user is finished and every chunk of its slice has published, pull
// the slice's chunk records into shared memory (one bulk copy per kGroup records) and
// merge them with an online rescale across batches: per window row the maximum and the
// normaliser, and the walk coefficients gamma_t / (sum gamma * Z_t) of Eq. (4); for
// W <= 32 it also turns them into the chunk's per-column weights.
template <int W, int D, int NWG>
__device__ void merge_warp(const Args& A, uint8_t* sm, int chunk_rows, int nbuf, float cl2,
                           uint64_t* bar_tempty, uint64_t* bar_mfull, uint64_t* bar_htx,
                           volatile int* abort_flag, int vcta, int vgrid) {
  using S = Smem<W, D, NWG>;
  constexpr int QW = (W + 31) / 32;       // columns per lane
  const int lane = threadIdx.x & 31;
  const int H = A.p.walk_len;
  float* stage = reinterpret_cast<float*>(sm + S::kOffStage);
  float* ms = reinterpret_cast<float*>(sm + S::kOffMs);     // [0]: maxima, [1]: normalisers
  uint32_t cnt = 0, htx = 0;
  if (A.pass == 1) return;                 // records only: nothing to merge
  if (!kFoldInMerge<W> && A.nbuf == 1) return;   // the epilogue merges (Epi::epi_merges)
  Sched sc;
  sched_init(sc, vcta, vgrid);
  int sl, kq, Tq;
  int last_slice = -1;
  uint32_t last_b = 0;
  float* mrec = reinterpret_cast<float*>(sm + S::kOffMrec);
  for (; !warp_flag(abort_flag) && sched_next(A, sc, chunk_rows, sl, kq, Tq); ++cnt) {
    const Chunk ch = make_chunk(A, sl, kq, Tq, chunk_rows, cnt, nbuf);
    int ok = 1;
    if (lane == 0) {
      // after a records-only pass every record of the slice is already in memory
      ok = mbar_wait(&bar_tempty[ch.b], (ch.use & 1) ^ 1, A.dev_status) &&
           (A.pass == 2 || wait_at_least(&A.arrive[ch.slice], ch.nchunks, A.dev_status));
      __threadfence();
      // the records were written through the generic proxy; the bulk copies read them
      // through the async proxy
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) { *abort_flag = 1; break; }
    if (A.pass == 2 && sl == last_slice) {
      // the second pass takes a slice's chunks one after another: the merged record is
      // the previous chunk slot's
      for (int x = lane; x < S::kMrec; x += 32)
        mrec[ch.b * S::kMrec + x] = mrec[last_b * S::kMrec + x];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_mfull[ch.b]);
      last_b = ch.b;
      continue;
    }
    last_slice = sl;
    last_b = ch.b;
    float M[QW], Z[QW];
#pragma unroll
    for (int q = 0; q < QW; ++q) {
      M[q] = -INFINITY;
      Z[q] = 0.f;
    }
    float G = 0.f;                          // lane k < kMaxPairs: Gram entry k
    int gu = 0, gt = 0;
    pair_of(lane < kMaxPairs ? lane : 0, gu, gt);
    const bool gact = lane < kMaxPairs && gt < H;
    const int wp = W - H + gu, wq = W - H + gt;
    const float* src = A.partial + (long long)ch.slice * A.maxc * A.stride;
    constexpr int NG = Roles<NWG>::kGroup;
    for (int b0 = 0; b0 < ch.nchunks && ok; b0 += NG) {
      const int n = min(NG, ch.nchunks - b0);
      if (lane == 0) {
        const uint32_t bytes = (uint32_t)(n * A.stride * 4);
        mbar_expect_tx(bar_htx, bytes);
        bulk_load(smem_u32(stage), src + (long long)b0 * A.stride, bytes, bar_htx);
        ok = mbar_wait(bar_htx, htx & 1, A.dev_status);
      }
      ++htx;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // new maxima, rescaled normalisers
      float Mn[QW];
#pragma unroll
      for (int q = 0; q < QW; ++q) {
        const int c = lane + 32 * q;
        float mb = M[q];
        if (c < W)
          for (int i = 0; i < n; ++i) mb = fmaxf(mb, stage[i * A.stride + c]);
        Mn[q] = mb;
        if (c < W) {
          float z = (M[q] == -INFINITY) ? 0.f : Z[q] * ex2_approx((M[q] - mb) * cl2);
          for (int i = 0; i < n; ++i)
            z += stage[i * A.stride + W + c] * ex2_approx((stage[i * A.stride + c] - mb) * cl2);
          Z[q] = z;
          ms[c] = mb;              // the Gram step needs every column's new maximum
          ms[W + c] = M[q];        // and its previous one
        }
      }
      __syncwarp();
      if (gact) {
        const float np = ms[wp], nq = ms[wq], op = ms[W + wp], oq = ms[W + wq];
        float g = (op == -INFINITY) ? 0.f : G * ex2_approx(((op - np) + (oq - nq)) * cl2);
        for (int i = 0; i < n; ++i) {
          const float* r = stage + i * A.stride;
          g += r[2 * W + lane] * ex2_approx(((r[wp] - np) + (r[wq] - nq)) * cl2);
        }
        G = g;
      }
#pragma unroll
      for (int q = 0; q < QW; ++q) M[q] = Mn[q];
      __syncwarp();
    }
    if (!ok) { *abort_flag = 1; break; }
    float* out = reinterpret_cast<float*>(sm + S::kOffMrec) + ch.b * S::kMrec;
#pragma unroll
    for (int q = 0; q < QW; ++q) {
      const int c = lane + 32 * q;
      if (c < W) {
        out[c] = M[q];
        out[W + c] = Z[q];
        ms[W + c] = Z[q];
      }
    }
    __syncwarp();
    // Eq. (4) in rank-1 form: gamma_t = 1 + sum_{u<t} gamma_u <P_t, P_u>, with
    // <P_u, P_t> = Gram / (Z_u Z_t); ||C||_1 = sum_t gamma_t (every row sums to one)
    const float gnorm = gact ? G / (ms[W + wp] * ms[W + wq]) : 0.f;
    float gam = 0.f, gsum = 0.f;               // lane t < H holds gamma_t
    for (int t = 0; t < H; ++t) {
      const float nt = __shfl_sync(0xffffffffu, gnorm, pair_index(lane < t ? lane : 0, t > 0 ? t : 1));
      float v = (lane < t) ? gam * nt : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      const float g = 1.f + v;
      if (lane == t) gam = g;
      gsum += g;
    }
    if (lane < H) out[2 * W + lane] = gam / (gsum * ms[W + (W - H + lane)]);
    __syncwarp();
    // fold this chunk's max shift (its maxima are in shared memory, stored before the
    // chunk was published) into the per-column weights the epilogue applies
    if (kFoldInMerge<W> && A.pass != 2) {
      const float* mch = reinterpret_cast<const float*>(sm + S::kOffMc) + ch.b * W;
      float* ca = reinterpret_cast<float*>(sm + S::kOffCa) + ch.b * W;
      float* cc = reinterpret_cast<float*>(sm + S::kOffCc) + ch.b * kMaxWalk;
#pragma unroll
      for (int q = 0; q < QW; ++q) {
        const int c = lane + 32 * q;
        if (c < W) {
          const float shift = ex2_approx((mch[c] - M[q]) * cl2);
          ca[c] = shift / ((float)W * Z[q]);
          if (c >= W - H) cc[c - (W - H)] = out[2 * W + (c - (W - H))] * shift;
          if (ch.k == 0 && (A.out.flags & kEmitStats)) {
            A.out.row_stats[((long long)ch.slice * W + c) * 2] = M[q] * rsqrtf((float)D);
            A.out.row_stats[((long long)ch.slice * W + c) * 2 + 1] = Z[q];
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&bar_mfull[ch.b]);
  }
}

// The publisher warp: once the epilogue warps have stored a chunk's lane-quarter partials
// (per-warp column maxima, sums and walk-row Gram sums), it builds the chunk's record
// (the four quarters rescaled to the chunk maxima, which also go to shared memory for the
// epilogue and the merge warp), releases the partials' shared memory, makes the record
// visible device-wide and counts it in for its slice -- all off the epilogue's path.
template <int W, int D, int NWG>
__device__ void publish_warp(const Args& A, uint8_t* sm, int chunk_rows, int nbuf, float cl2,
                             uint64_t* bar_pub, uint64_t* bar_rec, volatile int* abort_flag,
                             int vcta, int vgrid) {
  using S = Smem<W, D, NWG>;
  constexpr int CW = W / NWG;
  constexpr int RS = S::kRedStride;
  constexpr int kWalkWg = NWG - 1;
  const int lane = threadIdx.x & 31;
  const int H = A.p.walk_len;
  const float* red = reinterpret_cast<const float*>(sm + S::kOffRed);
  if (A.pass == 2) return;   // the second pass publishes nothing (the records are there)
  Sched sc;
  sched_init(sc, vcta, vgrid);
  int sl, kq, Tq;
  for (uint32_t cnt = 0; sched_next(A, sc, chunk_rows, sl, kq, Tq); ++cnt) {
    const uint32_t b = cnt % nbuf, use = cnt / nbuf;
    int ok = 1;
    if (lane == 0) ok = mbar_wait(&bar_pub[b], use & 1, A.dev_status) && !*abort_flag;
    if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    const float* mwb = reinterpret_cast<const float*>(sm + S::kOffMw) + b * 4 * W;
    float* m = reinterpret_cast<float*>(sm + S::kOffMc) + b * W;
    float* rec = A.partial + ((long long)sl * A.maxc + kq) * A.stride;
#pragma unroll
    for (int q0 = 0; q0 < (W + 31) / 32; ++q0) {
      const int col = lane + 32 * q0;
      if (col < W) {
        const int g = col / CW;
        float mq[4], mm = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mq[q] = mwb[q * W + col];
          mm = fmaxf(mm, mq[q]);
        }
        float x = 0.f;                  // quarter sums rescaled to the chunk maximum
#pragma unroll
        for (int q = 0; q < 4; ++q) x += red[(4 * g + q) * RS + col] * ex2_approx((mq[q] - mm) * cl2);
        m[col] = mm;
        rec[col] = mm;                  // chunk max (raw)
        rec[W + col] = x;               // sum relative to it
      }
    }
    if (lane < kMaxPairs) {
      const int k = lane;
      int u = 0, t = 0;
      pair_of(k, u, t);
      float x = 0.f;
      if (t < H) {
        const int cp = W - H + u, cq = W - H + t;
        float mp = -INFINITY, mq = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          mp = fmaxf(mp, mwb[q * W + cp]);
          mq = fmaxf(mq, mwb[q * W + cq]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          x += red[(4 * kWalkWg + q) * RS + W + k] *
               ex2_approx(((mwb[q * W + cp] - mp) + (mwb[q * W + cq] - mq)) * cl2);
      }
      rec[2 * W + k] = x;               // Gram entry
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(bar_rec);             // the partials may be overwritten
      __threadfence();
      atomicAdd(&A.arrive[sl], 1);
    }
    __syncwarp();
  }
}

// A CTA's warps are dealt round-robin to the SM's four sub-partitions, each with 16K
// registers: with NWG = 4 (one team of 20 warps) a sub-partition holds 5 warps, which caps
// a thread at 96 registers; with NWG = 2 (two teams of 12 warps) it holds 6, which caps a
// thread at 80.
template <int W, int D, int NWG>
__global__ void __launch_bounds__(Roles<NWG>::kBlockThreads, 1)
score_tc_kernel(const __grid_constant__ CUtensorMap tmap, const Args A) {
  using S = Smem<W, D, NWG>;
  using R = Roles<NWG>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm0 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
  // this thread's team: its shared-memory region, TMEM share and place in the schedule
  const int team = (int)threadIdx.x / R::kThreads;
  const int tid = (int)threadIdx.x - team * R::kThreads;
  uint8_t* sm = sm0 + team * S::kTeamBytes;
  const int vcta = (int)blockIdx.x * R::kTeams + team;
  const int vgrid = (int)gridDim.x * R::kTeams;
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + S::kOffBar);   // [S::kStages]
  uint64_t* bar_empty = bar_full + S::kStages;                           // [S::kStages]
  uint64_t* bar_tfull = bar_empty + S::kStages;                          // [3] TMEM buffer ready
  uint64_t* bar_tempty = bar_tfull + 3;                               // [3] TMEM buffer free
  uint64_t* bar_qfull = bar_tempty + 3;
  uint64_t* bar_qempty = bar_qfull + 1;
  uint64_t* bar_mfull = bar_full + 2 * S::kStages + 8;                 // [3] merged stats ready
  uint64_t* bar_htx = bar_mfull + 3;                                  // merge warp's copies
  uint64_t* bar_pub = bar_htx + 1;                                    // [3] records stored
  uint64_t* bar_rec = bar_pub + 3;                     // a chunk's partials taken (publisher)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm0 + S::kOffMisc);   // team 0's
  int* ctl = reinterpret_cast<int*>(sm + S::kOffMisc + 16);   // [1] abort, [2-3] snapshots

  const nx_cache& c = A.c;
  const int warp = tid >> 5, lane = tid & 31;
  const float cl2 = kLog2e * rsqrtf((float)D);   // raw accumulator -> log2 units
  constexpr uint32_t kIdesc = idesc_bf16<W>();
  const int chunk_rows = A.tiles_per_chunk * kTileRows;
  const int nbuf = A.nbuf;
  const uint32_t team_cols = A.tmem_cols / R::kTeams;
  const uint32_t buf_cols = (team_cols / (uint32_t)nbuf / W) * W;

  if (tid == 0) {
    trace_mark(A, vcta, 0, 7);
    for (int i = 0; i < S::kStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&bar_tfull[i], 1);
      mbar_init(&bar_tempty[i], 1);
    }
    mbar_init(bar_qfull, 1);
    mbar_init(bar_qempty, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&bar_mfull[i], 1);
    mbar_init(bar_htx, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&bar_pub[i], R::kEpiWarps);
    mbar_init(bar_rec, 1);
    ctl[0] = 0;
    ctl[1] = 0;
    ctl[2] = 0;
    ctl[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
  }
  if (team == 0 && warp == R::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(A.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the setup above overlaps the previous kernel; its outputs are read only from here on
  grid_dep_trigger();
  grid_dep_wait();
  const uint32_t tmem = *tmem_slot + (uint32_t)team * team_cols;   // column offset
  volatile int* abort_flag = ctl + 1;
  if (tid == 0) trace_mark(A, vcta, 1, 9);

  if (warp == R::kProducerWarp) {
    // =================== TMA producer: query images and K tiles ===================
    uint32_t u = 0, qn = 0;
    int prev_slice = -1, nev_p = 0;
    Sched sc;
    sched_init(sc, vcta, vgrid);
    int slice, k, T;
    while (!warp_flag(abort_flag) && sched_next(A, sc, chunk_rows, slice, k, T)) {
      int fail = 0;
      if (lane == 0) {
        int l, s, h;
        slice_coords(c, slice, l, s, h);
        const int j0 = k * chunk_rows;
        const int ntiles = min(A.tiles_per_chunk, (T - j0 + kTileRows - 1) / kTileRows);
        if (slice != prev_slice) {
          if (qn > 0 && !mbar_wait(bar_qempty, (qn - 1) & 1, A.dev_status)) fail = 1;
          if (!fail) {
            mbar_expect_tx(bar_qfull, S::kQBytes);
            bulk_load(smem_u32(sm + S::kOffQ), A.qimg + (long long)slice * S::kQBytes,
                      S::kQBytes, bar_qfull);
            ++qn;
            prev_slice = slice;
          }
        }
        for (int t = 0; t < ntiles && !fail; ++t, ++u) {
          const uint32_t st = u % S::kStages, ph = (u / S::kStages) & 1;
          if (!mbar_wait(&bar_empty[st], ph ^ 1, A.dev_status)) { fail = 1; break; }
          trace_role(A, vcta, 768, nev_p, 40 + t);
          const uint32_t dst = smem_u32(sm + S::kOffK + st * S::kTileBytes);
          const int r0 = j0 + t * kTileRows;
          if (c.page_size == 0) {
            mbar_expect_tx(&bar_full[st], S::kTileBytes);
            const int row = slice * c.capacity + r0;
#pragma unroll
            for (int kb = 0; kb < S::KB; ++kb)
              tma_load_2d(dst + kb * S::kRegionA, &tmap, kb * 64, row, &bar_full[st]);
          } else {
            const int ps = c.page_size;
            const int npg = min(kTileRows / ps, (T - r0 + ps - 1) / ps);
            mbar_expect_tx(&bar_full[st], (uint32_t)(npg * ps * 128 * S::KB));
            for (int pg = 0; pg < npg; ++pg) {
              const int page = c.block_table[(long long)s * c.max_pages_per_seq + (r0 / ps) + pg];
              const int row = (int)((((long long)l * c.num_pages + page) * c.kv_heads + h) * ps);
              for (int kb = 0; kb < S::KB; ++kb)
                tma_load_2d(dst + kb * S::kRegionA + pg * ps * 128, &tmap, kb * 64, row,
                            &bar_full[st]);
            }
          }
        }
        if (fail) *abort_flag = 1;
      }
      if (__shfl_sync(0xffffffffu, fail, 0)) break;
    }
  } else if (warp == R::kMmaWarp) {
    // =================== MMA issuer ===================
    uint32_t u = 0, qn = 0, cc = 0;
    int prev_slice = -1, nev_m = 0;
    const uint32_t qa = smem_u32(sm + S::kOffQ);
    Sched sc;
    sched_init(sc, vcta, vgrid);
    int slice, k, T;
    for (; !warp_flag(abort_flag) && sched_next(A, sc, chunk_rows, slice, k, T); ++cc) {
      int fail = 0;
      if (lane == 0) {
        const int j0 = k * chunk_rows;
        const int ntiles = min(A.tiles_per_chunk, (T - j0 + kTileRows - 1) / kTileRows);
        const uint32_t b = cc % nbuf, use = cc / nbuf;
        trace_role(A, vcta, 512, nev_m, 20);
        // the previous slice's query image may be replaced once its MMAs are done
        if (slice != prev_slice && prev_slice >= 0) mma_commit(bar_qempty);
        if (!mbar_wait(&bar_tempty[b], (use & 1) ^ 1, A.dev_status)) fail = 1;
        tc_fence_after();
        trace_role(A, vcta, 512, nev_m, 21);
        if (!fail && slice != prev_slice) {
          if (!mbar_wait(bar_qfull, qn & 1, A.dev_status)) fail = 1;
          ++qn;
          prev_slice = slice;
        }
        trace_role(A, vcta, 512, nev_m, 22);
        for (int t = 0; t < ntiles && !fail; ++t, ++u) {
          const uint32_t st = u % S::kStages, ph = (u / S::kStages) & 1;
          if (!mbar_wait(&bar_full[st], ph, A.dev_status)) { fail = 1; break; }
          if (t == 0 || t == ntiles - 1) trace_role(A, vcta, 512, nev_m, t == 0 ? 23 : 24);
          tc_fence_after();
          const uint32_t ka = smem_u32(sm + S::kOffK + st * S::kTileBytes);
          const uint32_t dt = tmem + b * buf_cols + (uint32_t)(t * W);
#pragma unroll
          for (int kb = 0; kb < S::KB; ++kb) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t da = sw128_desc(ka + kb * S::kRegionA + ks * 32);
              const uint64_t db = sw128_desc(qa + kb * S::kRegionB + ks * 32);
              mma_bf16(dt, da, db, kIdesc, (kb | ks) ? 1u : 0u);
            }
          }
          mma_commit(&bar_empty[st]);      // the stage's smem is free once these finish
        }
        if (!fail) mma_commit(&bar_tfull[b]);   // the chunk's logits are in TMEM buffer b
        trace_role(A, vcta, 512, nev_m, 25);
        if (fail) *abort_flag = 1;
      }
      if (__shfl_sync(0xffffffffu, fail, 0)) break;
    }
  } else if (warp == R::kMergeWarp) {
    // =================== slice merge ===================
    merge_warp<W, D, NWG>(A, sm, chunk_rows, nbuf, cl2, bar_tempty, bar_mfull, bar_htx,
                          abort_flag, vcta, vgrid);
  } else if (warp == R::kPublishWarp) {
    // =================== record publisher ===================
    publish_warp<W, D, NWG>(A, sm, chunk_rows, nbuf, cl2, bar_pub, bar_rec, abort_flag, vcta,
                            vgrid);
  } else {
    // =================== epilogue: warps [0, 4 NWG) ===================
    Epi<W, D, NWG> epi(A, sm, tmem, buf_cols, cl2, A.p.walk_len, tid, vcta, vgrid, 1 + team);
    switch (A.p.walk_len) {
      case 3: epi.template run<3>(bar_tfull, bar_tempty, bar_pub, chunk_rows, nbuf); break;
      case 5: epi.template run<5>(bar_tfull, bar_tempty, bar_pub, chunk_rows, nbuf); break;
      default: epi.template run<-1>(bar_tfull, bar_tempty, bar_pub, chunk_rows, nbuf); break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (team == 0 && warp == R::kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(*tmem_slot),
                 "r"(A.tmem_cols));
  }
  if (tid == 0) trace_mark(A, vcta, 2, 8);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
std::atomic<long long*> g_trace{nullptr};   // installed by nexus_debug_set_trace
std::atomic<int> g_layout{0};               // pipelines per CTA asked for (0: automatic)
thread_local int32_t g_last_cfg[8];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

template <int W, int D, int NWG>
cudaError_t launch_t(const nx_cache& c, const nx_params& p, const void* q, const WsLayout& L,
                     char* ws, const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                     int* launches, bool* used, bool* two_pass) {
  using S = Smem<W, D, NWG>;
  using R = Roles<NWG>;
  *used = false;
  for (int i = 0; i < 8; ++i) g_last_cfg[i] = 0;
  auto fn = encode_fn();
  if (!fn) { g_last_cfg[0] = -1; return cudaSuccess; }
  // the whole K tensor as rows of head_dim bf16 elements; boxes of 64 columns
  const long long rows = c.page_size
                             ? (long long)c.layers * c.num_pages * c.kv_heads * c.page_size
                             : (long long)c.layers * c.seqs * c.kv_heads * c.capacity;
  if (rows >= (1LL << 31)) { g_last_cfg[0] = -2; return cudaSuccess; }
  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(c.page_size ? c.page_size : kTileRows)};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.k, gdim, gstride, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
    g_last_cfg[0] = -3;
    return cudaSuccess;
  }

  if (L.stats_stride != S::kRecStride) { g_last_cfg[0] = -2; return cudaSuccess; }
  int dev = 0, sms = 0, per_sm_api = 0;
  cudaGetDevice(&dev);
  // per device and instantiation; setting the attributes twice (two host threads racing
  // on the first call) is harmless
  static std::atomic<bool> attr_set[64];
  if (dev < 0 || dev >= 64) return cudaSuccess;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<W, D, NWG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(score_tc_kernel<W, D, NWG>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm_api, score_tc_kernel<W, D, NWG>,
                                                R::kBlockThreads, S::kAlloc);
  if (per_sm_api < 1) {
    g_last_cfg[0] = -6;
    g_last_cfg[1] = per_sm_api;
    return cudaSuccess;
  }
  const long long slices = L.slices;
  const long long cap_tiles = (c.capacity + kTileRows - 1) / kTileRows;

  {
    const int per_sm = 1;
    const uint32_t tmem_cols = R::kTmemCols;                     // one team's share
    const long long grid_max = (long long)sms * R::kTeams;       // teams in the schedule
    // Chunk size and grid: every slice's chunks must be co-resident (the slice barrier),
    // and a round of the grid should hold whole slices (a slice split across two rounds
    // makes its first chunks wait a whole round). Among chunk sizes up to what a TMEM
    // buffer holds (and 16 tiles), pick the fewest rounds x chunk tiles; prefer two
    // buffers (the next chunk's MMAs overlap this chunk's epilogue).
    int nbuf = 0, tpc = 0, maxc = 0;
    long long grid_sel = 0, best = -1;
    for (int nb = 3; nb >= 1; --nb) {
      const int max_tiles = min(R::kMaxChunkTiles, (int)(tmem_cols / nb / W));
      for (int t = 1; t <= max_tiles; ++t) {
        const int mc = (int)((cap_tiles + t - 1) / t);
        if (mc > grid_max || mc > kMaxChunksPerSlice) continue;
        // Estimated time: rounds of the grid x (the chunk's tiles + about four tiles' worth
        // of fixed latency), 1.5x without a second buffer to overlap chunks. With two or
        // more buffers the next chunk's statistics overlap a slice's wait, so every
        // pipeline takes part and slices need not align with rounds (measured: 8-tile
        // chunks over all SMs beat 7-tile chunks in aligned rounds); with one buffer a
        // round holds whole slices (a slice split across rounds would stall its first
        // chunks for a whole round).
        long long rounds, gsel;
        if (nb == 1) {
          const long long per = grid_max / mc;                 // whole slices per round
          rounds = (slices + per - 1) / per;
          gsel = per * mc;
        } else {
          rounds = (slices * mc + grid_max - 1) / grid_max;
          gsel = grid_max;
        }
        const long long cost = rounds * (t + 4) * (nb == 1 ? 3 : 2) * 4 + (3 - nb);
        if (best < 0 || cost < best) {
          best = cost;
          nbuf = nb;
          tpc = t;
          maxc = mc;
          grid_sel = gsel;
        }
      }
    }
    // A slice with more chunks than there are co-resident pipelines cannot wait for its
    // own records at the slice barrier: two passes then, the first storing every chunk's
    // record, the second (which waits on no other CTA) recomputing the logits and going
    // straight to the emit against the complete records. K is read twice. (Measured: for
    // W = 64 slices of 131072 rows, which fit one pass with a single TMEM buffer, the two
    // passes -- 4-tile chunks at W = 64 -- took 1.47 ms against 1.05 ms for the one pass.)
    int passes = 1;
    if (!nbuf) {
      passes = 2;
      nbuf = 2;
      tpc = min(R::kMaxChunkTiles, (int)(tmem_cols / 2 / W));
      maxc = (int)((cap_tiles + tpc - 1) / tpc);
      grid_sel = grid_max;
    }
    Args a;
    a.c = c;
    a.p = p;
    (void)q;
    a.qimg = reinterpret_cast<const unsigned char*>(ws + L.qbar);
    a.tmem_cols = R::kTeams * tmem_cols;                        // the whole allocation
    a.partial = reinterpret_cast<float*>(ws + L.stats);
    a.arrive = reinterpret_cast<int*>(ws + L.barriers);
    a.newlen = reinterpret_cast<const int32_t*>(ws + L.newlen);
    a.out = out;
    a.dev_status = dev_status;
    a.tiles_per_chunk = tpc;
    a.nbuf = nbuf;
    a.maxc = maxc;
    a.stride = L.stats_stride;
    a.total_ids = slices * maxc;
    a.slices = (int)slices;
    a.trace = g_trace.load(std::memory_order_relaxed);
    const long long vgrid = a.total_ids < grid_sel ? a.total_ids : grid_sel;
    const long long grid = (vgrid + R::kTeams - 1) / R::kTeams;  // CTAs of kTeams teams

    for (int pass = (passes == 1 ? 0 : 1); pass <= (passes == 1 ? 0 : 2); ++pass) {
      a.pass = pass;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)grid);
      cfg.blockDim = dim3(R::kBlockThreads);
      cfg.dynamicSmemBytes = S::kAlloc;
      cfg.stream = st;
      cudaLaunchAttribute attr[2];
      attr[0].id = cudaLaunchAttributeCooperative;
      attr[0].val.cooperative = 1;
      attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[1].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 2;
      cudaError_t e = cudaLaunchKernelEx(&cfg, score_tc_kernel<W, D, NWG>, map, a);
      if (e == cudaErrorInvalidValue || e == cudaErrorNotSupported) {
        (void)cudaGetLastError();            // without the early start, then
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, score_tc_kernel<W, D, NWG>, map, a);
      }
      if (e == cudaErrorCooperativeLaunchTooLarge && pass <= 1) {
        (void)cudaGetLastError();
        g_last_cfg[0] = -5;
        g_last_cfg[1] = per_sm_api;
        return cudaSuccess;
      }
      if (e != cudaSuccess) return e;
      note_launch(st, launches, pass == 1 ? "score_tc_records" : "score_tc");
    }
    g_last_cfg[0] = R::kTeams;
    (void)per_sm;
    g_last_cfg[1] = per_sm_api;
    g_last_cfg[2] = (int32_t)grid;
    g_last_cfg[3] = tpc;
    g_last_cfg[4] = nbuf;
    g_last_cfg[5] = maxc;
    g_last_cfg[6] = (int32_t)tmem_cols;
    g_last_cfg[7] = S::kAlloc;
    *used = true;
    *two_pass = passes == 2;
    return cudaSuccess;
  }
  return cudaSuccess;
}

}  // namespace tc

void tc_set_trace(long long* buf) { tc::g_trace.store(buf); }
void tc_set_layout(int teams) { tc::g_layout.store(teams); }
void tc_last_config(int32_t* out) {
  for (int i = 0; i < 8; ++i) out[i] = tc::g_last_cfg[i];
}

bool tc_supported(const nx_cache& c, const nx_params& p) {
  if (c.dtype != NX_DTYPE_BF16) return false;
  if (c.head_dim != 64 && c.head_dim != 128) return false;
  if (p.window != 16 && p.window != 32 && p.window != 64) return false;
  if (p.walk_len > p.window / 4) return false;       // walk rows within one warpgroup
  if (c.page_size != 0 && c.page_size < 8) return false;
  return true;
}

cudaError_t launch_score_tc(const nx_cache& c, const nx_params& p, const void* q,
                            const WsLayout& L, char* ws, const ScoreOut& out,
                            int32_t* dev_status, cudaStream_t st, int* launches, bool* used,
                            bool* two_pass) {
  *used = false;
  *two_pass = false;
  if (!tc_supported(c, p)) return cudaSuccess;
  const bool d128 = c.head_dim == 128;
#define NX_TC_LAUNCH(WW, DD, NN) \
  tc::launch_t<WW, DD, NN>(c, p, q, L, ws, out, dev_status, st, launches, used, two_pass)
  // Windows of up to 32 rows may take two pipelines per CTA. Automatic choice: two for large
  // paged caches (one TMA copy per page: two producers keep more of them in flight), one
  // otherwise (measured faster for contiguous caches); a layout that cannot run falls back.
  const long long rows_all = (long long)c.layers * c.seqs * c.kv_heads * c.capacity;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool big = rows_all >= 8LL * 512 * (sms > 0 ? sms : 1) && c.page_size > 0;
  const int layout = tc::g_layout.load(std::memory_order_relaxed);
  if (p.window <= 32 && (layout == 2 || (layout == 0 && big))) {
    cudaError_t e = p.window == 16 ? (d128 ? NX_TC_LAUNCH(16, 128, 2) : NX_TC_LAUNCH(16, 64, 2))
                                   : (d128 ? NX_TC_LAUNCH(32, 128, 2) : NX_TC_LAUNCH(32, 64, 2));
    if (e != cudaSuccess || *used || layout == 2) return e;
  }
  switch (p.window) {
    case 16: return d128 ? NX_TC_LAUNCH(16, 128, 4) : NX_TC_LAUNCH(16, 64, 4);
    case 32: return d128 ? NX_TC_LAUNCH(32, 128, 4) : NX_TC_LAUNCH(32, 64, 4);
    default: return d128 ? NX_TC_LAUNCH(64, 128, 4) : NX_TC_LAUNCH(64, 64, 4);
  }
#undef NX_TC_LAUNCH
}

}  // namespace nx
