// nx_score_tc.cu -- fused direct scores + Nexus walk + selection keys on the tensor cores
// (bf16 caches, head_dim 64 or 128, W in {16, 32, 64}, contiguous or paged).
//
// Nexus Sampling paper, §2.1 Eq. (1) (b = 1), §2.2 Eqs. (2)-(5), §2.3 (keys of Eq. (6),
// n = 1). One persistent, cooperatively launched kernel; two CTAs per SM. A CTA takes
// chunks of up to 256/W tiles of 128 cached rows of one slice and:
//   1. stages each K tile in shared memory with TMA (128-byte swizzle, one box per
//      64-element column block -- per page when paged), double-buffered;
//   2. one thread issues tcgen05.mma (kind::f16, bf16 x bf16 -> fp32), M = 128 rows,
//      N = W window rows, K = head_dim, twice: against bf16(Qbar) and against
//      bf16(Qbar - bf16(Qbar)), accumulating in the same TMEM columns, so the logits
//      keep fp32 accuracy although the tensor cores take bf16 operands. Every tile's
//      logits stay in TMEM (tile t -> columns [t*W, (t+1)*W)) until the chunk is done;
//   3. four epilogue warps (one TMEM lane = one row each) take the chunk maxima, then
//      e = exp((l - max_chunk)/sqrt(d)) written back to TMEM, the chunk sums and the
//      H x H Gram of the walk rows, and publish them;
//   4. a bounded slice-wide barrier: the last chunk of the slice to arrive merges all
//      chunk statistics, runs the walk recurrence (gamma_t = 1 + sum_{u<t} gamma_u
//      <P_t, P_u>, the rank-1 form of Eq. (4)) and publishes the per-row coefficients;
//   5. every chunk turns its TMEM e values into a, c~, w and the order key of every row.
// K is read from HBM exactly once; nothing but one key (and optional outputs) per row
// goes back to memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "nx_internal.cuh"

namespace nx {
namespace tc {

constexpr int kThreads = 192;          // warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer
constexpr int kTileRows = 128;
constexpr int kStages = 2;
constexpr long long kWaitLimit = 1LL << 22;   // mbarrier polls before giving up
constexpr float kLog2e = 1.4426950408889634f;

struct Args {
  nx_cache c;
  nx_params p;
  const unsigned char* qimg;   // [slices] shared-memory images of bf16 hi/lo queries
  uint32_t tmem_cols;      // 256 with two CTAs per SM, 512 with one
  float* partial;          // [slices][maxc][stride]
  float* fin;              // [slices][3W + kMaxWalk]
  int* arrive;             // [slices] groups of the slice merged
  int* ready;              // [slices] final coefficients published
  int* garrive;            // [slices][ngroups] chunks of each group published
  float* grec;             // [slices][ngroups][stride] merged group records
  int ngroups;             // group records per slice (chunks are merged 16 at a time)
  const int32_t* newlen;   // [slices]
  ScoreOut out;
  int32_t* dev_status;
  int tiles_per_chunk;
  int maxc;                // chunk ids per slice
  int stride;              // floats per partial record
  long long total_ids;     // slices * maxc
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

// 32 lanes x 16 / 32 columns of 32-bit TMEM words into registers (and back).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
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

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Named barrier of the four epilogue warps (barrier 1; __syncthreads uses barrier 0).
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---------------------------------------------------------------------------
// Merging chunk statistics
// ---------------------------------------------------------------------------
constexpr int kGroup = 16;    // records merged at a time

// A record holds, for the rows it covers: per window row w the maximum raw logit m_w and
// sum_j exp((l_wj - m_w)/sqrt(d)) (natural-log units), and per walk-row pair (p, q) the
// Gram sum_j exp((l_pj - m_p)/sqrt(d)) exp((l_qj - m_q)/sqrt(d)). merge_records combines
// n <= 16 records (global memory, `stride` floats apart) into one record `dst` of the same
// form, with the 128 epilogue threads: every value is loaded into shared memory at once
// (independent loads, one round trip), then combined in a fixed order.
template <int W>
__device__ __forceinline__ void merge_records(const float* src, int n, int stride, float* dst,
                                              float* stage, int H, float cl2) {
  constexpr int R = 2 * W + kMaxPairs;
  const int tid = threadIdx.x;
  for (int idx = tid; idx < n * R; idx += 128) {
    const int i = idx / R, f = idx - i * R;
    stage[idx] = __ldcg(&src[(long long)i * stride + f]);
  }
  float* sM = stage + kGroup * R;      // merged maxima (the Gram step needs them)
  epi_sync();
  if (tid < W) {
    float M = -INFINITY;
    for (int i = 0; i < n; ++i) M = fmaxf(M, stage[i * R + tid]);
    float Z = 0.f;
    for (int i = 0; i < n; ++i) Z += stage[i * R + W + tid] * exp2f((stage[i * R + tid] - M) * cl2);
    sM[tid] = M;
    dst[tid] = M;
    dst[W + tid] = Z;
  }
  epi_sync();
  if (tid < kMaxPairs) {
    int t, u;
    pair_of(tid, t, u);
    float g = 0.f;
    if (u < H) {
      const int wp = W - H + t, wq = W - H + u;
      for (int i = 0; i < n; ++i) {
        const float* r = stage + i * R;
        g += r[2 * W + tid] * exp2f(((r[wp] - sM[wp]) + (r[wq] - sM[wq])) * cl2);
      }
    }
    dst[2 * W + tid] = g;
  }
  epi_sync();
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int W, int D>
struct Smem {
  static constexpr int KB = D / 64;                       // 128-byte column blocks per row
  static constexpr int kRegionA = kTileRows * 128;        // one column block of a K tile
  static constexpr int kTileBytes = KB * kRegionA;
  static constexpr int kRegionB = W * 128;                // one column block of Qbar
  static constexpr int kOffK = 0;
  static constexpr int kOffQ = kStages * kTileBytes;      // [hi, lo][KB][kRegionB]
  static constexpr int kOffBar = kOffQ + 2 * KB * kRegionB;
  static constexpr int kOffMisc = kOffBar + 64;           // tmem slot + control words
  static constexpr int kQBytes = 2 * KB * kRegionB;       // hi + lo query image
  static constexpr int kOffRed = kOffMisc + 64;           // [4][W + kMaxPairs] floats
  static constexpr int kOffCoef = kOffRed + 4 * (W + kMaxPairs) * 4;  // mc[W] ca[W] cc[8]
  static constexpr int kRec = 2 * W + kMaxPairs;          // floats of one chunk record
  static constexpr int kOffStage = kOffCoef + (2 * W + kMaxWalk) * 4;  // [16][kRec] + M Z G
  // staging for 16 records, the merged maxima (<= 64 floats), then one merged record
  static constexpr int kBytes = kOffStage + (16 * kRec + 64 + kRec) * 4;
  static constexpr int kAlloc = kBytes + 1024;            // slack for 1024-byte alignment
};

template <int W, int D>
__global__ void __launch_bounds__(kThreads, 2)
score_tc_kernel(const __grid_constant__ CUtensorMap tmap, const Args A) {
  using S = Smem<W, D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(sm + S::kOffBar);
  uint64_t* bar_empty = bar_full + kStages;
  uint64_t* bar_mma = bar_empty + kStages;
  uint64_t* bar_q = bar_mma + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + S::kOffMisc);
  int* ctl = reinterpret_cast<int*>(sm + S::kOffMisc + 16);   // [0] last-arriver, [1] abort
  float* red = reinterpret_cast<float*>(sm + S::kOffRed);
  float* s_mc = reinterpret_cast<float*>(sm + S::kOffCoef);   // chunk maxima (raw logits)
  float* s_ca = s_mc + W;                                     // per-row a coefficients
  float* s_cc = s_ca + W;                                     // walk coefficients

  const nx_cache& c = A.c;
  const nx_params& p = A.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.walk_len;
  const float cl2 = kLog2e * rsqrtf((float)D);   // raw accumulator -> log2 units
  constexpr uint32_t kIdesc = idesc_bf16<W>();
  const int chunk_rows = A.tiles_per_chunk * kTileRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar_full[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(bar_mma, 1);
    mbar_init(bar_q, 1);
    ctl[1] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(A.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  uint32_t it = 0;          // tiles streamed by this CTA (stage/phase bookkeeping)
  uint32_t chunks_done = 0;
  uint32_t q_loads = 0;     // query images fetched (bar_q phase bookkeeping)
  int prev_slice = -1;

  for (long long id = blockIdx.x; id < A.total_ids; id += gridDim.x) {
    const int slice = (int)(id / A.maxc);
    const int k = (int)(id % A.maxc);
    if (A.newlen[slice] < 0) continue;
    const int T = c.lens[slice];
    const int nchunks = (T + chunk_rows - 1) / chunk_rows;
    if (k >= nchunks) continue;
    if (ctl[1]) break;                       // an earlier wait gave up
    int l, s, h;
    slice_coords(c, slice, l, s, h);
    const int j0 = k * chunk_rows;
    const int ntiles = min(A.tiles_per_chunk, (T - j0 + kTileRows - 1) / kTileRows);

    // the slice's query image is fetched by the producer below when the slice changes;
    // the previous chunk's MMAs (its only readers) completed before the last barrier
    const bool new_q = slice != prev_slice;
    prev_slice = slice;
    __syncthreads();

    if (warp == 4) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        if (new_q) {
          mbar_expect_tx(bar_q, S::kQBytes);
          bulk_load(smem_u32(sm + S::kOffQ), A.qimg + (long long)slice * S::kQBytes, S::kQBytes,
                    bar_q);
        }
        for (int t = 0; t < ntiles; ++t) {
          const uint32_t u = it + t, st = u % kStages, ph = (u / kStages) & 1;
          if (!mbar_wait(&bar_empty[st], ph ^ 1, A.dev_status)) { ctl[1] = 1; break; }
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
      }
    } else if (warp == 5) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        tc_fence_after();
        const uint32_t qa = smem_u32(sm + S::kOffQ);
        if (new_q && !mbar_wait(bar_q, q_loads & 1, A.dev_status)) ctl[1] = 1;
        for (int t = 0; t < ntiles && !ctl[1]; ++t) {
          const uint32_t u = it + t, st = u % kStages, ph = (u / kStages) & 1;
          if (!mbar_wait(&bar_full[st], ph, A.dev_status)) { ctl[1] = 1; break; }
          tc_fence_after();
          const uint32_t ka = smem_u32(sm + S::kOffK + st * S::kTileBytes);
          const uint32_t dt = tmem + (uint32_t)(t * W);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
#pragma unroll
            for (int kb = 0; kb < S::KB; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint64_t da = sw128_desc(ka + kb * S::kRegionA + ks * 32);
                const uint64_t db = sw128_desc(qa + (half * S::KB + kb) * S::kRegionB + ks * 32);
                mma_bf16(dt, da, db, kIdesc, (half | kb | ks) ? 1u : 0u);
              }
            }
          }
          mma_commit(&bar_empty[st]);      // the stage's smem is free once these finish
        }
        mma_commit(bar_mma);               // all tiles of the chunk are in TMEM
      }
    } else {
      // ---------------- epilogue: warps 0-3, TMEM lane = row ----------------
      const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
      bool ok = mbar_wait(bar_mma, chunks_done & 1, A.dev_status);
      tc_fence_after();
      // pass 1a: chunk maxima of the raw accumulators
      float mx[W];
#pragma unroll
      for (int w = 0; w < W; ++w) mx[w] = -INFINITY;
      for (int t = 0; t < ntiles && ok; ++t) {
        const bool valid = j0 + t * kTileRows + warp * 32 + lane < T;
#pragma unroll
        for (int cb = 0; cb < W; cb += 16) {
          float v[16];
          tmem_ld16(lane_base + t * W + cb, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) mx[cb + i] = fmaxf(mx[cb + i], valid ? v[i] : -INFINITY);
        }
      }
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float m = warp_max(mx[w]);
        if (lane == 0) red[warp * (W + kMaxPairs) + w] = m;
      }
      epi_sync();
      if (threadIdx.x < W) {
        float m = red[threadIdx.x];
        for (int q4 = 1; q4 < 4; ++q4) m = fmaxf(m, red[q4 * (W + kMaxPairs) + threadIdx.x]);
        s_mc[threadIdx.x] = m;
      }
      epi_sync();
      // pass 1b: e = exp((l - max)/sqrt(d)) back into TMEM, chunk sums and walk Gram
      float z[W], gp[kMaxPairs];
#pragma unroll
      for (int w = 0; w < W; ++w) z[w] = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPairs; ++i) gp[i] = 0.f;
      for (int t = 0; t < ntiles && ok; ++t) {
        const bool valid = j0 + t * kTileRows + warp * 32 + lane < T;
        float ew[kMaxWalk];
#pragma unroll
        for (int cb = 0; cb < W; cb += 16) {
          float v[16];
          tmem_ld16(lane_base + t * W + cb, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e = valid ? exp2f((v[i] - s_mc[cb + i]) * cl2) : 0.f;
            v[i] = e;
            z[cb + i] += e;
          }
          tmem_st16(lane_base + t * W + cb, v);
          if (cb + 16 >= W) {   // the walk rows W-H .. W-1 lie in the last 16 columns
#pragma unroll
            for (int tt = 0; tt < kMaxWalk; ++tt) {
              float x = 0.f;
#pragma unroll
              for (int i = 0; i < 16; ++i)
                if (tt < H && cb + i == W - H + tt) x = v[i];
              ew[tt] = x;
            }
          }
        }
#pragma unroll
        for (int tt = 0; tt < kMaxWalk; ++tt)
#pragma unroll
          for (int uu = tt; uu < kMaxWalk; ++uu) gp[pair_index(tt, uu)] += ew[tt] * ew[uu];
      }
      tmem_st_wait();
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float v = warp_sum(z[w]);
        if (lane == 0) red[warp * (W + kMaxPairs) + w] = v;
      }
#pragma unroll
      for (int i = 0; i < kMaxPairs; ++i) {
        const float v = warp_sum(gp[i]);
        if (lane == 0) red[warp * (W + kMaxPairs) + W + i] = v;
      }
      epi_sync();
      float* rec = A.partial + ((long long)slice * A.maxc + k) * A.stride;
      if (threadIdx.x < W + kMaxPairs) {
        float v = 0.f;
        for (int q4 = 0; q4 < 4; ++q4) v += red[q4 * (W + kMaxPairs) + threadIdx.x];
        if (threadIdx.x < W) {
          rec[threadIdx.x] = s_mc[threadIdx.x];     // chunk max (raw)
          rec[W + threadIdx.x] = v;                 // chunk sum relative to that max
        } else {
          rec[2 * W + (threadIdx.x - W)] = v;       // Gram entry
        }
      }
      // ---- slice-wide barrier: two-level merge of the chunk records ----
      // chunks arrive in groups of kGroup; the last of a group merges the group, the last
      // group of the slice merges the group records and publishes the coefficients
      __threadfence();
      epi_sync();
      const int ngs = (nchunks + kGroup - 1) / kGroup;
      const int grp = k / kGroup;
      const int gsize = min(kGroup, nchunks - grp * kGroup);
      float* stage = reinterpret_cast<float*>(sm + S::kOffStage);
      float* merged = stage + kGroup * S::kRec;   // sM scratch then the slice record
      if (threadIdx.x == 0) {
        ctl[0] = 0;
        if (!ok) {
          ctl[1] = 1;
        } else {
          const int prev = atomicAdd(&A.garrive[(long long)slice * A.ngroups + grp], 1);
          ctl[0] = (prev == gsize - 1) ? 1 : 0;
        }
      }
      epi_sync();
      if (ctl[0]) {
        __threadfence();
        float* grec = A.grec + ((long long)slice * A.ngroups + grp) * A.stride;
        merge_records<W>(A.partial + ((long long)slice * A.maxc + grp * kGroup) * A.stride,
                         gsize, A.stride, grec, stage, H, cl2);
        __threadfence();
        epi_sync();
        if (threadIdx.x == 0) {
          const int prev = atomicAdd(&A.arrive[slice], 1);
          ctl[0] = (prev == ngs - 1) ? 2 : 0;
        }
        epi_sync();
      }
      float* fin = A.fin + (long long)slice * (3 * W + kMaxWalk);
      if (ctl[0] == 2) {
        __threadfence();
        float* rec = merged + 64;               // after the sM scratch (W <= 64)
        merge_records<W>(A.grec + (long long)slice * A.ngroups * A.stride, ngs, A.stride, rec,
                         stage, H, cl2);
        if (threadIdx.x == 0) {
          // Eq. (4) in rank-1 form on <P_p, P_q> = Gram / (Z_p Z_q)
          float gam[kMaxWalk], gsum = 0.f;
          for (int t = 0; t < H; ++t) {
            float g = 1.f;
            for (int u = 0; u < t; ++u) {
              const int wp = W - H + u, wq = W - H + t;
              g += gam[u] * rec[2 * W + pair_index(u, t)] / (rec[W + wp] * rec[W + wq]);
            }
            gam[t] = g;
            gsum += g;
          }
          // ||C||_1 = sum_t gamma_t since every row P sums to one
          for (int t = 0; t < kMaxWalk; ++t)
            fin[3 * W + t] = (t < H) ? gam[t] / (gsum * rec[W + (W - H + t)]) : 0.f;
        }
        if (threadIdx.x < W) {
          const int w = threadIdx.x;
          fin[w] = rec[w];                                     // raw max
          fin[W + w] = rec[W + w];                             // normaliser
          fin[2 * W + w] = 1.0f / ((float)W * rec[W + w]);
        }
        __threadfence();
        epi_sync();
        if (threadIdx.x == 0) st_release(&A.ready[slice], 1);
      } else {
        if (threadIdx.x == 0 && !ctl[1])
          if (!wait_at_least(&A.ready[slice], 1, A.dev_status)) ctl[1] = 1;
        epi_sync();
      }
      ok = ok && !ctl[1];
      // ---- per-chunk coefficients: fold the chunk-max shift into the final weights ----
      if (ok && threadIdx.x < W) {
        const int w = threadIdx.x;
        const float shift = exp2f((s_mc[w] - __ldcg(&fin[w])) * cl2);
        s_ca[w] = __ldcg(&fin[2 * W + w]) * shift;
        if (w >= W - H) s_cc[w - (W - H)] = __ldcg(&fin[3 * W + (w - (W - H))]) * shift;
      }
      if (ok && k == 0 && (A.out.flags & kEmitStats) && threadIdx.x < W) {
        const int w = threadIdx.x;
        A.out.row_stats[((long long)slice * W + w) * 2] = __ldcg(&fin[w]) * rsqrtf((float)D);
        A.out.row_stats[((long long)slice * W + w) * 2 + 1] = __ldcg(&fin[W + w]);
      }
      epi_sync();
      // pass 2: a, c~, w and the order key of every row
      const uint32_t head_id = (uint32_t)((p.layer_id_base + l) * c.kv_heads + h);
      const uint32_t seq_id = (uint32_t)(p.seq_id_base + s);
      for (int t = 0; t < ntiles && ok; ++t) {
        const int j = j0 + t * kTileRows + warp * 32 + lane;
        float a = 0.f, ct = 0.f;
#pragma unroll
        for (int cb = 0; cb < W; cb += 16) {
          float v[16];
          tmem_ld16(lane_base + t * W + cb, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            a = fmaf(v[i], s_ca[cb + i], a);
            if (cb + i >= W - H) ct = fmaf(v[i], s_cc[cb + i - (W - H)], ct);
          }
        }
        if (j < T) {
          const float sj = a + p.lambda * ct;
          const float ramp = (T > 1) ? (float)j / (float)(T - 1) : 0.f;
          const float wj = sj + p.eps_tie * ramp;
          const long long o = (long long)slice * c.capacity + j;
          if (A.out.flags & kEmitA) A.out.a[o] = a;
          if (A.out.flags & kEmitC) A.out.ctilde[o] = ct;
          if (A.out.flags & kEmitW) A.out.w[o] = wj;
          if (A.out.flags & kEmitKeys) {
            uint32_t key = kForcedKey;
            if (!(j < p.n_sink || j >= T - p.n_recent))
              key = candidate_key(wj, c.pos[row_of(c, l, s, h, j)], p, head_id, seq_id);
            A.out.keys[o] = key;
          }
        }
      }
      if (!ok && threadIdx.x == 0) ctl[1] = 1;
    }
    // ---- end of chunk: TMEM reads done before the next chunk's MMAs overwrite it ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    it += ntiles;
    ++chunks_done;
    if (new_q) ++q_loads;
  }

  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(A.tmem_cols));
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
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

template <int W, int D>
cudaError_t launch_t(const nx_cache& c, const nx_params& p, const void* q, const WsLayout& L,
                     char* ws, const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                     int* launches, bool* used) {
  using S = Smem<W, D>;
  *used = false;
  auto fn = encode_fn();
  if (!fn) return cudaSuccess;
  // the whole K tensor as rows of head_dim bf16 elements; boxes of 64 columns
  const long long rows = c.page_size
                             ? (long long)c.layers * c.num_pages * c.kv_heads * c.page_size
                             : (long long)c.layers * c.seqs * c.kv_heads * c.capacity;
  if (rows >= (1LL << 31)) return cudaSuccess;
  CUtensorMap map;
  cuuint64_t gdim[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t gstride[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(c.page_size ? c.page_size : kTileRows)};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c.k, gdim, gstride, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaSuccess;

  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaSuccess;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(score_tc_kernel<W, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kAlloc);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(score_tc_kernel<W, D>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, score_tc_kernel<W, D>, kThreads, S::kAlloc);
  if (per_sm < 1) return cudaSuccess;
  if (per_sm > 2) per_sm = 2;                 // TMEM: 512 columns per SM, split evenly
  const uint32_t tmem_cols = per_sm == 2 ? 256u : 512u;
  const long long grid_max = (long long)sms * per_sm;

  // chunk size: as many tiles as TMEM holds, but enough chunks to fill the grid
  const long long slices = L.slices;
  const int max_tiles = (int)(tmem_cols / W);
  const long long cap_tiles = (c.capacity + kTileRows - 1) / kTileRows;
  // the smallest power-of-two chunk that still fits every chunk in one round of the grid
  int tpc = max_tiles;
  while (tpc > 1 && slices * ((cap_tiles + tpc / 2 - 1) / (tpc / 2)) <= grid_max) tpc >>= 1;
  const int maxc = (int)((cap_tiles + tpc - 1) / tpc);
  if (maxc > grid_max) return cudaSuccess;    // the slice barrier needs co-resident chunks
  if (maxc > kGroup * kGroup) return cudaSuccess;   // two merge levels of 16
  if ((long long)maxc * (long long)((c.capacity + 127) / 128) > (1LL << 40)) return cudaSuccess;

  Args a;
  a.c = c;
  a.p = p;
  (void)q;
  a.qimg = reinterpret_cast<const unsigned char*>(ws + L.qbar);
  a.tmem_cols = tmem_cols;
  a.partial = reinterpret_cast<float*>(ws + L.stats);
  a.fin = reinterpret_cast<float*>(ws + L.fin);
  a.arrive = reinterpret_cast<int*>(ws + L.barriers);
  a.ready = a.arrive + slices;
  a.garrive = reinterpret_cast<int*>(ws + L.group_arrive);
  a.grec = reinterpret_cast<float*>(ws + L.group_rec);
  a.ngroups = L.groups_per_slice;
  a.newlen = reinterpret_cast<const int32_t*>(ws + L.newlen);
  a.out = out;
  a.dev_status = dev_status;
  a.tiles_per_chunk = tpc;
  a.maxc = maxc;
  a.stride = L.stats_stride;
  a.total_ids = slices * maxc;
  long long grid = a.total_ids < grid_max ? a.total_ids : grid_max;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = S::kAlloc;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, score_tc_kernel<W, D>, map, a);
  if (e != cudaSuccess) return e;
  note_launch(st, launches, "score_tc");
  *used = true;
  return cudaSuccess;
}

}  // namespace tc

bool tc_supported(const nx_cache& c, const nx_params& p) {
  if (c.dtype != NX_DTYPE_BF16) return false;
  if (c.head_dim != 64 && c.head_dim != 128) return false;
  if (p.window != 16 && p.window != 32 && p.window != 64) return false;
  if (c.page_size != 0 && c.page_size < 8) return false;
  return true;
}

cudaError_t launch_score_tc(const nx_cache& c, const nx_params& p, const void* q,
                            const WsLayout& L, char* ws, const ScoreOut& out,
                            int32_t* dev_status, cudaStream_t st, int* launches, bool* used) {
  *used = false;
  if (!tc_supported(c, p)) return cudaSuccess;
  const bool d128 = c.head_dim == 128;
  switch (p.window) {
    case 16:
      return d128 ? tc::launch_t<16, 128>(c, p, q, L, ws, out, dev_status, st, launches, used)
                  : tc::launch_t<16, 64>(c, p, q, L, ws, out, dev_status, st, launches, used);
    case 32:
      return d128 ? tc::launch_t<32, 128>(c, p, q, L, ws, out, dev_status, st, launches, used)
                  : tc::launch_t<32, 64>(c, p, q, L, ws, out, dev_status, st, launches, used);
    default:
      return d128 ? tc::launch_t<64, 128>(c, p, q, L, ws, out, dev_status, st, launches, used)
                  : tc::launch_t<64, 64>(c, p, q, L, ws, out, dev_status, st, launches, used);
  }
}

}  // namespace nx
