// nx_internal.cuh -- device helpers and the workspace layout shared by the CUDA sources
// of libnexus.so. Nothing here is part of the public ABI (include/nexus.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <utility>
#include <stdint.h>

#include "nexus.h"

namespace nx {

// ---------------------------------------------------------------------------
// Limits and tiling
// ---------------------------------------------------------------------------
constexpr int kMaxWindow = 64;        // W <= 64
constexpr int kMaxWalk = 8;           // H <= 8
constexpr int kMaxAvg = 1024;         // n_avg <= 1024 (256 Philox draw groups)
constexpr int kBlockRows = 32;        // the block size b > 1 (one warp's rows)
constexpr int kMaxPairs = kMaxWalk * (kMaxWalk - 1) / 2;   // walk-row pairs u < t
constexpr int kSimtRows = 256;        // rows per thread block in the CUDA-core scorer
constexpr int kCompactRows = 32;      // destination rows per compaction tile
constexpr long long kSpinLimit = 1LL << 22;   // bounded waits: ~0.3-1 s at most
// the multi-block selection serves up to kMultiSlices slices, kMultiStride ints of scratch each
constexpr int kMultiSlices = 256;
constexpr int kMultiStride = 512;
constexpr uint32_t kForcedKey = 0xFFFFFFFFu;  // order key of a forced (always kept) slot

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the caller's workspace, 256-byte aligned)
// ---------------------------------------------------------------------------
struct WsLayout {
  size_t counters;       // int32 region zeroed at the start of every call
  size_t counters_bytes;
  size_t tile_flags;     // int32 [slices][tiles_per_slice]  (inside counters)
  size_t work;           // int32 [8] global work counters     (inside counters)
  size_t barriers;       // int32 [2][slices] slice arrival counts (inside counters)
  size_t select_scratch; // int32 [min(slices, kMultiSlices)][kMultiStride] multi-block
                         // selection scratch (inside counters)
  size_t keys;           // uint32 [slices][capacity] order keys
  size_t stats;          // float [slices][max_chunks][stats_stride] partial softmax stats
  size_t qbar;           // float [slices][W][head_dim] group-mean window queries, or the
                         // tensor-core scorer's bf16 image (half the size)
  size_t newlen;         // int32 [slices]
  size_t keep;           // int32 [slices][capacity] kept slots (when the caller gives none)
  size_t total;
  int stats_stride;      // floats per chunk: 2W maxima/sums + kMaxPairs Gram entries (padded)
  int max_chunks;        // chunk records per slice (128-row granularity, covers both scorers)
  int tiles_per_slice;   // compaction tiles per slice (budget_max / kCompactRows, rounded up)
  long long slices;
};

// Walk-row pairs (u, t), u < t < kMaxWalk, packed in the order of t then u. The walk
// recurrence gamma_t = 1 + sum_{u<t} gamma_u <P_t, P_u> uses exactly these entries.
__host__ __device__ constexpr int pair_index(int u, int t) { return t * (t - 1) / 2 + u; }
__host__ __device__ inline void pair_of(int k, int& u, int& t) {
  t = 1;
  while (k >= t) {
    k -= t;
    ++t;
  }
  u = k;
}

// ---------------------------------------------------------------------------
// Small device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ld_elem(const void* base, int dtype, long long idx) {
  if (dtype == NX_DTYPE_BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// Row index (in rows of head_dim elements) of slot j of slice (l, s, h); -1 if the
// page table entry is out of range.
__device__ __forceinline__ long long row_of(const nx_cache& c, int l, int s, int h, int j) {
  if (c.page_size == 0)
    return (((long long)l * c.seqs + s) * c.kv_heads + h) * (long long)c.capacity + j;
  int page = c.block_table[(long long)s * c.max_pages_per_seq + j / c.page_size];
  if (page < 0 || page >= c.num_pages) return -1;
  return (((long long)l * c.num_pages + page) * c.kv_heads + h) * (long long)c.page_size +
         (j % c.page_size);
}

__device__ __forceinline__ void slice_coords(const nx_cache& c, int slice, int& l, int& s,
                                             int& h) {
  h = slice % c.kv_heads;
  s = (slice / c.kv_heads) % c.seqs;
  l = slice / (c.kv_heads * c.seqs);
}

// Monotone map from binary32 to uint32: a > b as floats iff key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11). Each round multiplies
// words 0 and 2 by the round constants; the high product halves, XOR-ed with the
// other two words and the key, become words 0 and 2 of the next state, the low halves
// words 1 and 3. The key advances by the golden-ratio / sqrt(3) Weyl increments.
__device__ __forceinline__ uint4 philox4x32_10(uint4 ctr, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t a = ctr.x, b = ctr.y, cc = ctr.z, d = ctr.w;
    const uint32_t hi_a = __umulhi(0xD2511F53u, a), lo_a = 0xD2511F53u * a;
    const uint32_t hi_c = __umulhi(0xCD9E8D57u, cc), lo_c = 0xCD9E8D57u * cc;
    ctr = make_uint4(hi_c ^ b ^ k0, lo_c, hi_a ^ d ^ k1, lo_a);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return ctr;
}

// The uniform of a Philox word: (2 * (x >> 9) + 1) * 2^-24, exact, in (0, 1).
__device__ __forceinline__ float word_to_uniform(uint32_t x) {
  return __fmul_rn(__uint2float_rn(((x >> 9) << 1) | 1u), 5.9604644775390625e-8f);
}

// Specified binary32 logarithm for u in (0, 1) (normal): reduce u = 2^e m with m in
// [sqrt(1/2), sqrt(2)], then ln m = 2 atanh((m - 1)/(m + 1)) by its odd series through
// the f^13 term (Horner in f^2), and ln u = e*ln2_hi + (e*ln2_lo + ln m) with a
// Cody-Waite split of ln 2 (ln2_hi has 16 significant bits). Every operation is one
// IEEE round-to-nearest operation in a fixed order (no contraction), so the result is
// reproducible bit for bit by any implementation of the same recipe.
__device__ __forceinline__ float ln_spec(float u) {
  constexpr float kLn2Hi = 45426.0f / 65536.0f;
  constexpr float kLn2Lo = (float)(0.69314718055994530942 - 45426.0 / 65536.0);
  constexpr float k3 = 1.0f / 3.0f, k5 = 1.0f / 5.0f, k7 = 1.0f / 7.0f;
  constexpr float k9 = 1.0f / 9.0f, k11 = 1.0f / 11.0f, k13 = 1.0f / 13.0f;
  const uint32_t bits = __float_as_uint(u);
  const uint32_t mant = bits & 0x007FFFFFu;
  int e = (int)((bits >> 23) & 0xFFu) - 127;
  uint32_t mbits = mant | 0x3F800000u;       // m in [1, 2)
  if (mant > 0x003504F3u) {                  // m > sqrt(2): halve it
    mbits = mant | 0x3F000000u;
    e += 1;
  }
  const float m = __uint_as_float(mbits);
  const float f = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float s = __fmul_rn(f, f);
  const float t = __fadd_rn(f, f);
  float h = k13;
  h = __fadd_rn(__fmul_rn(h, s), k11);
  h = __fadd_rn(__fmul_rn(h, s), k9);
  h = __fadd_rn(__fmul_rn(h, s), k7);
  h = __fadd_rn(__fmul_rn(h, s), k5);
  h = __fadd_rn(__fmul_rn(h, s), k3);
  const float lnm = __fadd_rn(t, __fmul_rn(t, __fmul_rn(s, h)));
  const float ef = (float)e;
  return __fadd_rn(__fmul_rn(ef, kLn2Hi), __fadd_rn(__fmul_rn(ef, kLn2Lo), lnm));
}

// Specified binary32 exponential (Cody & Waite): k = round-half-even(x * (1/ln 2)),
// r = (x - k ln2_hi) - k ln2_lo with the 16-bit ln2_hi of ln_spec (k ln2_hi exact),
// e^r by its Taylor series through r^7/7! (Horner from the top term), times 2^k; k < -126
// flushes to 0, k > 127 gives +inf. One IEEE round-to-nearest operation per step, in a
// fixed order, so any implementation of the same recipe gives the same bits.
__device__ __forceinline__ float exp_spec(float x) {
  constexpr float kInvLn2 = 1.44269504088896340736f;
  constexpr float kLn2Hi = 45426.0f / 65536.0f;
  constexpr float kLn2Lo = (float)(0.69314718055994530942 - 45426.0 / 65536.0);
  constexpr float c2 = 1.0f / 2.0f, c3 = 1.0f / 6.0f, c4 = 1.0f / 24.0f;
  constexpr float c5 = 1.0f / 120.0f, c6 = 1.0f / 720.0f, c7 = 1.0f / 5040.0f;
  if (x != x) return x;
  const float kf = rintf(__fmul_rn(x, kInvLn2));
  if (kf < -126.0f) return 0.0f;
  if (kf > 127.0f) return __int_as_float(0x7F800000);
  float r = __fsub_rn(x, __fmul_rn(kf, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(kf, kLn2Lo));
  float h = c7;
  h = __fadd_rn(__fmul_rn(h, r), c6);
  h = __fadd_rn(__fmul_rn(h, r), c5);
  h = __fadd_rn(__fmul_rn(h, r), c4);
  h = __fadd_rn(__fmul_rn(h, r), c3);
  h = __fadd_rn(__fmul_rn(h, r), c2);
  h = __fadd_rn(__fmul_rn(h, r), 1.0f);
  h = __fadd_rn(__fmul_rn(h, r), 1.0f);
  return __fmul_rn(h, __uint_as_float((uint32_t)((int)kf + 127) << 23));
}

// The Philox block of draw group g of one candidate: counter (pos, step, head id,
// seq id | g << 24), key = the 64-bit seed.
__device__ __forceinline__ uint4 draw_block(int32_t pos, const nx_params& p, uint32_t head_id,
                                            uint32_t seq_id, uint32_t g) {
  return philox4x32_10(
      make_uint4((uint32_t)pos, p.step, head_id, (seq_id & 0x00FFFFFFu) | (g << 24)),
      (uint32_t)p.seed, (uint32_t)(p.seed >> 32));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ln of uniform i of a candidate (word i mod 4 of draw group i / 4)
__device__ __forceinline__ float log_draw(int32_t pos, const nx_params& p, uint32_t head_id,
                                          uint32_t seq_id, int i) {
  return ln_spec(word_to_uniform(word_of(draw_block(pos, p, head_id, seq_id, (uint32_t)i >> 2),
                                         i & 3)));
}

// §2.3 Eq. (6) for n > 1, in the log domain: with l_i = ln(u_i), M = max_i l_i and
// r = 1/w, key = M r + ln(sum_{i < n} exp((l_i - M) r)) = ln(n pi_j); -inf for w = 0.
// NT > 0: n = NT draws, unrolled and kept in registers. NT = 0: n = p.n_avg draws, taken
// twice (the same values both times) so that nothing is indexed at run time. The sum runs
// over i = 0, 1, ..., n - 1 in that order either way, so both give the same bits.
template <int NT>
__device__ __forceinline__ float averaged_key(float w, int32_t pos, const nx_params& p,
                                              uint32_t head_id, uint32_t seq_id) {
  const float r = __fdiv_rn(1.0f, w);
  if (!(r < __int_as_float(0x7F800000))) return -__int_as_float(0x7F800000);
  float M = -__int_as_float(0x7F800000);
  float S = 0.0f;
  if constexpr (NT > 0) {
    float l[NT];
#pragma unroll
    for (int g = 0; g < (NT + 3) / 4; ++g) {
      const uint4 blk = draw_block(pos, p, head_id, seq_id, (uint32_t)g);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < NT) l[4 * g + i] = ln_spec(word_to_uniform(word_of(blk, i)));
    }
#pragma unroll
    for (int i = 0; i < NT; ++i) M = fmaxf(M, l[i]);
#pragma unroll
    for (int i = 0; i < NT; ++i) S = __fadd_rn(S, exp_spec(__fmul_rn(__fsub_rn(l[i], M), r)));
  } else {
    const int n = p.n_avg;
    for (int g = 0; 4 * g < n; ++g) {
      const uint4 blk = draw_block(pos, p, head_id, seq_id, (uint32_t)g);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < n) M = fmaxf(M, ln_spec(word_to_uniform(word_of(blk, i))));
    }
    for (int g = 0; 4 * g < n; ++g) {
      const uint4 blk = draw_block(pos, p, head_id, seq_id, (uint32_t)g);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * g + i < n) {
          const float l = ln_spec(word_to_uniform(word_of(blk, i)));
          S = __fadd_rn(S, exp_spec(__fmul_rn(__fsub_rn(l, M), r)));
        }
    }
  }
  return __fadd_rn(__fmul_rn(M, r), ln_spec(S));
}

// Order key of one candidate unit at n = 1 (§2.3, Eq. (6)): ln(u)/w for the reservoir
// (Efraimidis-Spirakis), w itself for the top-K template.
__device__ __forceinline__ uint32_t candidate_key1(float w, int32_t pos, const nx_params& p,
                                                   uint32_t head_id, uint32_t seq_id) {
  if (p.mode == NX_MODE_TOPK) return order_key(w);
  const uint4 r = draw_block(pos, p, head_id, seq_id, 0);
  return order_key(__fdiv_rn(ln_spec(word_to_uniform(r.x)), w));
}

// Order key of one candidate unit (§2.3, Eq. (6)) with NT draws known at compile time
// (NT = 1: ln(u)/w, Efraimidis-Spirakis; 0: p.n_avg draws), w itself for the top-K template.
template <int NT>
__device__ __forceinline__ uint32_t candidate_key(float w, int32_t pos, const nx_params& p,
                                                  uint32_t head_id, uint32_t seq_id) {
  if constexpr (NT == 1) {
    return candidate_key1(w, pos, p, head_id, seq_id);
  } else {
    if (p.mode == NX_MODE_TOPK) return order_key(w);
    return order_key(averaged_key<NT>(w, pos, p, head_id, seq_id));
  }
}

// The budget (units kept) of a slice: its own when the caller gives per-slice budgets.
__device__ __forceinline__ int budget_of(const nx_params& p, int slice, int s) {
  return p.slice_budget ? p.slice_budget[slice] : p.budget[s];
}

// Rows left in a slice of T rows after keeping B units of b rows (B >= 1): every kept
// unit is whole except the newest block, which is always kept (n_recent >= 1 at b > 1).
__host__ __device__ __forceinline__ int rows_kept(int T, int B, int b) {
  const int N = (T + b - 1) / b;
  return N <= B ? T : (B - 1) * b + (T - (N - 1) * b);
}

// Units of a slice of T rows.
__host__ __device__ __forceinline__ int units_of(int T, int b) { return (T + b - 1) / b; }

__device__ __forceinline__ int ld_acquire(const int* addr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int* addr, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// Bounded wait until *addr >= target. On giving up, flags NX_DEV_TIMEOUT and returns false.
__device__ __forceinline__ bool wait_at_least(const int* addr, int target, int32_t* dev_status) {
  for (long long it = 0; it < kSpinLimit; ++it) {
    if (ld_acquire(addr) >= target) return true;
    __nanosleep(it < 64 ? 20 : 200);
  }
  atomicOr(dev_status, NX_DEV_TIMEOUT);
  return false;
}

// Bookkeeping after every kernel launch of an entry point: counts it, remembers its
// name and, when a benchmark armed nexus_profile_next_call, records its event.
void note_launch(cudaStream_t st, int* launches, const char* name);
// Every entry point calls begin_call() first and returns through finish() once it has
// enqueued its kernels (launch count and names, the profiling request, the status).
void begin_call();
nx_status finish(cudaError_t e, int launches);

// ---------------------------------------------------------------------------
// Kernel launchers (one per source file)
// ---------------------------------------------------------------------------
enum EmitFlags { kEmitA = 1, kEmitW = 2, kEmitKeys = 4, kEmitC = 8, kEmitStats = 16 };

struct ScoreOut {
  float* a;          // [slices][cap]
  float* w;          // [slices][cap]
  float* ctilde;     // [slices][cap]
  float* row_stats;  // [slices][W][2]
  uint32_t* keys;    // [slices][cap]
  int flags;
};

// Programmatic dependent launch. A kernel launched with launch_after() may be scheduled
// while the kernel before it on the stream is still running: it calls grid_dep_wait()
// before touching anything that kernel writes (the wait returns once that kernel has
// completed and its memory operations are visible; it returns at once when there is no
// such dependency). grid_dep_trigger() lets the next kernel be scheduled early.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// nx_score.cu
cudaError_t launch_prep(const nx_cache& c, const void* q, const nx_params& p, const WsLayout& L,
                        char* ws, int32_t* dev_status, cudaStream_t st, int* launches,
                        int mode);   // 0: validity only, 1: fp32 Qbar, 2: tensor-core image;
                                     // also zeroes the workspace counters
// nx_score_tc.cu: *used is false when the shape is not covered (the caller falls back)
bool tc_supported(const nx_cache& c, const nx_params& p);
void tc_set_trace(long long* buf);
void tc_set_layout(int teams);
void tc_last_config(int32_t* out);
cudaError_t launch_score_tc(const nx_cache& c, const nx_params& p, const void* q,
                            const WsLayout& L, char* ws, const ScoreOut& out,
                            int32_t* dev_status, cudaStream_t st, int* launches, bool* used,
                            bool* two_pass);
cudaError_t launch_score_simt(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                              const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                              int* launches);
// nx_select.cu
cudaError_t launch_keys_from_w(const nx_cache& c, const nx_params& p, const float* w,
                               uint32_t* keys, const int32_t* newlen, cudaStream_t st,
                               int* launches);
cudaError_t launch_select(const nx_cache& c, const uint32_t* keys, int32_t* keep,
                          const int32_t* newlen, int block_size, int* scratch,
                          int32_t* dev_status, cudaStream_t st, int* launches);
// nx_compact.cu
cudaError_t launch_newlen(const nx_cache& c, const nx_params& p, int32_t* newlen,
                          int32_t* dev_status, cudaStream_t st, int* launches);
cudaError_t launch_compact(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                           const int32_t* keep, const int32_t* newlen, int32_t* dev_status,
                           cudaStream_t st, int* launches, long long skip_signal_tile = -1);
// which compaction kernel launch_compact() takes: 0 automatic, 1 tiles, 2 a warp per slice
void compact_set_kernel(int which);

}  // namespace nx
