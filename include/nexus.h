/*
 * nexus.h -- C ABI of the GB300 (sm_103a) per-step eviction library (libnexus.so).
 *
 * The library implements one eviction step of Nexus Sampling as defined in
 * "Forget Without Compromise: Nexus Sampling for Streaming KV-Cache Eviction Under
 * Fixed Budgets": direct scores (§2.1 Eq. (1), §2.2 Eq. (3)), the Nexus walk and
 * weight (§2.2 Eqs. (2), (4), (5)), weighted reservoir selection of B survivors
 * (§2.3 Eq. (6): Efraimidis-Spirakis keys ln(u)/w at n = 1, the n-averaged
 * priority for n > 1), and the in-place compaction that lets inference continue
 * with K_S, V_S (§2.1, "streaming view"). Decisions are made per token (b = 1) or
 * per block of 32 consecutive slots (§2.1 "Block granularity", b = 32).
 *
 * Terms
 *   slice   one (layer l, sequence s, KV head h); slices are independent.
 *           slice id = (l * seqs + s) * kv_heads + h.
 *   row     one cached (key, value) of one slice; slot j = its index 0..T-1.
 *   T       rows currently cached in a slice (lens[slice]).
 *   unit    what one keep/evict decision covers: a row (block_size b = 1) or a block
 *           of b consecutive slots [u b, (u + 1) b) (the slice's last block holds the
 *           T mod b remaining rows when b does not divide T); N = ceil(T / b) units.
 *   B       the budget: units kept per slice of sequence s (budget[s], or
 *           slice_budget[slice] when given).
 *   W, H    window rows and walk length; G = query heads per KV head.
 *
 * Conventions (every entry point)
 *   - All buffer pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or synchronises; scratch memory is the caller's
 *     workspace of nexus_workspace_bytes() bytes (256-byte aligned).
 *   - Calls are asynchronous on `stream`. The returned nx_status covers argument
 *     checks and launch errors only. Conditions found on the device are OR-ed into
 *     *dev_status (an int32 in device memory, caller-owned, which the caller zeroes
 *     and reads after synchronising): NX_DEV_* bits below.
 *   - Calls on different streams are independent when their workspaces and
 *     outputs are disjoint. Two calls must not share a workspace concurrently.
 *   - Block granularity is b = 1 (one decision per token) or b = 32 (block_size).
 */
#ifndef NEXUS_H_
#define NEXUS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* nx_stream_t;

typedef enum nx_status {
  NX_OK = 0,
  NX_ERR_INVALID_ARG = 1,   /* a size, pointer, alignment or parameter is out of range */
  NX_ERR_UNSUPPORTED = 2,   /* valid for the method, not built here (block size not 1/32)*/
  NX_ERR_CUDA = 3,          /* a CUDA launch or memset failed                           */
  NX_ERR_TIMEOUT = 4,       /* reserved: device waits report through dev_status         */
  NX_ERR_WORKSPACE = 5,     /* ws is NULL, misaligned or smaller than required          */
  NX_ERR_DEVICE_FAULT = 6   /* reserved                                                 */
} nx_status;

/* Bits OR-ed into *dev_status by the device. */
enum {
  NX_DEV_TIMEOUT = 1,       /* a bounded wait between thread blocks gave up; outputs of
                               the affected call are incomplete (the cache may be
                               partially compacted) */
  NX_DEV_BAD_LEN = 2,       /* lens[slice] < 0 or > capacity: slice left untouched */
  NX_DEV_BAD_BUDGET = 4,    /* the slice's budget < n_sink + n_recent or > budget_max:
                               slice left untouched */
  NX_DEV_BAD_PAGE = 8       /* a block_table entry is outside [0, num_pages): untouched */
};

enum { NX_DTYPE_F32 = 0, NX_DTYPE_BF16 = 1 };
enum { NX_MODE_RESERVOIR = 0, NX_MODE_TOPK = 1 };

/*
 * The KV cache. Two layouts:
 *   contiguous (page_size == 0): k, v [layers][seqs][kv_heads][capacity][head_dim],
 *                                pos    [layers][seqs][kv_heads][capacity];
 *   paged (page_size > 0):       k, v [layers][num_pages][kv_heads][page_size][head_dim],
 *                                pos    [layers][num_pages][kv_heads][page_size];
 *     slot j of (l, s, h) lives in page block_table[s * max_pages_per_seq + j / page_size]
 *     at row j % page_size; capacity = max_pages_per_seq * page_size.
 * lens [layers][seqs][kv_heads] int32: rows cached per slice (read, then set to
 * min(T, B) by kv_compact / nexus_evict_step). pos holds each row's absolute token
 * position (the token index of the Philox counter); it moves with its row.
 */
typedef struct nx_cache {
  int32_t layers, seqs, kv_heads;
  int32_t group;               /* G: query heads per KV head (GQA) */
  int32_t head_dim;            /* 64 or 128 */
  int32_t capacity;            /* rows per slice */
  int32_t page_size;           /* 0 (contiguous) or 8, 16, 32, 64, 128 */
  int32_t num_pages;           /* paged: pages per layer */
  int32_t max_pages_per_seq;   /* paged: columns of block_table */
  int32_t dtype;               /* NX_DTYPE_BF16 or NX_DTYPE_F32, for k, v and the queries */
  void* k;                     /* 16-byte aligned */
  void* v;                     /* 16-byte aligned */
  int32_t* pos;
  int32_t* lens;
  const int32_t* block_table;  /* paged only, [seqs][max_pages_per_seq] */
} nx_cache;

/*
 * Step parameters. Defaults from the paper's implementation details (§5.1):
 * lambda = 0.5, eps_tie = 1e-6, n = 5, b = 32; the paper's W = 16, H = 3. n_sink /
 * n_recent are the forced attention-sink and recency units of §2.3 (counted inside B;
 * at b = 1, 32 each is the default reading, one paper block each; at b = 32, one
 * block each).
 *
 * Reservoir keys (§2.3 Eq. (6)), per candidate unit j with weight w_j, from Philox4x32-10
 * with counter (pos_j, step, head id, seq id | g << 24) and key = seed, where pos_j is
 * the absolute position of the unit's first row and g the draw group:
 *   n_avg = 1: u = uniform(word 0 of group 0), key = ln(u) / w_j;
 *   n_avg = n > 1: u_i = uniform(word i mod 4 of group i / 4), l_i = ln(u_i),
 *     M = max_i l_i, r = 1 / w_j, key = M r + ln(sum_i exp((l_i - M) r)) = ln(n pi_j)
 *     (the order of pi_j = (1/n) sum_i u_i^(1/w_j); -ln n is left out as it does not
 *     change the order); a zero weight gives -inf.
 * uniform(x) = (2 (x >> 9) + 1) 2^-24; ln and exp are the library's specified binary32
 * functions (argument reduction by the exponent / Cody-Waite, then the atanh series
 * through f^13 / the Taylor series through r^7, each operation one IEEE rounding), so
 * the keys are reproducible bit for bit.
 */
typedef struct nx_params {
  int32_t window;              /* W, 1..64 */
  int32_t walk_len;            /* H, 0..min(W, 8): the last H window rows, oldest first */
  int32_t n_sink;              /* first n_sink units always kept */
  int32_t n_recent;            /* last n_recent units always kept (>= 1 when b > 1) */
  int32_t n_avg;               /* reservoir averaging count n of Eq. (6), 1..1024 */
  int32_t mode;                /* NX_MODE_RESERVOIR, or NX_MODE_TOPK (keep the top by w) */
  float lambda;                /* mixing weight of Eq. (2), >= 0 */
  float eps_tie;               /* recency tie-break of Eq. (5), >= 0 */
  const int32_t* budget;       /* device int32 [seqs]: B (units) per sequence */
  int32_t budget_max;          /* host bound: every budget <= budget_max <= ceil(capacity / b) */
  int32_t seq_id_base;         /* Philox sequence id of s is seq_id_base + s (< 2^24) */
  int32_t layer_id_base;       /* Philox head id of (l, h) is (layer_id_base + l) * kv_heads + h */
  uint32_t step;               /* Philox step id; callers advance it per eviction step */
  uint64_t seed;               /* Philox key */
  int32_t block_size;          /* b: 1 (decisions per token) or 32 (per 32-slot block) */
  int32_t reserved;            /* 0 */
  const int32_t* slice_budget; /* nullable device int32 [slices]: a budget per slice (e.g.
                                  from a head-adaptive allocation, §10); overrides
                                  budget[s] for every slice when given */
} nx_params;

/*
 * Bytes of workspace every entry point below needs for these arguments (0 on
 * invalid arguments). One workspace may serve all five calls in turn.
 */
size_t nexus_workspace_bytes(const nx_cache* cache, const nx_params* params);

/*
 * Direct scores, §2.1 Eq. (1) and §2.2 Eq. (3):
 *   Qbar_w = (1/G) sum_g q[g][w];  P_w = softmax_j(Qbar_w . k_j / sqrt(head_dim)) over
 *   the whole cache (no mask);     a_j = (1/W) sum_w P_w[j]; at b > 1, P_w is summed
 *   over each block (BlockSum; its rows still sum to 1, so rownorm is the identity)
 *   and a has one entry per block.
 * q: [layers][seqs][kv_heads * group][window][head_dim] in cache->dtype (device,
 *    16-byte aligned); query head kv_head * group + g belongs to KV head kv_head.
 * a_out: float [slices][capacity], entries j < N (units) written.
 * row_stats_out (nullable): float [slices][window][2] = (max_j logit, sum_j exp(logit - max)).
 * Errors: NX_ERR_INVALID_ARG, NX_ERR_WORKSPACE, NX_ERR_CUDA. Empty slices (T = 0)
 * write nothing.
 */
nx_status nexus_direct_scores(const nx_cache* cache, const void* q, const nx_params* params,
                              float* a_out, float* row_stats_out, void* ws, size_t ws_bytes,
                              int32_t* dev_status, nx_stream_t stream);

/*
 * Nexus weight, §2.2 Eqs. (4), (2), (5), over the N units (rows, or blocks whose rows
 * P_q are the block sums):
 *   C = 0; for the last H window rows q, oldest first: gamma_q = 1 + <P_q, C>,
 *   C += gamma_q P_q;  c~ = C / ||C||_1 (0 when H = 0);  s = a + lambda c~;
 *   w_j = s_j + eps_tie * j / (N - 1)  (the ramp is 0 when N = 1).
 * Computes everything from the cache and q (same layout as nexus_direct_scores).
 * w_out: float [slices][capacity]; ctilde_out (nullable): float [slices][capacity];
 * entries j < N written.
 */
nx_status nexus_walk(const nx_cache* cache, const void* q, const nx_params* params, float* w_out,
                     float* ctilde_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                     nx_stream_t stream);

/*
 * Weighted reservoir selection, §2.3 and Eq. (6), over the N units of each slice:
 *   forced F = units [0, n_sink) and [N - n_recent, N); K = B - |F|;
 *   for j not in F: kappa_j = the reservoir key of nx_params (n_avg = 1: ln(u)/w_j,
 *   Efraimidis-Spirakis; n_avg > 1: ln of the n-averaged priority); keep the K
 *   largest (kappa desc, then unit desc) -- in NX_MODE_TOPK kappa_j = w_j.
 * w: float [slices][capacity] (device), entries j < N. keep_idx: int32
 * [slices][capacity]: the first min(N, B) entries receive the kept units in ascending
 * order (0..N-1 when N <= B); the rest are not written. The cache is read (lens,
 * pos), not modified.
 */
nx_status nexus_reservoir_select(const float* w, const nx_cache* cache, const nx_params* params,
                                 int32_t* keep_idx, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, nx_stream_t stream);

/*
 * In-place compaction (§2.1: inference continues with K_S, V_S): the rows of the kept
 * units move, in order, to slots 0 .. n - 1 (k, v and pos), then lens = n. At b = 1,
 * n = min(T, B) and row i <- row keep_idx[i]; at b > 1 row i <- row keep_idx[i / b] b +
 * i mod b, and n = T when N <= B, else (B - 1) b + the size of the newest block (always
 * kept: n_recent >= 1). keep_idx: int32 [slices][capacity], ascending kept units, as
 * written by nexus_reservoir_select.
 * Rows at or beyond n and the block table are not modified; rows with
 * keep_idx[i] == i are not rewritten. Uses the workspace for tile flags; bounded
 * waits report NX_DEV_TIMEOUT.
 */
nx_status kv_compact(nx_cache* cache, const int32_t* keep_idx, const nx_params* params,
                     void* ws, size_t ws_bytes, int32_t* dev_status, nx_stream_t stream);

/*
 * kv_compact without a workspace, for callers that cannot allocate device memory:
 * code that runs where the CUDA allocator must not be called, such as inference
 * runtimes that plan and own every device byte up front, or real-time paths that may
 * not pay for (or fail on) an allocation in the middle of a step. The paper has no
 * counterpart; it is the same compaction as kv_compact, with the same arguments minus
 * the workspace, and the same results.
 *
 * Its scratch (a tile counter, the new lengths, one flag per tile of kCompactRows = 32
 * rows) lives in a 4 MiB static device array inside libnexus.so, held by every GPU
 * that loads the library until the process exits. Limit: 256 + 4 * slices (rounded
 * up to 256) + 4 * slices * ceil(budget_max * b / 32) (rounded up to 256) bytes must fit
 * in 4 MiB; larger calls return NX_ERR_WORKSPACE without launching anything. The
 * function calls no cudaMalloc, cudaFree or other allocating routine.
 * Every call made outside a stream capture looks up the array's device address for the
 * current device (a host-side query that allocates nothing) and remembers it; a call
 * made while its stream is being captured uses the remembered address, so the first
 * call on each device must come before any capture that includes this function (after
 * cudaDeviceReset, make one uncaptured call again). All calls share the one array,
 * which keeps the previous call's contents until the next call clears what must start
 * at zero: calls that overlap on the GPU (other streams, other host threads) race and
 * must be serialised by the caller.
 */
nx_status kv_compact_noalloc(nx_cache* cache, const int32_t* keep_idx, const nx_params* params,
                             int32_t* dev_status, nx_stream_t stream);

/*
 * One whole eviction step: scores, walk, reservoir selection and compaction for every
 * slice, with the same results as the four calls above in sequence.
 * keep_idx_out (nullable): int32 [slices][capacity] receives the kept slots.
 * The call only enqueues work on `stream` (four kernels), so it can
 * be captured into a CUDA graph; a replay reuses the captured arguments, `step`
 * included.
 */
nx_status nexus_evict_step(nx_cache* cache, const void* q, const nx_params* params,
                           int32_t* keep_idx_out, void* ws, size_t ws_bytes,
                           int32_t* dev_status, nx_stream_t stream);

/*
 * Testing hook for failure detection (not part of the method): kv_compact, except that
 * compaction tile number skip_signal_tile (slice * tiles_per_slice + tile, -1 for none)
 * never publishes its "read done" flag. Tiles that depend on it give up after their
 * bounded wait, skip their writes and set NX_DEV_TIMEOUT; nothing hangs and the CUDA
 * context stays usable. The cache is left partially compacted.
 */
nx_status nexus_debug_compact(nx_cache* cache, const int32_t* keep_idx, const nx_params* params,
                              void* ws, size_t ws_bytes, int32_t* dev_status, nx_stream_t stream,
                              long long skip_signal_tile);

/*
 * Testing hook: with on != 0, the scoring entry points use the CUDA-core scorer even
 * for shapes the tensor-core scorer covers (process-wide; 0 restores the default).
 */
void nexus_debug_force_simt(int32_t on);

/*
 * Testing hook: which kernel the compaction takes, process-wide. 1: the tile kernel
 * (32-row destination tiles claimed in order by persistent blocks, each waiting until the
 * earlier tiles of its slice have read their sources); 2: one warp per slice, its rows in
 * order through registers (rows of 128, 256 or 512 bytes); any other value: the automatic
 * choice (a warp per slice when there are at least eight slices per SM and the row size
 * allows). nexus_debug_compact always takes the tile kernel.
 */
void nexus_debug_compact_kernel(int32_t which);

/*
 * Testing hook: the tensor-core scorer's layout, process-wide. teams = 2 asks for two
 * independent pipelines per CTA (256 TMEM columns and eight epilogue warps each), 1 for
 * one pipeline per CTA (512 columns, sixteen epilogue warps), any other value for the
 * automatic choice (two for windows of up to 32 rows). Windows of 64 rows always take one.
 * When the two-pipeline layout cannot run, the automatic choice falls back to one and an
 * explicit 2 to the CUDA-core scorer.
 */
void nexus_debug_scorer_layout(int32_t teams);

/*
 * Diagnostics of the tensor-core scorer (not part of the method):
 * nexus_debug_set_trace installs a device buffer of grid x 1024 x 2 int64 that later
 * launches fill with (phase tag, globaltimer ns) pairs per pipeline; NULL turns it off.
 * nexus_debug_scorer_config writes the last launch's configuration from this host
 * thread: pipelines per CTA, CTAs per SM reported by the occupancy API, grid (CTAs),
 * tiles per chunk, TMEM buffers per pipeline, chunks per slice, TMEM columns per pipeline,
 * dynamic shared memory bytes. When the last call could not use the tensor-core scorer,
 * the first entry is negative: -1 no tensor-map encoder, -2 too many rows for one tensor
 * map, -3 tensor map rejected, -4 a slice has more chunks than co-resident pipelines,
 * -5 the cooperative launch did not fit, -6 no CTA fits on an SM.
 */
void nexus_debug_set_trace(long long* device_buffer);
void nexus_debug_scorer_config(int32_t* out8);

/* Static, human-readable name of a status code. */
const char* nx_status_string(nx_status status);

/*
 * Which scorer the most recent entry-point call made from this host thread used for the
 * direct scores and the walk (not part of the method; lets a caller see a fallback):
 *   NX_SCORER_NONE         the call computed no scores (selection or compaction only, or
 *                          it was rejected before launching anything);
 *   NX_SCORER_TENSOR_CORE  the tcgen05 scorer, which reads every cached key once;
 *   NX_SCORER_CUDA_CORE    the CUDA-core scorer (fp32 caches, shapes the tensor-core
 *                          scorer does not cover), which reads every cached key twice;
 *   NX_SCORER_TENSOR_CORE_TWO_PASS  the tcgen05 scorer in two launches, used when a
 *                          slice is longer than the single pass holds on chip at once
 *                          (152 SMs x 8 tiles x 128 rows = 155,648 rows on a GB300,
 *                          e.g. a one-shot eviction at the end of a long prefill):
 *                          the first stores every chunk's softmax record, the second
 *                          recomputes the logits and finishes; every key is read twice.
 * The results are the same within the score tolerance either way.
 */
enum { NX_SCORER_NONE = 0, NX_SCORER_TENSOR_CORE = 1, NX_SCORER_CUDA_CORE = 2,
       NX_SCORER_TENSOR_CORE_TWO_PASS = 3 };
int32_t nexus_last_scorer(void);

/* Kernels launched by the most recent call made from this host thread. */
int32_t nexus_last_launch_count(void);

/* Name of kernel launch i (0-based) of that call; "" when out of range. Static storage. */
const char* nexus_last_launch_name(int32_t i);

/*
 * Benchmark hook: the next entry-point call made from this host thread records
 * events[i] (cudaEvent_t handles, caller-owned) on its stream right after its i-th
 * kernel launch, for i < n. The request is consumed by that call; events must stay
 * valid until it returns.
 */
void nexus_profile_next_call(void* const* events, int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* NEXUS_H_ */
