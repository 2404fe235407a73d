// nx_api.cu -- the C ABI of libnexus.so (declared in include/nexus.h): argument checks,
// the workspace layout, and the kernel sequence of every entry point.
#include <math.h>
#include <string.h>

#include <atomic>

#include "nx_internal.cuh"

namespace nx {
namespace {

thread_local int32_t g_last_launches = 0;
thread_local int32_t g_last_scorer = NX_SCORER_NONE;
std::atomic<bool> g_force_simt{false};   // set by nexus_debug_force_simt (tests, comparisons)
constexpr int kMaxLaunchNames = 16;
thread_local const char* g_launch_names[kMaxLaunchNames];
thread_local void* const* g_prof_events = nullptr;   // armed by nexus_profile_next_call
thread_local int32_t g_prof_n = 0;
thread_local bool g_prof_active = false;

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool valid_cache(const nx_cache* c) {
  if (!c) return false;
  if (c->layers < 1 || c->seqs < 1 || c->kv_heads < 1 || c->group < 1) return false;
  if (c->head_dim != 64 && c->head_dim != 128) return false;
  if (c->dtype != NX_DTYPE_BF16 && c->dtype != NX_DTYPE_F32) return false;
  if (c->capacity < 1 || c->capacity > (1 << 24)) return false;
  if (!c->k || !c->v || !c->pos || !c->lens) return false;
  if (((uintptr_t)c->k & 15u) || ((uintptr_t)c->v & 15u)) return false;
  const long long slices = (long long)c->layers * c->seqs * c->kv_heads;
  if (slices > (1LL << 31) - 1 || slices * c->capacity > (1LL << 40)) return false;
  if (c->page_size != 0) {
    const int ps = c->page_size;
    if (ps != 8 && ps != 16 && ps != 32 && ps != 64 && ps != 128) return false;
    if (c->num_pages < 1 || c->max_pages_per_seq < 1 || !c->block_table) return false;
    if ((long long)c->max_pages_per_seq * ps != c->capacity) return false;
  }
  return true;
}

nx_status check_params(const nx_cache* c, const nx_params* p) {
  if (!p) return NX_ERR_INVALID_ARG;
  if (p->window < 1 || p->window > kMaxWindow) return NX_ERR_INVALID_ARG;
  if (p->walk_len < 0 || p->walk_len > kMaxWalk || p->walk_len > p->window)
    return NX_ERR_INVALID_ARG;
  if (p->n_sink < 0 || p->n_recent < 0) return NX_ERR_INVALID_ARG;
  if (p->mode != NX_MODE_RESERVOIR && p->mode != NX_MODE_TOPK) return NX_ERR_INVALID_ARG;
  if (!(p->lambda >= 0.f) || !isfinite(p->lambda)) return NX_ERR_INVALID_ARG;
  if (!(p->eps_tie >= 0.f) || !isfinite(p->eps_tie)) return NX_ERR_INVALID_ARG;
  if (!p->budget) return NX_ERR_INVALID_ARG;
  if (p->block_size != 1 && p->block_size != 32) {
    if (p->block_size < 1) return NX_ERR_INVALID_ARG;
    return NX_ERR_UNSUPPORTED;
  }
  if (p->block_size > 1 && p->n_recent < 1) return NX_ERR_INVALID_ARG;   // newest block kept
  if (p->reserved != 0) return NX_ERR_INVALID_ARG;
  const int max_units = (c->capacity + p->block_size - 1) / p->block_size;
  if (p->budget_max < p->n_sink + p->n_recent || p->budget_max > max_units)
    return NX_ERR_INVALID_ARG;
  if (p->seq_id_base < 0 || (long long)p->seq_id_base + c->seqs > (1LL << 24))
    return NX_ERR_INVALID_ARG;
  if (p->layer_id_base < 0) return NX_ERR_INVALID_ARG;
  if (p->n_avg < 1 || p->n_avg > kMaxAvg) return NX_ERR_INVALID_ARG;
  return NX_OK;
}

WsLayout layout_of(const nx_cache* c, const nx_params* p) {
  WsLayout L{};
  L.slices = (long long)c->layers * c->seqs * c->kv_heads;
  L.max_chunks = (c->capacity + 127) / 128;
  L.stats_stride = (int)align_up(2 * p->window + kMaxPairs, 4);
  L.tiles_per_slice =
      (int)(((long long)p->budget_max * p->block_size + kCompactRows - 1) / kCompactRows);
  if (L.tiles_per_slice < 1) L.tiles_per_slice = 1;
  size_t o = 0;
  L.counters = o;
  L.work = o;
  o += 64;
  L.barriers = o;
  o += align_up((size_t)L.slices * 8, 256);
  L.tile_flags = o;
  o += align_up((size_t)L.slices * L.tiles_per_slice * 4, 256);
  L.select_scratch = o;
  o += align_up((size_t)(L.slices < kMultiSlices ? L.slices : kMultiSlices) * kMultiStride * 4, 256);
  L.counters_bytes = o - L.counters;
  const size_t cells = (size_t)L.slices * c->capacity;
  L.keys = o;
  o += align_up(cells * 4, 256);
  L.stats = o;
  o += align_up((size_t)L.slices * L.max_chunks * L.stats_stride * 4, 256);
  L.qbar = o;
  o += align_up((size_t)L.slices * p->window * c->head_dim * 4, 256);
  L.newlen = o;
  o += align_up((size_t)L.slices * 4, 256);
  L.keep = o;
  o += align_up(cells * 4, 256);
  L.total = o;
  return L;
}

nx_status common_checks(const nx_cache* c, const nx_params* p, void* ws, size_t ws_bytes,
                        int32_t* dev_status, WsLayout* L) {
  if (!valid_cache(c)) return NX_ERR_INVALID_ARG;
  const nx_status ps = check_params(c, p);
  if (ps != NX_OK) return ps;
  if (!dev_status) return NX_ERR_INVALID_ARG;
  *L = layout_of(c, p);
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < L->total) return NX_ERR_WORKSPACE;
  return NX_OK;
}

}  // namespace

nx_status finish(cudaError_t e, int launches) {
  g_last_launches = launches;
  if (g_prof_active) {
    g_prof_active = false;
    g_prof_events = nullptr;
    g_prof_n = 0;
  }
  return e == cudaSuccess ? NX_OK : NX_ERR_CUDA;
}

// Called at the start of every entry point: consumes an armed profiling request.
void begin_call() {
  g_last_launches = 0;
  g_last_scorer = NX_SCORER_NONE;
  g_prof_active = g_prof_events != nullptr;
}

namespace {

#define NX_TRY(expr)                         \
  do {                                       \
    cudaError_t e_ = (expr);                 \
    if (e_ != cudaSuccess) return finish(e_, launches); \
  } while (0)

// Scores (and whatever `out` asks for) for every slice: the tensor-core scorer for the
// shapes it covers, the CUDA-core scorer otherwise. The counters region must be zero.
cudaError_t run_scores(const nx_cache& c, const void* q, const nx_params& p, const WsLayout& L,
                       char* ws, const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                       int* launches) {
  const bool tc = tc_supported(c, p) && !g_force_simt.load(std::memory_order_relaxed);
  cudaError_t e = launch_prep(c, q, p, L, ws, dev_status, st, launches, tc ? 2 : 1);
  if (e != cudaSuccess) return e;
  if (tc) {
    bool used = false, two_pass = false;
    e = launch_score_tc(c, p, q, L, ws, out, dev_status, st, launches, &used, &two_pass);
    if (e != cudaSuccess) return e;
    if (used) {
      g_last_scorer = two_pass ? NX_SCORER_TENSOR_CORE_TWO_PASS : NX_SCORER_TENSOR_CORE;
      return e;
    }
    // not launchable for this size: the CUDA-core path needs the fp32 queries
    e = launch_prep(c, q, p, L, ws, dev_status, st, launches, 1);
    if (e != cudaSuccess) return e;
  }
  g_last_scorer = NX_SCORER_CUDA_CORE;
  return launch_score_simt(c, p, L, ws, out, dev_status, st, launches);
}

}  // namespace

void note_launch(cudaStream_t st, int* launches, const char* name) {
  if (*launches < kMaxLaunchNames) g_launch_names[*launches] = name;
  // Inside a stream capture the records must be external to become event-record nodes
  // of the graph (so that replays time the launches too).
  if (g_prof_active && *launches < g_prof_n && g_prof_events[*launches]) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(st, &cs);
    cudaEvent_t ev = reinterpret_cast<cudaEvent_t>(g_prof_events[*launches]);
    if (cs == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
    else
      cudaEventRecord(ev, st);
  }
  *launches += 1;
}

}  // namespace nx

using namespace nx;

extern "C" {

size_t nexus_workspace_bytes(const nx_cache* cache, const nx_params* params) {
  if (!valid_cache(cache) || check_params(cache, params) != NX_OK) return 0;
  return layout_of(cache, params).total;
}

nx_status nexus_direct_scores(const nx_cache* cache, const void* q, const nx_params* params,
                              float* a_out, float* row_stats_out, void* ws, size_t ws_bytes,
                              int32_t* dev_status, nx_stream_t stream) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!q || ((uintptr_t)q & 15u) || !a_out) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  // the counters are zeroed by the first kernel (prep)
  ScoreOut out{};
  out.a = a_out;
  out.row_stats = row_stats_out;
  out.flags = kEmitA | (row_stats_out ? kEmitStats : 0);
  NX_TRY(run_scores(*cache, q, *params, L, w, out, dev_status, st, &launches));
  return finish(cudaSuccess, launches);
}

nx_status nexus_walk(const nx_cache* cache, const void* q, const nx_params* params, float* w_out,
                     float* ctilde_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                     nx_stream_t stream) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!q || ((uintptr_t)q & 15u) || !w_out) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  // the counters are zeroed by the first kernel (prep)
  ScoreOut out{};
  out.w = w_out;
  out.ctilde = ctilde_out;
  out.flags = kEmitW | (ctilde_out ? kEmitC : 0);
  NX_TRY(run_scores(*cache, q, *params, L, w, out, dev_status, st, &launches));
  return finish(cudaSuccess, launches);
}

nx_status nexus_reservoir_select(const float* w_in, const nx_cache* cache, const nx_params* params,
                                 int32_t* keep_idx, void* ws, size_t ws_bytes,
                                 int32_t* dev_status, nx_stream_t stream) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!w_in || !keep_idx) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int32_t* newlen = reinterpret_cast<int32_t*>(w + L.newlen);
  uint32_t* keys = reinterpret_cast<uint32_t*>(w + L.keys);
  NX_TRY(cudaMemsetAsync(w + L.counters, 0, L.counters_bytes, st));
  NX_TRY(launch_newlen(*cache, *params, newlen, dev_status, st, &launches));
  NX_TRY(launch_keys_from_w(*cache, *params, w_in, keys, newlen, st, &launches));
  NX_TRY(launch_select(*cache, keys, keep_idx, newlen, params->block_size,
                       reinterpret_cast<int*>(w + L.select_scratch), dev_status, st, &launches));
  return finish(cudaSuccess, launches);
}

nx_status kv_compact(nx_cache* cache, const int32_t* keep_idx, const nx_params* params, void* ws,
                     size_t ws_bytes, int32_t* dev_status, nx_stream_t stream) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!keep_idx) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int32_t* newlen = reinterpret_cast<int32_t*>(w + L.newlen);
  NX_TRY(cudaMemsetAsync(w + L.counters, 0, L.counters_bytes, st));
  NX_TRY(launch_newlen(*cache, *params, newlen, dev_status, st, &launches));
  NX_TRY(launch_compact(*cache, *params, L, w, keep_idx, newlen, dev_status, st, &launches));
  return finish(cudaSuccess, launches);
}

nx_status nexus_evict_step(nx_cache* cache, const void* q, const nx_params* params,
                           int32_t* keep_idx_out, void* ws, size_t ws_bytes,
                           int32_t* dev_status, nx_stream_t stream) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!q || ((uintptr_t)q & 15u)) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int32_t* newlen = reinterpret_cast<int32_t*>(w + L.newlen);
  uint32_t* keys = reinterpret_cast<uint32_t*>(w + L.keys);
  int32_t* keep = keep_idx_out ? keep_idx_out : reinterpret_cast<int32_t*>(w + L.keep);
  // the counters are zeroed by the first kernel (prep)
  ScoreOut out{};
  out.keys = keys;
  out.flags = kEmitKeys;
  NX_TRY(run_scores(*cache, q, *params, L, w, out, dev_status, st, &launches));
  // n > 1: the scorers left w in the key array; the n-averaged keys replace it in place
  if (params->n_avg > 1)
    NX_TRY(launch_keys_from_w(*cache, *params, reinterpret_cast<const float*>(keys), keys,
                              newlen, st, &launches));
  NX_TRY(launch_select(*cache, keys, keep, newlen, params->block_size,
                       reinterpret_cast<int*>(w + L.select_scratch), dev_status, st, &launches));
  NX_TRY(launch_compact(*cache, *params, L, w, keep, newlen, dev_status, st, &launches));
  return finish(cudaSuccess, launches);
}

nx_status nexus_debug_compact(nx_cache* cache, const int32_t* keep_idx, const nx_params* params,
                              void* ws, size_t ws_bytes, int32_t* dev_status, nx_stream_t stream,
                              long long skip_signal_tile) {
  int launches = 0;
  begin_call();
  WsLayout L;
  nx_status s = common_checks(cache, params, ws, ws_bytes, dev_status, &L);
  if (s != NX_OK) return s;
  if (!keep_idx) return NX_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  int32_t* newlen = reinterpret_cast<int32_t*>(w + L.newlen);
  NX_TRY(cudaMemsetAsync(w + L.counters, 0, L.counters_bytes, st));
  NX_TRY(launch_newlen(*cache, *params, newlen, dev_status, st, &launches));
  NX_TRY(launch_compact(*cache, *params, L, w, keep_idx, newlen, dev_status, st, &launches,
                        skip_signal_tile));
  return finish(cudaSuccess, launches);
}

const char* nx_status_string(nx_status status) {
  switch (status) {
    case NX_OK: return "NX_OK";
    case NX_ERR_INVALID_ARG: return "NX_ERR_INVALID_ARG";
    case NX_ERR_UNSUPPORTED: return "NX_ERR_UNSUPPORTED";
    case NX_ERR_CUDA: return "NX_ERR_CUDA";
    case NX_ERR_TIMEOUT: return "NX_ERR_TIMEOUT";
    case NX_ERR_WORKSPACE: return "NX_ERR_WORKSPACE";
    case NX_ERR_DEVICE_FAULT: return "NX_ERR_DEVICE_FAULT";
  }
  return "NX_UNKNOWN_STATUS";
}

int32_t nexus_last_launch_count(void) { return g_last_launches; }

int32_t nexus_last_scorer(void) { return g_last_scorer; }

void nexus_debug_force_simt(int32_t on) { g_force_simt.store(on != 0); }

void nexus_debug_compact_kernel(int32_t which) { nx::compact_set_kernel(which); }

void nexus_debug_scorer_layout(int32_t teams) {
  nx::tc_set_layout(teams == 1 || teams == 2 ? teams : 0);
}

void nexus_debug_set_trace(long long* device_buffer) { tc_set_trace(device_buffer); }

void nexus_debug_scorer_config(int32_t* out8) {
  if (out8) tc_last_config(out8);
}

const char* nexus_last_launch_name(int32_t i) {
  return (i >= 0 && i < g_last_launches && i < kMaxLaunchNames) ? g_launch_names[i] : "";
}

void nexus_profile_next_call(void* const* events, int32_t n) {
  g_prof_events = events;
  g_prof_n = n;
}

}  // extern "C"
