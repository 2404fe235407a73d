// nx_select.cu -- retention set of every slice (Nexus Sampling paper, §2.3).
//
// Every slot j carries a 32-bit order key: 0xFFFFFFFF for the forced sink and recency
// slots, else the monotone image of kappa_j = ln(u_j)/w_j (reservoir) or w_j (top-K).
// Keeping the B largest composite keys (key, slot) keeps the forced slots plus the K
// largest kappa, ties to the newer slot. One thread block per slice finds the B-th
// largest composite by an MSB-first radix select (four 8-bit digit passes on the key,
// four more on the slot only when the threshold key is tied), then writes the kept
// slots in ascending order (per-warp runs, ballots, one scan of the warp totals).
#include <atomic>

#include "nx_internal.cuh"

namespace nx {
namespace {

constexpr int kSelThreads = 1024;

// Order key of every unit of every slice from caller-given weights (one thread per unit;
// a unit's Philox position is that of its first row). w may alias keys (each thread reads
// its unit's weight before writing its key).
template <int NT>
__global__ void keys_from_w_kernel(nx_cache c, nx_params p, const float* w, uint32_t* keys,
                                   const int32_t* __restrict__ newlen) {
  const int slice = blockIdx.x;
  if (newlen[slice] < 0) return;
  const int N = units_of(c.lens[slice], p.block_size);
  const int u = blockIdx.y * blockDim.x + threadIdx.x;
  if (u >= N) return;
  int l, s, h;
  slice_coords(c, slice, l, s, h);
  const long long o = (long long)slice * c.capacity + u;
  uint32_t key = kForcedKey;
  if (!(u < p.n_sink || u >= N - p.n_recent)) {
    const uint32_t head_id = (uint32_t)((p.layer_id_base + l) * c.kv_heads + h);
    key = candidate_key<NT>(w[o], c.pos[row_of(c, l, s, h, u * p.block_size)], p, head_id,
                            (uint32_t)(p.seq_id_base + s));
  }
  keys[o] = key;
}

constexpr int kDigitBits = 8;                   // four passes cover 32 bits
constexpr int kBins = 1 << kDigitBits;
constexpr int kBinsPerLane = kBins / 32;

// Find digit d with above(d) < need <= above(d) + hist[d], where above(d) counts
// elements whose digit is larger than d. Run by warp 0; writes (d, above(d), hist[d]).
__device__ __forceinline__ void pick_digit(const unsigned* hist, int need, int* out3) {
  const int lane = threadIdx.x & 31;
  unsigned cnt[kBinsPerLane];
  unsigned mine = 0;
#pragma unroll
  for (int b = 0; b < kBinsPerLane; ++b) {
    cnt[b] = hist[lane * kBinsPerLane + b];
    mine += cnt[b];
  }
  // above_lane = sum over lanes > lane (bins above this lane's 8 bins)
  unsigned incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += y;
  }
  unsigned above = incl - mine;
#pragma unroll
  for (int b = kBinsPerLane - 1; b >= 0; --b) {
    if ((int)above < need && need <= (int)(above + cnt[b])) {
      out3[0] = lane * kBinsPerLane + b;
      out3[1] = (int)above;
      out3[2] = (int)cnt[b];
    }
    above += cnt[b];
  }
}

// Histogram of kDigitBits-bit digits of the elements matching a prefix, with plain
// shared-memory atomics (measured faster than aggregating equal digits per warp first).
template <bool SMEM>
__device__ __forceinline__ void digit_hist(const uint32_t* keys, int T, uint32_t pmask,
                                           uint32_t prefix, int shift, bool by_slot,
                                           uint32_t tau, unsigned* hist) {
  // (keys in global memory: U loads in flight per thread before their atomics)
  constexpr int U = SMEM ? 1 : 8;
  for (int j0 = threadIdx.x; j0 < T; j0 += U * blockDim.x) {
    uint32_t kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * blockDim.x;
      kv[u] = j < T ? keys[j] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + u * blockDim.x;
      if (j >= T) break;
      const uint32_t k = kv[u];
      if (!by_slot) {
        if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (kBins - 1u)], 1u);
      } else if (k == tau && ((uint32_t)j & pmask) == prefix) {
        atomicAdd(&hist[((uint32_t)j >> shift) & (kBins - 1u)], 1u);
      }
    }
  }
}

template <bool SMEM>
__global__ void __launch_bounds__(kSelThreads)
select_kernel(nx_cache c, const uint32_t* __restrict__ keys, int32_t* __restrict__ keep,
              const int32_t* __restrict__ newlen, int bs) {
  extern __shared__ __align__(16) uint32_t s_keys[];
  grid_dep_trigger();
  grid_dep_wait();                 // keys and new lengths come from the kernels before
  const int slice = blockIdx.x;
  const int rows_left = newlen[slice];
  if (rows_left < 0) return;
  // decision units: the slice's T units, of which nl are kept (the new length in rows
  // covers nl units: whole ones and the newest, possibly partial, block)
  const int T = units_of(c.lens[slice], bs);
  const int nl = units_of(rows_left, bs);
  int32_t* out = keep + (long long)slice * c.capacity;
  if (T <= nl) {
    for (int j = threadIdx.x; j < T; j += blockDim.x) out[j] = j;
    return;
  }
  const int B = nl;
  const uint32_t* gk = keys + (long long)slice * c.capacity;
  const uint32_t* kk = gk;
  if (SMEM) {
    // stage the slice's keys: 16-byte loads, eight in flight per thread
    int j_tail = 0;
    if ((c.capacity & 3) == 0) {
      const int nv = T >> 2;
      const uint4* gv = reinterpret_cast<const uint4*>(gk);
      uint4* sv = reinterpret_cast<uint4*>(s_keys);
      constexpr int U = 8;
      for (int v0 = threadIdx.x; v0 < nv; v0 += U * blockDim.x) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * blockDim.x;
          if (v < nv) x[u] = __ldcs(gv + v);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * blockDim.x;
          if (v < nv) sv[v] = x[u];
        }
      }
      j_tail = nv * 4;
    }
    for (int j = j_tail + threadIdx.x; j < T; j += blockDim.x) s_keys[j] = __ldcs(gk + j);
    kk = s_keys;
    __syncthreads();
  }
  __shared__ unsigned hist[kBins];
  __shared__ int pick[3];
  __shared__ int wcount[kSelThreads / 32];

  // ---- radix select on the key ----
  uint32_t prefix = 0, pmask = 0;
  int need = B;
  int eq_count = 0;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    const uint32_t dmask = 0xFFu;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    digit_hist<SMEM>(kk, T, pmask, prefix, shift, false, 0, hist);
    __syncthreads();
    if (threadIdx.x < 32) pick_digit(hist, need, pick);
    __syncthreads();
    need -= pick[1];
    eq_count = pick[2];
    prefix |= (uint32_t)pick[0] << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  const uint32_t tau = prefix;   // the B-th largest key; keep `need` of its eq_count copies
  // ---- ties at tau: keep the `need` largest slots among key == tau ----
  int slot_tau = 0;
  if (eq_count > need) {
    uint32_t sp = 0, sm = 0;
    int sneed = need;
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      const uint32_t dmask = 0xFFu;
      for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      digit_hist<SMEM>(kk, T, sm, sp, shift, true, tau, hist);
      __syncthreads();
      if (threadIdx.x < 32) pick_digit(hist, sneed, pick);
      __syncthreads();
      sneed -= pick[1];
      sp |= (uint32_t)pick[0] << shift;
      sm |= dmask << shift;
      __syncthreads();
    }
    slot_tau = (int)sp;
  }
  // ---- write kept slots, ascending: every warp owns a contiguous run of slots, which it
  // reads 32 at a time (ballots count and place its survivors); one scan of the warp
  // totals gives each warp its output offset ----
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int span = ((T + nw - 1) / nw + 31) / 32 * 32;
  const int w0 = min(T, warp * span), w1 = min(T, w0 + span);
  // (keys in global memory: U rows of 32 loads in flight per warp)
  constexpr int U = SMEM ? 1 : 8;
  auto load = [&](int j0, bool (&t)[U]) {
    uint32_t kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + 32 * u + lane;
      kv[u] = j < w1 ? kk[j] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = j0 + 32 * u + lane;
      t[u] = j < w1 && ((kv[u] > tau) || (kv[u] == tau && j >= slot_tau));
    }
  };
  int cnt = 0;
  for (int j0 = w0; j0 < w1; j0 += 32 * U) {
    bool t[U];
    load(j0, t);
#pragma unroll
    for (int u = 0; u < U; ++u) cnt += __popc(__ballot_sync(0xffffffffu, t[u]));
  }
  if (lane == 0) wcount[warp] = cnt;
  __syncthreads();
  if (warp == 0) {
    const int cw = lane < nw ? wcount[lane] : 0;
    int wi = cw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) wcount[lane] = wi - cw;        // exclusive prefix of the warp totals
  }
  __syncthreads();
  int o = wcount[warp];
  for (int j0 = w0; j0 < w1; j0 += 32 * U) {
    bool t[U];
    load(j0, t);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const unsigned bal = __ballot_sync(0xffffffffu, t[u]);
      if (t[u]) out[o + __popc(bal & ((1u << lane) - 1u))] = j0 + 32 * u + lane;
      o += __popc(bal);
    }
  }
}


// ---------------------------------------------------------------------------
// Few, long slices: P blocks per slice, each holding one segment of the slice's keys in
// shared memory. Every radix pass, each block adds its segment's digit histogram into the
// slice's histogram in global memory and counts itself in; the slice's first block waits
// (bounded) for all P, picks the digit, clears the histogram and publishes the pick, which
// the others wait for (bounded). The kept units are then counted per segment and written
// at offsets that follow from the counts of the earlier segments. All P x slices blocks
// are co-resident (the host keeps their number within one per SM), so the waits end.
// ---------------------------------------------------------------------------
constexpr int kMultiMaxParts = 128;    // segments per slice
// scratch per slice: [0, 256) digit histogram; kArrive: pass arrivals; kPublished: passes
// published; kPick: the last pick (digit, above, count); kOutArrive: counts posted;
// kCounts: survivors per segment
constexpr int kArrive = 256, kPublished = 257, kPick = 260, kOutArrive = 264, kCounts = 320;
static_assert(kCounts + kMultiMaxParts <= kMultiStride, "scratch layout");

__device__ __forceinline__ void segment_hist(const uint32_t* keys, int j0, int n, uint32_t pmask,
                                             uint32_t prefix, int shift, bool by_slot,
                                             uint32_t tau, unsigned* hist) {
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const uint32_t k = keys[i];
    const uint32_t j = (uint32_t)(j0 + i);
    if (!by_slot) {
      if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & (kBins - 1u)], 1u);
    } else if (k == tau && (j & pmask) == prefix) {
      atomicAdd(&hist[(j >> shift) & (kBins - 1u)], 1u);
    }
  }
}

// One radix pass across the slice's P blocks; returns false when a wait ran out.
__device__ bool multi_pass(int* sc, int part, int P, int q, const unsigned* lhist, int need,
                           int* pick, int32_t* dev_status) {
  __shared__ int s_ok;
  __shared__ unsigned ghist[kBins];
  for (int i = threadIdx.x; i < kBins; i += blockDim.x)
    if (lhist[i]) atomicAdd(reinterpret_cast<unsigned*>(sc) + i, lhist[i]);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(sc + kArrive, 1);
    s_ok = 1;
  }
  __syncthreads();
  if (part == 0) {
    if (threadIdx.x == 0 && !wait_at_least(sc + kArrive, (q + 1) * P, dev_status)) s_ok = 0;
    __syncthreads();
    if (s_ok) {
      for (int i = threadIdx.x; i < kBins; i += blockDim.x) {
        ghist[i] = __ldcg(reinterpret_cast<const unsigned*>(sc) + i);
        sc[i] = 0;                      // cleared for the next pass
      }
      __syncthreads();
      if (threadIdx.x < 32) pick_digit(ghist, need, pick);
      __syncthreads();
      if (threadIdx.x == 0) {
        sc[kPick] = pick[0];
        sc[kPick + 1] = pick[1];
        sc[kPick + 2] = pick[2];
        __threadfence();
        st_release(sc + kPublished, q + 1);
      }
    }
  } else if (threadIdx.x == 0) {
    if (wait_at_least(sc + kPublished, q + 1, dev_status)) {
      pick[0] = __ldcg(sc + kPick);
      pick[1] = __ldcg(sc + kPick + 1);
      pick[2] = __ldcg(sc + kPick + 2);
    } else {
      s_ok = 0;
    }
  }
  __syncthreads();
  return s_ok != 0;
}

__global__ void __launch_bounds__(kSelThreads)
select_multi_kernel(nx_cache c, const uint32_t* __restrict__ keys, int32_t* __restrict__ keep,
                    const int32_t* __restrict__ newlen, int bs, int P, int seg, int* scratch,
                    int32_t* dev_status) {
  extern __shared__ __align__(16) uint32_t s_keys[];
  grid_dep_trigger();
  grid_dep_wait();                 // keys and new lengths come from the kernels before
  const int slice = blockIdx.x / P, part = blockIdx.x % P;
  const int rows_left = newlen[slice];
  if (rows_left < 0) return;
  const int T = units_of(c.lens[slice], bs);
  const int nl = units_of(rows_left, bs);
  int32_t* out = keep + (long long)slice * c.capacity;
  const int j0 = part * seg;
  const int n = max(0, min(T, j0 + seg) - j0);       // this block's units
  if (T <= nl) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[j0 + i] = j0 + i;
    return;
  }
  int* sc = scratch + (long long)slice * kMultiStride;
  // stage the segment's keys (16-byte loads: j0 and the capacity are multiples of 4)
  const uint32_t* gk = keys + (long long)slice * c.capacity + j0;
  {
    const int nv = (c.capacity & 3) == 0 ? (n >> 2) : 0;
    const uint4* gv = reinterpret_cast<const uint4*>(gk);
    uint4* sv = reinterpret_cast<uint4*>(s_keys);
    for (int v = threadIdx.x; v < nv; v += blockDim.x) sv[v] = __ldcs(gv + v);
    for (int i = nv * 4 + threadIdx.x; i < n; i += blockDim.x) s_keys[i] = __ldcs(gk + i);
  }
  __shared__ unsigned hist[kBins];
  __shared__ int pick[3];
  __shared__ int wcount[kSelThreads / 32];
  __syncthreads();
  // ---- radix select on the key, then (ties at the threshold) on the unit ----
  uint32_t prefix = 0, pmask = 0;
  int need = nl;
  int eq_count = 0;
  int q = 0;
  for (int pass = 0; pass < 4; ++pass, ++q) {
    const int shift = 24 - 8 * pass;
    for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    segment_hist(s_keys, j0, n, pmask, prefix, shift, false, 0, hist);
    __syncthreads();
    if (!multi_pass(sc, part, P, q, hist, need, pick, dev_status)) return;
    need -= pick[1];
    eq_count = pick[2];
    prefix |= (uint32_t)pick[0] << shift;
    pmask |= 0xFFu << shift;
    __syncthreads();
  }
  const uint32_t tau = prefix;
  int slot_tau = 0;
  if (eq_count > need) {
    uint32_t sp = 0, sm = 0;
    int sneed = need;
    for (int pass = 0; pass < 4; ++pass, ++q) {
      const int shift = 24 - 8 * pass;
      for (int i = threadIdx.x; i < kBins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      segment_hist(s_keys, j0, n, sm, sp, shift, true, tau, hist);
      __syncthreads();
      if (!multi_pass(sc, part, P, q, hist, sneed, pick, dev_status)) return;
      sneed -= pick[1];
      sp |= (uint32_t)pick[0] << shift;
      sm |= 0xFFu << shift;
      __syncthreads();
    }
    slot_tau = (int)sp;
  }
  // ---- kept units of this segment, ascending: per-warp runs, ballots, one scan ----
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int span = ((n + nw - 1) / nw + 31) / 32 * 32;
  const int w0 = min(n, warp * span), w1 = min(n, w0 + span);
  auto kept = [&](int i) {
    if (i >= w1) return false;
    const uint32_t k = s_keys[i];
    return (k > tau) || (k == tau && j0 + i >= slot_tau);
  };
  int cnt = 0;
  for (int i0 = w0; i0 < w1; i0 += 32) cnt += __popc(__ballot_sync(0xffffffffu, kept(i0 + lane)));
  if (lane == 0) wcount[warp] = cnt;
  __syncthreads();
  __shared__ int s_base, s_ok2;
  if (warp == 0) {
    const int cw = lane < nw ? wcount[lane] : 0;
    int wi = cw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) wcount[lane] = wi - cw;        // exclusive prefix of the warp totals
    const int total = __shfl_sync(0xffffffffu, wi, 31);
    if (lane == 0) {
      // post this segment's count, then wait for every segment's and add the earlier ones
      sc[kCounts + part] = total;
      __threadfence();
      atomicAdd(sc + kOutArrive, 1);
      s_ok2 = wait_at_least(sc + kOutArrive, P, dev_status) ? 1 : 0;
      int base = 0;
      for (int p2 = 0; p2 < part; ++p2) base += __ldcg(sc + kCounts + p2);
      s_base = base;
    }
  }
  __syncthreads();
  if (!s_ok2) return;
  int o = s_base + wcount[warp];
  for (int i0 = w0; i0 < w1; i0 += 32) {
    const bool t = kept(i0 + lane);
    const unsigned bal = __ballot_sync(0xffffffffu, t);
    if (t) out[o + __popc(bal & ((1u << lane) - 1u))] = j0 + i0 + lane;
    o += __popc(bal);
  }
}

}  // namespace

cudaError_t launch_keys_from_w(const nx_cache& c, const nx_params& p, const float* w,
                               uint32_t* keys, const int32_t* newlen, cudaStream_t st,
                               int* launches) {
  const long long slices = (long long)c.layers * c.seqs * c.kv_heads;
  dim3 grid((unsigned)slices, (c.capacity + 255) / 256);
  // the usual draw counts unrolled with their draws in registers; the rest drawn twice
  switch (p.n_avg) {
    case 1: keys_from_w_kernel<1><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 2: keys_from_w_kernel<2><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 3: keys_from_w_kernel<3><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 4: keys_from_w_kernel<4><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 5: keys_from_w_kernel<5><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 6: keys_from_w_kernel<6><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 7: keys_from_w_kernel<7><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    case 8: keys_from_w_kernel<8><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
    default: keys_from_w_kernel<0><<<grid, 256, 0, st>>>(c, p, w, keys, newlen); break;
  }
  note_launch(st, launches, "keys_from_w");
  return cudaGetLastError();
}

cudaError_t launch_select(const nx_cache& c, const uint32_t* keys, int32_t* keep,
                          const int32_t* newlen, int block_size, int* scratch,
                          int32_t* dev_status, cudaStream_t st, int* launches) {
  const long long slices = (long long)c.layers * c.seqs * c.kv_heads;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Few slices too long for one block's shared memory (over 48K units; at least two SMs
  // per slice): P co-resident blocks per slice, one segment of at most 48K units each
  // (measured: 86 -> 45 us for 32 slices of 131072 units; for slices of 8192 units the
  // passes' inter-block waits cost more than they save, 14 -> 24 us)
  const int cap_units = (c.capacity + block_size - 1) / block_size;
  if (scratch && slices <= kMultiSlices && 2 * slices <= sms && cap_units > 48 * 1024 &&
      dev >= 0 && dev < 64) {
    int P = (int)min((long long)kMultiMaxParts, sms / slices);
    const int seg = ((cap_units + P - 1) / P + 31) / 32 * 32;
    if (seg <= 48 * 1024) {
      P = (cap_units + seg - 1) / seg;
      static std::atomic<bool> multi_set[64];   // a racing second set is harmless
      if (!multi_set[dev].load(std::memory_order_acquire)) {
        const cudaError_t e = cudaFuncSetAttribute(
            select_multi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 48 * 1024 * 4);
        if (e != cudaSuccess) return e;
        multi_set[dev].store(true, std::memory_order_release);
      }
      const cudaError_t e = launch_after(select_multi_kernel, dim3((unsigned)(slices * P)),
                                         dim3(kSelThreads), (size_t)seg * 4, st, c, keys, keep,
                                         newlen, block_size, P, seg, scratch, dev_status);
      if (e != cudaSuccess) return e;
      note_launch(st, launches, "select_multi");
      return cudaGetLastError();
    }
  }
  // keys of a slice in shared memory when they fit (up to 48K slots), else from L2
  constexpr int kSmemKeys = 48 * 1024;
  if (c.capacity <= kSmemKeys) {
    const size_t bytes = (size_t)c.capacity * 4;
    static std::atomic<bool> attr_set[64];   // a racing second set is harmless
    if (dev >= 0 && dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
      cudaError_t e = cudaFuncSetAttribute(select_kernel<true>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kSmemKeys * 4);
      if (e != cudaSuccess) return e;
      attr_set[dev].store(true, std::memory_order_release);
    }
    const cudaError_t e = launch_after(select_kernel<true>, dim3((unsigned)slices),
                                       dim3(kSelThreads), bytes, st, c, keys, keep, newlen,
                                       block_size);
    if (e != cudaSuccess) return e;
  } else {
    const cudaError_t e = launch_after(select_kernel<false>, dim3((unsigned)slices),
                                       dim3(kSelThreads), 0, st, c, keys, keep, newlen,
                                       block_size);
    if (e != cudaSuccess) return e;
  }
  note_launch(st, launches, "select");
  return cudaGetLastError();
}

}  // namespace nx
