// nx_compact.cu -- in-place stable compaction (Nexus Sampling paper, §2.1: inference
// continues with K_S, V_S): row i <- row src(i) for k, v and pos, i < n, where src(i) =
// keep[i] at block size b = 1 and keep[i / b] b + i mod b for blocks of b rows (keep holds
// the kept units, ascending).
//
// keep is ascending with keep[u] >= u, so src(i) >= i and writing row i can only destroy a
// source that a destination i' <= i still needs. Destinations are cut into tiles of kCompactRows rows,
// claimed in increasing order through one global counter (which skips the empty tail
// tiles of each slice). A tile first copies all its
// sources into shared memory, then publishes "read done", then waits (bounded) until the
// earlier tiles of its slice have published, and only then writes. Each block holds two
// tiles: the next one's reads (cp.async) overlap the current one's wait and writes.
// No deadlock: the lowest unpublished tile is either a block's current tile, published
// without waiting, or its next one, published once the current tile -- which only waits
// on lower, hence published, tiles -- is written. Rows with keep[i] == i are neither
// read nor written.
#include <atomic>

#include "nx_internal.cuh"

namespace nx {
namespace {

constexpr int kCompactThreads = 256;

__device__ __forceinline__ bool slice_ok(const nx_cache& c, const nx_params& p, int slice,
                                         int32_t* dev_status) {
  int l, s, h;
  slice_coords(c, slice, l, s, h);
  const int T = c.lens[slice];
  const int B = budget_of(p, slice, s);
  if (T < 0 || T > c.capacity) {
    atomicOr(dev_status, NX_DEV_BAD_LEN);
    return false;
  }
  if (B < p.n_sink + p.n_recent || B > p.budget_max) {
    atomicOr(dev_status, NX_DEV_BAD_BUDGET);
    return false;
  }
  if (c.page_size > 0) {
    const int npg = (T + c.page_size - 1) / c.page_size;
    if (npg > c.max_pages_per_seq) {
      atomicOr(dev_status, NX_DEV_BAD_PAGE);
      return false;
    }
    for (int i = 0; i < npg; ++i) {
      const int pg = c.block_table[(long long)s * c.max_pages_per_seq + i];
      if (pg < 0 || pg >= c.num_pages) {
        atomicOr(dev_status, NX_DEV_BAD_PAGE);
        return false;
      }
    }
  }
  return true;
}

// new length per slice (-1: invalid slice, left untouched)
__global__ void newlen_kernel(nx_cache c, nx_params p, int32_t* __restrict__ newlen,
                              int32_t* dev_status, long long slices) {
  const long long slice = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (slice >= slices) return;
  int l, s, h;
  slice_coords(c, (int)slice, l, s, h);
  newlen[slice] = slice_ok(c, p, (int)slice, dev_status)
                      ? rows_kept(c.lens[slice], budget_of(p, (int)slice, s), p.block_size)
                      : -1;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Per-buffer description of a claimed tile.
struct TileSlot {
  long long tile;   // >= total: none
  int slice, t, i0, n, nl, l, s, h;
  int moves;        // any row with keep[i] != i
};

// Two shared-memory buffers: while tile c's rows are written from one, tile c+1's sources
// stream into the other with cp.async.
__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(nx_cache c, const int32_t* __restrict__ keep, const int32_t* __restrict__ newlen,
               int* tile_flags, unsigned long long* work, int tiles_per_slice,
               long long total_tiles, int32_t* dev_status, long long skip_signal_tile, int bs) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int row_bytes = c.head_dim * (c.dtype == NX_DTYPE_BF16 ? 2 : 4);
  const int chunks = row_bytes / 16;                    // 16-byte pieces per row
  const int per_buf = 2 * kCompactRows * chunks;        // K then V
  uint4* bufs = reinterpret_cast<uint4*>(smem);
  __shared__ int s_src[2][kCompactRows];
  __shared__ int s_pos[2][kCompactRows];
  __shared__ long long s_srow[2][kCompactRows];   // source and destination row indices
  __shared__ long long s_drow[2][kCompactRows];
  __shared__ TileSlot s_slot[2];
  __shared__ long long s_claim;
  __shared__ int s_ok;
  grid_dep_wait();                 // kept slots and new lengths come from the kernels before
  uint4* K = reinterpret_cast<uint4*>(c.k);
  uint4* V = reinterpret_cast<uint4*>(c.v);

  // claim the next tile (in increasing order over the whole grid) and start its reads
  auto stage = [&](int b) {
    if (threadIdx.x == 0) {
      // Claim the next tile; tiles past their slice's new length (and every tile of a
      // rejected slice) hold no rows and are waited on by nobody, so once one is met the
      // counter jumps to the next slice. Tile 0 of a valid slice is always taken (it
      // writes the new length).
      long long x = (long long)atomicAdd(work, 1ULL);
      while (x < total_tiles) {
        const int sx = (int)(x / tiles_per_slice), tx = (int)(x % tiles_per_slice);
        const int nx = newlen[sx];
        if (nx >= 0 && (tx == 0 || tx * kCompactRows < nx)) break;
        atomicMax(work, (unsigned long long)(sx + 1) * (unsigned long long)tiles_per_slice);
        x = (long long)atomicAdd(work, 1ULL);
      }
      s_claim = x;
    }
    __syncthreads();
    TileSlot sl;
    sl.tile = s_claim;
    sl.moves = 0;
    sl.n = 0;
    if (sl.tile < total_tiles) {
      sl.slice = (int)(sl.tile / tiles_per_slice);
      sl.t = (int)(sl.tile % tiles_per_slice);
      sl.nl = newlen[sl.slice];
      sl.i0 = sl.t * kCompactRows;
      slice_coords(c, sl.slice, sl.l, sl.s, sl.h);
      if (sl.nl >= 0 && sl.i0 < sl.nl) sl.n = min(kCompactRows, sl.nl - sl.i0);
    }
    const int32_t* kp = (sl.n > 0) ? keep + (long long)sl.slice * c.capacity : nullptr;
    bool mv = false;
    if (threadIdx.x < kCompactRows) {
      const int i = threadIdx.x;
      // source slot of destination slot i0 + i: the kept unit's row at the same offset
      // (units are rows at b = 1, blocks of bs rows otherwise)
      const int dst = sl.i0 + i;
      const int src = (i < sl.n) ? (bs == 1 ? kp[dst] : kp[dst / bs] * bs + dst % bs) : 0;
      s_src[b][i] = src;
      mv = i < sl.n && src != sl.i0 + i;
      if (mv) {
        const long long sr = row_of(c, sl.l, sl.s, sl.h, src);
        s_srow[b][i] = sr;
        s_drow[b][i] = row_of(c, sl.l, sl.s, sl.h, sl.i0 + i);
        s_pos[b][i] = c.pos[sr];
      }
    }
    sl.moves = __syncthreads_or(mv);      // any row of the tile moves
    if (threadIdx.x == 0) s_slot[b] = sl;
    __syncthreads();
    sl = s_slot[b];
    if (sl.moves) {
      uint4* bk = bufs + b * per_buf;
      uint4* bv = bk + kCompactRows * chunks;
      for (int e = threadIdx.x; e < sl.n * chunks; e += blockDim.x) {
        const int i = e / chunks, ch = e - i * chunks;
        if (s_src[b][i] != sl.i0 + i) {
          const long long r = s_srow[b][i];
          cp_async16(bk + e, K + r * chunks + ch);
          cp_async16(bv + e, V + r * chunks + ch);
        }
      }
    }
    cp_async_commit();
  };

  int b = 0;
  stage(b);
  for (;;) {
    const TileSlot cur = s_slot[b];
    if (cur.tile >= total_tiles) break;
    // the current tile's reads are complete: publish "read done"
    cp_async_wait_all();
    __syncthreads();
    if (threadIdx.x == 0) {
      // the release store orders the block's completed reads (barrier above) before the
      // flag; tiles past the slice's new length are read by no later tile of the slice
      if (cur.n > 0 && cur.tile != skip_signal_tile) st_release(tile_flags + cur.tile, 1);
      if (cur.t == 0 && cur.tile < total_tiles && cur.nl >= 0) c.lens[cur.slice] = cur.nl;
      s_ok = 1;
    }
    // start the next tile's reads; they proceed while this tile waits and writes
    stage(b ^ 1);
    if (cur.moves) {
      // every earlier tile of the slice has read its sources (only those can read rows
      // [i0, i0 + n); none of them waits before publishing)
      const long long first = (long long)cur.slice * tiles_per_slice;
      for (long long u = first + threadIdx.x; u < cur.tile; u += blockDim.x)
        if (!wait_at_least(tile_flags + u, 1, dev_status)) s_ok = 0;
      __syncthreads();
      if (s_ok) {
        const uint4* bk = bufs + b * per_buf;
        const uint4* bv = bk + kCompactRows * chunks;
        for (int e = threadIdx.x; e < cur.n * chunks; e += blockDim.x) {
          const int i = e / chunks, ch = e - i * chunks;
          if (s_src[b][i] != cur.i0 + i) {
            const long long r = s_drow[b][i];
            K[r * chunks + ch] = bk[e];
            V[r * chunks + ch] = bv[e];
          }
        }
        if (threadIdx.x < cur.n && s_src[b][threadIdx.x] != cur.i0 + (int)threadIdx.x)
          c.pos[s_drow[b][threadIdx.x]] = s_pos[b][threadIdx.x];
      }
    }
    __syncthreads();
    b ^= 1;
  }
  cp_async_wait_all();
}


// Caches with many slices: one warp per slice, its destination rows in increasing order,
// with no flags and no shared memory. The warp takes 32 destinations at a time (their
// kept units read once, the next 32's read meanwhile) and moves their K and V rows through
// registers in batches of 2 KB per tensor, the next batch's loads in flight while this
// one is written. Nothing else needs ordering: a batch reads rows at or after its own
// destinations, which lie after every earlier batch's destinations, so a write never
// destroys a row that a later read of the slice still needs. CH = 16-byte pieces per row.
__device__ __forceinline__ int src_row_of(const int32_t* kp, int i, int bs) {
  return bs == 1 ? kp[i] : kp[i / bs] * bs + i % bs;
}

template <int CH>
__device__ __forceinline__ void slice_batch_load(const uint4* K, const uint4* V, long long srow,
                                                 long long drow, int b, int lane, uint4* k,
                                                 uint4* v, long long* d) {
  constexpr int RPL = 32 / CH;                     // rows per warp-wide 16-byte load
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int rr = b * 4 * RPL + q * RPL + lane / CH;   // this lane's row of the group
    const long long sr = __shfl_sync(0xffffffffu, srow, rr);
    d[q] = __shfl_sync(0xffffffffu, drow, rr);
    if (d[q] >= 0) {
      k[q] = K[sr * CH + lane % CH];
      v[q] = V[sr * CH + lane % CH];
    }
  }
}

template <int CH>
__device__ __forceinline__ void slice_batch_store(uint4* K, uint4* V, int lane, const uint4* k,
                                                  const uint4* v, const long long* d) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (d[q] >= 0) {
      K[d[q] * CH + lane % CH] = k[q];
      V[d[q] * CH + lane % CH] = v[q];
    }
  }
}

template <int CH>
__global__ void __launch_bounds__(kCompactThreads)
compact_slices_kernel(nx_cache c, const int32_t* __restrict__ keep,
                      const int32_t* __restrict__ newlen, long long slices, int bs) {
  constexpr int NB = 32 / (4 * (32 / CH));   // batches per group of 32 destination rows
  grid_dep_wait();                 // kept slots and new lengths come from the kernels before
  const int lane = threadIdx.x & 31;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  uint4* K = reinterpret_cast<uint4*>(c.k);
  uint4* V = reinterpret_cast<uint4*>(c.v);
  for (long long sl = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; sl < slices;
       sl += nwarps) {
    const int nl = newlen[sl];
    if (nl < 0) continue;
    int l, s, h;
    slice_coords(c, (int)sl, l, s, h);
    const int32_t* kp = keep + sl * (long long)c.capacity;
    int srcn = lane < nl ? src_row_of(kp, lane, bs) : 0;
    for (int g0 = 0; g0 < nl; g0 += 32) {
      const int i = g0 + lane;
      const int src = srcn;
      srcn = i + 32 < nl ? src_row_of(kp, i + 32, bs) : 0;   // the next group's sources
      const bool mv = i < nl && src != i;
      const long long srow = mv ? row_of(c, l, s, h, src) : -1;
      const long long drow = mv ? row_of(c, l, s, h, i) : -1;
      const int pv = mv ? c.pos[srow] : 0;
      if (__ballot_sync(0xffffffffu, mv) == 0) continue;   // nothing of this group moves
      uint4 ka[4], va[4], kb[4], vb[4];
      long long da[4], db[4];
      slice_batch_load<CH>(K, V, srow, drow, 0, lane, ka, va, da);
#pragma unroll
      for (int b = 0; b < NB; b += 2) {
        if (b + 1 < NB) slice_batch_load<CH>(K, V, srow, drow, b + 1, lane, kb, vb, db);
        slice_batch_store<CH>(K, V, lane, ka, va, da);
        if (b + 2 < NB) slice_batch_load<CH>(K, V, srow, drow, b + 2, lane, ka, va, da);
        if (b + 1 < NB) slice_batch_store<CH>(K, V, lane, kb, vb, db);
      }
      if (mv) c.pos[drow] = pv;
    }
    if (lane == 0) c.lens[sl] = nl;
  }
}

std::atomic<int> g_compact_kernel{0};   // 0: automatic, 1: tiles, 2: one warp per slice

template <int CH>
cudaError_t launch_slices(const nx_cache& c, const int32_t* keep, const int32_t* newlen,
                          long long slices, int bs, int sms, cudaStream_t st) {
  int per_sm = 0;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_slices_kernel<CH>,
                                                kCompactThreads, 0);
  constexpr int kWarps = kCompactThreads / 32;
  // as many warps as fit, but the same number of slices for each: with k slices per warp
  // at most, ceil(slices / k) warps (a warp with one slice more than the others would set
  // the kernel's time alone)
  const long long fit = (long long)sms * (per_sm > 0 ? per_sm : 1) * kWarps;
  const long long k = (slices + fit - 1) / fit;
  const long long warps = (slices + k - 1) / k;
  long long grid = (warps + kWarps - 1) / kWarps;
  if (grid < 1) grid = 1;
  return launch_after(compact_slices_kernel<CH>, dim3((unsigned)grid), dim3(kCompactThreads),
                      0, st, c, keep, newlen, slices, bs);
}

}  // namespace

cudaError_t launch_newlen(const nx_cache& c, const nx_params& p, int32_t* newlen,
                          int32_t* dev_status, cudaStream_t st, int* launches) {
  const long long slices = (long long)c.layers * c.seqs * c.kv_heads;
  newlen_kernel<<<(unsigned)((slices + 255) / 256), 256, 0, st>>>(c, p, newlen, dev_status, slices);
  note_launch(st, launches, "newlen");
  return cudaGetLastError();
}

cudaError_t launch_compact(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                           const int32_t* keep, const int32_t* newlen, int32_t* dev_status,
                           cudaStream_t st, int* launches, long long skip_signal_tile) {
  const int row_bytes = c.head_dim * (c.dtype == NX_DTYPE_BF16 ? 2 : 4);
  const size_t smem = 2 * 2 * (size_t)kCompactRows * row_bytes;   // two buffers of K + V
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // Many slices (at least eight per SM): one warp per slice, no cross-block ordering.
  // Otherwise (and for the failure-detection hook) the tile kernel, which spreads a
  // slice over many blocks.
  const int which = g_compact_kernel.load(std::memory_order_relaxed);
  const int ch = row_bytes / 16;
  const bool fits = row_bytes % 16 == 0 && (ch == 8 || ch == 16 || ch == 32);
  if (skip_signal_tile < 0 && fits &&
      (which == 2 || (which == 0 && L.slices >= 8LL * (sms > 0 ? sms : 1)))) {
    const int32_t* nlp = newlen;
    const cudaError_t e =
        ch == 8 ? launch_slices<8>(c, keep, nlp, L.slices, p.block_size, sms, st)
        : ch == 16 ? launch_slices<16>(c, keep, nlp, L.slices, p.block_size, sms, st)
                   : launch_slices<32>(c, keep, nlp, L.slices, p.block_size, sms, st);
    if (e != cudaSuccess) return e;
    note_launch(st, launches, "compact_slices");
    return cudaGetLastError();
  }
  // the tile bookkeeping lives in static shared memory: the opt-in is needed as soon as
  // static + dynamic bytes pass the 48 KB default
  static const size_t static_bytes = [] {
    cudaFuncAttributes fa{};
    return cudaFuncGetAttributes(&fa, compact_kernel) == cudaSuccess ? fa.sharedSizeBytes
                                                                     : (size_t)4096;
  }();
  if (smem + static_bytes > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        compact_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_kernel, kCompactThreads, smem);
  const long long total = L.slices * L.tiles_per_slice;
  long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  const cudaError_t e = launch_after(
      compact_kernel, dim3((unsigned)grid), dim3(kCompactThreads), smem, st, c, keep, newlen,
      reinterpret_cast<int*>(ws + L.tile_flags), reinterpret_cast<unsigned long long*>(ws + L.work),
      (int)L.tiles_per_slice, total, dev_status, skip_signal_tile, p.block_size);
  if (e != cudaSuccess) return e;
  note_launch(st, launches, "compact");
  return cudaGetLastError();
}

void compact_set_kernel(int which) { g_compact_kernel.store(which == 1 || which == 2 ? which : 0); }

}  // namespace nx
