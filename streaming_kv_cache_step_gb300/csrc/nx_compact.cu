// nx_compact.cu -- in-place stable compaction (Nexus Sampling paper, §2.1: inference
// continues with K_S, V_S): row i <- row keep[i] for k, v and pos, i < n = min(T, B).
//
// keep is ascending with keep[i] >= i, so writing row i can only destroy a source that a
// destination i' <= i still needs. Destinations are cut into tiles of kCompactRows rows,
// claimed in increasing order through one global counter. A tile first copies all its
// sources into shared memory, then publishes "read done", then waits (bounded) until the
// earlier tiles of its slice have published, and only then writes. Waits point only to
// lower tiles, which never wait before publishing, so the scheme cannot deadlock. Rows
// with keep[i] == i are neither read nor written.
#include "nx_internal.cuh"

namespace nx {
namespace {

constexpr int kCompactThreads = 256;

__device__ __forceinline__ bool slice_ok(const nx_cache& c, const nx_params& p, int slice,
                                         int32_t* dev_status) {
  int l, s, h;
  slice_coords(c, slice, l, s, h);
  const int T = c.lens[slice];
  const int B = p.budget[s];
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
  newlen[slice] = slice_ok(c, p, (int)slice, dev_status) ? min(c.lens[slice], p.budget[s]) : -1;
}

__global__ void __launch_bounds__(kCompactThreads)
compact_kernel(nx_cache c, const int32_t* __restrict__ keep, const int32_t* __restrict__ newlen,
               int* tile_flags, unsigned long long* work, int tiles_per_slice,
               long long total_tiles, int32_t* dev_status, long long skip_signal_tile) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int row_bytes = c.head_dim * (c.dtype == NX_DTYPE_BF16 ? 2 : 4);
  const int chunks = row_bytes / 16;                    // 16-byte pieces per row
  uint4* sk = reinterpret_cast<uint4*>(smem);
  uint4* sv = sk + kCompactRows * chunks;
  __shared__ int s_src[kCompactRows];
  __shared__ int s_pos[kCompactRows];
  __shared__ long long s_tile;
  __shared__ int s_any, s_ok;
  uint4* K = reinterpret_cast<uint4*>(c.k);
  uint4* V = reinterpret_cast<uint4*>(c.v);

  for (;;) {
    if (threadIdx.x == 0) s_tile = (long long)atomicAdd(work, 1ULL);
    __syncthreads();
    const long long tile = s_tile;
    if (tile >= total_tiles) return;
    const int slice = (int)(tile / tiles_per_slice);
    const int t = (int)(tile % tiles_per_slice);
    const int nl = newlen[slice];
    int* flag = tile_flags + tile;
    const int i0 = t * kCompactRows;
    if (nl < 0 || i0 >= nl) {
      if (threadIdx.x == 0) {
        if (t == 0 && nl >= 0) c.lens[slice] = nl;
        st_release(flag, 1);
      }
      __syncthreads();
      continue;
    }
    int l, s, h;
    slice_coords(c, slice, l, s, h);
    const int n = min(kCompactRows, nl - i0);
    const int32_t* kp = keep + (long long)slice * c.capacity;
    if (threadIdx.x == 0) s_any = 0;
    __syncthreads();
    if (threadIdx.x < n) {
      const int src = kp[i0 + threadIdx.x];
      s_src[threadIdx.x] = src;
      if (src != i0 + threadIdx.x) s_any = 1;
    }
    __syncthreads();
    if (!s_any) {            // identity tile: nothing to move
      if (threadIdx.x == 0) {
        if (t == 0) c.lens[slice] = nl;
        st_release(flag, 1);
      }
      __syncthreads();
      continue;
    }
    // ---- read every moved source row into shared memory ----
    for (int e = threadIdx.x; e < n * chunks; e += blockDim.x) {
      const int i = e / chunks, ch = e % chunks;
      const int src = s_src[i];
      if (src != i0 + i) {
        const long long r = row_of(c, l, s, h, src);
        sk[e] = K[r * chunks + ch];
        sv[e] = V[r * chunks + ch];
      }
    }
    if (threadIdx.x < n) {
      const int src = s_src[threadIdx.x];
      if (src != i0 + (int)threadIdx.x) s_pos[threadIdx.x] = c.pos[row_of(c, l, s, h, src)];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      if (tile != skip_signal_tile) st_release(flag, 1);   // test hook: -1 in normal calls
      s_ok = 1;
    }
    __syncthreads();
    // ---- wait until every earlier tile of the slice has read its sources: only those
    // can read rows [i0, i0 + n), and none of them waits before publishing ----
    const long long first = (long long)slice * tiles_per_slice;
    for (long long u = first + threadIdx.x; u < tile; u += blockDim.x)
      if (!wait_at_least(tile_flags + u, 1, dev_status)) s_ok = 0;
    __syncthreads();
    if (s_ok) {
      for (int e = threadIdx.x; e < n * chunks; e += blockDim.x) {
        const int i = e / chunks, ch = e % chunks;
        if (s_src[i] != i0 + i) {
          const long long r = row_of(c, l, s, h, i0 + i);
          K[r * chunks + ch] = sk[e];
          V[r * chunks + ch] = sv[e];
        }
      }
      if (threadIdx.x < n && s_src[threadIdx.x] != i0 + (int)threadIdx.x)
        c.pos[row_of(c, l, s, h, i0 + threadIdx.x)] = s_pos[threadIdx.x];
      if (threadIdx.x == 0 && t == 0) c.lens[slice] = nl;
    }
    __syncthreads();
  }
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
  (void)p;
  const int row_bytes = c.head_dim * (c.dtype == NX_DTYPE_BF16 ? 2 : 4);
  const size_t smem = 2 * (size_t)kCompactRows * row_bytes;
  int dev = 0, sms = 0, per_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compact_kernel, kCompactThreads, smem);
  const long long total = L.slices * L.tiles_per_slice;
  long long grid = (long long)sms * (per_sm > 0 ? per_sm : 1);
  if (grid > total) grid = total;
  if (grid < 1) grid = 1;
  compact_kernel<<<(unsigned)grid, kCompactThreads, smem, st>>>(
      c, keep, newlen, reinterpret_cast<int*>(ws + L.tile_flags),
      reinterpret_cast<unsigned long long*>(ws + L.work), L.tiles_per_slice, total, dev_status, skip_signal_tile);
  note_launch(st, launches, "compact");
  return cudaGetLastError();
}

}  // namespace nx
