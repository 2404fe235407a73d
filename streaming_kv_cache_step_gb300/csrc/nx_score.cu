// nx_score.cu -- direct scores and the Nexus walk on CUDA cores (the generic path: any
// W <= 64, H <= 8, head_dim 64/128, fp32 or bf16 caches, contiguous or paged).
//
// Per slice the work is split into chunks of kSimtRows rows (one row per thread):
//   stats pass  logits l[w][j] = Qbar_w . k_j / sqrt(d), per-chunk row maxima, sums of
//               exp(l - max), and the H x H Gram of the walk rows (Nexus Sampling paper,
//               §2.1 Eq. (1), §2.2 Eq. (4) through <P_p, P_q>);
//   emit pass   every block combines its slice's chunk statistics (a log-sum-exp merge),
//               runs the walk recurrence on the Gram (gamma_q = 1 + sum_{p<q} gamma_p
//               <P_q, P_p>, the rank-1 expansion of Eq. (4)), recomputes its rows'
//               logits and writes a (Eq. (3)), c~, w (Eqs. (2), (5)) and/or the
//               selection keys of §2.3.
// K is read twice; the tensor-core path (nx_score_tc.cu) reads it once.
#include <math.h>

#include "nx_internal.cuh"

namespace nx {
namespace {

__device__ __forceinline__ void unpack_bf16x8(const uint4 raw, float* out) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    out[2 * i] = __uint_as_float(w[i] << 16);
    out[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Per-slice validity and new length, plus the group-mean window queries Qbar, a tensor of
// the model's dtype (for bf16 caches the mean rounded once to bf16, as a bf16 model's head
// average is): fp32 rows for the CUDA-core scorer (mode 1), or the tensor-core scorer's
// shared-memory image (mode 2) of the bf16 Qbar as head_dim/64 column blocks of W rows x
// 128 bytes in the 128-byte swizzled K-major layout
// (16-byte chunk c of row n stored at chunk c ^ (n mod 8); 8-row groups 1024 bytes apart).
// Grid: one 256-thread block per slice, or (few slices) up to W 64-thread blocks per
// slice, block y of a slice taking the window rows n = y mod gridDim.y.
__global__ void prep_kernel(nx_cache c, const void* __restrict__ q, nx_params p,
                            void* __restrict__ qout, int32_t* __restrict__ newlen,
                            int32_t* dev_status, int mode, int4* __restrict__ counters,
                            long long counter_vecs) {
  // the step's counters (slice arrivals, compaction claims and flags) start at zero; the
  // kernels that use them run after this one
  {
    const long long n = (long long)gridDim.x * gridDim.y * blockDim.x;
    for (long long i = ((long long)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x +
                       threadIdx.x;
         i < counter_vecs; i += n)
      counters[i] = make_int4(0, 0, 0, 0);
  }
  const int slice = blockIdx.x;
  int l, s, h;
  slice_coords(c, slice, l, s, h);
  const int W = p.window, D = c.head_dim, G = c.group;
  const int ny = gridDim.y;                         // blocks sharing the slice's rows
  if (blockIdx.y == 0) {
    const int T = c.lens[slice];
    __shared__ int bad;
    if (threadIdx.x == 0) {
      bad = 0;
      const int B = budget_of(p, slice, s);
      if (T < 0 || T > c.capacity) {
        atomicOr(dev_status, NX_DEV_BAD_LEN);
        bad = 1;
      } else if (B < p.n_sink + p.n_recent || B > p.budget_max) {
        atomicOr(dev_status, NX_DEV_BAD_BUDGET);
        bad = 1;
      }
    }
    __syncthreads();
    if (!bad && c.page_size > 0) {
      const int npg = (T + c.page_size - 1) / c.page_size;
      for (int i = threadIdx.x; i < npg; i += blockDim.x) {
        const int pg = i < c.max_pages_per_seq
                           ? c.block_table[(long long)s * c.max_pages_per_seq + i] : -1;
        if (pg < 0 || pg >= c.num_pages) {
          atomicOr(dev_status, NX_DEV_BAD_PAGE);
          bad = 1;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0)
      newlen[slice] = bad ? -1 : rows_kept(T, budget_of(p, slice, s), p.block_size);
  }
  if (mode == 0) return;
  // query head h*G + g belongs to KV head h; the window query is their mean, summed in the
  // order g = 0, 1, ..., G - 1
  const long long qslice = (((long long)l * c.seqs + s) * (c.kv_heads * (long long)G) +
                            (long long)h * G) * W * D;
  const float invG = 1.0f / (float)G;
  if (mode == 2) {
    // the bf16 image in the MMA's 128-byte-swizzled K-major layout; 8 features (16 B) per
    // item, which stay contiguous under the 16-byte swizzle
    const int KB = D / 64, region = W * 128, groups = D / 8;
    unsigned char* img = reinterpret_cast<unsigned char*>(qout) + (long long)slice * KB * region;
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(q);
    const int rows = (W - (int)blockIdx.y + ny - 1) / ny;     // this block's window rows
    for (int it = threadIdx.x; it < rows * groups; it += blockDim.x) {
      const int r = it / groups, kk = (it - r * groups) * 8;
      const int n = (int)blockIdx.y + r * ny;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
      for (int g = 0; g < G; ++g) {
        const uint4 raw = *reinterpret_cast<const uint4*>(qb + qslice + (long long)g * W * D +
                                                           (long long)n * D + kk);
        const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] += __low2float(e2[i]);
          v[2 * i + 1] += __high2float(e2[i]);
        }
      }
      uint4 hw;
      __nv_bfloat162* hp = reinterpret_cast<__nv_bfloat162*>(&hw);
#pragma unroll
      for (int i = 0; i < 4; ++i) hp[i] = __floats2bfloat162_rn(v[2 * i] * invG, v[2 * i + 1] * invG);
      const int kb = kk >> 6, byte = (kk & 63) * 2;
      const int off = (n >> 3) * 1024 + (n & 7) * 128 + (((byte >> 4) ^ (n & 7)) << 4);
      *reinterpret_cast<uint4*>(img + kb * region + off) = hw;
    }
    return;
  }
  // group means as fp32 rows for the CUDA-core scorer (bf16 caches: the bf16 mean)
  const int rows = (W - (int)blockIdx.y + ny - 1) / ny;
  for (int it = threadIdx.x; it < rows * D; it += blockDim.x) {
    const int r = it / D, kk = it - r * D;
    const int n = (int)blockIdx.y + r * ny;
    float v = 0.f;
    for (int g = 0; g < G; ++g)
      v += ld_elem(q, c.dtype, qslice + (long long)g * W * D + (long long)n * D + kk);
    const float m = v * invG;
    reinterpret_cast<float*>(qout)[((long long)slice * W + n) * D + kk] =
        c.dtype == NX_DTYPE_BF16 ? __bfloat162float(__float2bfloat16_rn(m)) : m;
  }
}

template <int N>
__device__ __forceinline__ void block_reduce(float (&v)[N], int n, bool is_max, float* red,
                                             float* result) {
  // red: [warps][N] shared scratch; result: [N] shared
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (i < n) {
      float x = v[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, o);
        x = is_max ? fmaxf(x, y) : x + y;
      }
      if (lane == 0) red[warp * N + i] = x;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    float x = red[i];
    for (int w = 1; w < nw; ++w) x = is_max ? fmaxf(x, red[w * N + i]) : x + red[w * N + i];
    result[i] = x;
  }
  __syncthreads();
}

template <int WMAX, int D, bool BF16, bool EMIT>
__global__ void __launch_bounds__(kSimtRows)
score_simt_kernel(nx_cache c, nx_params p, const float* __restrict__ qbar,
                  float* __restrict__ stats, int stride, int max_chunks,
                  const int32_t* __restrict__ newlen, ScoreOut out, int32_t* dev_status) {
  const int slice = blockIdx.x, chunk = blockIdx.y;
  if (newlen[slice] < 0) return;
  const int T = c.lens[slice];
  const int j0 = chunk * kSimtRows;
  if (j0 >= T) return;
  int l, s, h;
  slice_coords(c, slice, l, s, h);
  const int W = p.window, H = p.walk_len;

  __shared__ __align__(16) float sq[WMAX * D];
  __shared__ float red[(kSimtRows / 32) * (WMAX > kMaxPairs ? WMAX : kMaxPairs)];
  __shared__ float smax[WMAX], ssum[WMAX], sgram[kMaxPairs], scoef[WMAX], swalk[kMaxWalk];

  for (int i = threadIdx.x; i < W * D; i += blockDim.x)
    sq[i] = qbar[(long long)slice * W * D + i];
  __syncthreads();

  const int j = j0 + threadIdx.x;
  const bool valid = j < T;
  float lg[WMAX];
#pragma unroll
  for (int w = 0; w < WMAX; ++w) lg[w] = 0.f;
  long long r = -1;
  if (valid) {
    r = row_of(c, l, s, h, j);
    if (BF16) {
      const uint4* kr = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(c.k) + r * D);
#pragma unroll 1
      for (int k8 = 0; k8 < D / 8; ++k8) {
        float kv[8];
        unpack_bf16x8(__ldg(kr + k8), kv);
#pragma unroll
        for (int w = 0; w < WMAX; ++w) {
          if (w < W) {
            const float4 q0 = *reinterpret_cast<const float4*>(&sq[w * D + k8 * 8]);
            const float4 q1 = *reinterpret_cast<const float4*>(&sq[w * D + k8 * 8 + 4]);
            float a = lg[w];
            a = fmaf(q0.x, kv[0], a); a = fmaf(q0.y, kv[1], a);
            a = fmaf(q0.z, kv[2], a); a = fmaf(q0.w, kv[3], a);
            a = fmaf(q1.x, kv[4], a); a = fmaf(q1.y, kv[5], a);
            a = fmaf(q1.z, kv[6], a); a = fmaf(q1.w, kv[7], a);
            lg[w] = a;
          }
        }
      }
    } else {
      const float4* kr = reinterpret_cast<const float4*>(
          reinterpret_cast<const float*>(c.k) + r * D);
#pragma unroll 1
      for (int k4 = 0; k4 < D / 4; ++k4) {
        const float4 kv = __ldg(kr + k4);
#pragma unroll
        for (int w = 0; w < WMAX; ++w) {
          if (w < W) {
            const float4 q0 = *reinterpret_cast<const float4*>(&sq[w * D + k4 * 4]);
            float a = lg[w];
            a = fmaf(q0.x, kv.x, a); a = fmaf(q0.y, kv.y, a);
            a = fmaf(q0.z, kv.z, a); a = fmaf(q0.w, kv.w, a);
            lg[w] = a;
          }
        }
      }
    }
  }
  const float scale = rsqrtf((float)D);
#pragma unroll
  for (int w = 0; w < WMAX; ++w) lg[w] = valid ? lg[w] * scale : -INFINITY;

  float* st = stats + ((long long)slice * max_chunks + chunk) * stride;
  if (!EMIT) {
    // ---- per-chunk statistics: maxima, sums of exp(l - max), Gram of walk rows ----
    block_reduce<WMAX>(lg, W, true, red, smax);
    float e[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w) e[w] = (w < W && valid) ? expf(lg[w] - smax[w]) : 0.f;
    float tmp[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w) tmp[w] = e[w];
    block_reduce<WMAX>(tmp, W, false, red, ssum);
    // walk-row exponentials ew[t] = e[W - H + t]; Gram entries in the fixed pair
    // layout pair_index(u, t), u < t, zero for t >= H.
    float ew[kMaxWalk];
#pragma unroll
    for (int t = 0; t < kMaxWalk; ++t) {
      float x = 0.f;
#pragma unroll
      for (int w = 0; w < WMAX; ++w)
        if (t < H && w == W - H + t) x = e[w];
      ew[t] = x;
    }
    if (p.block_size > 1) {
      // b = 32: the walk takes inner products between block rows (sums over the 32 rows
      // of a block, which are this warp's rows); lane 0 carries the block's terms
      const int lane = threadIdx.x & 31;
#pragma unroll
      for (int t = 0; t < kMaxWalk; ++t) {
        float x = ew[t];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        ew[t] = lane == 0 ? x : 0.f;
      }
    }
    float gc[kMaxPairs];
#pragma unroll
    for (int t = 0; t < kMaxWalk; ++t)
#pragma unroll
      for (int u = 0; u < t; ++u) gc[pair_index(u, t)] = ew[u] * ew[t];
    block_reduce<kMaxPairs>(gc, kMaxPairs, false, red, sgram);
    for (int i = threadIdx.x; i < W; i += blockDim.x) {
      st[i] = smax[i];
      st[W + i] = ssum[i];
    }
    for (int i = threadIdx.x; i < kMaxPairs; i += blockDim.x) st[2 * W + i] = sgram[i];
    return;
  }

  // ---- emit: merge the slice's chunk statistics ----
  const int nch = (T + kSimtRows - 1) / kSimtRows;
  const float* st0 = stats + (long long)slice * max_chunks * stride;
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    float M = -INFINITY;
    for (int ch = 0; ch < nch; ++ch) M = fmaxf(M, st0[(long long)ch * stride + w]);
    float Z = 0.f;
    for (int ch = 0; ch < nch; ++ch)
      Z += st0[(long long)ch * stride + W + w] * expf(st0[(long long)ch * stride + w] - M);
    smax[w] = M;
    ssum[w] = Z;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < kMaxPairs; k += blockDim.x) {
    int u = 0, t = 0;
    pair_of(k, u, t);
    float g = 0.f;
    if (t < H) {
      const int wp = W - H + u, wq = W - H + t;
      for (int ch = 0; ch < nch; ++ch) {
        const float* sc = st0 + (long long)ch * stride;
        g += sc[2 * W + k] * expf(sc[wp] - smax[wp]) * expf(sc[wq] - smax[wq]);
      }
      g /= ssum[wp] * ssum[wq];   // <P_p, P_q> with the final normalisers
    }
    sgram[k] = g;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Eq. (4) in rank-1 form: C_t = sum_{u<=t} gamma_u P_u, so
    // gamma_t = 1 + <P_t, C_{t-1}> = 1 + sum_{u<t} gamma_u <P_t, P_u>.
    float gam[kMaxWalk];
    float gsum = 0.f;
    for (int t = 0; t < H; ++t) {
      float g = 1.f;
      for (int u = 0; u < t; ++u) {
        g += gam[u] * sgram[pair_index(u, t)];
      }
      gam[t] = g;
      gsum += g;
    }
    // ||C||_1 = sum_t gamma_t because every P row sums to one.
    for (int t = 0; t < H; ++t) swalk[t] = gam[t] / (gsum * ssum[W - H + t]);
  }
  for (int w = threadIdx.x; w < W; w += blockDim.x) scoef[w] = 1.0f / ((float)W * ssum[w]);
  __syncthreads();
  if (chunk == 0 && out.row_stats && (out.flags & kEmitStats)) {
    for (int w = threadIdx.x; w < W; w += blockDim.x) {
      out.row_stats[((long long)slice * W + w) * 2] = smax[w];
      out.row_stats[((long long)slice * W + w) * 2 + 1] = ssum[w];
    }
  }
  const int bs = p.block_size;
  if (bs == 1 && !valid) return;
  float a = 0.f, ct = 0.f;
#pragma unroll
  for (int w = 0; w < WMAX; ++w) {
    if (w < W) {
      const float e = valid ? expf(lg[w] - smax[w]) : 0.f;
      a = fmaf(e, scoef[w], a);
      if (w >= W - H) ct = fmaf(e, swalk[w - (W - H)], ct);
    }
  }
  int u = j;                      // the decision unit: this row, or its 32-row block
  if (bs > 1) {
    // Eq. (1) BlockSum: a block's scores are the sums over its rows (this warp's 32
    // rows, blocks being aligned to warps); lane 0 finalizes the block
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      ct += __shfl_xor_sync(0xffffffffu, ct, o);
    }
    if ((threadIdx.x & 31) != 0 || !valid) return;
    u = j / bs;
  }
  const int N = units_of(T, bs);
  const float sj = a + p.lambda * ct;
  const float ramp = (N > 1) ? (float)u / (float)(N - 1) : 0.f;
  const float wj = sj + p.eps_tie * ramp;
  const long long o = (long long)slice * c.capacity + u;
  if (out.flags & kEmitA) out.a[o] = a;
  if (out.flags & kEmitC) out.ctilde[o] = ct;
  if (out.flags & kEmitW) out.w[o] = wj;
  if (out.flags & kEmitKeys) {
    uint32_t key = kForcedKey;
    if (p.n_avg > 1) {
      key = __float_as_uint(wj);   // the averaged keys are drawn by a pass of their own
    } else if (!(u < p.n_sink || u >= N - p.n_recent)) {
      const uint32_t head_id = (uint32_t)((p.layer_id_base + l) * c.kv_heads + h);
      key = candidate_key1(wj, c.pos[r], p, head_id, (uint32_t)(p.seq_id_base + s));
    }
    out.keys[o] = key;
  }
}

template <int WMAX, int D, bool BF16>
cudaError_t launch_simt_t(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                          const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                          int* launches) {
  dim3 grid((unsigned)L.slices, L.max_chunks);
  const float* qbar = reinterpret_cast<const float*>(ws + L.qbar);
  float* stats = reinterpret_cast<float*>(ws + L.stats);
  const int32_t* nl = reinterpret_cast<const int32_t*>(ws + L.newlen);
  score_simt_kernel<WMAX, D, BF16, false><<<grid, kSimtRows, 0, st>>>(
      c, p, qbar, stats, L.stats_stride, L.max_chunks, nl, out, dev_status);
  note_launch(st, launches, "score_stats_simt");
  score_simt_kernel<WMAX, D, BF16, true><<<grid, kSimtRows, 0, st>>>(
      c, p, qbar, stats, L.stats_stride, L.max_chunks, nl, out, dev_status);
  note_launch(st, launches, "score_emit_simt");
  return cudaGetLastError();
}

template <int WMAX>
cudaError_t launch_simt_w(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                          const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                          int* launches) {
  const bool bf = c.dtype == NX_DTYPE_BF16;
  if (c.head_dim == 128)
    return bf ? launch_simt_t<WMAX, 128, true>(c, p, L, ws, out, dev_status, st, launches)
              : launch_simt_t<WMAX, 128, false>(c, p, L, ws, out, dev_status, st, launches);
  return bf ? launch_simt_t<WMAX, 64, true>(c, p, L, ws, out, dev_status, st, launches)
            : launch_simt_t<WMAX, 64, false>(c, p, L, ws, out, dev_status, st, launches);
}

}  // namespace

cudaError_t launch_prep(const nx_cache& c, const void* q, const nx_params& p, const WsLayout& L,
                        char* ws, int32_t* dev_status, cudaStream_t st, int* launches,
                        int mode) {
  // few slices: spread each slice's window rows over several blocks
  const int ny = L.slices >= 1024 ? 1 : (int)min((long long)p.window, (1024 + L.slices - 1) / L.slices);
  dim3 grid((unsigned)L.slices, (unsigned)(mode == 0 ? 1 : ny));
  // counters_bytes is a multiple of 64 and the region 256-byte aligned; a block that takes
  // a few rows of its slice needs fewer threads
  prep_kernel<<<grid, grid.y > 1 ? 64 : 256, 0, st>>>(c, q, p, ws + L.qbar,
                                   reinterpret_cast<int32_t*>(ws + L.newlen), dev_status, mode,
                                   reinterpret_cast<int4*>(ws + L.counters),
                                   (long long)(L.counters_bytes / 16));
  note_launch(st, launches, "prep");
  return cudaGetLastError();
}

cudaError_t launch_score_simt(const nx_cache& c, const nx_params& p, const WsLayout& L, char* ws,
                              const ScoreOut& out, int32_t* dev_status, cudaStream_t st,
                              int* launches) {
  if (p.window <= 16) return launch_simt_w<16>(c, p, L, ws, out, dev_status, st, launches);
  if (p.window <= 32) return launch_simt_w<32>(c, p, L, ws, out, dev_status, st, launches);
  return launch_simt_w<64>(c, p, L, ws, out, dev_status, st, launches);
}

}  // namespace nx
