// nx_noalloc.cu -- kv_compact_noalloc: the in-place compaction for callers that cannot
// allocate device memory themselves (no workspace argument).
//
// The compaction's scratch (a tile-claim counter, the new length of every slice and one
// "read done" flag per tile) lives in the file-scope array below, which every GPU that
// loads the library holds until the process exits. Host code cannot pass the array's
// name to a kernel (on the host it is only a stand-in for the device symbol), so each
// call outside a stream capture looks up the array's device address with
// cudaGetSymbolAddress for the current device (the lookup allocates nothing) and
// remembers it; a call inside a capture uses the remembered address. Looking it up
// again on every uncaptured call keeps the address right after cudaDeviceReset, which
// can load the module's symbols at a new address.
#include <mutex>

#include "nx_internal.cuh"

namespace nx {
namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;   // 4 MiB per device
constexpr int kNoallocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoallocMaxDevices];

cudaError_t noalloc_scratch_of_current_device(cudaStream_t st, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kNoallocMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_ptr[dev] = p;
  }
  if (!g_noalloc_ptr[dev]) return cudaErrorStreamCaptureUnsupported;
  *out = g_noalloc_ptr[dev];
  return cudaSuccess;
}

constexpr size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace nx

extern "C" nx_status kv_compact_noalloc(nx_cache* cache, const int32_t* keep_idx,
                                        const nx_params* params, int32_t* dev_status,
                                        nx_stream_t stream) {
  using namespace nx;
  int launches = 0;
  begin_call();
  // Same argument checks as the workspace-taking entry points (0 = rejected).
  if (nexus_workspace_bytes(cache, params) == 0) {
    if (params && cache && params->block_size > 1 && params->block_size != 32)
      return NX_ERR_UNSUPPORTED;
    return NX_ERR_INVALID_ARG;
  }
  if (!keep_idx || !dev_status) return NX_ERR_INVALID_ARG;

  // Scratch layout inside the static array: claim counter | new lengths | tile flags.
  WsLayout L{};
  L.slices = (long long)cache->layers * cache->seqs * cache->kv_heads;
  L.tiles_per_slice = (int)(((long long)params->budget_max * params->block_size +
                             kCompactRows - 1) / kCompactRows);
  if (L.tiles_per_slice < 1) L.tiles_per_slice = 1;
  L.work = 0;
  L.newlen = 256;
  L.tile_flags = L.newlen + round256((size_t)L.slices * 4);
  const size_t need = L.tile_flags + round256((size_t)L.slices * L.tiles_per_slice * 4);
  if (need > kNoallocScratchBytes) return NX_ERR_WORKSPACE;   // sizes beyond the 4 MiB limit

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  void* scratch = nullptr;
  cudaError_t e = noalloc_scratch_of_current_device(st, &scratch);
  if (e != cudaSuccess) return finish(e, launches);
  char* ws = static_cast<char*>(scratch);
  // The array keeps the previous call's contents: the counter, lengths and flags must
  // start at zero.
  e = cudaMemsetAsync(ws, 0, need, st);
  if (e != cudaSuccess) return finish(e, launches);
  int32_t* newlen = reinterpret_cast<int32_t*>(ws + L.newlen);
  e = launch_newlen(*cache, *params, newlen, dev_status, st, &launches);
  if (e != cudaSuccess) return finish(e, launches);
  e = launch_compact(*cache, *params, L, ws, keep_idx, newlen, dev_status, st, &launches);
  return finish(e, launches);
}
