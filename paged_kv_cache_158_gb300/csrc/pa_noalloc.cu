// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory when they decode.
//
// pa_decode needs a scratch workspace for its per-partition partial results
// and its work counter, and leaves it to the caller to provide one.  Some
// callers have no way to get one at that point: serving processes that
// reserve all of HBM for the KV pool at start-up and keep no allocator
// headroom, runtimes that must not call cudaMalloc / cudaFree on their hot
// path because those calls can synchronise the device, and host code that
// owns no allocator at all (a plain C caller handed device pointers by
// someone else).  This entry point gives them the same decode with the
// scratch taken from a fixed array in the library's own device memory.
//
// The array is a file-scope __device__ variable.  This file's device code is
// a module of its own, and under CUDA's lazy module loading (the default) a
// module is loaded into a device's context the first time it is used, not
// when the library is loaded: the array's PA_DECODE_NOALLOC_SCRATCH_BYTES are
// committed on a device by the first pa_decode_noalloc call there, and stay
// until the process exits.  Host code cannot use the array's name as a
// device address, so that first call also looks the address up with
// cudaGetSymbolAddress (with the device current) and caches it; later calls
// reuse the cached address.  The first call on each device is therefore a
// warm-up: make it before the rest of device memory is handed to the KV pool
// and before any stream capture.
#include <mutex>

#include "pa_internal.h"

static __device__ __align__(256) unsigned char g_pa_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices];

// Device address of this device's scratch array (looked up once per device).
pa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_decode_scratch) != cudaSuccess || p == nullptr) {
      // Typically out of memory while loading the module: clear the sticky
      // last error so it is not reported again by a later, unrelated check.
      cudaGetLastError();
      return PA_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* query, const void* key_cache,
                                       const void* value_cache, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_heads, int head_dim, int block_size,
                                       int num_blocks, float scale, int max_context_len,
                                       pa_stream_t stream) {
  // A shape whose scratch would not fit is refused before anything runs.
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len);
  if (need > (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const pa_status st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  // pa_decode zeroes the work counters at the start of every call; the
  // partial results need no clearing (each is written before it is read).
  return pa_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                   context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                   max_context_len, scratch, (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
