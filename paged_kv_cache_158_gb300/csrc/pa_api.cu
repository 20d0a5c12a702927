// C ABI of libpa.so: argument checks, launch planning and the device error
// word.  Every computation runs in the kernels of the other translation
// units; this file only validates, sizes and launches.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <vector>

#include "pa_internal.h"

namespace pa {
#define PA_DECLARE_DECODE(sfx)                                                           \
  cudaError_t launch_decode_partition_##sfx(const DecodeParams&, int, int, size_t,      \
                                            cudaStream_t);                              \
  int decode_ctas_per_sm_##sfx(int, size_t, bool);                                      \
  size_t decode_fixed_smem_##sfx(int);                                                  \
  cudaError_t decode_prepare_##sfx();
PA_DECLARE_DECODE(d64)
PA_DECLARE_DECODE(d128)
PA_DECLARE_DECODE(f8_d64)
PA_DECLARE_DECODE(f8_d128)
#undef PA_DECLARE_DECODE
cudaError_t launch_decode_reduce_d64(const DecodeParams&, int, int, cudaStream_t);
cudaError_t launch_decode_reduce_d128(const DecodeParams&, int, int, cudaStream_t);

cudaError_t launch_decode_partition(const DecodeParams& p, bool fp8, int head_dim, int block_size,
                                    int grid, size_t smem, cudaStream_t st) {
  if (fp8)
    return head_dim == 64 ? launch_decode_partition_f8_d64(p, block_size, grid, smem, st)
                          : launch_decode_partition_f8_d128(p, block_size, grid, smem, st);
  return head_dim == 64 ? launch_decode_partition_d64(p, block_size, grid, smem, st)
                        : launch_decode_partition_d128(p, block_size, grid, smem, st);
}

cudaError_t launch_decode_reduce(const DecodeParams& p, int head_dim, int block_size,
                                 int total_seqs, cudaStream_t st) {
  return head_dim == 64 ? launch_decode_reduce_d64(p, block_size, total_seqs, st)
                        : launch_decode_reduce_d128(p, block_size, total_seqs, st);
}

size_t decode_smem_bytes(bool fp8, int head_dim, int block_size, int part_tokens,
                         int seqs_in_launch) {
  const size_t fixed =
      fp8 ? (head_dim == 64 ? decode_fixed_smem_f8_d64(block_size)
                            : decode_fixed_smem_f8_d128(block_size))
          : (head_dim == 64 ? decode_fixed_smem_d64(block_size) : decode_fixed_smem_d128(block_size));
  const size_t bt = 2 * (size_t)(part_tokens / block_size + 1) * 4;
  const size_t seq = (2 * (size_t)seqs_in_launch + 1) * 4 + (size_t)seqs_in_launch;  // + clip flags
  return (fixed + bt + seq + 15) & ~size_t(15);
}

int decode_ctas_per_sm(bool fp8, int head_dim, int block_size, size_t smem, bool append) {
  if (fp8)
    return head_dim == 64 ? decode_ctas_per_sm_f8_d64(block_size, smem, append)
                          : decode_ctas_per_sm_f8_d128(block_size, smem, append);
  return head_dim == 64 ? decode_ctas_per_sm_d64(block_size, smem, append)
                        : decode_ctas_per_sm_d128(block_size, smem, append);
}

cudaError_t decode_prepare_device(int) {
  cudaError_t e;
  if ((e = decode_prepare_d64()) != cudaSuccess) return e;
  if ((e = decode_prepare_d128()) != cudaSuccess) return e;
  if ((e = decode_prepare_f8_d64()) != cudaSuccess) return e;
  return decode_prepare_f8_d128();
}

}  // namespace pa

// The library's device error word: one per device (a static device variable
// is instantiated in every context that loads the module).
static __device__ unsigned int g_pa_error_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];
bool g_prepared[kMaxDevices];
std::atomic<int> g_part_override{0};

struct DeviceState {
  unsigned int* err;
  int sms;
};

pa_status device_state(DeviceState* out, bool prepare_decode) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_error_word) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    g_sms[dev] = sms;
    g_err_ptr[dev] = static_cast<unsigned int*>(p);
  }
  if (prepare_decode && !g_prepared[dev]) {
    if (pa::decode_prepare_device(dev) != cudaSuccess) return PA_ERR_CUDA;
    g_prepared[dev] = true;
  }
  out->err = g_err_ptr[dev];
  out->sms = g_sms[dev];
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }
bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7) == 0; }
bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool block_size_ok(int b) { return b == 4 || b == 8 || b == 16 || b == 32; }
// The address under which the device reaches p: device memory as is,
// pinned (page-locked) host memory through its mapping; nullptr when the
// device cannot reach it (pageable host memory, another device's memory).
const void* device_address(const void* p, int dev) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: return at.device == dev ? p : nullptr;
    case cudaMemoryTypeManaged: return p;
    case cudaMemoryTypeHost: return at.devicePointer;
    default: return nullptr;
  }
}

// True when the host can read p directly: pinned (page-locked) host memory.
bool host_readable(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}

// Conflicts of a block mapping the host can read (int64 [num_pairs][2] of
// (src, dst)): a destination that appears twice, or, with dst_also_src, a
// destination that is also another pair's source.  O(P log P).
bool host_mapping_conflicts(const int64_t* m, int num_pairs, bool dst_also_src) {
  std::vector<int64_t> d((size_t)num_pairs);
  for (int i = 0; i < num_pairs; ++i) d[(size_t)i] = m[2 * (size_t)i + 1];
  std::sort(d.begin(), d.end());
  if (std::adjacent_find(d.begin(), d.end()) != d.end()) return true;
  if (dst_also_src) {
    // Destinations are distinct here, so a source found among them is another
    // pair's destination unless it is the pair's own (a copy onto itself).
    for (int i = 0; i < num_pairs; ++i) {
      const int64_t src = m[2 * (size_t)i], dst = m[2 * (size_t)i + 1];
      if (src != dst && std::binary_search(d.begin(), d.end(), src)) return true;
    }
  }
  return false;
}

bool scale_ok(float s) { return s > 0.f && s <= 3.4028234663852886e38f; }  // finite, positive

// Tokens per partition.  Batches with few items per resident CTA (fewer
// than kSmallBatchItems items of 512 tokens, about 8 per CTA on a 152-SM
// GPU at 3 CTAs per SM) end on a tail of their last items, so their contexts
// are cut into 256-token partitions; larger batches balance anyway and keep
// 512, where the per-item barrier and merge cost less.  Measured (GB/s,
// 256 vs 512): 7B-shaped batch 4693 vs 4519, 13B-shaped 6503 vs 6433 (FP8
// 5347 vs 5322); long-context 7095 vs 7110 (FP8 6177 vs 6575),
// shared-prefix 3405 vs 3437.  A pure function of the sizes, so
// pa_decode_workspace_size and the call agree.
constexpr long long kSmallBatchItems = 4096;

int part_tokens_for(int num_seqs, int num_heads, int max_context_len) {
  const int o = g_part_override.load(std::memory_order_relaxed);
  if (o > 0) return (o + 31) / 32 * 32;
  const long long items512 =
      (long long)num_seqs * num_heads * ((max_context_len + 511) / 512);
  return items512 < kSmallBatchItems ? 256 : 512;
}

struct WsLayout {
  int part_tokens;
  int max_parts;
  int launches;
  size_t counters_off, zero_bytes, ml_off, o_off, total;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(int S, int H, int D, int max_context_len) {
  WsLayout w{};
  w.part_tokens = part_tokens_for(S, H, max_context_len);
  w.max_parts = max_context_len > 0 ? (max_context_len + w.part_tokens - 1) / w.part_tokens : 1;
  w.launches = (S + pa::kMaxSeqsPerLaunch - 1) / pa::kMaxSeqsPerLaunch;
  if (w.launches < 1) w.launches = 1;
  // The work counters are zeroed by every call; the partials after them are
  // always written before they are read.
  w.counters_off = 0;
  size_t off = (size_t)w.launches * 4;
  w.zero_bytes = off;
  off = round256(off);
  w.ml_off = off;
  w.o_off = off;
  if (w.max_parts > 1) {
    const size_t slots = (size_t)S * H * w.max_parts;
    w.o_off = round256(off + slots * 2 * 4);
    off = round256(w.o_off + slots * (size_t)D * 4);
  }
  w.total = off;
  return w;
}

// The decode call for both cache element types (fp8: E4M3 caches with
// per-tensor scales; k_scale and v_scale are 1 for fp16).
pa_status decode_impl(bool fp8, void* out, const void* query, const void* key_cache,
                      const void* value_cache, const int32_t* block_tables,
                      int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                      int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                      float k_scale, float v_scale, int max_context_len, void* workspace,
                      size_t workspace_bytes, unsigned int flags, pa_stream_t stream,
                      const void* key_new = nullptr, const void* value_new = nullptr) {
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (flags & ~(PA_DECODE_ZEROED_WORKSPACE | PA_DECODE_INPUTS_READY)) return PA_ERR_INVALID_ARG;
  if ((key_new == nullptr) != (value_new == nullptr)) return PA_ERR_INVALID_ARG;
  if (key_new && (!aligned16(key_new) || !aligned16(value_new))) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
      max_context_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens || !workspace)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned16(workspace) || !aligned4(block_tables) || !aligned4(context_lens))
    return PA_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(num_seqs, num_heads, head_dim, max_context_len);
  if (workspace_bytes < w.total) return PA_ERR_INVALID_ARG;
  if ((long long)num_seqs * num_heads * w.max_parts >= (1LL << 31)) return PA_ERR_UNSUPPORTED;

  DeviceState ds;
  pa_status st = device_state(&ds, true);
  if (st != PA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  pa::DecodeParams p{};
  p.out = out;
  p.query = query;
  p.key_cache = key_cache;
  p.value_cache = value_cache;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.ws_ml = reinterpret_cast<float*>(ws + w.ml_off);
  p.ws_o = reinterpret_cast<float*>(ws + w.o_off);
  p.err = ds.err;
  p.num_heads = num_heads;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = num_blocks;
  p.max_context_len = max_context_len;
  p.part_tokens = w.part_tokens;
  p.max_parts = w.max_parts;
  p.scale_log2 = (float)((double)scale * (double)k_scale * 1.4426950408889634073599246810019);
  p.v_scale = v_scale;
  p.key_new = key_new;
  p.value_new = value_new;
  p.k_scale = k_scale;

  // The kernels leave the counters zero; a caller that keeps them so skips the
  // zeroing kernel.
  unsigned int* counters = reinterpret_cast<unsigned int*>(ws + w.counters_off);
  if (!(flags & PA_DECODE_ZEROED_WORKSPACE) &&
      pa::launch_zero_words(counters, (int)(w.zero_bytes / 4), cs) != cudaSuccess)
    return PA_ERR_CUDA;
  for (int b = 0; b < w.launches; ++b) {
    p.seq_begin = b * pa::kMaxSeqsPerLaunch;
    p.num_seqs = num_seqs - p.seq_begin < pa::kMaxSeqsPerLaunch ? num_seqs - p.seq_begin
                                                                 : pa::kMaxSeqsPerLaunch;
    p.counter = counters + b;
    // The zeroing kernel, or the previous launch, waited before it triggered
    // this one; otherwise only the caller's word says the inputs are complete.
    p.inputs_ready = b > 0 || !(flags & PA_DECODE_ZEROED_WORKSPACE) ||
                     (flags & PA_DECODE_INPUTS_READY) != 0;
    const size_t smem = pa::decode_smem_bytes(fp8, head_dim, block_size, w.part_tokens, p.num_seqs);
    const int per_sm = pa::decode_ctas_per_sm(fp8, head_dim, block_size, smem, key_new != nullptr);
    long long grid = (long long)per_sm * ds.sms;
    const long long items_ub = (long long)p.num_seqs * num_heads * w.max_parts;
    if (grid > items_ub) grid = items_ub;
    if (pa::launch_decode_partition(p, fp8, head_dim, block_size, (int)grid, smem, cs) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  if (w.max_parts > 1) {
    p.seq_begin = 0;
    p.num_seqs = num_seqs;
    if (pa::launch_decode_reduce(p, head_dim, block_size, num_seqs, cs) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status copy_blocks_impl(int elem_bytes, void* const* key_caches, void* const* value_caches,
                           int num_layers, const int64_t* block_mapping, int num_pairs,
                           int num_heads, int head_dim, int block_size, int num_blocks,
                           pa_stream_t stream) {
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_layers < 0 || num_pairs < 0 || num_heads <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (!key_caches || !value_caches || !block_mapping || !aligned8(block_mapping))
    return PA_ERR_INVALID_ARG;
  for (int l = 0; l < num_layers; ++l) {
    if (!key_caches[l] || !value_caches[l] || !aligned16(key_caches[l]) ||
        !aligned16(value_caches[l]))
      return PA_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  const void* map_dev = device_address(block_mapping, dev);
  if (!map_dev) return PA_ERR_INVALID_ARG;
  const bool on_host = host_readable(block_mapping);
  if (on_host && host_mapping_conflicts(block_mapping, num_pairs, true)) return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_copy_blocks(key_caches, value_caches, num_layers,
                                static_cast<const int64_t*>(map_dev), num_pairs,
                                num_heads, head_dim, block_size, elem_bytes, num_blocks, !on_host,
                                ds.err,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
  }
  return "PA_ERR_UNKNOWN";
}

int pa_decode_partition_tokens(int num_seqs, int num_heads, int max_context_len) {
  if (num_seqs < 0 || num_heads <= 0 || max_context_len < 0) return 0;
  return part_tokens_for(num_seqs, num_heads, max_context_len);
}

void pa_decode_set_partition_tokens(int tokens) {
  g_part_override.store(tokens > 0 ? tokens : 0, std::memory_order_relaxed);
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len) {
  if (num_seqs < 0 || num_heads <= 0 || !head_dim_ok(head_dim) || max_context_len < 0) return 0;
  return ws_layout(num_seqs, num_heads, head_dim, max_context_len).total;
}

pa_status pa_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                    int block_size, int num_blocks, float scale, int max_context_len,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream) {
  return decode_impl(false, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     1.f, 1.f, max_context_len, workspace, workspace_bytes, 0u, stream);
}

pa_status pa_decode_ex(void* out, const void* query, const void* key_cache,
                       const void* value_cache, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                       int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                       int max_context_len, void* workspace, size_t workspace_bytes,
                       unsigned int flags, pa_stream_t stream) {
  return decode_impl(false, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     1.f, 1.f, max_context_len, workspace, workspace_bytes, flags, stream);
}

pa_status pa_decode_fp8(void* out, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                        int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                        float k_scale, float v_scale, int max_context_len, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream) {
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID_ARG;
  return decode_impl(true, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     k_scale, v_scale, max_context_len, workspace, workspace_bytes, 0u, stream);
}

pa_status pa_decode_fp8_ex(void* out, const void* query, const void* key_cache,
                           const void* value_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                           int num_heads, int head_dim, int block_size, int num_blocks,
                           float scale, float k_scale, float v_scale, int max_context_len,
                           void* workspace, size_t workspace_bytes, unsigned int flags,
                           pa_stream_t stream) {
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID_ARG;
  return decode_impl(true, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     k_scale, v_scale, max_context_len, workspace, workspace_bytes, flags, stream);
}

pa_status pa_decode_append(void* out, const void* query, const void* key_new,
                           const void* value_new, void* key_cache, void* value_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                           int block_size, int num_blocks, float scale, int max_context_len,
                           void* workspace, size_t workspace_bytes, unsigned int flags,
                           pa_stream_t stream) {
  if (!key_new || !value_new) return PA_ERR_INVALID_ARG;
  return decode_impl(false, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     1.f, 1.f, max_context_len, workspace, workspace_bytes, flags, stream,
                     key_new, value_new);
}

pa_status pa_decode_append_fp8(void* out, const void* query, const void* key_new,
                               const void* value_new, void* key_cache, void* value_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_heads,
                               int head_dim, int block_size, int num_blocks, float scale,
                               float k_scale, float v_scale, int max_context_len,
                               void* workspace, size_t workspace_bytes, unsigned int flags,
                               pa_stream_t stream) {
  if (!key_new || !value_new) return PA_ERR_INVALID_ARG;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID_ARG;
  return decode_impl(true, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, head_dim, block_size, num_blocks, scale,
                     k_scale, v_scale, max_context_len, workspace, workspace_bytes, flags, stream,
                     key_new, value_new);
}

pa_status pa_reshape_and_cache(const void* key, const void* value, void* key_cache,
                               void* value_cache, const int64_t* slot_mapping, int num_tokens,
                               int num_heads, int head_dim, int block_size, int num_blocks,
                               pa_stream_t stream) {
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned8(slot_mapping))
    return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, num_tokens,
                                      num_heads, head_dim, block_size, num_blocks, ds.err,
                                      reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                         const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim,
                         int block_size, int num_blocks, pa_stream_t stream) {
  return copy_blocks_impl(2, key_caches, value_caches, num_layers, block_mapping, num_pairs,
                          num_heads, head_dim, block_size, num_blocks, stream);
}

pa_status pa_copy_blocks_fp8(void* const* key_caches, void* const* value_caches, int num_layers,
                             const int64_t* block_mapping, int num_pairs, int num_heads,
                             int head_dim, int block_size, int num_blocks, pa_stream_t stream) {
  return copy_blocks_impl(1, key_caches, value_caches, num_layers, block_mapping, num_pairs,
                          num_heads, head_dim, block_size, num_blocks, stream);
}

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int64_t* slot_mapping, int num_tokens,
                                   int num_heads, int head_dim, int block_size, int num_blocks,
                                   float k_scale, float v_scale, pa_stream_t stream) {
  if (!head_dim_ok(head_dim) || !block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned8(slot_mapping))
    return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping,
                                          num_tokens, num_heads, head_dim, block_size, num_blocks,
                                          k_scale, v_scale, ds.err,
                                          reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_convert_cache_fp8(const void* src, void* dst, size_t num_elems, float scale,
                               pa_stream_t stream) {
  if (!scale_ok(scale) || (num_elems & 15) != 0) return PA_ERR_INVALID_ARG;
  if (num_elems == 0) return PA_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_convert_cache_fp8(src, dst, (long long)num_elems, scale,
                                      reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_swap_blocks(void* const* dst_caches, const void* const* src_caches, int num_caches,
                         const int64_t* block_mapping, int num_pairs, size_t block_bytes,
                         int64_t src_num_blocks, int64_t dst_num_blocks, pa_stream_t stream) {
  if (num_caches < 0 || num_pairs < 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 ||
      block_bytes == 0 || (block_bytes & 15) != 0)
    return PA_ERR_INVALID_ARG;
  if (num_caches == 0 || num_pairs == 0) return PA_OK;
  if (!dst_caches || !src_caches || !block_mapping || !aligned8(block_mapping))
    return PA_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  const void* map_dev = device_address(block_mapping, dev);
  if (!map_dev) return PA_ERR_INVALID_ARG;
  const bool on_host = host_readable(block_mapping);
  if (on_host && host_mapping_conflicts(block_mapping, num_pairs, false)) return PA_ERR_INVALID_ARG;
  std::vector<void*> dst(num_caches);
  std::vector<const void*> src(num_caches);
  for (int c = 0; c < num_caches; ++c) {
    if (!dst_caches[c] || !src_caches[c] || !aligned16(dst_caches[c]) || !aligned16(src_caches[c]))
      return PA_ERR_INVALID_ARG;
    dst[c] = const_cast<void*>(device_address(dst_caches[c], dev));
    src[c] = device_address(src_caches[c], dev);
    if (!dst[c] || !src[c] || !aligned16(dst[c]) || !aligned16(src[c])) return PA_ERR_INVALID_ARG;
  }
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_swap_blocks(dst.data(), src.data(), num_caches,
                                static_cast<const int64_t*>(map_dev), num_pairs,
                                (long long)block_bytes, (long long)src_num_blocks,
                                (long long)dst_num_blocks, !on_host, ds.err,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

// Shared by pa_prefill and pa_prefill_fp8 (the latter with E4M3 caches and
// their scales).
static pa_status prefill_impl(bool fp8, void* out, const void* query, const void* key_cache,
                              const void* value_cache, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens,
                              const int32_t* query_start, int num_seqs, int num_query_tokens,
                              int num_heads, int head_dim, int block_size, int num_blocks,
                              float scale, float k_scale, float v_scale, int max_query_len,
                              int num_decode_rows, unsigned int flags, pa_stream_t stream) {
  if (!head_dim_ok(head_dim) || !(block_size == 8 || block_size == 16 || block_size == 32))
    return PA_ERR_UNSUPPORTED;
  if (flags & ~PA_PREFILL_INPUTS_READY) return PA_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_query_tokens < 0 || num_heads <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || max_query_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_decode_rows < -1 || num_decode_rows > num_seqs || num_decode_rows > num_query_tokens)
    return PA_ERR_INVALID_ARG;
  if (fp8 && (!scale_ok(k_scale) || !scale_ok(v_scale))) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0 || num_query_tokens == 0 || max_query_len == 0) return PA_OK;
  if (!pa::prefill_rows_fit(num_blocks, num_heads, block_size)) return PA_ERR_UNSUPPORTED;
  if ((long long)num_seqs * ((max_query_len + 127) / 128) * num_heads >= (1LL << 31))
    return PA_ERR_UNSUPPORTED;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !context_lens ||
      !query_start)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache) ||
      !aligned4(block_tables) || !aligned4(context_lens) || !aligned4(query_start))
    return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  pa::PrefillArgs g{};
  g.out = out;
  g.query = query;
  g.key_cache = key_cache;
  g.value_cache = value_cache;
  g.block_tables = block_tables;
  g.context_lens = context_lens;
  g.query_start = query_start;
  g.err = ds.err;
  g.num_seqs = num_seqs;
  g.num_query_tokens = num_query_tokens;
  g.num_heads = num_heads;
  g.head_dim = head_dim;
  g.block_size = block_size;
  g.num_blocks = num_blocks;
  g.max_blocks = max_blocks_per_seq;
  g.max_query_len = max_query_len;
  g.fp8 = fp8;
  g.v_scale = fp8 ? v_scale : 1.f;
  g.scale_log2 = (float)((double)scale * (fp8 ? (double)k_scale : 1.0) *
                         1.4426950408889634073599246810019);
  g.inputs_ready = (flags & PA_PREFILL_INPUTS_READY) != 0;
  g.num_decode_rows = num_decode_rows;
  return pa::launch_prefill(g, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_prefill(void* out, const void* query, const void* key_cache, const void* value_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start, int num_seqs,
                     int num_query_tokens, int num_heads, int head_dim, int block_size,
                     int num_blocks, float scale, int max_query_len, pa_stream_t stream) {
  return prefill_impl(false, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, query_start, num_seqs, num_query_tokens, num_heads, head_dim,
                      block_size, num_blocks, scale, 1.f, 1.f, max_query_len, -1, 0u, stream);
}

pa_status pa_prefill_ex(void* out, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        const int32_t* query_start, int num_seqs, int num_query_tokens,
                        int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                        int max_query_len, int num_decode_rows, unsigned int flags,
                        pa_stream_t stream) {
  return prefill_impl(false, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, query_start, num_seqs, num_query_tokens, num_heads, head_dim,
                      block_size, num_blocks, scale, 1.f, 1.f, max_query_len, num_decode_rows,
                      flags, stream);
}

pa_status pa_prefill_fp8(void* out, const void* query, const void* key_cache,
                         const void* value_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens,
                         const int32_t* query_start, int num_seqs, int num_query_tokens,
                         int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                         float k_scale, float v_scale, int max_query_len, pa_stream_t stream) {
  return prefill_impl(true, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, query_start, num_seqs, num_query_tokens, num_heads, head_dim,
                      block_size, num_blocks, scale, k_scale, v_scale, max_query_len, -1, 0u,
                      stream);
}

pa_status pa_prefill_fp8_ex(void* out, const void* query, const void* key_cache,
                            const void* value_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens,
                            const int32_t* query_start, int num_seqs, int num_query_tokens,
                            int num_heads, int head_dim, int block_size, int num_blocks,
                            float scale, float k_scale, float v_scale, int max_query_len,
                            int num_decode_rows, unsigned int flags, pa_stream_t stream) {
  return prefill_impl(true, out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, query_start, num_seqs, num_query_tokens, num_heads, head_dim,
                      block_size, num_blocks, scale, k_scale, v_scale, max_query_len,
                      num_decode_rows, flags, stream);
}

pa_status pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                          int max_blocks_per_seq, const int32_t* token_seq,
                          const int32_t* token_pos, int num_tokens, int num_seqs, int block_size,
                          int num_blocks, pa_stream_t stream) {
  if (!block_size_ok(block_size)) return PA_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!slot_mapping || !block_tables || !token_seq || !token_pos || !aligned8(slot_mapping) ||
      !aligned4(block_tables) || !aligned4(token_seq) || !aligned4(token_pos))
    return PA_ERR_INVALID_ARG;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_slot_mapping(slot_mapping, block_tables, max_blocks_per_seq, token_seq,
                                 token_pos, num_tokens, num_seqs, block_size, num_blocks, ds.err,
                                 reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_selftest_wait_timeout(pa_stream_t stream) {
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  return pa::launch_selftest_wait(ds.err, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_check_errors(pa_stream_t stream, uint32_t* error_bits) {
  if (error_bits) *error_bits = 0;
  DeviceState ds;
  pa_status st = device_state(&ds, false);
  if (st != PA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, ds.err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return PA_ERR_CUDA;
  if (word != 0 && cudaMemset(ds.err, 0, sizeof(word)) != cudaSuccess) return PA_ERR_CUDA;
  if (error_bits) *error_bits = word;
  if (word & PA_ERRBIT_TIMEOUT) return PA_ERR_TIMEOUT;
  return word ? PA_ERR_OUT_OF_RANGE : PA_OK;
}

}  // extern "C"
