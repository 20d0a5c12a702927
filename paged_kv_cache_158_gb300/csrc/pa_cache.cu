// Cache write, copy-on-write block copy and slot map for sm_103a.
//
// All three are bit copies or integer index arithmetic over KB- to MB-scale
// data: they are bound by launch latency or by HBM, and move 16-byte
// vectors with fully coalesced accesses.
#include <cuda_fp16.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.cuh"

namespace pa {
namespace {

// ---- cache write ("深入解析LLM推理引擎：从PagedAttention到调度优化" §3.2;
// "vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制" §2.3)
// Thread i moves 16-byte vector i of the [T][H][D] key/value inputs to its
// slot: block slot/B, offset slot%B, same head and dimensions.
template <int D>
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                             const int64_t* __restrict__ slot_mapping, int num_tokens,
                             int num_heads, int log2_block, long long num_slots,
                             unsigned int* err) {
  constexpr int V = D / 8;  // 16-byte vectors per head row
  pdl_wait();
  pdl_launch_dependents();
  const long long per_token = (long long)num_heads * V;
  const long long total = (long long)num_tokens * per_token;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long t = i / per_token;
    const int rem = (int)(i - t * per_token);
    const long long slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (rem == 0) atomicOr(err, PA_ERRBIT_SLOT);
      continue;
    }
    const int h = rem / V;
    const int v = rem - h * V;
    const long long blk = slot >> log2_block;
    const long long off = slot & ((1 << log2_block) - 1);
    const long long dst = ((blk * num_heads + h) << log2_block | off) * V + v;
    key_cache[dst] = key[i];
    value_cache[dst] = value[i];
  }
}

// ---- cache write into an FP8 (E4M3) cache
// ("vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §3.3 names FP8 KV
// caches; format and scaling as stated in the public header).  Thread i makes
// 16-byte output vector i (16 codes) of the [T][H][D] inputs: it reads the
// 16 fp16 values (32 bytes), divides each by the tensor's scale in IEEE
// binary32 (round to nearest) and rounds the quotient to the nearest E4M3
// code, saturating to +-448 (quantize16, shared with the decode that writes
// its new token itself).

template <int D>
__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                 uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                 const int64_t* __restrict__ slot_mapping, int num_tokens,
                                 int num_heads, int log2_block, long long num_slots,
                                 float k_scale, float v_scale, unsigned int* err) {
  constexpr int V = D / 16;  // 16-byte code vectors per head row
  pdl_wait();
  pdl_launch_dependents();
  const long long per_token = (long long)num_heads * V;
  const long long total = (long long)num_tokens * per_token;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const long long t = i / per_token;
    const int rem = (int)(i - t * per_token);
    const long long slot = slot_mapping[t];
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (rem == 0) atomicOr(err, PA_ERRBIT_SLOT);
      continue;
    }
    const int h = rem / V;
    const int v = rem - h * V;
    const long long blk = slot >> log2_block;
    const long long off = slot & ((1 << log2_block) - 1);
    const long long dst = ((blk * num_heads + h) << log2_block | off) * V + v;
    key_cache[dst] = quantize16(key[2 * i], key[2 * i + 1], k_scale);
    value_cache[dst] = quantize16(value[2 * i], value[2 * i + 1], v_scale);
  }
}

// Elementwise quantisation of a whole fp16 buffer (a cache, layout kept):
// vector i of 16 codes from fp16 vectors 2i and 2i+1.
__global__ void __launch_bounds__(256)
    convert_cache_fp8_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                             long long vecs, float scale) {
  pdl_wait();
  pdl_launch_dependents();
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += stride)
    dst[i] = quantize16(src[2 * i], src[2 * i + 1], scale);
}

// ---- copy-on-write block copy
// ("vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制" §2.3)
// blockIdx.y = pair, blockIdx.z = layer * 2 + (0 key | 1 value); blockIdx.x
// and the threads stride over the block's H*B*D/8 16-byte vectors.
struct LayerPtrs {
  uint4* k[kCopyMaxLayers];
  uint4* v[kCopyMaxLayers];
};

// Block copies and swaps check their whole mapping for conflicting pairs on
// the device: every CTA scans all pairs for the one it copies (the mapping's
// 16 bytes per pair stay in L2).  Up to this many pairs
// one CTA copies one (pair, cache, chunk) and the grid covers every cache;
// above it one CTA copies its pair's whole block in every cache, so each
// pair's scan runs once instead of once per cache and chunk (the scans then
// cost pairs^2 x 16 bytes of L2 reads in all).
constexpr int kMappingScanPerCachePairs = 1024;

// True when another pair of the mapping writes `dst` or reads it (with
// `dst_also_src`), i.e. copying this pair would race.  Every thread of the
// CTA must call it (it ends with a CTA-wide vote).  With scan false (the
// host already checked the whole mapping) it returns false at once.
__device__ __forceinline__ bool mapping_conflict(const int64_t* __restrict__ block_mapping,
                                                 int num_pairs, int pair, long long dst,
                                                 bool dst_also_src, bool scan) {
  if (!scan) return false;
  int hit = 0;
  for (int q = threadIdx.x; q < num_pairs; q += blockDim.x) {
    const long long qd = block_mapping[2 * q + 1];
    const long long qs = dst_also_src ? block_mapping[2 * q] : -1;
    if (q != pair && (qd == dst || qs == dst)) hit = 1;
  }
  return __syncthreads_or(hit) != 0;
}

__device__ __forceinline__ void copy_vecs(const uint4* __restrict__ s, uint4* __restrict__ d,
                                          long long n, long long first, long long stride) {
  for (long long i = first; i < n; i += stride) d[i] = s[i];
}

// blockIdx.y = pair; blockIdx.z = layer * 2 + (0 key | 1 value) when
// per_cache, else the CTA loops over all 2 * num_layers caches of the launch.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(LayerPtrs ptrs, const int64_t* __restrict__ block_mapping, int pair_base,
                       int num_pairs, long long block_vecs, long long num_blocks, int num_caches,
                       bool per_cache, bool scan, unsigned int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = pair_base + blockIdx.y;
  const long long src = block_mapping[2 * pair];
  const long long dst = block_mapping[2 * pair + 1];
  // every thread of the CTA reaches the check's vote
  const bool conflict = mapping_conflict(block_mapping, num_pairs, pair, dst, true, scan);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks || conflict) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) atomicOr(err, PA_ERRBIT_COPY);
    return;
  }
  const long long stride = (long long)gridDim.x * blockDim.x;
  const long long first = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int z0 = per_cache ? (int)blockIdx.z : 0;
  const int z1 = per_cache ? z0 + 1 : num_caches;
  for (int z = z0; z < z1; ++z) {
    uint4* base = (z & 1) ? ptrs.v[z >> 1] : ptrs.k[z >> 1];
    copy_vecs(base + src * block_vecs, base + dst * block_vecs, block_vecs, first, stride);
  }
}

// ---- block swap between device and host pools
// ("【硬核】啃透vLLM源码：从PagedAttention到连续批处理，大模型推理加速24倍的秘密" §三:
// blocks_to_swap_out / blocks_to_swap_in).  One launch moves every (pair,
// cache): blockIdx.y = pair, blockIdx.z = cache; blockIdx.x and the threads
// stride over the block's 16-byte vectors.  One side is host memory reached
// over the CPU-GPU link (pinned, mapped into the device's address space),
// so each thread keeps kSwapUnroll independent loads in flight before it
// stores.
struct SwapPtrs {
  const uint4* src[kSwapMaxCaches];
  uint4* dst[kSwapMaxCaches];
};

constexpr int kSwapUnroll = 4;

// blockIdx.y = pair; blockIdx.z = cache when per_cache, else the CTA loops
// over all caches of the launch.
__global__ void __launch_bounds__(256)
    swap_blocks_kernel(SwapPtrs ptrs, const int64_t* __restrict__ block_mapping, int pair_base,
                       int num_pairs, long long block_vecs, long long src_num_blocks,
                       long long dst_num_blocks, int num_caches, bool per_cache, bool scan,
                       unsigned int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int pair = pair_base + blockIdx.y;
  const long long src = block_mapping[2 * pair];
  const long long dst = block_mapping[2 * pair + 1];
  // every thread of the CTA reaches the check's vote
  const bool conflict = mapping_conflict(block_mapping, num_pairs, pair, dst, false, scan);
  if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks || conflict) {
    if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) atomicOr(err, PA_ERRBIT_COPY);
    return;
  }
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int z0 = per_cache ? (int)blockIdx.z : 0;
  const int z1 = per_cache ? z0 + 1 : num_caches;
  for (int z = z0; z < z1; ++z) {
    const uint4* s = ptrs.src[z] + src * block_vecs;
    uint4* d = ptrs.dst[z] + dst * block_vecs;
    long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kSwapUnroll - 1) * stride < block_vecs; i += kSwapUnroll * stride) {
      uint4 t[kSwapUnroll];
#pragma unroll
      for (int u = 0; u < kSwapUnroll; ++u) t[u] = s[i + u * stride];
#pragma unroll
      for (int u = 0; u < kSwapUnroll; ++u) d[i + u * stride] = t[u];
    }
    for (; i < block_vecs; i += stride) d[i] = s[i];
  }
}

// ---- slot map ("vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §2.3)
__global__ void __launch_bounds__(256)
    slot_mapping_kernel(int64_t* __restrict__ slot_mapping, const int32_t* __restrict__ block_tables,
                        int max_blocks, const int32_t* __restrict__ token_seq,
                        const int32_t* __restrict__ token_pos, int num_tokens, int num_seqs,
                        int block_size, int num_blocks, unsigned int* err) {
  pdl_wait();
  pdl_launch_dependents();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  const int s = token_seq[t];
  const int pos = token_pos[t];
  int64_t slot = -1;
  if (s >= 0) {
    bool ok = s < num_seqs && pos >= 0 && pos / block_size < max_blocks;
    if (ok) {
      const int phys = block_tables[(long long)s * max_blocks + pos / block_size];
      ok = phys >= 0 && phys < num_blocks;
      if (ok) slot = (int64_t)phys * block_size + pos % block_size;
    }
    if (!ok) atomicOr(err, PA_ERRBIT_TOKEN);
  }
  slot_mapping[t] = slot;
}

// Zeroes n 32-bit words (the decode workspace's work counters); a kernel
// rather than a memset so the decode call stays one chain of kernels.
__global__ void __launch_bounds__(128) zero_words_kernel(unsigned int* __restrict__ w, int n) {
  pdl_wait();
  pdl_launch_dependents();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) w[i] = 0u;
}

int log2_exact(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// A wait that nothing completes.  The barrier expects two arrivals and gets
// one, so its first phase never ends; the thread waits through the same
// bounded wait as the library's copy pipelines, which gives up after
// kWaitLimitNs and reports the timeout in the device error word.  No copy
// or other asynchronous operation is in flight when the kernel returns.
__global__ void selftest_wait_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 2);
  fence_mbar_init();
  mbar_arrive(b);
  if (!mbar_wait_bounded(b, 0)) atomicOr(err, PA_ERRBIT_TIMEOUT);
}

int sm_count() {
  int dev = 0, n = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

}  // namespace

cudaError_t launch_zero_words(unsigned int* words, int n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  return launch_pdl(zero_words_kernel, dim3(1), dim3(128), 0, stream, words, n);
}

cudaError_t launch_selftest_wait(unsigned int* err, cudaStream_t stream) {
  return launch_pdl(selftest_wait_kernel, dim3(1), dim3(32), 0, stream, err);
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int64_t* slot_mapping,
                                     int num_tokens, int num_heads, int head_dim, int block_size,
                                     int num_blocks, unsigned int* err, cudaStream_t stream) {
  const long long vecs = (long long)num_tokens * num_heads * (head_dim / 8);
  if (vecs == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (vecs + threads - 1) / threads;
  const long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const int lb = log2_exact(block_size);
  const long long slots = (long long)num_blocks * block_size;
  auto k = static_cast<const uint4*>(key);
  auto v = static_cast<const uint4*>(value);
  auto kc = static_cast<uint4*>(key_cache);
  auto vc = static_cast<uint4*>(value_cache);
  if (head_dim == 64)
    return launch_pdl(reshape_and_cache_kernel<64>, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, k, v, kc, vc, slot_mapping, num_tokens, num_heads, lb, slots, err);
  return launch_pdl(reshape_and_cache_kernel<128>, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    k, v, kc, vc, slot_mapping, num_tokens, num_heads, lb, slots, err);
}

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                         void* value_cache, const int64_t* slot_mapping,
                                         int num_tokens, int num_heads, int head_dim,
                                         int block_size, int num_blocks, float k_scale,
                                         float v_scale, unsigned int* err, cudaStream_t stream) {
  const long long vecs = (long long)num_tokens * num_heads * (head_dim / 16);
  if (vecs == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (vecs + threads - 1) / threads;
  const long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  const int lb = log2_exact(block_size);
  const long long slots = (long long)num_blocks * block_size;
  auto k = static_cast<const uint4*>(key);
  auto v = static_cast<const uint4*>(value);
  auto kc = static_cast<uint4*>(key_cache);
  auto vc = static_cast<uint4*>(value_cache);
  if (head_dim == 64)
    return launch_pdl(reshape_and_cache_fp8_kernel<64>, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, k, v, kc, vc, slot_mapping, num_tokens, num_heads, lb, slots,
                      k_scale, v_scale, err);
  return launch_pdl(reshape_and_cache_fp8_kernel<128>, dim3((unsigned)blocks), dim3(threads), 0,
                    stream, k, v, kc, vc, slot_mapping, num_tokens, num_heads, lb, slots, k_scale,
                    v_scale, err);
}

cudaError_t launch_convert_cache_fp8(const void* src, void* dst, long long num_elems, float scale,
                                     cudaStream_t stream) {
  const long long vecs = num_elems / 16;
  if (vecs == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (vecs + threads - 1) / threads;
  const long long cap = (long long)sm_count() * 16;
  if (blocks > cap) blocks = cap;
  return launch_pdl(convert_cache_fp8_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), vecs, scale);
}

cudaError_t launch_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                               const int64_t* block_mapping, int num_pairs, int num_heads,
                               int head_dim, int block_size, int elem_bytes, int num_blocks,
                               bool scan, unsigned int* err, cudaStream_t stream) {
  if (num_pairs == 0 || num_layers == 0) return cudaSuccess;
  const long long block_vecs = (long long)num_heads * block_size * head_dim * elem_bytes / 16;
  const int threads = 256;
  long long xblocks = (block_vecs + threads - 1) / threads;
  if (xblocks > 64) xblocks = 64;
  for (int l0 = 0; l0 < num_layers; l0 += kCopyMaxLayers) {
    const int nl = num_layers - l0 < kCopyMaxLayers ? num_layers - l0 : kCopyMaxLayers;
    LayerPtrs ptrs{};
    for (int i = 0; i < nl; ++i) {
      ptrs.k[i] = static_cast<uint4*>(key_caches[l0 + i]);
      ptrs.v[i] = static_cast<uint4*>(value_caches[l0 + i]);
    }
    const bool per_cache = num_pairs <= kMappingScanPerCachePairs;
    for (int p0 = 0; p0 < num_pairs; p0 += 65535) {
      const int np = num_pairs - p0 < 65535 ? num_pairs - p0 : 65535;
      dim3 grid(per_cache ? (unsigned)xblocks : 1u, (unsigned)np, per_cache ? (unsigned)(2 * nl) : 1u);
      const cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(threads), 0, stream, ptrs,
                                       block_mapping, p0, num_pairs, block_vecs,
                                       (long long)num_blocks, 2 * nl, per_cache, scan, err);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_swap_blocks(void* const* dst_caches, const void* const* src_caches,
                               int num_caches, const int64_t* block_mapping, int num_pairs,
                               long long block_bytes, long long src_num_blocks,
                               long long dst_num_blocks, bool scan, unsigned int* err,
                               cudaStream_t stream) {
  if (num_pairs == 0 || num_caches == 0) return cudaSuccess;
  const long long block_vecs = block_bytes / 16;
  const int threads = 256;
  long long xblocks = (block_vecs + threads * kSwapUnroll - 1) / (threads * kSwapUnroll);
  if (xblocks > 64) xblocks = 64;
  for (int c0 = 0; c0 < num_caches; c0 += kSwapMaxCaches) {
    const int nc = num_caches - c0 < kSwapMaxCaches ? num_caches - c0 : kSwapMaxCaches;
    SwapPtrs ptrs{};
    for (int i = 0; i < nc; ++i) {
      ptrs.src[i] = static_cast<const uint4*>(src_caches[c0 + i]);
      ptrs.dst[i] = static_cast<uint4*>(dst_caches[c0 + i]);
    }
    const bool per_cache = num_pairs <= kMappingScanPerCachePairs;
    for (int p0 = 0; p0 < num_pairs; p0 += 65535) {
      const int np = num_pairs - p0 < 65535 ? num_pairs - p0 : 65535;
      dim3 grid(per_cache ? (unsigned)xblocks : 1u, (unsigned)np, per_cache ? (unsigned)nc : 1u);
      const cudaError_t e = launch_pdl(swap_blocks_kernel, grid, dim3(threads), 0, stream, ptrs,
                                       block_mapping, p0, num_pairs, block_vecs, src_num_blocks,
                                       dst_num_blocks, nc, per_cache, scan, err);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

cudaError_t launch_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                                int max_blocks, const int32_t* token_seq,
                                const int32_t* token_pos, int num_tokens, int num_seqs,
                                int block_size, int num_blocks, unsigned int* err,
                                cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = (num_tokens + threads - 1) / threads;
  return launch_pdl(slot_mapping_kernel, dim3(blocks), dim3(threads), 0, stream, slot_mapping,
                    block_tables, max_blocks, token_seq, token_pos, num_tokens, num_seqs,
                    block_size, num_blocks, err);
}

}  // namespace pa
