// Internal declarations shared by the library's translation units (not part
// of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Sequences handled by one launch of the partition kernel: their per-sequence
// item counts and prefix sums live in shared memory.
constexpr int kMaxSeqsPerLaunch = 1024;
// Layers handled by one launch of the block-copy kernel (pointer table passed
// by value as a kernel parameter).
constexpr int kCopyMaxLayers = 32;
// Caches handled by one launch of the block-swap kernel.
constexpr int kSwapMaxCaches = 64;

struct DecodeParams {
  void* out;                  // fp16 [S][H][D]
  const void* query;          // fp16 [S][H][D]
  const void* key_cache;      // fp16 or E4M3 [NB][H][B][D]
  const void* value_cache;    // fp16 or E4M3 [NB][H][B][D]
  const int32_t* block_tables;  // [S][max_blocks]
  const int32_t* context_lens;  // [S]
  float* ws_ml;               // [S][H][max_parts][2]: running max (base-2 units) and sum
  float* ws_o;                // [S][H][max_parts][D]: unnormalised output
  unsigned int* counter;      // work counter of this launch (zeroed before it)
  unsigned int* err;          // device error word
  int seq_begin;              // first sequence of this launch
  int num_seqs;               // sequences in this launch
  int num_heads;
  int max_blocks;             // block-table row length
  int num_blocks;             // pool size
  int max_context_len;        // host bound; larger lengths are clipped and flagged
  int part_tokens;            // tokens per partition (multiple of 32)
  int max_parts;              // ceil(max_context_len / part_tokens)
  float scale_log2;           // scale * log2(e) (* k_scale for E4M3 caches): base-2 logits
  float v_scale;              // E4M3 caches: multiplies the output (unused for fp16)
  // Decode with the cache write fused in (null otherwise): fp16 [S][H][D]
  // rows written to position context_len - 1 of each sequence before use.
  const void* key_new;
  const void* value_new;
  float k_scale;              // E4M3 caches: quantisation scale of key_new (v_scale for values)
  // 1: a kernel before this one in the same call already waited for the
  // stream's earlier work, so the inputs are complete when this launch starts
  // and its prologue reads them before its own wait; 0: it waits first.
  int inputs_ready;
};

// Partition-kernel launch: picks the instantiation for (cache element type,
// head_dim, block_size); fp8 selects E4M3 caches.
cudaError_t launch_decode_partition(const DecodeParams& p, bool fp8, int head_dim, int block_size,
                                    int grid, size_t smem_bytes, cudaStream_t stream);
// LSE-merge launch over all (seq, head) pairs of the batch.
cudaError_t launch_decode_reduce(const DecodeParams& p, int head_dim, int block_size,
                                 int total_seqs, cudaStream_t stream);
// Dynamic shared memory of the partition kernel.
size_t decode_smem_bytes(bool fp8, int head_dim, int block_size, int part_tokens,
                         int seqs_in_launch);
// Resident CTAs per SM of the partition kernel (append: the variant with the
// cache write fused in) for that shared-memory size.
int decode_ctas_per_sm(bool fp8, int head_dim, int block_size, size_t smem_bytes, bool append);
// One-time per-device kernel attributes (dynamic shared memory opt-in).
cudaError_t decode_prepare_device(int device);

// Zeroes n 32-bit words on the stream (one small kernel).
cudaError_t launch_zero_words(unsigned int* words, int n, cudaStream_t stream);
// One thread waits, through the kernels' bounded wait, on a barrier that
// never completes; the wait gives up and sets PA_ERRBIT_TIMEOUT in `err`.
cudaError_t launch_selftest_wait(unsigned int* err, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int64_t* slot_mapping,
                                     int num_tokens, int num_heads, int head_dim, int block_size,
                                     int num_blocks, unsigned int* err, cudaStream_t stream);

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                         void* value_cache, const int64_t* slot_mapping,
                                         int num_tokens, int num_heads, int head_dim,
                                         int block_size, int num_blocks, float k_scale,
                                         float v_scale, unsigned int* err, cudaStream_t stream);

// num_elems: a multiple of 16.
cudaError_t launch_convert_cache_fp8(const void* src, void* dst, long long num_elems, float scale,
                                     cudaStream_t stream);

// elem_bytes: 2 for fp16 caches, 1 for E4M3 caches.
cudaError_t launch_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                               const int64_t* block_mapping, int num_pairs, int num_heads,
                               int head_dim, int block_size, int elem_bytes, int num_blocks,
                               bool scan, unsigned int* err, cudaStream_t stream);

// block_bytes: a multiple of 16; pointers are device addresses (device
// memory or mapped pinned host memory).  scan: the kernel checks the mapping
// for conflicting pairs (false when the host already checked it).
cudaError_t launch_swap_blocks(void* const* dst_caches, const void* const* src_caches,
                               int num_caches, const int64_t* block_mapping, int num_pairs,
                               long long block_bytes, long long src_num_blocks,
                               long long dst_num_blocks, bool scan, unsigned int* err,
                               cudaStream_t stream);

// Multi-query paged attention (tensor cores): arguments as in pa_prefill.
struct PrefillArgs {
  void* out;
  const void* query;
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  unsigned int* err;
  int num_seqs, num_query_tokens, num_heads, head_dim, block_size, num_blocks, max_blocks;
  int max_query_len;
  float scale_log2;   // scale * log2(e) (times the key scale for FP8 caches)
  bool fp8;           // E4M3 caches (uint8 codes)
  float v_scale;      // FP8 caches: value scale
  bool inputs_ready;  // the kernel before the call writes none of its inputs (read before the wait)
  int num_decode_rows;  // the call's one-token sequences, or -1 when the caller does not say
};
cudaError_t launch_prefill(const PrefillArgs& args, cudaStream_t stream);
// The cache's rows (num_blocks * num_heads * block_size) fit the kernel's int coordinates.
bool prefill_rows_fit(int num_blocks, int num_heads, int block_size);

cudaError_t launch_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                                int max_blocks, const int32_t* token_seq,
                                const int32_t* token_pos, int num_tokens, int num_seqs,
                                int block_size, int num_blocks, unsigned int* err,
                                cudaStream_t stream);

}  // namespace pa
