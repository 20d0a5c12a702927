/*
 * pa.h — C ABI of libpa.so, a GB300 (sm_103a) library for the PagedAttention
 * decode hot path: single-query attention over a paged fp16 (or FP8 E4M3)
 * KV cache, the cache write that scatters new tokens into their slots, the
 * copy-on-write block copy, and the slot map.
 *
 * Sources (page title, section):
 *   [P1] "深入解析LLM推理引擎：从PagedAttention到调度优化"
 *   [P2] "vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量"
 *   [P3] "vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制"
 *
 * Conventions for every call:
 *   - All array pointers are device memory owned by the caller, C-contiguous,
 *     16-byte aligned unless stated otherwise.  The library keeps no pointer
 *     after a call returns and allocates no device memory.
 *   - fp16 arrays are IEEE binary16; int32 / int64 arrays as named.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream) and never synchronise it, except pa_check_errors.
 *   - Host-detectable errors (null pointer, misalignment, unsupported shape,
 *     too small a workspace) return a status and launch nothing.
 *   - Index errors found on the device (a block id outside [0, num_blocks),
 *     a slot past the pool, a context length past the block table) never
 *     trap: the offending item is skipped, a bit is set in the library's
 *     device error word, and pa_check_errors reports it.
 *   - Cache layout per layer: key_cache and value_cache are fp16
 *     [num_blocks][num_heads][block_size][head_dim]; one (block, head) tile
 *     of block_size * head_dim values is contiguous.
 *   - Supported shapes: head_dim in {64, 128}; block_size in {4, 8, 16, 32}.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (same underlying type, without including CUDA headers). */
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,  /* null pointer, misaligned pointer, bad size, small workspace */
  PA_ERR_UNSUPPORTED = 2,  /* head_dim or block_size outside the supported set           */
  PA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed                        */
  PA_ERR_OUT_OF_RANGE = 4, /* the device found an index outside its array (see bits)      */
  PA_ERR_TIMEOUT = 5       /* a bounded wait inside a kernel gave up (see bits)           */
} pa_status;

/* Bits of the device error word, as returned by pa_check_errors. */
#define PA_ERRBIT_BLOCK_ID 0x1u  /* decode: a block-table entry outside [0, num_blocks)        */
#define PA_ERRBIT_CONTEXT 0x2u   /* decode: context_len < 0, > max_blocks_per_seq*block_size,
                                    or > max_context_len                                      */
#define PA_ERRBIT_SLOT 0x4u      /* cache write: slot >= num_blocks*block_size                 */
#define PA_ERRBIT_COPY 0x8u      /* block copy: a src/dst id outside [0, num_blocks)           */
#define PA_ERRBIT_TOKEN 0x10u    /* slot map: sequence, position or table entry out of range   */
#define PA_ERRBIT_TIMEOUT 0x20u  /* a kernel's bounded wait on its own copies gave up          */

/*
 * Bytes of device scratch pa_decode needs for this batch shape.  The decode
 * splits each sequence's context into partitions and keeps, per partition,
 * the running maximum, the softmax denominator and the unnormalised output
 * (fp32), plus a work counter that every call zeroes before its kernels
 * run.  0 on invalid arguments.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len);

/*
 * Decode attention over the paged cache [P2 §2.1 attention formula; P2 §2.3
 * paged formula and address map K_paged[i] = K_physical[BlockTable[i div B]][i mod B];
 * P1 §3.3 gather through the block table at attention time]:
 *
 *   out[s,h,:] = softmax( scale * q[s,h,:] . K_paged[s,h,i,:] for i < c_s ) . V_paged[s,h,:,:]
 *
 * with c_s = context_lens[s] (it counts the token written just before this
 * call), K_paged[s,h,i,:] = key_cache[block_tables[s][i / block_size]][h][i % block_size][:]
 * and the same for V.  A sequence with c_s == 0 gets a zero row.
 *
 *   out            fp16 [num_seqs][num_heads][head_dim]          (written)
 *   query          fp16 [num_seqs][num_heads][head_dim]
 *   key_cache,
 *   value_cache    fp16 [num_blocks][num_heads][block_size][head_dim]
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(c_s / block_size) are never read (any value)
 *   context_lens   int32 [num_seqs]
 *   scale          multiplier of q.k (normally 1/sqrt(head_dim))
 *   max_context_len  host-side upper bound of context_lens (sizes the launch;
 *                  a larger c_s is clipped and flagged PA_ERRBIT_CONTEXT)
 *   workspace      device scratch of at least pa_decode_workspace_size(...)
 *                  bytes, 16-byte aligned; contents on entry are ignored (its
 *                  work counters are zeroed first) and on exit the counters
 *                  are zero and the rest undefined (see pa_decode_ex).  Calls
 *                  that share one workspace must not overlap on the GPU.
 *
 * Arithmetic: fp16 inputs, fp32 dot products, online softmax and
 * accumulation; the result is rounded once to fp16 (nearest even).  The
 * summation order depends only on logical token positions, so results are
 * bit-identical under any relabelling of physical blocks and between shared
 * and privately copied blocks with equal contents.
 */
pa_status pa_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, int max_blocks_per_seq,
                    const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                    int block_size, int num_blocks, float scale, int max_context_len,
                    void* workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode with flags.  With flags == 0 it is pa_decode.
 *
 * PA_DECODE_ZEROED_WORKSPACE: the workspace's work counters are zero when
 * the call starts, so the call launches no kernel to zero them (one kernel
 * fewer on each layer's dependency chain: 1.9 % on the 13B-shaped decode
 * step).  Every call leaves the counters zero, whatever its flags, so the
 * flag holds for a workspace that was zero-filled once before its first call
 * (e.g. cudaMemsetAsync) and since then only passed to pa_decode* calls.  A
 * call that timed out (PA_ERR_TIMEOUT) leaves them zero as well; a workspace
 * whose bytes anything else wrote must be zero-filled again.  Counters that
 * are not zero make the call skip or repeat work without any report.
 * The call's first kernel is then the decode itself, which may start while
 * the kernel enqueued just before the call still runs (programmatic launch):
 * it waits for that kernel before it reads any input, unless
 * PA_DECODE_INPUTS_READY is passed as well.
 *
 * PA_DECODE_INPUTS_READY (with PA_DECODE_ZEROED_WORKSPACE; alone it changes
 * nothing): the kernel enqueued on the stream just before this call writes
 * none of the call's inputs (query, caches, block tables, context lengths,
 * and for pa_decode_append the new keys and values).  The decode then reads
 * its context lengths, the first block-table slices and the first cache
 * chunks while that kernel finishes, instead of after it; the results are
 * written only after it has ended.  A preceding kernel that does write an
 * input (a cache write, a block copy or swap-in, a kernel producing the
 * queries) makes the call read stale values without any report.  The
 * library's decode step passes it for every layer but the first when the
 * cache write is fused in (the kernel before layer i's decode is then layer
 * i - 1's decode): 1 % on the 13B-shaped step.
 * Not part of the pages; launch-latency options.
 */
#define PA_DECODE_ZEROED_WORKSPACE 1u
#define PA_DECODE_INPUTS_READY 2u
pa_status pa_decode_ex(void* out, const void* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                       int block_size, int num_blocks, float scale, int max_context_len,
                       void* workspace, size_t workspace_bytes, unsigned int flags,
                       pa_stream_t stream);

/*
 * The decode step of one layer in one call: the cache write of each
 * sequence's new token [P1 §3.2: the new token's K/V go to slot
 * block*B + offset of its block; P3 §2.3] fused into pa_decode_ex.  For every
 * sequence s with c_s = context_lens[s] >= 1 the new token is the one at
 * position c_s - 1:
 *
 *   key_cache[block_tables[s][(c_s-1) / B]][h][(c_s-1) % B][:] = key_new[s][h][:]   (same for V)
 *
 * and the decode over [0, c_s) then uses it.  Result and cache contents are
 * bit-identical to pa_slot_mapping + pa_reshape_and_cache of those rows (the
 * token of sequence s at position c_s - 1) followed by pa_decode_ex, with one
 * kernel fewer on the layer's dependency chain.
 *
 *   key_new,
 *   value_new      fp16 [num_seqs][num_heads][head_dim], 16-byte aligned
 *   key_cache,
 *   value_cache    written (one row per (sequence, head)); otherwise as for
 *                  pa_decode_ex, as are the other arguments and flags
 * A sequence with c_s == 0 writes nothing.  A sequence whose c_s is clipped
 * (past its table or max_context_len; PA_ERRBIT_CONTEXT) or whose block for
 * position c_s - 1 is out of range (PA_ERRBIT_BLOCK_ID) writes nothing.
 */
pa_status pa_decode_append(void* out, const void* query, const void* key_new,
                           const void* value_new, void* key_cache, void* value_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* context_lens, int num_seqs, int num_heads, int head_dim,
                           int block_size, int num_blocks, float scale, int max_context_len,
                           void* workspace, size_t workspace_bytes, unsigned int flags,
                           pa_stream_t stream);

/* Size of the fixed scratch area pa_decode_noalloc uses (32 MiB per device). */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * pa_decode without a workspace argument, for callers that cannot allocate
 * device memory at the moment they decode: processes that give all of HBM
 * to the KV pool up front and keep no allocator headroom, hot paths that must
 * not call cudaMalloc/cudaFree because those may synchronise the device, and
 * plain C callers that own no device allocator.  The pages have no
 * counterpart; it is a deployment convenience.
 *
 * Same arguments, result and arithmetic as pa_decode.  The scratch is a fixed
 * array of PA_DECODE_NOALLOC_SCRATCH_BYTES in the library's own device memory
 * (a __device__ variable).  This call allocates nothing and calls no
 * allocating routine.
 *   - If pa_decode_workspace_size(num_seqs, num_heads, head_dim,
 *     max_context_len) exceeds PA_DECODE_NOALLOC_SCRATCH_BYTES the call
 *     returns PA_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on each device is a warm-up.  Under CUDA's lazy module
 *     loading (the default) it loads the module that holds the array, which
 *     commits the array's bytes on that device until the process exits, and
 *     it looks up the array's device address (cudaGetSymbolAddress, with that
 *     device current) and caches it.  Make that first call before the rest of
 *     device memory is reserved (for the KV pool, say) and before any stream
 *     capture on that device.  If it fails (PA_ERR_CUDA, typically out of
 *     memory) the CUDA last error is cleared and a later call may retry.
 *   - All calls on a device share the one array, which keeps the previous
 *     call's contents; the work counters are zeroed by every call.  Calls
 *     that overlap on the GPU (e.g. on two streams) race on the array and
 *     must be serialised by the caller.
 */
pa_status pa_decode_noalloc(void* out, const void* query, const void* key_cache,
                            const void* value_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                            int num_heads, int head_dim, int block_size, int num_blocks,
                            float scale, int max_context_len, pa_stream_t stream);

/*
 * Cache write [P1 §3.2: a block fills token by token, a new block is taken
 * when the last one is full; P3 §2.3: blocks are taken on demand every
 * block_size tokens]: token t's key and value vectors for every head go to
 * slot slot_mapping[t], i.e.
 *
 *   key_cache[slot / block_size][h][slot % block_size][:] = key[t][h][:]   (same for value)
 *
 * slot_mapping[t] < 0 marks a padding token: skipped, not an error.  A slot
 * >= num_blocks * block_size is skipped and flagged PA_ERRBIT_SLOT.  Two
 * tokens with the same slot race (the result is one of them).
 *
 *   key, value     fp16 [num_tokens][num_heads][head_dim]
 *   key_cache,
 *   value_cache    fp16 [num_blocks][num_heads][block_size][head_dim] (updated)
 *   slot_mapping   int64 [num_tokens]
 * num_tokens == 0 is a no-op.  Bit-exact copy; nothing else is touched.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* key_cache,
                               void* value_cache, const int64_t* slot_mapping, int num_tokens,
                               int num_heads, int head_dim, int block_size, int num_blocks,
                               pa_stream_t stream);

/*
 * Copy-on-write block copy [P3 §2.3: a shared block stays shared until a
 * request writes different content into it; then the block is copied and
 * that request's table is repointed; P3 §2.1 components table: the block
 * manager owns allocation, release and copy-on-write]: for every pair p
 * and every layer l,
 *
 *   key_caches[l][dst_p][:][:][:] = key_caches[l][src_p][:][:][:]   (same for value_caches)
 *
 * with (src_p, dst_p) = (block_mapping[2p], block_mapping[2p+1]).
 *
 *   key_caches,
 *   value_caches   HOST arrays of num_layers device pointers, each to an fp16
 *                  [num_blocks][num_heads][block_size][head_dim] cache
 *   block_mapping  int64 [num_pairs][2], device memory or pinned host memory
 *                  (the kernel reads pinned memory over the CPU-GPU link);
 *                  pageable host memory returns PA_ERR_INVALID_ARG
 * Preconditions: destination ids are distinct and no destination is also a
 * source in the same call (a pair copying a block onto itself is allowed).
 * They are checked for any num_pairs:
 *   - a pinned host mapping is checked on the host when the call is made
 *     (O(P log P)); a violation returns PA_ERR_INVALID_ARG and launches
 *     nothing.  The mapping must not change until the stream reaches the
 *     copy (a CUDA graph that captured the call does not re-check it);
 *   - a device mapping is checked on the device: every pair's CTA scans the
 *     whole mapping, and a pair whose destination is another pair's
 *     destination or source is skipped (not copied) and sets
 *     PA_ERRBIT_COPY, so nothing races.  The scans cost num_pairs^2 x 16
 *     bytes of L2 reads in all (above 1024 pairs one CTA copies a pair's
 *     block in every layer, so each pair is scanned once).
 * An id outside [0, num_blocks) skips that pair and sets PA_ERRBIT_COPY.
 * num_pairs == 0 is a no-op.  Bit-exact.
 */
pa_status pa_copy_blocks(void* const* key_caches, void* const* value_caches, int num_layers,
                         const int64_t* block_mapping, int num_pairs, int num_heads, int head_dim,
                         int block_size, int num_blocks, pa_stream_t stream);

/*
 * Multi-query paged attention: chunked prefill and mixed prefill + decode
 * batches [P2 §4.3: prefill (the prompt) and decode (generated tokens) can
 * share one batch; P2 §2.1 and §2.3: attention over K/V gathered through the
 * block table; P1 §3.3].  Sequence s brings
 * q_len_s = query_start[s+1] - query_start[s] new tokens, which are the last
 * q_len_s of its c_s = context_lens[s] cached tokens (written before this
 * call by pa_reshape_and_cache).  New token j of sequence s sits at position
 * p = c_s - q_len_s + j and attends causally:
 *
 *   out[query_start[s]+j, h, :] = softmax( scale * q . K_paged[s,h,i,:] for i <= p ) . V_paged[s,h,:,:]
 *
 * A one-token chunk is decode; q_len_s == 0 contributes nothing.
 *
 *   out            fp16 [num_query_tokens][num_heads][head_dim]   (written for
 *                  the rows of valid sequences)
 *   query          fp16 [num_query_tokens][num_heads][head_dim]
 *   key_cache,
 *   value_cache    fp16 [num_blocks][num_heads][block_size][head_dim]
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   context_lens   int32 [num_seqs]
 *   query_start    int32 [num_seqs + 1], non-decreasing, query_start[0] = 0,
 *                  query_start[num_seqs] = num_query_tokens
 *   max_query_len  host-side upper bound of q_len (sizes the launch)
 * A sequence with q_len < 0, q_len > c_s, c_s past its table, q_len >
 * max_query_len or query rows outside [0, num_query_tokens) is skipped and
 * flagged PA_ERRBIT_CONTEXT; a block id outside
 * [0, num_blocks) reads zeros and is flagged PA_ERRBIT_BLOCK_ID.
 *
 * Supported: head_dim in {64, 128}, block_size in {8, 16, 32}, num_blocks *
 * num_heads * block_size < 2^31.  Chunks (q_len >= 2) run on the tensor
 * cores (tcgen05.mma, fp16 operands, fp32 accumulation in tensor memory);
 * one-token rows run in the same launch on CUDA cores, with the decode
 * kernel's fp32 online softmax over the whole context: one CTA per row and
 * head, or per row and four heads when the launch knows how many one-token
 * rows the batch holds (max_query_len == 1, or num_decode_rows given to
 * pa_prefill_ex / pa_prefill_fp8_ex).  The softmax weights
 * are computed in fp32 and rounded once to fp16 for the second product (the
 * denominator sums them in fp32); the result is rounded once to fp16.  The
 * call allocates nothing; batches of more than 4096 sequences take one
 * launch per 4096.
 */
pa_status pa_prefill(void* out, const void* query, const void* key_cache, const void* value_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, const int32_t* query_start, int num_seqs,
                     int num_query_tokens, int num_heads, int head_dim, int block_size,
                     int num_blocks, float scale, int max_query_len, pa_stream_t stream);

/*
 * pa_prefill over FP8 (E4M3) caches [P2 §3.3: FP8 KV caches; format and
 * scaling as for pa_decode_fp8]: the same causal attention with
 * K_paged[s,h,i,:] = E4M3(key code) * k_scale and V likewise with v_scale.
 * key_cache / value_cache are uint8 [num_blocks][num_heads][block_size]
 * [head_dim] codes; query and out stay fp16.  The kernel widens each K / V
 * tile to fp16 in shared memory (exact) and runs the same tensor-core
 * products; the key scale is folded into the logit scale and the value scale
 * applied with the final division.  k_scale and v_scale must be finite and
 * positive (else PA_ERR_INVALID_ARG).  Everything else as pa_prefill.
 */
pa_status pa_prefill_fp8(void* out, const void* query, const void* key_cache,
                         const void* value_cache, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* context_lens,
                         const int32_t* query_start, int num_seqs, int num_query_tokens,
                         int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                         float k_scale, float v_scale, int max_query_len, pa_stream_t stream);

/*
 * pa_prefill and pa_prefill_fp8 with a batch-composition hint and flags.
 * With num_decode_rows == -1 and flags == 0 they are pa_prefill and
 * pa_prefill_fp8.
 *
 * num_decode_rows: the number of sequences with q_len == 1 (decode rows), or
 * -1 when the caller does not know it.  Not part of the pages: the launch
 * is sized from it, so that a one-token row CTA can cover up to four heads
 * of its row (one plan, one start-up latency and one CTA turnover instead
 * of four; the last wave of rows keeps one head per CTA) with no idle CTAs.
 * Used when num_seqs <= 4096 (one launch); ignored otherwise.  A count
 * other than the true one makes the launch either larger than needed (idle
 * CTAs, correct results) or too small: then the units past the grid are not
 * computed, their output rows are left as they were, and PA_ERRBIT_CONTEXT
 * is set.  Outside [-1, min(num_seqs, num_query_tokens)]:
 * PA_ERR_INVALID_ARG.
 *
 * The kernel may start while the kernel enqueued just before the call still
 * runs (programmatic launch); by default it waits for that kernel before it
 * reads any input.
 *
 * PA_PREFILL_INPUTS_READY: the kernel enqueued on the stream just before this
 * call writes none of the call's inputs (query, caches, block tables,
 * context lengths, query_start).  The kernel then plans its work, loads its
 * query and K/V tiles and computes while that kernel finishes, and waits for
 * it only before it stores the output.  Calls on independent data (other
 * layers' or other batches' prefill calls, say) then overlap: a call's first
 * CTAs fill the SMs the previous call's last wave leaves idle.  A preceding
 * kernel that writes an input (a cache write, a projection producing the
 * queries) makes the call read stale values without any report.  Not part
 * of the pages; a launch-latency option.  Unknown flag bits return
 * PA_ERR_INVALID_ARG.
 */
#define PA_PREFILL_INPUTS_READY 2u
pa_status pa_prefill_ex(void* out, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens,
                        const int32_t* query_start, int num_seqs, int num_query_tokens,
                        int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                        int max_query_len, int num_decode_rows, unsigned int flags,
                        pa_stream_t stream);
pa_status pa_prefill_fp8_ex(void* out, const void* query, const void* key_cache,
                            const void* value_cache, const int32_t* block_tables,
                            int max_blocks_per_seq, const int32_t* context_lens,
                            const int32_t* query_start, int num_seqs, int num_query_tokens,
                            int num_heads, int head_dim, int block_size, int num_blocks,
                            float scale, float k_scale, float v_scale, int max_query_len,
                            int num_decode_rows, unsigned int flags, pa_stream_t stream);

/*
 * Block swap between the device cache and a host copy [P4 §三: when GPU
 * memory runs short the scheduler moves some blocks to CPU memory and brings
 * them back when needed (blocks_to_swap_out / blocks_to_swap_in); P2 §4.3:
 * preemption pauses requests when memory runs short]: for every pair p and
 * every cache c,
 *
 *   dst_caches[c] block dst_p  :=  src_caches[c] block src_p   (block_bytes bytes)
 *
 * with (src_p, dst_p) = (block_mapping[2p], block_mapping[2p+1]) and block k
 * of a cache being bytes [k * block_bytes, (k+1) * block_bytes).  Pass every
 * layer's key and value caches (2 * num_layers caches; block_bytes =
 * num_heads * block_size * head_dim * element size).  Swap-out: sources on
 * the device, destinations in host memory; swap-in: the reverse.  One launch
 * moves all pairs of all caches.
 *
 *   dst_caches,
 *   src_caches     HOST arrays of num_caches pointers.  Each pointer is device
 *                  memory of the current device or pinned (page-locked:
 *                  cudaHostAlloc / cudaHostRegister) host memory; the kernel
 *                  reaches host memory directly over the CPU-GPU link.
 *                  Pageable host memory or another device's memory returns
 *                  PA_ERR_INVALID_ARG.  16-byte aligned.
 *   block_mapping  int64 [num_pairs][2], device memory or pinned host memory
 *   block_bytes    a multiple of 16
 *   src_num_blocks, dst_num_blocks  pool sizes; an id outside [0, n) skips
 *                  the pair and sets PA_ERRBIT_COPY
 * Destination blocks must be distinct, for any num_pairs: a pinned host
 * mapping is checked on the host when the call is made (a repeated
 * destination returns PA_ERR_INVALID_ARG and launches nothing; the mapping
 * must not change until the stream reaches the copy), and a device mapping
 * on the device, where every pair's CTA scans the whole mapping, so a pair
 * whose destination repeats another's is skipped and sets PA_ERRBIT_COPY.  Source and
 * destination pools must not overlap.  Bit-exact.  The
 * host side must stay allocated and unchanged until the stream reaches the
 * copy.
 */
pa_status pa_swap_blocks(void* const* dst_caches, const void* const* src_caches, int num_caches,
                         const int64_t* block_mapping, int num_pairs, size_t block_bytes,
                         int64_t src_num_blocks, int64_t dst_num_blocks, pa_stream_t stream);

/* ---- FP8 KV cache ------------------------------------------------------
 * [P2 §3.3 lists FP8 KV caches among the memory optimisations; the pages fix
 * neither the format nor the scaling.]  The library's reading: OCP FP8 E4M3
 * ("e4m3fn": 1 sign bit, 4 exponent bits of bias 7, 3 fraction bits, no
 * infinities, codes 0x7F and 0xFF are NaN, largest finite value 448) with one
 * fp32 scale per cache tensor.  An FP8 cache has the fp16 cache's layout
 * with one-byte elements, uint8 [num_blocks][num_heads][block_size][head_dim],
 * and code c stands for the value E4M3(c) * scale.  It holds a token in half
 * the bytes, so decode reads half as much.  Scales must be finite and
 * positive (PA_ERR_INVALID_ARG otherwise).
 */

/*
 * Cache write into FP8 caches: the slots, padding and error rules of
 * pa_reshape_and_cache, storing for each element x (fp16) the code
 *
 *   E4M3( fl32(x / scale) )   with scale = k_scale for keys, v_scale for values,
 *
 * where fl32 is IEEE binary32 division rounded to nearest and E4M3(.) rounds
 * to the nearest code (ties to even), saturating to +-448.  Bit-exact.
 *
 *   key, value     fp16 [num_tokens][num_heads][head_dim]
 *   key_cache,
 *   value_cache    uint8 [num_blocks][num_heads][block_size][head_dim] (updated)
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int64_t* slot_mapping, int num_tokens,
                                   int num_heads, int head_dim, int block_size, int num_blocks,
                                   float k_scale, float v_scale, pa_stream_t stream);

/*
 * Decode attention over FP8 caches: pa_decode's formula, shapes, workspace
 * (pa_decode_workspace_size) and error rules, on the dequantised cache
 * K = E4M3(code) * k_scale, V = E4M3(code) * v_scale.
 *
 *   key_cache,
 *   value_cache    uint8 [num_blocks][num_heads][block_size][head_dim]
 *
 * Arithmetic: the codes are widened to fp16 exactly; dot products, softmax
 * and accumulation as in pa_decode with the logit multiplier
 * fl32(scale * k_scale * log2 e) (base-2 exponentials); the merged output is
 * multiplied by v_scale in fp32 and rounded once to fp16.
 */
pa_status pa_decode_fp8(void* out, const void* query, const void* key_cache,
                        const void* value_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                        int num_heads, int head_dim, int block_size, int num_blocks, float scale,
                        float k_scale, float v_scale, int max_context_len, void* workspace,
                        size_t workspace_bytes, pa_stream_t stream);

/*
 * pa_decode_append over FP8 caches: the new rows are quantised as
 * pa_reshape_and_cache_fp8 quantises them (k_scale for keys, v_scale for
 * values; bit-identical codes) and the decode is pa_decode_fp8_ex's.
 */
pa_status pa_decode_append_fp8(void* out, const void* query, const void* key_new,
                               const void* value_new, void* key_cache, void* value_cache,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_heads,
                               int head_dim, int block_size, int num_blocks, float scale,
                               float k_scale, float v_scale, int max_context_len,
                               void* workspace, size_t workspace_bytes, unsigned int flags,
                               pa_stream_t stream);

/* pa_decode_fp8 with flags (see pa_decode_ex). */
pa_status pa_decode_fp8_ex(void* out, const void* query, const void* key_cache,
                           const void* value_cache, const int32_t* block_tables,
                           int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                           int num_heads, int head_dim, int block_size, int num_blocks,
                           float scale, float k_scale, float v_scale, int max_context_len,
                           void* workspace, size_t workspace_bytes, unsigned int flags,
                           pa_stream_t stream);

/*
 * Converts a whole fp16 buffer to E4M3 codes element by element with the
 * rule of pa_reshape_and_cache_fp8 (code = E4M3(fl32(x / scale))), keeping
 * the layout: turns an fp16 cache into the equivalent FP8 cache.
 *
 *   src            fp16 [num_elems]
 *   dst            uint8 [num_elems] (written); must not overlap src
 *   num_elems      a multiple of 16 (PA_ERR_INVALID_ARG otherwise)
 */
pa_status pa_convert_cache_fp8(const void* src, void* dst, size_t num_elems, float scale,
                               pa_stream_t stream);

/* Copy-on-write block copy for FP8 caches: pa_copy_blocks on uint8 caches. */
pa_status pa_copy_blocks_fp8(void* const* key_caches, void* const* value_caches, int num_layers,
                             const int64_t* block_mapping, int num_pairs, int num_heads,
                             int head_dim, int block_size, int num_blocks, pa_stream_t stream);

/*
 * Slot map [P2 §2.3 address map; P1 §3.2 worked block-table example]: for
 * token t of sequence s = token_seq[t] at logical position pos = token_pos[t],
 *
 *   slot_mapping[t] = block_tables[s][pos / block_size] * block_size + pos % block_size
 *
 * token_seq[t] < 0 marks a padding token and yields -1.  A sequence outside
 * [0, num_seqs), a position outside the table, or a table entry outside
 * [0, num_blocks) yields -1 and sets PA_ERRBIT_TOKEN.
 *
 *   slot_mapping   int64 [num_tokens] (written)
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]
 *   token_seq,
 *   token_pos      int32 [num_tokens]
 */
pa_status pa_slot_mapping(int64_t* slot_mapping, const int32_t* block_tables,
                          int max_blocks_per_seq, const int32_t* token_seq,
                          const int32_t* token_pos, int num_tokens, int num_seqs, int block_size,
                          int num_blocks, pa_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the calling device's error
 * word.  Returns PA_ERR_CUDA if a CUDA error is pending, PA_ERR_TIMEOUT if
 * the timeout bit is set, PA_ERR_OUT_OF_RANGE if any other bit is set, else
 * PA_OK.  If error_bits is not NULL it receives the word (0 when clean).
 */
pa_status pa_check_errors(pa_stream_t stream, uint32_t* error_bits);

/*
 * Self-test of the library's stall handling.  Every wait of a library kernel
 * on its own asynchronous copies is bounded: after about one second it gives
 * up, the kernel finishes the work it can, sets PA_ERRBIT_TIMEOUT in the
 * device error word and returns, so a stalled pipeline ends as a reported
 * status instead of a hung GPU.  This call launches one thread that waits,
 * through that same bounded wait, on a shared-memory barrier that never
 * completes (it expects two arrivals and receives one); about one second
 * later the wait gives up and the timeout bit is set.  The next
 * pa_check_errors returns PA_ERR_TIMEOUT with error_bits ==
 * PA_ERRBIT_TIMEOUT (and clears the word); the context stays usable.
 * Asynchronous on `stream`; returns PA_ERR_CUDA if the launch fails.
 */
pa_status pa_selftest_wait_timeout(pa_stream_t stream);

/* A static, human-readable name of a status. */
const char* pa_status_string(pa_status status);

/*
 * Tokens per context partition pa_decode will use for this shape (a
 * multiple of 32): 256 when num_seqs * num_heads * ceil(max_context_len /
 * 512) < 4096 (small batches, which would otherwise end on a tail of their
 * last items), else 512; the override below wins.  A pure function of the
 * arguments.  Exposed so callers can reason about workspace use; 0 on
 * invalid arguments.
 */
int pa_decode_partition_tokens(int num_seqs, int num_heads, int max_context_len);

/*
 * Process-wide override of the partition size used by pa_decode and
 * pa_decode_workspace_size (rounded up to a multiple of 32; 0 restores the
 * automatic choice).  Meant for tuning and for tests that force many
 * partitions on small inputs.  Not thread-safe with concurrent decodes.
 */
void pa_decode_set_partition_tokens(int tokens);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
