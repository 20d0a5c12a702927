// Paged decode attention for sm_103a: partition pass + log-sum-exp merge.
//
// What is computed ("vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量"
// §2.1 and §2.3): for each sequence s and head h,
//   out = softmax(scale * q . K_paged^T) V_paged,
//   K_paged[i] = key_cache[block_tables[s][i / B]][h][i % B]   (same for V).
//
// Design (GB300):
//  * Work items are (sequence, head, context partition) triples of at most
//    `part_tokens` tokens, numbered sequence-major, then partition, then
//    head.  A persistent grid of CTAs (resident CTAs per SM x SM count) takes
//    items from an atomic counter, so skewed batches balance to within one
//    item and no CTA is launched for an empty partition.  Handing items out
//    in this order keeps the CTAs running at any moment on the same few
//    sequences and partitions, so they read the head tiles of the same
//    physical blocks (one contiguous region per block in the [NB][H][B][D]
//    layout) at about the same time.  (A balanced static split of the
//    batch's token space over the CTAs, which removes the tail of the last
//    items, was built and measured slower: each CTA then streams its own
//    region of the batch, HBM sees scattered 4-8 KB tiles instead of
//    contiguous blocks, and the long-context batch fell from 6.9 to
//    5.9 TB/s.)
//  * Each CTA has NW warps.  A partition is cut into chunks of TC tokens
//    (TC = min(B, 16)) lying inside one physical block; chunk j goes to warp
//    j mod NW.  Each warp runs its own ring of NST shared-memory stages: lane
//    0 issues two 1-D bulk copies per chunk (the K rows and the V rows of one
//    (block, head) tile, contiguous in the [NB][H][B][D] layout) completing on
//    the stage's mbarrier; only the live rows of a ragged last chunk are
//    copied.  A warp's chunk stream runs across items: as soon as a stage is
//    free and the current item has no chunk left for the warp, lane 0 issues
//    the warp's first chunks of the next item, so copies stay in flight
//    through the end-of-item barrier and merge.
//  * The partition's block-table slice sits in shared memory; the next
//    item's slice is prefetched with cp.async while the current item runs
//    (the few entries needed to start the next item early are loaded into
//    registers by lane 0).
//  * Inside a warp each lane owns 8 dimensions (16 bytes) of a token row;
//    D/8 lanes cover one row.  q.k uses fp16 x fp16 -> fp32 fused
//    multiply-adds; the per-lane partial dots are combined by a shuffle
//    reduce-scatter, after which each lane holds one token's logit.  The
//    online softmax keeps (m, l) in fp32 in base-2 units (logits are scaled
//    by scale*log2(e) and exponentiated with ex2), with shuffle max/sum
//    reductions.  p.V accumulates in fp32, 8 dimensions per lane.
//  * At the end of an item the warps' (m, l, o) merge in shared memory.  A
//    sequence with one partition writes fp16 output directly; otherwise the
//    partition's (m, l, o) go to the workspace and a second kernel merges the
//    partitions (log-sum-exp weights), one warp per (sequence, head).  Two
//    in-kernel merges were built and measured slower: merging item by item
//    (a GPU-scope fence and an arrival atomic after every partition stall all
//    four warps), and deferring each CTA's merges to when it runs out of work
//    (the pending merges form a serial latency chain in the kernel's tail).
//  * The summation order depends only on logical token positions, so the
//    result is bit-identical under any relabelling of physical blocks.
//  * Cache write fused in (key_new set): the new token of each sequence sits
//    at position c - 1, in the last chunk of its last partition.  The warp
//    that owns that chunk, once the chunk has landed, writes the new key and
//    value rows (quantised for FP8 caches, as the cache-write kernel does)
//    to the cache and over the stale rows of its stage, then proceeds: the
//    same result and cache contents as the cache write followed by decode,
//    in one kernel.
//  * FP8 caches (F8: one E4M3 byte per element, one scale per cache tensor)
//    read a token's row in half the bytes, so per byte of HBM the kernel
//    does twice the arithmetic; the fp16 layout above is then bound by
//    instruction issue, not by HBM.  The FP8 layout cuts the instructions
//    per token: a lane owns 16 dimensions (16 codes = 16 bytes), a chunk is
//    16 tokens (it spans 16/B physical blocks when B < 16, one bulk copy per
//    block for K and for V), codes are widened to fp16 pairs in registers
//    (exact), and p.V runs as fp16 x fp16 -> fp32 fused multiply-adds with
//    the softmax weights rounded to fp16 (relative error <= 2^-11 per
//    weight; the denominator sums the same rounded weights).  The key scale is folded
//    into the logit scale and the value scale multiplies the CTA's merged
//    output.
#pragma once

#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.cuh"

namespace pa {

template <int D, int B, bool F8 = false>
struct DecodeTraits {
  static constexpr int NW = 4;                // warps per CTA
  // Stages per warp.  Two stages instead of three leave room for more
  // resident CTAs (fp16: 3 per SM instead of 2, by shared memory; FP8: 5
  // instead of 4, with the register budget below) at the same bytes in
  // flight per SM, and more warps hide more latency.
  static constexpr int NST = 2;
  static constexpr int THREADS = NW * 32;
  // Tokens per chunk: fp16 chunks lie inside one block; FP8 chunks are 16
  // tokens and span BPC = 16 / B blocks when B < 16 (partitions are
  // multiples of 32 tokens, so a chunk never straddles a partition).
  static constexpr int TC = F8 ? 16 : (B < 16 ? B : 16);
  static constexpr int BPC = TC > B ? TC / B : 1;  // blocks per chunk
  static constexpr int DPL = F8 ? 16 : 8;     // dimensions per lane (16 bytes either way)
  static constexpr int LR = D / DPL;          // lanes per token row
  static constexpr int RI = 32 / LR;          // token rows per warp-wide load
  static constexpr int TPL = TC / RI;         // token rows per lane
  static constexpr int DUP = LR / TPL;        // lanes sharing a logit after the reduction
  static constexpr int ELEM = F8 ? 1 : 2;    // bytes per cache element
  static constexpr int CHUNK_ELEMS = TC * D;
  static constexpr int CHUNK_BYTES = CHUNK_ELEMS * ELEM;
  static constexpr int STAGE_BYTES = 2 * CHUNK_BYTES;  // K rows then V rows
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(TPL >= 1 && TPL <= LR && (TPL & (TPL - 1)) == 0, "lane layout");
  static_assert(NST == 2 || NST == 3, "stage ring");

  // Fixed part of the dynamic shared memory (bytes), in layout order.
  static constexpr size_t kStages = size_t(NW) * NST * STAGE_BYTES;
  static constexpr size_t kBars = size_t(NW) * NST * 8;
  static constexpr size_t kP = size_t(NW) * TC * 4;  // softmax weights (fp32, or fp16 for F8)
  static constexpr int MS = D + 4;            // merge stride (floats): o[D], m, l, pad
  static constexpr size_t kMerge = 2 * size_t(NW) * MS * 4;
  static constexpr size_t kMisc = 16 * 4;     // item ring, warp sums, flags
  static constexpr size_t kFixed = kStages + kBars + kP + kMerge + kMisc;
};

// Effective context length: clipped to what the table and the launch cover.
__device__ __forceinline__ int effective_len(int c, const DecodeParams& a, int B, bool report) {
  int e = 0;
  if (c < 0) { c = 0; e = 1; }
  const long long cap_table = (long long)a.max_blocks * B;
  if (c > cap_table) { c = (int)cap_table; e = 1; }
  if (c > a.max_context_len) { c = a.max_context_len; e = 1; }
  if (report && e) atomicOr(a.err, PA_ERRBIT_CONTEXT);
  return c;
}

__device__ __forceinline__ int num_parts(int c, int part_tokens) {
  return c > 0 ? (c + part_tokens - 1) / part_tokens : 1;  // an empty sequence is one item
}

struct ItemInfo {
  int s;        // sequence within the launch
  int h;
  int p;        // partition
  int c;        // effective context length
  int t_begin, t_end;
  int n_parts;
  int blk0;     // first logical block of the partition
  int nblk;     // logical blocks it touches
};

template <int B>
__device__ __forceinline__ ItemInfo locate_item(int item, const int* cum, const int* ctx_s,
                                                int nseq, int H, int part_tokens) {
  int lo = 0, hi = nseq - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cum[mid] <= item) lo = mid; else hi = mid - 1;
  }
  ItemInfo it;
  it.s = lo;
  it.c = ctx_s[lo];
  it.n_parts = num_parts(it.c, part_tokens);
  const int within = item - cum[lo];
  it.p = within / H;  // head-innermost: concurrent CTAs read the same physical blocks
  it.h = within - it.p * H;
  it.t_begin = it.p * part_tokens;
  it.t_end = min(it.c, it.t_begin + part_tokens);
  it.blk0 = it.t_begin / B;
  it.nblk = it.t_end > it.t_begin ? (it.t_end - 1) / B - it.blk0 + 1 : 0;
  return it;
}

// Chunks of an item that warp `warp` processes (chunks warp, warp+NW, ...).
template <int D, int B, bool F8>
__device__ __forceinline__ int warp_chunks(const ItemInfo& it, int warp) {
  using T = DecodeTraits<D, B, F8>;
  const int n = (it.t_end - it.t_begin + T::TC - 1) / T::TC;
  return warp < n ? (n - 1 - warp) / T::NW + 1 : 0;
}

// Physical ids of the blocks of chunk `chunk` of an item, from the item's
// block-table slice in shared memory (-1 for blocks past the live rows).
template <int D, int B, bool F8>
__device__ __forceinline__ void chunk_ids(int (&phys)[DecodeTraits<D, B, F8>::BPC], const int* bt,
                                          const ItemInfo& it, int chunk) {
  using T = DecodeTraits<D, B, F8>;
  const int t0 = it.t_begin + chunk * T::TC;
#pragma unroll
  for (int b = 0; b < T::BPC; ++b) phys[b] = t0 + b * B < it.t_end ? bt[t0 / B + b - it.blk0] : -1;
}

// True when every block of the chunk that holds live rows has a valid id.
template <int D, int B, bool F8>
__device__ __forceinline__ bool chunk_ids_ok(const DecodeParams& a, const int (&phys)[DecodeTraits<D, B, F8>::BPC],
                                             int rows) {
  bool ok = true;
#pragma unroll
  for (int b = 0; b < DecodeTraits<D, B, F8>::BPC; ++b)
    if (b * B < rows && (phys[b] < 0 || phys[b] >= a.num_blocks)) ok = false;
  return ok;
}

// Issues the bulk copies of one chunk into a stage: for each block of the
// chunk with live rows, its K rows and its V rows (contiguous in the
// [NB][H][B][D] layout); only live rows are copied.  kn, vn (fp16 caches with
// the cache write fused in, for the chunk holding a sequence's new token;
// null otherwise): the chunk's last row comes from these new rows instead of
// the cache, which does not hold them yet.  Warp-uniform: every lane executes
// it with the same operands and only `leader` issues.
template <int D, int B, bool F8>
__device__ __forceinline__ void issue_chunk(const DecodeParams& a, const ItemInfo& it,
                                            const int (&phys)[DecodeTraits<D, B, F8>::BPC],
                                            int chunk, uint32_t stage, uint32_t bar,
                                            uint64_t policy, bool leader,
                                            const void* kn = nullptr, const void* vn = nullptr) {
  using T = DecodeTraits<D, B, F8>;
  const int t0 = it.t_begin + chunk * T::TC;
  const int rows = min(T::TC, it.t_end - t0);
  if (rows <= 0) {  // not a chunk of this item (cannot happen): complete the phase empty
    mbar_arrive_if(leader, bar);
    return;
  }
  if (!chunk_ids_ok<D, B, F8>(a, phys, rows)) {
    if (leader) atomicOr(a.err, PA_ERRBIT_BLOCK_ID);
    mbar_arrive_if(leader, bar);  // completes the phase with no data; the chunk is skipped
    return;
  }
  mbar_arrive_expect_tx_if(leader, bar, 2u * (uint32_t)rows * D * T::ELEM);
  const int crows = kn != nullptr ? rows - 1 : rows;  // rows that come from the cache
  if (kn != nullptr) {
    const uint32_t soff = (uint32_t)(rows - 1) * D * T::ELEM;
    bulk_g2s_hint_if(leader, stage + soff, kn, D * T::ELEM, bar, policy);
    bulk_g2s_hint_if(leader, stage + T::CHUNK_BYTES + soff, vn, D * T::ELEM, bar, policy);
  }
  // Byte offset of (block 0, head h, row t0 % B) and the stride between blocks.
  const size_t head_off = ((size_t)it.h * B + (t0 % B)) * D * T::ELEM;
  const size_t blk_stride = (size_t)a.num_heads * B * D * T::ELEM;
#pragma unroll
  for (int b = 0; b < T::BPC; ++b) {
    const int r = min(B, crows - b * B);
    if (r <= 0) break;
    const size_t off = (size_t)phys[b] * blk_stride + head_off;
    const uint32_t bytes = (uint32_t)r * D * T::ELEM;
    const uint32_t soff = b * B * D * T::ELEM;
    bulk_g2s_hint_if(leader, stage + soff, static_cast<const unsigned char*>(a.key_cache) + off,
                     bytes, bar, policy);
    bulk_g2s_hint_if(leader, stage + T::CHUNK_BYTES + soff,
                     static_cast<const unsigned char*>(a.value_cache) + off, bytes, bar, policy);
  }
}

// The fused cache write of one sequence's new token (warp-wide; call only
// for the chunk that holds position pos = c - 1).  Lanes 0..15 carry the new
// key row and lanes 16..31 the value row of (sequence, head h), 16 bytes of
// fp16 each (lanes whose index within the half is >= D/8 carry nothing): w
// is that piece, or for FP8 caches its 8 E4M3 codes in w.x, w.y (quantised
// as the cache-write kernel quantises them).  The piece goes to the cache
// slot of pos; for FP8 caches also over the chunk's staged row `row` (K rows
// at Ks, V rows at Vs), which the bulk copy filled with the slot's old codes
// (for fp16 caches the copy already took that row from the new rows).
template <int D, int B, bool F8>
__device__ __forceinline__ void append_new_token(const DecodeParams& a, int h, int phys, int pos,
                                                 int row, unsigned char* Ks, unsigned char* Vs,
                                                 int lane, const uint4& w) {
  using T = DecodeTraits<D, B, F8>;
  constexpr int PIECE = 8 * T::ELEM;  // bytes of one lane's piece in the cache
  const bool is_v = lane >= 16;
  const int idx = lane & 15;
  const size_t dst = (((size_t)phys * a.num_heads + h) * B + pos % B) * D * T::ELEM +
                     (size_t)idx * PIECE;  // bytes
  unsigned char* c = static_cast<unsigned char*>(const_cast<void*>(is_v ? a.value_cache : a.key_cache));
  unsigned char* st = (is_v ? Vs : Ks) + (size_t)row * D * T::ELEM + idx * PIECE;
  // The staged row first, then the fence that keeps the next bulk copy into
  // this stage from overtaking it; the cache store goes last, so the fence
  // does not wait for it.
  if constexpr (F8) {
    if (idx < D / 8) *reinterpret_cast<uint2*>(st) = make_uint2(w.x, w.y);
    fence_proxy_async_smem();
    __syncwarp();
  }
  if (idx < D / 8) {
    if constexpr (F8)
      *reinterpret_cast<uint2*>(c + dst) = make_uint2(w.x, w.y);
    else
      *reinterpret_cast<uint4*>(c + dst) = w;
  }
}

// A lane's query slice: DPL fp16 values (16 or 32 bytes).
template <int DPL>
struct QSlice {
  uint4 v[DPL / 8];
};

// Partial dot of the lane's query slice with its slice of cache row t.
template <int D, bool F8>
__device__ __forceinline__ float row_dot(const QSlice<F8 ? 16 : 8>& q, const unsigned char* rows,
                                         int t, int cidx) {
  if constexpr (F8) {
    const uint4 c = lds128(rows + t * D + 16 * cidx);
    const float a = dot8_f16(q.v[0], e4m3x8_to_f16x8(make_uint2(c.x, c.y)));
    return a + dot8_f16(q.v[1], e4m3x8_to_f16x8(make_uint2(c.z, c.w)));
  } else {
    return dot8_f16(q.v[0], lds128(rows + (t * D + 8 * cidx) * 2));
  }
}

// One chunk for one warp: logits, online-softmax update, p.V accumulation.
template <int D, int B, bool F8, bool FULL>
__device__ __forceinline__ void process_chunk(const unsigned char* Ks, const unsigned char* Vs,
                                              int rows, const QSlice<DecodeTraits<D, B, F8>::DPL>& q,
                                              float scale_log2, float* p_w, int lane, float& m,
                                              float& l, float (&o)[DecodeTraits<D, B, F8>::DPL]) {
  using T = DecodeTraits<D, B, F8>;
  const int cidx = lane % T::LR;  // which DPL dimensions
  const int r = lane / T::LR;     // which row group

  // Partial dots over this lane's dimensions for its TPL rows.
  float v[T::TPL];
#pragma unroll
  for (int k = 0; k < T::TPL; ++k) v[k] = row_dot<D, F8>(q, Ks, r + T::RI * k, cidx);
  // Reduce-scatter over the LR lanes of the row group: at each halving step a
  // lane keeps one half of its values and adds its partner's copy of it.
#pragma unroll
  for (int cnt = T::TPL, msk = T::LR / 2; cnt > 1; cnt >>= 1, msk >>= 1) {
    const bool upper = (lane & msk) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float send = upper ? v[i] : v[i + cnt / 2];
      const float keep = upper ? v[i + cnt / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, msk);
    }
  }
#pragma unroll
  for (int msk = T::DUP / 2; msk >= 1; msk >>= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], msk);
  const int kl = cidx / T::DUP;          // this lane's logit: row r + RI*kl
  const int tl = r + T::RI * kl;
  float x = v[0] * scale_log2;
  if (!FULL && tl >= rows) x = -INFINITY;

  float cm = x;
#pragma unroll
  for (int msk = T::DUP; msk < 32; msk <<= 1) cm = fmaxf(cm, __shfl_xor_sync(kFullMask, cm, msk));
  const float m_new = fmaxf(m, cm);
  const float alpha = exp2_approx(m - m_new);  // 0 on the first chunk (m = -inf)
  float pv = exp2_approx(x - m_new);           // 0 for masked rows
  if constexpr (F8) {
    // The weight p.V uses, rounded to fp16; the denominator sums the same value.
    const __half ph = __float2half_rn(pv);
    pv = __half2float(ph);
    if ((cidx % T::DUP) == 0)
      reinterpret_cast<__half*>(p_w)[r * T::TPL + kl] = ph;
  } else {
    if ((cidx % T::DUP) == 0) p_w[r * T::TPL + kl] = pv;
  }
  float ps = pv;
#pragma unroll
  for (int msk = T::DUP; msk < 32; msk <<= 1) ps += __shfl_xor_sync(kFullMask, ps, msk);
  l = l * alpha + ps;
  m = m_new;
  __syncwarp();
  if (alpha != 1.f) {  // warp-uniform; skipping a multiply by 1 changes no bit
#pragma unroll
    for (int i = 0; i < T::DPL; ++i) o[i] *= alpha;
  }

  if constexpr (F8) {
    // The row group's TPL fp16 weights, contiguous in shared memory.
    static_assert(T::TPL == 2 || T::TPL == 4 || T::TPL == 8, "FP8 weight load");
    uint32_t pk[T::TPL / 2];
    const __half* pw = reinterpret_cast<const __half*>(p_w) + r * T::TPL;
    if constexpr (T::TPL == 8) {
      const uint4 w4 = lds128(pw);
      pk[0] = w4.x;
      pk[1] = w4.y;
      pk[2] = w4.z;
      pk[3] = w4.w;
    } else if constexpr (T::TPL == 4) {
      const uint2 w2 = lds64(pw);
      pk[0] = w2.x;
      pk[1] = w2.y;
    } else {
      pk[0] = *reinterpret_cast<const uint32_t*>(pw);
    }
#pragma unroll
    for (int k = 0; k < T::TPL; ++k) {
      const int t = r + T::RI * k;
      if (FULL || t < rows) {
        const uint16_t p16 = (uint16_t)(pk[k / 2] >> (16 * (k & 1)));
        const uint4 c = lds128(Vs + t * D + 16 * cidx);
        const uint4 h0 = e4m3x8_to_f16x8(make_uint2(c.x, c.y));
        const uint4 h1 = e4m3x8_to_f16x8(make_uint2(c.z, c.w));
        const uint32_t w[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) fma2_f16_f32(p16, w[j], o[2 * j], o[2 * j + 1]);
      }
    }
  } else {
    float pk[T::TPL];
#pragma unroll
    for (int k = 0; k < T::TPL; ++k) pk[k] = p_w[r * T::TPL + k];
#pragma unroll
    for (int k = 0; k < T::TPL; ++k) {
      const int t = r + T::RI * k;
      if (FULL || t < rows) {
        const uint4 vv = lds128(Vs + (t * D + 8 * cidx) * 2);
        const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = half2_bits_to_float2(w[j]);
          o[2 * j] = fmaf(pk[k], f.x, o[2 * j]);
          o[2 * j + 1] = fmaf(pk[k], f.y, o[2 * j + 1]);
        }
      }
    }
  }
}

// APPEND: the variant with the new token's cache write fused in (a separate
// instantiation, so the plain decode keeps its registers and schedule).
template <int D, int B, bool F8, bool APPEND>
__global__ void __launch_bounds__(DecodeTraits<D, B, F8>::THREADS, F8 ? 5 : 1)
    decode_partition_kernel(const DecodeParams a) {
  using T = DecodeTraits<D, B, F8>;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* cur_ptr = smem;
  unsigned char* stages = cur_ptr;
  cur_ptr += T::kStages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(cur_ptr);
  cur_ptr += T::kBars;
  float* p_s = reinterpret_cast<float*>(cur_ptr);
  cur_ptr += T::kP;
  float* merge = reinterpret_cast<float*>(cur_ptr);
  cur_ptr += T::kMerge;
  // misc: [1..3] item ring, [4..7] warp sums, [8] failure flag
  int* misc = reinterpret_cast<int*>(cur_ptr);
  cur_ptr += T::kMisc;
  const int bt_cap = a.part_tokens / B + 1;
  int* bt_s = reinterpret_cast<int*>(cur_ptr);  // 2 x bt_cap
  cur_ptr += 2 * bt_cap * 4;
  int* cum = reinterpret_cast<int*>(cur_ptr);   // nseq + 1
  int* ctx_s = cum + (a.num_seqs + 1);          // nseq
  // nseq flags: the sequence's context length was clipped (APPEND: no write)
  unsigned char* clip_s = reinterpret_cast<unsigned char*>(ctx_s + a.num_seqs);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nseq = a.num_seqs;
  const int H = a.num_heads;
  const int P = a.part_tokens;

  if (lane == 0) {
    for (int j = 0; j < T::NST; ++j) mbar_init(smem_u32(&bars[warp * T::NST + j]), 1);
  }
  if (tid == 0) misc[8] = 0;
  fence_mbar_init();
  // A launch may start while the kernel before it on the stream still runs
  // (programmatic launch).  The call's inputs (context lengths, block tables,
  // queries, caches) may come from that kernel (a cache write, say), so the
  // first kernel of a call waits before it reads them.  When an earlier
  // kernel of the same call has waited already (the counter-zeroing kernel,
  // or the previous launch of a split batch), it triggered this launch only
  // after its wait: the inputs are complete here, and the scan, the first
  // item's block-table slice and its first copies run before pdl_wait, over
  // the previous kernel's tail.  The work counter and the workspace partials
  // are touched only after the wait.
  if (!a.inputs_ready) pdl_wait();

  // ---- per-sequence item counts and their exclusive prefix sums ---------
  {
    constexpr int PER = (kMaxSeqsPerLaunch + T::THREADS - 1) / T::THREADS;
    int vals[PER];
    int local = 0;
    const int base = tid * PER;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = base + j;
      int v = 0;
      if (i < nseq) {
        const int raw = a.context_lens[a.seq_begin + i];
        const int c = effective_len(raw, a, B, blockIdx.x == 0);
        ctx_s[i] = c;
        if constexpr (APPEND) clip_s[i] = raw != c;
        v = H * num_parts(c, P);
      }
      vals[j] = v;
      local += v;
    }
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullMask, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) misc[4 + warp] = x;
    __syncthreads();
    int run = x - local;
    for (int w = 0; w < warp; ++w) run += misc[4 + w];
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int i = base + j;
      if (i < nseq) {
        cum[i] = run;
        run += vals[j];
        if (i == nseq - 1) cum[nseq] = run;
      }
    }
  }
  __syncthreads();
  const int total = cum[nseq];
  // Item blockIdx.x is this CTA's first; later items come from the counter,
  // numbered from gridDim.x on.
  int cur = blockIdx.x;
  if (cur >= total) return;

  // First item's block-table slice (synchronous).
  ItemInfo it = locate_item<B>(cur, cum, ctx_s, nseq, H, P);
  {
    const int32_t* row = a.block_tables + (size_t)(a.seq_begin + it.s) * a.max_blocks;
    for (int i = tid; i < it.nblk; i += T::THREADS) bt_s[i] = row[it.blk0 + i];
  }
  __syncthreads();

  const uint64_t policy = policy_evict_first();
  unsigned char* my_stages = stages + (size_t)warp * T::NST * T::STAGE_BYTES;
  uint64_t* my_bars = bars + warp * T::NST;
  float* my_p = p_s + warp * T::TC;
  const int cidx = lane % T::LR;
  const int rgrp = lane / T::LR;
  // Per-warp running chunk counts across items (warp-uniform): consumed and
  // issued.  Chunk g of the warp's stream lives in stage g % NST and is the
  // (g / NST)-th use of that stage's barrier.
  uint32_t u = 0, iss = 0;
  int buf = 0;
  int iter = 0;

  const bool leader = lane == 0;
  const uint32_t my_stages_s = smem_u32(my_stages);
  const uint32_t my_bars_s = smem_u32(my_bars);
  // fp16 caches with the cache write fused in: the new K and V rows that
  // replace the last row of the chunk holding c - 1 in an item's last
  // partition (null for every other chunk, and for clipped contexts).
  auto new_rows = [&](const ItemInfo& x, int chunk, const void*& kn, const void*& vn) {
    kn = vn = nullptr;
    if constexpr (APPEND && !F8) {
      if (x.t_end == x.c && x.c > 0 && !clip_s[x.s] && chunk == (x.c - 1 - x.t_begin) / T::TC) {
        const size_t off = ((size_t)(a.seq_begin + x.s) * H + x.h) * D;
        kn = static_cast<const __half*>(a.key_new) + off;
        vn = static_cast<const __half*>(a.value_new) + off;
      }
    }
  };
  // The first item's first copies, still before the wait (warp-uniform; the
  // leader issues).
  {
    const int n0 = warp_chunks<D, B, F8>(it, warp);
    for (; (int)iss < n0 && iss < (uint32_t)T::NST; ++iss) {
      const int chunk = warp + (int)iss * T::NW;
      int ph[T::BPC];
      chunk_ids<D, B, F8>(ph, bt_s, it, chunk);
      const void *kn, *vn;
      new_rows(it, chunk, kn, vn);
      issue_chunk<D, B, F8>(a, it, ph, chunk, my_stages_s + iss * T::STAGE_BYTES,
                            my_bars_s + 8 * iss, policy, leader, kn, vn);
    }
  }
  // Stage of the next issue and of the next consumption (with its phase).
  int st_i = (int)iss % T::NST, st_c = 0;
  uint32_t ph_c = 0;
  pdl_wait();
  pdl_launch_dependents();
  // Fetches from the work counter.  Every CTA with a first item fetches once
  // before its loop and once per item it runs, so a launch makes exactly
  // min(grid, total) + total fetches; the one that gets the last value puts
  // the counter back to zero for the next call.
  const unsigned last_fetch = (unsigned)(min((int)gridDim.x, total) + total - 1);
  auto fetch = [&]() {
    const unsigned v = atomicAdd(a.counter, 1u);
    if (v == last_fetch) atomicExch(a.counter, 0u);
    return (int)(gridDim.x + v);
  };
  if (tid == 0) misc[1] = fetch();
  __syncthreads();
  int nxt = misc[1];

  while (true) {
    const bool has_next = nxt < total;
    ItemInfo nx;
    nx.t_begin = nx.t_end = 0;
    if (has_next) {
      nx = locate_item<B>(nxt, cum, ctx_s, nseq, H, P);
      const int32_t* row = a.block_tables + (size_t)(a.seq_begin + nx.s) * a.max_blocks;
      int* dst = bt_s + (buf ^ 1) * bt_cap;
      for (int i = tid; i < nx.nblk; i += T::THREADS) cp_async_4(dst + i, row + nx.blk0 + i);
    }
    cp_async_commit();
    if (tid == 0) misc[2 + (iter & 1)] = fetch();

    const int* bt = bt_s + buf * bt_cap;
    const size_t sh = (size_t)(a.seq_begin + it.s) * H + it.h;
    const int n_my = warp_chunks<D, B, F8>(it, warp);
    const int n_nx = has_next ? warp_chunks<D, B, F8>(nx, warp) : 0;
    const uint32_t base = u;

    // Block ids of this warp's first NST chunks of the next item (every lane
    // loads the same ids: the issue code is warp-uniform).
    int nxp[T::NST][T::BPC];
#pragma unroll
    for (int j = 0; j < T::NST; ++j)
#pragma unroll
      for (int b = 0; b < T::BPC; ++b) nxp[j][b] = -1;
    if (n_nx > 0) {
      const int32_t* row = a.block_tables + (size_t)(a.seq_begin + nx.s) * a.max_blocks;
#pragma unroll
      for (int j = 0; j < T::NST; ++j) {
        const int t0 = nx.t_begin + (warp + j * T::NW) * T::TC;
#pragma unroll
        for (int b = 0; b < T::BPC; ++b)
          if (j < n_nx && t0 + b * B < nx.t_end) nxp[j][b] = row[t0 / B + b];
      }
    }
    // Fill free stages: the rest of this item's chunks, then the next item's
    // (warp-uniform; the leader issues).
    auto issue_upto = [&]() {
      while (iss < u + T::NST) {
        const int k = (int)(iss - base);
        const uint32_t stage = my_stages_s + st_i * T::STAGE_BYTES;
        const uint32_t bar = my_bars_s + 8 * st_i;
        if (k < n_my) {
          const int chunk = warp + k * T::NW;
          int ph[T::BPC];
          chunk_ids<D, B, F8>(ph, bt, it, chunk);
          const void *kn, *vn;
          new_rows(it, chunk, kn, vn);
          issue_chunk<D, B, F8>(a, it, ph, chunk, stage, bar, policy, leader, kn, vn);
        } else if (k - n_my < n_nx) {
          const int j = k - n_my;
          int ph[T::BPC];
#pragma unroll
          for (int b = 0; b < T::BPC; ++b) {  // j < NST: a register select, no local memory
            int v = nxp[0][b];
#pragma unroll
            for (int jj = 1; jj < T::NST; ++jj)
              if (j == jj) v = nxp[jj][b];
            ph[b] = v;
          }
          const void *kn, *vn;
          new_rows(nx, warp + j * T::NW, kn, vn);
          issue_chunk<D, B, F8>(a, nx, ph, warp + j * T::NW, stage, bar, policy, leader, kn, vn);
        } else {
          break;
        }
        ++iss;
        st_i = st_i + 1 == T::NST ? 0 : st_i + 1;
      }
    };
    issue_upto();

    QSlice<T::DPL> q;
#pragma unroll
    for (int j = 0; j < T::DPL / 8; ++j)
      q.v[j] = *reinterpret_cast<const uint4*>(static_cast<const __half*>(a.query) + sh * D +
                                               T::DPL * cidx + 8 * j);
    float m = -INFINITY, l = 0.f;
    float o[T::DPL];
#pragma unroll
    for (int i = 0; i < T::DPL; ++i) o[i] = 0.f;
    // APPEND: the last item of a (sequence, head) holds its new token in
    // chunk a_chunk; the warp that owns that chunk loads the new rows now
    // (lanes 0..15 the key row, 16..31 the value row), so the loads are long
    // done when the chunk lands.
    int a_chunk = -1;
    uint4 a_w = make_uint4(0, 0, 0, 0);
    if constexpr (APPEND) {
      if (it.t_end == it.c && it.c > 0 && !clip_s[it.s] &&
          ((it.c - 1 - it.t_begin) / T::TC) % T::NW == warp) {
        a_chunk = (it.c - 1 - it.t_begin) / T::TC;
        const __half* row = static_cast<const __half*>(lane >= 16 ? a.value_new : a.key_new) + sh * D;
        if ((lane & 15) < D / 8) a_w = reinterpret_cast<const uint4*>(row)[lane & 15];
      }
    }

    for (int i = 0; i < n_my; ++i) {
      const int st = st_c;
      const uint32_t bar = my_bars_s + 8 * st;
      const int chunk = warp + i * T::NW;
      // FP8: the new rows' codes are made while this chunk's copy is still in
      // flight (eight IEEE divisions per lane).
      if constexpr (APPEND && F8) {
        if (chunk == a_chunk) {
          const uint2 q = quantize8(a_w, lane >= 16 ? a.v_scale : a.k_scale);
          a_w.x = q.x;
          a_w.y = q.y;
        }
      }
      bool ok = mbar_wait_bounded(bar, ph_c);
      ok = __all_sync(kFullMask, ok);
      if (!ok) {
        // Drain this warp's copies still in flight (bounded), then give up.
        for (uint32_t g = u + 1; g < iss; ++g)
          mbar_wait_bounded(smem_u32(&my_bars[g % T::NST]), (g / T::NST) & 1);
        u = iss;
        if (lane == 0) {
          atomicOr(a.err, PA_ERRBIT_TIMEOUT);
          misc[8] = 1;
        }
        break;
      }
      const int t0 = it.t_begin + chunk * T::TC;
      const int rows = min(T::TC, it.t_end - t0);
      int ph[T::BPC];
      chunk_ids<D, B, F8>(ph, bt, it, chunk);
      if (rows > 0 && chunk_ids_ok<D, B, F8>(a, ph, rows)) {
        unsigned char* Ks = my_stages + st * T::STAGE_BYTES;
        // Fused cache write: this chunk holds the sequence's new token (a
        // clipped context length was reported and writes nothing).
        if (APPEND && chunk == a_chunk) {
          const int row = it.c - 1 - t0;
          int phys = ph[0];  // the block of that row (a register select, no local memory)
#pragma unroll
          for (int b = 1; b < T::BPC; ++b)
            if (row / B == b) phys = ph[b];
          append_new_token<D, B, F8>(a, it.h, phys, it.c - 1, row, Ks, Ks + T::CHUNK_BYTES, lane,
                                     a_w);
        }
        if (rows == T::TC)
          process_chunk<D, B, F8, true>(Ks, Ks + T::CHUNK_BYTES, rows, q, a.scale_log2, my_p, lane,
                                        m, l, o);
        else
          process_chunk<D, B, F8, false>(Ks, Ks + T::CHUNK_BYTES, rows, q, a.scale_log2, my_p,
                                         lane, m, l, o);
      }
      __syncwarp();
      ++u;
      if (++st_c == T::NST) {
        st_c = 0;
        ph_c ^= 1;
      }
      issue_upto();
    }

    // Combine the row groups, then publish this warp's (m, l, o).
#pragma unroll
    for (int msk = T::LR; msk < 32; msk <<= 1) {
#pragma unroll
      for (int i = 0; i < T::DPL; ++i) o[i] += __shfl_xor_sync(kFullMask, o[i], msk);
    }
    float* mw = merge + (iter & 1) * T::NW * T::MS + warp * T::MS;
    if (rgrp == 0) {
#pragma unroll
      for (int i = 0; i < T::DPL / 4; ++i)
        reinterpret_cast<float4*>(mw + T::DPL * cidx)[i] =
            make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
    if (lane == 0) {
      mw[D] = m;
      mw[D + 1] = l;
    }
    cp_async_wait_all();
    __syncthreads();

    // Merge the warps of this item and write the output or the partial.
    const float* mb = merge + (iter & 1) * T::NW * T::MS;
    for (int d = tid; d < D; d += T::THREADS) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < T::NW; ++w) M = fmaxf(M, mb[w * T::MS + D]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < T::NW; ++w) {
        const float mwv = mb[w * T::MS + D];
        const float sc = (mwv == -INFINITY) ? 0.f : exp2_approx(mwv - M);
        L = fmaf(sc, mb[w * T::MS + D + 1], L);
        O = fmaf(sc, mb[w * T::MS + d], O);
      }
      if constexpr (F8) O *= a.v_scale;
      if (it.n_parts == 1) {
        const float r = (it.c > 0 && L > 0.f) ? O / L : 0.f;
        static_cast<__half*>(a.out)[sh * D + d] = __float2half_rn(r);
      } else {
        const size_t slot = sh * a.max_parts + it.p;
        a.ws_o[slot * D + d] = O;
        if (d == 0) {
          a.ws_ml[slot * 2] = M;
          a.ws_ml[slot * 2 + 1] = L;
        }
      }
    }
    if (misc[8] != 0 || !has_next) {
      // A CTA that gave up still makes the fetches it would have made (the
      // items it skips are lost and the call reports the timeout), so the
      // counter comes back to zero.
      if (misc[8] != 0 && tid == 0) {
        int n1 = nxt, n2 = misc[2 + (iter & 1)];
        while (n1 < total) {
          n1 = n2;
          n2 = fetch();
        }
      }
      // No copy of this warp may still be in flight when the CTA exits.
      for (uint32_t g = u; g < iss; ++g)
        mbar_wait_bounded(smem_u32(&my_bars[g % T::NST]), (g / T::NST) & 1);
      break;
    }
    cur = nxt;
    nxt = misc[2 + (iter & 1)];
    it = nx;
    buf ^= 1;
    ++iter;
  }
}

// Merge the partitions of each (sequence, head): one warp per pair.  The
// context length is read before pdl_wait (the partition launch before this
// one triggered it only after its own wait, so the call's inputs are
// complete); after the wait, the partitions' (m, l) and their first kPre partial
// outputs are loaded together, then the warp reduces max and sum by shuffles
// and accumulates the weighted partials in partition order, D/32 dimensions
// per lane.
template <int D, int B>
__global__ void __launch_bounds__(128) decode_reduce_kernel(const DecodeParams a, int total_seqs) {
  constexpr int DPL = D / 32;
  constexpr int kPre = 8;
  using Vec = typename std::conditional<DPL == 4, float4, float2>::type;
  const int lane = threadIdx.x & 31;
  const long long pair = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const bool live = pair < (long long)total_seqs * a.num_heads;
  int n = 0;
  if (live) n = num_parts(effective_len(a.context_lens[pair / a.num_heads], a, B, false), a.part_tokens);
  pdl_wait();
  pdl_launch_dependents();
  if (n <= 1) return;
  const float* ml = a.ws_ml + (size_t)pair * a.max_parts * 2;
  const float* ob = a.ws_o + (size_t)pair * a.max_parts * D + lane * DPL;
  float mp = -INFINITY, lp = 0.f;
  if (lane < n) {
    mp = ml[2 * lane];
    lp = ml[2 * lane + 1];
  }
  Vec pre[kPre];
#pragma unroll
  for (int j = 0; j < kPre; ++j)
    if (j < n) pre[j] = *reinterpret_cast<const Vec*>(ob + (size_t)j * D);
  float M = mp;
  for (int p = lane + 32; p < n; p += 32) M = fmaxf(M, ml[2 * p]);
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, msk));
  float L = (mp == -INFINITY) ? 0.f : exp2_approx(mp - M) * lp;
  for (int p = lane + 32; p < n; p += 32) {
    const float m2 = ml[2 * p];
    L += (m2 == -INFINITY ? 0.f : exp2_approx(m2 - M)) * ml[2 * p + 1];
  }
#pragma unroll
  for (int msk = 16; msk >= 1; msk >>= 1) L += __shfl_xor_sync(kFullMask, L, msk);
  float acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) acc[i] = 0.f;
  for (int p0 = 0; p0 < n; p0 += 32) {
    const int pl = p0 + lane;
    const float m2 = pl < n ? (p0 == 0 ? mp : ml[2 * pl]) : -INFINITY;
    const float wl = m2 == -INFINITY ? 0.f : exp2_approx(m2 - M);
    const int cnt = min(32, n - p0);
    for (int j = 0; j < cnt; ++j) {
      const float w = __shfl_sync(kFullMask, wl, j);
      const int p = p0 + j;
      Vec v = pre[0];  // a register select over pre[] (no local memory)
      if (p < kPre) {
#pragma unroll
        for (int k = 1; k < kPre; ++k)
          if (k == p) v = pre[k];
      } else {
        v = *reinterpret_cast<const Vec*>(ob + (size_t)p * D);
      }
      acc[0] = fmaf(w, v.x, acc[0]);
      acc[1] = fmaf(w, v.y, acc[1]);
      if constexpr (DPL == 4) {
        acc[2] = fmaf(w, reinterpret_cast<const float4&>(v).z, acc[2]);
        acc[3] = fmaf(w, reinterpret_cast<const float4&>(v).w, acc[3]);
      }
    }
  }
  __half* out = static_cast<__half*>(a.out) + (size_t)pair * D + lane * DPL;
#pragma unroll
  for (int i = 0; i < DPL; ++i) out[i] = __float2half_rn(L > 0.f ? acc[i] / L : 0.f);
}

template <int D, int B>
cudaError_t launch_reduce_t(const DecodeParams& p, int total_seqs, cudaStream_t st) {
  const long long warps = (long long)total_seqs * p.num_heads;
  const int blocks = (int)((warps + 3) / 4);
  return launch_pdl(decode_reduce_kernel<D, B>, dim3(blocks), dim3(128), 0, st, p, total_seqs);
}

template <int D, int B, bool F8>
cudaError_t launch_partition_t(const DecodeParams& p, int grid, size_t smem, cudaStream_t st) {
  if (p.key_new != nullptr)
    return launch_pdl(decode_partition_kernel<D, B, F8, true>, dim3(grid),
                      dim3(DecodeTraits<D, B, F8>::THREADS), smem, st, p);
  return launch_pdl(decode_partition_kernel<D, B, F8, false>, dim3(grid),
                    dim3(DecodeTraits<D, B, F8>::THREADS), smem, st, p);
}

template <int D, int B, bool F8>
int ctas_per_sm_t(size_t smem, bool append) {
  int n = 0;
  const cudaError_t e =
      append ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                   &n, decode_partition_kernel<D, B, F8, true>, DecodeTraits<D, B, F8>::THREADS, smem)
             : cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                   &n, decode_partition_kernel<D, B, F8, false>, DecodeTraits<D, B, F8>::THREADS,
                   smem);
  if (e != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

template <int D, int B, bool F8>
cudaError_t prepare_t() {
  const cudaError_t e = cudaFuncSetAttribute(decode_partition_kernel<D, B, F8, false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_partition_kernel<D, B, F8, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

}  // namespace pa
