// Multi-query paged attention (chunked prefill, mixed prefill + decode
// batches) on the sm_103a tensor cores.
//
// What is computed ("vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量"
// §4.3: prefill and decode share a batch; §2.1/§2.3: attention through the
// block table): sequence s brings q_len new tokens, the last q_len of its c
// cached tokens; new token j (position p = c - q_len + j) attends causally
//   out = softmax_{i <= p}(scale * q . K_i) V.
//
// Design (GB300):
//  * One CTA per (sequence, head, pair of 128-row query tiles), 12 warps:
//    two softmax warpgroups (one query row per thread) and a producer
//    warpgroup whose first warp issues the MMAs and second the TMA copies.
//    Q (128 x D per tile) and the paged K/V tiles (128 tokens = 128/B
//    blocks) arrive by TMA tensor copies with 128-byte swizzle, one box per
//    physical block, into two-stage rings; a block past the context is
//    fetched from an out-of-range coordinate (zero fill).
//  * One thread issues tcgen05.mma: S = Q K^T (M = 128 queries, N = 128
//    tokens, fp32 in TMEM columns [0, 128)), then O += P V (N = D, TMEM
//    columns [128, 128 + D)), each as D/16 or 8 instructions of K = 16 with
//    shared-memory descriptors; completion is signalled by tcgen05.commit to
//    an mbarrier.
//  * Each thread owns one query row (TMEM lane = row): it reads its S row
//    with tcgen05.ld, applies the causal and context masks, keeps the online
//    softmax (m in raw logit units, l in fp32, exponentials in base 2 with
//    the scale folded into a packed fused multiply-add; the exponentials run
//    in fp32 and each pair is rounded once to an fp16 pair, which is the P
//    operand of the second MMA and is summed in fp32 for l).  m is a
//    reference, not necessarily the maximum: it is set to the row's maximum
//    on its first tile and moves only when a weight would overflow fp16 (a
//    logit more than 16 above m in base-2 units); only then is the tile's
//    maximum computed, the tile's weights redone and the O row in TMEM
//    rescaled.  (The exponentials were once one packed fp16 ex2 per pair,
//    with the arguments rounded to fp16: at logit scales of 4.5 / sqrt(D)
//    that cost up to 1 % relative error on an output, and the fp32 form
//    measured the same speed.)
//    Masks are applied only on tiles that reach the diagonal or the context
//    end.  V rows past the context are zeroed in shared memory (0 * NaN in
//    stale slots would poison the sum).
//  * Work per KV tile: the TMA of the next tile overlaps the softmax and
//    both MMAs of the current one; the softmax and the MMAs of one CTA run
//    back to back (one CTA per SM by shared memory).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.cuh"
#include "pa_prefill_rows.cuh"
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kQT = 128;   // query rows per CTA (MMA M)
constexpr int kKT = 128;   // KV tokens per tile (MMA N of S, K of P.V)

template <int D, bool F8>
struct PrefillTraits {
  static constexpr int NA = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int ATOM = 128 * 128;            // bytes of one [128 rows][64 fp16] atom array
  static constexpr int QB = kQT * D * 2;
  static constexpr int KB = kKT * D * 2;
  static constexpr int STB = kKT * D;               // FP8 caches: one tile of codes
  // V stages.  A third one for fp16 caches (a V tile's copy could start a
  // whole KV-tile period earlier) fits the shared memory but measured 2 %
  // slower on the 7B-shaped chunked prefill (1086 vs 1108 TFLOP/s); FP8
  // caches have no room for it.
  static constexpr int NVS = 2;
  static constexpr int OFF_Q = 0;                   // Q tile x at OFF_Q + x*QB
  static constexpr int OFF_K0 = 2 * QB;             // K stage s at OFF_K0 + s*KB (s < 2)
  static constexpr int OFF_V0 = OFF_K0 + 2 * KB;    // V stage s at OFF_V0 + s*KB (s < NVS)
  static constexpr int OFF_ST = OFF_V0 + NVS * KB;  // FP8 caches: K codes, then V codes
  static constexpr int OFF_BAR = OFF_ST + (F8 ? 2 * STB : 0);
  // Decode rows: their rings use the Q and K/V stage area, their mbarriers
  // (up to 12 warps x 4 stages) and softmax weights follow the barriers.
  static constexpr int ROW_AREA = 2 * QB + 4 * KB;
  static constexpr int OFF_RBAR = OFF_BAR + 256;
  static constexpr int OFF_RPW = OFF_RBAR + prows::kRowWarps * 4 * 8;
  // Barriers, TMEM slot, decode-row metadata and alignment slack; at least
  // 120 KB so that one CTA holds an SM (each CTA allocates all 512 TMEM
  // columns).
  static constexpr int SMEM_USED = OFF_RPW + prows::kRowWarps * 16 * 4 + 1024;
  static constexpr int SMEM = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static_assert(SMEM <= 232448, "beyond the opt-in shared memory of one CTA");
  // Two softmax warpgroups and one producer warpgroup (its first warp issues
  // the MMAs, its second the TMA copies; with FP8 caches the other two widen
  // the codes to fp16).  Registers: the kernel is compiled for 384 threads at
  // kRegsLaunch each; the producer warpgroup gives registers back and the
  // softmax warpgroups take them (the split never exceeds the launch
  // allocation: kRegsSplit <= 384 * registers per thread at launch).
  static constexpr int THREADS = 384;
  static constexpr uint32_t TMEM_COLS = 512;        // S_x: 128 columns each, O_x: D columns each
  static constexpr uint32_t COL_O = 256;
  static_assert(D == 64 || D == 128, "head_dim");
};

constexpr int kRegsSoftmax = 200;
constexpr int kRegsProducer = 96;
// Registers the split needs at launch (per block); the launcher checks the
// compiled kernel's count against it before the first launch, since a
// setmaxnreg.inc beyond the block's allocation would wait forever.
constexpr int kRegsSplit = 2 * 128 * kRegsSoftmax + 128 * kRegsProducer;
static_assert(kRegsSplit <= 65536, "register split exceeds the register file");

// Sequences per launch: the unit table of one launch lives in the Q area.
constexpr int kSeqsPerLaunch = 4096;

struct PrefillParams {
  void* out;                     // fp16 [TQ][H][D]
  const void* query;             // fp16 [TQ][H][D] (decode rows read it directly)
  const void* key_cache;         // caches (decode rows copy from them directly)
  const void* value_cache;
  const int32_t* block_tables;   // [S][max_blocks]
  const int32_t* context_lens;   // [S]
  const int32_t* query_start;    // [S + 1]
  unsigned int* err;
  int seq_begin;                 // first sequence of this launch
  int num_seqs;                  // sequences of this launch
  int num_heads;
  int max_blocks;
  int num_blocks;
  int block_size;
  int qpairs;                    // most pairs of query tiles a sequence may need
  int sms;                       // SM count (one CTA per SM)
  int max_query_len;             // host bound of the chunk lengths
  int oob_row;                   // a row coordinate past the cache (zero-filled loads)
  float scale_log2;              // scale * log2(e), times the key scale for FP8 caches
  float v_scale;                 // value scale (1 for fp16 caches)
  int inputs_ready;              // 1: inputs are read before the wait, outputs stored after it
  int row_heads;                 // heads per decode-row unit (1 .. prows::kMaxRowHeads)
  int num_query_tokens;          // rows of query and out
};

// Per-CTA geometry of one query tile (x = 0, 1 of the pair).
struct QTile {
  int rows;      // valid rows (<= 0: inactive)
  int pos_min;   // position of row 0
  int n_kv;      // KV tiles it needs
};

// FP8 caches: widens one tile of codes (kKT rows x D codes, row-major) into
// the fp16 operand layout the TMA copies of an fp16 cache produce with
// 128-byte swizzle (atoms of 128 rows x 64 halves; the 16-byte chunk c of
// row r at r * 128 + ((c ^ (r & 7)) * 16)).  64 threads; E4M3 -> fp16 is
// exact.
template <int D>
__device__ __forceinline__ void widen_tile(const unsigned char* src, unsigned char* dst, int ctid) {
  constexpr int CPR = D / 16;     // 16-code chunks per row
  constexpr int ATOM = 128 * 128;
  constexpr int STEP = 64 / CPR;  // rows between one thread's chunks
  static_assert(STEP % 8 == 0, "a thread's chunks share one swizzle phase");
  // Thread ctid widens chunk j of rows r0, r0 + STEP, ...: the chunk column
  // and the row's swizzle phase (r & 7) are the same for all of them, so the
  // addresses are two bases and compile-time offsets.
  const int j = ctid % CPR, r0 = ctid / CPR;
  const int c0 = 2 * (j % 4);
  const unsigned char* sp = src + r0 * D + 16 * j;
  unsigned char* dp = dst + (j / 4) * ATOM + r0 * 128;
  const int o0 = (c0 ^ (r0 & 7)) << 4, o1 = ((c0 + 1) ^ (r0 & 7)) << 4;
#pragma unroll 4
  for (int k = 0; k < kKT / STEP; ++k) {
    const uint4 c = lds128(sp + k * STEP * D);
    const uint4 h0 = e4m3x8_to_f16x8(make_uint2(c.x, c.y));
    const uint4 h1 = e4m3x8_to_f16x8(make_uint2(c.z, c.w));
    *reinterpret_cast<uint4*>(dp + k * STEP * 128 + o0) = h0;
    *reinterpret_cast<uint4*>(dp + k * STEP * 128 + o1) = h1;
  }
}

// A waiting thread's view of an mbarrier: the next phase it expects.  Used
// only where at most one phase can complete between two waits (a parity
// wait cannot tell phase k from phase k + 2).
struct Waiter {
  uint32_t bar;
  uint32_t phase = 0;
  __device__ bool wait() {
    const bool ok = mbar_wait_bounded(bar, phase & 1);
    ++phase;
    return ok;
  }
};

template <int D, bool F8>
__global__ void __launch_bounds__(PrefillTraits<D, F8>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PrefillParams a) {
  using T = PrefillTraits<D, F8>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + T::OFF_BAR);
  // barriers: 0 q_full; 1,2 k_full[st]; 3,4 s_full[x]; 5,6 p_full[x]; 7,8 o_full[x]; 9 done;
  // 10,11 k_empty[st]; 12,13,20 v_full[st]; 14,15,21 v_empty[st]; FP8 caches: 16 kc_full,
  // 17 kc_empty, 18 vc_full, 19 vc_empty (the staged codes of the next K / V tile).  With FP8
  // caches the fp16 stages are filled by the two widening warps (k_full / v_full: one arrival
  // each).
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  auto v_full = [&](int st) { return bar(st < 2 ? 12 + st : 20); };
  auto v_empty = [&](int st) { return bar(st < 2 ? 14 + st : 21); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + T::OFF_BAR + 192);
  int* fail = reinterpret_cast<int*>(sm + T::OFF_BAR + 196);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int H = a.num_heads;
  // Set-up that does not depend on the unit runs beside the planning: warp 2
  // initialises the tensor-core path's barriers and prefetches the tensor
  // maps, warp 0 allocates the tensor memory (all CTAs; a decode row gives it
  // back unused).
  if (tid == 64) {
    mbar_init(bar(0), 1);
    mbar_init(bar(1), F8 ? 2 : 1);
    mbar_init(bar(2), F8 ? 2 : 1);
    mbar_init(bar(3), 1);
    mbar_init(bar(4), 1);
    mbar_init(bar(5), 128);
    mbar_init(bar(6), 128);
    mbar_init(bar(7), 1);
    mbar_init(bar(8), 1);
    mbar_init(bar(9), T::THREADS);
    mbar_init(bar(10), 1);
    mbar_init(bar(11), 1);
    mbar_init(bar(12), F8 ? 2 : 1);
    mbar_init(bar(13), F8 ? 2 : 1);
    mbar_init(bar(14), 1);
    mbar_init(bar(15), 1);
    mbar_init(bar(16), 1);
    mbar_init(bar(17), 2);
    mbar_init(bar(18), 1);
    mbar_init(bar(19), 2);
    mbar_init(bar(20), F8 ? 2 : 1);
    mbar_init(bar(21), 1);
    *fail = 0;
    fence_mbar_init();
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
    tmem_relinquish();
  }
  // The launch may start while the kernel before it on the stream still runs
  // (programmatic launch).  That kernel may write this call's inputs, so by
  // default everything below runs after the wait; the set-up above overlaps
  // its tail.  With inputs_ready (the caller's word that it writes none of
  // them) the planning, the loads and the products run at once, and only the
  // output stores wait (decode rows wait first).
  if (!a.inputs_ready) pdl_wait();
  // This CTA's unit (see pa_prefill_rows.cuh for the order), with its
  // sequence's query rows and context length; the table and scratch live in
  // the Q area until the first loads.  Up to 32 sequences: warp 1 alone;
  // more: the whole block.
  int* scratch = reinterpret_cast<int*>(sm) + kSeqsPerLaunch;
  prows::Unit* unit_s = reinterpret_cast<prows::Unit*>(scratch + 20);
  if (a.num_seqs <= 32) {
    if (warp == 1)
      prows::plan_small(a.query_start + a.seq_begin, a.context_lens + a.seq_begin, a.num_seqs, H,
                        a.row_heads, a.qpairs, a.sms, (int)blockIdx.x, unit_s, scratch + 19);
  } else {
    int tot = 0;
    const prows::Unit u = prows::plan_unit_block(a.query_start + a.seq_begin,
                                                 a.context_lens + a.seq_begin, a.num_seqs, H,
                                                 a.row_heads, a.qpairs, a.sms, (int)blockIdx.x,
                                                 reinterpret_cast<int*>(sm), scratch, &tot);
    if (tid == 0) {
      *unit_s = u;
      scratch[19] = tot;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const prows::Unit unit = *unit_s;
  if (blockIdx.x == 0 && tid == 0 && scratch[19] > (int)gridDim.x)
    atomicOr(a.err, PA_ERRBIT_CONTEXT);  // inconsistent query_start: units beyond the grid
  if (unit.kind != 1) {
    // No tensor-core work: a decode row runs on CUDA cores; then the tensor
    // memory goes back.
    if (unit.kind == 2) {
      pdl_wait();
      pdl_launch_dependents();
      const int s = a.seq_begin + unit.s, q_len = unit.q_len, c = unit.c;
      const bool bad = q_len != 1 || c < 1 || c > a.max_blocks * a.block_size ||
                       q_len > a.max_query_len || unit.q0 < 0 ||
                       unit.q0 > a.num_query_tokens - q_len;
      if (bad && unit.h == 0 && tid == 0) atomicOr(a.err, PA_ERRBIT_CONTEXT);
      if (!bad) {
        const int32_t* bt = a.block_tables + (size_t)s * a.max_blocks;
        uint64_t* dbars = reinterpret_cast<uint64_t*>(sm + T::OFF_RBAR);
        float* pw = reinterpret_cast<float*>(sm + T::OFF_RPW);
        if (tid < prows::kRowWarps * 4) {
          mbar_init(smem_u32(&dbars[tid]), 1);
          fence_mbar_init();
        }
        __syncthreads();
        if (a.block_size == 8) {
          constexpr int NST = prows::row_stages<D, 8, F8>(T::ROW_AREA);
          prows::decode_row<D, 8, F8, NST>(a.query, a.key_cache, a.value_cache, bt, H,
                                            a.block_size, a.num_blocks, a.scale_log2, a.v_scale,
                                            a.err, a.out, unit.h, unit.nh, unit.q0, c, sm, dbars,
                                            pw, fail);
        } else {
          constexpr int NST = prows::row_stages<D, 16, F8>(T::ROW_AREA);
          prows::decode_row<D, 16, F8, NST>(a.query, a.key_cache, a.value_cache, bt, H,
                                             a.block_size, a.num_blocks, a.scale_log2, a.v_scale,
                                             a.err, a.out, unit.h, unit.nh, unit.q0, c, sm, dbars,
                                             pw, fail);
        }
      }
    }
    if (warp == 0) tmem_dealloc(tmem, T::TMEM_COLS);
    return;
  }
  // The unit's values came through shared memory; a shuffle from lane 0 lets
  // the compiler keep them in uniform registers (as values derived from
  // blockIdx would be), which leaves the softmax warps their registers: read
  // as plain per-thread values they cost the kernel 5 % in throughput.
  const int s = __shfl_sync(kFullMask, a.seq_begin + unit.s, 0);
  const int h = __shfl_sync(kFullMask, unit.h, 0);
  const int pq = __shfl_sync(kFullMask, unit.pq, 0);

  pdl_launch_dependents();

  const int q0 = __shfl_sync(kFullMask, unit.q0, 0);
  const int q_len = __shfl_sync(kFullMask, unit.q_len, 0);
  const int c = __shfl_sync(kFullMask, unit.c, 0);
  const bool bad = q_len < 0 || q_len > c || c > a.max_blocks * a.block_size ||
                   q_len > a.max_query_len || q0 < 0 || q0 > a.num_query_tokens - q_len;
  if (bad && pq == 0 && h == 0 && tid == 0) atomicOr(a.err, PA_ERRBIT_CONTEXT);
  QTile qx[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    const int qt = 2 * pq + x;
    qx[x].rows = bad ? 0 : min(kQT, q_len - qt * kQT);
    qx[x].pos_min = c - q_len + qt * kQT;
    qx[x].n_kv = qx[x].rows > 0 ? (qx[x].pos_min + qx[x].rows - 1) / kKT + 1 : 0;
  }
  const int n_kv = max(qx[0].n_kv, qx[1].n_kv);

  // The roles never meet again: each ends by arriving on the done barrier,
  // after which warp 0 frees the tensor memory.
  if (warp >= 8) {
    setmaxnreg_dec<kRegsProducer>();
    // K of tile t sits in stage t & 1 of a two-stage ring, V in stage t % NVS of
    // its own ring: k_full / v_full complete once per tile, parity (t >> 1) & 1
    // and (t / NVS) & 1; k_empty / v_empty once per tile that used the stage.
    // K is released after the tile's QK products, V after its P.V products.
    constexpr int NVS = T::NVS;
    auto wait_k = [&](int t) { return mbar_wait_bounded(bar(1 + (t & 1)), (t >> 1) & 1); };
    auto wait_v = [&](int t) { return mbar_wait_bounded(v_full(t % NVS), (t / NVS) & 1); };
    if (warp == 9 && n_kv > 0) {
      // ---------------- TMA warp: Q tiles, then K/V tiles into a two-stage ring
      const int32_t* bt = a.block_tables + (size_t)s * a.max_blocks;
      const int bpt = kKT / a.block_size;
      // Cache row of block `lane` of KV tile t (lanes < bpt; one load per lane,
      // fetched a tile ahead so no copy waits on the block table).
      auto tile_row = [&](int t) {
        const int lb = t * bpt + lane;
        int row = a.oob_row;
        if (lane < bpt && t < n_kv && lb * a.block_size < c) {
          const int phys = bt[lb];
          if (phys >= 0 && phys < a.num_blocks)
            row = (phys * H + h) * a.block_size;
          else
            atomicOr(a.err, PA_ERRBIT_BLOCK_ID);
        }
        return row;
      };
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(0), (qx[1].rows > 0 ? 2 : 1) * T::QB);
#pragma unroll
        for (int x = 0; x < 2; ++x)
          if (qx[x].rows > 0)
#pragma unroll
            for (int at = 0; at < T::NA; ++at)
              tma_load_3d(s_base + T::OFF_Q + x * T::QB + at * T::ATOM, &tq, at * 64, h,
                          q0 + (2 * pq + x) * kQT, bar(0));
      }
      // Program order per tile: K(t) then V(t); K(t + 1) needs the QK of
      // tile t - 1, which the MMA warp issues after the P.V of tile t - 2 that
      // frees V(t)'s stage, so this order never waits on a later release.
      // FP8 caches: the codes of tile t go to the staging buffer (one tile of K
      // codes and one of V codes, row-major, one box of B rows per block) once
      // the widening warps have read tile t - 1's; the fp16 stages are theirs.
      auto issue = [&](int t, int row, bool is_v) {
        if constexpr (F8) {
          const uint32_t dst = s_base + T::OFF_ST + (is_v ? T::STB : 0);
          const uint32_t fb = bar(is_v ? 18 : 16);
          if (lane == 0) mbar_arrive_expect_tx(fb, T::STB);
          __syncwarp();
          if (lane < bpt)
            tma_load_2d(dst + (uint32_t)(lane * a.block_size * D), is_v ? &tv : &tk, 0, row, fb);
        } else {
          const uint32_t dst = is_v ? s_base + T::OFF_V0 + (t % NVS) * T::KB
                                    : s_base + T::OFF_K0 + (t & 1) * T::KB;
          const uint32_t fb = is_v ? v_full(t % NVS) : bar(1 + (t & 1));
          if (lane == 0) mbar_arrive_expect_tx(fb, T::KB);
          __syncwarp();
          if (lane < bpt) {  // lane b issues block b's boxes
            const uint32_t roff = (uint32_t)(lane * a.block_size * 128);
#pragma unroll
            for (int at = 0; at < T::NA; ++at)
              tma_load_2d(dst + at * T::ATOM + roff, is_v ? &tv : &tk, at * 64, row, fb);
          }
        }
      };
      // The barrier a copy of tile t waits on before it may start, and its parity.
      auto free_bar = [&](int t, bool is_v) {
        return F8 ? bar(is_v ? 19 : 17) : is_v ? v_empty(t % NVS) : bar(10 + (t & 1));
      };
      auto free_par = [&](int t, bool is_v) {
        return F8 ? (uint32_t)((t - 1) & 1)
                  : is_v ? (uint32_t)((t / NVS - 1) & 1) : (uint32_t)(((t >> 1) - 1) & 1);
      };
      auto first_wait = [&](bool is_v) { return F8 ? 1 : is_v ? NVS : 2; };
      int row = tile_row(0);
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int t = 0; t < n_kv && ok; ++t) {
        if (t >= first_wait(false))
          ok = __all_sync(kFullMask, mbar_wait_bounded(free_bar(t, false), free_par(t, false)));
        if (!ok) break;
        issue(t, row, false);
        ++k_issued;
        if (t >= first_wait(true))
          ok = __all_sync(kFullMask, mbar_wait_bounded(free_bar(t, true), free_par(t, true)));
        if (!ok) break;
        issue(t, row, true);
        ++v_issued;
        row = tile_row(t + 1);
      }
      if (!ok && lane == 0) {
        *fail = 1;
        // Let the copies this warp started land (bounded) before the shared
        // memory is released.
        if constexpr (F8) {
          if (k_issued > 0) mbar_wait_bounded(bar(16), (k_issued - 1) & 1);
          if (v_issued > 0) mbar_wait_bounded(bar(18), (v_issued - 1) & 1);
        } else {
          for (int u = max(0, k_issued - 2); u < k_issued; ++u) wait_k(u);
          for (int u = max(0, v_issued - NVS); u < v_issued; ++u) wait_v(u);
        }
      }
    } else if (F8 && (warp == 10 || warp == 11) && n_kv > 0) {
      // ---------------- FP8 caches: the two widening warps.  Per tile t, in
      // the order K then V: wait for the staged codes and for the fp16 stage
      // t & 1 to be free (the QK / P.V products of tile t - 2 are done), widen,
      // make the writes visible to the tensor cores, then release the staging
      // buffer and fill the stage (one arrival per warp on each barrier).
      const int ctid = tid - 320;
      bool ok = true;
      for (int t = 0; t < n_kv && ok; ++t) {
        const int st = t & 1;
#pragma unroll
        for (int kv = 0; kv < 2 && ok; ++kv) {
          ok = __all_sync(kFullMask, mbar_wait_bounded(bar(kv ? 18 : 16), t & 1));
          static_assert(!F8 || NVS == 2, "the widening warps fill two-stage rings");
          if (ok && t >= 2)
            ok = __all_sync(kFullMask, mbar_wait_bounded(bar((kv ? 14 : 10) + st), ((t >> 1) - 1) & 1));
          // Warp-uniform: the failure flag may be set by another warp between
          // two lanes' reads, and the widening ends in a __syncwarp.
          ok = __all_sync(kFullMask, ok && !*fail);
          if (!ok) break;
          widen_tile<D>(sm + T::OFF_ST + kv * T::STB,
                        sm + (kv ? T::OFF_V0 : T::OFF_K0) + st * T::KB, ctid);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(kv ? 19 : 17));
            mbar_arrive(bar((kv ? 12 : 1) + st));
          }
        }
      }
      if (!ok && lane == 0) *fail = 1;
    } else if (warp == 8 && n_kv > 0) {
    // ---------------- MMA issuer (lane 0; the warp zeroes V rows past the context)
    int qk[2] = {0, 0}, pv[2] = {0, 0}, krel = 0, vrel = 0;
    constexpr uint32_t kIdQK = umma_idesc_f16(kQT, kKT, false, false);
    constexpr uint32_t kIdPV = umma_idesc_f16(kQT, D, false, true);
    // The whole warp runs the issue code (warp-uniform operands); lane 0
    // alone issues each instruction.
    const bool leader = lane == 0;
    // Base descriptors, computed once; the descriptor of a K step or stage
    // differs only in its start address field (16-byte units), so each MMA
    // adds a compile-time offset.
    const uint64_t q_desc0 = umma_desc_sw128(s_base + T::OFF_Q, 16, 1024);
    const uint64_t k_desc0 = umma_desc_sw128(s_base + T::OFF_K0, 16, 1024);
    const uint64_t v_desc0 = umma_desc_sw128(s_base + T::OFF_V0, T::ATOM, 1024);
    constexpr uint64_t kStageStep = (uint64_t)T::KB >> 4;
    auto qk_mma = [&](int x, int t, bool release) {
      const uint64_t qd = q_desc0 + (uint64_t)((x * T::QB) >> 4);
      const uint64_t kd = k_desc0 + (t & 1) * kStageStep;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint64_t off = (uint64_t)(((k / 4) * T::ATOM + (k % 4) * 32) >> 4);
        umma_f16_if(leader, tmem + 128 * x, qd + off, kd + off, kIdQK, k > 0);
      }
      umma_commit_if(leader, bar(3 + x));
      ++qk[x];
      if (release) {  // the last reader of K stage t & 1
        umma_commit_if(leader, bar(10 + (t & 1)));
        ++krel;
      }
    };
    auto pv_mma = [&](int x, int t, bool release) {
      const uint64_t vd = v_desc0 + (t % NVS) * kStageStep;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kKT / 16; ++k)
        umma_f16_tmem_a_if(leader, tmem + T::COL_O + D * x, tmem + 128 * x + 8 * k,
                           vd + (uint64_t)((k * 16 * 128) >> 4), kIdPV, t > 0 || k > 0);
      umma_commit_if(leader, bar(7 + x));
      ++pv[x];
      if (release) {  // the last reader of V stage t & 1
        umma_commit_if(leader, v_empty(t % NVS));
        ++vrel;
      }
    };
    // V rows of tile t past the context: zeroed by the whole warp after the
    // tile has landed (stale slots may hold anything; 0 * NaN would poison O).
    auto zero_v_tail = [&](int t) {
      const int first = c - t * kKT;
      if (first >= kKT) return;
      unsigned char* v = sm + T::OFF_V0 + (t % NVS) * T::KB;
      const int nchunks = (kKT - max(first, 0)) * 8;
      for (int i = lane; i < nchunks * T::NA; i += 32) {
        const int at = i / nchunks, r = max(first, 0) + (i % nchunks) / 8, ch = i % 8;
        *reinterpret_cast<uint4*>(v + at * T::ATOM + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
    };
    Waiter p_w[2] = {{bar(5)}, {bar(6)}};
    bool ok = __all_sync(kFullMask, mbar_wait_bounded(bar(0), 0) && wait_k(0));
    if (ok) {
      qk_mma(0, 0, qx[1].n_kv == 0);
      if (qx[1].n_kv > 0) qk_mma(1, 0, true);
    }
    // S(x, t + 1) overwrites the columns P(x, t) occupies; tcgen05.mma issued
    // by one thread execute in issue order, so QK(x, t + 1) is issued right
    // after P.V(x, t) without waiting for it.
    // Every wait result is made warp-uniform at once, so all branches below
    // are taken by the whole warp.
    auto uni = [&](bool v) { return __all_sync(kFullMask, v); };
    for (int t = 0; t < n_kv && ok; ++t) {
      const bool a0 = t < qx[0].n_kv, a1 = t < qx[1].n_kv;
      const bool n0 = t + 1 < qx[0].n_kv, n1 = t + 1 < qx[1].n_kv;
      ok = uni(wait_v(t));
      if (ok) zero_v_tail(t);
      if (ok && a0) ok = uni(p_w[0].wait());
      if (ok && a0) pv_mma(0, t, !a1);
      if (ok && t + 1 < n_kv) ok = uni(wait_k(t + 1));
      if (ok && n0) qk_mma(0, t + 1, !n1);
      if (ok && a1) ok = uni(p_w[1].wait());
      if (ok && a1) pv_mma(1, t, true);
      if (ok && n1) qk_mma(1, t + 1, true);
    }
    if (!ok) {
      if (lane == 0) {
        atomicOr(a.err, PA_ERRBIT_TIMEOUT);
        *fail = 1;
        // Let every MMA this warp started finish (bounded) before the TMEM and
        // shared memory are released.
        for (int i = 0; i < 2; ++i) {
          if (qk[i] > 0) mbar_wait_bounded(bar(3 + i), (qk[i] - 1) & 1);
          if (pv[i] > 0) mbar_wait_bounded(bar(7 + i), (pv[i] - 1) & 1);
        }
        if (krel > 0) mbar_wait_bounded(bar(10 + ((krel - 1) & 1)), ((krel - 1) >> 1) & 1);
        if (vrel > 0) mbar_wait_bounded(v_empty((vrel - 1) % NVS), ((vrel - 1) / NVS) & 1);
      }
    }
    }
    tc_fence_before();
    mbar_arrive(bar(9));
    return;
  }
  setmaxnreg_inc<kRegsSoftmax>();
  {
    // ---------------- softmax warpgroup x: one query row per thread
    const int x = warp >> 2;
    const int row = tid & 127;
    const QTile qt = qx[x];
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + 128 * x + lane_off;
    const uint32_t t_o = tmem + T::COL_O + D * x + lane_off;
    const int qpos = qt.pos_min + row;
    float m = -INFINITY, l = 0.f;
    Waiter s_w{bar(3 + x)};
    bool ok = true;
    for (int t = 0; t < qt.n_kv; ++t) {
      // Warp-uniform outcome: the tensor-memory accesses below are warp-collective.
      ok = __all_sync(kFullMask, s_w.wait() && !*fail);
      if (!ok) break;
      tc_fence_after();
      // The row's logits of this tile, masked past the diagonal and the
      // context end (only on tiles that reach them).
      const int kv0 = t * kKT;
      auto load_logits = [&](float (&xv)[kKT]) {
        uint32_t sr[kKT];
#pragma unroll
        for (int cb = 0; cb < kKT / 32; ++cb)
          tmem_ld32(t_s + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[cb * 32]));
        tmem_wait_ld();  // one wait for all four loads
#pragma unroll
        for (int j = 0; j < kKT; ++j) xv[j] = __uint_as_float(sr[j]);
        if (kv0 + kKT - 1 > qt.pos_min) {
          const int lim = min(qpos, c - 1) - kv0;
#pragma unroll
          for (int j = 0; j < kKT; ++j)
            if (j > lim) xv[j] = -INFINITY;
        }
      };
      // Weights against the row's reference m (raw logit units): fp32
      // exponentials rounded to fp16 pairs (they feed the fp16 P.V product);
      // the row sum adds those exact fp16 values in fp32.  m is only a
      // reference, so weights may exceed 1: the tile's maximum is computed only
      // on the row's first tile and when a weight overflows fp16 (the tile
      // holds a logit more than 16 above m in base-2 units; the sum is then not
      // finite).  Then m moves to the maximum and the weights are recomputed
      // from the logits reloaded from tensor memory (S is intact until P is
      // written over it).
      float sq[4];
      uint32_t pk[kKT / 2];
      const uint64_t sc2 = f32x2_splat(a.scale_log2);
      auto weights = [&](const float (&xv)[kKT], float ref) {
        const uint64_t neg2 = f32x2_splat(ref == -INFINITY ? 0.f : -ref * a.scale_log2);
#pragma unroll
        for (int u = 0; u < 4; ++u) sq[u] = 0.f;
#pragma unroll
        for (int j = 0; j < kKT / 2; ++j) {
          const float2 y = ffma2(xv[2 * j], xv[2 * j + 1], sc2, neg2);  // packed: two fmas at once
          pk[j] = exp2_f32_to_f16x2(y.x, y.y);
          sq[j & 3] = add_f16x2_f32(pk[j], sq[j & 3]);
        }
        return (sq[0] + sq[1]) + (sq[2] + sq[3]);
      };
      // The tensor-memory loads are warp-collective, so the choice of path is
      // made for the whole warp: if any row needs the maximum, every row of the
      // warp recomputes against its own (still exact for the others).
      float mx = m, ls = 0.f;
      bool slow = __any_sync(kFullMask, m == -INFINITY);
      if (!slow) {
        float xv[kKT];
        load_logits(xv);
        ls = weights(xv, m);
        // a weight overflowed (or a NaN logit) in some row of the warp
        slow = __any_sync(kFullMask, !(ls <= 3.4028234663852886e38f));
      }
      if (slow) {
        float xv[kKT];
        load_logits(xv);
        // Independent partial maxima keep the dependency chains short.
        float mq[4] = {m, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < kKT; j += 8)
#pragma unroll
          for (int u = 0; u < 4; ++u) mq[u] = fmax3(mq[u], xv[j + 2 * u], xv[j + 2 * u + 1]);
        mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        ls = weights(xv, mx);
      }
      const float alpha = (mx == -INFINITY || mx == m) ? 1.f : exp2_approx((m - mx) * a.scale_log2);
      l = l * alpha + ls;
      m = mx;
      // O(x, t - 1) is complete here: S(x, t) was computed after it.
      if (t > 0 && __any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll
        for (int cb = 0; cb < D / 32; cb += 2) {
          uint32_t r[2][32];
          tmem_ld32(t_o + cb * 32, r[0]);
          tmem_ld32(t_o + cb * 32 + 32, r[1]);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[u][j] = __float_as_uint(__uint_as_float(r[u][j]) * alpha);
            tmem_st32(t_o + (cb + u) * 32, r[u]);
          }
        }
      }
      // P (fp16 pairs) over the first 64 columns of this tile's S.
      {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = pk[j];
        tmem_st32(t_s, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = pk[32 + j];
        tmem_st32(t_s + 32, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(5 + x));
    }
    if (ok && qt.n_kv > 0) {
      // The last P.V of this tile (phase n_kv - 1; the earlier ones completed
      // before S of the last tile was computed, so the parity is unambiguous).
      const bool done = __all_sync(kFullMask, mbar_wait_bounded(bar(7 + x), (qt.n_kv - 1) & 1) && !*fail);
      pdl_wait();  // the output may be read or written by the kernel before this one
      if (done) {
        tc_fence_after();
        const float inv = l > 0.f ? a.v_scale / l : 0.f;  // v_scale: FP8 values (1 for fp16)
        __half* orow = static_cast<__half*>(a.out) +
                       ((size_t)(q0 + (2 * pq + x) * kQT + row) * H + h) * D;
#pragma unroll
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t r[32];
          tmem_ld32(t_o + cb * 32, r);
          tmem_wait_ld();
          if (row < qt.rows) {
#pragma unroll
            for (int j8 = 0; j8 < 4; ++j8) {
              uint32_t w[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const __half2 hv = __floats2half2_rn(__uint_as_float(r[8 * j8 + 2 * u]) * inv,
                                                     __uint_as_float(r[8 * j8 + 2 * u + 1]) * inv);
                w[u] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              *reinterpret_cast<uint4*>(orow + cb * 32 + j8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  mbar_arrive(bar(9));
  if (warp == 0) {
    if (!mbar_wait_bounded(bar(9), 0) && lane == 0) atomicOr(a.err, PA_ERRBIT_TIMEOUT);
    tc_fence_after();
    tmem_dealloc(tmem, T::TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// fp16 tensors with 128-byte swizzle (operand layout), or bytes unswizzled
// (FP8 codes, widened in shared memory).
bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box, bool bytes = false) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool F8>
cudaError_t launch_prefill_t(const PrefillArgs& g, cudaStream_t stream) {
  using T = PrefillTraits<D, F8>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    cudaFuncAttributes fa{};
    attr_err = cudaFuncGetAttributes(&fa, prefill_kernel<D, F8>);
    if (attr_err == cudaSuccess && fa.numRegs * T::THREADS < kRegsSplit)
      attr_err = cudaErrorInvalidConfiguration;  // never launch a split that could not be granted
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(prefill_kernel<D, F8>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tq, tk, tv;
  const cuuint64_t qdims[3] = {(cuuint64_t)D, (cuuint64_t)g.num_heads, (cuuint64_t)g.num_query_tokens};
  const cuuint64_t qstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)g.num_heads * D * 2};
  const cuuint32_t qbox[3] = {64, 1, (cuuint32_t)kQT};
  const long long rows = (long long)g.num_blocks * g.num_heads * g.block_size;
  const cuuint64_t kdims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t kstr[1] = {(cuuint64_t)D * (F8 ? 1 : 2)};
  // fp16: boxes of one 64-element swizzle atom; FP8: one box covers a row.
  const cuuint32_t kbox[2] = {(cuuint32_t)(F8 ? D : 64), (cuuint32_t)g.block_size};
  if (!encode(&tq, g.query, 3, qdims, qstr, qbox) ||
      !encode(&tk, g.key_cache, 2, kdims, kstr, kbox, F8) ||
      !encode(&tv, g.value_cache, 2, kdims, kstr, kbox, F8))
    return cudaErrorInvalidValue;
  PrefillParams p{};
  p.out = g.out;
  p.query = g.query;
  p.key_cache = g.key_cache;
  p.value_cache = g.value_cache;
  p.block_tables = g.block_tables;
  p.context_lens = g.context_lens;
  p.query_start = g.query_start;
  p.err = g.err;
  p.num_heads = g.num_heads;
  p.max_blocks = g.max_blocks;
  p.num_blocks = g.num_blocks;
  p.block_size = g.block_size;
  p.qpairs = (g.max_query_len + 2 * kQT - 1) / (2 * kQT);
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cudaErrorInvalidValue;
    p.sms = sms;
  }
  p.max_query_len = g.max_query_len;
  p.oob_row = (int)rows;
  p.scale_log2 = g.scale_log2;
  p.v_scale = F8 ? g.v_scale : 1.f;
  p.inputs_ready = g.inputs_ready ? 1 : 0;
  p.num_query_tokens = g.num_query_tokens;
  // One launch per window of sequences.  The grid bounds the window's units:
  // a sequence of q tokens needs ceil(q / 256) units per head, at most qpairs,
  // and over the window sum(ceil(q / 256)) <= (TQ + 255 * n) / 256.  A decode
  // row (q = 1) is one unit per head within that bound.  When the window's
  // count r of decode rows is known, the rows' units are counted exactly
  // (RowSplit) and the other n - r sequences hold the other TQ - r tokens; a
  // unit then covers up to kMaxRowHeads heads of a row.  r
  // is known when no sequence has more than one token (r <= n; shorter ones
  // have no units) or from the caller for a call of one window.
  for (int sb = 0; sb < g.num_seqs; sb += kSeqsPerLaunch) {
    const int n = g.num_seqs - sb < kSeqsPerLaunch ? g.num_seqs - sb : kSeqsPerLaunch;
    p.seq_begin = sb;
    p.num_seqs = n;
    const int r = g.max_query_len == 1 ? n
                  : g.num_seqs <= kSeqsPerLaunch ? g.num_decode_rows : -1;
    p.row_heads = r >= 0 ? prows::kMaxRowHeads : 1;
    const int nc = r >= 0 ? (n > r ? n - r : 0) : n;  // the other sequences and their tokens
    long long tc = r >= 0 ? (long long)g.num_query_tokens - r : g.num_query_tokens;
    if (tc < 0) tc = 0;
    long long per_head = (long long)nc * p.qpairs;
    const long long by_tokens = (tc + 255LL * nc) / 256;
    if (by_tokens < per_head) per_head = by_tokens;
    long long grid = per_head * g.num_heads;
    if (r > 0) grid += prows::RowSplit(r, g.num_heads, p.row_heads, p.sms).units(g.num_heads);
    if (grid <= 0) continue;
    const cudaError_t e = launch_pdl(prefill_kernel<D, F8>, dim3((unsigned)grid),
                                     dim3(T::THREADS), (size_t)T::SMEM, stream, tq, tk, tv, p);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

bool prefill_rows_fit(int num_blocks, int num_heads, int block_size) {
  return (long long)num_blocks * num_heads * block_size < (1LL << 31) - 1;
}

cudaError_t launch_prefill(const PrefillArgs& g, cudaStream_t stream) {
  if (g.num_seqs == 0 || g.max_query_len == 0) return cudaSuccess;
  if (g.fp8)
    return g.head_dim == 64 ? launch_prefill_t<64, true>(g, stream)
                            : launch_prefill_t<128, true>(g, stream);
  return g.head_dim == 64 ? launch_prefill_t<64, false>(g, stream)
                          : launch_prefill_t<128, false>(g, stream);
}

}  // namespace pa
