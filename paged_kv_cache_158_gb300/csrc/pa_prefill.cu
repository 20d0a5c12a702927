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
//  * One CTA of four warps per (sequence, head, tile of 128 new tokens).
//    Q (128 x D) and the paged K/V tiles (128 tokens = 128/B blocks) arrive
//    by TMA tensor copies with 128-byte swizzle, one box per physical block,
//    into a two-stage ring; a block past the context is fetched from an
//    out-of-range coordinate (zero fill).
//  * One thread issues tcgen05.mma: S = Q K^T (M = 128 queries, N = 128
//    tokens, fp32 in TMEM columns [0, 128)), then O += P V (N = D, TMEM
//    columns [128, 128 + D)), each as D/16 or 8 instructions of K = 16 with
//    shared-memory descriptors; completion is signalled by tcgen05.commit to
//    an mbarrier.
//  * Each thread owns one query row (TMEM lane = row): it reads its S row
//    with tcgen05.ld, applies the causal and context masks, keeps the online
//    softmax (m in raw logit units, l in fp32, exponentials in base 2 with
//    the scale folded into one fused multiply-add), rounds P to fp16 for the
//    second MMA and writes it to shared memory in the swizzled K-major
//    layout that MMA reads, and rescales its O row in TMEM when the running
//    maximum grows.  Masks are applied only on tiles that reach the
//    diagonal or the context end.  V rows past the context are zeroed in shared
//    memory (0 * NaN in stale slots would poison the sum).
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
#include "pa_umma.cuh"

namespace pa {
namespace {

constexpr int kQT = 128;   // query rows per CTA (MMA M)
constexpr int kKT = 128;   // KV tokens per tile (MMA N of S, K of P.V)

template <int D>
struct PrefillTraits {
  static constexpr int NA = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int ATOM = 128 * 128;            // bytes of one [128 rows][64 fp16] atom array
  static constexpr int QB = kQT * D * 2;
  static constexpr int KB = kKT * D * 2;
  static constexpr int PB = kQT * kKT * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K0 = QB;                 // stage s: K at OFF_K0 + s*2*KB, V after it
  static constexpr int OFF_P = QB + 4 * KB;
  static constexpr int OFF_BAR = OFF_P + PB;        // q, kv[2], s, o barriers; TMEM slot; flags
  static constexpr int SMEM = OFF_BAR + 128 + 1024;  // + alignment slack
  static constexpr uint32_t TMEM_COLS = 256;        // S: 128 columns, O: D columns
  static_assert(D == 64 || D == 128, "head_dim");
};

struct PrefillParams {
  void* out;                     // fp16 [TQ][H][D]
  const int32_t* block_tables;   // [S][max_blocks]
  const int32_t* context_lens;   // [S]
  const int32_t* query_start;    // [S + 1]
  unsigned int* err;
  int num_seqs;
  int num_heads;
  int max_blocks;
  int num_blocks;
  int block_size;
  int qtiles;                    // query tiles per sequence covered by the grid
  int max_query_len;             // host bound of the chunk lengths
  int oob_row;                   // a row coordinate past the cache (zero-filled loads)
  float scale_log2;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk16) {
  return (uint32_t)(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(128, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const PrefillParams a) {
  using T = PrefillTraits<D>;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_base = smem_u32(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + T::OFF_BAR);
  const uint32_t q_bar = smem_u32(&bars[0]);
  const uint32_t kv_bar0 = smem_u32(&bars[1]);
  const uint32_t s_bar = smem_u32(&bars[3]);
  const uint32_t o_bar = smem_u32(&bars[4]);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + T::OFF_BAR + 64);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int H = a.num_heads;
  const int h = blockIdx.x % H;
  const int rest = blockIdx.x / H;
  const int s = rest % a.num_seqs;
  const int qt = a.qtiles - 1 - rest / a.num_seqs;  // heaviest tiles first

  if (tid == 0) {
    mbar_init(q_bar, 1);
    mbar_init(kv_bar0, 1);
    mbar_init(kv_bar0 + 8, 1);
    mbar_init(s_bar, 1);
    mbar_init(o_bar, 1);
    fence_mbar_init();
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), T::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  pdl_wait();
  pdl_launch_dependents();

  const int q0 = a.query_start[s];
  const int q_len = a.query_start[s + 1] - q0;
  const int c = a.context_lens[s];
  const bool bad = q_len < 0 || q_len > c || c > a.max_blocks * a.block_size ||
                   q_len > a.max_query_len;
  if (bad && qt == a.qtiles - 1 && h == 0 && tid == 0) atomicOr(a.err, PA_ERRBIT_CONTEXT);
  const int rows_valid = bad ? 0 : min(kQT, q_len - qt * kQT);

  if (rows_valid > 0) {
    const int pos_min = c - q_len + qt * kQT;          // position of this tile's row 0
    const int n_t = (pos_min + rows_valid - 1) / kKT + 1;
    const int32_t* bt = a.block_tables + (size_t)s * a.max_blocks;
    const int bpt = kKT / a.block_size;                // blocks per KV tile

    // Thread 0: K and V tile t into stage st (one box per block and atom).
    auto issue_kv = [&](int t, int st) {
      const uint32_t bar = kv_bar0 + 8 * st;
      const uint32_t kdst = s_base + T::OFF_K0 + st * 2 * T::KB;
      const uint32_t vdst = kdst + T::KB;
      mbar_arrive_expect_tx(bar, 2 * T::KB);
      for (int b = 0; b < bpt; ++b) {
        const int lb = t * bpt + b;
        int row = a.oob_row;
        if (lb * a.block_size < c) {
          const int phys = bt[lb];
          if (phys >= 0 && phys < a.num_blocks)
            row = (phys * H + h) * a.block_size;
          else
            atomicOr(a.err, PA_ERRBIT_BLOCK_ID);
        }
        const uint32_t roff = (uint32_t)(b * a.block_size * 128);
#pragma unroll
        for (int at = 0; at < T::NA; ++at) {
          tma_load_2d(kdst + at * T::ATOM + roff, &tk, at * 64, row, bar);
          tma_load_2d(vdst + at * T::ATOM + roff, &tv, at * 64, row, bar);
        }
      }
    };

    if (tid == 0) {
      mbar_arrive_expect_tx(q_bar, T::QB);
#pragma unroll
      for (int at = 0; at < T::NA; ++at)
        tma_load_3d(s_base + T::OFF_Q + at * T::ATOM, &tq, at * 64, h, q0 + qt * kQT, q_bar);
      issue_kv(0, 0);
    }

    constexpr uint32_t kIdQK = umma_idesc_f16(kQT, kKT, false, false);
    constexpr uint32_t kIdPV = umma_idesc_f16(kQT, D, false, true);
    const int qpos = pos_min + tid;                    // this thread's query position
    float m = -INFINITY, l = 0.f;
    // Thread 0's record of what it started, for a clean exit after a timeout.
    int kv_issued = 1, qk_done = 0, pv_done = 0;
    bool good = true;
    int t = 0;
    for (; t < n_t; ++t) {
      const int st = t & 1;
      const uint32_t kaddr = s_base + T::OFF_K0 + st * 2 * T::KB;
      const uint32_t vaddr = kaddr + T::KB;
      // Every wait is bounded; a thread that gives up skips the work but still
      // reaches the block-wide vote below, so all threads leave together.
      good = mbar_wait_bounded(kv_bar0 + 8 * st, (t >> 1) & 1);
      if (t == 0) good = good && mbar_wait_bounded(q_bar, 0);

      // S = Q K^T
      if (tid == 0 && good) {
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const int at = k / 4, kk = k % 4;
          const uint64_t da = umma_desc_sw128(s_base + T::OFF_Q + at * T::ATOM + kk * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(kaddr + at * T::ATOM + kk * 32, 16, 1024);
          umma_f16(tmem_s, da, db, kIdQK, k > 0);
        }
        umma_commit(s_bar);
        ++qk_done;
      }
      good = good && mbar_wait_bounded(s_bar, t & 1);
      if (t > 0) good = good && mbar_wait_bounded(o_bar, (t - 1) & 1);  // P.V of t-1 done
      if (good) {
        tc_fence_after();
        if (tid == 0 && t + 1 < n_t) {
          issue_kv(t + 1, st ^ 1);
          ++kv_issued;
        }

        // Online softmax on this thread's row, in raw logit units for the
        // maximum (scale > 0) and base 2 for the exponentials.
        float x[kKT];
#pragma unroll
        for (int cb = 0; cb < kKT / 32; ++cb) {
          uint32_t r[32];
          tmem_ld32(tmem_s + lane_off + cb * 32, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) x[cb * 32 + j] = __uint_as_float(r[j]);
        }
        const int kv0 = t * kKT;
        if (kv0 + kKT - 1 > pos_min) {  // tile reaches the diagonal (or the context end)
          const int lim = min(qpos, c - 1) - kv0;   // last visible column of this row
#pragma unroll
          for (int j = 0; j < kKT; ++j)
            if (j > lim) x[j] = -INFINITY;
        }
        float mx = m;
#pragma unroll
        for (int j = 0; j < kKT; j += 2) mx = fmax3(mx, x[j], x[j + 1]);
        const float alpha = (mx == -INFINITY) ? 1.f : exp2_approx((m - mx) * a.scale_log2);
        const float neg = (mx == -INFINITY) ? 0.f : -mx * a.scale_log2;
        float ps = 0.f;
        unsigned char* prow = sm + T::OFF_P;
#pragma unroll
        for (int j8 = 0; j8 < kKT / 8; ++j8) {
          uint32_t w[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float p0 = exp2_approx(fmaf(x[8 * j8 + 2 * u], a.scale_log2, neg));
            const float p1 = exp2_approx(fmaf(x[8 * j8 + 2 * u + 1], a.scale_log2, neg));
            ps += p0 + p1;
            const __half2 hp = __floats2half2_rn(p0, p1);
            w[u] = *reinterpret_cast<const uint32_t*>(&hp);
          }
          const int at = j8 / 8, ch = j8 % 8;
          *reinterpret_cast<uint4*>(prow + at * T::ATOM + swz128(tid, ch)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
        l = l * alpha + ps;
        m = mx;
        // Rescale this row of O when the maximum grew (warp-collective access).
        if (t > 0 && __any_sync(kFullMask, alpha != 1.f)) {
#pragma unroll
          for (int cb = 0; cb < D / 32; ++cb) {
            uint32_t r[32];
            tmem_ld32(tmem_o + lane_off + cb * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tmem_st32(tmem_o + lane_off + cb * 32, r);
          }
          tmem_wait_st();
        }
        // Zero V rows past the context (stale slots may hold anything).
        if (kv0 + tid >= c) {
          unsigned char* vrow = sm + (vaddr - s_base) + tid * 128;
#pragma unroll
          for (int at = 0; at < T::NA; ++at)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vrow + at * T::ATOM + ch * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      good = __syncthreads_and(good) != 0;
      tc_fence_after();
      if (!good) break;

      // O += P V
      if (tid == 0) {
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k) {
          const int at = k / 4, kk = k % 4;
          const uint64_t da = umma_desc_sw128(s_base + T::OFF_P + at * T::ATOM + kk * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(vaddr + k * 16 * 128, T::ATOM, 1024);
          umma_f16(tmem_o, da, db, kIdPV, t > 0 || k > 0);
        }
        umma_commit(o_bar);
        ++pv_done;
      }
    }
    if (good) good = mbar_wait_bounded(o_bar, (n_t - 1) & 1);
    good = __syncthreads_and(good) != 0;
    if (!good) {
      if (tid == 0) {
        atomicOr(a.err, PA_ERRBIT_TIMEOUT);
        // Let every copy and MMA this CTA started finish (bounded) before
        // its TMEM and shared memory are released.
        for (int u = t; u < kv_issued; ++u) mbar_wait_bounded(kv_bar0 + 8 * (u & 1), (u >> 1) & 1);
        if (qk_done > 0) mbar_wait_bounded(s_bar, (qk_done - 1) & 1);
        if (pv_done > 0) mbar_wait_bounded(o_bar, (pv_done - 1) & 1);
      }
    } else {
      tc_fence_after();
      // Epilogue: O / l -> fp16 rows of the output.
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __half* orow = static_cast<__half*>(a.out) + ((size_t)(q0 + qt * kQT + tid) * H + h) * D;
#pragma unroll
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem_o + lane_off + cb * 32, r);
        tmem_wait_ld();
        if (tid < rows_valid) {
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
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
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

bool encode(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
            strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_prefill_t(const PrefillArgs& g, cudaStream_t stream) {
  using T = PrefillTraits<D>;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    T::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tq, tk, tv;
  const cuuint64_t qdims[3] = {(cuuint64_t)D, (cuuint64_t)g.num_heads, (cuuint64_t)g.num_query_tokens};
  const cuuint64_t qstr[2] = {(cuuint64_t)D * 2, (cuuint64_t)g.num_heads * D * 2};
  const cuuint32_t qbox[3] = {64, 1, (cuuint32_t)kQT};
  const long long rows = (long long)g.num_blocks * g.num_heads * g.block_size;
  const cuuint64_t kdims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  const cuuint64_t kstr[1] = {(cuuint64_t)D * 2};
  const cuuint32_t kbox[2] = {64, (cuuint32_t)g.block_size};
  if (!encode(&tq, g.query, 3, qdims, qstr, qbox) || !encode(&tk, g.key_cache, 2, kdims, kstr, kbox) ||
      !encode(&tv, g.value_cache, 2, kdims, kstr, kbox))
    return cudaErrorInvalidValue;
  PrefillParams p{};
  p.out = g.out;
  p.block_tables = g.block_tables;
  p.context_lens = g.context_lens;
  p.query_start = g.query_start;
  p.err = g.err;
  p.num_seqs = g.num_seqs;
  p.num_heads = g.num_heads;
  p.max_blocks = g.max_blocks;
  p.num_blocks = g.num_blocks;
  p.block_size = g.block_size;
  p.qtiles = (g.max_query_len + kQT - 1) / kQT;
  p.max_query_len = g.max_query_len;
  p.oob_row = (int)rows;
  p.scale_log2 = g.scale_log2;
  const long long grid = (long long)g.num_seqs * p.qtiles * g.num_heads;
  return launch_pdl(prefill_kernel<D>, dim3((unsigned)grid), dim3(128), (size_t)T::SMEM, stream, tq,
                    tk, tv, p);
}

}  // namespace

bool prefill_rows_fit(int num_blocks, int num_heads, int block_size) {
  return (long long)num_blocks * num_heads * block_size < (1LL << 31) - 1;
}

cudaError_t launch_prefill(const PrefillArgs& g, cudaStream_t stream) {
  if (g.num_seqs == 0 || g.max_query_len == 0) return cudaSuccess;
  return g.head_dim == 64 ? launch_prefill_t<64>(g, stream) : launch_prefill_t<128>(g, stream);
}

}  // namespace pa
