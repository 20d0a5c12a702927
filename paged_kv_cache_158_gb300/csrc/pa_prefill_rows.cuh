// Work units of the multi-query attention kernel, and its CUDA-core path for
// one-token rows.
//
// Units.  A launch covers a window of sequences.  Sequence s with q_len new
// tokens contributes, for each head, ceil(q_len / 256) units of two 128-row
// query tiles (tensor cores), or decode-row units when q_len == 1 (run on
// CUDA cores: "vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §4.3,
// prefill and decode rows share a batch), or none when q_len == 0.  Units are
// numbered densely, so a batch of many decode rows and a few chunks launches
// (almost) no CTA without work:
//   * chunk groups (sequence, head), sequence-major, come first.  As many
//     whole groups as fit one CTA per SM come first, each group's pairs
//     adjacent and heaviest first (they share K/V tiles through L2); the
//     other groups follow rank by rank, every group's heaviest remaining pair
//     before any group's next one;
//   * the decode rows follow, sequence-major (RowSplit): one unit per head,
//     or, when the launch was sized from a known count of decode rows, one
//     unit per G = kMaxRowHeads heads of a row except for the last wave of
//     rows, which keeps one unit per head so that the launch ends on short
//     units.
// Every CTA derives its unit from query_start: up to 32 sequences on one
// warp, more with the whole block (one pass writes a per-sequence table to
// shared memory, pairs or kDecodeRowKind, then weighted selections over it,
// block-wide scans, find the unit).
//
// Decode rows.  A unit of nh heads runs on the CTA's twelve warps, 12 / nh
// per head: warp w takes head w mod nh and every (12 / nh)-th 16-token chunk
// of its context, and runs the decode kernel's per-chunk step (fp32 online
// softmax over bulk-copied K/V rows).  Each warp owns a ring of
// shared-memory stages with one mbarrier per stage; lane 0 copies a chunk's
// K rows and V rows with 1-D bulk copies.  The heads of a unit advance
// through the row's blocks side by side, so their K/V tiles, neighbours in
// the [block][head] layout, are read together.  At the end each head's
// warps merge their (m, l, o) in shared memory and the CTA writes the heads'
// fp16 outputs.  No workspace, no merge kernel; the hardware's CTA dispatch
// balances rows of different lengths.  Grouping heads spreads one plan, one
// start-up latency and one CTA turnover (together about 6 us against about
// 6 us of streaming for one head of a 1300-token FP8 row) over four heads.
#pragma once

#include "pa_decode.cuh"

namespace pa {
namespace prows {

constexpr int kDecodeRowKind = -1;  // table entry of a one-token row (CUDA-core path)
constexpr int kNW = 12;             // warps per CTA
constexpr int kThreads = kNW * 32;
constexpr int kRowWarps = 12;       // warps that run a decode row
constexpr int kMaxRowHeads = 4;     // most heads of one decode-row unit
static_assert(kRowWarps % 2 == 0 && kRowWarps % 3 == 0 && kRowWarps % 4 == 0,
              "every head count up to kMaxRowHeads divides the row warps");

// Exclusive scan of one int per thread over the block; *total gets the sum.
// scratch[0..11] is used; ends with a barrier, so scratch may be reused.
__device__ __forceinline__ int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kNW; ++w) {
    const int t = scratch[w];
    if (w < warp) base += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return base + x - v;
}

// Sum over the table of weight(i, table[i]).
template <class W>
__device__ __forceinline__ int block_sum(const int* table, int n, W weight, int* scratch) {
  int local = 0;
  for (int i = threadIdx.x; i < n; i += kThreads) local += weight(i, table[i]);
  int total;
  block_exclusive_scan(local, scratch, &total);
  return total;
}

// Weighted selection: the first index i whose inclusive prefix of
// weight(i, table[i]) exceeds target, and target minus the prefix before it;
// (n, target - total) when the total does not exceed target.
template <class W>
__device__ __forceinline__ int2 block_select(const int* table, int n, int target, W weight,
                                             int* scratch) {
  const int per = (n + kThreads - 1) / kThreads;
  const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
  int local = 0;
  for (int i = i0; i < i1; ++i) local += weight(i, table[i]);
  int total;
  const int base = block_exclusive_scan(local, scratch, &total);
  if (target >= base && target < base + local) {
    int acc = base;
    for (int i = i0; i < i1; ++i) {
      const int w = weight(i, table[i]);
      if (target < acc + w) {
        scratch[16] = i;
        scratch[17] = target - acc;
        break;
      }
      acc += w;
    }
  }
  if (threadIdx.x == 0 && target >= total) {
    scratch[16] = n;
    scratch[17] = target - total;
  }
  __syncthreads();
  const int2 r = make_int2(scratch[16], scratch[17]);
  __syncthreads();
  return r;
}

struct Unit {
  int kind;  // 0: none (past the launch's units), 1: pair of query tiles, 2: decode row
  int s;     // sequence within the launch
  int h;     // head (kind 1); first head (kind 2)
  int pq;    // pair of query tiles (kind 1)
  int q0;    // the sequence's first query row, its query length and context length
  int q_len;
  int c;
  int nh;    // heads h .. h + nh - 1 (kind 2)
};

// Decode-row units.  With G heads per unit (G > 1) the rows come first in
// units of G heads (a row's last unit may hold fewer), except the last
// `tail` rows, which take one unit per head so that the launch ends on short
// units; with G == 1 every row is one unit per head.  nd: the launch's decode
// rows; sms: the SM count.
struct RowSplit {
  int ru;    // units of a grouped row
  int tail;  // rows at one unit per head
  int gu;    // units of the grouped rows
  __host__ __device__ RowSplit(int nd, int H, int G, int sms) {
    ru = (H + G - 1) / G;
    const int wave = (sms + H - 1) / H;  // rows that fill one wave at one unit per head
    tail = G == 1 ? nd : (nd < wave ? nd : wave);
    gu = (nd - tail) * ru;
  }
  __host__ __device__ int units(int H) const { return gu + tail * H; }
};

// Row unit rho (0 <= rho < RowSplit::units): the row's index among the
// launch's decode rows (sequence order), its first head and head count.
__device__ __forceinline__ int3 row_unit(const RowSplit& rs, int H, int G, int rho) {
  if (rho < rs.gu) {
    const int i = rho / rs.ru;
    const int h = (rho - i * rs.ru) * G;
    return make_int3(i, h, min(G, H - h));
  }
  rho -= rs.gu;
  const int i = rho / H;
  return make_int3(rs.gu / rs.ru + i, rho - i * H, 1);
}

// Table entry of a sequence with q new tokens: pairs of query tiles, a decode
// row, or nothing.  A negative length gets one unit, which reports it; a
// length beyond the call's max_query_len is clamped to qpairs pairs and
// reported by its unit.
__device__ __forceinline__ int table_entry(int q, int qpairs) {
  return q < 0 ? 1 : q == 1 ? kDecodeRowKind : min((q + 2 * 128 - 1) / (2 * 128), qpairs);
}

// Warp-wide selection over one weight per lane (lanes >= n hold 0): the first
// lane whose inclusive prefix exceeds target and target minus the prefix
// before it; (32, target - total) when the total does not exceed target.
__device__ __forceinline__ int2 warp_select(int w, int target) {
  const int lane = threadIdx.x & 31;
  int incl = w;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned m = __ballot_sync(kFullMask, target < incl);
  const int total = __shfl_sync(kFullMask, incl, 31);
  if (m == 0) return make_int2(32, target - total);
  const int l = __ffs(m) - 1;
  return make_int2(l, target - (__shfl_sync(kFullMask, incl, l) - __shfl_sync(kFullMask, w, l)));
}

// The unit order of plan_unit for at most 32 sequences, on one warp (lane i
// holds sequence i's table entry k).  G: heads per decode-row unit.
__device__ __forceinline__ Unit plan_unit_warp(int k, int H, int G, int qpairs, int sms, int b,
                                               int* total_units) {
  Unit u{0, 0, 0, 0, 0, 0, 0, 0};
  const int lane = threadIdx.x & 31;
  const int cu = __reduce_add_sync(kFullMask, k > 0 ? H * k : 0);
  const int nd = __reduce_add_sync(kFullMask, k == kDecodeRowKind ? 1 : 0);
  const RowSplit rs(nd, H, G, sms);
  *total_units = cu + rs.units(H);
  if (b >= cu + rs.units(H)) return u;
  if (b >= cu) {
    const int3 r = row_unit(rs, H, G, b - cu);
    u.kind = 2;
    u.s = warp_select(k == kDecodeRowKind ? 1 : 0, r.x).x;
    u.h = r.y;
    u.nh = r.z;
    return u;
  }
  const int wu = k > 0 ? H * k : 0;
  const int2 w = warp_select(wu, sms);
  int u1, s_w, g_w;
  if (w.x >= 32) {
    u1 = cu;
    s_w = 32;
    g_w = 0;
  } else {
    const int kw = __shfl_sync(kFullMask, k, w.x);
    g_w = w.y / kw;
    s_w = w.x;
    u1 = (sms - w.y) + g_w * kw;
  }
  if (b < u1) {
    const int2 r = warp_select(wu, b);
    const int kr = __shfl_sync(kFullMask, k, r.x);
    u.kind = 1;
    u.s = r.x;
    u.h = r.y / kr;
    u.pq = kr - 1 - r.y % kr;
    return u;
  }
  int t = b - u1;
  for (int rank = 0; rank < qpairs; ++rank) {
    const int wr = k <= rank ? 0 : lane < s_w ? 0 : lane == s_w ? H - g_w : H;
    const int cnt = __reduce_add_sync(kFullMask, wr);
    if (t < cnt) {
      const int2 r = warp_select(wr, t);
      u.kind = 1;
      u.s = r.x;
      u.h = r.x == s_w ? g_w + r.y : r.y;
      u.pq = __shfl_sync(kFullMask, k, r.x) - 1 - rank;
      return u;
    }
    t -= cnt;
  }
  return u;
}

// plan_unit_warp's order in closed form for a launch whose nseq sequences all
// have the same k > 0 pairs (fixed-size chunks): the first wave's whole
// groups, then rank by rank, with integer arithmetic instead of warp-wide
// selections (every lane computes the same unit).
__device__ __forceinline__ Unit plan_unit_uniform(int nseq, int k, int H, int sms, int b,
                                                  int* total_units) {
  Unit u{0, 0, 0, 0, 0, 0, 0, 0};
  const int G = H * k;  // units of one sequence
  const int cu = nseq * G;
  *total_units = cu;
  if (b >= cu) return u;
  int u1, s_w, g_w;  // units of the first wave; its last sequence and whole groups in it
  const int s = sms / G;
  if (s >= nseq) {
    u1 = cu;
    s_w = nseq;
    g_w = 0;
  } else {
    g_w = (sms - s * G) / k;
    s_w = s;
    u1 = s * G + g_w * k;
  }
  u.kind = 1;
  if (b < u1) {
    u.s = b / G;
    const int r = b - u.s * G;
    u.h = r / k;
    u.pq = k - 1 - r % k;
    return u;
  }
  // Rank r: the remaining groups' pair k - 1 - r (H - g_w groups of sequence s_w, then H
  // of each later sequence).
  const int per_rank = (H - g_w) + (nseq - s_w - 1) * H;
  int t = b - u1;
  const int rank = t / per_rank;
  t -= rank * per_rank;
  u.pq = k - 1 - rank;
  if (t < H - g_w) {
    u.s = s_w;
    u.h = g_w + t;
  } else {
    t -= H - g_w;
    u.s = s_w + 1 + t / H;
    u.h = t % H;
  }
  return u;
}

// This CTA's unit over many sequences: the table in shared memory and
// block-wide selections.  Every thread calls it (block barriers inside).
__device__ __forceinline__ Unit plan_unit_table(const int32_t* qs, int nseq, int H, int G,
                                               int qpairs, int sms, int b, int* table,
                                               int* scratch, int* total_units) {
  for (int i = threadIdx.x; i < nseq; i += kThreads) table[i] = table_entry(qs[i + 1] - qs[i], qpairs);
  __syncthreads();
  auto chunk_units = [H](int, int k) { return k > 0 ? H * k : 0; };
  const int cu = block_sum(table, nseq, chunk_units, scratch);
  const int nd = block_sum(table, nseq, [](int, int k) { return k == kDecodeRowKind ? 1 : 0; },
                           scratch);
  Unit u{0, 0, 0, 0, 0, 0, 0, 0};
  const RowSplit rs(nd, H, G, sms);
  *total_units = cu + rs.units(H);
  if (b >= cu + rs.units(H)) return u;
  if (b >= cu) {  // a decode row
    const int3 r = row_unit(rs, H, G, b - cu);
    u.kind = 2;
    u.s = block_select(table, nseq, r.x, [](int, int k) { return k == kDecodeRowKind ? 1 : 0; },
                       scratch).x;
    u.h = r.y;
    u.nh = r.z;
    return u;
  }
  // Chunk pairs.  First wave: the whole groups whose pairs fit one CTA per SM.
  const int2 w = block_select(table, nseq, sms, chunk_units, scratch);
  int u1, s_w, g_w;  // units of the first wave; its last sequence and whole groups in it
  if (w.x >= nseq) {
    u1 = cu;
    s_w = nseq;
    g_w = 0;
  } else {
    const int k = table[w.x];
    g_w = w.y / k;
    s_w = w.x;
    u1 = (sms - w.y) + g_w * k;
  }
  if (b < u1) {
    const int2 r = block_select(table, nseq, b, chunk_units, scratch);
    const int k = table[r.x];
    u.kind = 1;
    u.s = r.x;
    u.h = r.y / k;
    u.pq = k - 1 - r.y % k;
    return u;
  }
  // Later groups, rank by rank: rank r holds each remaining group with more
  // than r pairs (its pair k - 1 - r).
  int t = b - u1;
  for (int rank = 0; rank < qpairs; ++rank) {
    auto in_rank = [H, rank, s_w, g_w](int i, int k) {
      if (k <= rank) return 0;
      return i < s_w ? 0 : i == s_w ? H - g_w : H;
    };
    const int cnt = block_sum(table, nseq, in_rank, scratch);
    if (t < cnt) {
      const int2 r = block_select(table, nseq, t, in_rank, scratch);
      u.kind = 1;
      u.s = r.x;
      u.h = r.x == s_w ? g_w + r.y : r.y;
      u.pq = table[r.x] - 1 - rank;
      return u;
    }
    t -= cnt;
  }
  return u;  // not reached for a consistent table
}

// plan_unit_table with the unit's query rows and context length.
__device__ __noinline__ Unit plan_unit_block(const int32_t* qs, const int32_t* ctx, int nseq,
                                             int H, int G, int qpairs, int sms, int b, int* table,
                                             int* scratch, int* total_units) {
  Unit u = plan_unit_table(qs, nseq, H, G, qpairs, sms, b, table, scratch, total_units);
  if (u.kind != 0) {
    u.q0 = qs[u.s];
    u.q_len = qs[u.s + 1] - u.q0;
    u.c = ctx[u.s];
  }
  return u;
}

// This CTA's unit for at most 32 sequences, on one warp (the caller's warp;
// no block barrier): written to *res with its sequence's query rows and
// context length, and the launch's unit count to *total_units.  qs, ctx:
// query_start and context_lens of the launch's first sequence.
__device__ __noinline__ void plan_small(const int32_t* qs, const int32_t* ctx, int nseq, int H,
                                        int G, int qpairs, int sms, int b, Unit* res,
                                        int* total_units) {
  const int lane = threadIdx.x & 31;
  int q0 = 0, q1 = 0, c = 0;
  if (lane < nseq) {
    q0 = qs[lane];
    q1 = qs[lane + 1];
    c = ctx[lane];
  }
  const int k = lane < nseq ? table_entry(q1 - q0, qpairs) : 0;
  int tot = 0;
  const int kmin = __reduce_min_sync(kFullMask, lane < nseq ? k : 0x7fffffff);
  const int kmax = __reduce_max_sync(kFullMask, lane < nseq ? k : -0x7fffffff);
  Unit u = kmin == kmax && kmin > 0 ? plan_unit_uniform(nseq, kmin, H, sms, b, &tot)
                                    : plan_unit_warp(k, H, G, qpairs, sms, b, &tot);
  const int src = u.kind != 0 ? u.s : 0;
  u.q0 = __shfl_sync(kFullMask, q0, src);
  u.q_len = __shfl_sync(kFullMask, q1, src) - u.q0;
  u.c = __shfl_sync(kFullMask, c, src);
  if (lane == 0) {
    *res = u;
    *total_units = tot;
  }
}

// Stages per warp for the decode-row rings in the `area` bytes of shared
// memory the rows may use: as many as fit, at most 4.
template <int D, int TCB, bool F8>
constexpr int row_stages(int area) {
  return area / (kRowWarps * DecodeTraits<D, TCB, F8>::STAGE_BYTES) >= 4
             ? 4
             : area / (kRowWarps * DecodeTraits<D, TCB, F8>::STAGE_BYTES);
}

// One decode row (query/output row q0, context length c) for the nh heads
// h0 .. h0 + nh - 1 (nh divides kRowWarps) on kRowWarps warps: warp w runs
// head w mod nh, chunk w / nh, w / nh + kRowWarps / nh, ... of it.  So the
// heads advance through the row's blocks side by side and their K/V tiles
// (neighbours in the [block][head] layout) are read together.  ring: shared
// memory of at least kRowWarps * NST * STAGE_BYTES bytes; bars: kRowWarps *
// NST initialised mbarriers (count 1); pw: kRowWarps * 16 floats; fail: a
// shared flag.  Every thread of the CTA calls it (one block barrier inside).
template <int D, int TCB, bool F8, int NST>
__device__ __noinline__ void decode_row(const void* query, const void* key_cache,
                                        const void* value_cache, const int32_t* bt, int num_heads,
                                        int block_size, int num_blocks, float scale_log2,
                                        float v_scale, unsigned int* err, void* out, int h0,
                                        int nh, int q0, int c, unsigned char* ring,
                                        uint64_t* bars, float* pw, int* fail) {
  using T = DecodeTraits<D, TCB, F8>;
  static_assert(NST >= 2 && NST <= 4, "stages");
  constexpr int PR = T::TC / T::BPC;   // rows per piece (a piece lies in one block)
  constexpr int PPW = 32 / T::BPC;     // chunks one warp-wide id load covers
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool leader = lane == 0;
  const int B = block_size, H = num_heads;
  const int wph = kRowWarps / nh;      // warps per head
  const int g = warp % nh, wi = warp / nh;
  const int h = h0 + g;
  const int n_chunks = (c + T::TC - 1) / T::TC;
  const int n_my = wi < n_chunks ? (n_chunks - 1 - wi) / wph + 1 : 0;
  const uint64_t policy = policy_evict_first();
  const uint32_t ring_s = smem_u32(ring) + (uint32_t)(warp * NST * T::STAGE_BYTES);
  const uint32_t bar_s = smem_u32(bars) + (uint32_t)(warp * NST * 8);
  const unsigned char* kc = static_cast<const unsigned char*>(key_cache);
  const unsigned char* vc = static_cast<const unsigned char*>(value_cache);

  // Block ids of this warp's chunks k in [base, base + PPW): lane L holds the
  // id of piece L % BPC of chunk base + L / BPC (-1 past the live rows).
  auto load_ids = [&](int base) {
    const int k = base + lane / T::BPC;
    int id = -1;
    if (k < n_my) {
      const int t = (wi + k * wph) * T::TC + (lane % T::BPC) * PR;
      if (t < c) id = bt[t / B];
    }
    return id;
  };
  int id_base = 0;
  int ids_cur = load_ids(0);
  int ids_next = load_ids(PPW);
  uint32_t valid = 0;  // bit st: the chunk in stage st had valid ids

  // Warp-uniform; lane 0 issues.  Chunk k of this warp into stage st.
  auto issue = [&](int k, int st) {
    if (k - id_base >= 2 * PPW) {
      id_base += PPW;
      ids_cur = ids_next;
      ids_next = load_ids(id_base + PPW);
    }
    const int t0 = (wi + k * wph) * T::TC;
    const int rows = min(T::TC, c - t0);
    const int wsel = (k - id_base) / PPW;
    const int src = ((k - id_base) % PPW) * T::BPC;
    int ph[T::BPC];
    bool ok = true;
#pragma unroll
    for (int p = 0; p < T::BPC; ++p) {
      const int a0 = __shfl_sync(kFullMask, ids_cur, src + p);
      const int a1 = __shfl_sync(kFullMask, ids_next, src + p);
      ph[p] = wsel ? a1 : a0;
      if (p * PR < rows && (ph[p] < 0 || ph[p] >= num_blocks)) ok = false;
    }
    const uint32_t bar = bar_s + 8 * st;
    if (!ok) {
      if (leader) atomicOr(err, PA_ERRBIT_BLOCK_ID);
      mbar_arrive_if(leader, bar);  // completes the phase with no data; the chunk is skipped
      valid &= ~(1u << st);
      return;
    }
    valid |= 1u << st;
    mbar_arrive_expect_tx_if(leader, bar, 2u * (uint32_t)rows * D * T::ELEM);
    const uint32_t stage = ring_s + (uint32_t)(st * T::STAGE_BYTES);
#pragma unroll
    for (int p = 0; p < T::BPC; ++p) {
      const int r = min(PR, rows - p * PR);
      if (r <= 0) break;
      const int tok = t0 + p * PR;
      const size_t off = (((size_t)ph[p] * H + h) * B + tok % B) * D * T::ELEM;
      const uint32_t bytes = (uint32_t)r * D * T::ELEM;
      const uint32_t soff = (uint32_t)(p * PR * D * T::ELEM);
      bulk_g2s_hint_if(leader, stage + soff, kc + off, bytes, bar, policy);
      bulk_g2s_hint_if(leader, stage + T::CHUNK_BYTES + soff, vc + off, bytes, bar, policy);
    }
  };

  int iss = 0;
  for (; iss < n_my && iss < NST; ++iss) issue(iss, iss);

  const int cidx = lane % T::LR;
  const int rgrp = lane / T::LR;
  QSlice<T::DPL> q;
#pragma unroll
  for (int j = 0; j < T::DPL / 8; ++j)
    q.v[j] = *reinterpret_cast<const uint4*>(static_cast<const __half*>(query) +
                                             ((size_t)q0 * H + h) * D + T::DPL * cidx + 8 * j);
  float m = -INFINITY, l = 0.f;
  float o[T::DPL];
#pragma unroll
  for (int i = 0; i < T::DPL; ++i) o[i] = 0.f;
  float* my_pw = pw + warp * 16;

  for (int k = 0; k < n_my; ++k) {
    const int st = k % NST;
    const bool ok = __all_sync(kFullMask, mbar_wait_bounded(bar_s + 8 * st, (uint32_t)(k / NST) & 1));
    if (!ok) {
      // Let this warp's other copies in flight land (bounded), then give up.
      for (int i = k + 1; i < iss; ++i)
        mbar_wait_bounded(bar_s + 8 * (i % NST), (uint32_t)(i / NST) & 1);
      if (leader) {
        atomicOr(err, PA_ERRBIT_TIMEOUT);
        *fail = 1;
      }
      break;
    }
    if (valid & (1u << st)) {
      const int rows = min(T::TC, c - (wi + k * wph) * T::TC);
      const unsigned char* Ks = ring + (size_t)(warp * NST + st) * T::STAGE_BYTES;
      if (rows == T::TC)
        process_chunk<D, TCB, F8, true>(Ks, Ks + T::CHUNK_BYTES, rows, q, scale_log2, my_pw, lane,
                                        m, l, o);
      else
        process_chunk<D, TCB, F8, false>(Ks, Ks + T::CHUNK_BYTES, rows, q, scale_log2, my_pw, lane,
                                         m, l, o);
    }
    __syncwarp();
    if (iss < n_my) {  // stage st is free: the chunk NST ahead goes into it
      issue(iss, iss % NST);
      ++iss;
    }
  }

  // Combine the row groups, publish the warp's (m, l, o) in its own first
  // stage (all of its copies have landed), merge each head's warps, write the
  // heads' output rows (contiguous, like the query rows).
#pragma unroll
  for (int msk = T::LR; msk < 32; msk <<= 1) {
#pragma unroll
    for (int i = 0; i < T::DPL; ++i) o[i] += __shfl_xor_sync(kFullMask, o[i], msk);
  }
  __syncwarp();
  float* mw = reinterpret_cast<float*>(ring + (size_t)(warp * NST) * T::STAGE_BYTES);
  if (rgrp == 0) {
#pragma unroll
    for (int i = 0; i < T::DPL / 4; ++i)
      reinterpret_cast<float4*>(mw + T::DPL * cidx)[i] =
          make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
  if (leader) {
    mw[D] = m;
    mw[D + 1] = l;
  }
  __syncthreads();
  if (*fail != 0) return;
  auto slot = [&](int w) {
    return reinterpret_cast<const float*>(ring + (size_t)(w * NST) * T::STAGE_BYTES);
  };
  for (int i = tid; i < nh * D; i += kThreads) {
    const int gi = i / D, d = i - gi * D;
    float M = -INFINITY;
    for (int w = gi; w < kRowWarps; w += nh) M = fmaxf(M, slot(w)[D]);
    float L = 0.f, O = 0.f;
    for (int w = gi; w < kRowWarps; w += nh) {
      const float* mb = slot(w);
      const float sc = mb[D] == -INFINITY ? 0.f : exp2_approx(mb[D] - M);
      L = fmaf(sc, mb[D + 1], L);
      O = fmaf(sc, mb[d], O);
    }
    if constexpr (F8) O *= v_scale;
    const float r = (c > 0 && L > 0.f) ? O / L : 0.f;
    static_cast<__half*>(out)[((size_t)q0 * H + h0) * D + i] = __float2half_rn(r);
  }
}

}  // namespace prows
}  // namespace pa
