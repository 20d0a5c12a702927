"""The synthetic workloads: shapes, context-length mixes and block orders.

All five are LLaMA-shaped paged-decode batches in fp16 with the cache laid
out as [num_blocks, num_heads, block_size, head_dim] per layer.  Discrete
structure is drawn in a fixed order from one SplitMix64 stream seeded with
``158000 + config_id``: context lengths (or suffix lengths) first, then the
physical block order.  Values come from ``synth`` banks seeded the same way.

Block tables for workloads 1, 2, 3 and 5 are static assignments: each
sequence takes its ceil(c/B) blocks in order from a seeded permutation of the
pool (plain structure of the input, like a sparsity pattern).  Workload 4's
tables are not drawn here: its prefix sharing and copy-on-write are the block
manager's job, so this module only supplies the prefix length, the suffix
lengths and the free-list order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import synth

SEED_BASE = 158000
POOL_CAP_BYTES = 120 * 10 ** 9


@dataclass
class Workload:
    name: str
    config_id: int
    seed: int
    num_layers: int
    num_seqs: int
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    context_lens: np.ndarray              # int32 [S]
    block_tables: np.ndarray | None       # int32 [S, max_blocks_per_seq], -1 padded
    kv_sigma: float = 1.0
    q_sigma: float = 1.0
    # Workload 4 (shared prefix): inputs for the block manager.
    prefix_len: int = 0
    suffix_lens: np.ndarray | None = None
    free_order: np.ndarray | None = None
    description: str = ""
    extra: dict = field(default_factory=dict)
    logit_scale: float | None = None      # the attention scale if not 1/sqrt(head_dim)

    @property
    def scale(self) -> float:
        return self.logit_scale if self.logit_scale is not None else 1.0 / math.sqrt(self.head_dim)

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if len(self.context_lens) else 0

    @property
    def tile_elems(self) -> int:
        """fp16 elements of one physical block across all heads."""
        return self.num_heads * self.block_size * self.head_dim

    @property
    def pool_elems(self) -> int:
        return self.num_blocks * self.tile_elems

    def pool_bytes_all_layers(self) -> int:
        return self.num_layers * 2 * self.pool_elems * 2

    # Streams of the value generator.
    def key_pool_stream(self, layer: int) -> int:
        return synth.stream_id(layer, synth.KEY_POOL)

    def value_pool_stream(self, layer: int) -> int:
        return synth.stream_id(layer, synth.VALUE_POOL)

    def query_stream(self, layer: int) -> int:
        return synth.stream_id(layer, synth.QUERY)

    def key_new_stream(self, layer: int) -> int:
        return synth.stream_id(layer, synth.KEY_NEW)

    def value_new_stream(self, layer: int) -> int:
        return synth.stream_id(layer, synth.VALUE_NEW)

    def kv_bank(self) -> np.ndarray:
        return synth.fp16_bank(self.seed, self.kv_sigma)

    def q_bank(self) -> np.ndarray:
        return synth.fp16_bank(self.seed, self.q_sigma)

    def new_tokens(self):
        """(token_seq, token_pos) of the tokens written by the cache-write step.

        Decode workloads write one token per sequence at position c_s - 1 (the
        context length counts the token just written).  Workload 4 writes its
        whole suffix, sequence by sequence.
        """
        if self.suffix_lens is not None:
            seqs = np.repeat(np.arange(self.num_seqs, dtype=np.int32), self.suffix_lens)
            pos = np.concatenate([self.prefix_len + np.arange(n, dtype=np.int32)
                                  for n in self.suffix_lens]).astype(np.int32)
            return seqs, pos
        live = self.context_lens > 0
        seqs = np.arange(self.num_seqs, dtype=np.int32)[live]
        return seqs, (self.context_lens[live] - 1).astype(np.int32)


def _tables_from_permutation(perm: np.ndarray, ctx: np.ndarray, block_size: int,
                             max_blocks: int) -> np.ndarray:
    bt = np.full((len(ctx), max_blocks), -1, dtype=np.int32)
    off = 0
    for s, c in enumerate(ctx):
        nb = -(-int(c) // block_size)
        bt[s, :nb] = perm[off:off + nb]
        off += nb
    return bt


def config1() -> Workload:
    """Tiny single-layer decode: S4 H8 D64 B4, c ~ U{1..64}, 128-block pool."""
    cid = 1
    seed = SEED_BASE + cid
    d = synth.Draws(seed)
    S, H, D, B, NB = 4, 8, 64, 4, 128
    ctx = np.array([d.integer(1, 64) for _ in range(S)], dtype=np.int32)
    perm = d.permutation(NB)
    mb = 64 // B
    return Workload("c1_tiny_S4_H8_D64_B4", cid, seed, 1, S, H, D, B, NB, mb, ctx,
                    _tables_from_permutation(perm, ctx, B, mb),
                    description="tiny single-layer decode, pool of 128 blocks")


def config2() -> Workload:
    """LLaMA-7B-shaped single layer: S32 H32 D128 B16, c ~ U{200..500}, pool 2x need."""
    cid = 2
    seed = SEED_BASE + cid
    d = synth.Draws(seed)
    S, H, D, B = 32, 32, 128, 16
    ctx = np.array([d.integer(200, 500) for _ in range(S)], dtype=np.int32)
    need = int(sum(-(-int(c) // B) for c in ctx))
    NB = 2 * need
    perm = d.permutation(NB)
    mb = -(-500 // B)
    return Workload("c2_llama7b_S32_H32_D128_B16", cid, seed, 1, S, H, D, B, NB, mb, ctx,
                    _tables_from_permutation(perm, ctx, B, mb),
                    description="7B-shaped single-layer decode, random non-contiguous tables")


def config3(num_layers: int = 40) -> Workload:
    """LLaMA-13B-shaped: 40 layers x (S32 H40 D128 B16, c = 1024), K/V ~ 0.5 N(0,1)."""
    cid = 3
    seed = SEED_BASE + cid
    d = synth.Draws(seed)
    S, H, D, B, c = 32, 40, 128, 16, 1024
    ctx = np.full(S, c, dtype=np.int32)
    NB = S * (c // B)
    perm = d.permutation(NB)
    mb = c // B
    return Workload("c3_llama13b_L40_S32_H40_D128_B16_c1024", cid, seed, num_layers, S, H, D, B,
                    NB, mb, ctx, _tables_from_permutation(perm, ctx, B, mb), kv_sigma=0.5,
                    description="13B-shaped decode step over 40 layers, shuffled blocks")


def config4() -> Workload:
    """Shared 520-token prefix + per-sequence suffix U{1..1536}: S64 H32 D128 B16."""
    cid = 4
    seed = SEED_BASE + cid
    d = synth.Draws(seed)
    S, H, D, B, prefix = 64, 32, 128, 16, 520
    suffix = np.array([d.integer(1, 1536) for _ in range(S)], dtype=np.int32)
    ctx = (prefix + suffix).astype(np.int32)
    prefix_blocks = -(-prefix // B)                      # 33: 32 full + 1 partial
    own = int(sum(-(-int(c) // B) - prefix_blocks for c in ctx))
    copies = S - 1 if prefix % B else 0                  # writers of the shared partial block
    NB = prefix_blocks + copies + own
    free_order = d.permutation(NB)
    mb = -(-(prefix + 1536) // B)
    return Workload("c4_shared_prefix_S64_H32_D128_B16", cid, seed, 1, S, H, D, B, NB, mb, ctx,
                    None, prefix_len=prefix, suffix_lens=suffix, free_order=free_order,
                    description="shared-prefix decode with copy-on-write")


def config5(num_layers: int = 32, sigma: float = 0.75) -> Workload:
    """Long-context skewed: 32 layers x (S256 H32 D128 B32), c log-normal, median 600."""
    cid = 5
    seed = SEED_BASE + cid
    d = synth.Draws(seed)
    S, H, D, B = 256, 32, 128, 32
    ctx = np.array([min(4096, max(16, math.floor(math.exp(math.log(600.0) + sigma * d.normal())
                                                     + 0.5))) for _ in range(S)], dtype=np.int32)
    NB = int(sum(-(-int(c) // B) for c in ctx))
    perm = d.permutation(NB)
    mb = 4096 // B
    w = Workload("c5_longctx_L32_S256_H32_D128_B32_lognormal600", cid, seed, num_layers, S, H, D,
                 B, NB, mb, ctx, _tables_from_permutation(perm, ctx, B, mb),
                 description=f"long-context skewed batch, log-normal sigma={sigma}")
    if w.pool_bytes_all_layers() > POOL_CAP_BYTES:
        raise ValueError(f"workload 5 pool {w.pool_bytes_all_layers() / 1e9:.1f} GB exceeds the "
                         f"{POOL_CAP_BYTES / 1e9:.0f} GB cap")
    return w


def small_random(seed: int, num_seqs: int, num_heads: int, head_dim: int, block_size: int,
                 max_context: int, min_context: int = 0, spare_blocks: int = 3,
                 kv_sigma: float = 1.0, q_sigma: float = 1.0) -> Workload:
    """A small random paged batch: c ~ U{min..max}, tables from a permutation of a pool
    with a few spare blocks."""
    d = synth.Draws(seed)
    ctx = np.array([d.integer(min_context, max_context) for _ in range(num_seqs)], dtype=np.int32)
    need = int(sum(-(-int(c) // block_size) for c in ctx))
    NB = need + spare_blocks
    perm = d.permutation(NB)
    mb = max(1, -(-max_context // block_size))
    return Workload(f"rand_S{num_seqs}_H{num_heads}_D{head_dim}_B{block_size}_c{max_context}", 0,
                    seed, 1, num_seqs, num_heads, head_dim, block_size, NB, mb, ctx,
                    _tables_from_permutation(perm, ctx, block_size, mb), kv_sigma=kv_sigma,
                    q_sigma=q_sigma)


def prefill_workload(name: str, seed: int, q_lens, ctx, num_heads: int, head_dim: int,
                     block_size: int, spare_blocks: int = 3, kv_sigma: float = 1.0,
                     q_sigma: float = 1.0, cid: int = 0) -> Workload:
    """A chunked-prefill / mixed batch on one layer: sequence s has ctx[s] cached tokens,
    the last q_lens[s] of which are its new query tokens (q_lens[s] == 1: decode).
    Blocks come from a seeded permutation of a pool with a few spare blocks."""
    d = synth.Draws(seed)
    ctx = np.asarray(ctx, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    need = int(sum(-(-int(c) // block_size) for c in ctx))
    NB = need + spare_blocks
    perm = d.permutation(NB)
    mb = max(1, -(-int(ctx.max()) // block_size))
    return Workload(name, cid, seed, 1, len(ctx), num_heads, head_dim, block_size, NB, mb, ctx,
                    _tables_from_permutation(perm, ctx, block_size, mb), kv_sigma=kv_sigma,
                    q_sigma=q_sigma, description="chunked prefill / mixed batch",
                    extra={"q_lens": q_lens})


def query_start(w: Workload) -> np.ndarray:
    """int32 [S + 1]: prefix sums of the prefill workload's chunk lengths."""
    return np.concatenate([[0], np.cumsum(w.extra["q_lens"])]).astype(np.int32)


def prefill_7b() -> Workload:
    """LLaMA-7B-shaped chunked prefill: 4 sequences x a 512-token chunk after a 1536-token
    cached prefix (context 2048), H32 D128 B16."""
    return prefill_workload("p1_chunked_prefill_S4_H32_D128_B16_q512_c2048", SEED_BASE + 6,
                            [512] * 4, [2048] * 4, 32, 128, 16, spare_blocks=0, cid=6)


def prefill_7b_mixed() -> Workload:
    """LLaMA-7B-shaped mixed batch: 2 sequences with a 512-token chunk after a 1536-token
    cached prefix (context 2048) and 64 decode sequences (one new token each, contexts
    U{512..2048}), H32 D128 B16."""
    d = synth.Draws(SEED_BASE + 7)
    dec_ctx = [d.integer(512, 2048) for _ in range(64)]
    return prefill_workload("p2_mixed_S66_H32_D128_B16_q2x512_64x1", SEED_BASE + 7,
                            [512] * 2 + [1] * 64, [2048] * 2 + dec_ctx, 32, 128, 16,
                            spare_blocks=0, cid=7)


def fp8_scales(w: Workload) -> tuple[float, float]:
    """Per-tensor scales (k_scale, v_scale) of a workload's FP8 caches: about
    1/70 and 1/84 of the values' standard deviation, so that values up to
    about 6 and 5.3 sigma lie inside E4M3's finite range (448) and the rare
    larger ones saturate.  Two different, non-power-of-two values, rounded to
    binary32 (the type the library takes)."""
    k = float(np.float32(w.kv_sigma * 0.0137))
    v = float(np.float32(w.kv_sigma * 0.0119))
    return k, v


ALL = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}
