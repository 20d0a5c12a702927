"""Paged KV pool: device buffers and the host-side block manager.

The block manager is host bookkeeping, as in the pages' engine: it decides
which physical block every logical block of a sequence uses and when a
shared block must be copied.  It moves no data; the copies it asks for are
done on the GPU by pa_copy_blocks, the slots of new tokens are computed on
the GPU by pa_slot_mapping from the tables it produces, and the token data
is written by pa_reshape_and_cache.

Semantics ("深入解析LLM推理引擎：从PagedAttention到调度优化" §3.2-§3.3;
"vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §4.1;
"vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制" §2.3):
  * the free list is a stack: allocation takes its last entry, freeing
    pushes; an empty list is an out-of-blocks error;
  * every table entry holds one reference; forking a sequence shares all of
    its blocks (reference +1 each);
  * a sequence takes a new block when its last block is full; a write into a
    block whose reference count is above one first copies the block to a
    fresh one (copy-on-write) and repoints the table; the last holder writes
    in place;
  * freeing a sequence drops its references; blocks reaching zero return to
    the free list;
  * swapping ("【硬核】啃透vLLM源码：从PagedAttention到连续批处理，大模型推理加速24倍的秘密"
    §三: when GPU memory runs short, blocks go to CPU memory and come back
    when needed): swap-out gives each of the sequence's blocks a host block
    and drops the sequence's reference to the GPU block (a block still held
    by another sequence stays; the host gets a copy); swap-in gives each host
    block a fresh GPU block and frees the host block.  The (src, dst) pairs
    returned are what pa_swap_blocks moves.
This implementation is array based and appends tokens in bulk per sequence.
"""
from __future__ import annotations

import numpy as np
import torch


def kv_bytes_per_token(num_layers: int, num_heads: int, head_dim: int, dtype_bytes: int = 2) -> int:
    """Bytes of K and V cached per token: 2 (K and V) x layers x heads x head_dim x dtype size
    ("vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §2.1, KV_Size)."""
    return 2 * int(num_layers) * int(num_heads) * int(head_dim) * int(dtype_bytes)


class OutOfBlocksError(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, max_seqs: int, max_blocks_per_seq: int,
                 free_order=None, num_host_blocks: int = 0):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = np.arange(self.num_blocks) if free_order is None else np.asarray(free_order)
        self._free = np.empty(self.num_blocks, dtype=np.int64)
        self._free[:len(order)] = order
        self._top = len(order)                       # stack height
        self.ref = np.zeros(self.num_blocks, dtype=np.int32)
        self.tables = np.full((int(max_seqs), int(max_blocks_per_seq)), -1, dtype=np.int32)
        self.nblocks = np.zeros(int(max_seqs), dtype=np.int32)
        self.lengths = np.zeros(int(max_seqs), dtype=np.int64)
        self.live = np.zeros(int(max_seqs), dtype=bool)
        self.pending_copies: list[tuple[int, int]] = []
        # host (CPU) blocks for swapped-out sequences: a stack like the GPU list
        self.num_host_blocks = int(num_host_blocks)
        self._hfree = np.arange(self.num_host_blocks, dtype=np.int64)[::-1].copy()
        self._htop = self.num_host_blocks
        self.swapped = np.zeros(int(max_seqs), dtype=bool)

    # -- free list ---------------------------------------------------------
    def num_free(self) -> int:
        return self._top

    def _take(self) -> int:
        if self._top == 0:
            raise OutOfBlocksError("no free blocks")
        self._top -= 1
        b = int(self._free[self._top])
        self.ref[b] = 1
        return b

    def _drop(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self._free[self._top] = b
            self._top += 1

    # -- sequences -----------------------------------------------------------
    def add_sequence(self, seq: int) -> None:
        if self.live[seq]:
            raise ValueError(f"sequence {seq} exists")
        self.live[seq] = True
        self.nblocks[seq] = 0
        self.lengths[seq] = 0

    def fork(self, src: int, dst: int) -> None:
        """dst starts with src's contents, sharing every block."""
        if self.swapped[src]:
            raise ValueError(f"sequence {src} is swapped out")
        self.add_sequence(dst)
        n = int(self.nblocks[src])
        blocks = self.tables[src, :n]
        self.tables[dst, :n] = blocks
        np.add.at(self.ref, blocks, 1)
        self.nblocks[dst] = n
        self.lengths[dst] = self.lengths[src]

    def append_tokens(self, seq: int, n: int) -> np.ndarray:
        """Reserve slots for n more tokens of seq; returns their logical positions.
        Copy-on-write pairs (src, dst) accumulate in pending_copies."""
        B = self.block_size
        if self.swapped[seq]:
            raise ValueError(f"sequence {seq} is swapped out")
        pos0 = int(self.lengths[seq])
        if n <= 0:
            return np.empty(0, dtype=np.int32)
        if pos0 % B:
            j = pos0 // B
            b = int(self.tables[seq, j])
            if self.ref[b] > 1:
                fresh = self._take()
                self.pending_copies.append((b, fresh))
                self.ref[b] -= 1
                self.tables[seq, j] = fresh
        have = int(self.nblocks[seq])
        need = -(-(pos0 + n) // B)
        if need > self.tables.shape[1]:
            raise ValueError("sequence longer than the block-table width")
        for j in range(have, need):
            self.tables[seq, j] = self._take()
        self.nblocks[seq] = need
        self.lengths[seq] = pos0 + n
        return np.arange(pos0, pos0 + n, dtype=np.int32)

    def num_free_host(self) -> int:
        return self._htop

    def swap_out(self, seq: int) -> np.ndarray:
        """Move seq's blocks to host blocks; returns (gpu_block, host_block) pairs, int64 [n, 2]."""
        if not self.live[seq] or self.swapped[seq]:
            raise ValueError(f"sequence {seq} is not resident")
        n = int(self.nblocks[seq])
        if n > self._htop:
            raise OutOfBlocksError("no free host blocks")
        pairs = np.empty((n, 2), dtype=np.int64)
        for j in range(n):
            b = int(self.tables[seq, j])
            self._htop -= 1
            hb = int(self._hfree[self._htop])
            pairs[j] = (b, hb)
            self._drop(b)
            self.tables[seq, j] = hb
        self.swapped[seq] = True
        return pairs

    def swap_in(self, seq: int) -> np.ndarray:
        """Bring seq's blocks back into fresh GPU blocks; returns (host_block, gpu_block) pairs."""
        if not self.live[seq] or not self.swapped[seq]:
            raise ValueError(f"sequence {seq} is not swapped out")
        n = int(self.nblocks[seq])
        if n > self._top:
            raise OutOfBlocksError("no free blocks")
        pairs = np.empty((n, 2), dtype=np.int64)
        for j in range(n):
            hb = int(self.tables[seq, j])
            g = self._take()
            pairs[j] = (hb, g)
            self._hfree[self._htop] = hb
            self._htop += 1
            self.tables[seq, j] = g
        self.swapped[seq] = False
        return pairs

    def free_sequence(self, seq: int) -> None:
        if self.swapped[seq]:
            for hb in self.tables[seq, :int(self.nblocks[seq])]:
                self._hfree[self._htop] = int(hb)
                self._htop += 1
            self.swapped[seq] = False
        else:
            for b in self.tables[seq, :int(self.nblocks[seq])]:
                self._drop(int(b))
        self.tables[seq, :] = -1
        self.nblocks[seq] = 0
        self.lengths[seq] = 0
        self.live[seq] = False

    def take_copies(self) -> np.ndarray:
        """The copy-on-write pairs recorded since the last call, as int64 [P, 2]."""
        pairs = np.asarray(self.pending_copies, dtype=np.int64).reshape(-1, 2)
        self.pending_copies = []
        return pairs

    def block_tables(self, seqs=None) -> np.ndarray:
        return self.tables.copy() if seqs is None else self.tables[np.asarray(seqs)].copy()

    def context_lens(self, seqs=None) -> np.ndarray:
        lens = self.lengths if seqs is None else self.lengths[np.asarray(seqs)]
        return lens.astype(np.int32)


class KVPool:
    """Per-layer paged caches in HBM: key/value fp16 [num_blocks, num_heads, block_size, head_dim]
    (allocated through torch)."""

    def __init__(self, num_layers: int, num_blocks: int, num_heads: int, block_size: int,
                 head_dim: int, device="cuda"):
        shape = (int(num_blocks), int(num_heads), int(block_size), int(head_dim))
        self.shape = shape
        self.key_caches = [torch.empty(shape, dtype=torch.float16, device=device) for _ in range(num_layers)]
        self.value_caches = [torch.empty(shape, dtype=torch.float16, device=device) for _ in range(num_layers)]

    @property
    def num_layers(self) -> int:
        return len(self.key_caches)

    def bytes(self) -> int:
        return sum(t.numel() * 2 for t in self.key_caches + self.value_caches)
