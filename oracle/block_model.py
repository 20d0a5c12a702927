"""Plain model of the pages' KV block manager — TEST INFRASTRUCTURE ONLY.

Written from:
  * "深入解析LLM推理引擎：从PagedAttention到调度优化" §3.2 (blocks fill token
    by token; a new physical block is taken when the last one is full; a
    request's block table maps logical to physical blocks) and §3.3 (the
    free list starts as all block ids and allocation pops from its end; an
    empty free list is an out-of-memory error; a block returns to the free
    list only when its reference count is zero).
  * "vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §4.1 (allocation
    appends the new block to the request's table and raises its reference
    count; sharing appends the source request's physical block to the
    destination's table and raises its count).
  * "vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制"
    §2.3 (shared blocks stay shared until a request has to write different
    content into one; then that block is copied and the request's table is
    repointed — copy-on-write; finishing a request lowers the counts of its
    blocks and returns those that reach zero).

Reading taken where the pages are silent: a write copies a block exactly
when that block's reference count is above one at the time of the write (the
usual operating-system copy-on-write rule); the last remaining holder writes
in place.  Eviction is not modelled (serving policy, not this path).
"""
from __future__ import annotations

import numpy as np


class OutOfBlocks(Exception):
    """Raised when a block is needed and the free list is empty."""


class BlockModel:
    def __init__(self, num_blocks: int, block_size: int, free_list=None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.free = list(range(self.num_blocks)) if free_list is None else [int(b) for b in free_list]
        self.ref = [0] * self.num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}
        self.copies: list[tuple[int, int]] = []

    def allocate(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free blocks")
        b = self.free.pop()
        self.ref[b] += 1
        return b

    def release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def add_sequence(self, seq: int) -> None:
        self.tables[seq] = []
        self.lengths[seq] = 0

    def share(self, src: int, dst: int, logical_block: int) -> None:
        """Append src's physical block `logical_block` to dst's table."""
        b = self.tables[src][logical_block]
        self.tables[dst].append(b)
        self.ref[b] += 1

    def fork(self, src: int, dst: int) -> None:
        """dst starts as a copy of src's whole table (every block shared)."""
        self.add_sequence(dst)
        for j in range(len(self.tables[src])):
            self.share(src, dst, j)
        self.lengths[dst] = self.lengths[src]

    def append_token(self, seq: int) -> int:
        """Reserve room for one more token of `seq`; returns its logical position."""
        pos = self.lengths[seq]
        table = self.tables[seq]
        if pos == len(table) * self.block_size:
            table.append(self.allocate())
        else:
            j = pos // self.block_size
            b = table[j]
            if self.ref[b] > 1:
                n = self.allocate()
                self.copies.append((b, n))
                self.ref[b] -= 1
                table[j] = n
        self.lengths[seq] = pos + 1
        return pos

    def free_sequence(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self.release(b)
        del self.lengths[seq]

    def slot(self, seq: int, pos: int) -> int:
        return self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size

    def table_array(self, seqs, width: int) -> np.ndarray:
        out = np.full((len(seqs), width), -1, dtype=np.int32)
        for i, s in enumerate(seqs):
            t = self.tables[s]
            out[i, :len(t)] = t
        return out


def shared_prefix_flow(num_seqs: int, prefix_len: int, suffix_lens, num_blocks: int,
                       block_size: int, free_list):
    """The shared-prefix workload as the pages describe it.

    Sequence 0 stores the prefix, sequences 1..S-1 share all of its blocks,
    then every sequence in turn appends its own suffix.  Returns the model and
    the (seq, pos) list of the appended suffix tokens, in order.
    """
    m = BlockModel(num_blocks, block_size, free_list)
    m.add_sequence(0)
    for _ in range(prefix_len):
        m.append_token(0)
    for s in range(1, num_seqs):
        m.fork(0, s)
    appended = []
    for s in range(num_seqs):
        for _ in range(int(suffix_lens[s])):
            appended.append((s, m.append_token(s)))
    return m, appended
