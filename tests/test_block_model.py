"""Pins for the oracle's block-manager model against the pages' statements.

* "深入解析LLM推理引擎：从PagedAttention到调度优化" §3.2: a block fills token
  by token and a new block is taken when it is full; the worked example's
  table [0, 1, 3]; waste only in the last block (ceil(len/B) blocks).
  §3.3: free list list(range(N)), allocation pops its end, empty list is an
  out-of-memory error, a block is freed only at reference count zero.
* "vLLM推理加速深度解读：PagedAttention如何提升10x吞吐量" §4.1: allocation
  and sharing raise the reference count; sharing appends the source's
  physical block to the destination's table.
* "vLLM基础架构：核心组件、PagedAttention原理、KV Cache管理与连续批处理机制"
  §2.3: copy-on-write on the first differing write to a shared block;
  finishing lowers counts and frees those reaching zero.
"""
import json
import os

import numpy as np
import pytest

from oracle.block_model import BlockModel, OutOfBlocks, shared_prefix_flow
from workloads import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_free_list_pops_from_the_end():
    m = BlockModel(5, 4)
    assert [m.allocate() for _ in range(5)] == [4, 3, 2, 1, 0]
    with pytest.raises(OutOfBlocks):
        m.allocate()


def test_worked_example_table():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_block_table.json")))
    B = g["block_size"]
    # A free list handing out 0, 1, 2, ... in order (pop from the end of a reversed list).
    m = BlockModel(8, B, free_list=list(range(8))[::-1])
    m.add_sequence("A")
    m.add_sequence("B")
    for _ in range(8):
        m.append_token("A")          # tokens 1-4 -> block 0, tokens 5-8 -> block 1
    m.append_token("B")              # another request takes physical block 2
    m.append_token("A")              # token 9 -> a new block: 3
    assert m.tables["A"] == g["block_table_A"]
    for pos, blk, off in g["position_to_block_offset"][:9]:
        assert m.slot("A", pos) == blk * B + off


def test_block_count_is_ceil_len_over_b():
    g = json.load(open(os.path.join(GOLDEN, "worked_example_block_table.json")))
    for tokens, blocks in g["blocks_for_tokens"]:
        m = BlockModel(16, g["block_size"])
        m.add_sequence(0)
        for _ in range(tokens):
            m.append_token(0)
        assert len(m.tables[0]) == blocks


def test_share_raises_ref_and_free_waits_for_zero():
    m = BlockModel(4, 2)
    m.add_sequence(0)
    m.append_token(0)
    b = m.tables[0][0]
    m.add_sequence(1)
    m.share(0, 1, 0)
    assert m.tables[1] == [b] and m.ref[b] == 2
    m.free_sequence(0)
    assert b not in m.free and m.ref[b] == 1
    m.free_sequence(1)
    assert b in m.free and m.ref[b] == 0


def test_copy_on_write_iff_shared():
    m = BlockModel(8, 4)
    m.add_sequence(0)
    for _ in range(6):                # blocks: one full, one partial (2 tokens)
        m.append_token(0)
    m.fork(0, 1)
    m.fork(0, 2)
    full, part = m.tables[0]
    assert m.ref[full] == 3 and m.ref[part] == 3
    m.append_token(1)                 # writes into the shared partial block -> copy
    assert len(m.copies) == 1 and m.copies[0][0] == part
    assert m.tables[1][1] == m.copies[0][1] and m.ref[part] == 2
    m.append_token(0)                 # still shared with seq 2 -> copy
    assert len(m.copies) == 2 and m.ref[part] == 1
    m.append_token(2)                 # last holder writes in place
    assert len(m.copies) == 2 and m.tables[2][1] == part
    m.append_token(2)                 # the full block is never written: no copy
    m.append_token(2)
    assert len(m.copies) == 2 and m.ref[full] == 3


def test_shared_prefix_workload_structure():
    w = configs.config4()
    m, appended = shared_prefix_flow(w.num_seqs, w.prefix_len, w.suffix_lens, w.num_blocks,
                                     w.block_size, w.free_order)
    B = w.block_size
    # 63 copies: every writer of the shared partial block but the last.
    assert len(m.copies) == w.num_seqs - 1
    srcs = {s for s, _ in m.copies}
    assert len(srcs) == 1 and m.tables[w.num_seqs - 1][w.prefix_len // B] == srcs.pop()
    # the pool is sized exactly: nothing left over
    assert m.free == []
    for s in range(w.num_seqs):
        assert m.lengths[s] == w.context_lens[s]
        assert len(m.tables[s]) == -(-int(w.context_lens[s]) // B)
        assert m.tables[s][:w.prefix_len // B] == m.tables[0][:w.prefix_len // B]
    assert len(appended) == int(w.suffix_lens.sum())
    # distinct destinations, none of them a source
    dsts = [d for _, d in m.copies]
    assert len(set(dsts)) == len(dsts) and not set(dsts) & {s for s, _ in m.copies}
