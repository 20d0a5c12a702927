"""The product's host block manager against the oracle's plain model of the
pages' block manager, and the KV-size closed form against the pages' figures."""
import json
import os

import numpy as np
import pytest

from oracle.block_model import BlockModel, OutOfBlocks, shared_prefix_flow
from paged_kv_cache_158_gb300.pool import BlockManager, OutOfBlocksError, kv_bytes_per_token
from workloads import configs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_kv_bytes_per_token_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "kv_cache_sizes.json")))
    for c in g["cases"]:
        assert kv_bytes_per_token(c["layers"], c["heads"], c["head_dim"]) == c["bytes_per_token"]
    per_tok = kv_bytes_per_token(40, 40, 128)
    assert per_tok * 1024 == g["llama13b_1024_tokens_bytes"]
    assert per_tok * 1024 == g["llama13b_1024_tokens_mib"] * 2 ** 20
    assert per_tok * 1024 * 32 == g["llama13b_batch32_1024_tokens_gib"] * 2 ** 30


def product_shared_prefix(w):
    bm = BlockManager(w.num_blocks, w.block_size, w.num_seqs, w.max_blocks_per_seq, w.free_order)
    bm.add_sequence(0)
    bm.append_tokens(0, w.prefix_len)
    for s in range(1, w.num_seqs):
        bm.fork(0, s)
    positions = [bm.append_tokens(s, int(w.suffix_lens[s])) for s in range(w.num_seqs)]
    return bm, positions


def test_shared_prefix_flow_matches_model():
    w = configs.config4()
    bm, positions = product_shared_prefix(w)
    model, appended = shared_prefix_flow(w.num_seqs, w.prefix_len, w.suffix_lens, w.num_blocks,
                                         w.block_size, w.free_order)
    assert np.array_equal(bm.block_tables(), model.table_array(range(w.num_seqs), w.max_blocks_per_seq))
    assert np.array_equal(bm.take_copies(), np.array(model.copies, dtype=np.int64))
    assert np.array_equal(bm.context_lens(), w.context_lens)
    assert list(bm.ref) == model.ref and bm.num_free() == len(model.free) == 0
    seqs, pos = w.new_tokens()
    assert np.array_equal(np.concatenate(positions), pos)
    assert [(int(s), int(p)) for s, p in zip(seqs, pos)] == appended


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_model(seed):
    rng = np.random.default_rng(seed)
    NB, B, MS = 40, 4, 8
    order = rng.permutation(NB)
    bm = BlockManager(NB, B, MS, 32, order)
    model = BlockModel(NB, B, order)
    live = []
    for _ in range(200):
        op = rng.integers(0, 4)
        if True:
            if op == 0 and len(live) < MS:
                s = next(i for i in range(MS) if i not in live)
                bm.add_sequence(s)
                model.add_sequence(s)
                live.append(s)
            elif op == 1 and live and len(live) < MS:
                src = int(rng.choice(live))
                dst = next(i for i in range(MS) if i not in live)
                bm.fork(src, dst)
                model.fork(src, dst)
                live.append(dst)
            elif op == 2 and live:
                s = int(rng.choice(live))
                n = int(rng.integers(1, 9))
                if model.lengths[s] + n > 32 * B:
                    continue
                try:
                    bm.append_tokens(s, n)
                    bm_err = None
                except OutOfBlocksError as e:
                    bm_err = e
                try:
                    for _ in range(n):
                        model.append_token(s)
                    model_err = None
                except OutOfBlocks as e:
                    model_err = e
                assert (bm_err is None) == (model_err is None)
                if bm_err is not None:
                    return  # both ran out of blocks; state after a failed append is unspecified
            elif op == 3 and live:
                s = int(rng.choice(live))
                bm.free_sequence(s)
                model.free_sequence(s)
                live.remove(s)
        for s in live:
            assert list(bm.tables[s, :bm.nblocks[s]]) == model.tables[s]
            assert bm.lengths[s] == model.lengths[s]
        assert list(bm.ref) == model.ref
        assert [tuple(p) for p in bm.take_copies()] == model.copies
        model.copies = []
        assert bm.num_free() == len(model.free)
