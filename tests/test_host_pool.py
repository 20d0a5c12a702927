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


def gather(pool: np.ndarray, table: np.ndarray, n: int) -> np.ndarray:
    """A sequence's blocks in logical order (pool: [NB, ...])."""
    return pool[table[:n]].copy()


def test_swap_out_and_in_round_trip_restores_every_sequence():
    """Swap a shared-prefix sequence out and back in with the pairs the manager
    returns, moving block contents with the oracle's swap: every sequence's
    logical contents are unchanged, the other sequences' blocks untouched, and
    the free counts come back."""
    import oracle
    rng = np.random.default_rng(4)
    B, NB, NH = 4, 40, 16
    bm = BlockManager(NB, B, 4, 12, num_host_blocks=NH)
    dev = rng.integers(0, 1 << 16, (NB, 2, B, 8), dtype=np.uint16)
    host = np.zeros((NH, 2, B, 8), dtype=np.uint16)
    bm.add_sequence(0)
    bm.append_tokens(0, 10)            # 3 blocks, the last partial
    bm.fork(0, 1)                      # seq 1 shares all three
    bm.append_tokens(1, 5)             # copy-on-write of the partial block + 1 new
    cow = bm.take_copies()
    for src, dst in cow:
        dev[dst] = dev[src]
    bm.add_sequence(2)
    bm.append_tokens(2, 7)
    before = {s: gather(dev, bm.tables[s], int(bm.nblocks[s])) for s in (0, 1, 2)}
    free0, hfree0 = bm.num_free(), bm.num_free_host()

    out = bm.swap_out(1)
    assert out.shape == (int(bm.nblocks[1]), 2) and bm.swapped[1]
    assert oracle.swap_blocks([host], [dev], out) == 0
    assert bm.num_free_host() == hfree0 - len(out)
    # blocks still shared with sequence 0 stay allocated; the rest are free
    shared = set(bm.tables[0, :int(bm.nblocks[0])].tolist())
    assert bm.num_free() == free0 + sum(1 for g, _ in out if int(g) not in shared)
    # the freed GPU blocks are reused (and overwritten) by a new sequence
    bm.add_sequence(3)
    bm.append_tokens(3, B * min(bm.num_free(), 12))
    dev[bm.tables[3, :int(bm.nblocks[3])]] = 0xDEAD
    bm.free_sequence(3)

    back = bm.swap_in(1)
    assert not bm.swapped[1] and bm.num_free_host() == hfree0
    assert oracle.swap_blocks([dev], [host], back) == 0
    for s in (0, 1, 2):
        assert np.array_equal(gather(dev, bm.tables[s], int(bm.nblocks[s])), before[s])
    # blocks sequence 1 shared with sequence 0 came back as private copies
    n_shared = sum(1 for g, _ in out if int(g) in shared)
    assert n_shared == 2 and bm.num_free() == free0 - n_shared


def test_swap_errors_leave_state_unchanged():
    bm = BlockManager(8, 4, 2, 4, num_host_blocks=1)
    bm.add_sequence(0)
    bm.append_tokens(0, 9)             # 3 blocks, more than the one host block
    tables, free = bm.tables.copy(), bm.num_free()
    with pytest.raises(OutOfBlocksError):
        bm.swap_out(0)
    assert np.array_equal(bm.tables, tables) and bm.num_free() == free and not bm.swapped[0]
    with pytest.raises(ValueError):
        bm.swap_in(0)                  # not swapped out
    bm2 = BlockManager(8, 4, 2, 4, num_host_blocks=4)
    bm2.add_sequence(0)
    bm2.append_tokens(0, 8)
    bm2.swap_out(0)
    with pytest.raises(ValueError):
        bm2.append_tokens(0, 1)        # a swapped-out sequence takes no tokens
    with pytest.raises(ValueError):
        bm2.fork(0, 1)
    bm2.free_sequence(0)               # freeing returns its host blocks
    assert bm2.num_free_host() == 4 and bm2.num_free() == 8
