"""Host logic of the decode step that runs without a GPU: merging the copies of back-to-back
layer buffers into one copy per run, the byte-range overlap test behind
PA_DECODE_INPUTS_READY, and the layer groups the copies are issued in."""
import torch

from paged_kv_cache_158_gb300.step import _copy_runs, _overlap, _pow2_groups


def test_views_of_one_tensor_merge_into_one_copy():
    src, dst = torch.arange(4 * 6, dtype=torch.float32).view(4, 2, 3), torch.zeros(4, 2, 3)
    runs = _copy_runs([(src[i], dst[i]) for i in range(4)])
    assert len(runs) == 1
    s, d = runs[0]
    assert s.numel() == d.numel() == 24 and s.data_ptr() == src.data_ptr()
    d.copy_(s)
    assert torch.equal(dst, src)


def test_separate_or_gapped_buffers_stay_separate_copies():
    dst = torch.zeros(4, 5)
    sep = [torch.full((5,), float(i)) for i in range(4)]
    assert len(_copy_runs([(sep[i], dst[i]) for i in range(4)])) == 4
    src = torch.arange(20, dtype=torch.float32).view(4, 5)
    runs = _copy_runs([(src[i], dst[i]) for i in (0, 1, 3)])      # layer 2 missing: two runs
    assert [r[0].numel() for r in runs] == [10, 5]
    for s, d in runs:
        d.copy_(s)
    assert torch.equal(dst[[0, 1, 3]], src[[0, 1, 3]]) and torch.equal(dst[2], torch.zeros(5))
    # back to back on one side only: no merge
    assert len(_copy_runs([(src[i], sep[i]) for i in range(4)])) == 4
    # other dtype or a strided view never merges with its neighbour
    half = torch.zeros(10, dtype=torch.float16)
    assert len(_copy_runs([(src[0], half[:5].float()), (src[1], dst[1])])) == 2
    cols = torch.zeros(5, 4)
    assert len(_copy_runs([(src[i], cols[:, i]) for i in range(2)])) == 2


def test_overlap_is_byte_range_intersection():
    t = torch.zeros(100)
    assert _overlap(t[10:20], t[15:30]) and _overlap(t[0:50], t[49:50])
    assert not _overlap(t[0:10], t[10:20]) and not _overlap(t, torch.zeros(100))


def test_copy_groups_cover_every_layer_once_in_powers_of_two():
    for n in range(1, 70):
        g = _pow2_groups(n)
        assert g[0][0] == 0 and g[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(g, g[1:]))
        assert all(b - a <= max(1, a) for a, b in g)
