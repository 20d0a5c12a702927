"""The decode tolerance gate itself (CPU): each bound catches what it should
and lets pass what it should, so a loosened or mis-indexed gate fails here."""
import numpy as np
import pytest
import torch

from pa_testlib import decode_gate, gate_errors


def _check(g, r):
    return gate_errors(np.asarray(g, dtype=np.float64), np.asarray(r, dtype=np.float64))


def test_abs_bound_below_four():
    _, _, bad_abs, _ = _check([1.0021, 1.0019, -3.9981], [1.0, 1.0, -4.0 + 1e-9])
    assert bad_abs.tolist() == [True, False, False]


def test_abs_bound_one_fp16_step_from_four():
    # fp16 step in [4, 8) is 2^-8 = 3.90625e-3; in [8, 16) it is 2^-7.
    _, _, bad_abs, _ = _check([5.0038, 5.0040, 9.0077, 9.0080], [5.0, 5.0, 9.0, 9.0])
    assert bad_abs.tolist() == [False, True, False, True]


def test_rel_bound_only_from_one_tenth():
    # 0.1 with error 1.5e-3 is 1.5 % relative: above 1e-2.  0.05 with the same
    # error is 3 % relative but below the floor, and within the abs bound.
    max_abs, max_rel, bad_abs, bad_rel = _check([0.1015, 0.0515, 0.5009], [0.1, 0.05, 0.5])
    assert bad_rel.tolist() == [True, False, False]
    assert not bad_abs.any()
    assert max_rel == pytest.approx(0.015, rel=1e-6)
    assert max_abs == pytest.approx(1.5e-3, rel=1e-6)


def test_gate_asserts_and_reports():
    ref = np.array([[0.25, -1.5, 3.0, 0.0]])
    ok = torch.tensor(ref + np.array([[1e-4, -2e-4, 1.5e-3, 1e-3]]), dtype=torch.float32)
    a, r = decode_gate(ok, ref, "within", record=False)
    assert a == pytest.approx(1.5e-3, rel=1e-3) and r == pytest.approx(5e-4, rel=1e-3)
    with pytest.raises(AssertionError):
        decode_gate(torch.tensor(ref + np.array([[0.0, 2.5e-3, 0.0, 0.0]])), ref, "abs", record=False)
    with pytest.raises(AssertionError):
        decode_gate(torch.tensor([[0.25, -1.5, 3.0, float("nan")]]), ref, "nan", record=False)


def test_prefill_gate_is_the_same_tolerance():
    from pa_testlib import GATE_LOG, prefill_gate
    ref = np.array([[1.0, 0.3]])
    with pytest.raises(AssertionError):
        prefill_gate(torch.tensor(ref + np.array([[2.6e-3, 0.0]])), ref, "abs", record=False)
    n = len(GATE_LOG)
    prefill_gate(torch.tensor(ref + np.array([[1e-3, 0.0]])), ref, "ok")
    assert GATE_LOG[-1][0] == "ok" and GATE_LOG[-1][4] == "prefill"
    del GATE_LOG[n:]
