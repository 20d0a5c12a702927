"""pa_decode_noalloc, the decode entry point for callers that cannot allocate
device memory when they decode (all of HBM given to the KV pool, a hot path
where cudaMalloc/cudaFree may synchronise the device, or a plain C caller with
no device allocator).  It must give the same result as pa_decode with a
caller-allocated workspace, on two calls in a row (the fixed scratch keeps the
previous call's contents), and refuse shapes whose scratch would not fit.

Called through the C ABI with ctypes.  Collected last on purpose, so that a
run stopping at its first failure has run every other test first; it passes
alone in a fresh process too (its first call is then the per-device warm-up
that loads the scratch array)."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_158_gb300 as pa
from pa_testlib import ATOL, RTOL
from workloads import configs, gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _entry():
    f = ctypes.CDLL(pa.LIB_PATH).pa_decode_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    f.restype = i32
    return f


def _call(f, w, out, q, kc, vc, bt, ctx):
    return f(out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), bt.shape[1],
             ctx.data_ptr(), w.num_seqs, w.num_heads, w.head_dim, w.block_size, w.num_blocks,
             w.scale, w.max_context_len, torch.cuda.current_stream().cuda_stream)


def test_noalloc_decode_matches_workspace_decode_twice():
    f = _entry()
    w = configs.config2()
    # 128-token partitions: every sequence (200..500 tokens) has several, so the
    # partial results and the merge go through the scratch area.
    pa.pa_decode_set_partition_tokens(128)
    try:
        assert pa.pa_decode_workspace_size(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len) > 4096
        dw = gpu.materialize(w, layers=[0, 1], device=DEV)
        ws = pa.decode_workspace(w.num_seqs, w.num_heads, w.head_dim, w.max_context_len)
        for i in (0, 1):                 # two calls in a row, different inputs
            ref = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=DEV)
            pa.pa_decode(ref, dw.queries[i], dw.key_caches[i], dw.value_caches[i], dw.block_tables,
                         dw.context_lens, w.scale, w.max_context_len, ws)
            got = torch.full_like(ref, float("nan"))
            assert _call(f, w, got, dw.queries[i], dw.key_caches[i], dw.value_caches[i],
                         dw.block_tables, dw.context_lens) == pa.PA_OK
            torch.cuda.synchronize()
            g = got.float().cpu().numpy()
            r = ref.float().cpu().numpy()
            assert np.all(np.isfinite(g))
            assert np.all(np.abs(g - r) <= ATOL + RTOL * np.abs(r))
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
            via = torch.full_like(ref, float("nan"))     # the Python binding of the same call
            pa.pa_decode_noalloc(via, dw.queries[i], dw.key_caches[i], dw.value_caches[i],
                                 dw.block_tables, dw.context_lens, w.scale, w.max_context_len)
            torch.cuda.synchronize()
            assert torch.equal(via.view(torch.int16), ref.view(torch.int16))
        assert pa.pa_check_errors() == (pa.PA_OK, 0)
    finally:
        pa.pa_decode_set_partition_tokens(0)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    """1024 sequences x 64 heads up to 4096 tokens needs far more than 32 MiB of
    partials; the call is refused on the host and launches nothing."""
    f = _entry()
    S, H, D, B, NB, ctx_max = 1024, 64, 128, 16, 8, 4096
    assert pa.pa_decode_workspace_size(S, H, D, ctx_max) > (32 << 20)
    dummy = torch.zeros(64, dtype=torch.float16, device=DEV)
    ints = torch.zeros(64, dtype=torch.int32, device=DEV)
    p = dummy.data_ptr()
    rc = f(p, p, p, p, ints.data_ptr(), 1, ints.data_ptr(), S, H, D, B, NB, 0.1, ctx_max,
           torch.cuda.current_stream().cuda_stream)
    assert rc == pa.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
