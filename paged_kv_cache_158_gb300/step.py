"""One decode step over every layer, replayable as a CUDA graph.

A decode step is: (optional) the copy-on-write block copies the block
manager planned, the slot map of the new tokens, then for every layer the
cache write of the new tokens and the paged decode.  When every sequence
brings one new token at position context_len - 1 (append=True), each layer's
cache write is fused into its decode (pa_decode_append) and the slot map is
not needed: one kernel fewer per layer.  Launching it takes
~2-3 library calls per layer; capturing it once in a CUDA graph and
replaying it removes the per-launch CPU cost and most launch gaps, as the
pages' model runner does for decode ("【硬核】啃透vLLM源码：从PagedAttention到
连续批处理，大模型推理加速24倍的秘密" §四: warm up twice, capture, replay).

All buffers are fixed at construction (a graph replays the same pointers):
callers update the step's inputs in place (queries, new keys/values, token
positions, block tables, context lengths) and read the outputs in place.
Every launch goes through the library's C ABI; every library call is safe to
capture (no allocation, no synchronisation).  The first call of the library
on a device does one-time set-up, so run the step eagerly at least once
before capturing (``capture`` does this).

With ``fp8_scales=(k_scale, v_scale)`` the caches are FP8 (E4M3 codes in
uint8 tensors) and the step uses the library's FP8 cache write, block copy
and decode.

Host-resident inputs (``bind_host``): every step copies the step's inputs
from pinned host buffers and its outputs back.  A layer needs only its own
query and new key/value rows, so the uploads run on a copy stream ahead of
the compute stream, and each layer's output goes back on a second copy
stream after its decode: only the first layer's upload and the last layer's
download are not hidden behind the decode kernels.  The compute stream waits
for the uploads only at layers 0, 1, 2, 4, 8, ... (each wait covers the next
power-of-two group of layers, which the copy stream, several times faster
than the decode, has finished by then), and hands outputs to the download
stream in the mirror-image groups (..., 4, 2, 1, 1 layers at the end), so
most consecutive kernels keep their programmatic launch chaining.  The small
per-step inputs (token ids and positions, block tables, context lengths) are
copied first, on the compute stream.  The whole fork/join captures into one
CUDA graph like the device-resident step.
"""
from __future__ import annotations

import torch

from . import (PA_DECODE_INPUTS_READY, PA_DECODE_ZEROED_WORKSPACE, decode_workspace, pa_copy_blocks, pa_copy_blocks_fp8,
               pa_decode_append, pa_decode_append_fp8, pa_decode_ex, pa_decode_fp8_ex,
               pa_reshape_and_cache, pa_reshape_and_cache_fp8, pa_slot_mapping)


def _overlap(a: torch.Tensor, b: torch.Tensor) -> bool:
    """The two tensors' byte ranges intersect."""
    a0, b0 = a.data_ptr(), b.data_ptr()
    return a0 < b0 + b.numel() * b.element_size() and b0 < a0 + a.numel() * a.element_size()


def _follows(a: torch.Tensor, b: torch.Tensor) -> bool:
    """b starts where a ends, in the same storage (both contiguous, same dtype)."""
    return (a.dtype == b.dtype and a.is_contiguous() and b.is_contiguous()
            and a.untyped_storage().data_ptr() == b.untyped_storage().data_ptr()
            and b.storage_offset() == a.storage_offset() + a.numel())


def _span(ts: list[torch.Tensor]) -> torch.Tensor:
    """One flat view over tensors that follow each other in one storage."""
    if len(ts) == 1:
        return ts[0]
    t0 = ts[0]
    return t0.new_empty(0).set_(t0.untyped_storage(), t0.storage_offset(),
                                (sum(t.numel() for t in ts),))


def _copy_runs(pairs: list[tuple[torch.Tensor, torch.Tensor]]) -> list[tuple[torch.Tensor, torch.Tensor]]:
    """(source, destination) pairs merged into one pair per maximal run whose sources follow
    each other in one storage and whose destinations do too: one copy instead of several."""
    runs, i = [], 0
    while i < len(pairs):
        j = i + 1
        while j < len(pairs) and _follows(pairs[j - 1][0], pairs[j][0]) and \
                _follows(pairs[j - 1][1], pairs[j][1]):
            j += 1
        runs.append((_span([p[0] for p in pairs[i:j]]), _span([p[1] for p in pairs[i:j]])))
        i = j
    return runs


def _pow2_groups(n: int) -> list[tuple[int, int]]:
    """Layer ranges [0, 1), [1, 2), [2, 4), [4, 8), ... covering n layers."""
    out, a = [], 0
    while a < n:
        b = min(n, max(1, 2 * a))
        out.append((a, b))
        a = b
    return out


class DecodeStep:
    def __init__(self, key_caches, value_caches, queries, keys_new, values_new, outs,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, token_seq: torch.Tensor,
                 token_pos: torch.Tensor, block_size: int, num_blocks: int, scale: float,
                 max_context_len: int, copy_pairs: torch.Tensor | None = None,
                 fp8_scales: tuple[float, float] | None = None, append: bool = False):
        n = len(key_caches)
        if not (len(value_caches) == len(queries) == len(keys_new) == len(values_new) == len(outs) == n):
            raise ValueError("one cache, query, new key/value and output per layer")
        self.key_caches, self.value_caches = list(key_caches), list(value_caches)
        self.queries, self.keys_new, self.values_new = list(queries), list(keys_new), list(values_new)
        self.outs = list(outs)
        self.block_tables, self.context_lens = block_tables, context_lens
        self.token_seq, self.token_pos = token_seq, token_pos
        self.block_size, self.num_blocks = int(block_size), int(num_blocks)
        self.scale, self.max_context_len = float(scale), int(max_context_len)
        self.copy_pairs = copy_pairs
        self.fp8_scales = None if fp8_scales is None else (float(fp8_scales[0]), float(fp8_scales[1]))
        # append: the decode step's usual shape, one new token per sequence at position
        # context_lens[s] - 1 with its rows keys_new[i][s] / values_new[i][s]; each layer's cache
        # write is then fused into its decode (pa_decode_append), and the slot map is not needed.
        self.append = bool(append)
        if self.append and any(k.shape != queries[0].shape for k in list(keys_new) + list(values_new)):
            raise ValueError("append: new keys/values must be [S, H, D], one row per sequence")
        # In append mode the kernel just before layer i's decode (i >= 1) is layer i - 1's
        # decode, which writes only its output: layer i's decode may then read its inputs
        # while that one finishes (PA_DECODE_INPUTS_READY), unless the output is one of them.
        self._ready = [False] * n
        for i in range(1, n if self.append else 0):
            ins = (queries[i], keys_new[i], values_new[i], key_caches[i], value_caches[i],
                   block_tables, context_lens)
            self._ready[i] = not any(_overlap(outs[i - 1], t) for t in ins)
        dev = queries[0].device
        S, H, D = queries[0].shape
        self.slots = torch.empty(token_seq.numel(), dtype=torch.int64, device=dev)
        self.workspace = decode_workspace(S, H, D, self.max_context_len, dev)
        self.graph: torch.cuda.CUDAGraph | None = None        # device-resident step
        self.host_graph: torch.cuda.CUDAGraph | None = None   # step from / to the host buffers
        self.host = None

    @property
    def num_layers(self) -> int:
        return len(self.key_caches)

    def run(self, stream=None, decode_events=None) -> None:
        """Launch the step eagerly on `stream` (default: the current stream).
        decode_events, if given, holds one (start, end) CUDA event pair per layer
        recorded around that layer's decode call."""
        s = stream if stream is not None else torch.cuda.current_stream()
        f8 = self.fp8_scales
        if self.copy_pairs is not None and self.copy_pairs.numel():
            (pa_copy_blocks_fp8 if f8 else pa_copy_blocks)(self.key_caches, self.value_caches,
                                                           self.copy_pairs, s)
        if not self.append:
            pa_slot_mapping(self.slots, self.block_tables, self.token_seq, self.token_pos,
                            self.block_size, self.num_blocks, s)
        for i in range(self.num_layers):
            self._write(i, s)
            if decode_events is not None:
                decode_events[i][0].record(s)
            self._decode(i, s)
            if decode_events is not None:
                decode_events[i][1].record(s)

    def bind_host(self, queries, keys_new, values_new, outs, block_tables, context_lens, token_seq,
                  token_pos) -> None:
        """Pinned host buffers the step reads its inputs from and writes its outputs to (one
        query / new key / new value / output tensor per layer, shaped like the device ones)."""
        n = self.num_layers
        if not (len(queries) == len(keys_new) == len(values_new) == len(outs) == n):
            raise ValueError("one host query, new key/value and output per layer")
        pairs = list(zip(queries, self.queries)) + list(zip(keys_new, self.keys_new)) + \
            list(zip(values_new, self.values_new)) + list(zip(outs, self.outs)) + \
            [(block_tables, self.block_tables), (context_lens, self.context_lens),
             (token_seq, self.token_seq), (token_pos, self.token_pos)]
        for h, d in pairs:
            if h.is_cuda or not h.is_pinned():
                raise ValueError("host buffers must be pinned host memory")
            if h.shape != d.shape or h.dtype != d.dtype or not h.is_contiguous():
                raise ValueError("a host buffer does not match its device buffer")
        dev = self.queries[0].device
        # The copies of each layer group (uploads) and of each mirror-image group (downloads),
        # merged where consecutive layers' buffers lie back to back on both sides (for example
        # views of one [L, ...] tensor): fewer, larger copies on the copy engines.
        groups = _pow2_groups(n)
        up_runs = {g0: _copy_runs([(h[i], d[i]) for h, d in ((queries, self.queries),
                                                              (keys_new, self.keys_new),
                                                              (values_new, self.values_new))
                                   for i in range(g0, g1)])
                   for g0, g1 in groups}
        down_runs = {n - g0: _copy_runs([(self.outs[j], outs[j]) for j in range(n - g1, n - g0)])
                     for g0, g1 in groups}
        small = [(block_tables, self.block_tables), (context_lens, self.context_lens),
                 (token_seq, self.token_seq), (token_pos, self.token_pos)]
        self.host = {
            "up_runs": up_runs, "down_runs": down_runs, "small_runs": _copy_runs(small),
            "q": list(queries), "k": list(keys_new), "v": list(values_new), "out": list(outs),
            "small": [(block_tables, self.block_tables), (context_lens, self.context_lens),
                      (token_seq, self.token_seq), (token_pos, self.token_pos)],
            "up": torch.cuda.Stream(dev), "down": torch.cuda.Stream(dev),
            "ev_in": [torch.cuda.Event() for _ in range(n)],
            "ev_gate": [torch.cuda.Event() for _ in range(n)],
            "ev_out": [torch.cuda.Event() for _ in range(n)],
        }

    def run_host(self, stream=None) -> None:
        """One step from the bound host buffers to the bound host outputs (see bind_host),
        launched eagerly on `stream` with the copies overlapped layer by layer."""
        if self.host is None:
            raise RuntimeError("bind_host() first")
        hb = self.host
        s = stream if stream is not None else torch.cuda.current_stream()
        up, down = hb["up"], hb["down"]
        # The copy streams start after everything queued before this step.
        up.wait_stream(s)
        down.wait_stream(s)
        groups = _pow2_groups(self.num_layers)
        L = self.num_layers

        def upload(g0):
            with torch.cuda.stream(up):
                for h, d in hb["up_runs"][g0]:
                    d.copy_(h, non_blocking=True)
                hb["ev_in"][g0].record(up)

        # Uploads are paced: group [g0, g1) starts copying when the compute reaches layer
        # g0 // 2, half the group's length ahead of its first use.  Issuing every upload at the
        # step's start makes a burst of host-to-device writes that slows the first layers'
        # decode more than its bytes suggest (13B-shaped step: 4.16 vs 4.05 ms).
        gate = {}
        for g0, _ in groups:
            gate.setdefault(g0 // 2, []).append(g0)
        with torch.cuda.stream(s):
            for h, d in hb["small_runs"]:
                d.copy_(h, non_blocking=True)
        f8 = self.fp8_scales
        if self.copy_pairs is not None and self.copy_pairs.numel():
            (pa_copy_blocks_fp8 if f8 else pa_copy_blocks)(self.key_caches, self.value_caches,
                                                           self.copy_pairs, s)
        if not self.append:
            pa_slot_mapping(self.slots, self.block_tables, self.token_seq, self.token_pos,
                            self.block_size, self.num_blocks, s)
        starts = {g0 for g0, _ in groups}
        # Downloads in the mirror-image groups: ..., 4, 2, 1, 1 layers at the end.
        ends = {L - g0: L - g1 for g0, g1 in groups}   # group end (exclusive) -> group start
        for i in range(L):
            for g0 in gate.get(i, []):
                if i > 0:
                    hb["ev_gate"][g0].record(s)
                    up.wait_event(hb["ev_gate"][g0])
                upload(g0)
            if i in starts:
                s.wait_event(hb["ev_in"][i])
            self._write(i, s)
            self._decode(i, s)
            if i + 1 in ends:
                hb["ev_out"][i].record(s)
                down.wait_event(hb["ev_out"][i])
                with torch.cuda.stream(down):
                    for d, h in hb["down_runs"][i + 1]:
                        h.copy_(d, non_blocking=True)
        # The step ends when its last output is on the host.
        s.wait_stream(down)
        s.wait_stream(up)

    def _write(self, i: int, s) -> None:
        """Layer i's cache write of the new tokens (in append mode it is part of the decode)."""
        if self.append:
            return
        f8 = self.fp8_scales
        if f8:
            pa_reshape_and_cache_fp8(self.keys_new[i], self.values_new[i], self.key_caches[i],
                                     self.value_caches[i], self.slots, f8[0], f8[1], s)
        else:
            pa_reshape_and_cache(self.keys_new[i], self.values_new[i], self.key_caches[i],
                                 self.value_caches[i], self.slots, s)

    def _decode(self, i: int, s) -> None:
        """Layer i's paged decode.  The step's workspace is zero-filled at construction and
        only ever passed to the decode calls, which leave its counters zero, so no call needs
        to zero them first (PA_DECODE_ZEROED_WORKSPACE)."""
        f8 = self.fp8_scales
        fl = PA_DECODE_ZEROED_WORKSPACE | (PA_DECODE_INPUTS_READY if self._ready[i] else 0)
        if self.append:
            if f8:
                pa_decode_append_fp8(self.outs[i], self.queries[i], self.keys_new[i],
                                     self.values_new[i], self.key_caches[i], self.value_caches[i],
                                     self.block_tables, self.context_lens, self.scale, f8[0], f8[1],
                                     self.max_context_len, self.workspace, fl, s)
            else:
                pa_decode_append(self.outs[i], self.queries[i], self.keys_new[i], self.values_new[i],
                                 self.key_caches[i], self.value_caches[i], self.block_tables,
                                 self.context_lens, self.scale, self.max_context_len,
                                 self.workspace, fl, s)
            return
        if f8:
            pa_decode_fp8_ex(self.outs[i], self.queries[i], self.key_caches[i],
                             self.value_caches[i], self.block_tables, self.context_lens, self.scale,
                             f8[0], f8[1], self.max_context_len, self.workspace, fl, s)
        else:
            pa_decode_ex(self.outs[i], self.queries[i], self.key_caches[i], self.value_caches[i],
                         self.block_tables, self.context_lens, self.scale, self.max_context_len,
                         self.workspace, fl, s)

    def capture(self, warmup: int = 2, host: bool = False) -> None:
        """Warm up (eager runs), then capture one step into a CUDA graph; with host=True the
        captured step is run_host (copies from / to the bound host buffers included)."""
        fn = self.run_host if host else self.run
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(max(1, warmup)):
                fn(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        if host:
            self.host_graph = g
        else:
            self.graph = g

    def replay(self, host: bool = False) -> None:
        g = self.host_graph if host else self.graph
        if g is None:
            raise RuntimeError("capture() first")
        g.replay()
