"""One decode step over every layer, replayable as a CUDA graph.

A decode step is: (optional) the copy-on-write block copies the block
manager planned, the slot map of the new tokens, then for every layer the
cache write of the new tokens and the paged decode.  Launching it takes
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
"""
from __future__ import annotations

import torch

from . import (decode_workspace, pa_copy_blocks, pa_copy_blocks_fp8, pa_decode, pa_decode_fp8,
               pa_reshape_and_cache, pa_reshape_and_cache_fp8, pa_slot_mapping)


class DecodeStep:
    def __init__(self, key_caches, value_caches, queries, keys_new, values_new, outs,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, token_seq: torch.Tensor,
                 token_pos: torch.Tensor, block_size: int, num_blocks: int, scale: float,
                 max_context_len: int, copy_pairs: torch.Tensor | None = None,
                 fp8_scales: tuple[float, float] | None = None):
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
        dev = queries[0].device
        S, H, D = queries[0].shape
        self.slots = torch.empty(token_seq.numel(), dtype=torch.int64, device=dev)
        self.workspace = decode_workspace(S, H, D, self.max_context_len, dev)
        self.graph: torch.cuda.CUDAGraph | None = None

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
        pa_slot_mapping(self.slots, self.block_tables, self.token_seq, self.token_pos, self.block_size,
                        self.num_blocks, s)
        for i in range(self.num_layers):
            if f8:
                pa_reshape_and_cache_fp8(self.keys_new[i], self.values_new[i], self.key_caches[i],
                                         self.value_caches[i], self.slots, f8[0], f8[1], s)
            else:
                pa_reshape_and_cache(self.keys_new[i], self.values_new[i], self.key_caches[i],
                                     self.value_caches[i], self.slots, s)
            if decode_events is not None:
                decode_events[i][0].record(s)
            if f8:
                pa_decode_fp8(self.outs[i], self.queries[i], self.key_caches[i], self.value_caches[i],
                              self.block_tables, self.context_lens, self.scale, f8[0], f8[1],
                              self.max_context_len, self.workspace, s)
            else:
                pa_decode(self.outs[i], self.queries[i], self.key_caches[i], self.value_caches[i],
                          self.block_tables, self.context_lens, self.scale, self.max_context_len,
                          self.workspace, s)
            if decode_events is not None:
                decode_events[i][1].record(s)

    def capture(self, warmup: int = 2) -> None:
        """Warm up (eager runs), then capture one step into a CUDA graph."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(max(1, warmup)):
                self.run(side)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(torch.cuda.current_stream())
        self.graph = g

    def replay(self) -> None:
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
