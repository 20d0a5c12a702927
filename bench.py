"""Benchmark of the paged decode hot path on GB300.

One step = one decode step of the workload through the library: for every
layer the cache write of the new tokens and the paged decode (partition pass
+ merge).  When every sequence brings one new token at position c - 1 (all
decode workloads but the shared-prefix one) and the caches are fp16, the write
is fused into the decode (pa_decode_append); otherwise (and with --append off)
the step runs the slot map and a cache-write kernel before each decode.  The headline metric
is paged-decode KV GB/s: algorithmic bytes of all decode calls of the step
(q + the gathered K/V of the c_s live tokens + out + block-table entries and
context lengths) over the step time; also reported as % of the measured HBM
peak, attention tokens/s per layer and us per layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c3|c5|c2|c4|c1]
                    [--kv-dtype fp16|fp8]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm
    python bench.py --op scan [--kv-dtype fp8]  # time per call vs context length

--kv-dtype fp8 runs the same step on FP8 (E4M3) caches: the bytes count one
byte per cached K/V element, so compare it with fp16 on tokens/s as well.

N > 1 runs under torch.distributed.run: every rank runs its own replica of
the workload (sequences shard across GPUs with no exchange: weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import configs  # noqa: E402

FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c3", choices=["c1", "c2", "c3", "c4", "c5"])
    ap.add_argument("--layers", type=int, default=0, help="use only the first L layers (profiling)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--partition-tokens", type=int, default=0)
    ap.add_argument("--eager", action="store_true", help="time eager launches only (no CUDA graph)")
    ap.add_argument("--op", choices=["step", "swap", "prefill", "cache", "scan"], default="step",
                    help="swap: time block swap-out/in of whole sequences to pinned host memory; "
                         "prefill: time multi-query paged attention on the 7B-shaped chunked prefill; "
                         "cache: time the cache write and the copy-on-write block copy of a step; "
                         "scan: decode time per call against context length (fixed + marginal)")
    ap.add_argument("--kv-dtype", choices=["fp16", "fp8"], default="fp16",
                    help="KV-cache element type (fp8: E4M3 codes with per-tensor scales)")
    ap.add_argument("--prefill-workload", choices=["chunked", "mixed"], default="chunked",
                    help="--op prefill: 4 x 512-token chunks (chunked) or 2 chunks plus 64 decode "
                         "rows in one call (mixed; also timed as separate prefill and decode calls)")
    ap.add_argument("--append", choices=["auto", "on", "off"], default="auto",
                    help="cache write fused into the decode (pa_decode_append: on), or its own "
                         "kernel after a slot map (off); auto: fused for fp16 caches, separate "
                         "for FP8 caches (the faster of the two on each)")
    ap.add_argument("--no-append", dest="append", action="store_const", const="off",
                    help="same as --append off")
    ap.add_argument("--also", default="c5",
                    help="comma-separated workloads measured after the main one in the same run "
                         "(single GPU only; 'none' to skip); each gets its own record under 'also'")
    return ap.parse_args()


def make_workload(name: str, layers: int):
    cid = int(name[1:])
    if cid == 3:
        return configs.config3(layers or 40)
    if cid == 5:
        return configs.config5(layers or 32)
    return configs.ALL[cid]()


def decode_bytes(w, bt, ctx, kv_elem_bytes: int = 2) -> int:
    """Algorithmic bytes of one decode call: per (s, h): q (2D) + K and V of the c_s live
    tokens (2 * c_s * D * kv_elem_bytes) + out (2D); per s: ceil(c_s/B) table entries and
    one context length."""
    H, D, B = w.num_heads, w.head_dim, w.block_size
    ctx = np.asarray(ctx, dtype=np.int64)
    S = len(ctx)
    per_pair = 2 * D + 2 * kv_elem_bytes * ctx * D + 2 * D
    return int(H * per_pair.sum() + 4 * (-(-ctx // B)).sum() + 4 * S)


# Sources that define the decode kernels (the ncu traffic is tied to these).
DECODE_SOURCES = ("pa_decode.cuh", "pa_decode_inst.inc", "pa_decode_d64.cu", "pa_decode_d128.cu",
                  "pa_decode_f8_d64.cu", "pa_decode_f8_d128.cu", "pa_device.cuh", "pa_launch.cuh",
                  "pa_internal.h", "pa_api.cu")   # pa_api.cu: launch configuration (partition size)


def source_hash() -> str:
    """Hash of the decode kernels' sources."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_158_gb300", "csrc")
    for p in sorted(os.path.join(csrc, f) for f in DECODE_SOURCES):
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def committed_traffic(workload_name: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload_name)
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.path = os.path.join("/tmp", f"pa_clocks_{os.getpid()}.csv")

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(n_gpus: int):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar (timing only; no data-path collective)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank_step: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job GB/s: every rank processed bytes_per_rank_step per step; the job's step
    time is the slowest rank's."""
    return bytes_per_rank_step * world / (ms_per_step_max * 1e-3) / 1e9


# ---------------------------------------------------------------- our arm

class Step:
    """Device state of the workload and its decode step (the library's DecodeStep)."""

    def __init__(self, w, device, fp8: bool = False, append: str = "auto"):
        import torch

        import paged_kv_cache_158_gb300 as pa
        from paged_kv_cache_158_gb300.pool import BlockManager
        from paged_kv_cache_158_gb300.step import DecodeStep
        from workloads import gpu

        self.pa, self.w, self.dev = pa, w, device
        self.fp8_scales = configs.fp8_scales(w) if fp8 else None
        if fp8:
            dw = gpu.materialize(w, device=device, fp8_convert=pa.pa_convert_cache_fp8,
                                 fp8_scales=self.fp8_scales)
        else:
            dw = gpu.materialize(w, device=device)
        self.dw = dw
        copy_pairs = None
        if w.block_tables is None:          # shared-prefix workload: the block manager plans
            bm = BlockManager(w.num_blocks, w.block_size, w.num_seqs, w.max_blocks_per_seq, w.free_order)
            bm.add_sequence(0)
            bm.append_tokens(0, w.prefix_len)
            for s in range(1, w.num_seqs):
                bm.fork(0, s)
            for s in range(w.num_seqs):
                bm.append_tokens(s, int(w.suffix_lens[s]))
            copy_pairs = torch.from_numpy(bm.take_copies()).to(device)
            dw.block_tables = torch.from_numpy(bm.block_tables()).to(device)
        self.bt_host = dw.block_tables.cpu().numpy()
        self.ctx_host = w.context_lens.copy()
        self.max_ctx = int(self.ctx_host.max())
        # One [L, S, H, D] allocation: consecutive layers' outputs back to back (fewer, larger
        # read-back copies in the end-to-end step).
        outs = list(torch.empty((len(dw.layers), w.num_seqs, w.num_heads, w.head_dim),
                                dtype=torch.float16, device=device).unbind(0))
        # One new token per sequence at position c - 1 (every decode workload but the shared
        # prefix one, which writes whole suffixes): with fp16 caches the cache write rides in
        # the decode.  With FP8 caches the fused kernel measured slower than the separate write
        # (long-context step 6221 vs 6521 GB/s), so the FP8 step keeps the write kernel unless
        # --append forces the fused one.
        self.append = (append == "on" or (append == "auto" and not fp8)) and copy_pairs is None \
            and bool(np.all(w.context_lens > 0))
        self.step = DecodeStep(dw.key_caches, dw.value_caches, dw.queries, dw.keys_new, dw.values_new,
                               outs, dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos,
                               w.block_size, w.num_blocks, w.scale, self.max_ctx, copy_pairs,
                               self.fp8_scales, append=self.append)
        self.outs = outs
        self.copy_pairs = copy_pairs
        self.bytes_per_decode = decode_bytes(w, self.bt_host, self.ctx_host, 1 if fp8 else 2)
        self.partition_tokens = pa.pa_decode_partition_tokens(w.num_seqs, w.num_heads, self.max_ctx)
        self.max_parts = -(-self.max_ctx // self.partition_tokens)

    def launches_per_step(self) -> int:
        """Library kernels per step: slot map; per layer the cache write, the partition pass
        and (with several partitions) the merge (the step's workspace stays zeroed, so no
        work-counter init).  With the cache write fused into the decode: per layer the
        partition pass and the merge only."""
        L = len(self.dw.layers)
        if self.append:
            return L * (1 + (1 if self.max_parts > 1 else 0))
        per_layer = 2 + (1 if self.max_parts > 1 else 0)
        return 1 + L * per_layer + (1 if self.copy_pairs is not None else 0)


def timed(fn, K, device, world, stream):
    """Device time of K calls of fn (CUDA events on the launching stream, barrier and
    synchronize on both sides), max over ranks; ms for all K."""
    import torch
    barrier(world)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(K):
        fn(k)
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world)
    return max_over_ranks(t0.elapsed_time(t1), world)


def timed_flushed(fn, K, device, world, stream, flush):
    """Device time of K calls of fn, each timed alone with CUDA events on the launching stream
    after flush() has written a buffer of twice the L2 size (outside the events); sum over the
    calls in ms, max over ranks."""
    import torch
    barrier(world)
    torch.cuda.synchronize(device)
    evs = []
    for k in range(K):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn(k)
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize(device)
    barrier(world)
    return max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), world)


def measure_step(args, w, fp8: bool, device, world):
    """Everything the bench reports for one workload's decode step: the graph step (the
    value), the eager step with CUDA events around every decode call (the roofline's
    achieved), the clocks sampled during both, and the end-to-end step from pinned host
    buffers.  Returns (record, launches in the timed regions)."""
    import torch

    import paged_kv_cache_158_gb300 as pa

    st = Step(w, device, fp8, append=args.append)
    L = len(st.dw.layers)
    stream = torch.cuda.current_stream(device)
    for _ in range(args.warmup):
        st.step.run(stream)
    torch.cuda.synchronize(device)
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word after warm-up: {pa.pa_status_string(status)} 0x{bits:x}")

    K = args.steps
    # A step whose bytes fit in the L2 would be served from L2 when steps repeat: then every
    # timed step runs after a flush (a write of twice the L2 size, not timed).
    l2_bytes = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)) or (128 << 20)
    flush_buf = None
    if st.bytes_per_decode * L < l2_bytes:
        flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=device)

    def run_timed(fn):
        if flush_buf is None:
            return timed(fn, K, device, world, stream)
        return timed_flushed(fn, K, device, world, stream, lambda: flush_buf.fill_(1))

    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    time.sleep(0.3)
    # Eager pass: the step launched call by call, with CUDA events around every
    # decode call (the dominant kernel's duration, for the roofline).
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
          for _ in range(K)]
    ms_eager = run_timed(lambda k: st.step.run(stream, ev[k]))
    dec_ms = [a.elapsed_time(b) for row in ev for a, b in row]
    dec_avg_ms = sum(dec_ms) / len(dec_ms)
    # Graph pass: the same step captured once and replayed (the production configuration).
    ms_graph = None
    if not args.eager:
        st.step.capture(warmup=2)
        for _ in range(3):
            st.step.replay()
        ms_graph = run_timed(lambda k: st.step.replay())
    clk = clocks.stop()
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word after timing: {pa.pa_status_string(status)} 0x{bits:x}")

    ms_step = (ms_graph if ms_graph is not None else ms_eager) / K
    bytes_step = st.bytes_per_decode * L
    value = weak_scaling_value(bytes_step, world, ms_step)
    peak, peak_kind = measured_peak()
    achieved = st.bytes_per_decode / (dec_avg_ms * 1e-3) / 1e9
    ctx_tokens = int(st.ctx_host.sum())

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(st, args, world, device)
        if flush_buf is not None:
            e2e["l2"] = ("not flushed: consecutive steps run back to back, and this step's cache "
                         "fits in the L2, so it may be served from L2")
    rec = {
        "value": round(value, 2),
        "ms_per_step": round(ms_step, 4),
        "dtype": "e4m3 KV cache, f16 q/out, f32 accumulate" if fp8 else "f16 in, f32 accumulate",
        "config": {
            "workload": w.name,
            "kv_dtype": "fp8" if fp8 else "fp16",
            "layers": L, "num_seqs": w.num_seqs, "num_heads": w.num_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "num_blocks_per_layer": w.num_blocks,
            "context_tokens": ctx_tokens, "max_context_len": st.max_ctx,
            "partition_tokens": st.partition_tokens,
            "l2": ("inputs larger than L2: each layer's cache is read once per step"
                   if flush_buf is None else
                   f"L2 flushed before every timed step (a {2 * l2_bytes >> 20} MB write, not "
                   "timed); steps timed one by one with CUDA events"),
            "kv_pool_gb": round(w.pool_bytes_all_layers() / (2 if fp8 else 1) / 1e9, 3),
            "cuda_graph": ms_graph is not None,
            "cache_write": ("fused into the decode (pa_decode_append)" if st.append else
                            "slot map + pa_reshape_and_cache before each decode"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
        "us_per_layer": round(ms_step * 1e3 / L, 3),
        "decode_tokens_per_s_per_layer": round(w.num_seqs / (ms_step * 1e-3 / L), 1),
        "context_tokens_per_s_per_layer": round(ctx_tokens / (ms_step * 1e-3 / L), 1),
        "decode_bytes_per_layer": st.bytes_per_decode,
        "eager": {"value": round(weak_scaling_value(bytes_step, world, ms_eager / K), 2),
                  "ms_per_step": round(ms_eager / K, 4)},
        "roofline": {
            "bound": "hbm",
            "kernel": ("pa_decode_append" if st.append else "pa_decode") + ("_fp8" if fp8 else "") +
                      (" (partition kernel with the new token's cache write fused in, + merge;"
                       if st.append else " (partition + merge kernels;") +
                      " workspace kept zeroed; CUDA events bracket each call in the eager pass;"
                      " bytes are the decode's alone: the 4*S*H*D*elem of the fused write are"
                      " not counted)",
            "achieved": round(achieved, 2),
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "launch_us": round(dec_avg_ms * 1e3, 3),
            "launch_us_p10_p50_p90": [round(float(np.percentile(dec_ms, q)) * 1e3, 3) for q in (10, 50, 90)],
            "bytes_per_launch": st.bytes_per_decode,
            "traffic": committed_traffic(w.name + ("_fp8" if fp8 else "")),
        },
        "clocks": clk,
        "e2e": e2e,
    }
    launches = st.launches_per_step() * K * (2 if ms_graph is not None else 1)
    if e2e is not None:  # the end-to-end pass is timed too
        launches += st.launches_per_step() * e2e["steps"]
    del st
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()
    return rec, launches


def run_ours(args, rank, world, local):
    import torch

    import paged_kv_cache_158_gb300 as pa

    device = torch.device("cuda", local if world > 1 else 0)
    if args.partition_tokens:
        pa.pa_decode_set_partition_tokens(args.partition_tokens)
    w = make_workload(args.workload, args.layers)
    fp8 = args.kv_dtype == "fp8"
    rec, launches = measure_step(args, w, fp8, device, world)
    line = {
        "metric": "paged-decode KV GB/s (algorithmic q + gathered K/V + out bytes over step time)",
        "value": rec["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": rec["dtype"],
        "data": "synthetic (seeded SplitMix64 / Box-Muller values, seeded block tables)",
    }
    line.update({k: v for k, v in rec.items() if k not in line})
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=12.0, fp8=fp8)
    # The other workload with a bandwidth target, measured the same way in the same process
    # (single GPU only): one record per workload under "also".
    extra = [x for x in args.also.split(",") if x and x != "none" and x != args.workload]
    if world == 1 and extra:
        line["also"] = []
        for name in extra:
            wx = make_workload(name, 0)
            rx, lx = measure_step(args, wx, fp8, device, world)
            rx["metric"] = line["metric"]
            rx["unit"] = "GB/s"
            if rank == 0 and not args.no_cpu_baseline:
                rx["cpu_baseline"] = cpu_baseline(wx, budget_s=6.0, fp8=fp8, single_thread_s=0.0)
            line["also"].append(rx)
            launches += lx
    line["gpu_launches"] = launches
    return line


def measure_e2e(st, args, world, device):
    """Same metric through the public API with the step's inputs in pinned host memory:
    every step copies q / new K,V / token ids / tables / lengths host->device and reads every
    layer's output back (DecodeStep.bind_host: the uploads run ahead of the compute on a copy
    stream, the outputs go back on a second one right behind the decodes), as a graph replay
    unless --eager."""
    import torch
    dw = st.dw
    pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
    # Each kind's per-layer host buffers are views of one pinned [L, ...] tensor, like the
    # device ones, so the step merges consecutive layers' copies.
    h_q = list(pin(torch.stack(dw.queries)).unbind(0))
    h_k = list(pin(torch.stack(dw.keys_new)).unbind(0))
    h_v = list(pin(torch.stack(dw.values_new)).unbind(0))
    # The small int32 inputs back to back in one pinned buffer (one upload, like the device side).
    smalls = (dw.block_tables, dw.context_lens, dw.token_seq, dw.token_pos)
    flat = pin(torch.cat([t.reshape(-1) for t in smalls]))
    h_small, off = [], 0
    for t in smalls:
        h_small.append(flat[off:off + t.numel()].view(t.shape))
        off += t.numel()
    h_out = list(torch.empty((len(st.outs),) + tuple(st.outs[0].shape), dtype=st.outs[0].dtype,
                             pin_memory=True).unbind(0))
    h2d = sum(t.numel() * t.element_size() for t in h_q + h_k + h_v + h_small)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    st.step.bind_host(h_q, h_k, h_v, h_out, *h_small)
    K = max(3, min(args.steps, 100))
    use_graph = not args.eager
    if use_graph:
        st.step.capture(warmup=2, host=True)
        one = lambda: st.step.replay(host=True)  # noqa: E731
    else:
        one = st.step.run_host
    for _ in range(3):
        one()
    torch.cuda.synchronize(device)
    for i, o in enumerate(st.outs):  # the host copies are the device results
        if not torch.equal(h_out[i].view(torch.int16), o.cpu().view(torch.int16)):
            raise RuntimeError(f"host output of layer {i} differs from the device output")
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(K):
        one()
    torch.cuda.synchronize(device)
    dt = max_over_ranks(time.perf_counter() - t0, world) / K
    L = len(dw.layers)
    return {"value": round(st.bytes_per_decode * L * world / dt / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(dt * 1e3, 4), "steps": K, "cuda_graph": use_graph,
            "copies": "uploads on a copy stream ahead of the compute (waits at layers 0, 1, 2, 4, "
                      "...; the group starting at layer g is copied once the compute reaches "
                      "layer g // 2); outputs read back on a second copy stream right behind the "
                      "decodes; "
                      "one copy per layer group and tensor kind (per-layer buffers are views of "
                      "one [L, ...] tensor on each side)",
            "copies_per_step": sum(len(r) for r in st.step.host["up_runs"].values()) +
                               sum(len(r) for r in st.step.host["down_runs"].values()) +
                               len(st.step.host["small_runs"]),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def run_swap(args):
    """Swap-out and swap-in of whole sequences' blocks (every layer's K and V) between the
    device pool and pinned host memory through pa_swap_blocks, against one contiguous
    copy-engine transfer of the same bytes (torch copy_ between a device buffer and a
    pinned buffer) as the link's reference rate."""
    import torch

    import paged_kv_cache_158_gb300 as pa
    w = make_workload(args.workload, args.layers)
    dev = torch.device("cuda", 0)
    fp8 = args.kv_dtype == "fp8"
    dt = torch.uint8 if fp8 else torch.float16
    shape = (w.num_blocks, w.num_heads, w.block_size, w.head_dim)
    L = w.num_layers
    caches = [torch.empty(shape, dtype=dt, device=dev) for _ in range(2 * L)]
    for c in caches:
        c.view(torch.uint8).random_(0, 256)
    nswap = max(1, w.num_seqs // 16)
    blocks = np.concatenate([w.block_tables[s, :-(-int(w.context_lens[s]) // w.block_size)]
                             for s in range(nswap)]).astype(np.int64)
    nb = len(blocks)
    host = [torch.empty((nb,) + shape[1:], dtype=dt).pin_memory() for _ in range(2 * L)]
    out_map = torch.from_numpy(np.stack([blocks, np.arange(nb)], 1).copy()).to(dev)
    in_map = torch.from_numpy(np.stack([np.arange(nb), blocks], 1).copy()).to(dev)
    nbytes = nb * host[0][0].numel() * host[0].element_size() * 2 * L
    stream = torch.cuda.current_stream(dev)
    K, W = max(3, min(args.steps, 30)), max(3, args.warmup)

    def t_of(fn):
        for _ in range(W):
            fn()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / K * 1e-3

    t_out = t_of(lambda: pa.pa_swap_blocks(host, caches, out_map))
    t_in = t_of(lambda: pa.pa_swap_blocks(caches, host, in_map))
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word: {pa.pa_status_string(status)} 0x{bits:x}")
    flat_d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    t_d2h = t_of(lambda: flat_h.copy_(flat_d, non_blocking=True))
    t_h2d = t_of(lambda: flat_d.copy_(flat_h, non_blocking=True))
    gbs = lambda t: round(nbytes / t / 1e9, 2)  # noqa: E731
    return {
        "metric": "block swap GB/s (bytes of the swapped blocks over the call's device time)",
        "value": gbs(t_out), "unit": "GB/s", "n_gpus": 1, "steps": K, "warmup": W,
        "higher_is_better": True, "dtype": "e4m3" if fp8 else "f16", "data": "synthetic",
        "config": {"workload": w.name, "kv_dtype": args.kv_dtype, "layers": L,
                   "sequences_swapped": nswap, "blocks": nb, "caches": 2 * L,
                   "bytes_per_direction": nbytes},
        "swap_out_gbs": gbs(t_out), "swap_in_gbs": gbs(t_in),
        "swap_out_ms": round(t_out * 1e3, 3), "swap_in_ms": round(t_in * 1e3, 3),
        "copy_engine_reference": {"d2h_gbs": gbs(t_d2h), "h2d_gbs": gbs(t_h2d),
                                  "what": "one contiguous transfer of the same bytes"},
        "frac_of_copy_engine": {"out": round(t_d2h / t_out, 3), "in": round(t_h2d / t_in, 3)},
        "gpu_launches": 2 * (K + W),
        "cpu_baseline": None if args.no_cpu_baseline else swap_cpu_baseline(host, nb, budget_s=5.0),
    }


def swap_cpu_baseline(host_caches, nb: int, budget_s: float):
    """The oracle's block swap between two host pools with the blocks, caches and block size of
    the timed swap (the same bytes per call)."""
    import oracle
    src = [t.numpy().view(np.uint8).reshape(nb, -1) for t in host_caches]
    dst = [np.empty_like(a) for a in src]
    mapping = np.stack([np.arange(nb), np.arange(nb)[::-1]], 1).astype(np.int64)
    nbytes = sum(a.nbytes for a in src)
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps < 1:
        t0 = time.perf_counter()
        assert oracle.swap_blocks(dst, src, mapping) == 0
        t_total += time.perf_counter() - t0
        reps += 1
    return {"value": round(nbytes * reps / t_total / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "sample": f"{nb} blocks x {len(src)} caches host to host, {reps} repetitions, "
                                        f"{t_total:.1f} s", "host_cpus": os.cpu_count()}


def prefill_flops(w) -> int:
    """Algorithmic FLOPs of a chunked-prefill call: a new token at position p costs
    4*D*(p+1) FLOPs per head (2*D for each of its p+1 dot products q.K_i and 2*D for each
    of the p+1 accumulations p_i V_i); masked work is not counted."""
    tot = 0
    for ql, c in zip(w.extra["q_lens"], w.context_lens):
        ql, c = int(ql), int(c)
        pos = np.arange(c - ql, c, dtype=np.int64)
        tot += int((pos + 1).sum())
    return 4 * w.head_dim * w.num_heads * tot


def run_cache(args):
    """The step's cache write (layer 0: every new token of the step into its slot) and, for the
    shared-prefix workload, its copy-on-write block copies (every layer), each timed alone with
    CUDA events; GB/s = (bytes read + bytes written) / time.  KB-scale writes are launch-bound;
    the shared-prefix step writes 49 k tokens (0.8 GB each way)."""
    import torch

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = make_workload(args.workload, args.layers)
    fp8 = args.kv_dtype == "fp8"
    st = Step(w, dev, fp8=fp8)
    pa, dw = st.pa, st.dw
    T = dw.token_seq.numel()
    H, D, B = w.num_heads, w.head_dim, w.block_size
    elem = 1 if fp8 else 2
    slots = torch.empty(T, dtype=torch.int64, device=dev)
    pa.pa_slot_mapping(slots, dw.block_tables, dw.token_seq, dw.token_pos, B, w.num_blocks)
    K, W = max(3, min(args.steps, 200)), max(3, args.warmup)

    def timed(fn):
        """Mean device time of one call: K calls captured in a CUDA graph and replayed, so
        the host's per-call cost (argument marshalling, launch) is not timed."""
        for _ in range(W):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(K):
                fn()
        g.replay()
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        stream = torch.cuda.current_stream(dev)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / K * 1e-3

    def write():
        if fp8:
            pa.pa_reshape_and_cache_fp8(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                        dw.value_caches[0], slots, *st.fp8_scales)
        else:
            pa.pa_reshape_and_cache(dw.keys_new[0], dw.values_new[0], dw.key_caches[0],
                                    dw.value_caches[0], slots)

    t_w = timed(write)
    wbytes = T * H * D * (2 * 2 + elem * 2)          # fp16 K/V read, cache elements written
    out = {"metric": "cache write and copy-on-write block copy GB/s ((bytes read + bytes written) "
                     "over CUDA-event time)",
           "value": round(wbytes / t_w / 1e9, 2), "unit": "GB/s", "n_gpus": 1, "steps": K,
           "warmup": W, "higher_is_better": True, "dtype": args.kv_dtype, "data": "synthetic",
           "config": {"workload": w.name, "kv_dtype": args.kv_dtype, "new_tokens": T},
           "cache_write": {"tokens": T, "bytes": wbytes, "us": round(t_w * 1e6, 3),
                           "gbs": round(wbytes / t_w / 1e9, 2)},
           "timing": "K calls captured in one CUDA graph, one replay timed with CUDA events",
           "gpu_launches": 2 * K + W}
    if st.copy_pairs is not None and st.copy_pairs.numel():
        P = st.copy_pairs.shape[0]
        copy = (lambda: pa.pa_copy_blocks_fp8(dw.key_caches, dw.value_caches, st.copy_pairs)) if fp8 \
            else (lambda: pa.pa_copy_blocks(dw.key_caches, dw.value_caches, st.copy_pairs))
        t_c = timed(copy)
        cbytes = P * len(dw.layers) * 2 * H * B * D * elem * 2
        out["block_copy"] = {"pairs": P, "layers": len(dw.layers), "bytes": cbytes,
                             "us": round(t_c * 1e6, 3), "gbs": round(cbytes / t_c / 1e9, 2),
                             "note": "source and destination blocks fit in L2"}
        out["gpu_launches"] += 2 * K + W
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word: {pa.pa_status_string(status)} 0x{bits:x}")
    return out


def run_scan(args):
    """Decode time per call against context length: the workload's batch shape (S, H, D, B)
    with every sequence at one context length c in {256 .. 4096}, each point timed as a CUDA
    graph of calls over distinct layers (more than 2 GB of cache per replay, so nothing is
    served from L2).  A least-squares line time = fixed + bytes / marginal splits each call's
    time into a per-call fixed part (launch chain, ramp-up and drain, the tail of the last
    items, the merge) and the streaming rate of the partition pass."""
    import torch

    import paged_kv_cache_158_gb300 as pa

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = make_workload(args.workload, 1)
    S, H, D, B = w.num_seqs, w.num_heads, w.head_dim, w.block_size
    fp8 = args.kv_dtype == "fp8"
    elem = 1 if fp8 else 2
    if args.partition_tokens:
        pa.pa_decode_set_partition_tokens(args.partition_tokens)
    gen = torch.Generator(device=dev)
    gen.manual_seed(158100)
    K = max(3, min(args.steps, 20))
    points, launches = [], 0
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    clocks.start()
    for c in (256, 512, 1024, 2048, 4096):
        nbl = (c + B - 1) // B
        NB = S * nbl
        layer_bytes = 2 * NB * H * B * D * elem
        L = max(2, int(2.5e9 // layer_bytes))
        caches = []
        for _ in range(L):
            pair = []
            for _kv in range(2):
                if fp8:  # random codes with bit 3 clear: never an E4M3 NaN
                    x = torch.randint(0, 256, (NB, H, B, D), dtype=torch.uint8, device=dev,
                                      generator=gen) & 0xF7
                else:
                    x = torch.randn((NB, H, B, D), dtype=torch.float16, device=dev, generator=gen)
                pair.append(x)
            perm = torch.randperm(NB, device=dev, generator=gen).to(torch.int32)
            caches.append((pair[0], pair[1], perm.view(S, nbl).contiguous()))
        q = torch.randn((S, H, D), dtype=torch.float16, device=dev, generator=gen)
        out = torch.empty_like(q)
        ctx = torch.full((S,), c, dtype=torch.int32, device=dev)
        ws = pa.decode_workspace(S, H, D, c, device=dev)
        scale = 1.0 / D ** 0.5

        def calls():
            for kc, vc, bt in caches:
                if fp8:
                    pa.pa_decode_fp8(out, q, kc, vc, bt, ctx, scale, 0.02, 0.02, c, ws)
                else:
                    pa.pa_decode(out, q, kc, vc, bt, ctx, scale, c, ws)

        for _ in range(max(3, args.warmup)):
            calls()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                calls()
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        stream = torch.cuda.current_stream(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        us = a.elapsed_time(b) * 1e3 / (K * L)
        nbytes = decode_bytes(w, None, np.full(S, c), elem)
        points.append({"context_len": c, "layers": L, "us_per_call": round(us, 3),
                       "bytes_per_call": nbytes, "gbs": round(nbytes / us / 1e3, 1),
                       "partition_tokens": pa.pa_decode_partition_tokens(S, H, c)})
        launches += K * L * 3 + max(3, args.warmup) * L * 3
        del caches, g
        torch.cuda.empty_cache()
    clk = clocks.stop()
    pa.pa_decode_set_partition_tokens(0)
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word: {pa.pa_status_string(status)} 0x{bits:x}")
    xb = np.array([p["bytes_per_call"] for p in points], dtype=np.float64)
    yt = np.array([p["us_per_call"] for p in points], dtype=np.float64)
    slope, fixed = np.polyfit(xb, yt, 1)
    marginal = 1.0 / slope / 1e3  # bytes per us -> GB/s
    peak, kind = measured_peak()
    return {"metric": "paged-decode time per call vs context length: fixed us per call and "
                      "marginal GB/s (least-squares line over the points)",
            "value": round(marginal, 1), "unit": "GB/s", "n_gpus": 1, "steps": K,
            "warmup": max(3, args.warmup), "higher_is_better": True, "dtype": args.kv_dtype,
            "data": "synthetic (seeded torch generator; FP8 codes with bit 3 clear)",
            "config": {"workload": f"{w.name} batch shape, uniform context lengths",
                       "num_seqs": S, "num_heads": H, "head_dim": D, "block_size": B,
                       "kv_dtype": args.kv_dtype, "l2": "more than 2 GB of cache per replay"},
            "fixed_us_per_call": round(float(fixed), 2), "marginal_gbs": round(marginal, 1),
            "marginal_frac_of_peak": round(marginal / peak, 4), "peak_gbs": peak, "peak_kind": kind,
            "points": points, "clocks": clk, "gpu_launches": launches}


def run_prefill_bench(args):
    import torch

    import paged_kv_cache_158_gb300 as pa
    from workloads import gpu
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    w = configs.prefill_7b_mixed() if args.prefill_workload == "mixed" else configs.prefill_7b()
    fp8 = args.kv_dtype == "fp8"
    ks, vs = configs.fp8_scales(w)
    tq = int(np.sum(w.extra["q_lens"]))
    # Consecutive calls rotate over NCOPY separate copies of the inputs (queries, pool, tables,
    # outputs), NCOPY x 100-170 MB in all, so no call finds the previous one's data in L2.
    NCOPY = 3
    copies = []
    for _ in range(NCOPY):
        dv = gpu.materialize_prefill(w, dev)
        if fp8:  # the same pool as E4M3 codes (the library's conversion)
            for name, sc in (("key_cache", ks), ("value_cache", vs)):
                codes = torch.empty(dv[name].shape, dtype=torch.uint8, device=dev)
                pa.pa_convert_cache_fp8(dv[name], codes, sc)
                dv[name] = codes
        dv["out"] = torch.empty((tq, w.num_heads, w.head_dim), dtype=torch.float16, device=dev)
        copies.append(dv)
    max_q = int(max(w.extra["q_lens"]))
    stream = torch.cuda.current_stream(dev)
    input_bytes = sum(t.numel() * t.element_size() for t in copies[0].values())

    # Consecutive calls work on independent copies: the kernel before each call writes only its
    # own output, so the calls pass PA_PREFILL_INPUTS_READY and a call's first CTAs start on the
    # SMs the previous call's last wave leaves idle.  The same calls without the flag (each
    # waits for the previous one before it reads anything) are timed too: serial_ms_per_call.
    # The caller knows its batch: it passes the count of one-token sequences, which sizes the
    # launch exactly and lets one CTA run four heads of a decode row.
    n_rows = int(np.sum(np.asarray(w.extra["q_lens"]) == 1))

    def call(i=0, flags=pa.PA_PREFILL_INPUTS_READY):
        dv = copies[i % NCOPY]
        args = (dv["out"], dv["query"], dv["key_cache"], dv["value_cache"], dv["block_tables"],
                dv["context_lens"], dv["query_start"], w.scale)
        if fp8:
            pa.pa_prefill_fp8_ex(*args, ks, vs, max_q, n_rows, flags)
        else:
            pa.pa_prefill_ex(*args, max_q, n_rows, flags)

    K, W = max(3, min(args.steps, 200)), max(3, args.warmup)
    for i in range(W):
        call(i)
    torch.cuda.synchronize(dev)
    status, bits = pa.pa_check_errors()
    if status != pa.PA_OK:
        raise RuntimeError(f"device error word: {pa.pa_status_string(status)} 0x{bits:x}")
    clocks = ClockSampler(None)
    clocks.start()
    time.sleep(0.3)

    def time_calls(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(K):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / K * 1e-3

    sec = time_calls(call)
    sec_serial = time_calls(lambda i: call(i, 0))
    split = None
    if args.prefill_workload == "mixed":
        split = mixed_split_timing(w, copies, fp8, ks, vs, time_calls, W)
        # Both sides serial (no call starts before the previous one ends).
        split["mixed_ms"] = round(sec_serial * 1e3, 4)
        split["mixed_over_separate"] = round(sec_serial * 1e3 / split["separate_ms"], 4)
    clk = clocks.stop()
    flops = prefill_flops(w)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; fp16 runs at the bf16 rate)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    kv_bytes = int(np.sum(w.context_lens)) * w.num_heads * w.head_dim * 2 * (1 if fp8 else 2)
    tflops = flops / sec / 1e12
    return {
        "metric": "multi-query paged attention TFLOP/s (causal algorithmic FLOPs over call time)",
        "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": 1, "steps": K, "warmup": W,
        "ms_per_call": round(sec * 1e3, 4), "higher_is_better": True,
        "serial_ms_per_call": round(sec_serial * 1e3, 4),
        "serial_tflops": round(flops / sec_serial / 1e12, 2),
        "dtype": ("e4m3 KV cache widened to f16" if fp8 else "f16") + " operands, f32 accumulate",
        "data": "synthetic", "config": {"workload": w.name, "kv_dtype": args.kv_dtype,
                                        "num_seqs": w.num_seqs,
                                        "num_heads": w.num_heads, "head_dim": w.head_dim,
                                        "block_size": w.block_size, "query_tokens": tq,
                                        "context_tokens": int(np.sum(w.context_lens)),
                                        "num_decode_rows_passed": n_rows,
                                        "l2": f"inputs larger than L2: consecutive calls rotate "
                                              f"over {NCOPY} copies of the inputs "
                                              f"({NCOPY * input_bytes / 1e6:.0f} MB in all)"},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "peak_kind": kind,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "flops_per_call": flops,
                     "kv_bytes_per_call": kv_bytes,
                     "kv_gbs": round(kv_bytes / sec / 1e9, 1)},
        "clocks": clk, "gpu_launches": (2 * K + W) * (1 if split is None else 4),
        "separate_calls": split,
        "cpu_baseline": None if args.no_cpu_baseline else prefill_cpu_baseline(w, budget_s=10.0,
                                                                               fp8=fp8),
    }


def mixed_split_timing(w, copies, fp8, ks, vs, time_calls, warmup):
    """The mixed batch's two parts as separate calls on the same inputs: pa_prefill over the
    chunk sequences only and pa_decode over the decode sequences only (their query rows are
    contiguous after the chunks'), each timed over the same input rotation."""
    import torch

    import paged_kv_cache_158_gb300 as pa
    ql = np.asarray(w.extra["q_lens"])
    nch = int(np.sum(ql > 1))
    assert np.all(ql[:nch] > 1) and np.all(ql[nch:] == 1), "chunks first, then decode rows"
    qs = configs.query_start(w)
    r0 = int(qs[nch])
    max_q = int(ql[:nch].max())
    dec_ctx = int(w.context_lens[nch:].max())
    ws = [pa.decode_workspace(len(ql) - nch, w.num_heads, w.head_dim, dec_ctx) for _ in copies]
    n = len(copies)

    def chunks(i):
        dv = copies[i % n]
        args = (dv["out"][:r0], dv["query"][:r0], dv["key_cache"], dv["value_cache"],
                dv["block_tables"][:nch], dv["context_lens"][:nch], dv["query_start"][:nch + 1],
                w.scale)
        if fp8:
            pa.pa_prefill_fp8(*args, ks, vs, max_q)
        else:
            pa.pa_prefill(*args, max_q)

    def decode(i):
        dv = copies[i % n]
        args = (dv["out"][r0:], dv["query"][r0:], dv["key_cache"], dv["value_cache"],
                dv["block_tables"][nch:], dv["context_lens"][nch:], w.scale)
        if fp8:
            pa.pa_decode_fp8(*args, ks, vs, dec_ctx, ws[i % n])
        else:
            pa.pa_decode(*args, dec_ctx, ws[i % n])

    for i in range(warmup):
        chunks(i)
        decode(i)
    torch.cuda.synchronize()
    t_c = time_calls(chunks)
    t_d = time_calls(decode)
    t_both = time_calls(lambda i: (chunks(i), decode(i)))
    return {"chunk_sequences": nch, "decode_sequences": len(ql) - nch,
            "prefill_chunks_ms": round(t_c * 1e3, 4), "decode_rows_ms": round(t_d * 1e3, 4),
            "separate_ms": round(t_both * 1e3, 4),
            "what": "pa_prefill over the chunk sequences then pa_decode over the decode "
                    "sequences, back to back on one stream"}


def prefill_cpu_baseline(w, budget_s: float, fp8: bool = False):
    """The oracle's multi-query attention on a bounded sample of the same workload: the last
    32 new tokens of sequence 0 over its whole context, every head (the causally truncated
    problem that gives exactly those rows)."""
    import oracle
    from workloads import gpu
    kc, vc = gpu.host_pool(w, 0)
    ks, vs = configs.fp8_scales(w)
    if fp8:
        kc, vc = oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)
    q = gpu.host_queries(w)
    qs = configs.query_start(w)
    ql, c, n = int(w.extra["q_lens"][0]), int(w.context_lens[0]), 32
    rows = q[qs[0] + ql - n:qs[0] + ql]
    bt = w.block_tables[0:1]
    flops = 4 * w.head_dim * w.num_heads * sum(range(c - n + 1, c + 1))
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps < 1:
        t0 = time.perf_counter()
        if fp8:
            _, _, rc = oracle.prefill_fp8(rows, kc, vc, bt, np.array([c], np.int32),
                                          np.array([0, n], np.int32), w.scale, ks, vs, want64=False)
        else:
            _, _, rc = oracle.prefill(rows, kc, vc, bt, np.array([c], np.int32),
                                      np.array([0, n], np.int32), w.scale, want64=False)
        t_total += time.perf_counter() - t0
        reps += 1
        assert rc == 0
    return {"value": round(flops * reps / t_total / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{w.name}: last {n} new tokens of sequence 0 over its {c}-token context, "
                      f"all {w.num_heads} heads, {reps} repetitions, {t_total:.1f} s",
            "host_cpus": os.cpu_count()}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, fp8: bool = False, seqs: int | None = None):
    """Host inputs of the bounded sample: layer 0 of the workload, every head of the first
    `seqs` sequences (default: all), and a call running the oracle's decode on them (FP8: the
    oracle quantises the pool)."""
    import oracle
    from workloads import gpu
    if w.block_tables is None:
        raise ValueError("the CPU baseline sample needs static block tables")
    kc, vc = gpu.host_pool(w, 0)
    q, _, _ = gpu.host_small(w, 0)
    n = w.num_seqs if seqs is None else seqs
    q, bt, ctx = q[:n], w.block_tables[:n], w.context_lens[:n]
    if fp8:
        ks, vs = configs.fp8_scales(w)
        kc, vc = oracle.quantize_e4m3(kc, ks), oracle.quantize_e4m3(vc, vs)
        return oracle, lambda: oracle.decode_fp8(q, kc, vc, bt, ctx, w.scale, ks, vs, want64=False)
    return oracle, lambda: oracle.decode(q, kc, vc, bt, ctx, w.scale, want64=False)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _time_oracle(run, budget_s: float):
    reps, t_total = 0, 0.0
    while t_total < budget_s or reps < 1:
        t0 = time.perf_counter()
        _, _, rc = run()
        t_total += time.perf_counter() - t0
        reps += 1
        assert rc == 0
    return reps, t_total


def cpu_baseline(w, budget_s: float, fp8: bool = False, single_thread_s: float = 4.0):
    """The oracle's decode of layer 0 on all host cores for about budget_s seconds, and (if
    single_thread_s > 0) on one core for about that long over the first 4 sequences."""
    oracle, run = oracle_sample(w, fp8)
    nbytes = decode_bytes(w, w.block_tables, w.context_lens, 1 if fp8 else 2)
    reps, t_total = _time_oracle(run, budget_s)
    out = {"value": round(nbytes * reps / t_total / 1e9, 4), "unit": "GB/s",
           "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{w.name} layer 0 decode (all {w.num_seqs} seqs x {w.num_heads} heads), "
                     f"{reps} repetitions, {t_total:.1f} s",
           "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}
    if single_thread_s > 0:
        n = min(4, w.num_seqs)
        _, run1 = oracle_sample(w, fp8, seqs=n)
        nb1 = decode_bytes(w, w.block_tables[:n], w.context_lens[:n], 1 if fp8 else 2)
        threads = oracle.num_threads()
        oracle.set_num_threads(1)
        try:
            r1, t1 = _time_oracle(run1, single_thread_s)
        finally:
            oracle.set_num_threads(threads)
        out["single_thread"] = {"value": round(nb1 * r1 / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                                "sample": f"{w.name} layer 0 decode of sequences 0..{n - 1} (all "
                                          f"{w.num_heads} heads), {r1} repetitions, {t1:.1f} s"}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = make_workload(args.workload, 1)
    fp8 = args.kv_dtype == "fp8"
    oracle, run = oracle_sample(w, fp8)
    nbytes = decode_bytes(w, w.block_tables, w.context_lens, 1 if fp8 else 2)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = f"{w.name} layer 0 decode per step (all {w.num_seqs} seqs x {w.num_heads} heads)"
    return {
        "impl": "reference",
        "metric": "paged-decode KV GB/s (algorithmic q + gathered K/V + out bytes over step time)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "kv_dtype": args.kv_dtype, "layers": 1, "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        line = run_reference(args, int(os.environ.get("RANK", "0")), world_env)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.op == "prefill":
        print(json.dumps(run_prefill_bench(args)), flush=True)
        return
    if args.op == "swap":
        import torch
        torch.cuda.set_device(0)
        print(json.dumps(run_swap(args)), flush=True)
        return
    if args.op == "cache":
        print(json.dumps(run_cache(args)), flush=True)
        return
    if args.op == "scan":
        print(json.dumps(run_scan(args)), flush=True)
        return
    rank, world, local = dist_setup(args.gpus)
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
