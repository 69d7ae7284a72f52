#!/usr/bin/env python
"""Decode-step benchmark of the quantized paged KV path on GB300.

One step = one decode step through every layer of a workload's model.  Each
layer appends the new token's K/V row (quantized into its page) and runs the
decode attention over the layer's whole cache, in one fused call
(kvq_append_decode_attention, or kvq_append_window_decode for a sliding-window
layer).  The step is captured once in a CUDA graph and replayed.

The headline workload (default: the continuous batch, the largest single-GPU
configuration) is timed, and so is every other configuration in `per_config`:
the Llama-3.1-8B-shaped model, the sliding-window and the global layers of the
sliding + global mix (separately and together) and the long mixed-dtype
context.  Each is timed in blocks of exactly K steps, each block bracketed by a
barrier and a device synchronize, and reports the median block.  A model whose
caches together are smaller than twice the L2 cache gets an L2 flush before
every timed step instead.

Printed (rank 0, one JSON line): decode-attention KV GB/s for the whole job
(algorithmic bytes / step time), query and context tokens/s, the roofline of
the fused call, the end-to-end number through host buffers, clocks seen during
the timed region, per-configuration results, and the CPU oracle timed on a
bounded sample of the same work.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...      # the CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kvq_workloads as wl  # noqa: E402

METRIC = "decode-attention KV GB/s and % of HBM peak; attention tokens/s at 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0

# Layers of each model: (workload, number of layers, window decode?)
MODELS = {
    "contbatch": [("contbatch", 1, False)],                    # 1.16 GB per layer already > L2
    "llama8b": [("llama8b", 32, False)],                       # Llama-3.1-8B: 32 layers
    "gemma_mix": [("gemma_mix", 25, True), ("gemma_mix", 5, False)],   # 25 window + 5 global
    "gemma_window": [("gemma_mix", 25, True)],                 # the window layers of gemma_mix
    "gemma_global": [("gemma_mix", 5, False)],                 # the global layers of gemma_mix
    "long_mixed": [("long_mixed", 4, False)],
    # the unquantised f16 K/V the pages compare with (8K and 64K)
    "llama8b_f16": [("llama8b_f16", 32, False)],
    "long_f16": [("long_f16", 4, False)],
    # the /7.5 offset-8 4-bit codec (8K and 64K)
    "llama8b_shimmy": [("llama8b_shimmy", 32, False)],
    "long_shimmy": [("long_shimmy", 4, False)],
}
# Configurations timed besides the headline one.
PER_CONFIG = ("contbatch", "llama8b", "gemma_window", "gemma_global", "gemma_mix", "long_mixed")


# ----------------------------------------------------------------------------- helpers


def kv_bytes_per_token_head(kind: str, head_dim: int, group: int, param: str) -> int:
    """Stored bytes of one token's K or V vector for one kv head: codes plus the
    scale (and bias) of every group; f16 rows have no scale."""
    if kind == "f16":
        return 2 * head_dim
    bits = 8 if kind == "sym8" else 4
    n_par = 2 if kind == "affine4" else 1
    return head_dim * bits // 8 + (head_dim // group) * n_par * (4 if param == "f32" else 2)


def algorithmic_bytes(w: dict, lens: np.ndarray, window: int) -> tuple[int, int]:
    """(decode-call bytes, append-call bytes) the method must move.

    Decode: K/V codes and scales of every attended token, q, out, the block-table
    entries it reads and seq_lens.  Append: the new K/V rows, the RoPE row,
    positions, and the codes and scales written.
    """
    hd, hkv, hq = w["head_dim"], w["n_kv_heads"], w["n_heads"]
    act = 4 if w["act"] == "f32" else 2
    per_tok = (kv_bytes_per_token_head(w["k_kind"], hd, w["k_group"], w["k_param"])
               + kv_bytes_per_token_head(w["v_kind"], hd, w["v_group"], w["v_param"]))
    att = np.minimum(lens, window) if window else lens
    B = len(lens)
    dec = int(att.sum()) * hkv * per_tok + 2 * B * hq * hd * act + 4 * int(np.ceil(att / 16).sum()) + 4 * B
    app = B * (2 * hkv * hd * act + 4 * hd + 8 + hkv * per_tok)
    return dec, app


KERNEL_SOURCES = tuple("int8_quantized_paged_gb300/csrc/" + f for f in (
    "kvq_decode_tc.cuh", "kvq_tc_ptx.cuh", "kvq_decode.cu", "kvq_quant.cuh", "kvq_decode_impl.cuh", "kvq_device.cuh"))


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes (read + write) of one decode launch of this workload from the
    committed ncu summary (profiles/traffic.txt), or None when there is none or
    the kernel sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload:
                    return int(parts[2]) if parts[1] == kernel_source_hash() else None
    except OSError:
        pass
    return None


def load_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or 'unknown'."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


class _Cu:
    """Driver-API events that can be recorded as graph nodes (external records)."""

    def __init__(self):
        self.lib = ctypes.CDLL("libcuda.so.1")
        self.lib.cuEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_uint]
        self.lib.cuEventRecordWithFlags.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]
        self.lib.cuEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        self.lib.cuEventDestroy_v2.argtypes = [ctypes.c_void_p]

    def event(self):
        e = ctypes.c_void_p()
        r = self.lib.cuEventCreate(ctypes.byref(e), 0)
        if r != 0:
            raise RuntimeError(f"cuEventCreate failed: {r}")
        return e

    def record_external(self, ev, stream_handle: int):
        r = self.lib.cuEventRecordWithFlags(ev, ctypes.c_void_p(stream_handle), 1)  # CU_EVENT_RECORD_EXTERNAL
        if r != 0:
            raise RuntimeError(f"cuEventRecordWithFlags failed: {r}")

    def elapsed_ms(self, a, b) -> float:
        ms = ctypes.c_float()
        r = self.lib.cuEventElapsedTime(ctypes.byref(ms), a, b)
        if r != 0:
            raise RuntimeError(f"cuEventElapsedTime failed: {r}")
        return ms.value


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # KVQ_CLOCKS_DIR keeps the samples where the caller wants them
        out = os.environ.get("KVQ_CLOCKS_DIR")
        self.path = os.path.join(out, f"clocks_gpu{gpu_index}.csv") if out and os.path.isdir(out) \
            else f"/tmp/kvq_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed


def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest value over all ranks (every rank gets it)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(units_per_rank: float, world: int, ms_max: float) -> float:
    """Units per second for the whole job: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def n_blocks_for(block_ms: float, min_blocks: int = 5, min_seconds: float = 1.0, max_blocks: int = 400) -> int:
    """How many timed blocks of block_ms each: at least min_blocks, and enough
    for about min_seconds of timed work (so the clock sampler sees the load),
    at most max_blocks."""
    want = math.ceil(min_seconds * 1e3 / max(block_ms, 1e-6))
    return int(min(max_blocks, max(min_blocks, want)))


def check_gpus_flag(gpus: int, world: int) -> str | None:
    """An error message when --gpus disagrees with the launch (WORLD_SIZE)."""
    if gpus != world:
        return (f"--gpus {gpus} but WORLD_SIZE is {world}: launch N ranks with "
                f"torch.distributed.run --nproc-per-node N bench.py --gpus N")
    return None


# ----------------------------------------------------------------------------- GPU arm


class BenchLayer:
    def __init__(self, w: dict, window: bool, layer: int, device, gen, chunk_tokens: int = 0,
                 rope_tab=None, flags: int = 0):
        import torch
        from int8_quantized_paged_gb300 import kvq
        from int8_quantized_paged_gb300.cache import LayerCache
        self.w = w
        self.lens = wl.seq_lens(w)
        self.B = len(self.lens)
        self.window = int(w["window"]) if window else 0
        self.ring = int(w["ring_rows"]) if window else 0
        cfg = kvq.config(**w, flags=flags)
        P = 16
        if self.ring:
            max_pages = self.ring // P
            n_pages = self.B * max_pages
        else:
            max_pages = int(math.ceil(self.lens.max() / P))
            n_pages = int(sum(math.ceil(L / P) for L in self.lens))
        pool = kvq.Pool(n_pages)
        if w.get("shuffle_pages"):
            pool.alloc(n_pages)
            pool.free(wl.page_free_order(w, n_pages))
        rope_max = int(self.lens.max()) + 1
        self.cache = LayerCache(cfg, self.B, max_pages, n_pages, rope_max, self.ring, device=device, pool=pool,
                                rope_tab=rope_tab)
        for b, L in enumerate(self.lens):
            self.cache.reserve(b, self.ring if self.ring else int(L))
        self.cache.sync_table()
        act = self.cache.act_dtype
        hkv, hd, hq = w["n_kv_heads"], w["head_dim"], w["n_heads"]

        def rows(n):
            x = torch.randn((n, hkv, hd), generator=gen, device=device, dtype=torch.float32)
            if w.get("outlier_frac", 0):
                m = torch.rand((n, hkv, hd), generator=gen, device=device) < w["outlier_frac"]
                x = torch.where(m, x * 8, x)
            return x.to(act)

        # Prefill every sequence (the product's append path, chunked so no call
        # writes one ring row twice).
        for b, L in enumerate(self.lens):
            step = self.ring if self.ring else int(L)
            for s in range(0, int(L), step):
                e = min(int(L), s + step)
                self.cache.append(rows(e - s), rows(e - s),
                                  torch.arange(s, e, dtype=torch.int32, device=device),
                                  torch.full((e - s,), b, dtype=torch.int32, device=device))
        # This step's inputs: the token at position L-1 of every sequence.
        self.q = torch.randn((self.B, hq, hd), generator=gen, device=device).to(act)
        self.k_new, self.v_new = rows(self.B), rows(self.B)
        self.pos = torch.from_numpy(self.lens - 1).to(device)
        self.seq_lens = torch.from_numpy(self.lens).to(device)
        self.out = torch.empty_like(self.q)
        self.chunk = chunk_tokens
        self.ws = self.cache.workspace(self.B, chunk_tokens, self.window)
        self.dec_bytes, self.app_bytes = algorithmic_bytes(w, self.lens, self.window)
        self.use_fused = True

    def append(self):
        self.cache.append(self.k_new, self.v_new, self.pos)

    def decode(self):
        if self.window:
            self.cache.window_decode(self.q, self.seq_lens, self.out, self.ws, self.window, self.chunk)
        else:
            self.cache.decode(self.q, self.seq_lens, self.out, self.ws, self.chunk)

    def fused(self) -> bool:
        """Whether step() makes one fused call (kvq_append_decode_attention or
        kvq_append_window_decode)."""
        return self.use_fused

    def step(self):
        """This layer's share of a decode step: append the new row, then decode."""
        if self.fused() and self.window:
            self.cache.append_window_decode(self.q, self.k_new, self.v_new, self.pos, self.seq_lens, self.out,
                                            self.ws, self.window, self.chunk)
        elif self.fused():
            self.cache.append_decode(self.q, self.k_new, self.v_new, self.pos, self.seq_lens, self.out, self.ws,
                                     self.chunk)
        else:
            self.append()
            self.decode()

    def launches(self) -> int:
        from int8_quantized_paged_gb300 import kvq
        if self.fused():
            return kvq.append_decode_launches(self.cache.cfg)
        return 1 + kvq.decode_launches(self.cache.cfg)


def early_reads(model: str, args) -> bool:
    """Whether a model's calls may read their pages before the kernel before
    them ends (KVQ_FLAG_EARLY_READS).  That kernel must write none of those
    inputs: true when it is another layer's fused call, not when a one-layer
    model's call follows its own previous step or a separate append."""
    n_layers = sum(n for _, n, _ in MODELS[model])
    return n_layers > 1 and not args.separate and not getattr(args, "no_early_reads", False)


def build_layers(model: str, args, dev, seed: int) -> list:
    """The layers of a model, caches prefilled on the device."""
    import torch
    from int8_quantized_paged_gb300 import kvq
    layers = []
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    flags = kvq.FLAG_EARLY_READS if early_reads(model, args) else 0
    rope_tabs = {}   # one RoPE table per model: every layer reads the same positions
    for name, n, window in MODELS[model]:
        w = wl.workload(name, **({"batch": args.batch} if args.batch else {}))
        if name not in rope_tabs:
            cfg = kvq.config(**w)
            rows = int(wl.seq_lens(w).max()) + 1
            rope_tabs[name] = (torch.from_numpy(kvq.rope_table(cfg, rows)).to(dev)
                               if cfg.rope != kvq.ROPE_NONE else None)
        for i in range(n):
            layers.append(BenchLayer(w, window, len(layers), dev, gen, args.chunk_tokens, rope_tabs[name], flags))
    # One decode step has one seq_lens and one positions array for all layers
    # of a model, as the model's layers share them; q and the new K/V rows
    # stay per layer.
    first = {}
    for L in layers:
        L.use_fused = not args.separate
        key = (L.w["name"], tuple(L.lens.tolist()))
        if key in first:
            L.seq_lens, L.pos = first[key].seq_lens, first[key].pos
        else:
            first[key] = L
    return layers


def stage_io(layers, dev):
    """Every layer's step inputs (q, k_new, v_new) as views of one device buffer
    and its outputs as views of another: a step's inputs then come over from
    host memory in one copy and its outputs go back in one, as a server would
    batch them.  Each view starts on a multiple of head_dim elements (>= 128 B).
    Returns (inputs, outputs), the two flat buffers."""
    import torch
    act = layers[0].q.dtype
    assert all(L.q.dtype == act for L in layers), "one activation dtype per model"

    def pack(tensors):
        buf = torch.empty(sum(t.numel() for t in tensors), dtype=act, device=dev)
        views, o = [], 0
        for t in tensors:
            v = buf[o:o + t.numel()].view(t.shape)
            v.copy_(t)
            views.append(v)
            o += t.numel()
        return buf, views

    io_in, v_in = pack([t for L in layers for t in (L.q, L.k_new, L.v_new)])
    io_out, v_out = pack([L.out for L in layers])
    for i, L in enumerate(layers):
        L.q, L.k_new, L.v_new = v_in[3 * i:3 * i + 3]
        L.out = v_out[i]
    return io_in, io_out


def run_profile(args) -> None:
    """The timed decode call of every layer (the fused append + decode call, or the
    decode alone), layer after layer, for profiler captures (no timing)."""
    import torch
    dev = torch.device("cuda", 0)
    from int8_quantized_paged_gb300 import build as _build
    _build.build()
    layers = build_layers(args.workload, args, dev, 1000)
    torch.cuda.synchronize()
    for _ in range(args.profile_decode):
        for L in layers:
            L.step() if L.fused() else L.decode()
    torch.cuda.synchronize()
    assert all(L.cache.status_bits() == 0 for L in layers), "a kernel flagged a bad input"
    print(f"profile-decode: {args.workload}, {len(layers)} layers x {args.profile_decode} calls, "
          f"{layers[0].dec_bytes} algorithmic bytes per call", flush=True)


def l2_bytes(dev) -> int:
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))


def time_blocks(run_step, steps: int, stream, world: int, n_blocks: int, flush=None) -> list[float]:
    """ms per step of each of n_blocks blocks of exactly `steps` steps.  Every
    block is bracketed by a barrier and a device synchronize.  Without `flush`
    the block's steps run back to back between two events; with it, `flush`
    (a write larger than L2) runs before every step, and the block's time is
    the sum of its steps' own event intervals."""
    import torch
    out = []
    for _ in range(n_blocks):
        barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            if flush is None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(steps):
                    run_step()
                e1.record(stream)
            else:
                evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                       for _ in range(steps)]
                for a, b in evs:
                    flush()
                    a.record(stream)
                    run_step()
                    b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        if flush is None:
            out.append(e0.elapsed_time(e1) / steps)
        else:
            out.append(sum(a.elapsed_time(b) for a, b in evs) / steps)
    return out


def time_pipelined(graphs, ins, outs, h_in, h_out, stream, steps: int, world: int, n_blocks: int) -> list[float]:
    """ms per step of n_blocks blocks of `steps` end-to-end steps, pipelined over
    two buffer sets: step i uploads its inputs into set i % 2 on a copy stream
    (once the step that last read that set has run), the compute stream replays
    that set's graph, and a second copy stream brings its outputs back.  So the
    upload of step i+1 and the download of step i-1 overlap the compute of step
    i.  Each block's time runs from before its first upload to after its last
    download."""
    import torch
    up, down = torch.cuda.Stream(device=stream.device), torch.cuda.Stream(device=stream.device)
    out = []
    for _ in range(n_blocks):
        barrier(world)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        drained = [torch.cuda.Event() for _ in range(2)]
        e0.record(stream)
        up.wait_stream(stream)
        for i in range(steps):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(done[b])            # step i-2 has read set b's inputs
                ins[b].copy_(h_in, non_blocking=True)
                ready[b].record(up)
            stream.wait_event(ready[b])
            if i >= 2:
                stream.wait_event(drained[b])         # step i-2's outputs are back on the host
            with torch.cuda.stream(stream):
                graphs[b].replay()
            done[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(done[b])
                h_out.copy_(outs[b], non_blocking=True)
                drained[b].record(down)
        stream.wait_stream(down)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        out.append(e0.elapsed_time(e1) / steps)
    return out


def measure_model(model: str, args, dev, world: int, rank: int, headline: bool, clocks=None) -> dict:
    """Builds, times and frees one model.  Returns the numbers of one bench line
    (for the headline: with the bracketed launch time and the end-to-end leg)."""
    import torch
    layers = build_layers(model, args, dev, 1000 + 97 * rank)
    io_in, io_out = stage_io(layers, dev)
    torch.cuda.synchronize()
    for L in layers:
        assert L.cache.status_bits() == 0, "prefill flagged a bad page or position"

    step_bytes = sum(L.dec_bytes + L.app_bytes for L in layers)
    kv_bytes = sum(L.dec_bytes for L in layers)
    query_tokens = layers[0].B
    ctx_tokens = sum(int((np.minimum(L.lens, L.window) if L.window else L.lens).sum()) for L in layers)
    stream = torch.cuda.Stream(device=dev)
    flush_buf = None
    if kv_bytes < 2 * l2_bytes(dev):
        flush_buf = torch.empty(2 * l2_bytes(dev) // 4, dtype=torch.float32, device=dev)

    def step():
        for L in layers:
            L.step()

    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    g_a = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_a, stream=stream):
        step()
    launches_per_step = sum(L.launches() for L in layers)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_a.replay()
    torch.cuda.synchronize()

    flush = (lambda: flush_buf.zero_()) if flush_buf is not None else None
    # one calibration block sizes the timed run (the same block count on every rank)
    cal = time_blocks(g_a.replay, args.steps, stream, world, 1, flush)[0]
    n_blocks = int(max_over_ranks(n_blocks_for(cal * args.steps, min_seconds=args.min_seconds), world))
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    blocks = time_blocks(g_a.replay, args.steps, stream, world, n_blocks, flush)
    ms = statistics.median(blocks)
    ms_max = max_over_ranks(ms, world)
    res = {"layers": len(layers), "batch": layers[0].B, "ctx": int(layers[0].lens.max()),
           "kv_bytes_per_step": step_bytes, "ms_per_step": ms_max, "blocks": n_blocks,
           "block_ms_per_step": {"median": round(ms, 5), "min": round(min(blocks), 5),
                                 "max": round(max(blocks), 5)},
           "l2": ("an L2 flush (a write of twice the L2 size) before every timed step: the caches "
                  "together (%.1f MB) are smaller than twice L2" % (kv_bytes / 1e6)) if flush else
                 ("inputs larger than L2: %d layer caches of %.1f MB each are read in turn"
                  % (len(layers), statistics.mean(L.dec_bytes for L in layers) / 1e6)),
           "step_bytes": step_bytes, "query_tokens": query_tokens, "ctx_tokens": ctx_tokens,
           "launches_per_step": launches_per_step,
           "fused": any(L.fused() for L in layers),
           "early_reads": bool(layers[0].cache.cfg.flags & 1),
           "one_kernel": all(L.fused() and L.launches() == 1 for L in layers),
           "call_bytes": statistics.mean(L.dec_bytes + (L.app_bytes if L.fused() else 0) for L in layers),
           "workloads": sorted({L.w["name"] for L in layers})}

    if headline:
        # decode-call durations: a second graph with external event records
        # around every call, one step per replay
        cu = _Cu()
        evs = [(cu.event(), cu.event()) for _ in layers]
        g_b = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_b, stream=stream):
            for L, (e0, e1) in zip(layers, evs):
                if not L.fused():
                    L.append()
                cu.record_external(e0, torch.cuda.current_stream().cuda_stream)
                L.step() if L.fused() else L.decode()
                cu.record_external(e1, torch.cuda.current_stream().cuda_stream)
        dec_ms = []
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                if flush:
                    flush()
                g_b.replay()
                stream.synchronize()
                dec_ms.extend(cu.elapsed_ms(e0, e1) for e0, e1 in evs)
        torch.cuda.synchronize()
        res["bracketed_ms"] = statistics.mean(dec_ms)

        # end to end: every layer's inputs from pinned host memory in one copy, the
        # step (the public call per layer), every layer's outputs back in one copy
        h_in = io_in.cpu().pin_memory()
        h_out = io_out.cpu().pin_memory()

        def e2e_step():
            io_in.copy_(h_in, non_blocking=True)
            g_a.replay()
            h_out.copy_(io_out, non_blocking=True)
            stream.synchronize()

        e2e = time_blocks(e2e_step, args.steps, stream, world, 5, flush)
        res["e2e_serial_ms"] = max_over_ranks(statistics.median(e2e), world)
        res["e2e_ms"] = res["e2e_serial_ms"]
        res["e2e_pipelined"] = False
        res["h2d"] = h_in.numel() * h_in.element_size()
        res["d2h"] = h_out.numel() * h_out.element_size()
        if flush is None:
            # the same steps pipelined over a second set of input and output
            # buffers (and a graph of the step over them)
            io_in2, io_out2 = stage_io(layers, dev)
            g_a2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_a2, stream=stream):
                step()
            with torch.cuda.stream(stream):
                g_a2.replay()
            torch.cuda.synchronize()
            pip = time_pipelined([g_a, g_a2], [io_in, io_in2], [io_out, io_out2], h_in, h_out, stream,
                                 args.steps, world, 5)
            res["e2e_ms"] = max_over_ranks(statistics.median(pip), world)
            res["e2e_pipelined"] = True
            del g_a2, io_in2, io_out2
    if clocks is not None:
        res["clocks"] = clocks.stop()
    for L in layers:
        assert L.cache.status_bits() == 0, "a kernel flagged a bad page, position or length"
    del layers, io_in, io_out, g_a, flush_buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def summarize(r: dict, world: int, peak: float) -> dict:
    """value, fractions and rates of one measured model."""
    ms = r["ms_per_step"]
    launch_ms = ms / r["launches_per_step"] if r["one_kernel"] else r.get("bracketed_ms", float("nan"))
    achieved = r["call_bytes"] / (launch_ms / 1e3) / 1e9
    value = whole_job(r["step_bytes"], world, ms) / 1e9
    return {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "frac": round(achieved / peak, 4), "avg_launch_us": round(launch_ms * 1e3, 3),
        "tokens_per_s": round(whole_job(r["query_tokens"], world, ms), 1),
        "context_tokens_per_s": round(whole_job(r["ctx_tokens"], world, ms), 1),
        "layers": r["layers"], "batch": r["batch"], "ctx": r["ctx"], "kv_bytes_per_step": r["step_bytes"],
        "blocks": r["blocks"], "block_ms_per_step": r["block_ms_per_step"], "l2": r["l2"],
        "early_reads": r.get("early_reads", False),
        "_achieved": achieved, "_launch_ms": launch_ms,
    }


def run_gpu(args) -> dict | None:
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    from int8_quantized_paged_gb300 import build as _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)

    peak, peak_kind = load_peaks()
    clocks = ClockSampler(local)
    head = measure_model(args.workload, args, dev, world, rank, True, clocks)
    hs = summarize(head, world, peak)
    per_config = {}
    if not args.no_per_config:
        for m in PER_CONFIG:
            if m == args.workload:
                continue
            s = summarize(measure_model(m, args, dev, world, rank, False), world, peak)
            s.pop("_achieved")
            s.pop("_launch_ms")
            s["traffic"] = profiled_traffic(m)   # DRAM bytes of one launch, when profiled
            per_config[m] = s
    ms_max = head["ms_per_step"]
    res = {
        "metric": METRIC,
        "value": hs["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4/int8 codes; fp32 softmax and accumulation, fp16 hi/lo tensor-core operands",
        "data": "synthetic: seeded N(0,1) activations of the workload's shapes; no model weights",
        "config": {
            "workload": args.workload,
            "layers": head["layers"],
            "batch": head["batch"],
            "ctx": head["ctx"],
            "kv_bytes_per_step": head["step_bytes"],
            "l2": head["l2"],
            "timing": (f"{head['blocks']} blocks of exactly {args.steps} steps, each bracketed by a barrier and a "
                       f"device synchronize; ms_per_step is the median block"),
            "block_ms_per_step": head["block_ms_per_step"],
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "graph": "CUDA graph of one step",
            "chunk_tokens": args.chunk_tokens or "library default",
            "step_call": ("kvq_append_decode_attention (window layers: kvq_append_window_decode)"
                          if head["fused"] else
                          "kvq_append + kvq_decode_attention (window layers: kvq_window_decode)"),
        },
        "tokens_per_s": hs["tokens_per_s"],
        "context_tokens_per_s": hs["context_tokens_per_s"],
        "pct_of_hbm_peak": hs["pct_of_hbm_peak"],
        "pct_of_nominal_hbm": hs["pct_of_nominal_hbm"],
        "roofline": {
            "bound": "hbm",
            "kernel": ("decode_tc_kernel (kvq_append_decode_attention: the step's append, split-K decode "
                       "and the LSE combine in one launch)" if head["fused"] else
                       "decode_tc_kernel (kvq_decode_attention: split-K decode with the LSE combine fused)"),
            "achieved": round(hs["_achieved"], 1),
            "peak": peak,
            "peak_source": f"{peak_kind} hbm_gbs",
            "unit": "GB/s",
            "frac": round(hs["_achieved"] / peak, 4),
            "traffic": profiled_traffic(args.workload),
            "algorithmic_bytes_per_launch": int(head["call_bytes"]),
            "avg_launch_us": round(hs["_launch_ms"] * 1e3, 3),
            "launch_us_from": ("timed region / launches (the step is only this kernel)" if head["one_kernel"]
                               else "CUDA events around each call in a graph of the step"),
            "bracketed_launch_us": round(head["bracketed_ms"] * 1e3, 3),
        },
        "e2e": {
            "value": round(whole_job(head["step_bytes"], world, head["e2e_ms"]) / 1e9, 2),
            "unit": "GB/s",
            "ms_per_step": round(head["e2e_ms"], 5),
            "h2d_bytes_per_step": head["h2d"],
            "d2h_bytes_per_step": head["d2h"],
            "method": ("pipelined over two buffer sets: step i+1's inputs copied up and step i-1's "
                       "outputs copied down while step i computes; every copy inside the timed region"
                       if head["e2e_pipelined"] else
                       "serial: upload, step, download and a host synchronize every step"),
            "serial": {"value": round(whole_job(head["step_bytes"], world, head["e2e_serial_ms"]) / 1e9, 2),
                       "ms_per_step": round(head["e2e_serial_ms"], 5)},
        },
        "gpu_launches": head["launches_per_step"] * args.steps * head["blocks"],
        "clocks": head["clocks"],
        "per_config": per_config,
    }
    return res if rank == 0 else None


# ----------------------------------------------------------------------------- CPU oracle


def oracle_sample(workload: str):
    """One bounded unit of the workload for the CPU oracle: the first layer of the
    model with its cache filled by the oracle's own append (set-up, untimed).  For
    the continuous batch the sample is its first 4 sequences."""
    from oracle import kvq_oracle as O
    name, _, window = MODELS[workload][0]
    w = wl.workload(name)
    lens = wl.seq_lens(w)
    if workload == "contbatch":
        lens = lens[:4]
    spec = O.Spec.from_workload(w)
    ring = int(w["ring_rows"]) if window else 0
    win = int(w["window"]) if window else 0
    P = 16
    maxp = ring // P if ring else int(math.ceil(lens.max() / P))
    bt = np.arange(len(lens) * maxp, dtype=np.int32).reshape(len(lens), maxp)
    pools = {"k": np.zeros(bt.size * O.page_bytes(spec, "k"), np.uint8),
             "v": np.zeros(bt.size * O.page_bytes(spec, "v"), np.uint8)}
    tab = O.rope_table(spec.head_dim, spec.rope_base, int(lens.max()) + 1)
    for b, L in enumerate(lens):
        k, v = wl.kv_rows(w, b, "k", int(L)), wl.kv_rows(w, b, "v", int(L))
        O.append(spec, pools, k, v, np.full(int(L), b), np.arange(int(L)), bt, ring, tab)
    q = wl.queries(dict(w, batch=len(lens)))
    knew = wl.new_rows(w, "k", len(lens))
    vnew = wl.new_rows(w, "v", len(lens))
    dec, app = algorithmic_bytes(w, lens, win)

    def step():
        O.append(spec, pools, knew, vnew, np.arange(len(lens)), lens - 1, bt, ring, tab)
        O.decode(spec, q, pools, bt, lens, win, ring)

    desc = (f"oracle append + decode of 1 {name} layer ({len(lens)} seq, "
            f"{int((np.minimum(lens, win) if win else lens).sum())} attended tokens), "
            f"cache filled by the oracle untimed")
    return step, dec + app, desc


ORACLE_KIND = "oracle (numpy, 1 thread, OPENBLAS_NUM_THREADS=1)"


def cpu_worker(workload: str, seconds: float, steps: int, warmup: int) -> dict:
    step, nbytes, desc = oracle_sample(workload)
    for _ in range(warmup):
        step()
    times = []
    t_end = time.perf_counter() + seconds
    while (steps and len(times) < steps) or (not steps and (time.perf_counter() < t_end or not times)):
        t = time.perf_counter()
        step()
        times.append(time.perf_counter() - t)
    mean = sum(times) / len(times)
    return {"value": round(nbytes / mean / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": ORACLE_KIND,
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "sample": f"{desc}; {len(times)} timed calls, {mean * 1e3:.1f} ms each",
            "ms_per_step": mean * 1e3}


def run_cpu_worker_subprocess(workload: str, seconds: float, steps: int = 0, warmup: int = 1) -> dict:
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "NUMEXPR_NUM_THREADS"):
        env[k] = "1"
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-worker", "--workload", workload,
           "--cpu-seconds", str(seconds), "--steps", str(steps), "--warmup", str(warmup)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
    if r.returncode != 0:
        raise RuntimeError(f"cpu worker failed:\n{r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    r = run_cpu_worker_subprocess(args.workload, 0.0, steps=args.steps, warmup=args.warmup)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": r["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(r["ms_per_step"], 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (codes in fp32)",
        "data": "synthetic: seeded N(0,1) activations of the workload's shapes; no model weights",
        "config": {"workload": args.workload, "sample": r["sample"]},
        "cpu_baseline": {"value": r["value"], "unit": "GB/s", "cores": r["cores"], "kind": r["kind"],
                         "cpu_model": r["cpu_model"], "host_cpus": r["host_cpus"], "sample": r["sample"]},
        "e2e": {"value": r["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--workload", choices=list(MODELS), default="contbatch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="timed work per configuration, at least (whole blocks, at least 5)")
    ap.add_argument("--chunk-tokens", type=int, default=0,
                    help="tokens per split-K chunk (0: the library chooses)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile-decode", type=int, default=0, metavar="CALLS",
                    help="only run CALLS decode calls per layer (for profiler captures)")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling)")
    ap.add_argument("--no-early-reads", action="store_true",
                    help="multi-layer models: read every input after the previous kernel ends")
    ap.add_argument("--separate", action="store_true",
                    help="time kvq_append + kvq_decode_attention instead of the fused call")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker:
        print(json.dumps(cpu_worker(args.workload, args.cpu_seconds, args.steps, args.warmup)))
        return
    rank, world, _ = dist_env()
    err = check_gpus_flag(args.gpus, world)
    if err:
        print(f"bench.py: {err}", file=sys.stderr)
        sys.exit(2)
    if args.profile_decode:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")

    res = run_gpu(args)
    if res is not None:
        if world == 1 and not args.no_cpu_baseline:
            cb = run_cpu_worker_subprocess(args.workload, args.cpu_seconds)
            cb.pop("ms_per_step", None)
            res["cpu_baseline"] = cb
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
