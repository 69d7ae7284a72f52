"""KVQ_FLAG_EARLY_READS on the GPU: layers whose inputs come from the call before.

A model of four layers runs two decode steps as one stream of fused calls,
launched back to back with no synchronisation, so each call can start while the
call before it still runs.  Layer i's query (and, at batch 1, its new K and V
rows) is a slice of layer i-1's output, written by the very kernel launched
before it: a call that read those inputs before its dependency wait would see
the NaNs the outputs start as, or the previous step's values.  The oracle runs
the same chain from the outputs the GPU produced: the appended pages are
bytewise equal and every output is within 2e-3 row-relative error.  The
decode-only calls are chained the same way, the whole-context ones through the
no-alloc entry point, whose calls all share the library's one scratch
workspace.
"""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, floor_for, max_row_err, oracle_rope
from int8_quantized_paged_gb300 import kvq
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu

N_LAYERS, N_STEPS = 4, 2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.init()


# lens: the prefilled rows (each row L, L + 1 the steps write lies in a mapped
# page); chain_kv: the new K and V rows are slices of the previous output too
# (batch 1, where those slices are contiguous)
CASES = {
    "llama8b_b1": dict(name="llama8b", lens=[8200], chain_kv=True),
    "llama8b_b3": dict(name="llama8b", lens=[1000, 33, 2049], over=dict(batch=3), chain_kv=False),
    "long_mixed": dict(name="long_mixed", lens=[5000, 777], over=dict(batch=2), chain_kv=False),
    "gemma_window": dict(name="gemma_mix", lens=[3001], ring=1152, window=1024, chain_kv=True),
    # head_dim 256, whole context, affine K: four warps of each cluster CTA
    # build the query fragments and per-unit q sums after their waits
    "gemma_global": dict(name="gemma_mix", lens=[3001], chain_kv=True),
}


@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("key", list(CASES))
def test_chained_layers_with_early_reads_match_oracle(key, chunk):
    spec = CASES[key]
    w = wl.workload(spec["name"], **spec.get("over", {}))
    ring, window = spec.get("ring", 0), spec.get("window", 0)
    layers = [Case(w, spec["lens"], ring_rows=ring, extra_positions=N_STEPS) for _ in range(N_LAYERS)]
    for c in layers:
        c.cfg.flags = kvq.FLAG_EARLY_READS   # the cache's own config object
    c0 = layers[0]
    dev, B, hkv = c0.cache.device, c0.B, w["n_kv_heads"]
    assert spec["chain_kv"] == (B == 1)
    act = c0.cache.act_dtype

    # every input and output allocated and filled before the first call
    lens0 = c0.lens.astype(np.int64)
    steps = []
    for s in range(N_STEPS):
        pos = (lens0 + s).astype(np.int32)
        st = dict(pos=torch.from_numpy(pos).to(dev),
                  lens=torch.from_numpy(pos + 1).to(dev),
                  q0=torch.from_numpy(wl.queries(dict(w, batch=B), step=10 + s)).to(dev),
                  k0=torch.from_numpy(wl.new_rows(w, "k", B, step=10 + s)).to(dev),
                  v0=torch.from_numpy(wl.new_rows(w, "v", B, step=10 + s)).to(dev),
                  outs=[torch.full((B, w["n_heads"], w["head_dim"]), float("nan"), dtype=act, device=dev)
                        for _ in range(N_LAYERS)],
                  ws=[c.cache.workspace(B, chunk, window) for c in layers])
        steps.append(st)
    torch.cuda.synchronize()

    def inputs(st, i):
        if i == 0:
            return st["q0"], st["k0"], st["v0"]
        prev = st["outs"][i - 1]
        if spec["chain_kv"]:
            return prev, prev[:, :hkv], prev[:, hkv:2 * hkv]
        return prev, st["k0"], st["v0"]

    for st in steps:
        for i, c in enumerate(layers):
            q, k_new, v_new = inputs(st, i)
            if window:
                c.cache.append_window_decode(q, k_new, v_new, st["pos"], st["lens"], st["outs"][i], st["ws"][i],
                                             window, chunk)
            else:
                c.cache.append_decode(q, k_new, v_new, st["pos"], st["lens"], st["outs"][i], st["ws"][i], chunk)
    torch.cuda.synchronize()
    assert all(c.cache.status_bits() == 0 for c in layers)

    # the oracle, step by step and layer by layer, from the GPU's own outputs
    s_ = c0.spec
    tab = oracle_rope(s_.head_dim, s_.rope_base, c0.rope_max)
    host = lambda t: t.cpu().numpy()
    for s, st in enumerate(steps):
        pos = (lens0 + s).astype(np.int64)
        for i, c in enumerate(layers):
            q, k_new, v_new = (host(t) for t in inputs(st, i))
            assert np.isfinite(q.astype(np.float64)).all()
            O.append(s_, c.pools, np.ascontiguousarray(k_new), np.ascontiguousarray(v_new), np.arange(B), pos,
                     c.bt, ring, tab)
            ref = O.decode(s_, q, c.pools, c.bt, pos + 1, window, ring, seqs=list(range(B)))
            got = host(st["outs"][i]).astype(np.float64)
            assert max_row_err(got, ref, floor=floor_for(w)) <= TOL, (s, i)
    for c in layers:
        k, v = c.gpu_pools()
        assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])



DECODE_CASES = {
    # whole context through the no-alloc entry point: every layer's call
    # shares the library's one scratch workspace with the call before it
    "llama8b_noalloc": dict(name="llama8b", lens=[1000, 33, 2049], over=dict(batch=3)),
    "gemma_window": dict(name="gemma_mix", lens=[3001, 700], over=dict(batch=2), ring=1152, window=1024),
    "gemma_global": dict(name="gemma_mix", lens=[3001, 700], over=dict(batch=2)),
}


@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("key", list(DECODE_CASES))
def test_chained_decode_calls_with_early_reads_match_oracle(key, chunk):
    """The decode-only calls: layer i's query is layer i-1's output."""
    spec = DECODE_CASES[key]
    w = wl.workload(spec["name"], **spec.get("over", {}))
    ring, window = spec.get("ring", 0), spec.get("window", 0)
    layers = [Case(w, spec["lens"], ring_rows=ring) for _ in range(N_LAYERS)]
    for c in layers:
        c.cfg.flags = kvq.FLAG_EARLY_READS
    c0 = layers[0]
    dev, B = c0.cache.device, c0.B
    lens = torch.from_numpy(c0.lens).to(dev)
    passes = []
    for p in range(N_STEPS):
        passes.append(dict(q0=torch.from_numpy(wl.queries(dict(w, batch=B), step=20 + p)).to(dev),
                           outs=[torch.full((B, w["n_heads"], w["head_dim"]), float("nan"), dtype=c0.cache.act_dtype,
                                            device=dev) for _ in range(N_LAYERS)],
                           ws=[c.cache.workspace(B, chunk, window) for c in layers]))
    torch.cuda.synchronize()
    for ps in passes:
        for i, c in enumerate(layers):
            q = ps["q0"] if i == 0 else ps["outs"][i - 1]
            if window:
                c.cache.window_decode(q, lens, ps["outs"][i], ps["ws"][i], window, chunk)
            else:
                kvq.decode_attention_noalloc(c.cfg, q, c.cache.k_pool, c.cache.v_pool, c.n_pages,
                                             c.cache.block_table, c.max_pages, lens, c.cache.rope_tab,
                                             c.rope_max, ps["outs"][i], c.cache.status, chunk)
    torch.cuda.synchronize()
    assert all(c.cache.status_bits() == 0 for c in layers)
    for ps in passes:
        for i, c in enumerate(layers):
            q = (ps["q0"] if i == 0 else ps["outs"][i - 1]).cpu().numpy()
            assert np.isfinite(q.astype(np.float64)).all()
            ref = O.decode(c.spec, q, c.pools, c.bt, c.lens, window, ring, seqs=list(range(B)))
            got = ps["outs"][i].cpu().numpy().astype(np.float64)
            assert max_row_err(got, ref, floor=floor_for(w)) <= TOL, i
