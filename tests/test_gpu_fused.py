"""The fused decode step, kvq_append_decode_attention, on the GPU.

Against the oracle's append of the step's rows followed by its decode: pools
bytewise equal, outputs within 2e-3 row-relative error.  Against the library's
own separate calls: the output equals, bit for bit, a plain decode of the
pools the fused call left behind (the row the fused call used from shared
memory is the row it wrote), and re-appending the same rows with kvq_append
leaves the pools unchanged.  Positions cover the first row of a page, the last
row of a page, mid-page rows, a row past the attended length and bad input.
"""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, floor_for, max_row_err, oracle_rope
from int8_quantized_paged_gb300 import kvq
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.init()


# lens: the prefilled rows; the step rewrites row L - 1 of every sequence
CASES = {
    "tiny": dict(lens=[256]),
    "llama8b": dict(lens=[1000, 33, 2049], over=dict(batch=3)),
    "llama8b_8k": dict(name="llama8b", lens=[8192]),
    "contbatch": dict(lens=[1, 16, 17, 700, 2900], over=dict(batch=5)),
    "gemma_mix": dict(lens=[3001, 5], over=dict(batch=2)),
    "long_mixed": dict(lens=[5000, 777], over=dict(batch=2)),
    "llama8b_f16": dict(lens=[1000, 33, 2049], over=dict(batch=3)),
    "long_f16": dict(lens=[3000, 77], over=dict(batch=2)),
    "llama8b_shimmy": dict(lens=[1000, 33, 2049], over=dict(batch=3)),
    "long_shimmy": dict(lens=[3000, 77], over=dict(batch=2)),
}


def _case(key):
    spec = CASES[key]
    w = wl.workload(spec.get("name", key), **spec.get("over", {}))
    return Case(w, spec["lens"])


def _step(c: Case, pos, seq_lens, chunk: int, step: int = 1):
    """Runs the fused call with new rows at `pos`; returns (out, k_new, v_new)."""
    dev = c.cache.device
    k_new = wl.new_rows(c.w, "k", c.B, step=step)
    v_new = wl.new_rows(c.w, "v", c.B, step=step)
    q = c.queries(step=step)
    qt = torch.from_numpy(q).to(dev)
    out = torch.full_like(qt, float("nan"))
    ws = c.cache.workspace(c.B, chunk)
    c.cache.append_decode(qt, torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                          torch.as_tensor(np.asarray(pos, np.int32), device=dev),
                          torch.as_tensor(np.asarray(seq_lens, np.int32), device=dev), out, ws, chunk)
    torch.cuda.synchronize()
    return q, out.float().cpu().numpy().astype(np.float64), k_new, v_new


def _oracle_append(c: Case, k_new, v_new, pos):
    s = c.spec
    tab = oracle_rope(s.head_dim, s.rope_base, c.rope_max)
    keep = [b for b in range(c.B) if pos[b] >= 0]
    O.append(s, c.pools, k_new[keep], v_new[keep], np.asarray(keep), np.asarray(pos)[keep], c.bt, 0, tab)


@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("key", list(CASES))
def test_fused_step_matches_oracle_and_separate_calls(key, chunk):
    c = _case(key)
    pos = c.lens - 1
    q, got, k_new, v_new = _step(c, pos, c.lens, chunk)
    assert c.cache.status_bits() == 0
    _oracle_append(c, k_new, v_new, pos)
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"])
    assert np.array_equal(v, c.pools["v"])
    assert max_row_err(got, c.oracle_decode(q), floor=floor_for(c.w)) <= TOL
    # the plain decode over the pools the fused call wrote gives the same bits
    assert np.array_equal(got, c.gpu_decode(q, chunk_tokens=chunk))
    # the separate append of the same rows rewrites the same bytes
    dev = c.cache.device
    c.cache.append(torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                   torch.as_tensor(pos.astype(np.int32), device=dev))
    torch.cuda.synchronize()
    k2, v2 = c.gpu_pools()
    assert np.array_equal(k2, k) and np.array_equal(v2, v)


def test_fused_step_uses_the_cluster_mode_for_a_short_batch():
    c = _case("llama8b_8k")
    assert kvq.decode_cluster_ctas(c.cfg, c.B, c.max_pages) > 0
    assert kvq.decode_cluster_ctas(c.cfg, c.B, c.max_pages, chunk_tokens=64) == 0
    assert kvq.append_decode_launches(c.cfg) == 1


def test_row_past_the_attended_length_is_written_not_attended():
    w = wl.workload("llama8b", batch=2)
    c = Case(w, [49, 40])
    # sequence 0: row 48 (page 3) with only 37 keys attended -> written by the
    # prologue path; sequence 1: row 39, 38 attended -> written, masked
    pos = np.array([48, 39])
    lens = np.array([37, 38])
    q, got, k_new, v_new = _step(c, pos, lens, 0)
    assert c.cache.status_bits() == 0
    _oracle_append(c, k_new, v_new, pos)
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    ref = O.decode(c.spec, q, c.pools, c.bt, lens)
    assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL


def test_bad_position_flags_and_skips_the_row():
    w = wl.workload("llama8b", batch=2)
    c = Case(w, [100, 30])
    before_k, before_v = c.gpu_pools()
    q, got, _, _ = _step(c, np.array([-1, 10 ** 6]), c.lens, 0)
    assert c.cache.status_bits() == kvq.DEV_BAD_POS
    k, v = c.gpu_pools()
    assert np.array_equal(k, before_k) and np.array_equal(v, before_v)
    assert max_row_err(got, c.oracle_decode(q), floor=floor_for(c.w)) <= TOL   # the decode itself is unaffected


def test_fused_argument_checks():
    w = wl.workload("llama8b", batch=1)
    c = Case(w, [64], fill_oracle=False)
    dev = c.cache.device
    q = torch.zeros((1, w["n_heads"], w["head_dim"]), dtype=torch.float16, device=dev)
    rows = torch.zeros((2 * w["n_kv_heads"] * w["head_dim"] + 8,), dtype=torch.float16, device=dev)
    k_bad = rows[1:1 + w["n_kv_heads"] * w["head_dim"]].view(1, w["n_kv_heads"], w["head_dim"])
    pos = torch.tensor([63], dtype=torch.int32, device=dev)
    lens = torch.tensor([64], dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    ws = c.cache.workspace(1)
    with pytest.raises(kvq.KvqError):
        c.cache.append_decode(q, k_bad, k_bad, pos, lens, out, ws)
    with pytest.raises(kvq.KvqError):
        kvq.append_decode_attention(c.cfg, q, k_bad, k_bad, None, c.cache.k_pool, c.cache.v_pool,
                                    c.n_pages, c.cache.block_table, c.max_pages, lens, c.cache.rope_tab,
                                    c.rope_max, out, ws, c.cache.status)


def _window_step(c: Case, window: int, chunk: int, step: int = 1):
    dev = c.cache.device
    k_new = wl.new_rows(c.w, "k", c.B, step=step)
    v_new = wl.new_rows(c.w, "v", c.B, step=step)
    q = c.queries(step=step)
    qt = torch.from_numpy(q).to(dev)
    out = torch.full_like(qt, float("nan"))
    ws = c.cache.workspace(c.B, chunk, window)
    pos = (c.lens - 1).astype(np.int32)
    c.cache.append_window_decode(qt, torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                                 torch.from_numpy(pos).to(dev), torch.from_numpy(c.lens).to(dev), out, ws,
                                 window, chunk)
    torch.cuda.synchronize()
    return q, out.float().cpu().numpy().astype(np.float64), k_new, v_new, pos


@pytest.mark.parametrize("name", ["gemma_mix", "llama8b_f16"])
@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("L", [5, 1024, 1153, 3000])
def test_fused_window_step_matches_oracle(L, chunk, name):
    """Ring of 1152 rows, window 1024: the new row overwrites ring row (L-1) mod 1152."""
    w = wl.workload(name, batch=1)
    c = Case(w, [L], ring_rows=1152)
    q, got, k_new, v_new, pos = _window_step(c, 1024, chunk)
    assert c.cache.status_bits() == 0
    s = c.spec
    O.append(s, c.pools, k_new, v_new, np.array([0]), pos, c.bt, 1152, oracle_rope(s.head_dim, s.rope_base,
                                                                                      c.rope_max))
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    assert max_row_err(got, c.oracle_decode(q, window=1024), floor=floor_for(c.w)) <= TOL
    assert np.array_equal(got, c.gpu_decode(q, chunk_tokens=chunk, window=1024))


def test_window_uses_the_cluster_mode():
    w = wl.workload("gemma_mix", batch=1)
    cfg = kvq.config(**w)
    assert kvq.decode_cluster_ctas(cfg, 1, 1152 // 16, window=1024) > 0
