"""The bench workloads at their full sizes, in the launch configuration the
bench times (library-chosen chunks), checked on sequences the oracle can
compute one by one: their pages bytewise and their outputs at 2e-3.  Each
case runs the plain decode of the filled cache, then the bench's step, the
fused call that writes a new token's K/V at row L - 1 and attends over it."""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, floor_for, max_row_err, oracle_rope, pages_of, pool_slice
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _pages_equal(c: Case):
    kp, vp = c.gpu_pools()
    for b in c.oracle_seqs:
        pg = pages_of(c, b)
        for which, gpu in (("k", kp), ("v", vp)):
            pb = O.page_bytes(c.spec, which)
            assert np.array_equal(pool_slice(gpu, pb, pg), pool_slice(c.pools[which], pb, pg)), (b, which)


def _fused_step(c: Case, window: int = 0):
    """The bench's step: new K/V rows at L - 1 (a ring row for a window), written
    and attended by one kvq_append_decode_attention / kvq_append_window_decode."""
    dev = c.cache.device
    k_new = wl.new_rows(c.w, "k", c.B, step=1)
    v_new = wl.new_rows(c.w, "v", c.B, step=1)
    q = c.queries(step=1)
    pos = (c.lens - 1).astype(np.int32)
    qt = torch.from_numpy(q).to(dev)
    out = torch.full_like(qt, float("nan"))
    ws = c.cache.workspace(c.B, 0, window)
    args = (qt, torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev), torch.from_numpy(pos).to(dev),
            torch.from_numpy(c.lens).to(dev), out, ws)
    if window:
        c.cache.append_window_decode(*args, window, 0)
    else:
        c.cache.append_decode(*args, 0)
    torch.cuda.synchronize()
    got = out.float().cpu().numpy().astype(np.float64)
    seqs = np.asarray(c.oracle_seqs)
    s = c.spec
    O.append(s, c.pools, k_new[seqs], v_new[seqs], seqs, pos[seqs], c.bt, c.ring_rows,
             oracle_rope(s.head_dim, s.rope_base, c.rope_max))
    _pages_equal(c)
    assert np.all(np.isfinite(got[seqs]))
    assert max_row_err(got, c.oracle_decode(q, window=window), seqs=c.oracle_seqs, floor=floor_for(c.w)) <= TOL
    assert c.cache.status_bits() == 0


def _check(c: Case, window: int = 0):
    _pages_equal(c)
    q = c.queries()
    got = c.gpu_decode(q, window=window)
    assert np.all(np.isfinite(got))
    ref = c.oracle_decode(q, window=window)
    assert max_row_err(got, ref, seqs=c.oracle_seqs, floor=floor_for(c.w)) <= TOL
    assert c.cache.status_bits() == 0
    _fused_step(c, window)


def test_llama8b_full():
    w = wl.workload("llama8b")
    _check(Case(w, wl.seq_lens(w), shuffle=False))


def test_contbatch_full_sampled():
    w = wl.workload("contbatch")
    lens = wl.seq_lens(w)
    pick = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 17})
    _check(Case(w, lens, oracle_seqs=pick))


def test_gemma_global_full():
    w = wl.workload("gemma_mix")
    _check(Case(w, [w["ctx"]], shuffle=False))


def test_gemma_window_full():
    w = wl.workload("gemma_mix")
    _check(Case(w, [w["ctx"]], ring_rows=w["ring_rows"]), window=w["window"])


def test_long_mixed_full_sampled():
    w = wl.workload("long_mixed")
    _check(Case(w, wl.seq_lens(w), oracle_seqs=[2]))


@pytest.mark.parametrize("name", ["llama8b_f16", "llama8b_shimmy"])
def test_llama8b_kinds_full(name):
    w = wl.workload(name)
    _check(Case(w, wl.seq_lens(w), shuffle=False))


@pytest.mark.parametrize("name", ["long_f16", "long_shimmy"])
def test_long_kinds_full_sampled(name):
    w = wl.workload(name)
    _check(Case(w, wl.seq_lens(w), oracle_seqs=[1]))
