"""The five workloads at their full sizes, in the launch configuration the
bench times (library-chosen chunks), checked on sequences the oracle can
compute one by one: their pages bytewise and their outputs at 2e-3."""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, max_row_err, pages_of, pool_slice
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _check(c: Case, window: int = 0):
    kp, vp = c.gpu_pools()
    for b in c.oracle_seqs:
        pg = pages_of(c, b)
        for which, gpu in (("k", kp), ("v", vp)):
            pb = O.page_bytes(c.spec, which)
            assert np.array_equal(pool_slice(gpu, pb, pg), pool_slice(c.pools[which], pb, pg)), (b, which)
    q = c.queries()
    got = c.gpu_decode(q, window=window)
    assert np.all(np.isfinite(got))
    ref = c.oracle_decode(q, window=window)
    assert max_row_err(got, ref, seqs=c.oracle_seqs) <= TOL
    assert c.cache.status_bits() == 0
    return got


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
