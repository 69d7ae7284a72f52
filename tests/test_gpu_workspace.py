"""The workspace mode at batches the cluster mode cannot hold, against the oracle.

Split-K chunks of every (sequence, kv head) go through the workspace and the
last chunk to finish combines them.  The cases: many mixed lengths with empty
sequences and page edges; a bad length; the fused append; a sliding window
over ring pages at batch 80; single-block sequences; one 64K-token sequence
split into many chunks a stream.  Pools bytewise equal to the oracle's,
outputs within 2e-3 row-relative error.
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


def _lens(n, lo, hi, seed, edges=()):
    r = np.random.default_rng(seed)
    L = r.integers(lo, hi, size=n, endpoint=True).astype(np.int32)
    L[:len(edges)] = edges
    return L


def _workspace_mode(c: Case, window: int = 0):
    assert kvq.decode_cluster_ctas(c.cfg, c.B, c.max_pages, window=window) == 0


def test_mixed_lengths_and_empty_sequences():
    lens = _lens(48, 1, 3000, 11, edges=(0, 1, 15, 16, 17, 0, 2900))
    c = Case(wl.workload("contbatch", batch=48), lens)
    _workspace_mode(c)
    q = c.queries()
    got = c.gpu_decode(q)
    assert c.cache.status_bits() == 0
    ref = c.oracle_decode(q)
    assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL
    assert np.all(got[lens == 0] == 0)
    # a length past the table's capacity: a zero row and the flag, the rest unchanged
    bad = lens.copy()
    bad[3] = 10 ** 6
    got2 = c.gpu_decode(q, lens=bad)
    assert c.cache.status_bits() & kvq.DEV_BAD_LEN
    assert np.all(got2[3] == 0)
    keep = [b for b in range(c.B) if b != 3]
    assert max_row_err(got2, ref, seqs=keep, floor=floor_for(c.w)) <= TOL


def test_fused_append_decode():
    lens = _lens(40, 1, 3000, 12, edges=(1, 16, 17, 32))
    c = Case(wl.workload("contbatch", batch=40), lens)
    _workspace_mode(c)
    dev = c.cache.device
    pos = (lens - 1).astype(np.int32)
    k_new, v_new = wl.new_rows(c.w, "k", c.B, step=3), wl.new_rows(c.w, "v", c.B, step=3)
    q = c.queries(step=3)
    qt = torch.from_numpy(q).to(dev)
    out = torch.full_like(qt, float("nan"))
    ws = c.cache.workspace(c.B)
    c.cache.append_decode(qt, torch.from_numpy(k_new).to(dev), torch.from_numpy(v_new).to(dev),
                          torch.from_numpy(pos).to(dev), torch.from_numpy(lens).to(dev), out, ws)
    torch.cuda.synchronize()
    assert c.cache.status_bits() == 0
    s = c.spec
    O.append(s, c.pools, k_new, v_new, np.arange(c.B), pos, c.bt, 0, oracle_rope(s.head_dim, s.rope_base, c.rope_max))
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    got = out.double().cpu().numpy()
    assert max_row_err(got, c.oracle_decode(q), floor=floor_for(c.w)) <= TOL
    assert np.array_equal(got, c.gpu_decode(q))   # the decode of the pools it wrote, bit for bit


def test_sliding_window_over_ring_pages():
    lens = _lens(80, 1, 1500, 13, edges=(1, 1024, 1025, 1152, 1153))
    c = Case(wl.workload("gemma_mix", batch=80), lens, ring_rows=1152)
    _workspace_mode(c, window=1024)
    q = c.queries()
    got = c.gpu_decode(q, window=1024)
    assert c.cache.status_bits() == 0
    assert max_row_err(got, c.oracle_decode(q, window=1024), floor=floor_for(c.w)) <= TOL


def test_single_block_sequences():
    lens = _lens(80, 1, 16, 14)
    c = Case(wl.workload("contbatch", batch=80), lens)
    _workspace_mode(c)
    q = c.queries()
    got = c.gpu_decode(q)
    assert c.cache.status_bits() == 0
    assert max_row_err(got, c.oracle_decode(q), floor=floor_for(c.w)) <= TOL


def test_one_long_sequence_in_many_chunks():
    # fp32 activations: at 64K tokens the outputs are ~1/256 and an fp16
    # output's own rounding near the 0.1 % row floor is already ~2e-3 of it
    c = Case(wl.workload("llama8b", act="f32"), [65536])
    _workspace_mode(c)
    q = c.queries()
    got = c.gpu_decode(q)
    assert c.cache.status_bits() == 0
    assert max_row_err(got, c.oracle_decode(q), floor=floor_for(c.w)) <= TOL
