"""kvq_decode_attention_noalloc against kvq_decode_attention.

The no-allocation entry point is for callers that cannot allocate device
memory themselves.  Examples are a plugin running inside an engine that owns
all of HBM through its own pool, and a latency-critical path where an
allocation and the synchronization it may bring are not allowed.  Its split-K
workspace is a fixed array inside the library, so the caller passes only
inputs and outputs.  These tests call it through the C ABI twice in a row,
with different queries and lengths, and check each result against the entry
point that takes a caller workspace.  The second call shows that the shared
scratch left by the first call does not leak into the next result.  An
oversized request must be refused before any launch.
"""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case
from int8_quantized_paged_gb300 import kvq
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _both(c: Case, q: np.ndarray, lens, chunk: int = 0):
    dev = c.cache.device
    qt = torch.from_numpy(q).to(dev)
    lt = torch.from_numpy(np.asarray(lens, np.int32)).to(dev)
    ref = torch.full_like(qt, float("nan"))
    got = torch.full_like(qt, float("nan"))
    ws = c.cache.workspace(c.B, chunk)
    c.cache.decode(qt, lt, ref, ws, chunk)
    kvq.decode_attention_noalloc(c.cfg, qt, c.cache.k_pool, c.cache.v_pool, c.n_pages, c.cache.block_table,
                                 c.max_pages, lt, c.cache.rope_tab, c.rope_max, got, c.cache.status, chunk)
    torch.cuda.synchronize()
    return got.double().cpu().numpy(), ref.double().cpu().numpy()


def test_noalloc_matches_workspace_entry_twice():
    w = wl.workload("llama8b", batch=3)
    c = Case(w, [1000, 37, 2049], fill_oracle=False)
    for step, lens, chunk in ((0, [1000, 37, 2049], 0), (1, [999, 5, 1500], 64)):
        got, ref = _both(c, c.queries(step=step), lens, chunk)
        assert np.all(np.isfinite(got))
        assert float(np.max(O.row_rel_error(got, ref))) <= TOL, step
    assert c.cache.status_bits() == 0


def test_noalloc_other_codec():
    w = wl.workload("long_mixed", batch=2)
    c = Case(w, [3000, 333], fill_oracle=False)
    for step in (0, 1):
        got, ref = _both(c, c.queries(step=step), [3000 - 7 * step, 333])
        assert float(np.max(O.row_rel_error(got, ref))) <= TOL


def test_noalloc_rejects_oversized_workspace():
    w = wl.workload("llama8b", batch=64)
    cfg = kvq.config(**w)
    max_pages = 4096
    need = kvq.decode_workspace_bytes(cfg, 64, max_pages, 16)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    q = torch.zeros(64, 32, 128, dtype=torch.float16, device=dev)
    out = torch.full_like(q, 3.0)
    dummy = torch.zeros(64, dtype=torch.int32, device=dev)
    pool = torch.zeros(16, dtype=torch.uint8, device=dev)
    rope = torch.zeros(2, 64, 2, dtype=torch.float32, device=dev)
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention_noalloc(cfg, q, pool, pool, 1, dummy, max_pages, dummy, rope, 2, out, dummy, 16)
    assert e.value.status == kvq.ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
