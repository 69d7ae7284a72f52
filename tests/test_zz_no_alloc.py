"""kvq_decode_attention_noalloc against kvq_decode_attention and the oracle.

The no-allocation entry point is for callers that cannot allocate device
memory themselves.  Examples are a plugin running inside an engine that owns
all of HBM through its own pool, and a latency-critical path where an
allocation and the synchronization it may bring are not allowed.  Its split-K
workspace is a fixed array inside the library, so the caller passes only
inputs and outputs.

These tests call it through the C ABI several times in a row.  With
chunk_tokens = 64 every call takes the workspace mode, whose last-arriving CTA
of each (sequence, kv head) combines the partials through arrival counters in
that shared array; two such calls back to back, then a third with another
batch, show that what one call leaves in the array does not reach the next
result.  Each result must equal, bit for bit, the entry point that takes a
caller workspace (the same kernel on the same inputs), and match the oracle
within the parity tolerance.  An oversized request must be refused before
any launch.
"""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, floor_for, max_row_err
from int8_quantized_paged_gb300 import kvq
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _both(c: Case, q: np.ndarray, lens, chunk: int = 0, batch: int = 0):
    """(no-alloc output, workspace-entry output) for the first `batch`
    sequences (all when 0)."""
    dev = c.cache.device
    B = batch or c.B
    qt = torch.from_numpy(np.ascontiguousarray(q[:B])).to(dev)
    lt = torch.from_numpy(np.asarray(lens, np.int32)[:B]).to(dev)
    table = c.cache.block_table[:B]          # rows 0 .. B-1: a contiguous prefix of the table
    ref = torch.full_like(qt, float("nan"))
    got = torch.full_like(qt, float("nan"))
    ws = torch.zeros(kvq.decode_workspace_bytes(c.cfg, B, c.max_pages, chunk), dtype=torch.uint8, device=dev)
    kvq.decode_attention(c.cfg, qt, c.cache.k_pool, c.cache.v_pool, c.n_pages, table, c.max_pages, lt,
                         c.cache.rope_tab, c.rope_max, ref, ws, c.cache.status, chunk)
    kvq.decode_attention_noalloc(c.cfg, qt, c.cache.k_pool, c.cache.v_pool, c.n_pages, table, c.max_pages, lt,
                                 c.cache.rope_tab, c.rope_max, got, c.cache.status, chunk)
    torch.cuda.synchronize()
    return got.double().cpu().numpy(), ref.double().cpu().numpy()


def _oracle(c: Case, q: np.ndarray, lens, batch: int = 0):
    B = batch or c.B
    return O.decode(c.spec, q[:B], c.pools, c.bt[:B], np.asarray(lens, np.int32)[:B])


def test_noalloc_counter_path_twice_then_another_batch():
    w = wl.workload("llama8b", batch=3)
    c = Case(w, [1000, 37, 2049])
    calls = ((0, [1000, 37, 2049], 0), (1, [999, 5, 1500], 0), (2, [640, 33, 2049], 2))
    for step, lens, batch in calls:
        q = c.queries(step=step)
        got, ref = _both(c, q, lens, chunk=64, batch=batch)
        assert np.all(np.isfinite(got)), step
        assert np.array_equal(got, ref), step
        assert max_row_err(got, _oracle(c, q, lens, batch), floor=floor_for(c.w)) <= TOL, step
    assert c.cache.status_bits() == 0


def test_noalloc_library_chunks_and_other_codec():
    w = wl.workload("long_mixed", batch=2)
    c = Case(w, [3000, 333])
    for step in (0, 1):
        lens = [3000 - 7 * step, 333]
        q = c.queries(step=step)
        got, ref = _both(c, q, lens)
        assert np.array_equal(got, ref), step
        assert max_row_err(got, _oracle(c, q, lens), floor=floor_for(c.w)) <= TOL, step
    assert c.cache.status_bits() == 0


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
