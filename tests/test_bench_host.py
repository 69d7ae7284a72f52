"""Host-side pieces of the bench that need no GPU: the staging of every layer's
step inputs and outputs into two flat buffers (one copy each way per
end-to-end step), and the kernel-source hash that keys the profiled traffic."""
import os
from types import SimpleNamespace

import torch

import bench


def _layer(seed: int, B: int, hq: int, hkv: int, hd: int, dtype=torch.float16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, hq, hd), generator=g).to(dtype)
    return SimpleNamespace(q=q, k_new=torch.randn((B, hkv, hd), generator=g).to(dtype),
                           v_new=torch.randn((B, hkv, hd), generator=g).to(dtype), out=torch.zeros_like(q))


def test_stage_io_keeps_values_and_shares_two_buffers():
    layers = [_layer(i, 2, 32, 8, 128) for i in range(5)]
    before = [(L.q.clone(), L.k_new.clone(), L.v_new.clone()) for L in layers]
    io_in, io_out = bench.stage_io(layers, torch.device("cpu"))
    assert io_in.dim() == 1 and io_out.dim() == 1
    assert io_in.numel() == sum(t.numel() for b in before for t in b)
    assert io_out.numel() == sum(L.out.numel() for L in layers)
    base_in = io_in.data_ptr()
    for L, (q, k, v) in zip(layers, before):
        assert torch.equal(L.q, q) and torch.equal(L.k_new, k) and torch.equal(L.v_new, v)
        for t in (L.q, L.k_new, L.v_new):
            assert t.untyped_storage().data_ptr() == io_in.untyped_storage().data_ptr()
            off = t.data_ptr() - base_in
            assert off % (128 * t.element_size()) == 0   # every view starts on a head_dim boundary
            assert t.is_contiguous()
        assert L.out.untyped_storage().data_ptr() == io_out.untyped_storage().data_ptr()
    # one copy into the flat buffer reaches every layer's view
    io_in.fill_(1.5)
    assert all(float(L.q[0, 0, 0]) == 1.5 and float(L.v_new[-1, -1, -1]) == 1.5 for L in layers)
    layers[3].out.fill_(2.0)
    n = sum(L.out.numel() for L in layers[:3])
    assert torch.all(io_out[n:n + layers[3].out.numel()] == 2.0) and float(io_out[:n].abs().sum()) == 0.0


def test_kernel_source_hash_covers_the_kernel_files():
    for rel in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(bench.ROOT, rel)), rel
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert bench.kernel_source_hash() == h   # a pure function of the files


def test_profiled_traffic_is_keyed_by_the_source_hash():
    # a workload the summary does not list has no figure; a listed one has its
    # bytes while the hash matches and none once the kernel sources change
    assert bench.profiled_traffic("no_such_workload") is None
    t = bench.profiled_traffic("llama8b")
    assert t is None or (isinstance(t, int) and t > 0)
