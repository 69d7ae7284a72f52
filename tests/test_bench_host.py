"""Host-side pieces of the bench that need no GPU: the staging of every layer's
step inputs and outputs into two flat buffers (one copy each way per
end-to-end step), and the kernel-source hash that keys the profiled traffic."""
import os
from types import SimpleNamespace

import pytest
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


def test_closed_form_bytes_match_the_library_and_the_oracle():
    """The bench's per-token byte count (no library call) equals the oracle's
    sizing and the library's kvq_cache_bytes for every bench workload."""
    import kvq_workloads as wl
    from int8_quantized_paged_gb300 import kvq
    from oracle import kvq_oracle as O
    for name in wl.WORKLOADS:
        w = wl.workload(name)
        hd, hkv = w["head_dim"], w["n_kv_heads"]
        per = (bench.kv_bytes_per_token_head(w["k_kind"], hd, w["k_group"], w["k_param"])
               + bench.kv_bytes_per_token_head(w["v_kind"], hd, w["v_group"], w["v_param"]))
        for which in ("k", "v"):
            kind, grp, par = w[which + "_kind"], w[which + "_group"], w[which + "_param"]
            assert bench.kv_bytes_per_token_head(kind, hd, grp, par) == O.bytes_per_token_head(kind, hd, grp, par)
        assert per * 16 * hkv == kvq.cache_bytes(kvq.config(**w), 1, 16), name


def test_algorithmic_bytes_of_the_llama8b_layer():
    import numpy as np
    import kvq_workloads as wl
    w = wl.workload("llama8b")
    dec, app = bench.algorithmic_bytes(w, np.array([8192]), 0)
    # 8192 tokens x 8 kv heads x (68 + 68) B, q and out (2 x 32 x 128 x 2 B),
    # 512 block-table entries and one length
    assert dec == 8192 * 8 * 136 + 2 * 32 * 128 * 2 + 4 * 512 + 4
    assert app == 2 * 8 * 128 * 2 + 4 * 128 + 8 + 8 * 136


def test_block_count_and_gpus_flag():
    assert bench.n_blocks_for(1000.0) == 5            # long blocks: the minimum of 5
    assert bench.n_blocks_for(5.0) == 200             # about a second of timed work
    assert bench.n_blocks_for(0.001) == 400           # capped
    assert bench.check_gpus_flag(1, 1) is None
    assert "WORLD_SIZE" in bench.check_gpus_flag(8, 1)


def test_gpus_flag_mismatch_exits_nonzero():
    import subprocess
    import sys
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    r = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 2 and "--gpus 2" in r.stderr


def test_oracle_sample_loads_no_product_library():
    """The CPU arm (cpu_baseline, --impl reference) runs the oracle only: its
    process imports no part of the package and maps no libkvq.so."""
    import subprocess
    import sys
    code = ("import sys, bench\n"
            "step, nbytes, desc = bench.oracle_sample('tiny_model')\n"
            "step()\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert 'libkvq' not in maps, 'libkvq mapped'\n"
            "assert not any(m.startswith('int8_quantized_paged_gb300') for m in sys.modules), 'package imported'\n"
            "print(nbytes)\n")
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1")
    pre = ("import bench; bench.MODELS['tiny_model'] = [('tiny', 1, False)]\n")
    r = subprocess.run([sys.executable, "-c", pre + code], capture_output=True, text=True, env=env,
                       cwd=bench.ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert int(r.stdout.split()[-1]) > 0


def test_summarize_rates_and_fractions():
    """One measured model's numbers: whole-job GB/s from the step bytes, the
    launch time from the step (one kernel a layer) and the roofline fraction."""
    r = {"ms_per_step": 0.25, "launches_per_step": 32, "one_kernel": True, "call_bytes": 8.0e6,
         "step_bytes": 2.56e8, "query_tokens": 1, "ctx_tokens": 32 * 8192, "layers": 32, "batch": 1,
         "ctx": 8192, "blocks": 7, "block_ms_per_step": {"median": 0.25}, "l2": "x"}
    s = bench.summarize(r, 1, 6000.0)
    assert s["value"] == pytest.approx(1024.0)                 # 2.56e8 B / 0.25 ms
    assert s["avg_launch_us"] == pytest.approx(0.25e3 / 32, abs=1e-3)   # the step over its launches
    assert s["frac"] == pytest.approx(8.0e6 / (0.25e-3 / 32) / 1e9 / 6000.0, rel=1e-3)
    assert s["pct_of_hbm_peak"] == pytest.approx(100 * 1024.0 / 6000.0, abs=0.01)
    assert s["pct_of_nominal_hbm"] == pytest.approx(100 * 1024.0 / 8000.0, abs=0.01)
    assert s["tokens_per_s"] == pytest.approx(4000.0)
    assert s["context_tokens_per_s"] == pytest.approx(32 * 8192 / 0.25e-3)
    # two replicas: the job's value counts both ranks' bytes over the slowest rank's time
    s2 = bench.summarize(r, 2, 6000.0)
    assert s2["value"] == pytest.approx(2048.0) and s2["pct_of_hbm_peak"] == s["pct_of_hbm_peak"]
    # with more than one launch a layer, the launch time is the bracketed one
    r3 = dict(r, one_kernel=False, bracketed_ms=0.01)
    assert bench.summarize(r3, 1, 6000.0)["avg_launch_us"] == pytest.approx(10.0)


def test_early_reads_only_where_the_previous_kernel_is_another_layer():
    """KVQ_FLAG_EARLY_READS lets a call read its pages before the kernel before
    it ends, so the bench sets it only for models of several layers, each call
    following another layer's, and never for the separate append + decode."""
    a = SimpleNamespace(separate=False, no_early_reads=False)
    assert bench.early_reads("llama8b", a) and bench.early_reads("gemma_window", a)
    assert bench.early_reads("long_mixed", a)
    assert not bench.early_reads("contbatch", a)            # one layer: its own previous step
    assert not bench.early_reads("llama8b", SimpleNamespace(separate=True, no_early_reads=False))
    assert not bench.early_reads("llama8b", SimpleNamespace(separate=False, no_early_reads=True))
