"""The C-ABI library on the host (no GPU): exports, sizing, RoPE table, page
pool, block tables and argument checks."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import kvq_workloads as wl
from int8_quantized_paged_gb300 import kvq
from oracle import kvq_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not os.path.exists(kvq.LIB_PATH):
        from int8_quantized_paged_gb300 import build
        build.build()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", text)))


def test_header_symbols_exported_and_bound():
    declared = _declared()
    assert len(declared) >= 25
    lib = C.CDLL(kvq.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(kvq.exported_symbols()) == declared


def test_abi_version_matches_header():
    m = re.search(r"#define KVQ_ABI_VERSION (\d+)", open(HEADER).read())
    assert kvq.abi_version() == int(m.group(1))


def _cfg(w):
    return kvq.config(**w)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_cache_and_page_bytes_match_oracle(name):
    w = wl.workload(name)
    cfg = _cfg(w)
    s = O.Spec.from_workload(w)
    for layers, ctx in [(1, w["ctx"]), (32, 8192), (3, 17), (1, 0)]:
        want = O.cache_bytes(layers, w["n_kv_heads"], w["head_dim"], ctx, 16, w["k_kind"], w["v_kind"],
                             w["k_group"], w["v_group"], w["k_param"], w["v_param"])
        assert kvq.cache_bytes(cfg, layers, ctx) == want
    assert kvq.page_bytes(cfg, 0) == O.page_bytes(s, "k")
    assert kvq.page_bytes(cfg, 1) == O.page_bytes(s, "v")
    assert kvq.page_bytes(cfg, 0) % 16 == 0 and kvq.page_bytes(cfg, 1) % 16 == 0


def test_cache_bytes_pages_values():
    # the pages' printed sizes, through the library
    f32 = kvq.config(32, 8, 128, k_kind="f32", v_kind="f32")
    assert kvq.cache_bytes(f32, 1, 2048) == 16777216
    assert kvq.cache_bytes(f32, 28, 2048) == 448 * 2 ** 20
    f16 = kvq.config(32, 8, 128, k_kind="f16", v_kind="f16")
    assert kvq.cache_bytes(f16, 32, 8192) == 2 * 32 * 8 * 128 * 8192 * 2
    i4 = kvq.config(32, 8, 128, k_group=128, v_group=128, k_param="f32")
    assert kvq.cache_bytes(i4, 1, 128) / (2 * 8 * 128 * 128) == 0.53125
    assert kvq.cache_bytes(kvq.config(0, 8, 128), 1, 16) == 0      # invalid config -> 0
    assert kvq.cache_bytes(i4, -1, 16) == 0


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_rope_table_bitwise_equals_oracle(name):
    w = wl.workload(name)
    cfg = _cfg(w)
    n = 2048 if name != "tiny" else 256
    lib_tab = kvq.rope_table(cfg, n)
    ora_tab = O.rope_table(w["head_dim"], w["rope_base"], n)
    assert lib_tab.dtype == ora_tab.dtype == np.float32
    assert np.array_equal(lib_tab.view(np.uint32), ora_tab.view(np.uint32))


@pytest.mark.slow
def test_rope_table_high_positions_bitwise():
    w = wl.workload("long_mixed")
    cfg = _cfg(w)
    lib_tab = kvq.rope_table(cfg, 65536)
    rows = [65535, 40000, 32767, 9999]
    th = O.rope_theta(128, w["rope_base"])
    import math
    for p in rows:
        want = np.array([[math.cos(p * t), math.sin(p * t)] for t in th], dtype=np.float32)
        assert np.array_equal(lib_tab[p].view(np.uint32), want.view(np.uint32))


def test_validate_config():
    kvq.validate_config(_cfg(wl.workload("llama8b")))
    bad = [
        (dict(n_heads=30), kvq.ERR_INVALID_ARG),          # not a multiple of n_kv_heads
        (dict(n_heads=48, n_kv_heads=3), kvq.ERR_UNSUPPORTED),   # G = 16
        (dict(head_dim=96, k_group=32, v_group=32), kvq.ERR_UNSUPPORTED),
        (dict(page_size=32), kvq.ERR_UNSUPPORTED),
        (dict(k_group=48), kvq.ERR_INVALID_ARG),          # does not divide 128
        (dict(k_group=8, v_group=8), kvq.ERR_UNSUPPORTED),  # not a multiple of 16
        (dict(k_kind="sym4", v_kind="sym8"), kvq.ERR_UNSUPPORTED),
        (dict(k_kind="f16", v_kind="f16", head_dim=256, k_group=256, v_group=256), kvq.ERR_UNSUPPORTED),
        (dict(k_kind="f16", v_kind="sym4"), kvq.ERR_UNSUPPORTED),
        (dict(k_kind="shimmy4", v_kind="shimmy4", k_param="f16", v_param="f16"), kvq.ERR_UNSUPPORTED),
        (dict(k_kind="shimmy4", v_kind="shimmy4", k_group=16, v_group=16), kvq.ERR_UNSUPPORTED),
        (dict(rope_base=-1.0), kvq.ERR_INVALID_ARG),
    ]
    kvq.validate_config(_cfg(wl.workload("llama8b_f16")))   # unquantised f16 K/V at head_dim 128
    kvq.validate_config(_cfg(wl.workload("llama8b_shimmy")))  # the /7.5 offset-8 codec
    for over, want in bad:
        w = dict(wl.workload("llama8b"))
        w.update(over)
        with pytest.raises(kvq.KvqError) as e:
            kvq.validate_config(_cfg(w))
        assert e.value.status == want, over
    c = _cfg(wl.workload("llama8b"))
    c.flags = kvq.FLAG_EARLY_READS
    kvq.validate_config(c)                            # the one defined flag
    c.flags = 2
    with pytest.raises(kvq.KvqError):
        kvq.validate_config(c)                        # an unknown bit


def test_pool_lifo_and_errors():
    p = kvq.Pool(8)
    assert p.num_pages == 8 and p.num_free == 8
    assert list(p.alloc(3)) == [0, 1, 2]
    p.free([1, 0])
    assert list(p.alloc(2)) == [0, 1]                 # last freed comes out first
    with pytest.raises(kvq.KvqError) as e:
        p.alloc(7)                                    # only 5 free: all or nothing
    assert e.value.status == kvq.ERR_OUT_OF_PAGES and p.num_free == 5
    for ids in ([9], [-1], [3], [0, 0]):              # foreign, foreign, free, repeated
        before = p.num_free
        with pytest.raises(kvq.KvqError) as e:
            p.free(ids)
        assert e.value.status == kvq.ERR_INVALID_ARG and p.num_free == before
    p.free([0, 1, 2])
    assert p.num_free == 8
    with pytest.raises(kvq.KvqError):
        kvq.Pool(0)


def test_pool_shuffled_free_list():
    # Freeing a fresh pool's pages in a seeded order leaves its free list shuffled.
    w = wl.workload("contbatch")
    order = wl.page_free_order(w, 64)
    p = kvq.Pool(64)
    p.alloc(64)
    p.free(order)
    assert list(p.alloc(64)) == list(order[::-1])


def test_table_reserve_release_isolation():
    pool = kvq.Pool(10)
    t = kvq.Table(pool, 3, 4, 16)
    t.reserve(0, 17)                                  # 2 pages
    t.reserve(1, 16)                                  # 1 page
    t.reserve(0, 32)                                  # still 2 pages
    assert (t.num_pages(0), t.num_pages(1), t.num_pages(2)) == (2, 1, 0)
    d = t.data()
    assert list(d[0]) == [0, 1, -1, -1] and list(d[1]) == [2, -1, -1, -1]
    t.reserve(2, 64)
    held = d[:2][d[:2] >= 0].tolist() + t.data()[2].tolist()
    assert len(set(held)) == len(held) == 7           # no page in two sequences
    t.reserve(1, 64)                                  # needs 3 more: exactly the 3 free
    assert pool.num_free == 0
    with pytest.raises(kvq.KvqError) as e:
        t.reserve(0, 64)                              # 2 more pages, none free
    assert e.value.status == kvq.ERR_OUT_OF_PAGES and t.num_pages(0) == 2
    with pytest.raises(kvq.KvqError) as e:
        t.reserve(0, 65)                              # 5 pages > 4 per sequence
    assert e.value.status == kvq.ERR_INVALID_ARG
    t.release(2)                                      # sequence 2 finished
    assert pool.num_free == 4 and list(t.data()[2]) == [-1] * 4
    t.reserve(0, 64)
    assert t.num_pages(0) == 4
    t.close()                                         # returns every page
    assert pool.num_free == 10


def _host_cfg():
    return kvq.config(32, 8, 128)


def test_device_calls_reject_bad_arguments_before_launch():
    """These fail in host validation, so they run without a GPU."""
    import torch
    cfg = _host_cfg()
    dummy = torch.zeros(16, dtype=torch.uint8)   # host tensor: never dereferenced
    with pytest.raises(kvq.KvqError) as e:       # NULL pools
        kvq.append(cfg, torch.zeros(1, 8, 128, dtype=torch.float16), torch.zeros(1, 8, 128,
                   dtype=torch.float16), None, dummy, dummy, 1, 4, 0, None, 0, None, None, 4, dummy,
                   stream=0)
    assert e.value.status == kvq.ERR_INVALID_ARG
    with pytest.raises(kvq.KvqError) as e:       # ring_rows not a multiple of the page
        kvq.append(cfg, torch.zeros(1, 8, 128, dtype=torch.float16), torch.zeros(1, 8, 128,
                   dtype=torch.float16), None, dummy, dummy, 1, 4, 20, dummy, 1, dummy, dummy, 4,
                   dummy, stream=0)
    assert e.value.status == kvq.ERR_INVALID_ARG
    ws_need = kvq.decode_workspace_bytes(cfg, 2, 512)
    small = torch.zeros(ws_need - 256, dtype=torch.uint8)
    q = torch.zeros(2, 32, 128, dtype=torch.float16)
    lens = torch.zeros(2, dtype=torch.int32)
    aligned = kvq.lib()  # noqa: F841
    # the workspace check comes before any launch; alignment of host tensors is not guaranteed,
    # so accept either "too small" or "alignment" as the rejection reason
    with pytest.raises(kvq.KvqError) as e:
        kvq.decode_attention(cfg, q, dummy, dummy, 4, dummy, 512, lens, dummy, 1, q, small, dummy,
                             stream=0)
    assert e.value.status in (kvq.ERR_WORKSPACE_TOO_SMALL, kvq.ERR_INVALID_ARG)
    with pytest.raises(kvq.KvqError) as e:       # chunk not a multiple of the page
        kvq.decode_attention(cfg, q, dummy, dummy, 4, dummy, 512, lens, dummy, 1, q, small, dummy,
                             chunk_tokens=24, stream=0)
    assert e.value.status == kvq.ERR_INVALID_ARG
    with pytest.raises(kvq.KvqError) as e:       # window larger than the ring
        kvq.window_decode(cfg, q, dummy, dummy, 4, dummy, 64, 65, lens, dummy, 1, q, small, dummy,
                          stream=0)
    assert e.value.status == kvq.ERR_INVALID_ARG
    # zero rows / zero batch are no-ops
    kvq.append(cfg, torch.zeros(0, 8, 128, dtype=torch.float16), torch.zeros(0, 8, 128,
               dtype=torch.float16), None, dummy, dummy, 1, 4, 0, dummy, 1, dummy, dummy, 4, dummy, stream=0)


def test_workspace_sizes():
    cfg = _host_cfg()
    a = kvq.decode_workspace_bytes(cfg, 4, 512, 256)
    # counters (4 seqs x 8 kv heads, 256-aligned), then 32 chunks x 4 q heads x 128 fp32 partial
    # sums per (seq, kv head), then (max, sum) pairs
    counters = 256
    acc = 4 * 8 * 32 * 4 * 128 * 4
    assert a == counters + (acc + 255) // 256 * 256 + 4 * 8 * 32 * 4 * 2 * 4
    assert kvq.window_workspace_bytes(cfg, 1, 1024, 64) < kvq.decode_workspace_bytes(cfg, 1, 1024, 64)
    with pytest.raises(kvq.KvqError):
        kvq.decode_workspace_bytes(cfg, 1, 512, 20)


def test_pool_finalized_before_its_table_is_safe():
    """The cyclic garbage collector may finalize a pool before a table that
    holds it; neither order may touch freed host memory."""
    import gc
    for first in ("pool", "table"):
        pool = kvq.Pool(8)
        table = kvq.Table(pool, 2, 4)
        table.reserve(0, 40)
        assert pool.num_free == 5
        if first == "pool":
            pool.close()              # destroys the table first, then the pool
            table.close()             # a no-op now
        else:
            table.close()
            assert pool.num_free == 8
            pool.close()
        cycle = [kvq.Pool(4)]
        cycle.append(kvq.Table(cycle[0], 1, 4))
        cycle[1].reserve(0, 16)
        cycle.append(cycle)           # a reference cycle the collector has to break
        del cycle
        gc.collect()


@pytest.mark.parametrize("name", ["kvq_append", "kvq_decode_attention", "kvq_decode_attention_noalloc",
                                  "kvq_window_decode", "kvq_append_decode_attention",
                                  "kvq_append_window_decode"])
def test_unknown_flag_bits_refused_by_every_entry_point(name):
    """An unknown kvq_config.flags bit fails the host checks of every device
    entry point before any pointer is touched or anything is launched."""
    c = _cfg(wl.workload("llama8b"))
    c.flags = 1 << 4
    fn = getattr(kvq.lib(), name)
    args = []
    for t in fn.argtypes:
        if t is C.c_void_p:
            args.append(None)
        elif t in (C.c_int32, C.c_int64, C.c_size_t):
            args.append(1)
        else:                               # the config pointer
            args.append(C.byref(c))
    assert fn(*args) == kvq.ERR_INVALID_ARG
    assert "flags" in kvq.last_error()
