"""GPU path (through the C ABI) against the CPU oracle on the same seeded inputs.

Codes and scales: bytewise equal pools.  Outputs: max row-relative error
<= 2e-3 and max normwise error <= 2e-3 in every decode check.  Elements below
0.1 % of the row's largest magnitude compare against that floor; layers with
a raised score scale pass a wider floor (gpu_cases.floor_for).  Sizes span
several chunks, several pages and ragged tails.
"""
import numpy as np
import pytest
import torch

import kvq_workloads as wl
from gpu_cases import TOL, Case, floor_for, max_row_err, oracle_rope
from int8_quantized_paged_gb300 import kvq
from int8_quantized_paged_gb300.cache import LayerCache
from oracle import kvq_oracle as O

pytestmark = pytest.mark.gpu

needs_cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    torch.cuda.init()


SMALL = {
    "tiny": dict(lens=[256]),
    "llama8b": dict(lens=[1000, 37, 2049], over=dict(batch=3)),
    "contbatch": dict(lens=[0, 1, 16, 17, 700, 2900], over=dict(batch=6)),
    "gemma_mix": dict(lens=[3001, 5], over=dict(batch=2)),
    "long_mixed": dict(lens=[5000, 777], over=dict(batch=2)),
    "llama8b_f16": dict(lens=[1000, 37, 2049], over=dict(batch=3)),
    "long_f16": dict(lens=[3000, 777], over=dict(batch=2)),
    "llama8b_shimmy": dict(lens=[1000, 37, 2049], over=dict(batch=3)),
    "long_shimmy": dict(lens=[3000, 777], over=dict(batch=2)),
}


def test_normwise_error_small():
    w = wl.workload("gemma_mix", batch=2)
    c = Case(w, [3001, 5])
    q = c.queries()
    got = c.gpu_decode(q)
    ref = c.oracle_decode(q)
    assert float(np.max(O.row_norm_error(got, ref))) <= TOL
    assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL


def _case(name, **kw):
    spec = SMALL[name]
    w = wl.workload(name, **spec.get("over", {}))
    return Case(w, spec["lens"], **kw)


@pytest.fixture(scope="module", params=list(SMALL))
def case(request):
    return _case(request.param)


def test_append_codes_bytewise(case):
    k, v = case.gpu_pools()
    assert np.array_equal(k, case.pools["k"])
    assert np.array_equal(v, case.pools["v"])
    assert case.cache.status_bits() == 0


@pytest.mark.parametrize("chunk", [0, 16, 64, 512])
def test_decode_matches_oracle(case, chunk):
    q = case.queries()
    ref = case.oracle_decode(q)
    got = case.gpu_decode(q, chunk_tokens=chunk)
    assert np.all(np.isfinite(got))
    assert max_row_err(got, ref, floor=floor_for(case.w)) <= TOL
    for b, L in enumerate(case.lens):
        if L == 0:
            assert np.all(got[b] == 0)
    assert case.cache.status_bits() == 0


def test_chunk_count_invariance(case):
    q = case.queries(step=1)
    a = case.gpu_decode(q, chunk_tokens=16)
    b = case.gpu_decode(q, chunk_tokens=1024)
    c = case.gpu_decode(q)
    ref = case.oracle_decode(q)
    for x in (a, b, c):
        assert max_row_err(x, ref, floor=floor_for(case.w)) <= TOL
    assert np.max(np.abs(a - c)) <= 4e-3 * max(1e-6, np.max(np.abs(ref)))


@pytest.mark.parametrize("L", [1, 1000, 1024, 1025, 1152, 1153, 3000])
def test_window_ring_matches_oracle(L):
    w = wl.workload("gemma_mix")
    c = Case(w, [L], ring_rows=1152)
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    q = c.queries()
    ref = c.oracle_decode(q, window=1024)
    for chunk in (0, 64):
        got = c.gpu_decode(q, chunk_tokens=chunk, window=1024)
        assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL, (L, chunk)


def test_window_small_ring_other_codec():
    # a symmetric-INT4 layer with a 64-row ring and a 40-token window
    w = wl.workload("llama8b", batch=3)
    c = Case(w, [10, 64, 333], ring_rows=64)
    q = c.queries()
    ref = c.oracle_decode(q, window=40)
    got = c.gpu_decode(q, window=40)
    assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL


def test_length_one_returns_its_value():
    w = wl.workload("llama8b", batch=1)
    c = Case(w, [1])
    q = c.queries()
    got = c.gpu_decode(q)
    ref = c.oracle_decode(q)                       # = the dequantized v of token 0
    assert max_row_err(got, ref, floor=floor_for(c.w)) <= TOL


def test_non_default_stream_and_isolation():
    w = wl.workload("llama8b", batch=2)
    c = Case(w, [300, 500], extra_pages=4)
    q = c.queries()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        before = c.gpu_decode(q, stream=s)
    ref = c.oracle_decode(q)
    assert max_row_err(before, ref, floor=floor_for(c.w)) <= TOL
    # grow sequence 0 by one token: sequence 1's output must not change at all
    c.cache.reserve(0, 301)
    c.cache.sync_table()
    dev = c.cache.device
    rows = torch.from_numpy(wl.new_rows(w, "k", 1)).to(dev)
    c.cache.append(rows, rows, torch.tensor([300], dtype=torch.int32, device=dev),
                   torch.tensor([0], dtype=torch.int32, device=dev))
    after = c.gpu_decode(q, lens=[301, 500])
    assert np.array_equal(before[1], after[1])
    assert not np.array_equal(before[0], after[0])


def test_device_status_flags_bad_inputs():
    w = wl.workload("llama8b", batch=3)
    c = Case(w, [40, 40, 40], fill_oracle=True)
    q = c.queries()
    ref = c.oracle_decode(q)
    dev = c.cache.device
    # a page id outside the pool in sequence 1
    bad = c.bt.copy()
    bad[1, 1] = c.n_pages + 5
    c.cache.set_table(bad)
    kvq.clear_device_status(c.cache.status)
    got = c.gpu_decode(q)
    assert c.cache.status_bits() & kvq.DEV_BAD_PAGE
    assert max_row_err(got, ref, seqs=[0, 2], floor=floor_for(c.w)) <= TOL   # other sequences unaffected
    assert np.all(np.isfinite(got[1]))                         # the bad page's rows are left out
    c.cache.set_table(c.bt)
    # a length past the table's capacity gives a zero row and a flag
    kvq.clear_device_status(c.cache.status)
    got = c.gpu_decode(q, lens=[40, 10 ** 6, 40])
    assert c.cache.status_bits() & kvq.DEV_BAD_LEN
    assert np.all(got[1] == 0) and max_row_err(got, ref, seqs=[0, 2], floor=floor_for(c.w)) <= TOL
    # append: a sequence id and a position outside the table are flagged and skipped
    kvq.clear_device_status(c.cache.status)
    k0 = c.cache.k_pool.clone()
    rows = torch.zeros(2, 8, 128, dtype=torch.float16, device=dev)
    c.cache.append(rows, rows, torch.tensor([5, 10 ** 5], dtype=torch.int32, device=dev),
                   torch.tensor([7, 0], dtype=torch.int32, device=dev))
    bits = c.cache.status_bits()
    assert bits & kvq.DEV_BAD_SEQ and bits & kvq.DEV_BAD_POS
    assert torch.equal(k0, c.cache.k_pool)
    kvq.clear_device_status(c.cache.status)
    assert c.cache.status_bits() == 0


def test_empty_batch_is_noop():
    w = wl.workload("tiny")
    c = Case(w, [256], fill_oracle=False)
    cfg = c.cfg
    q = torch.zeros(0, 4, 64, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    kvq.decode_attention(cfg, q, c.cache.k_pool, c.cache.v_pool, c.n_pages, c.cache.block_table,
                         c.max_pages, c.cache.block_table, c.cache.rope_tab, c.rope_max, q, ws, c.cache.status)


def test_group16_runs_on_cuda_core_kernel():
    # groups of 16 elements go to the CUDA-core decode kernel (tensor-core path needs >= 32)
    w = wl.workload("llama8b", batch=2, k_group=16, v_group=16, k_param="f16", v_param="bf16")
    c = Case(w, [700, 33])
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    q = c.queries()
    ref = c.oracle_decode(q)
    for chunk in (0, 64):
        assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk), ref, floor=floor_for(c.w)) <= TOL


@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("heads", [(64, 8), (32, 4)])
def test_wide_query_groups_match_oracle(heads, chunk):
    """G = 8 query heads per kv head with 4-bit K and V: the 8 heads share one
    MMA tile, the high and low parts of q and of the weights as two passes."""
    w = wl.workload("llama8b", batch=2, n_heads=heads[0], n_kv_heads=heads[1])
    c = Case(w, [700, 33])
    q = c.queries()
    assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk), c.oracle_decode(q), floor=floor_for(c.w)) <= TOL
    assert c.cache.status_bits() == 0


@pytest.mark.parametrize("chunk", [0, 64])
@pytest.mark.parametrize("heads", [(8, 8), (16, 8), (32, 8), (64, 8)])
@pytest.mark.parametrize("kv", [("sym8", "sym4", 32, "f16"), ("sym4", "sym4", 64, "f32"),
                                ("sym8", "sym8", 32, "bf16")])
def test_several_v_groups_match_oracle(kv, heads, chunk):
    """Symmetric V with several groups per head vector at G = 1, 2, 4 and 8:
    the weights of each group are formed in the P.V operand layout.  1 % of
    the elements x 8 move the groups' reference scales up between pages."""
    kk, vk, g, par = kv
    w = wl.workload("long_mixed", batch=2, n_heads=heads[0], n_kv_heads=heads[1], k_kind=kk, v_kind=vk,
                    k_group=g, v_group=g, k_param=par, v_param=par)
    c = Case(w, [1500, 41])
    q = c.queries()
    assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk), c.oracle_decode(q), floor=floor_for(c.w)) <= TOL
    assert c.cache.status_bits() == 0


def test_several_v_groups_window_matches_oracle():
    """The same weights at the window's first page, which starts mid-page."""
    w = wl.workload("long_mixed", batch=2, n_heads=32, n_kv_heads=4, ctx=4096)
    c = Case(w, [1500, 3000], ring_rows=1152)
    q = c.queries()
    ref = c.oracle_decode(q, window=1000)
    for chunk in (0, 64):
        assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk, window=1000), ref, floor=floor_for(c.w)) <= TOL


def test_wide_query_group_affine_matches_oracle():
    """G = 8 with affine 4-bit K/V (per-group q sums of the 8 heads)."""
    w = wl.workload("gemma_mix", batch=2, n_heads=64, n_kv_heads=8, head_dim=128)
    c = Case(w, [900, 17])
    q = c.queries()
    for chunk in (0, 64):
        assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk), c.oracle_decode(q), floor=floor_for(c.w)) <= TOL


def _tie_rows(w: dict, n_rows: int, seed: int) -> np.ndarray:
    """Rows whose quotients x / scale land on, and one or two ulps beside,
    half-integers: each group's largest magnitude is qmax * s for a random s,
    so the stored scale is (close to) s, and the other elements are
    (k + 1/2) * scale for the scale the quantizer will store."""
    rng = np.random.default_rng(seed)
    hkv, hd, g = w["n_kv_heads"], w["head_dim"], w["k_group"]
    qmax = {"sym8": 127.0, "shimmy4": 7.5}.get(w["k_kind"], 7.0)
    rows = np.zeros((n_rows, hkv, hd), np.float32)
    for r in range(n_rows):
        for h in range(hkv):
            for g0 in range(0, hd, g):
                s = np.float32(rng.uniform(0.05, 3.0))
                amax = np.float32(qmax) * s
                scale = np.float32(np.float32(amax) / np.float32(qmax))
                if w["k_param"] == "f16":
                    scale = np.float32(np.float16(scale))
                ks = rng.integers(-int(qmax + 0.5), int(qmax), g).astype(np.float32) + np.float32(0.5)
                x = (ks * scale).astype(np.float32)
                nudge = rng.integers(-2, 3, g)
                x = np.array([np.nextafter(v, np.float32(np.inf) if d > 0 else np.float32(-np.inf))
                              if d else v for v, d in zip(x, nudge)], np.float32)
                x[0] = amax * (1 if rng.random() < 0.5 else -1)
                rows[r, h, g0:g0 + g] = np.clip(x, -amax, amax)
    return rows


@pytest.mark.parametrize("name,over", [
    ("tiny", dict(rope="none")),
    ("long_mixed", dict(rope="none", act="f32", k_kind="sym8", v_kind="sym8")),
    ("llama8b", dict(rope="none", act="f32", k_kind="shimmy4", v_kind="shimmy4")),
])
def test_append_codes_at_rounding_ties(name, over):
    """Codes of quotients at and next to rounding ties: the append kernel and
    the fused call write the oracle's bytes (the division-free quotient falls
    back to the exact one there)."""
    w = wl.workload(name, batch=1, **over)
    cfg = kvq.config(**w)
    spec = O.Spec.from_workload(w)
    n = 48
    cache = LayerCache(cfg, 1, 4, 4, rope_max_pos=n + 1)
    cache.reserve(0, n)
    cache.sync_table()
    bt = cache.table.data()
    k, v = _tie_rows(w, n, 1), _tie_rows(w, n, 2)
    dev = cache.device
    cache.append(torch.from_numpy(k[:n - 1]).to(dev), torch.from_numpy(v[:n - 1]).to(dev),
                 torch.arange(n - 1, dtype=torch.int32, device=dev),
                 torch.zeros(n - 1, dtype=torch.int32, device=dev))
    # the last row through the fused call
    q = torch.from_numpy(wl.queries(dict(w, batch=1)).astype(np.float32)).to(dev)
    out = torch.empty_like(q)
    cache.append_decode(q, torch.from_numpy(k[n - 1:]).to(dev), torch.from_numpy(v[n - 1:]).to(dev),
                        torch.tensor([n - 1], dtype=torch.int32, device=dev),
                        torch.tensor([n], dtype=torch.int32, device=dev), out, cache.workspace(1))
    torch.cuda.synchronize()
    assert cache.status_bits() == 0
    pools = {"k": np.zeros(4 * O.page_bytes(spec, "k"), np.uint8), "v": np.zeros(4 * O.page_bytes(spec, "v"), np.uint8)}
    O.append(spec, pools, k, v, np.zeros(n, np.int64), np.arange(n), bt, 0, oracle_rope(spec.head_dim, spec.rope_base, n + 1))
    assert np.array_equal(cache.k_pool.cpu().numpy(), pools["k"])
    assert np.array_equal(cache.v_pool.cpu().numpy(), pools["v"])


# ---------------------------------------------------------------- bf16 activations

def _round_bf16(x: np.ndarray) -> np.ndarray:
    """x rounded once to bf16, as fp32 (input preparation: both sides read these values)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


class _Bf16Case(Case):
    """A Case with bf16 activations: rows and queries drawn in fp32 and rounded to
    bf16 once; the device gets the bf16 tensors, the oracle the same values."""

    def _draws(self) -> dict:
        return dict(self.w, act="f32")

    def _fill_gpu(self):
        dev = self.cache.device
        for b, L in enumerate(self.lens):
            k = _round_bf16(wl.kv_rows(self._draws(), b, "k", int(L)))
            v = _round_bf16(wl.kv_rows(self._draws(), b, "v", int(L)))
            if b in self.oracle_seqs:
                self.rows[b] = (k, v)
            for s, e in self._chunks(int(L)):
                self.cache.append(torch.from_numpy(k[s:e]).to(dev).to(torch.bfloat16),
                                  torch.from_numpy(v[s:e]).to(dev).to(torch.bfloat16),
                                  torch.arange(s, e, dtype=torch.int32, device=dev),
                                  torch.full((e - s,), b, dtype=torch.int32, device=dev))
        torch.cuda.synchronize()

    def queries(self, step: int = 0) -> np.ndarray:
        return _round_bf16(wl.queries(dict(self._draws(), batch=self.B), step=step))

    def gpu_decode(self, q: np.ndarray, chunk_tokens: int = 0, window: int = 0, lens=None, stream=None):
        dev = self.cache.device
        qt = torch.from_numpy(q).to(dev).to(torch.bfloat16)
        out = torch.full_like(qt, float("nan"))
        ws = self.cache.workspace(self.B, chunk_tokens, window)
        lt = torch.from_numpy(self.lens).to(dev)
        if window:
            self.cache.window_decode(qt, lt, out, ws, window, chunk_tokens)
        else:
            self.cache.decode(qt, lt, out, ws, chunk_tokens)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64)


# The output is rounded once to bf16 (8 significant bits): up to 2^-8 of its
# magnitude on top of the 2e-3 bound of the arithmetic before it.
TOL_BF16_OUT = TOL + 2.0 ** -8


@pytest.mark.parametrize("name", ["llama8b", "gemma_mix", "long_mixed"])
def test_bf16_activations_match_oracle(name):
    """bf16 q, K/V rows and output: pools bytewise, outputs within TOL_BF16_OUT,
    for the plain decode (both launch modes) and the fused step."""
    c = _Bf16Case(wl.workload(name, batch=2, act="bf16"), [700, 33])
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    q = c.queries()
    ref = c.oracle_decode(q)
    for chunk in (0, 64):
        assert max_row_err(c.gpu_decode(q, chunk_tokens=chunk), ref, floor=floor_for(c.w)) <= TOL_BF16_OUT, chunk
    # the fused step: new rows at L - 1
    dev = c.cache.device
    k_new = _round_bf16(wl.new_rows(c._draws(), "k", c.B, step=1))
    v_new = _round_bf16(wl.new_rows(c._draws(), "v", c.B, step=1))
    q1 = c.queries(step=1)
    pos = (c.lens - 1).astype(np.int32)
    qt = torch.from_numpy(q1).to(dev).to(torch.bfloat16)
    out = torch.full_like(qt, float("nan"))
    c.cache.append_decode(qt, torch.from_numpy(k_new).to(dev).to(torch.bfloat16),
                          torch.from_numpy(v_new).to(dev).to(torch.bfloat16), torch.from_numpy(pos).to(dev),
                          torch.from_numpy(c.lens).to(dev), out, c.cache.workspace(c.B))
    torch.cuda.synchronize()
    assert c.cache.status_bits() == 0
    s = c.spec
    O.append(s, c.pools, k_new, v_new, np.arange(c.B), pos, c.bt, 0, oracle_rope(s.head_dim, s.rope_base, c.rope_max))
    k, v = c.gpu_pools()
    assert np.array_equal(k, c.pools["k"]) and np.array_equal(v, c.pools["v"])
    got = out.float().cpu().numpy().astype(np.float64)
    assert max_row_err(got, c.oracle_decode(q1), floor=floor_for(c.w)) <= TOL_BF16_OUT
