"""Pins of the CPU oracle to facts the pages and mathematics fix (no GPU).

Each test targets a plausible mistake: a wrong rounding mode, clamp, scale
formula, nibble order, sign, pair index, theta exponent, GQA mapping, page or
ring index, window bound, or softmax normalisation.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import kvq_workloads as wl
from oracle import kvq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def _kv(line):
    parts = line.split()
    return parts[0], dict(p.split("=", 1) for p in parts[1:] if "=" in p), parts


# --------------------------------------------------------------------------- sizing


def test_sizing_values_printed_by_pages():
    for line in _golden_lines("kv_sizing.txt"):
        name, kv, _ = _kv(line)
        hd = int(kv["head_dim"])
        if name == "int4_per_elem":
            per = O.bytes_per_token_head(kv["kind"], hd, int(kv["group"]), kv["param"])
            assert per / hd == float(kv["expect_bytes_per_elem"])
            continue
        b = O.cache_bytes(int(kv["n_layers"]), int(kv["n_kv_heads"]), hd, int(kv["ctx"]),
                          16, kv["kind"], kv["kind"], hd, hd, "f32", "f32")
        if "expect_bytes" in kv:
            assert b == int(kv["expect_bytes"]), name
        else:
            assert b == int(kv["expect_mib"]) * 1024 * 1024, name


def test_sizing_formula_kaiwu_and_gqa():
    # KV_MB = 2 x layers x kv_heads x head_dim x ctx x bytes / 1024^2 (f16: bytes = 2)
    for layers, kvh, hd, ctx in [(32, 8, 128, 8192), (28, 4, 64, 4096), (1, 1, 256, 16)]:
        formula = 2 * layers * kvh * hd * ctx * 2
        assert O.cache_bytes(layers, kvh, hd, ctx, 16, "f16", "f16", hd, hd, "f32", "f32") == formula
    # GQA: the size follows kv_heads; counting query heads (32 vs 8) overestimates 4x.
    a = O.cache_bytes(32, 8, 128, 8192, 16, "sym4", "sym4", 128, 128, "f32", "f32")
    b = O.cache_bytes(32, 32, 128, 8192, 16, "sym4", "sym4", 128, 128, "f32", "f32")
    assert b == 4 * a


def test_sizing_workloads_and_page_rounding():
    # llama8b layer: 8 kv heads x 8192 tokens x (64 B codes + 4 B scale) x 2
    w = wl.workload("llama8b")
    s = O.Spec.from_workload(w)
    assert O.cache_bytes(1, 8, 128, 8192, 16, "sym4", "sym4", 128, 128, "f32", "f32") == 8912896
    assert O.page_bytes(s, "k") == 8 * 16 * 68
    # long_mixed: K 128 B + 4 fp16 scales, V 64 B + 4 fp16 scales -> 208 B per token-head
    assert O.cache_bytes(1, 4, 128, 65536, 16, "sym8", "sym4", 32, 32, "f16", "f16") == 4 * 65536 * 208
    # gemma_mix: 128 B codes + 4 groups x (scale, bias) bf16 = 144 B per token-head for K and V
    assert O.cache_bytes(1, 8, 256, 16384, 16, "affine4", "affine4", 64, 64, "bf16", "bf16") == 37748736
    # a partial page still costs a whole page
    assert O.cache_bytes(1, 2, 64, 17, 16, "sym4", "sym4", 64, 64, "f32", "f32") == \
        O.cache_bytes(1, 2, 64, 32, 16, "sym4", "sym4", 64, 64, "f32", "f32")


# --------------------------------------------------------------------------- codec


def _hexbytes(s):
    return np.array([int(t, 16) for t in s.split(",")], dtype=np.uint8)


def test_codec_hand_worked_examples():
    n = 0
    for line in _golden_lines("codec_examples.txt"):
        kind, group, param, xs, scale, bias, codes, bts = line.split()
        x = np.array([float(t) for t in xs.split(",")], dtype=np.float32)
        c, s, b = O.quantize(kind, x, int(group), param)
        assert np.array_equal(c.astype(int), [int(t) for t in codes.split(",")]), line
        assert s[0] == np.float32(float(scale)), line
        if bias != "-":
            assert b[0] == np.float32(float(bias)), line
        assert np.array_equal(O.pack_codes(kind, c), _hexbytes(bts)), line
        assert np.array_equal(O.unpack_codes(kind, _hexbytes(bts)), c.astype(np.int16)), line
        n += 1
    assert n >= 10


def _f32(v):
    return float(np.float32(v))


def _f16_struct(v):
    """fp32 -> fp16 -> float via Python's struct (independent of numpy)."""
    return struct.unpack("<e", struct.pack("<e", v))[0]


def _bf16_torch(v):
    torch = pytest.importorskip("torch")
    return float(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).float()[0])


def _stored(v, param):
    if param == "f32":
        return _f32(v)
    if param == "f16":
        return _f16_struct(v)
    return _bf16_torch(v)


def _nearest_even(y, lo, hi):
    """argmin_c |y - c| over integers in [lo, hi], ties to the even c (brute force)."""
    best = None
    for c in range(lo, hi + 1):
        d = abs(Fraction(y) - c)
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
            best = (d, c)
    return best[1]


@pytest.mark.parametrize("kind,bits,param", [("sym4", 4, "f32"), ("sym4", 4, "f16"),
                                             ("sym8", 8, "f16"), ("sym4", 4, "bf16")])
def test_sym_codec_matches_brute_force(kind, bits, param):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((40, 32)).astype(np.float32)
    x[3] *= 1e-6                                   # tiny groups exercise the floor
    x[5, :16] = 0.0                                # an all-zero group
    x[7] = np.round(x[7] * 4) / 4                  # many exact .5 quotients
    x[9] *= 300.0                                  # large magnitudes
    group = 16
    c, s, _ = O.quantize(kind, x, group, param)
    q = 2 ** (bits - 1) - 1
    floor = 2.0 ** -14 if param == "f16" else _f32(1e-8)
    for r in range(x.shape[0]):
        for g in range(x.shape[1] // group):
            xs = [float(v) for v in x[r, g * group:(g + 1) * group]]
            amax = max(abs(v) for v in xs)
            sc = _stored(max(_f32(amax / q), floor), param)
            assert s[r, g] == np.float32(sc)
            for j, v in enumerate(xs):
                y = _f32(v / sc)                 # fp32 division via exact double rounding
                assert c[r, g * group + j] == _nearest_even(y, -q, q), (r, g, j)


def test_affine_codec_matches_brute_force():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal((30, 64)) * 2 + 0.3).astype(np.float32)
    x[4, :32] = 1.25                               # constant group -> zero scale
    c, s, b = O.quantize("affine4", x, 32, "bf16")
    for r in range(x.shape[0]):
        for g in range(2):
            xs = [float(v) for v in x[r, g * 32:(g + 1) * 32]]
            sc = _bf16_torch(_f32(_f32(max(xs) - min(xs)) / 15.0))
            bi = _bf16_torch(min(xs))
            assert s[r, g] == np.float32(sc) and b[r, g] == np.float32(bi)
            for j, v in enumerate(xs):
                want = 0 if sc == 0 else _nearest_even(_f32(_f32(v - bi) / sc), 0, 15)
                assert c[r, g * 32 + j] == want


def test_round_trip_bound():
    # |x - x^| <= scale/2 for symmetric groups whose amax is at least Qmax * floor.
    rng = np.random.default_rng(3)
    for kind, bits in (("sym4", 4), ("sym8", 8)):
        x = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
        c, s, _ = O.quantize(kind, x, 32, "f32")
        xh = O.dequantize(c, s, None, 32)
        err = np.abs(x.astype(np.float64) - xh).reshape(200, 4, 32)
        assert np.all(err <= (s.astype(np.float64) / 2 * (1 + 2.0 ** -22))[..., None])
        # the largest element of each group gets the extreme code
        qmax = 2 ** (bits - 1) - 1
        assert np.all(np.max(np.abs(c.reshape(200, 4, 32)), axis=-1) == qmax)
    # the /7.5 codec: max|x| / scale = 7.5 up to the scale's rounding, so the
    # largest element lands on the clamp at +7 (or on -8) with an error of half
    # a step at most, the fp32 rounding of the scale aside (7.5 * 2^-24 of it)
    x = (rng.standard_normal((200, 128)) * rng.uniform(0.01, 50, (200, 1))).astype(np.float32)
    c, s, _ = O.quantize("shimmy4", x, 32, "f32")
    xh = O.dequantize(c, s, None, 32)
    err = np.abs(x.astype(np.float64) - xh).reshape(200, 4, 32)
    assert np.all(err <= (s.astype(np.float64) / 2 * (1 + 2.0 ** -19))[..., None])
    assert c.min() >= -8 and c.max() <= 7
    # the largest element's quotient is 7.5 up to the scale's rounding: code 7
    # (from +-7.5 down, or +8 clamped) or -8
    assert np.all(np.max(np.abs(c.reshape(200, 4, 32).astype(np.int64)), axis=-1) >= 7)
    # affine with bf16-exact min/max and an exact step: error <= scale/2
    mn = np.float32(-1.5)
    xs = (mn + np.arange(64, dtype=np.float32) * np.float32(15 / 63)).astype(np.float32)
    xs[-1] = np.float32(13.5)
    c, s, b = O.quantize("affine4", xs[None], 64, "bf16")
    assert s[0, 0] == 1.0 and b[0, 0] == -1.5
    assert np.all(np.abs(xs - O.dequantize(c, s, b, 64)[0]) <= 0.5)


def test_bf16_rounding_known_values():
    cases = {0.1: 0.10009765625, 1.0 + 2 ** -8: 1.0, 1.0 + 3 * 2 ** -8: 1.0 + 2 ** -6,
             -2.0 - 2 ** -7: -2.0, 3.0: 3.0}
    got = O.bf16_round(np.array(list(cases), dtype=np.float32))
    assert np.array_equal(got, np.array(list(cases.values()), dtype=np.float32))
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(5).standard_normal(10000).astype(np.float32) * 100
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    assert np.array_equal(O.bf16_round(x), ref)


# --------------------------------------------------------------------------- RoPE


def test_rope_closed_forms():
    for line in _golden_lines("rope_attention.txt"):
        name, kv, parts = _kv(line)
        if name != "rope":
            continue
        mode = parts[1]
        hd, base, pos = int(kv["hd"]), float(kv["base"]), int(kv["pos"])
        x = np.array([float(t) for t in kv["x"].split(",")])
        want = np.array([float(t) for t in kv["expect"].split(",")])
        assert np.allclose(O.rotate_f64(x, pos, hd, base, mode), want, rtol=0, atol=1e-15), line
        tab = O.rope_table(hd, base, pos + 1)
        got32 = O.rotate_f32(x.astype(np.float32), tab[pos], mode)
        assert np.allclose(got32, want, rtol=0, atol=4e-7), line


def test_rope_invariants():
    hd, base = 64, 10000.0
    tab = O.rope_table(hd, base, 300)
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0)
    th = O.rope_theta(hd, base)
    assert th[0] == 1.0 and math.isclose(th[-1], base ** (-(hd - 2) / hd), rel_tol=1e-15)
    x = np.random.default_rng(2).standard_normal(hd)
    for mode in ("normal", "neox"):
        i0, i1 = O.rope_pairs(hd, mode)
        for pos in (0, 1, 17, 299):
            y = O.rotate_f64(x, pos, hd, base, mode)
            assert np.allclose(np.hypot(y[i0], y[i1]), np.hypot(x[i0], x[i1]), rtol=1e-12)
            if pos == 0:
                assert np.array_equal(y, x)
        # composition: rotating by a then b equals rotating by a + b
        y = O.rotate_f64(O.rotate_f64(x, 5, hd, base, mode), 7, hd, base, mode)
        assert np.allclose(y, O.rotate_f64(x, 12, hd, base, mode), atol=1e-12)
    # NeoX pairing equals adjacent pairing on the interleaved vector
    perm = np.empty(hd, dtype=int)
    perm[0::2], perm[1::2] = np.arange(hd // 2), np.arange(hd // 2) + hd // 2
    a = O.rotate_f64(x, 9, hd, base, "neox")
    b = O.rotate_f64(x[perm], 9, hd, base, "normal")
    assert np.allclose(a[perm], b, atol=1e-13)
    # the fp32 rotation of K agrees with the fp64 one to fp32 accuracy
    x32 = x.astype(np.float32)
    for pos in (3, 150, 299):
        r32 = O.rotate_f32(x32, tab[pos], "normal")
        assert np.allclose(r32, O.rotate_f64(x32.astype(np.float64), pos, hd, base, "normal"),
                           atol=3e-6)


# --------------------------------------------------------------------------- attention


def _parse_mat(s):
    return np.array([[float(t) for t in row.split(",")] for row in s.split(";")])


def test_attention_closed_forms():
    n = 0
    for line in _golden_lines("rope_attention.txt"):
        name, kv, _ = _kv(line)
        if name != "attend":
            continue
        q = np.array([float(t) for t in kv["q"].split(",")])
        got = O.attend(q, _parse_mat(kv["k"]), _parse_mat(kv["v"]), float(kv["alpha"]))
        want = np.array([float(t) for t in kv["expect"].split(",")])
        assert np.allclose(got, want, rtol=1e-14, atol=1e-14), line
        n += 1
    assert n == 3


def _brute_attend(q, K, V, alpha):
    """Pure-Python softmax-weighted sum without max subtraction."""
    w = [math.exp(alpha * sum(qi * ki for qi, ki in zip(q, k))) for k in K]
    tot = sum(w)
    return [sum(wt * v[d] for wt, v in zip(w, V)) / tot for d in range(len(V[0]))]


def test_attention_brute_force_and_invariants():
    rng = np.random.default_rng(9)
    for L in (1, 2, 15, 16, 17, 40):
        q, K, V = rng.standard_normal(8), rng.standard_normal((L, 8)), rng.standard_normal((L, 8))
        got = O.attend(q, K, V, 0.35)
        assert np.allclose(got, _brute_attend(q.tolist(), K.tolist(), V.tolist(), 0.35), rtol=1e-12)
        if L == 1:
            assert np.array_equal(got, V[0])
        # constant keys average the values
        assert np.allclose(O.attend(q, np.tile(K[:1], (L, 1)), V, 0.35), V.mean(axis=0), rtol=1e-12)
        # permuting keys with their values changes nothing
        p = rng.permutation(L)
        assert np.allclose(O.attend(q, K[p], V[p], 0.35), got, rtol=1e-12)
    # one key with a far larger score dominates
    K = rng.standard_normal((30, 8)) * 0.1
    K[13] = 50 * np.ones(8)
    V = rng.standard_normal((30, 8))
    assert np.allclose(O.attend(np.ones(8), K, V, 1.0), V[13], atol=1e-12)
    # an empty context gives zeros (reading R7)
    assert np.array_equal(O.attend(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0), np.zeros(8))


def _fill(spec, w, lens, n_pages, bt, ring_rows=0, rope_tab=None, seed=0):
    """Append every token of every sequence (oracle only)."""
    pools = {"k": np.zeros(n_pages * O.page_bytes(spec, "k"), np.uint8),
             "v": np.zeros(n_pages * O.page_bytes(spec, "v"), np.uint8)}
    rng = np.random.default_rng(seed)
    ks, vs = [], []
    for b, L in enumerate(lens):
        k = rng.standard_normal((L, spec.n_kv_heads, spec.head_dim)).astype(np.float16)
        v = rng.standard_normal((L, spec.n_kv_heads, spec.head_dim)).astype(np.float16)
        ks.append(k)
        vs.append(v)
        O.append(spec, pools, k, v, np.full(L, b), np.arange(L), bt, ring_rows, rope_tab)
    return pools, ks, vs


def _small_spec(**kw):
    base = dict(n_heads=4, n_kv_heads=2, head_dim=32, page_size=16, k_kind="sym4",
                v_kind="sym4", k_group=16, v_group=32, k_param="f16", v_param="f32",
                act="f16", attn_scale=0.0, rope="normal", rope_base=10000.0)
    base.update(kw)
    return O.Spec(**base)


@pytest.mark.parametrize("kinds", [("sym4", "sym4"), ("sym8", "sym4"), ("affine4", "affine4"), ("f16", "f16"),
                                   ("shimmy4", "shimmy4")])
def test_paged_equals_contiguous(kinds):
    kk, vk = kinds
    par = "bf16" if kk == "affine4" else "f16"
    spec = _small_spec(k_kind=kk, v_kind=vk, k_param=par, v_param=par,
                       rope="neox" if kk == "affine4" else "normal")
    lens = [1, 16, 17, 45, 0]
    maxp = 4
    rope_tab = O.rope_table(spec.head_dim, spec.rope_base, 64)
    order = np.random.default_rng(1).permutation(40)     # shuffled physical pages
    bt = np.full((len(lens), maxp), -1, np.int32)
    k = 0
    for b, L in enumerate(lens):
        for j in range(-(-L // 16)):
            bt[b, j] = order[k]
            k += 1
    pools, ks, vs = _fill(spec, None, lens, 40, bt, rope_tab=rope_tab)
    q = np.random.default_rng(4).standard_normal((len(lens), 4, 32)).astype(np.float16)
    paged = O.decode(spec, q, pools, bt, np.array(lens))
    contig = O.decode_contiguous(spec, q, ks, vs, lens, rope_tab)
    assert np.allclose(paged, contig, rtol=1e-13, atol=1e-13)
    assert np.all(paged[4] == 0)
    # GQA: q heads 0,1 read kv head 0; heads 2,3 read kv head 1
    pools2 = {w: p.copy() for w, p in pools.items()}
    spec_v = O.Spec(**{**spec.__dict__})
    K = O.gather_dequant(spec, "k", pools["k"], bt[3], np.arange(45))
    V = O.gather_dequant(spec, "v", pools2["v"], bt[3], np.arange(45))
    for h in range(4):
        qh = O.rotate_f64(q[3, h].astype(np.float64), 44, 32, spec.rope_base, spec.rope)
        assert np.allclose(paged[3, h], O.attend(qh, K[:, h // 2], V[:, h // 2], spec_v.alpha()))


def test_page_layout_offsets():
    # llama8b-shaped K pool: sub-block = 16 x 64 B codes + 16 x 4 B scales = 1088 B, page = 8 x 1088
    spec = O.Spec(n_heads=32, n_kv_heads=8, head_dim=128, page_size=16, k_kind="sym4",
                  v_kind="sym4", k_group=128, v_group=128, k_param="f32", v_param="f32",
                  act="f16", rope="none")
    oc, op, cb, pb = O._slot_offsets(spec, "k", 3, 5, 2)
    assert (int(oc), int(op), cb, pb) == (3 * 8704 + 2 * 1088 + 5 * 64,
                                          3 * 8704 + 2 * 1088 + 1024 + 5 * 4, 64, 4)
    pools = {"k": np.zeros(5 * 8704, np.uint8), "v": np.zeros(5 * 8704, np.uint8)}
    row = np.zeros((1, 8, 128), np.float32)
    row[0, 2, 0], row[0, 2, 1], row[0, 2, 127] = 7.0, -7.0, 3.5   # scale 1
    bt = np.array([[9, 9, 3, 9]], np.int32)
    O.append(spec, pools, row, row, [0], [2 * 16 + 5], bt)
    base = 3 * 8704 + 2 * 1088
    assert pools["k"][base + 5 * 64] == 0x97              # codes 7 (low) and -7 (high)
    assert pools["k"][base + 5 * 64 + 63] == 0x40         # code 4 (3.5 -> 4) in the high nibble
    assert np.frombuffer(pools["k"][base + 1024 + 20: base + 1024 + 24].tobytes(), "<f4")[0] == 1.0
    sub = pools["k"][base: base + 1088]
    assert np.count_nonzero(sub) == 2 + 2                 # two code bytes; 1.0f has two nonzero bytes
    # the other heads' all-zero rows store the 1e-8 scale floor and zero codes
    other = pools["k"][3 * 8704 + 1088 * 5: 3 * 8704 + 1088 * 6]
    assert np.count_nonzero(other[:1024]) == 0
    assert np.frombuffer(other[1024 + 20: 1024 + 24].tobytes(), "<f4")[0] == np.float32(1e-8)


def test_f16_kv_layout_and_brute_force_attention():
    """The unquantised f16 KV type (reading R8, [Kaiwu] finding 2 "f16+f16"):
    a sub-block is 16 rows of 2 * head_dim bytes, each row the fp16 rounding of
    its elements with no scale; decode equals brute-force softmax attention
    over those fp16 values."""
    spec = O.Spec(n_heads=4, n_kv_heads=2, head_dim=32, page_size=16, k_kind="f16", v_kind="f16",
                  k_group=32, v_group=32, k_param="f32", v_param="f32", act="f32", rope="none")
    assert O.code_bytes("f16", 32) == 64 and O.param_row_bytes("f16", 32, 32, "f32") == 0
    assert O.page_bytes(spec, "k") == 2 * 16 * 64
    rng = np.random.default_rng(7)
    L = 21
    k = rng.standard_normal((L, 2, 32)).astype(np.float32) * 3
    v = rng.standard_normal((L, 2, 32)).astype(np.float32)
    bt = np.array([[4, 1]], np.int32)
    pools = {w: np.zeros(5 * O.page_bytes(spec, w), np.uint8) for w in ("k", "v")}
    O.append(spec, pools, k, v, np.zeros(L, np.int64), np.arange(L), bt)
    # token 17 sits in page bt[0][1] = 1, slot 1, kv head 1
    off = 1 * O.page_bytes(spec, "k") + 1 * 16 * 64 + 1 * 64
    assert pools["k"][off:off + 64].tobytes() == k[17, 1].astype("<f2").tobytes()
    q = rng.standard_normal((1, 4, 32))
    got = O.decode(spec, q, pools, bt, np.array([L]))
    K16 = k.astype(np.float16).astype(np.float64)
    V16 = v.astype(np.float16).astype(np.float64)
    for h in range(4):
        ref = _brute_attend(q[0, h].tolist(), K16[:, h // 2].tolist(), V16[:, h // 2].tolist(),
                            1.0 / np.sqrt(32.0))
        assert np.allclose(got[0, h], ref, rtol=1e-12, atol=1e-12)


def _rotate_closed_form(x, pos, base, mode):
    """The rotation written out from its definition, in pure Python:
    theta_i = base^(-2i/hd), pair i rotated by pos * theta_i; pairs (2i, 2i+1),
    or (i, i + hd/2) for NeoX ([Shimmy] §2.2/§2.3, [Fieldfare] "量化和精度")."""
    hd = len(x)
    out = [float(v) for v in x]
    for i in range(hd // 2):
        a, b = (2 * i, 2 * i + 1) if mode == "normal" else (i, i + hd // 2)
        ang = pos * base ** (-2.0 * i / hd)
        c, s = math.cos(ang), math.sin(ang)
        out[a] = float(x[a]) * c - float(x[b]) * s
        out[b] = float(x[a]) * s + float(x[b]) * c
    return out


@pytest.mark.parametrize("mode", ["normal", "neox"])
def test_rope_positions_against_brute_force(mode):
    """Where the rotation is applied ([Shimmy] §2.3: q and k are rotated;
    [Fieldfare] "KV Cache 的双布局设计": K is rotated before it is cached, V is
    not): key t at its own position t, the decode query at L - 1.  With the
    unquantised f16 kind (reading R8) no code intervenes, so the oracle's
    append + decode must equal brute-force attention over keys rotated by the
    closed form and rounded to fp16 once.  The same brute force with the keys
    one position late, or the query one position late, must differ widely, so a
    slip in either position fails here."""
    hd, base, L = 16, 100.0, 23
    spec = O.Spec(n_heads=4, n_kv_heads=2, head_dim=hd, page_size=16, k_kind="f16", v_kind="f16",
                  k_group=hd, v_group=hd, k_param="f32", v_param="f32", act="f32", rope=mode,
                  rope_base=base)
    rng = np.random.default_rng(21)
    k = rng.standard_normal((L, 2, hd)).astype(np.float32)
    v = rng.standard_normal((L, 2, hd)).astype(np.float32)
    q = rng.standard_normal((1, 4, hd)).astype(np.float32)
    bt = np.array([[3, 0]], np.int32)
    pools = {w: np.zeros(4 * O.page_bytes(spec, w), np.uint8) for w in ("k", "v")}
    O.append(spec, pools, k, v, np.zeros(L, np.int64), np.arange(L), bt, 0, O.rope_table(hd, base, L + 1))
    got = O.decode(spec, q, pools, bt, np.array([L]))
    alpha = 1.0 / math.sqrt(hd)

    def brute(k_shift, q_shift):
        o = np.zeros((4, hd))
        for h in range(4):
            kv = h // 2
            K = [np.float16(_rotate_closed_form(k[t, kv], t + k_shift, base, mode)).astype(np.float64).tolist()
                 for t in range(L)]
            V = [v[t, kv].astype(np.float16).astype(np.float64).tolist() for t in range(L)]
            qr = _rotate_closed_form(q[0, h], L - 1 + q_shift, base, mode)
            o[h] = _brute_attend(qr, K, V, alpha)
        return o

    ref = brute(0, 0)
    scale = np.max(np.abs(ref))
    # fp32 rotation with the fp32 table before the fp16 rounding, against the
    # fp64 closed form: at most a one-ulp fp16 difference in a few elements
    assert np.max(np.abs(got[0] - ref)) <= 1e-3 * scale
    for ks, qs in ((1, 0), (0, 1), (-1, 0), (0, -1)):
        assert np.max(np.abs(brute(ks, qs) - ref)) >= 3e-2 * scale, (ks, qs)


def test_rope_scores_depend_on_relative_position():
    """A rotation pair at positions (p, t) gives the same fp64 score as at
    (p + d, t + d): the scores see only p - t.  Moving the query alone changes
    them."""
    hd, base = 32, 500000.0
    rng = np.random.default_rng(5)
    q, kk = rng.standard_normal(hd), rng.standard_normal(hd)
    for mode in ("normal", "neox"):
        for p, t in ((0, 0), (7, 3), (8191, 100), (65535, 65000)):
            s0 = O.rotate_f64(q, p, hd, base, mode) @ O.rotate_f64(kk, t, hd, base, mode)
            for d in (1, 13, 4096):
                s1 = O.rotate_f64(q, p + d, hd, base, mode) @ O.rotate_f64(kk, t + d, hd, base, mode)
                assert abs(s1 - s0) <= 1e-12 * max(1.0, abs(s0)), (mode, p, t, d)
            s2 = O.rotate_f64(q, p + 1, hd, base, mode) @ O.rotate_f64(kk, t, hd, base, mode)
            assert abs(s2 - s0) > 1e-3, (mode, p, t)


def test_shimmy_codec_hand_worked_and_brute_force():
    """[Shimmy] §3.2 quantize_head_vector (reading R9): scale = max|x| / 7.5,
    code = clamp(round(x / scale), -8, 7) rounding half away from zero, stored
    as code + 8 with the even element in the low nibble."""
    x = np.array([[7.5, -7.5, 2.5, -2.5, 0.5, 3.75, -0.5, 1.25]], np.float32)
    c, s, b = O.quantize("shimmy4", x, 8, "f32")
    assert b is None and s[0, 0] == 1.0
    # 7.5 rounds to 8 and clamps to 7; ties 2.5 / -2.5 / 0.5 / -0.5 go away from zero
    assert c.tolist() == [[7, -8, 3, -3, 1, 4, -1, 1]]
    assert O.pack_codes("shimmy4", c).tolist() == [[0x0F, 0x5B, 0xC9, 0x97]]
    assert O.unpack_codes("shimmy4", O.pack_codes("shimmy4", c)).tolist() == c.tolist()
    assert O.bytes_per_token_head("shimmy4", 128, 128, "f32") == 68      # 0.53 B per element, as the page says
    # brute force: the nearest integer in [-8, 7], a tie to the one farther from zero
    rng = np.random.default_rng(3)
    xs = rng.standard_normal((64, 32)).astype(np.float32) * rng.uniform(0.1, 5, (64, 1)).astype(np.float32)
    xs[::7, 5] = 0.0
    codes, scales, _ = O.quantize("shimmy4", xs, 32, "f32")
    for r in range(xs.shape[0]):
        sc = np.float32(np.max(np.abs(xs[r])) / np.float32(7.5))
        assert scales[r, 0] == sc
        for j in range(32):
            y = float(np.float32(xs[r, j] / sc))
            best = min(range(-8, 8), key=lambda k: (abs(y - k), -abs(k)))
            assert codes[r, j] == best
            assert abs(xs[r, j] - codes[r, j] * sc) <= sc / 2 + 1e-6 * sc   # round-trip bound
    # an all-zero group: scale 0, codes 0 (nibbles 8)
    z, sz, _ = O.quantize("shimmy4", np.zeros((1, 8), np.float32), 8, "f32")
    assert sz[0, 0] == 0 and z.tolist() == [[0] * 8]
    assert O.pack_codes("shimmy4", z).tolist() == [[0x88] * 4]


def test_ring_equals_explicit_window():
    # [Fieldfare] "KV Cache 的双布局设计": 1152-row ring, 1024-token window
    spec = _small_spec(n_heads=2, n_kv_heads=1, head_dim=16, k_group=16, v_group=16,
                       rope="neox", rope_base=1e4)
    R, W = 1152, 1024
    rope_tab = O.rope_table(16, 1e4, 5000)
    assert list(O.attended_positions(1025, W)[[0, -1]]) == [1, 1024]
    assert list(O.attended_positions(700, W)[[0, -1]]) == [0, 699]
    for L in (1000, 1024, 1025, 1152, 1153, 5000):
        bt = np.arange(R // 16, dtype=np.int32)[None, ::-1].copy()
        pools, ks, vs = _fill(spec, None, [L], R // 16, bt, ring_rows=R, rope_tab=rope_tab, seed=L)
        q = np.random.default_rng(L).standard_normal((1, 2, 16)).astype(np.float16)
        ring = O.decode(spec, q, pools, bt, np.array([L]), window=W, ring_rows=R)
        expl = O.decode_contiguous(spec, q, ks, vs, [L], rope_tab, window=W)
        assert np.allclose(ring, expl, rtol=1e-13, atol=1e-13), L


def test_sequence_isolation():
    # [airllm] §5.4: sequences sharing one pool must not overwrite each other.
    spec = _small_spec()
    lens = [20, 33]
    bt = np.array([[5, 0, -1], [2, 7, 1]], np.int32)
    rope_tab = O.rope_table(32, 1e4, 64)
    pools, ks, vs = _fill(spec, None, lens, 8, bt, rope_tab=rope_tab)
    q = np.random.default_rng(0).standard_normal((2, 4, 32)).astype(np.float16)
    before = O.decode(spec, q, pools, bt, np.array(lens))
    extra = np.random.default_rng(1).standard_normal((1, 2, 32)).astype(np.float16)
    O.append(spec, pools, extra, extra, [0], [20], bt, 0, rope_tab)     # grow sequence 0
    after = O.decode(spec, q, pools, bt, np.array([21, 33]))
    assert np.array_equal(before[1], after[1])
    assert not np.allclose(before[0], after[0])


def test_row_rel_error_rule():
    ref = np.array([[1.0, -0.5, 1e-9, 0.0]])
    assert O.row_rel_error(ref, ref)[0] == 0
    got = ref + np.array([[1e-3, 0, 0, 0]])
    assert math.isclose(O.row_rel_error(got, ref)[0], 1e-3)
    got = ref + np.array([[0, 0, 1e-6, 0]])                # near-zero element uses the row floor (0.1 %)
    assert math.isclose(O.row_rel_error(got, ref)[0], 1e-3)
    assert math.isclose(O.row_rel_error(got, ref, floor=1e-2)[0], 1e-4)   # an explicit wider floor
    got = ref + np.array([[0, 2e-4, 0, 0]])                # 0.5 is above the floor: relative to itself
    assert math.isclose(O.row_rel_error(got, ref)[0], 4e-4)
    assert math.isclose(O.row_norm_error(got, ref)[0], 2e-4)
