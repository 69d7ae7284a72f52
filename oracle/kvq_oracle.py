"""CPU oracle for the quantized paged KV decode path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import
or run this module.  The product -- the ``kvq`` C-ABI library and its Python
binding -- never imports it, and this module imports nothing of the product.

Plain, slow, obviously-correct numpy.  Each function cites the passage of the
source pages it restates.  The four pages are referred to as:

* [Shimmy]  "Shimmy 深度解剖：Airframe 引擎与 TurboShimmy INT4 KV"
            (chenxutan.com/d/5228)
* [Fieldfare] the TurboFieldfare post on cnblogs (32bin/p/23195374)
* [airllm]  the airllm light-weight inference post (cf-1.com/news/5708464)
* [Kaiwu]   "我做了个工具让 8GB 显卡跑 30B 模型从 3 tok/s 提到 21 tok/s"
            (blog.xiaohack.org/244516)

Precision: the codec (RoPE on K, group amax/min-max, scale, division,
rounding) is evaluated in IEEE fp32 with one rounding per operation, exactly as
the numeric spec fixes it, because a quantised code is an integer decided by
floating point and both sides must decide it in the same precision.  Everything
after the codes (dequantisation, q rotation, scores, softmax, P.V) is fp64.

Readings taken where the pages are silent:
  R1  round-half-to-even for x/scale in the symmetric and affine kinds
      (torch.round in [airllm] §4.2 rounds half to even); the Rust ``round()``
      of [Shimmy] §3.2 rounds half away from zero and serves only its own
      codec, the "shimmy4" kind (R9).
  R2  symmetric scale = max|x| / 7 with clamp_min 1e-8 ([airllm] §4.2); for
      fp16-stored scales the floor is 2^-14 (1e-8 underflows in fp16); the
      floor is applied in fp32 before rounding to the stored type.
  R3  affine 4-bit ([Fieldfare] "量化和精度" names only "4-bit, group 64, bf16
      scale + bf16 bias"): scale = bf16(fl32(max-min)/15), bias = bf16(min),
      code = clamp(rne((x - bias)/scale), 0, 15), x^ = scale*code + bias; a
      zero scale gives code 0.
  R4  RoPE: theta_i = base^(-2i/hd); adjacent pairs (2i, 2i+1) unless NeoX
      (i, i+hd/2) is stated ([Fieldfare] "量化和精度"); position = absolute
      token index from 0; the decode query sits at position L-1.
  R5  GQA: q head h reads kv head h // (n_heads / n_kv_heads).
  R6  attention scale defaults to 1/sqrt(head_dim) ([Shimmy] §2.3 comment);
      the shader line that divides by head_dim is read as garbled.
  R7  an empty context (L = 0) yields a zero output row.
  R8  the unquantised "f16" KV type of [Kaiwu] finding 2 (f16 K + f16 V) stores
      each element of the (rotated, fp32) row rounded once to fp16 (nearest,
      ties to even), with no scale; its value is read back exactly.
  R9  the "shimmy4" kind is the codec of [Shimmy] §3.2 as written:
      scale = fl32(max|x| / 7.5) (stored in the param type), code =
      clamp(round(fl32(x / scale)), -8, 7) with round half away from zero (the
      Rust ``round`` it uses), nibble = code + 8 (offset binary, even element
      low), x^ = (nibble - 8) * scale; a zero scale gives code 0.  Groups of
      any size (the page uses one group per head vector).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

PARAM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
KV_KINDS = ("sym4", "sym8", "affine4", "f16", "f32", "shimmy4")


# ---------------------------------------------------------------------------
# Description of one attention layer's cache


@dataclass(frozen=True)
class Spec:
    n_heads: int
    n_kv_heads: int
    head_dim: int
    page_size: int
    k_kind: str
    v_kind: str
    k_group: int
    v_group: int
    k_param: str
    v_param: str
    act: str = "f16"
    attn_scale: float = 0.0
    rope: str = "normal"          # "none" | "normal" | "neox"
    rope_base: float = 10000.0

    @staticmethod
    def from_workload(w: dict) -> "Spec":
        return Spec(**{f: w[f] for f in Spec.__dataclass_fields__})

    @property
    def group_size(self) -> int:
        return self.n_heads // self.n_kv_heads

    def alpha(self) -> float:
        """Score scale; R6."""
        if self.attn_scale > 0.0:
            return float(self.attn_scale)
        return 1.0 / math.sqrt(self.head_dim)


# ---------------------------------------------------------------------------
# Cache sizing -- [Kaiwu] finding 2 (KV_MB = 2 x layers x kv_heads x head_dim x
# ctx x bytes / 1024^2), its "GQA 架构识别" note (kv_heads, not heads), and
# [Shimmy] §3.1 / §3.2 (16 MB per layer; 0.5 B per INT4 element plus one
# 4-byte scale per head vector).


def bytes_per_token_head(kind: str, head_dim: int, group: int, param: str) -> int:
    """Stored bytes of one token's vector for one kv head."""
    if kind == "f16":
        return 2 * head_dim
    if kind == "f32":
        return 4 * head_dim
    bits = 8 if kind == "sym8" else 4
    n_params = 2 if kind == "affine4" else 1
    return head_dim * bits // 8 + (head_dim // group) * n_params * PARAM_BYTES[param]


def cache_bytes(n_layers: int, n_kv_heads: int, head_dim: int, ctx: int,
                page_size: int, k_kind: str, v_kind: str, k_group: int,
                v_group: int, k_param: str, v_param: str) -> int:
    """K plus V bytes for ``n_layers`` layers holding ``ctx`` tokens.

    The context is rounded up to whole pages ([airllm] §2.3: the pool grows by
    whole blocks).  With equal K/V kinds and ctx a multiple of the page this is
    2 x layers x kv_heads x ctx x bytes_per_token_head.
    """
    ctx_pad = -(-ctx // page_size) * page_size
    per = (bytes_per_token_head(k_kind, head_dim, k_group, k_param)
           + bytes_per_token_head(v_kind, head_dim, v_group, v_param))
    return n_layers * n_kv_heads * ctx_pad * per


# ---------------------------------------------------------------------------
# Rounding to the stored parameter type


def bf16_round(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 -> fp32, round to nearest, ties to even (finite inputs)."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def round_param(x32: np.ndarray, param: str) -> np.ndarray:
    x32 = np.asarray(x32, dtype=np.float32)
    if param == "f32":
        return x32.copy()
    if param == "f16":
        return x32.astype(np.float16).astype(np.float32)
    if param == "bf16":
        return bf16_round(x32)
    raise ValueError(param)


def scale_floor(param: str) -> np.float32:
    """R2: smallest stored symmetric scale."""
    return np.float32(2.0 ** -14) if param == "f16" else np.float32(1e-8)


# ---------------------------------------------------------------------------
# Group-wise quantisation -- [airllm] §2.1 (group of contiguous elements) and
# §4.2 (group_quantize: scale = amax / (2^(bits-1) - 1), clamp_min 1e-8,
# round(t / scale) clamped to +-(2^(bits-1) - 1)); [Shimmy] §3.2 (one vector
# per kv head, codes stored with a scale); [Fieldfare] "量化和精度" (affine
# 4-bit, group 64, bf16 scale and bias).


def quantize_sym(x: np.ndarray, group: int, bits: int, param: str):
    """Symmetric codes of the last axis, in fp32 (readings R1, R2).

    Returns (codes int8 [..., hd], scales fp32 [..., hd // group]); the scales
    hold exactly the values stored in the ``param`` type.
    """
    x = np.asarray(x, dtype=np.float32)
    lead, hd = x.shape[:-1], x.shape[-1]
    qmax = np.float32(2 ** (bits - 1) - 1)
    xg = x.reshape(*lead, hd // group, group)
    amax = np.max(np.abs(xg), axis=-1)
    s = (amax / qmax).astype(np.float32)
    s = np.maximum(s, scale_floor(param)).astype(np.float32)
    s = round_param(s, param)
    y = (xg / s[..., None]).astype(np.float32)
    c = np.clip(np.rint(y), -qmax, qmax).astype(np.int8)
    return c.reshape(*lead, hd), s


def quantize_affine(x: np.ndarray, group: int, param: str):
    """Affine 4-bit codes of the last axis, in fp32 (reading R3).

    Returns (codes uint8 in [0, 15], scales fp32, biases fp32).
    """
    x = np.asarray(x, dtype=np.float32)
    lead, hd = x.shape[:-1], x.shape[-1]
    xg = x.reshape(*lead, hd // group, group)
    mn = np.min(xg, axis=-1)
    mx = np.max(xg, axis=-1)
    span = (mx - mn).astype(np.float32)
    s = round_param((span / np.float32(15.0)).astype(np.float32), param)
    b = round_param(mn, param)
    d = (xg - b[..., None]).astype(np.float32)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    y = (d / safe[..., None]).astype(np.float32)
    c = np.clip(np.rint(y), 0.0, 15.0)
    c = np.where((s == 0)[..., None], 0.0, c).astype(np.uint8)
    return c.reshape(*lead, hd), s, b


def quantize_shimmy(x: np.ndarray, group: int, param: str):
    """[Shimmy] §3.2 quantize_head_vector per group (reading R9).

    Returns (codes int8 in [-8, 7], scales fp32).
    """
    x = np.asarray(x, dtype=np.float32)
    lead, hd = x.shape[:-1], x.shape[-1]
    xg = x.reshape(*lead, hd // group, group)
    amax = np.max(np.abs(xg), axis=-1)
    s = round_param((amax / np.float32(7.5)).astype(np.float32), param)
    safe = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
    y = (xg / safe[..., None]).astype(np.float32).astype(np.float64)
    r = np.sign(y) * np.floor(np.abs(y) + 0.5)          # half away from zero, exact in fp64
    c = np.clip(r, -8, 7)
    c = np.where((s == 0)[..., None], 0, c).astype(np.int8)
    return c.reshape(*lead, hd), s


def quantize(kind: str, x: np.ndarray, group: int, param: str):
    """(codes, scales, biases-or-None) for any stored kind; "f16" (R8) keeps
    the fp16-rounded values as its codes and has no scales."""
    if kind == "f16":
        return np.asarray(x, dtype=np.float32).astype(np.float16), None, None
    if kind == "sym4":
        c, s = quantize_sym(x, group, 4, param)
        return c, s, None
    if kind == "sym8":
        c, s = quantize_sym(x, group, 8, param)
        return c, s, None
    if kind == "affine4":
        return quantize_affine(x, group, param)
    if kind == "shimmy4":
        c, s = quantize_shimmy(x, group, param)
        return c, s, None
    raise ValueError(kind)


def dequantize(codes: np.ndarray, scales: np.ndarray, biases, group: int) -> np.ndarray:
    """x^ = scale * code (+ bias), in fp64; an unscaled kind (no scales) is its codes."""
    c = np.asarray(codes).astype(np.float64)
    if scales is None:
        return c
    lead, hd = c.shape[:-1], c.shape[-1]
    cg = c.reshape(*lead, hd // group, group)
    out = cg * np.asarray(scales, dtype=np.float64)[..., None]
    if biases is not None:
        out = out + np.asarray(biases, dtype=np.float64)[..., None]
    return out.reshape(*lead, hd)


# ---------------------------------------------------------------------------
# RoPE -- [Shimmy] §2.2 (rope_freq_base) and §2.3 (rotation applied to query
# and key); [Fieldfare] "KV Cache 的双布局设计" (K is rotated before it is
# cached, V is not) and "量化和精度" (NeoX pairing for Gemma 4).  Reading R4.


def rope_theta(head_dim: int, base: float) -> list[float]:
    return [math.pow(base, -2.0 * i / head_dim) for i in range(head_dim // 2)]


def rope_table(head_dim: int, base: float, max_pos: int) -> np.ndarray:
    """fp32 [max_pos][head_dim/2][2] of (cos, sin) of pos*theta_i (fp64 math)."""
    th = rope_theta(head_dim, base)
    out = np.empty((max_pos, head_dim // 2, 2), dtype=np.float32)
    for p in range(max_pos):
        ang = [p * t for t in th]
        out[p, :, 0] = [math.cos(a) for a in ang]
        out[p, :, 1] = [math.sin(a) for a in ang]
    return out


def rope_pairs(head_dim: int, mode: str):
    half = head_dim // 2
    i = np.arange(half)
    if mode == "normal":
        return 2 * i, 2 * i + 1
    if mode == "neox":
        return i, i + half
    raise ValueError(mode)


def rotate_f32(x32: np.ndarray, cs: np.ndarray, mode: str) -> np.ndarray:
    """Rotate the last axis in fp32, one rounding per multiply and add.

    ``cs`` is a (cos, sin) table slice broadcastable to [..., hd/2, 2].
    x0' = x0*c - x1*s ; x1' = x0*s + x1*c.
    """
    x = np.asarray(x32, dtype=np.float32)
    if mode == "none":
        return x.copy()
    i0, i1 = rope_pairs(x.shape[-1], mode)
    c = cs[..., 0].astype(np.float32)
    s = cs[..., 1].astype(np.float32)
    x0, x1 = x[..., i0], x[..., i1]
    out = np.empty_like(x)
    out[..., i0] = (x0 * c).astype(np.float32) - (x1 * s).astype(np.float32)
    out[..., i1] = (x0 * s).astype(np.float32) + (x1 * c).astype(np.float32)
    return out


def rotate_f64(x: np.ndarray, pos: int, head_dim: int, base: float, mode: str) -> np.ndarray:
    """Rotate a query vector in fp64 at one position."""
    x = np.asarray(x, dtype=np.float64)
    if mode == "none":
        return x.copy()
    th = np.array(rope_theta(head_dim, base), dtype=np.float64)
    ang = np.array([pos * t for t in th], dtype=np.float64)
    c = np.array([math.cos(a) for a in ang])
    s = np.array([math.sin(a) for a in ang])
    i0, i1 = rope_pairs(head_dim, mode)
    out = np.empty_like(x)
    out[..., i0] = x[..., i0] * c - x[..., i1] * s
    out[..., i1] = x[..., i0] * s + x[..., i1] * c
    return out


# ---------------------------------------------------------------------------
# Page layout (the boundary's documented storage format) -- [airllm] §2.3
# (free-block pool, whole-block growth, an offset index inside each block) and
# §2.2 (the packing layout decides coalescing).  Two 4-bit codes per byte, low
# nibble = even element ([airllm] §4.2 packs quant[:, 0::2] low and quant[:,
# 1::2] high, two's-complement nibbles via & 0x0F).
#
#   pool   = n_pages x page
#   page   = n_kv_heads x sub-block
#   sub    = codes[page_size][code_bytes] , params[page_size][param_row_bytes]
#   params = per group: scale (symmetric) or scale, bias (affine)


def code_bytes(kind: str, head_dim: int) -> int:
    if kind == "f16":
        return 2 * head_dim
    return head_dim if kind == "sym8" else head_dim // 2


def param_row_bytes(kind: str, head_dim: int, group: int, param: str) -> int:
    if kind == "f16":
        return 0
    n_params = 2 if kind == "affine4" else 1
    return (head_dim // group) * n_params * PARAM_BYTES[param]


def sub_block_bytes(kind, head_dim, group, param, page_size) -> int:
    return page_size * (code_bytes(kind, head_dim)
                        + param_row_bytes(kind, head_dim, group, param))


def page_bytes(spec: Spec, which: str) -> int:
    kind, grp, par = _kv(spec, which)
    return spec.n_kv_heads * sub_block_bytes(kind, spec.head_dim, grp, par,
                                             spec.page_size)


def _kv(spec: Spec, which: str):
    if which == "k":
        return spec.k_kind, spec.k_group, spec.k_param
    return spec.v_kind, spec.v_group, spec.v_param


def pack_codes(kind: str, codes: np.ndarray) -> np.ndarray:
    """codes [..., hd] -> bytes [..., code_bytes]."""
    if kind == "f16":
        c = np.ascontiguousarray(codes, dtype="<f2")
        return c.view(np.uint8).reshape(*c.shape[:-1], 2 * c.shape[-1])
    if kind == "sym8":
        return np.asarray(codes, dtype=np.int8).view(np.uint8)
    if kind == "shimmy4":   # offset-binary nibbles: code + 8
        c = (np.asarray(codes).astype(np.int16) + 8) & 0xF
        return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)
    c = np.asarray(codes).astype(np.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_codes(kind: str, raw: np.ndarray) -> np.ndarray:
    """bytes [..., code_bytes] -> codes [..., hd] (int16)."""
    raw = np.asarray(raw, dtype=np.uint8)
    if kind == "f16":
        return np.ascontiguousarray(raw).view("<f2")
    if kind == "sym8":
        return raw.view(np.int8).astype(np.int16)
    lo = (raw & 0xF).astype(np.int16)
    hi = (raw >> 4).astype(np.int16)
    if kind == "sym4":
        lo = (lo ^ 8) - 8
        hi = (hi ^ 8) - 8
    if kind == "shimmy4":
        lo = lo - 8
        hi = hi - 8
    out = np.empty(raw.shape[:-1] + (raw.shape[-1] * 2,), dtype=np.int16)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _param_to_bytes(vals32: np.ndarray, param: str) -> np.ndarray:
    v = np.ascontiguousarray(vals32, dtype=np.float32)
    if param == "f32":
        b = v.astype("<f4")
    elif param == "f16":
        b = v.astype("<f2")
    else:  # bf16: the top half of the (already bf16-exact) fp32 pattern
        b = (v.view("<u4") >> 16).astype("<u2")
    return b.view(np.uint8).reshape(*v.shape[:-1], v.shape[-1] * PARAM_BYTES[param])


def _bytes_to_param(raw: np.ndarray, param: str) -> np.ndarray:
    raw = np.ascontiguousarray(raw, dtype=np.uint8)
    if param == "f32":
        return raw.view("<f4").astype(np.float32)
    if param == "f16":
        return raw.view("<f2").astype(np.float32)
    u = raw.view("<u2").astype(np.uint32) << 16
    return u.astype("<u4").view(np.float32)


def _params_row(kind, scales, biases, param):
    if scales is None:   # an unscaled kind: no parameter bytes
        return np.zeros(0, np.uint8)
    if kind == "affine4":
        inter = np.stack([scales, biases], axis=-1).reshape(
            *scales.shape[:-1], 2 * scales.shape[-1])
        return _param_to_bytes(inter, param)
    return _param_to_bytes(scales, param)


def _slot_offsets(spec, which, page_ids, slots, heads):
    """Byte offsets of (codes, params) of given (page, slot, kv head)."""
    kind, grp, par = _kv(spec, which)
    cb = code_bytes(kind, spec.head_dim)
    pb = param_row_bytes(kind, spec.head_dim, grp, par)
    sub = spec.page_size * (cb + pb)
    base = (np.asarray(page_ids, np.int64) * page_bytes(spec, which)
            + np.asarray(heads, np.int64) * sub)
    slots = np.asarray(slots, np.int64)
    return base + slots * cb, base + spec.page_size * cb + slots * pb, cb, pb


def token_location(block_table_row: np.ndarray, pos, page_size: int, ring_rows: int):
    """(page id, slot) of absolute token positions; a ring maps pos -> pos mod R.

    [Fieldfare] "KV Cache 的双布局设计": the window layer keeps its K/V in a
    1152-row ring and overwrites rows that left the window; the global layer
    is append-only.
    """
    pos = np.asarray(pos, np.int64)
    row = pos % ring_rows if ring_rows else pos
    return np.asarray(block_table_row)[row // page_size], row % page_size


# ---------------------------------------------------------------------------
# Quantise-on-append


def quantize_rows(spec: Spec, which: str, rows: np.ndarray, pos: np.ndarray,
                  rope_tab: np.ndarray | None):
    """Codes and params of new rows [n][n_kv_heads][hd] at positions ``pos``.

    K is rotated (fp32) at its own position before quantisation; V is not.
    """
    kind, grp, par = _kv(spec, which)
    x = np.asarray(rows).astype(np.float32)
    if which == "k" and spec.rope != "none":
        x = rotate_f32(x, rope_tab[np.asarray(pos)][:, None, :, :], spec.rope)
    return quantize(kind, x, grp, par)


def append(spec: Spec, pools: dict, k_rows: np.ndarray, v_rows: np.ndarray,
           seq_ids: np.ndarray, pos: np.ndarray, block_table: np.ndarray,
           ring_rows: int = 0, rope_tab: np.ndarray | None = None) -> None:
    """Write rows i (of sequence seq_ids[i], position pos[i]) into the pools.

    ``pools`` maps "k"/"v" to flat uint8 arrays in the page layout above.
    """
    seq_ids = np.asarray(seq_ids, np.int64)
    pos = np.asarray(pos, np.int64)
    n, hkv = len(pos), spec.n_kv_heads
    pages = np.empty(n, np.int64)
    slots = np.empty(n, np.int64)
    for i in range(n):
        pages[i], slots[i] = token_location(block_table[seq_ids[i]], pos[i],
                                            spec.page_size, ring_rows)
    heads = np.broadcast_to(np.arange(hkv)[None, :], (n, hkv))
    for which, rows in (("k", k_rows), ("v", v_rows)):
        kind = _kv(spec, which)[0]
        codes, scales, biases = quantize_rows(spec, which, rows, pos, rope_tab)
        oc, op, cb, pb = _slot_offsets(spec, which, pages[:, None], slots[:, None], heads)
        pool = pools[which]
        pool[oc[..., None] + np.arange(cb)] = pack_codes(kind, codes)
        pool[op[..., None] + np.arange(pb)] = _params_row(kind, scales, biases, _kv(spec, which)[2])


def read_tokens(spec: Spec, which: str, pool: np.ndarray, block_table_row,
                positions, ring_rows: int = 0):
    """(codes, scales, biases) of the given positions: [T][n_kv_heads][...]."""
    kind, grp, par = _kv(spec, which)
    pg, sl = token_location(block_table_row, positions, spec.page_size, ring_rows)
    heads = np.arange(spec.n_kv_heads)[None, :]
    oc, op, cb, pb = _slot_offsets(spec, which, pg[:, None], sl[:, None], heads)
    codes = unpack_codes(kind, pool[oc[..., None] + np.arange(cb)])
    if pb == 0:
        return codes, None, None
    prm = _bytes_to_param(pool[op[..., None] + np.arange(pb)], par)
    if kind == "affine4":
        return codes, prm[..., 0::2], prm[..., 1::2]
    return codes, prm, None


def gather_dequant(spec: Spec, which: str, pool, block_table_row, positions,
                   ring_rows: int = 0) -> np.ndarray:
    """fp64 K^ or V^ of the given positions: [T][n_kv_heads][hd]."""
    grp = _kv(spec, which)[1]
    codes, s, b = read_tokens(spec, which, pool, block_table_row, positions, ring_rows)
    return dequantize(codes, s, b, grp)


# ---------------------------------------------------------------------------
# Decode attention -- the method's softmax(q K^T * s) V read through the block
# table ([airllm] §2.3: queries may span blocks) over fp64 values
# ([airllm] §3.4: keep softmax out of fp16).


def attend(q: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: float) -> np.ndarray:
    """o = softmax(alpha * K q) V for one query (fp64); empty K gives zeros."""
    if k.shape[0] == 0:
        return np.zeros(v.shape[-1], dtype=np.float64)
    s = alpha * (np.asarray(k, np.float64) @ np.asarray(q, np.float64))
    s = s - np.max(s)
    p = np.exp(s)
    return (p @ np.asarray(v, np.float64)) / np.sum(p)


def attended_positions(L: int, window: int) -> np.ndarray:
    lo = max(0, L - window) if window else 0
    return np.arange(lo, L, dtype=np.int64)


def decode(spec: Spec, q: np.ndarray, pools: dict, block_table: np.ndarray,
           seq_lens: np.ndarray, window: int = 0, ring_rows: int = 0,
           seqs=None) -> np.ndarray:
    """Decode attention for each sequence b: fp64 [B][n_heads][hd].

    Query head h of sequence b sits at position L_b - 1 and attends positions
    [max(0, L_b - window), L_b) (all of [0, L_b) when window == 0).  ``seqs``
    restricts the work to some sequences (other rows are left as NaN).
    """
    q = np.asarray(q)
    B = q.shape[0]
    out = np.full((B, spec.n_heads, spec.head_dim), np.nan, dtype=np.float64)
    G = spec.group_size
    for b in (range(B) if seqs is None else seqs):
        L = int(seq_lens[b])
        t = attended_positions(L, window)
        K = gather_dequant(spec, "k", pools["k"], block_table[b], t, ring_rows)
        V = gather_dequant(spec, "v", pools["v"], block_table[b], t, ring_rows)
        for h in range(spec.n_heads):
            qh = q[b, h].astype(np.float64)
            if L > 0:
                qh = rotate_f64(qh, L - 1, spec.head_dim, spec.rope_base, spec.rope)
            out[b, h] = attend(qh, K[:, h // G], V[:, h // G], spec.alpha())
    return out


def row_norm_error(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per (b, h) row: max_i |got_i - ref_i| / max_i |ref_i| (normwise)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.max(np.abs(ref), axis=-1)
    return np.max(np.abs(got - ref), axis=-1) / np.where(den == 0, 1.0, den)


def decode_contiguous(spec: Spec, q: np.ndarray, k_rows: list, v_rows: list,
                      seq_lens, rope_tab, window: int = 0) -> np.ndarray:
    """Same result computed without pages: quantise each sequence's rows in
    order and attend over them directly (used to pin paged == contiguous)."""
    B = q.shape[0]
    G = spec.group_size
    out = np.zeros((B, spec.n_heads, spec.head_dim), dtype=np.float64)
    for b in range(B):
        L = int(seq_lens[b])
        t = attended_positions(L, window)
        kc, ks, kb = quantize_rows(spec, "k", k_rows[b][t], t, rope_tab)
        vc, vs, vb = quantize_rows(spec, "v", v_rows[b][t], t, rope_tab)
        K = dequantize(kc, ks, kb, spec.k_group)
        V = dequantize(vc, vs, vb, spec.v_group)
        for h in range(spec.n_heads):
            qh = q[b, h].astype(np.float64)
            if L > 0:
                qh = rotate_f64(qh, L - 1, spec.head_dim, spec.rope_base, spec.rope)
            out[b, h] = attend(qh, K[:, h // G], V[:, h // G], spec.alpha())
    return out


# ---------------------------------------------------------------------------
# Comparison rule for fp outputs


def row_rel_error(got: np.ndarray, ref: np.ndarray, floor: float = 1e-3) -> np.ndarray:
    """Per (b, h) row: max_i |got_i - ref_i| / max(|ref_i|, floor * max|ref_row|).

    Reading of "max relative error" on the output: elements within 1/floor of
    the row's largest magnitude are compared relatively; smaller ones against
    floor times that magnitude, since their own relative error is
    ill-conditioned.  The default floor is 0.1 %.  A caller whose scores carry
    a larger absolute fp32 error (a large attention scale) passes a larger
    floor explicitly.
    """
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rmax = np.max(np.abs(ref), axis=-1, keepdims=True)
    den = np.maximum(np.abs(ref), floor * rmax)
    den = np.where(den == 0, 1.0, den)
    return np.max(np.abs(got - ref) / den, axis=-1)
