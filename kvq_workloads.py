"""Seeded synthetic inputs for the quantized paged KV decode path.

This module is shared by the tests, the bench and the CPU oracle's callers. It
holds shapes and random numbers only: no quantisation, rotation, paging or
attention arithmetic lives here, so neither side of a parity check can borrow
the other's method through it.

Workloads (shapes follow the pages' problem statements; every value is drawn
from a seeded numpy ``Generator``):

* ``tiny``     -- 1 sequence, 4 q / 2 kv heads, head_dim 64, ctx 256, page 16,
                  symmetric INT4 K/V with group 64 and fp32 scales, fp32
                  activations ~N(0,1), RoPE base 1e4 (adjacent pairs).
* ``llama8b``  -- Llama-3.1-8B-shaped layer: batch 1, 32 q / 8 kv heads,
                  head_dim 128, ctx 8192, fp16 activations ~N(0,1), symmetric
                  INT4 K/V group 128 with fp32 scales, RoPE base 5e5.
* ``contbatch``-- continuous batch: 64 sequences, lengths uniform in
                  [512, 32768], otherwise as ``llama8b``; pages come from one
                  shared pool whose free list is shuffled.
* ``gemma_mix``-- sliding + global mix: 16 q / 8 kv heads, head_dim 256,
                  affine 4-bit group 64 with bf16 scale and bias, attention
                  scale 1.0, NeoX RoPE (base 1e4 is a reading), ctx 16384; the
                  window layer keeps a 1152-row ring and attends 1024 tokens,
                  the global layer is append-only.
* ``long_mixed``-- batch 4, 32 q / 4 kv heads, head_dim 128, ctx 65536, fp16 q;
                  K symmetric INT8 group 32 and V symmetric INT4 group 32, both
                  with fp16 scales; K/V ~N(0,1) with a seeded 1 % of elements
                  multiplied by 8.
* ``llama8b_f16``, ``long_f16`` -- the ``llama8b`` and ``long_mixed`` shapes
                  with unquantised f16 K and V (the "f16+f16" KV type the
                  pages compare the quantised ones with).
* ``llama8b_shimmy``, ``long_shimmy`` -- the ``llama8b`` and ``long_mixed``
                  shapes with the /7.5 offset-8 4-bit codec of the Shimmy post
                  ("shimmy4"), one fp32 scale per 128-element head vector.
"""
from __future__ import annotations

import numpy as np

# Plain descriptions of each workload.  Strings name the codec kinds:
#   "sym4"  symmetric 4-bit, "sym8" symmetric 8-bit, "affine4" affine 4-bit,
#   "f16"   unquantised f16, "shimmy4" the /7.5 offset-8 4-bit codec.
WORKLOADS: dict[str, dict] = {
    "tiny": dict(
        index=0, batch=1, n_heads=4, n_kv_heads=2, head_dim=64, ctx=256,
        page_size=16, k_kind="sym4", v_kind="sym4", k_group=64, v_group=64,
        k_param="f32", v_param="f32", act="f32", attn_scale=0.0,
        rope="normal", rope_base=10000.0, outlier_frac=0.0,
        window=0, ring_rows=0),
    "llama8b": dict(
        index=1, batch=1, n_heads=32, n_kv_heads=8, head_dim=128, ctx=8192,
        page_size=16, k_kind="sym4", v_kind="sym4", k_group=128, v_group=128,
        k_param="f32", v_param="f32", act="f16", attn_scale=0.0,
        rope="normal", rope_base=500000.0, outlier_frac=0.0,
        window=0, ring_rows=0, n_layers=32),
    "contbatch": dict(
        index=2, batch=64, n_heads=32, n_kv_heads=8, head_dim=128, ctx=32768,
        min_len=512, page_size=16, k_kind="sym4", v_kind="sym4",
        k_group=128, v_group=128, k_param="f32", v_param="f32", act="f16",
        attn_scale=0.0, rope="normal", rope_base=500000.0, outlier_frac=0.0,
        window=0, ring_rows=0, shuffle_pages=True),
    "gemma_mix": dict(
        index=3, batch=1, n_heads=16, n_kv_heads=8, head_dim=256, ctx=16384,
        page_size=16, k_kind="affine4", v_kind="affine4", k_group=64,
        v_group=64, k_param="bf16", v_param="bf16", act="f16",
        attn_scale=1.0, rope="neox", rope_base=10000.0, outlier_frac=0.0,
        window=1024, ring_rows=1152),
    "long_mixed": dict(
        index=4, batch=4, n_heads=32, n_kv_heads=4, head_dim=128, ctx=65536,
        page_size=16, k_kind="sym8", v_kind="sym4", k_group=32, v_group=32,
        k_param="f16", v_param="f16", act="f16", attn_scale=0.0,
        rope="normal", rope_base=500000.0, outlier_frac=0.01,
        window=0, ring_rows=0),
}

WORKLOADS["llama8b_f16"] = dict(WORKLOADS["llama8b"], index=5, k_kind="f16", v_kind="f16")
WORKLOADS["llama8b_shimmy"] = dict(WORKLOADS["llama8b"], index=7, k_kind="shimmy4", v_kind="shimmy4")
WORKLOADS["long_f16"] = dict(WORKLOADS["long_mixed"], index=6, k_kind="f16", v_kind="f16", k_group=128,
                             v_group=128, k_param="f32", v_param="f32")
WORKLOADS["long_shimmy"] = dict(WORKLOADS["long_mixed"], index=8, k_kind="shimmy4", v_kind="shimmy4",
                                k_group=128, v_group=128, k_param="f32", v_param="f32")

ACT_NUMPY = {"f32": np.float32, "f16": np.float16}


def workload(name: str, **overrides) -> dict:
    """A copy of a workload description with some fields replaced."""
    w = dict(WORKLOADS[name])
    w["name"] = name
    w.update(overrides)
    return w


def _rng(w: dict, *stream: int) -> np.random.Generator:
    """Independent stream per (workload seed, purpose, index...)."""
    seed = 1000 + int(w["index"])
    return np.random.default_rng(np.random.SeedSequence([seed, *stream]))


# Stream purposes (first entry of the stream key).
_S_LENS, _S_Q, _S_K, _S_V, _S_PAGES, _S_NEW = 1, 2, 3, 4, 5, 6


def seq_lens(w: dict) -> np.ndarray:
    """Per-sequence context lengths (int32 [batch])."""
    b = int(w["batch"])
    if "min_len" in w:
        r = _rng(w, _S_LENS)
        return r.integers(int(w["min_len"]), int(w["ctx"]), size=b,
                          endpoint=True).astype(np.int32)
    return np.full(b, int(w["ctx"]), dtype=np.int32)


def _normal(r: np.random.Generator, shape, w: dict, outliers: bool):
    x = r.standard_normal(size=shape, dtype=np.float32)
    frac = float(w.get("outlier_frac", 0.0))
    if outliers and frac > 0.0:
        mask = r.random(size=shape, dtype=np.float32) < np.float32(frac)
        x = np.where(mask, x * np.float32(8.0), x)
    return x.astype(ACT_NUMPY[w["act"]])


def kv_rows(w: dict, seq: int, which: str, n_tokens: int | None = None,
            layer: int = 0) -> np.ndarray:
    """New K or V rows of one sequence, tokens 0..n-1: [n][n_kv_heads][head_dim]."""
    n = int(seq_lens(w)[seq]) if n_tokens is None else int(n_tokens)
    r = _rng(w, _S_K if which == "k" else _S_V, layer, seq)
    return _normal(r, (n, w["n_kv_heads"], w["head_dim"]), w, outliers=True)


def queries(w: dict, layer: int = 0, step: int = 0) -> np.ndarray:
    """Decode-step queries [batch][n_heads][head_dim] in the activation dtype."""
    r = _rng(w, _S_Q, layer, step)
    return _normal(r, (w["batch"], w["n_heads"], w["head_dim"]), w,
                   outliers=False)


def new_rows(w: dict, which: str, n_rows: int, layer: int = 0,
             step: int = 0) -> np.ndarray:
    """Rows appended in one decode step: [n_rows][n_kv_heads][head_dim]."""
    r = _rng(w, _S_NEW, 0 if which == "k" else 1, layer, step)
    return _normal(r, (n_rows, w["n_kv_heads"], w["head_dim"]), w,
                   outliers=True)


def page_free_order(w: dict, n_pages: int) -> np.ndarray:
    """A seeded permutation of page ids (Fisher-Yates via numpy).

    Freeing every page of a fresh pool in this order leaves its LIFO free list
    shuffled, the way pages interleave when many sequences grow at once.
    """
    r = _rng(w, _S_PAGES)
    return r.permutation(n_pages).astype(np.int32)


def random_codes_input(seed: int, shape, scale: float = 1.0,
                       dtype=np.float32) -> np.ndarray:
    """Small generic N(0, scale^2) array for unit tests."""
    r = np.random.default_rng(seed)
    return (r.standard_normal(size=shape) * scale).astype(dtype)
