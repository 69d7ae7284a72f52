"""ctypes binding of libkvq.so (include/kvq.h), one Python function per C entry.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels or its C++ host runtime.  Device buffers are torch tensors (PyTorch is
used for device memory and streams); their data pointers go to the C ABI
unchanged.  A non-OK status raises KvqError with the library's message.  There
is no fallback: if libkvq.so is missing, the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

# Enumerations of kvq.h.
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_OUT_OF_PAGES, ERR_BAD_BLOCK_TABLE, \
    ERR_WORKSPACE_TOO_SMALL, ERR_CUDA = range(7)
DEV_BAD_PAGE, DEV_BAD_POS, DEV_BAD_SEQ, DEV_BAD_LEN = 1, 2, 4, 8
F32, F16, BF16 = 0, 1, 2
SYM_INT4, SYM_INT8, AFFINE_INT4, F16_KV, F32_KV, SHIMMY_INT4 = range(6)
ROPE_NONE, ROPE_NORMAL, ROPE_NEOX = 0, 1, 2
FLAG_EARLY_READS = 1

FLOATS = {"f32": F32, "f16": F16, "bf16": BF16}
KINDS = {"sym4": SYM_INT4, "sym8": SYM_INT8, "affine4": AFFINE_INT4, "f16": F16_KV, "f32": F32_KV,
         "shimmy4": SHIMMY_INT4}
ROPES = {"none": ROPE_NONE, "normal": ROPE_NORMAL, "neox": ROPE_NEOX}


class KvqError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"kvq status {status}: {message}")
        self.status = status


class Config(C.Structure):
    """struct kvq_config."""
    _fields_ = [("n_heads", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("page_size", C.c_int32), ("k_dtype", C.c_int32), ("v_dtype", C.c_int32),
                ("k_group", C.c_int32), ("v_group", C.c_int32), ("k_param_dtype", C.c_int32),
                ("v_param_dtype", C.c_int32), ("act_dtype", C.c_int32), ("rope", C.c_int32),
                ("attn_scale", C.c_float), ("flags", C.c_int32), ("rope_base", C.c_double)]


def config(n_heads, n_kv_heads, head_dim, page_size=16, k_kind="sym4", v_kind="sym4",
           k_group=128, v_group=128, k_param="f32", v_param="f32", act="f16",
           attn_scale=0.0, rope="normal", rope_base=10000.0, flags=0, **_ignored) -> Config:
    """A kvq_config from the names used in workload descriptions."""
    return Config(n_heads, n_kv_heads, head_dim, page_size, KINDS[k_kind], KINDS[v_kind],
                  k_group, v_group, FLOATS[k_param], FLOATS[v_param], FLOATS[act],
                  ROPES[rope], float(attn_scale), int(flags), float(rope_base))


_lib = None
_vp, _i32, _i64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
_cfgp = C.POINTER(Config)

_SIGS = {
    "kvq_abi_version": (_i32, []),
    "kvq_last_error": (C.c_char_p, []),
    "kvq_validate_config": (C.c_int, [_cfgp]),
    "kvq_decode_launches": (_i32, [_cfgp]),
    "kvq_decode_cluster_ctas": (_i32, [_cfgp, _i32, _i32, _i32, _i32]),
    "kvq_cache_bytes": (_sz, [_cfgp, _i32, _i64]),
    "kvq_page_bytes": (_sz, [_cfgp, _i32]),
    "kvq_pool_create": (C.c_int, [_i32, C.POINTER(_vp)]),
    "kvq_pool_destroy": (None, [_vp]),
    "kvq_pool_alloc": (C.c_int, [_vp, _i32, _vp]),
    "kvq_pool_free": (C.c_int, [_vp, _i32, _vp]),
    "kvq_pool_num_free": (_i32, [_vp]),
    "kvq_pool_num_pages": (_i32, [_vp]),
    "kvq_table_create": (C.c_int, [_vp, _i32, _i32, _i32, C.POINTER(_vp)]),
    "kvq_table_destroy": (None, [_vp]),
    "kvq_table_reserve": (C.c_int, [_vp, _i32, _i64]),
    "kvq_table_release": (C.c_int, [_vp, _i32]),
    "kvq_table_data": (_vp, [_vp]),
    "kvq_table_num_pages": (_i32, [_vp, _i32]),
    "kvq_rope_table": (C.c_int, [_cfgp, _i32, _vp]),
    "kvq_append": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp, _i32,
                             _vp, _vp, _i32, _vp, _vp]),
    "kvq_decode_workspace_bytes": (_sz, [_cfgp, _i32, _i32, _i32]),
    "kvq_decode_attention": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp,
                                       _i32, _vp, _vp, _sz, _i32, _vp, _vp]),
    "kvq_append_decode_attention": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32,
                                              _vp, _vp, _i32, _vp, _vp, _sz, _i32, _vp, _vp]),
    "kvq_append_decode_launches": (_i32, [_cfgp]),
    "kvq_append_window_decode": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32,
                                           _vp, _vp, _i32, _vp, _vp, _sz, _i32, _vp, _vp]),
    "kvq_window_workspace_bytes": (_sz, [_cfgp, _i32, _i32, _i32]),
    "kvq_window_decode": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _vp, _vp,
                                    _i32, _vp, _vp, _sz, _i32, _vp, _vp]),
    "kvq_decode_attention_noalloc": (C.c_int, [_cfgp, _i32, _vp, _vp, _vp, _i32, _vp, _i32, _vp, _vp,
                                               _i32, _vp, _i32, _vp, _vp]),
    "kvq_clear_device_status": (C.c_int, [_vp, _vp]),
    "kvq_get_device_status": (C.c_int, [_vp, _vp, C.POINTER(_i32)]),
}


def lib() -> C.CDLL:
    """The loaded libkvq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m int8_quantized_paged_gb300.build`")
        h = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _lib = h
    return _lib


def exported_symbols() -> list[str]:
    return list(_SIGS)


def last_error() -> str:
    return lib().kvq_last_error().decode()


def _check(st: int) -> None:
    if st != OK:
        raise KvqError(st, last_error())


def _ptr(t) -> int | None:
    """Data pointer of a torch tensor (or None)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to kvq must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ------------------------------------------------------------------ sizing


def abi_version() -> int:
    return lib().kvq_abi_version()


def validate_config(cfg: Config) -> None:
    _check(lib().kvq_validate_config(C.byref(cfg)))


def decode_launches(cfg: Config) -> int:
    """Kernel launches per decode call (1: tensor-core path, 2: CUDA-core path)."""
    n = lib().kvq_decode_launches(C.byref(cfg))
    if n == 0:
        raise KvqError(ERR_INVALID_ARG, last_error())
    return n


def decode_cluster_ctas(cfg: Config, batch: int, max_pages_per_seq: int, window: int = 0,
                        chunk_tokens: int = 0) -> int:
    """CTAs per cluster of a decode call (0: the partials go through the workspace)."""
    n = lib().kvq_decode_cluster_ctas(C.byref(cfg), batch, max_pages_per_seq, window, chunk_tokens)
    if n < 0:
        raise KvqError(ERR_INVALID_ARG, last_error())
    return n


def cache_bytes(cfg: Config, n_layers: int, ctx: int) -> int:
    return lib().kvq_cache_bytes(C.byref(cfg), n_layers, ctx)


def page_bytes(cfg: Config, which: int) -> int:
    return lib().kvq_page_bytes(C.byref(cfg), which)


def rope_table(cfg: Config, max_pos: int) -> np.ndarray:
    """float32 [max_pos][head_dim/2][2] computed by the library on the host."""
    out = np.empty((max_pos, cfg.head_dim // 2, 2), dtype=np.float32)
    _check(lib().kvq_rope_table(C.byref(cfg), max_pos, out.ctypes.data))
    return out


# -------------------------------------------------------- pool and tables


class Pool:
    """Host LIFO free list of page ids (kvq_pool_*)."""

    def __init__(self, n_pages: int):
        h = _vp()
        _check(lib().kvq_pool_create(n_pages, C.byref(h)))
        self._h = h
        # Handles of the live tables over this pool.  The cyclic garbage
        # collector may finalize a pool before a table that uses it; the pool
        # then destroys those tables first (their pages go back into it), and
        # a table destroys itself only while its pool still lists it.
        self._tables = set()

    @property
    def handle(self):
        return self._h

    def alloc(self, n: int) -> np.ndarray:
        ids = np.empty(n, dtype=np.int32)
        _check(lib().kvq_pool_alloc(self._h, n, ids.ctypes.data))
        return ids

    def free(self, ids) -> None:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        _check(lib().kvq_pool_free(self._h, len(ids), ids.ctypes.data))

    @property
    def num_free(self) -> int:
        return lib().kvq_pool_num_free(self._h)

    @property
    def num_pages(self) -> int:
        return lib().kvq_pool_num_pages(self._h)

    def close(self) -> None:
        if self._h:
            for t in list(self._tables):
                lib().kvq_table_destroy(_vp(t))
            self._tables.clear()
            lib().kvq_pool_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Table:
    """Per-sequence page lists with a dense host mirror (kvq_table_*)."""

    def __init__(self, pool: Pool, n_seqs: int, max_pages_per_seq: int, page_size: int = 16):
        h = _vp()
        _check(lib().kvq_table_create(pool.handle, n_seqs, max_pages_per_seq, page_size, C.byref(h)))
        self._h, self.pool = h, pool
        pool._tables.add(h.value)
        self.n_seqs, self.max_pages = n_seqs, max_pages_per_seq

    def reserve(self, seq: int, n_rows: int) -> None:
        _check(lib().kvq_table_reserve(self._h, seq, n_rows))

    def release(self, seq: int) -> None:
        _check(lib().kvq_table_release(self._h, seq))

    def num_pages(self, seq: int) -> int:
        return lib().kvq_table_num_pages(self._h, seq)

    def data(self) -> np.ndarray:
        """A copy of the dense table int32 [n_seqs][max_pages_per_seq]."""
        p = lib().kvq_table_data(self._h)
        buf = (C.c_int32 * (self.n_seqs * self.max_pages)).from_address(p)
        return np.frombuffer(buf, dtype=np.int32).reshape(self.n_seqs, self.max_pages).copy()

    def close(self) -> None:
        if self._h:
            if self._h.value in self.pool._tables:
                self.pool._tables.discard(self._h.value)
                lib().kvq_table_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------ device calls


def append(cfg: Config, k_new, v_new, seq_ids, pos, block_table, n_seqs: int,
           max_pages_per_seq: int, ring_rows: int, rope_tab, rope_max_pos: int,
           k_pool, v_pool, n_pool_pages: int, dev_status, stream=None) -> None:
    _check(lib().kvq_append(C.byref(cfg), k_new.shape[0], _ptr(k_new), _ptr(v_new), _ptr(seq_ids),
                            _ptr(pos), _ptr(block_table), n_seqs, max_pages_per_seq, ring_rows,
                            _ptr(rope_tab), rope_max_pos, _ptr(k_pool), _ptr(v_pool), n_pool_pages,
                            _ptr(dev_status), _stream(stream)))


def decode_workspace_bytes(cfg: Config, batch: int, max_pages_per_seq: int, chunk_tokens: int = 0) -> int:
    n = lib().kvq_decode_workspace_bytes(C.byref(cfg), batch, max_pages_per_seq, chunk_tokens)
    if n == 0:
        raise KvqError(ERR_INVALID_ARG, last_error())
    return n


def decode_attention(cfg: Config, q, k_pool, v_pool, n_pool_pages: int, block_table,
                     max_pages_per_seq: int, seq_lens, rope_tab, rope_max_pos: int, out,
                     workspace, dev_status, chunk_tokens: int = 0, stream=None) -> None:
    _check(lib().kvq_decode_attention(
        C.byref(cfg), q.shape[0], _ptr(q), _ptr(k_pool), _ptr(v_pool), n_pool_pages, _ptr(block_table),
        max_pages_per_seq, _ptr(seq_lens), _ptr(rope_tab), rope_max_pos, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), chunk_tokens, _ptr(dev_status), _stream(stream)))


def append_decode_attention(cfg: Config, q, k_new, v_new, pos, k_pool, v_pool, n_pool_pages: int,
                            block_table, max_pages_per_seq: int, seq_lens, rope_tab, rope_max_pos: int,
                            out, workspace, dev_status, chunk_tokens: int = 0, stream=None) -> None:
    """kvq_append of row b at pos[b] for every sequence b, then kvq_decode_attention, in one call."""
    _check(lib().kvq_append_decode_attention(
        C.byref(cfg), q.shape[0], _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(k_pool), _ptr(v_pool),
        n_pool_pages, _ptr(block_table), max_pages_per_seq, _ptr(seq_lens), _ptr(rope_tab), rope_max_pos,
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), chunk_tokens,
        _ptr(dev_status), _stream(stream)))


def append_window_decode(cfg: Config, q, k_new, v_new, pos, k_pool, v_pool, n_pool_pages: int, ring_table,
                         ring_rows: int, window: int, seq_lens, rope_tab, rope_max_pos: int, out, workspace,
                         dev_status, chunk_tokens: int = 0, stream=None) -> None:
    """kvq_append into the ring of row b at pos[b] for every sequence b, then kvq_window_decode."""
    _check(lib().kvq_append_window_decode(
        C.byref(cfg), q.shape[0], _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(pos), _ptr(k_pool), _ptr(v_pool),
        n_pool_pages, _ptr(ring_table), ring_rows, window, _ptr(seq_lens), _ptr(rope_tab), rope_max_pos,
        _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), chunk_tokens,
        _ptr(dev_status), _stream(stream)))


def append_decode_launches(cfg: Config) -> int:
    """Kernel launches per append_decode_attention call (1: tensor-core path)."""
    n = lib().kvq_append_decode_launches(C.byref(cfg))
    if n == 0:
        raise KvqError(ERR_INVALID_ARG, last_error())
    return n


NOALLOC_SCRATCH_BYTES = 8 << 20


def decode_attention_noalloc(cfg: Config, q, k_pool, v_pool, n_pool_pages: int, block_table,
                             max_pages_per_seq: int, seq_lens, rope_tab, rope_max_pos: int, out,
                             dev_status, chunk_tokens: int = 0, stream=None) -> None:
    """kvq_decode_attention with the library's built-in scratch as workspace."""
    _check(lib().kvq_decode_attention_noalloc(
        C.byref(cfg), q.shape[0], _ptr(q), _ptr(k_pool), _ptr(v_pool), n_pool_pages, _ptr(block_table),
        max_pages_per_seq, _ptr(seq_lens), _ptr(rope_tab), rope_max_pos, _ptr(out), chunk_tokens,
        _ptr(dev_status), _stream(stream)))


def window_workspace_bytes(cfg: Config, batch: int, window: int, chunk_tokens: int = 0) -> int:
    n = lib().kvq_window_workspace_bytes(C.byref(cfg), batch, window, chunk_tokens)
    if n == 0:
        raise KvqError(ERR_INVALID_ARG, last_error())
    return n


def window_decode(cfg: Config, q, k_pool, v_pool, n_pool_pages: int, ring_table, ring_rows: int,
                  window: int, seq_lens, rope_tab, rope_max_pos: int, out, workspace, dev_status,
                  chunk_tokens: int = 0, stream=None) -> None:
    _check(lib().kvq_window_decode(
        C.byref(cfg), q.shape[0], _ptr(q), _ptr(k_pool), _ptr(v_pool), n_pool_pages, _ptr(ring_table),
        ring_rows, window, _ptr(seq_lens), _ptr(rope_tab), rope_max_pos, _ptr(out), _ptr(workspace),
        workspace.numel() * workspace.element_size(), chunk_tokens, _ptr(dev_status), _stream(stream)))


def clear_device_status(dev_status, stream=None) -> None:
    _check(lib().kvq_clear_device_status(_ptr(dev_status), _stream(stream)))


def get_device_status(dev_status, stream=None) -> int:
    """Synchronize the stream and return the device status bits (0 when clean)."""
    bits = C.c_int32(0)
    st = lib().kvq_get_device_status(_ptr(dev_status), _stream(stream), C.byref(bits))
    if st not in (OK, ERR_BAD_BLOCK_TABLE):
        _check(st)
    return bits.value
