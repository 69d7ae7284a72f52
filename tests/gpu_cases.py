"""Shared set-up for the GPU parity tests: one layer's cache filled through the
C ABI (GPU) and, independently, through the oracle (CPU) from the same seeded
rows and the same block table."""
from __future__ import annotations

import numpy as np
import torch

import kvq_workloads as wl
from int8_quantized_paged_gb300 import kvq
from int8_quantized_paged_gb300.cache import LayerCache
from oracle import kvq_oracle as O

TOL = 2e-3            # max row-relative error of outputs (the required bound)
P = 16

_ORACLE_ROPE = {}


def oracle_rope(head_dim: int, base: float, max_pos: int) -> np.ndarray:
    key = (head_dim, base)
    tab = _ORACLE_ROPE.get(key)
    if tab is None or tab.shape[0] < max_pos:
        tab = O.rope_table(head_dim, base, max(max_pos, 64))
        _ORACLE_ROPE[key] = tab
    return tab


class Case:
    """A workload with explicit sequence lengths, filled on both sides."""

    def __init__(self, w: dict, lens, ring_rows: int = 0, shuffle: bool = True, extra_pages: int = 3,
                 oracle_seqs=None, fill_oracle: bool = True, extra_positions: int = 0):
        self.w = w
        self.lens = np.asarray(lens, dtype=np.int32)
        self.B = len(self.lens)
        self.cfg = kvq.config(**w)
        self.spec = O.Spec.from_workload(w)
        self.ring_rows = ring_rows
        if ring_rows:
            self.max_pages = ring_rows // P
            need = self.B * self.max_pages
        else:
            self.max_pages = max(1, -(-int(self.lens.max()) // P))
            need = int(sum(-(-int(L) // P) for L in self.lens))
        self.n_pages = need + extra_pages
        pool = kvq.Pool(self.n_pages)
        if shuffle:
            pool.alloc(self.n_pages)
            pool.free(wl.page_free_order(w, self.n_pages))
        self.rope_max = max(2, int(self.lens.max()) + 1 + extra_positions)
        self.cache = LayerCache(self.cfg, self.B, self.max_pages, self.n_pages, self.rope_max, ring_rows,
                                pool=pool)
        for b, L in enumerate(self.lens):
            self.cache.reserve(b, ring_rows if ring_rows else int(L))
        self.cache.sync_table()
        self.bt = self.cache.table.data()
        self.oracle_seqs = list(range(self.B)) if oracle_seqs is None else list(oracle_seqs)
        self.rows = {}
        self._fill_gpu()
        self.pools = None
        if fill_oracle:
            self._fill_oracle()

    def _chunks(self, L):
        step = self.ring_rows if self.ring_rows else max(L, 1)
        for s in range(0, L, step):
            yield s, min(L, s + step)

    def _fill_gpu(self):
        dev = self.cache.device
        for b, L in enumerate(self.lens):
            k, v = wl.kv_rows(self.w, b, "k", int(L)), wl.kv_rows(self.w, b, "v", int(L))
            if b in self.oracle_seqs:
                self.rows[b] = (k, v)
            for s, e in self._chunks(int(L)):   # rows of one call never share a ring slot
                kt = torch.from_numpy(np.ascontiguousarray(k[s:e])).to(dev)
                vt = torch.from_numpy(np.ascontiguousarray(v[s:e])).to(dev)
                pos = torch.arange(s, e, dtype=torch.int32, device=dev)
                sid = torch.full((e - s,), b, dtype=torch.int32, device=dev)
                self.cache.append(kt, vt, pos, sid)
        torch.cuda.synchronize()

    def _fill_oracle(self):
        s = self.spec
        self.pools = {"k": np.zeros(self.n_pages * O.page_bytes(s, "k"), np.uint8),
                      "v": np.zeros(self.n_pages * O.page_bytes(s, "v"), np.uint8)}
        tab = oracle_rope(s.head_dim, s.rope_base, self.rope_max)
        for b in self.oracle_seqs:
            L = int(self.lens[b])
            k, v = self.rows[b]
            O.append(s, self.pools, k, v, np.full(L, b), np.arange(L), self.bt, self.ring_rows, tab)

    def gpu_pools(self):
        return self.cache.k_pool.cpu().numpy(), self.cache.v_pool.cpu().numpy()

    def queries(self, step: int = 0) -> np.ndarray:
        return wl.queries(dict(self.w, batch=self.B), step=step)

    def gpu_decode(self, q: np.ndarray, chunk_tokens: int = 0, window: int = 0, lens=None, stream=None):
        dev = self.cache.device
        qt = torch.from_numpy(q).to(dev)
        lens = self.lens if lens is None else np.asarray(lens, np.int32)
        lt = torch.from_numpy(lens).to(dev)
        out = torch.full_like(qt, float("nan"))
        ws = self.cache.workspace(self.B, chunk_tokens, window)
        if window:
            self.cache.window_decode(qt, lt, out, ws, window, chunk_tokens, stream=stream)
        else:
            self.cache.decode(qt, lt, out, ws, chunk_tokens, stream=stream)
        torch.cuda.synchronize()
        return out.float().cpu().numpy().astype(np.float64)

    def oracle_decode(self, q: np.ndarray, window: int = 0, seqs=None):
        return O.decode(self.spec, q, self.pools, self.bt, self.lens, window, self.ring_rows,
                        seqs=self.oracle_seqs if seqs is None else seqs)


FLOOR = 1e-3          # row floor of the output comparison (0.1 % of the row's largest magnitude)


def floor_for(w: dict) -> float:
    """Row floor for a workload's outputs.

    The absolute fp32 error of a score grows with attn_scale * sum_d |q_d k_d|,
    about attn_scale * head_dim for N(0,1) rows, while the default scale
    1/sqrt(head_dim) keeps that at sqrt(head_dim).  So the floor is 0.1 %
    times attn_scale * sqrt(head_dim) (at least 1), and at most 1 %: only a
    layer with a raised score scale (attention scale 1.0, as the sliding +
    global mix uses) gets more than 0.1 %.
    """
    alpha = float(w.get("attn_scale", 0.0))
    if alpha <= 0.0:
        return FLOOR
    return min(1e-2, FLOOR * max(1.0, alpha * float(w["head_dim"]) ** 0.5))


def max_row_err(got, ref, seqs=None, floor=FLOOR):
    """The larger of the max row-relative error (with the given row floor) and
    the max normwise error, over the rows of the selected sequences."""
    if seqs is not None:
        got, ref = got[list(seqs)], ref[list(seqs)]
    return float(max(np.max(O.row_rel_error(got, ref, floor=floor)), np.max(O.row_norm_error(got, ref))))


def pages_of(case: Case, b: int):
    n = case.cache.table.num_pages(b)
    return case.bt[b, :n]


def pool_slice(pool: np.ndarray, page_bytes: int, pages) -> np.ndarray:
    return np.concatenate([pool[p * page_bytes:(p + 1) * page_bytes] for p in pages]) if len(pages) else \
        np.zeros(0, np.uint8)
