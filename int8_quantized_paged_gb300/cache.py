"""Device-memory plumbing around the C ABI for one attention layer's cache.

``LayerCache`` owns torch tensors for the K and V pools, a device copy of the
block table, the RoPE table and the status word, plus the library's host page
pool and block table.  Every computation is a call into libkvq.
"""
from __future__ import annotations

import numpy as np
import torch

from . import kvq

_TORCH_ACT = {kvq.F32: torch.float32, kvq.F16: torch.float16, kvq.BF16: torch.bfloat16}


class LayerCache:
    def __init__(self, cfg: kvq.Config, n_seqs: int, max_pages_per_seq: int, n_pool_pages: int,
                 rope_max_pos: int = 0, ring_rows: int = 0, device="cuda", pool: kvq.Pool | None = None,
                 rope_host: np.ndarray | None = None, rope_tab: torch.Tensor | None = None):
        self.cfg = cfg
        self.device = torch.device(device)
        self.n_seqs, self.max_pages, self.n_pool_pages = n_seqs, max_pages_per_seq, n_pool_pages
        self.ring_rows = ring_rows
        self.pool = pool if pool is not None else kvq.Pool(n_pool_pages)
        self.table = kvq.Table(self.pool, n_seqs, max_pages_per_seq, cfg.page_size)
        self.k_pool = torch.zeros(n_pool_pages * kvq.page_bytes(cfg, 0), dtype=torch.uint8, device=self.device)
        self.v_pool = torch.zeros(n_pool_pages * kvq.page_bytes(cfg, 1), dtype=torch.uint8, device=self.device)
        self.block_table = torch.full((n_seqs, max_pages_per_seq), -1, dtype=torch.int32, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.rope_max_pos = rope_max_pos
        self.rope_tab = None
        if cfg.rope != kvq.ROPE_NONE and rope_max_pos > 0:
            if rope_tab is not None:   # a table shared by the layers of a model
                if rope_tab.shape[0] < rope_max_pos:
                    raise ValueError("shared RoPE table has fewer rows than rope_max_pos")
                self.rope_tab = rope_tab
            else:
                host = rope_host if rope_host is not None else kvq.rope_table(cfg, rope_max_pos)
                self.rope_tab = torch.from_numpy(host).to(self.device)

    @property
    def act_dtype(self) -> torch.dtype:
        return _TORCH_ACT[self.cfg.act_dtype]

    def reserve(self, seq: int, n_rows: int) -> None:
        self.table.reserve(seq, n_rows)

    def sync_table(self) -> None:
        self.block_table.copy_(torch.from_numpy(self.table.data()))

    def set_table(self, table: np.ndarray) -> None:
        """Use an explicit block table (bypassing the host page pool)."""
        self.block_table.copy_(torch.as_tensor(table, dtype=torch.int32))

    def append(self, k_new, v_new, pos, seq_ids=None, stream=None) -> None:
        kvq.append(self.cfg, k_new, v_new, seq_ids, pos, self.block_table, self.n_seqs, self.max_pages,
                   self.ring_rows, self.rope_tab, self.rope_max_pos, self.k_pool, self.v_pool,
                   self.n_pool_pages, self.status, stream)

    def workspace(self, batch: int, chunk_tokens: int = 0, window: int = 0) -> torch.Tensor:
        if window:
            n = kvq.window_workspace_bytes(self.cfg, batch, window, chunk_tokens)
        else:
            n = kvq.decode_workspace_bytes(self.cfg, batch, self.max_pages, chunk_tokens)
        return torch.zeros(n, dtype=torch.uint8, device=self.device)   # counters start at zero

    def decode(self, q, seq_lens, out, workspace, chunk_tokens: int = 0, stream=None) -> None:
        kvq.decode_attention(self.cfg, q, self.k_pool, self.v_pool, self.n_pool_pages, self.block_table,
                             self.max_pages, seq_lens, self.rope_tab, self.rope_max_pos, out, workspace,
                             self.status, chunk_tokens, stream)

    def append_decode(self, q, k_new, v_new, pos, seq_lens, out, workspace, chunk_tokens: int = 0,
                      stream=None) -> None:
        """Append row b at pos[b] of every sequence b, then decode (one call)."""
        kvq.append_decode_attention(self.cfg, q, k_new, v_new, pos, self.k_pool, self.v_pool, self.n_pool_pages,
                                    self.block_table, self.max_pages, seq_lens, self.rope_tab, self.rope_max_pos,
                                    out, workspace, self.status, chunk_tokens, stream)

    def append_window_decode(self, q, k_new, v_new, pos, seq_lens, out, workspace, window: int,
                             chunk_tokens: int = 0, stream=None) -> None:
        """Append row b at pos[b] into the ring of every sequence b, then window-decode (one call)."""
        kvq.append_window_decode(self.cfg, q, k_new, v_new, pos, self.k_pool, self.v_pool, self.n_pool_pages,
                                 self.block_table, self.ring_rows, window, seq_lens, self.rope_tab,
                                 self.rope_max_pos, out, workspace, self.status, chunk_tokens, stream)

    def window_decode(self, q, seq_lens, out, workspace, window: int, chunk_tokens: int = 0,
                      stream=None) -> None:
        kvq.window_decode(self.cfg, q, self.k_pool, self.v_pool, self.n_pool_pages, self.block_table,
                          self.ring_rows, window, seq_lens, self.rope_tab, self.rope_max_pos, out, workspace,
                          self.status, chunk_tokens, stream)

    def status_bits(self) -> int:
        return kvq.get_device_status(self.status)

    def close(self) -> None:
        self.table.close()
