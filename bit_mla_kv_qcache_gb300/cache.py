"""Device buffers of one layer's low-bit dual-path MLA cache and the calls that use them.

PyTorch only allocates device memory and provides the stream; the writer and the decode
attention run in libmla_qcache.so.
"""
from __future__ import annotations

import torch

from . import binding


class QuantizedMLACache:
    """Page pool, BF16 sink/recent buffers, page table and lengths for B sequences.

    The page table is the caller's (a paged allocator maps positions to physical pages);
    by default sequence b owns pages [b*max_pages, (b+1)*max_pages).
    """

    def __init__(self, cfg: binding.Config, batch: int, max_pages: int, n_pages: int | None = None,
                 page_table: torch.Tensor | None = None, device="cuda"):
        self.cfg = cfg
        self.B = batch
        self.max_pages = max_pages
        self.n_pages = n_pages if n_pages is not None else batch * max_pages
        dev = torch.device(device)
        pb = binding.page_bytes(cfg)
        if pb == 0:
            raise binding.QCacheError(f"unsupported configuration {cfg}")
        self.pool = torch.zeros((self.n_pages, pb), dtype=torch.uint8, device=dev)
        self.sink = torch.zeros((batch, cfg.n_sink, 576), dtype=torch.int16, device=dev)
        self.ring = torch.zeros((batch, cfg.n_recent, 576), dtype=torch.int16, device=dev)
        if page_table is None:
            page_table = torch.arange(batch * max_pages, dtype=torch.int32, device=dev).view(batch, max_pages)
        self.page_table = page_table.to(device=dev, dtype=torch.int32).contiguous()
        self.seq_lens = torch.zeros(batch, dtype=torch.int32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self._ws = None
        self._ws_need = {}  # workspace bytes per head count
        self._lens_alt = None  # second length array for write_advance

    def write(self, c_new: torch.Tensor, kr_new: torch.Tensor, cu_new: torch.Tensor, max_new: int,
              advance: bool = True, stream=None) -> None:
        """Append rows cu_new[b]..cu_new[b+1]-1 to sequence b (BF16 c [N,512], k_R [N,64])."""
        binding.mla_qcache_write(self.cfg, c_new, kr_new, cu_new, self.seq_lens, max_new, self.page_table, self.pool,
                                 self.sink, self.ring, self.err, stream)
        if advance:
            binding.mla_qcache_advance(cu_new, self.seq_lens, stream)

    def write_advance(self, c_new: torch.Tensor, kr_new: torch.Tensor, cu_new: torch.Tensor, max_new: int,
                      stream=None) -> None:
        """write() with the length update in the same launch: the new lengths are stored into a
        second array, which then becomes ``self.seq_lens`` (the two arrays alternate)."""
        if self._lens_alt is None:
            self._lens_alt = torch.empty_like(self.seq_lens)
        binding.mla_qcache_write_advance(self.cfg, c_new, kr_new, cu_new, self.seq_lens, self._lens_alt, max_new,
                                         self.page_table, self.pool, self.sink, self.ring, self.err, stream)
        self.seq_lens, self._lens_alt = self._lens_alt, self.seq_lens

    def workspace(self, heads: int) -> torch.Tensor:
        need = self._ws_need.get(heads)
        if need is None:
            need = self._ws_need[heads] = binding.workspace_bytes(self.cfg, self.B, heads, self.max_pages)
        if self._ws is None or self._ws.numel() < need:
            # zeroed once: the decode keeps the merge counters at its start zero between calls
            self._ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=self.pool.device)
        return self._ws

    def decode(self, q_lat: torch.Tensor, q_rope: torch.Tensor, softmax_scale: float, out=None, lse=None,
               stream=None):
        """Attention readout O [B,H,512] (float32) and LSE [B,H] for one decode step."""
        B, H = q_lat.shape[0], q_lat.shape[1]
        if out is None:
            out = torch.empty((B, H, 512), dtype=torch.float32, device=q_lat.device)
        if lse is None:
            lse = torch.empty((B, H), dtype=torch.float32, device=q_lat.device)
        binding.mla_qcache_decode_attn(self.cfg, q_lat, q_rope, self.page_table, self.seq_lens, self.pool, self.sink,
                                       self.ring, softmax_scale, out, lse, self.workspace(H), self.err, stream)
        return out, lse

    def error_bits(self) -> int:
        return int(self.err.item())
