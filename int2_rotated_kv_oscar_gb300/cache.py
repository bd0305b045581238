"""Device memory for the OSCAR cache, allocated with PyTorch.

PyTorch is only the allocator here: these classes hold torch tensors and hand
their addresses to the C ABI (``abi.oscar_cache_view`` and friends).  No
arithmetic of the method happens in this file.
"""

import torch

from . import abi


class MixedCache:
    """Per-layer pools of one mixed-precision paged cache.

    int2_pages[l]  uint8  [num_pages, Hkv, 4608]
    k_sink[l], v_sink[l]  bf16 [num_sink_pages, Hkv, 64, 128]
    k_ring[l], v_ring[l]  bf16 [num_ring_slots, Hkv, 256, 128]
    page_table  int32 [batch, max_pages_per_req]   (shared by all layers)
    sink_page, ring_slot  int32 [batch]

    With ``recent_pages`` the recent window is paged instead: k_ring, v_ring
    are a pool of that many BF16 pages [recent_pages, Hkv, 64, 128] and
    recent_table int32 [batch, max_pages_per_req] (filled with -1; the caller
    assigns the pages of the logical pages the window touches).
    """

    def __init__(self, num_layers, num_kv_heads, num_pages, num_sink_pages, num_ring_slots, batch,
                 max_pages_per_req, device="cuda", recent_pages=None):
        self.num_layers = num_layers
        self.num_kv_heads = num_kv_heads
        self.num_pages = num_pages
        self.num_sink_pages = num_sink_pages
        self.num_ring_slots = num_ring_slots
        self.batch = batch
        self.max_pages_per_req = max_pages_per_req
        self.device = torch.device(device)
        H = num_kv_heads
        self.int2_pages = [torch.zeros((num_pages, H, abi.BLOCK_BYTES), dtype=torch.uint8, device=self.device)
                           for _ in range(num_layers)]
        self.k_sink = [torch.zeros((num_sink_pages, H, abi.SINK_TOKENS, abi.HEAD_DIM), dtype=torch.bfloat16,
                                   device=self.device) for _ in range(num_layers)]
        self.v_sink = [torch.zeros_like(t) for t in self.k_sink]
        self.paged_recent = recent_pages is not None
        if self.paged_recent:
            self.num_ring_slots = recent_pages
            rows = abi.PAGE_TOKENS
        else:
            rows = abi.RECENT_TOKENS
        self.k_ring = [torch.zeros((self.num_ring_slots, H, rows, abi.HEAD_DIM), dtype=torch.bfloat16,
                                   device=self.device) for _ in range(num_layers)]
        self.v_ring = [torch.zeros_like(t) for t in self.k_ring]
        self.recent_table = (torch.full((batch, max_pages_per_req), -1, dtype=torch.int32, device=self.device)
                             if self.paged_recent else None)
        self.page_table = torch.zeros((batch, max_pages_per_req), dtype=torch.int32, device=self.device)
        self.sink_page = torch.arange(batch, dtype=torch.int32, device=self.device) % max(num_sink_pages, 1)
        self.ring_slot = torch.arange(batch, dtype=torch.int32, device=self.device) % max(num_ring_slots, 1)

    def view(self, layer, batch=None):
        return abi.oscar_cache_view(
            int2_pages=self.int2_pages[layer].data_ptr(), num_pages=self.num_pages,
            k_sink=self.k_sink[layer].data_ptr(), v_sink=self.v_sink[layer].data_ptr(),
            num_sink_pages=self.num_sink_pages,
            k_ring=self.k_ring[layer].data_ptr(), v_ring=self.v_ring[layer].data_ptr(),
            num_ring_slots=self.num_ring_slots,
            page_table=self.page_table.data_ptr(), max_pages_per_req=self.max_pages_per_req,
            sink_page=self.sink_page.data_ptr(), ring_slot=self.ring_slot.data_ptr(),
            batch=self.batch if batch is None else batch,
            recent_page_table=self.recent_table.data_ptr() if self.paged_recent else None)

    def chunk_view(self, layer, b, n):
        """A view of n batch rows that all alias request b's page table row, sink
        page and ring slot (the queries of one chunk, for oscar_extend_attention).
        Returns (view, tables); keep ``tables`` alive while the view is in use."""
        pt = self.page_table[b:b + 1].expand(n, -1).contiguous()
        sp = self.sink_page[b:b + 1].expand(n).contiguous()
        rs = self.ring_slot[b:b + 1].expand(n).contiguous()
        rt = self.recent_table[b:b + 1].expand(n, -1).contiguous() if self.paged_recent else None
        view = abi.oscar_cache_view(
            int2_pages=self.int2_pages[layer].data_ptr(), num_pages=self.num_pages,
            k_sink=self.k_sink[layer].data_ptr(), v_sink=self.v_sink[layer].data_ptr(),
            num_sink_pages=self.num_sink_pages,
            k_ring=self.k_ring[layer].data_ptr(), v_ring=self.v_ring[layer].data_ptr(),
            num_ring_slots=self.num_ring_slots,
            page_table=pt.data_ptr(), max_pages_per_req=self.max_pages_per_req,
            sink_page=sp.data_ptr(), ring_slot=rs.data_ptr(), batch=n,
            recent_page_table=rt.data_ptr() if rt is not None else None)
        view._tensors = (pt, sp, rs, rt)
        return view, view._tensors


class BF16PagedCache:
    """A plain BF16 paged cache of one layer (the comparator)."""

    def __init__(self, num_kv_heads, num_pages, batch, max_pages_per_req, device="cuda"):
        self.k_pages = torch.zeros((num_pages, num_kv_heads, abi.PAGE_TOKENS, abi.HEAD_DIM), dtype=torch.bfloat16,
                                   device=device)
        self.v_pages = torch.zeros_like(self.k_pages)
        self.num_pages = num_pages
        self.batch = batch
        self.max_pages_per_req = max_pages_per_req
        self.page_table = torch.zeros((batch, max_pages_per_req), dtype=torch.int32, device=device)

    def view(self):
        return abi.oscar_bf16_cache_view(
            k_pages=self.k_pages.data_ptr(), v_pages=self.v_pages.data_ptr(), num_pages=self.num_pages,
            page_table=self.page_table.data_ptr(), max_pages_per_req=self.max_pages_per_req, batch=self.batch)


def append_args(k, v, pos, cu_seqlens=None, max_tokens_per_req=None, fresh_ring=False):
    """oscar_append_args for bf16 tensors k, v [n_tokens, Hkv, 128] and int32 device tensors.
    The struct keeps the tensors alive for as long as it lives (it holds their addresses)."""
    n = int(k.shape[0])
    a = abi.oscar_append_args(
        k=k.data_ptr(), v=v.data_ptr(), pos=pos.data_ptr(),
        cu_seqlens=None if cu_seqlens is None else cu_seqlens.data_ptr(), n_tokens=n,
        max_tokens_per_req=n if max_tokens_per_req is None else int(max_tokens_per_req),
        flags=abi.OSCAR_APPEND_FRESH_RING if fresh_ring else 0)
    a._tensors = (k, v, pos, cu_seqlens)
    return a


def decode_args(q, out, ctx_len, max_ctx_len, sm_scale=0.0):
    """oscar_decode_args; the struct keeps q, out and ctx_len alive (it holds their addresses)."""
    a = abi.oscar_decode_args(q=q.data_ptr(), out=out.data_ptr(), ctx_len=ctx_len.data_ptr(),
                              max_ctx_len=int(max_ctx_len), sm_scale=float(sm_scale))
    a._tensors = (q, out, ctx_len)
    return a


def extend_workspace(ctx, batch, chunk, max_ctx_len, device="cuda"):
    """A caller-owned workspace for oscar_extend_chunk (uint8 tensor, 256-byte
    aligned, zero-filled).  Returns (tensor, pointer, bytes)."""
    n = abi.oscar_extend_workspace_bytes(ctx, batch, chunk, max_ctx_len)
    t = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t, t.data_ptr() + off, n


def workspace(ctx, max_batch, max_ctx_len, device="cuda"):
    """A caller-owned decode workspace (uint8 tensor, 256-byte aligned, zero-filled
    as the fused decode step wants it before its first use)."""
    n = abi.oscar_decode_workspace_bytes(ctx, max_batch, max_ctx_len)
    t = torch.zeros(n + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t, t.data_ptr() + off, n
