"""CPU: the host side of the cache bindings (views, tables, argument structs).

No kernel runs here: the pools are CPU tensors, and the tests check what the
Python layer hands to the C ABI -- the pool addresses and counts of a view,
the paged recent window's table, the aliasing tables of a chunk view, and that
the argument structs keep alive the tensors whose addresses they hold.
"""

import gc

import torch

from int2_rotated_kv_oscar_gb300 import abi
from int2_rotated_kv_oscar_gb300 import cache as kvcache


def test_ring_view_points_at_the_pools():
    c = kvcache.MixedCache(2, 4, 10, 3, 3, 3, 6, device="cpu")
    v = c.view(1)
    assert v.int2_pages == c.int2_pages[1].data_ptr() and v.num_pages == 10
    assert v.k_sink == c.k_sink[1].data_ptr() and v.v_sink == c.v_sink[1].data_ptr() and v.num_sink_pages == 3
    assert v.k_ring == c.k_ring[1].data_ptr() and v.v_ring == c.v_ring[1].data_ptr() and v.num_ring_slots == 3
    assert v.page_table == c.page_table.data_ptr() and v.max_pages_per_req == 6 and v.batch == 3
    assert v.sink_page == c.sink_page.data_ptr() and v.ring_slot == c.ring_slot.data_ptr()
    assert v.recent_page_table is None
    assert tuple(c.k_ring[0].shape) == (3, 4, abi.RECENT_TOKENS, abi.HEAD_DIM)
    assert c.int2_pages[0].shape[-1] == abi.BLOCK_BYTES
    assert c.view(0, batch=1).batch == 1


def test_paged_recent_view():
    c = kvcache.MixedCache(1, 2, 8, 2, 2, 2, 5, device="cpu", recent_pages=11)
    assert tuple(c.k_ring[0].shape) == (11, 2, abi.PAGE_TOKENS, abi.HEAD_DIM)
    assert tuple(c.recent_table.shape) == (2, 5) and bool((c.recent_table == -1).all())
    v = c.view(0)
    assert v.num_ring_slots == 11 and v.recent_page_table == c.recent_table.data_ptr()


def test_chunk_view_aliases_one_request():
    c = kvcache.MixedCache(1, 2, 20, 3, 3, 3, 6, device="cpu", recent_pages=15)
    c.page_table.copy_(torch.arange(18, dtype=torch.int32).view(3, 6))
    c.recent_table.copy_(torch.arange(18, dtype=torch.int32).view(3, 6) % 15)
    view, tabs = c.chunk_view(0, 1, 4)
    pt, sp, rs, rt = tabs
    assert view.batch == 4 and view._tensors is tabs
    assert bool((pt == c.page_table[1]).all()) and tuple(pt.shape) == (4, 6)
    assert bool((sp == c.sink_page[1]).all()) and bool((rs == c.ring_slot[1]).all())
    assert bool((rt == c.recent_table[1]).all())
    assert view.page_table == pt.data_ptr() and view.recent_page_table == rt.data_ptr()


def test_argument_structs_keep_their_tensors_alive():
    # built from temporaries: the structs must hold them, so the addresses stay valid
    a = kvcache.append_args(torch.zeros(3, 2, 128, dtype=torch.bfloat16), torch.ones(3, 2, 128, dtype=torch.bfloat16),
                            torch.tensor([5], dtype=torch.int32), torch.tensor([0, 3], dtype=torch.int32), 3)
    d = kvcache.decode_args(torch.zeros(1, 8, 128, dtype=torch.bfloat16), torch.zeros(1, 8, 128),
                            torch.tensor([7], dtype=torch.int32), 7)
    gc.collect()
    k, v, pos, cu = a._tensors
    assert (a.k, a.v, a.pos, a.cu_seqlens) == (k.data_ptr(), v.data_ptr(), pos.data_ptr(), cu.data_ptr())
    assert a.n_tokens == 3 and a.max_tokens_per_req == 3 and int(pos[0]) == 5
    q, out, lens = d._tensors
    assert (d.q, d.out, d.ctx_len) == (q.data_ptr(), out.data_ptr(), lens.data_ptr()) and int(lens[0]) == 7
