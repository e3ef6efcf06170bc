"""quest_decode_static: the fused decode step for callers that cannot allocate device memory
(for example code hosted by a runtime that owns the allocator), which uses a scratch
array inside the library instead of a caller workspace.

Called through the C ABI directly and compared with quest_decode (which takes a
workspace) and with the CPU oracle on two calls in a row; a call that records a device
error reports it through status_out, and the next call starts clean.  This file is
collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import harness as H
import oracle
import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2
STATIC_SCRATCH_BYTES = 16 << 20


def _static_fn():
    lib = q.load()
    fn = lib.quest_decode_static
    V = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(q.QuestCacheDesc), V, ctypes.c_int32, V, V, V, V, V, V]
    fn.restype = ctypes.c_int
    return lib, fn


def _device_cache(w):
    dev = torch.device("cuda")
    cache = q.PagedCache.allocate_meta(w.k_pool.to(dev), w.v_pool.to(dev),
                                       w.block_table.to(dev), w.seq_lens.to(dev),
                                       w.num_q_heads)
    return cache


def _static_call(fn, cache, qd, K, stream):
    B, Hq, Hkv = cache.batch, cache.desc.num_q_heads, cache.num_kv_heads
    out = torch.empty((B, Hq, 128), dtype=torch.float16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, Hkv, K), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, Hkv), dtype=torch.int32, device="cuda")
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.byref(cache.desc), qd.data_ptr(), K, out.data_ptr(), lse.data_ptr(),
            idx.data_ptr(), cnt.data_ptr(), status.data_ptr(), stream)
    torch.cuda.synchronize()
    return rc, out, lse, idx, cnt, status.cpu().tolist()


def test_static_scratch_matches_workspace_path_twice():
    w = wl.build("no_alloc", batch=2, num_q_heads=8, num_kv_heads=4, page_size=16,
                 prefill_lens=[3000, 700], steps=2, budget=256, seed=5, outliers=4)
    cache = _device_cache(w)
    ref = oracle.Cache.from_arrays(w.k_pool.numpy(), w.v_pool.numpy(), w.block_table.numpy(),
                                   w.seq_lens.numpy(), w.num_q_heads)
    oracle.build_meta(ref)
    ws = q.workspace(cache, w.top_k)
    q.build_meta(cache, ws)
    lib, fn = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, Hq, Hkv, K = w.batch, w.num_q_heads, w.num_kv_heads, w.top_k
    for t in range(2):  # two calls in a row through the shared scratch
        qd = w.q[t].cuda().contiguous()
        ref_out, ref_lse = q.decode(cache, qd, K, ws)
        ref_idx = torch.empty((B, Hkv, K), dtype=torch.int32, device="cuda")
        ref_cnt = torch.empty((B, Hkv), dtype=torch.int32, device="cuda")
        q.decode(cache, qd, K, ws, idx_out=ref_idx, count_out=ref_cnt)
        out = torch.empty((B, Hq, 128), dtype=torch.float16, device="cuda")
        lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
        idx = torch.empty((B, Hkv, K), dtype=torch.int32, device="cuda")
        cnt = torch.empty((B, Hkv), dtype=torch.int32, device="cuda")
        status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
        rc = fn(ctypes.byref(cache.desc), qd.data_ptr(), K, out.data_ptr(), lse.data_ptr(),
                idx.data_ptr(), cnt.data_ptr(), status.data_ptr(), stream)
        assert rc == q.QUEST_OK, lib.quest_last_error()
        torch.cuda.synchronize()
        assert int(status[0]) == q.QUEST_OK
        assert torch.equal(cnt, ref_cnt) and torch.equal(idx, ref_idx)
        np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(),
                                   atol=ATOL, rtol=RTOL)
        np.testing.assert_allclose(lse.cpu().numpy(), ref_lse.cpu().numpy(), atol=ATOL, rtol=RTOL)
        # and against the oracle: selection (tie-window rule) and attention
        qh = w.q[t].numpy().astype(np.float32)
        rs = oracle.score(ref, qh)
        ri, rcnt = oracle.topk(ref, rs, K)
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        H.assert_selection(gi, gc, rs, ri, rcnt)
        out_ref, lse_ref = oracle.attend(ref, qh, gi, gc)
        H.assert_attention_close(out, lse, out_ref, lse_ref)
    rc, detail = q.read_status(ws)
    assert rc == q.QUEST_OK, detail


def test_static_scratch_reports_a_device_error_then_starts_clean():
    """A call that meets an unmapped page reports it through status_out; the next call on
    a good cache (through the same array) reports OK and matches quest_decode, so the
    per-call clear really runs.  A batch of 0 writes OK to status_out."""
    w = wl.build("no_alloc_bad", batch=2, num_q_heads=8, num_kv_heads=4, page_size=16,
                 prefill_lens=[300, 100], steps=1, budget=128, seed=6)
    good = _device_cache(w)
    ws = q.workspace(good, w.top_k)
    q.build_meta(good, ws)
    bad = _device_cache(w)
    bad.meta.copy_(good.meta)
    bad.block_table[1, 3] = w.num_phys + 5  # out of the pool; every page of row 1 is kept
    lib, fn = _static_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    K = w.top_k
    qd = w.q[0].cuda().contiguous()
    rc, _, _, _, _, status = _static_call(fn, bad, qd, K, stream)
    assert rc == q.QUEST_OK, lib.quest_last_error()
    assert status[0] == q.QUEST_ERR_BAD_PAGE, status
    rc, out, lse, idx, cnt, status = _static_call(fn, good, qd, K, stream)
    assert rc == q.QUEST_OK and status[0] == q.QUEST_OK, status
    ref_idx = torch.empty_like(idx)
    ref_cnt = torch.empty_like(cnt)
    ref_out, ref_lse = q.decode(good, qd, K, ws, idx_out=ref_idx, count_out=ref_cnt)
    assert torch.equal(idx, ref_idx) and torch.equal(cnt, ref_cnt)
    np.testing.assert_allclose(out.float().cpu().numpy(), ref_out.float().cpu().numpy(),
                               atol=ATOL, rtol=RTOL)
    empty = q.QuestCacheDesc(0, 8, 4, 128, 16, good.max_pages, w.num_phys,
                             good.k_pool.data_ptr(), good.v_pool.data_ptr(),
                             good.meta.data_ptr(), good.block_table.data_ptr(),
                             good.seq_lens.data_ptr())
    status_t = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    rc = fn(ctypes.byref(empty), qd.data_ptr(), K, None, None, None, None,
            status_t.data_ptr(), stream)
    torch.cuda.synchronize()
    assert rc == q.QUEST_OK and status_t.cpu().tolist() == [0, 0, 0, 0]


def test_static_scratch_rejects_oversized_workloads():
    # 64 sequences x 32 heads x 16384 pages of scores alone exceed the 16 MiB scratch
    desc = q.QuestCacheDesc(64, 32, 32, 128, 16, 16384, 16384, 256, 512, 768, 1024, 1280)
    lib, fn = _static_fn()
    assert lib.quest_workspace_size(ctypes.byref(desc), 128, None) > STATIC_SCRATCH_BYTES
    rc = fn(ctypes.byref(desc), 256, 128, 256, None, None, None, None, None)
    assert rc == q.QUEST_ERR_WORKSPACE
    assert b"static scratch" in lib.quest_last_error()
