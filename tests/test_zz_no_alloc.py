"""quest_decode_static: the fused decode step for callers that cannot allocate device memory
(for example code hosted by a runtime that owns the allocator), which uses a scratch
array inside the library instead of a caller workspace.

Called through the C ABI directly and compared with quest_decode (which takes a
workspace) on two calls in a row.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def test_static_scratch_matches_workspace_path_twice():
    w = wl.build("no_alloc", batch=2, num_q_heads=8, num_kv_heads=4, page_size=16,
                 prefill_lens=[3000, 700], steps=2, budget=256, seed=5, outliers=4)
    cache = _device_cache(w)
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
    rc, detail = q.read_status(ws)
    assert rc == q.QUEST_OK, detail


def test_static_scratch_rejects_oversized_workloads():
    # 64 sequences x 32 heads x 16384 pages of scores alone exceed the 16 MiB scratch
    desc = q.QuestCacheDesc(64, 32, 32, 128, 16, 16384, 16384, 256, 512, 768, 1024, 1280)
    lib, fn = _static_fn()
    assert lib.quest_workspace_size(ctypes.byref(desc), 128, None) > STATIC_SCRATCH_BYTES
    rc = fn(ctypes.byref(desc), 256, 128, 256, None, None, None, None, None)
    assert rc == q.QUEST_ERR_WORKSPACE
    assert b"static scratch" in lib.quest_last_error()
