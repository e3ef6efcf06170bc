"""GPU parity of the chunked-prefill write (quest_prefill) against the CPU oracle, through
the C ABI: the chunk's K/V rows, the page boxes and the lengths must be bit-exact with the
oracle appending the same tokens one at a time ("Guide to Quest", Solution step 1: boxes
formed as pages fill during prefill), and with quest_build_meta over the finished prompt.
"""
import numpy as np
import pytest
import torch

import harness as H
import oracle
import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def chunks_of(w, sizes):
    """The workload's per-step tokens regrouped as chunks [B][n][Hkv][d]."""
    t = 0
    for n in sizes:
        yield (w.k_new[t:t + n].permute(1, 0, 2, 3).contiguous(),
               w.v_new[t:t + n].permute(1, 0, 2, 3).contiguous())
        t += n


def assert_cache_equal(pair):
    assert pair.cache.seq_lens.cpu().tolist() == pair.ref.seq_lens.tolist()
    H.assert_meta_equal(pair)
    kp = pair.cache.k_pool.cpu().numpy()
    vp = pair.cache.v_pool.cpu().numpy()
    P = pair.w.page_size
    for b, p, ph in H.valid_pages(pair.ref):
        n = min(P, int(pair.ref.seq_lens[b]) - p * P)
        np.testing.assert_array_equal(kp[ph, :, :n].astype(np.float32), pair.ref.k_pool[ph, :, :n])
        np.testing.assert_array_equal(vp[ph, :, :n].astype(np.float32), pair.ref.v_pool[ph, :, :n])


GEOMS = [dict(hq=4, hkv=4, P=16), dict(hq=32, hkv=8, P=16), dict(hq=8, hkv=1, P=32),
         dict(hq=24, hkv=12, P=32)]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_chunks_match_token_by_token_append(geom):
    """Ragged starting lengths (mid-page, page-aligned, empty), chunks of 1, 15, 16, 37,
    100 and 3 tokens; compared after every chunk."""
    sizes = [1, 15, 16, 37, 100, 3]
    w = wl.build("prefill", batch=5, num_q_heads=geom["hq"], num_kv_heads=geom["hkv"],
                 page_size=geom["P"], prefill_lens=[30, 0, 47, 64, 5], steps=sum(sizes),
                 budget=128, seed=3, outliers=4)
    pair = H.on_device(w)
    for kc, vc in chunks_of(w, sizes):
        q.prefill(pair.cache, kc.cuda(), vc.cuda(), pair.ws)
        oracle.prefill(pair.ref, kc.numpy(), vc.numpy())
        H.assert_status_ok(pair.ws)
        assert_cache_equal(pair)


@pytest.mark.parametrize("P", [16, 32])
def test_whole_prompt_equals_build_meta(P):
    """A 2000-token prompt written in one chunk into an empty cache gives the boxes
    quest_build_meta computes afterwards, bit for bit, and the oracle's."""
    w = wl.build("prompt", batch=3, num_q_heads=8, num_kv_heads=8, page_size=P,
                 prefill_lens=[0, 0, 0], steps=2000, budget=128, seed=5)
    pair = H.on_device(w)
    pair.cache.meta.fill_(7.0)  # stale boxes must be replaced, not widened
    (kc, vc), = chunks_of(w, [2000])
    q.prefill(pair.cache, kc.cuda(), vc.cuda(), pair.ws)
    oracle.prefill(pair.ref, kc.numpy(), vc.numpy())
    H.assert_status_ok(pair.ws)
    assert_cache_equal(pair)
    written = pair.cache.meta.clone()
    q.build_meta(pair.cache, pair.ws)
    assert torch.equal(written.view(torch.int16), pair.cache.meta.view(torch.int16))


def test_then_decode_matches_oracle():
    """Prefill in chunks, then fused decode steps: the selection and attention rules of
    the decode path hold on the cache the prefill wrote."""
    sizes = [700, 513, 1]
    w = wl.build("prefill_decode", batch=2, num_q_heads=32, num_kv_heads=8, page_size=16,
                 prefill_lens=[0, 33], steps=sum(sizes), budget=256, seed=9)
    pair = H.on_device(w)
    for kc, vc in chunks_of(w, sizes):
        q.prefill(pair.cache, kc.cuda(), vc.cuda(), pair.ws)
        oracle.prefill(pair.ref, kc.numpy(), vc.numpy())
    H.assert_status_ok(pair.ws)
    assert_cache_equal(pair)
    for t in range(3):
        qd = w.q[t].cuda()
        qh = w.q[t].numpy().astype(np.float32)
        ref_scores = oracle.score(pair.ref, qh)
        ref_idx, ref_cnt = oracle.topk(pair.ref, ref_scores, w.top_k)
        idx = torch.empty((2, 8, w.top_k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((2, 8), dtype=torch.int32, device="cuda")
        out, lse = q.decode(pair.cache, qd, w.top_k, pair.ws, idx_out=idx, count_out=cnt)
        H.assert_status_ok(pair.ws)
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        H.assert_selection(gi, gc, ref_scores, ref_idx, ref_cnt)
        out_ref, lse_ref = oracle.attend(pair.ref, qh, gi, gc)
        H.assert_attention_close(out, lse, out_ref, lse_ref)


def test_sequence_without_room_is_reported_and_left_alone():
    """Sequence 0 has 60 of 64 slots filled: an 8-token chunk does not fit, is reported as
    QUEST_ERR_BAD_LENGTH, and leaves its length and boxes as they were; sequence 1 still
    takes the chunk."""
    w = wl.build("full", batch=2, num_q_heads=4, num_kv_heads=4, page_size=16,
                 prefill_lens=[60, 0], steps=4, budget=64, seed=1)
    assert w.max_pages == 4
    pair = H.on_device(w)
    before = pair.cache.meta[0].clone()
    kc = torch.randn(2, 8, 4, 128, generator=torch.Generator().manual_seed(2)).half()
    vc = torch.randn(2, 8, 4, 128, generator=torch.Generator().manual_seed(3)).half()
    q.prefill(pair.cache, kc.cuda(), vc.cuda(), pair.ws)
    rc, _ = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_LENGTH
    assert pair.cache.seq_lens.cpu().tolist() == [60, 8]
    assert torch.equal(pair.cache.meta[0], before)
    ph = int(w.block_table[1, 0])
    np.testing.assert_array_equal(pair.cache.k_pool[ph, :, :8].cpu().numpy(),
                                  kc[1].permute(1, 0, 2).numpy())
    box = pair.cache.meta[1, :, 0].float().cpu()
    keys = kc[1].float().permute(1, 0, 2)  # [Hkv][8][d]
    assert torch.equal(box[:, 0], keys.min(dim=1).values)
    assert torch.equal(box[:, 1], keys.max(dim=1).values)


def test_unmapped_page_is_reported_and_length_kept():
    """A block-table entry outside [0, num_phys) for a page the chunk reaches is reported
    as QUEST_ERR_BAD_PAGE; that sequence's length stays, the other sequence advances."""
    w = wl.build("badpage", batch=2, num_q_heads=4, num_kv_heads=4, page_size=16,
                 prefill_lens=[0, 0], steps=16, budget=64, seed=1)
    pair = H.on_device(w)
    pair.cache.block_table[1, 0] = w.num_phys
    kc = torch.zeros(2, 4, 4, 128, dtype=torch.float16)
    q.prefill(pair.cache, kc.cuda(), kc.cuda(), pair.ws)
    rc, _ = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_PAGE
    assert pair.cache.seq_lens.cpu().tolist() == [4, 0]
