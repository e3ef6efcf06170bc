"""GPU parity of every step of the decode path against the CPU oracle, through the C ABI.

Acceptance rules (see harness.py): boxes / appended tokens / lengths / top-K of identical
scores bit-exact; scores within the fp32 reordering bound; selections equal outside the
1e-5 relative tie window of the K-th score; attention |gpu - oracle| <= 2e-3 + 1e-2|oracle|.
"""
import numpy as np
import pytest
import torch

import harness as H
import oracle
import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def small(name="small", batch=3, hq=4, hkv=4, P=16, lens=(300, 1, 77), steps=4, budget=128,
          seed=0, **kw):
    return wl.build(name, batch=batch, num_q_heads=hq, num_kv_heads=hkv, page_size=P,
                    prefill_lens=list(lens), steps=steps, budget=budget, seed=seed, **kw)


GEOMS = [
    dict(hq=4, hkv=4, P=16),
    dict(hq=8, hkv=4, P=16),
    dict(hq=16, hkv=4, P=32),
    dict(hq=32, hkv=4, P=16),
    dict(hq=8, hkv=1, P=32),
]


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_build_meta_bit_exact(geom):
    w = small(lens=(300, 1, 77, 0, 64), batch=5, spare_pages=3, **geom)
    pair = H.on_device(w)
    H.assert_status_ok(pair.ws)
    H.assert_meta_equal(pair)


@pytest.mark.parametrize("geom", GEOMS[:3], ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_append_bit_exact(geom):
    w = small(lens=(30, 0, 47), steps=40, **geom)
    pair = H.on_device(w)
    for t in range(w.steps):
        q.append(pair.cache, w.k_new[t].cuda(), w.v_new[t].cuda(), pair.ws)
        oracle.append(pair.ref, w.k_new[t].numpy(), w.v_new[t].numpy())
    H.assert_status_ok(pair.ws)
    assert pair.cache.seq_lens.cpu().tolist() == pair.ref.seq_lens.tolist()
    H.assert_meta_equal(pair)
    kp = pair.cache.k_pool.cpu().numpy()
    vp = pair.cache.v_pool.cpu().numpy()
    for b, p, ph in H.valid_pages(pair.ref):
        n = min(w.page_size, int(pair.ref.seq_lens[b]) - p * w.page_size)
        np.testing.assert_array_equal(kp[ph, :, :n].astype(np.float32), pair.ref.k_pool[ph, :, :n])
        np.testing.assert_array_equal(vp[ph, :, :n].astype(np.float32), pair.ref.v_pool[ph, :, :n])


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_estimate_within_fp32_reordering(geom):
    w = small(lens=(1000, 1, 333), outliers=4, **geom)
    pair = H.on_device(w)
    qh = w.q[0].numpy().astype(np.float32)
    s = q.estimate(pair.cache, w.q[0].cuda(), pair.ws).cpu().numpy()
    H.assert_status_ok(pair.ws)
    ref = oracle.score(pair.ref, qh)
    H.assert_scores_close(s, ref, H.score_tolerance(pair.ref, qh))


@pytest.mark.parametrize("K", [1, 7, 16, 64, 200])
def test_topk_bit_exact_on_identical_scores(K):
    """Given the oracle's own scores, the selection must be exactly the oracle's."""
    w = small(lens=(16 * 150 - 3, 5, 16 * 40), budget=16 * K)
    pair = H.on_device(w)
    ref = oracle.score(pair.ref, w.q[0].numpy())
    idx, cnt = q.topk(pair.cache, torch.from_numpy(ref).cuda(), K, pair.ws)
    H.assert_status_ok(pair.ws)
    ri, rc = oracle.topk(pair.ref, ref, K)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    assert np.array_equal(gc, rc)
    for b in range(w.batch):
        for g in range(w.num_kv_heads):
            assert gi[b, g, :gc[b, g]].tolist() == sorted(ri[b, g, :rc[b, g]].tolist())
            assert np.all(gi[b, g, gc[b, g]:] == -1)


def test_topk_exact_ties_go_to_lower_index():
    w = small(lens=(16 * 500,), batch=1, hq=2, hkv=2)
    pair = H.on_device(w)
    rng = np.random.default_rng(1)
    scores = np.full((1, 2, w.block_table.shape[1]), -np.inf, np.float32)
    scores[0, 0, :500] = rng.integers(0, 5, 500).astype(np.float32)   # heavy ties
    scores[0, 1, :500] = 1.5                                           # all tied
    for K in (1, 37, 100, 499):
        idx, cnt = q.topk(pair.cache, torch.from_numpy(scores).cuda(), K, pair.ws)
        ri, rc = oracle.topk(pair.ref, scores, K)
        for g in range(2):
            assert idx[0, g, :K].cpu().tolist() == sorted(ri[0, g, :K].tolist())
    H.assert_status_ok(pair.ws)


@pytest.mark.parametrize("n", [1024, 1025, 2048, 2049, 3000, 4096, 4097])
def test_topk_row_sizes(n):
    """Rows around the register-resident selection's size classes (4, 8 and 16 keys per
    thread, then the shared-memory path), with outliers and exact ties."""
    w = small(lens=(16 * n,), batch=1, hq=2, hkv=2, steps=0, budget=16 * 128)
    pair = H.on_device(w, build_meta=False)
    rng = np.random.default_rng(n)
    scores = np.full((1, 2, w.block_table.shape[1]), -np.inf, np.float32)
    scores[0, 0, :n] = rng.normal(200.0, 30.0, n).astype(np.float32)
    scores[0, 0, rng.integers(0, n, 4)] = [5e3, 6e3, -7e3, 1e6]
    scores[0, 1, :n] = rng.integers(0, 9, n).astype(np.float32) * 0.5  # heavy ties
    for K in (1, 128, n // 2, n - 1):
        idx, cnt = q.topk(pair.cache, torch.from_numpy(scores).cuda(), K, pair.ws)
        ri, rc = oracle.topk(pair.ref, scores, K)
        for g in range(2):
            assert int(cnt[0, g]) == rc[0, g]
            assert idx[0, g, :K].cpu().tolist() == sorted(ri[0, g, :K].tolist()), (K, g)
    H.assert_status_ok(pair.ws)


def test_topk_near_ties_over_a_wide_range():
    """Distinct keys a few ulps apart at the threshold, in a row whose range spans the
    whole float line: the two histogram levels cannot separate them, the radix select
    must."""
    n = 2000
    w = small(lens=(16 * n,), batch=1, hq=1, hkv=1, steps=0, budget=16 * 100)
    pair = H.on_device(w, build_meta=False)
    scores = np.full((1, 1, w.block_table.shape[1]), -np.inf, np.float32)
    base = np.float32(1.0)
    near = np.nextafter(base, np.float32(2.0)) - base
    scores[0, 0, :n] = np.float32(-3.0e38)
    scores[0, 0, 1] = np.float32(3.0e38)
    scores[0, 0, 10:310] = base + near * np.arange(300, dtype=np.float32)[::-1]
    for K in (50, 100, 200):
        idx, cnt = q.topk(pair.cache, torch.from_numpy(scores).cuda(), K, pair.ws)
        ri, rc = oracle.topk(pair.ref, scores, K)
        assert idx[0, 0, :K].cpu().tolist() == sorted(ri[0, 0, :K].tolist()), K
    H.assert_status_ok(pair.ws)


@pytest.mark.parametrize("sink,local", [(2, 2), (0, 3), (4, 0), (8, 8)])
def test_topk_sink_and_local_pages(sink, local):
    """Sink and local pages ("Guide to Quest", Solution step 3 / Implementation step 2):
    the first `sink` and last `local` pages of a long sequence are always kept, the rest of
    the budget goes to the best of the others; short sequences keep everything."""
    w = small(lens=(16 * 300 - 7, 16 * 12, 16 * 64), batch=3, hq=4, hkv=2)
    pair = H.on_device(w, build_meta=False)
    rng = np.random.default_rng(sink * 10 + local)
    scores = np.full((3, 2, w.block_table.shape[1]), -np.inf, np.float32)
    for b, L in enumerate((16 * 300 - 7, 16 * 12, 16 * 64)):
        n = wl.pages_for(L, 16)
        scores[b, :, :n] = rng.standard_normal((2, n)).astype(np.float32)
        scores[b, 1, :n] = np.round(scores[b, 1, :n])          # exact ties
        scores[b, 0, n - 1] = -50.0                              # a weak last page
    for K in (16, 40):
        o = q.opts(sink_pages=sink, local_pages=local)
        idx, cnt = q.topk(pair.cache, torch.from_numpy(scores).cuda(), K, pair.ws, o)
        ri, rc = oracle.topk(pair.ref, scores, K, sink, local)
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        assert np.array_equal(gc, rc)
        for b in range(3):
            for g in range(2):
                assert gi[b, g, :gc[b, g]].tolist() == sorted(ri[b, g, :rc[b, g]].tolist())
    H.assert_status_ok(pair.ws)


@pytest.mark.parametrize("cs", [0, 1, 8, "stream"])
def test_fused_step_with_sink_and_local_pages(cs):
    w = small(lens=(2500, 1, 700, 16 * 9), batch=4, steps=2, hq=8, hkv=4, budget=256,
              outliers=4)
    pair = H.on_device(w)
    if cs == "stream":
        o = q.opts(path=q.QUEST_PATH_STREAM, sink_pages=2, local_pages=2)
    else:
        o = q.opts(cluster_size=cs, sink_pages=2, local_pages=2)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o, one_launch=True, sink=2, local=2,
                               check_cache=(t == w.steps - 1))


def test_estimate_heads_and_group_max():
    """Per-query-head bounds within fp32 reordering of the oracle's; their group maximum is
    bit-identical to quest_estimate."""
    w = small(lens=(1000, 1, 333), hq=8, hkv=2, outliers=4)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    sh = q.estimate_heads(pair.cache, qd, pair.ws).cpu().numpy()
    sk = q.estimate(pair.cache, qd, pair.ws).cpu().numpy()
    H.assert_status_ok(pair.ws)
    qh = w.q[0].numpy().astype(np.float32)
    ref = oracle.score_heads(pair.ref, qh)
    tol = H.score_tolerance(pair.ref, qh)  # [B][Hkv][max_pages], valid for every head of g
    tol_h = np.repeat(tol, 4, axis=1)
    H.assert_scores_close(sh, ref, tol_h)
    G = 4
    for g in range(2):
        np.testing.assert_array_equal(sh[:, g * G:(g + 1) * G].max(axis=1), sk[:, g])


@pytest.mark.parametrize("K", [1, 9, 40])
def test_topk_union_matches_oracle_on_identical_scores(K):
    """Union form ("Guide to Quest", Best Practices step 2): given the oracle's own
    per-head scores the union must be exactly the oracle's."""
    w = small(lens=(16 * 200 - 3, 16 * 6, 16 * 41), batch=3, hq=8, hkv=2, budget=16 * K)
    pair = H.on_device(w)
    sh = oracle.score_heads(pair.ref, w.q[0].numpy().astype(np.float32))
    sh[0, 1] = np.where(np.isfinite(sh[0, 1]), np.round(sh[0, 1] / 50.0), sh[0, 1])  # ties
    o = q.opts(gqa_union=True)
    idx, cnt = q.topk(pair.cache, torch.from_numpy(sh).cuda(), K, pair.ws, o)
    H.assert_status_ok(pair.ws)
    ri, rc = oracle.topk_union(pair.ref, sh, K)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    assert gi.shape == ri.shape
    assert np.array_equal(gc, rc)
    for b in range(3):
        for g in range(2):
            assert gi[b, g, :gc[b, g]].tolist() == ri[b, g, :rc[b, g]].tolist()
            assert np.all(gi[b, g, gc[b, g]:] == -1)


def test_union_chain_matches_oracle():
    """Per-head bounds, union selection and sparse decode over the union (rows of G*K),
    against the oracle: swaps only among pages near some head's K-th score; attention over
    the GPU's union."""
    w = small(lens=(3000, 700, 16 * 9), batch=3, hq=8, hkv=2, budget=256, outliers=4,
              steps=1)
    pair = H.on_device(w)
    K = w.top_k
    G = 4
    qd = w.q[0].cuda()
    qh = w.q[0].numpy().astype(np.float32)
    sh = q.estimate_heads(pair.cache, qd, pair.ws)
    idx, cnt = q.topk(pair.cache, sh, K, pair.ws, q.opts(gqa_union=True))
    cap = idx.shape[2]
    ws_u = q.workspace(pair.cache, cap)  # partials for rows of G*K pages
    out, lse = q.sparse_decode(pair.cache, qd, idx, cnt, cap, ws_u)
    H.assert_status_ok(pair.ws)
    H.assert_status_ok(ws_u)
    ref_sh = oracle.score_heads(pair.ref, qh)
    ri, rc = oracle.topk_union(pair.ref, ref_sh, K)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for b in range(3):
        n = wl.pages_for(int(pair.ref.seq_lens[b]), 16)
        for g in range(2):
            got = set(gi[b, g, :gc[b, g]].tolist())
            want = set(ri[b, g, :rc[b, g]].tolist())
            window = set()
            if n > K:
                for h in range(g * G, (g + 1) * G):
                    row = ref_sh[b, h, :n]
                    sk = float(np.sort(row)[::-1][K - 1])
                    window |= {p for p in range(n) if abs(float(row[p]) - sk) <= H.TIE_REL * abs(sk)}
            assert got - window == want - window, (b, g)
    out_ref, lse_ref = oracle.attend(pair.ref, qh, gi, gc)
    H.assert_attention_close(out, lse, out_ref, lse_ref)


def test_topk_at_max_pages():
    """The largest supported row: 16384 pages."""
    n = q.QUEST_MAX_PAGES
    w = small(lens=(16 * n,), batch=1, hq=1, hkv=1, steps=0, budget=16 * 512)
    pair = H.on_device(w, build_meta=False)
    rng = np.random.default_rng(2)
    scores = rng.standard_normal((1, 1, n)).astype(np.float32)
    scores[0, 0, ::7] = scores[0, 0, 3]  # some exact ties
    for K in (1, 512, n - 1, n):
        idx, cnt = q.topk(pair.cache, torch.from_numpy(scores).cuda(), K, pair.ws)
        ri, rc = oracle.topk(pair.ref, scores, K)
        assert int(cnt[0, 0]) == rc[0, 0]
        assert idx[0, 0, :K].cpu().tolist() == sorted(ri[0, 0, :K].tolist())
    H.assert_status_ok(pair.ws)


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
@pytest.mark.parametrize("pps", [0, 1, 5])
def test_sparse_decode_on_oracle_selection(geom, pps):
    w = small(lens=(900, 1, 333, 0), batch=4, **geom)
    pair = H.on_device(w, opts=q.opts(pages_per_split=pps))
    qh = w.q[0].numpy()
    ref_s = oracle.score(pair.ref, qh)
    ri, rc = oracle.topk(pair.ref, ref_s, w.top_k)
    out, lse = q.sparse_decode(pair.cache, w.q[0].cuda(), torch.from_numpy(ri).cuda(),
                               torch.from_numpy(rc).cuda(), w.top_k, pair.ws,
                               q.opts(pages_per_split=pps))
    H.assert_status_ok(pair.ws)
    ro, rl = oracle.attend(pair.ref, qh, ri, rc)
    H.assert_attention_close(out, lse, ro, rl)


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_dense_decode_matches_oracle(geom):
    w = small(lens=(2000, 1, 333, 0), batch=4, **geom)
    pair = H.on_device(w)
    qh = w.q[0].numpy()
    out, lse = q.dense_decode(pair.cache, w.q[0].cuda(), pair.ws)
    H.assert_status_ok(pair.ws)
    ro, rl = oracle.dense(pair.ref, qh)
    H.assert_attention_close(out, lse, ro, rl)


@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
@pytest.mark.parametrize("fused", [True, False], ids=["fused", "chain"])
def test_decode_steps_match_oracle(geom, fused):
    w = small(lens=(1500, 1, 333, 0, 16 * 30), batch=5, steps=6, outliers=4, **geom)
    pair = H.on_device(w)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, fused=fused)


ALL_PATHS = [q.QUEST_PATH_FUSED, q.QUEST_PATH_CHAIN, q.QUEST_PATH_STREAM]
ALL_PATH_IDS = ["fused", "chain", "stream"]


@pytest.mark.parametrize("path", ALL_PATHS, ids=ALL_PATH_IDS)
@pytest.mark.parametrize("geom", GEOMS, ids=lambda g: f"hq{g['hq']}_hkv{g['hkv']}_p{g['P']}")
def test_one_launch_step_matches_oracle(geom, path):
    """quest_decode_step through each path (the cluster kernel and the stream kernel with
    the append folded in, and the chain of separate kernels): boxes, pools, lengths,
    selection and attention all match the oracle step after step (pages open and fill)."""
    w = small(lens=(1500, 1, 333, 0, 16 * 30 - 2), batch=5, steps=20, outliers=4, **geom)
    pair = H.on_device(w)
    o = q.opts(path=path)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o, one_launch=True,
                               check_cache=(t % 5 == 4))


def test_decode_path_choice():
    """Short rows with a resident cluster per pair take the one launch, long rows and
    forced paths take what they are given."""
    w = wl.tiny(seed=0)
    pair = H.on_device(w)
    assert q.decode_path(pair.cache, w.top_k) == q.QUEST_PATH_FUSED
    assert q.decode_path(pair.cache, w.top_k, q.opts(path=q.QUEST_PATH_CHAIN)) == \
        q.QUEST_PATH_CHAIN
    long_w = small(lens=(20000, 3000), batch=2, hq=8, hkv=8, steps=1, budget=512)
    long_pair = H.on_device(long_w)
    assert long_pair.cache.max_pages >= 1024
    assert q.decode_path(long_pair.cache, long_w.top_k) == q.QUEST_PATH_CHAIN
    assert q.decode_path(long_pair.cache, long_w.top_k, q.opts(cluster_size=2)) == \
        q.QUEST_PATH_FUSED
    assert q.decode_path(long_pair.cache, long_w.top_k, n_layers=4) == q.QUEST_PATH_CHAIN


def test_chain_path_window_and_no_selection_outputs():
    """The chain path honours sink / local pages and runs without idx_out / count_out (the
    selection then stays in the workspace)."""
    w = small(lens=(3000, 700), batch=2, hq=8, hkv=4, steps=2, budget=256, outliers=4)
    pair = H.on_device(w)
    o = q.opts(path=q.QUEST_PATH_CHAIN, sink_pages=2, local_pages=3)
    H.run_step_and_compare(pair, 0, w.top_k, opts=o, one_launch=True, sink=2, local=3,
                           check_cache=True)
    out, lse = q.decode_step(pair.cache, w.q[1].cuda(), w.k_new[1].cuda(), w.v_new[1].cuda(),
                             w.top_k, pair.ws, o)
    oracle.append(pair.ref, w.k_new[1].numpy(), w.v_new[1].numpy())
    H.assert_status_ok(pair.ws)
    qh = w.q[1].numpy().astype(np.float32)
    ref_scores = oracle.score(pair.ref, qh)
    ri, rc = oracle.topk(pair.ref, ref_scores, w.top_k, 2, 3)
    out_ref, lse_ref = oracle.attend(pair.ref, qh, ri, rc)
    H.assert_attention_close(out, lse, out_ref, lse_ref)


def test_tiny_config():
    w = wl.tiny(seed=0)
    pair = H.on_device(w)
    H.run_step_and_compare(pair, 0, w.top_k, one_launch=True, check_cache=True)


def test_stream_cta_counts_agree():
    """The stream kernel with any number of CTAs (one CTA doing every pair's scoring,
    selection, decode and merge; a few; one per SM) gives bit-identical selections and
    outputs: each decode piece's partial and the merge order do not depend on which CTA
    ran them."""
    w = small(lens=(4000, 2100, 5000), batch=3, hq=8, hkv=4, budget=512, outliers=4)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    idx0 = torch.empty((3, 4, w.top_k), dtype=torch.int32, device="cuda")
    cnt0 = torch.empty((3, 4), dtype=torch.int32, device="cuda")
    o = q.opts(path=q.QUEST_PATH_STREAM)
    base, base_lse = q.decode(pair.cache, qd, w.top_k, pair.ws, o, idx_out=idx0, count_out=cnt0)
    H.assert_status_ok(pair.ws)
    qh = w.q[0].numpy().astype(np.float32)
    ref_scores = oracle.score(pair.ref, qh)
    ri, rc = oracle.topk(pair.ref, ref_scores, w.top_k)
    H.assert_selection(idx0.cpu().numpy(), cnt0.cpu().numpy(), ref_scores, ri, rc)
    ro, rl = oracle.attend(pair.ref, qh, idx0.cpu().numpy(), cnt0.cpu().numpy())
    H.assert_attention_close(base, base_lse, ro, rl)
    for ctas in [1, 2, 3, 7, 300]:
        idx = torch.empty_like(idx0)
        cnt = torch.empty_like(cnt0)
        out, lse = q.decode(pair.cache, qd, w.top_k, pair.ws,
                            q.opts(path=q.QUEST_PATH_STREAM, max_ctas=ctas),
                            idx_out=idx, count_out=cnt)
        assert torch.equal(idx, idx0) and torch.equal(cnt, cnt0), ctas
        assert torch.equal(out, base) and torch.equal(lse, base_lse), ctas
    H.assert_status_ok(pair.ws)


@pytest.mark.parametrize("cs", [0, 1, 2, 3, 4, 5, 8, 9, 12, 16])
def test_every_cluster_size_matches_oracle(cs):
    """The fused step with clusters of 1..16 CTAs per (sequence, kv head); 0 = automatic."""
    w = small(lens=(2500, 1, 700, 0, 16 * 9), batch=5, steps=3, hq=8, hkv=4, budget=256, outliers=4)
    pair = H.on_device(w)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=q.opts(cluster_size=cs), one_launch=True,
                               check_cache=(t == w.steps - 1))


def test_stream_variant_matches_cluster_variant():
    w = small(lens=(4000, 2100, 5000), batch=3, hq=8, hkv=4, budget=512, outliers=4)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    idx0 = torch.empty((3, 4, w.top_k), dtype=torch.int32, device="cuda")
    cnt0 = torch.empty((3, 4), dtype=torch.int32, device="cuda")
    base, base_lse = q.decode(pair.cache, qd, w.top_k, pair.ws, q.opts(path=q.QUEST_PATH_FUSED),
                              idx_out=idx0, count_out=cnt0)
    idx = torch.empty_like(idx0)
    cnt = torch.empty_like(cnt0)
    out, lse = q.decode(pair.cache, qd, w.top_k, pair.ws, q.opts(path=q.QUEST_PATH_STREAM),
                        idx_out=idx, count_out=cnt)
    H.assert_status_ok(pair.ws)
    assert torch.equal(idx, idx0) and torch.equal(cnt, cnt0)
    torch.testing.assert_close(out.float(), base.float(), atol=2e-3, rtol=0)
    torch.testing.assert_close(lse, base_lse, atol=1e-4, rtol=0)


@pytest.mark.parametrize("cs", [0, 1, 3, 16, "stream"])
def test_fused_step_long_rows(cs):
    """Rows of 1.2K-3.2K pages in the one-launch steps, two decode steps."""
    w = small(lens=(33000, 20000, 51000), batch=3, hq=8, hkv=4, steps=2, budget=2048,
              outliers=4, needles_per_head=2)
    pair = H.on_device(w)
    o = q.opts(path=q.QUEST_PATH_STREAM) if cs == "stream" else q.opts(cluster_size=cs)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o, one_launch=True, check_needles=True)


def test_trace_records_a_timeline():
    w = small(lens=(3000, 700), batch=2, budget=256)
    pair = H.on_device(w)
    cap = 64 * 16 * w.batch * w.num_kv_heads  # 64 records per CTA, at most 16 CTAs per pair
    tr = torch.zeros(1 + 2 * cap, dtype=torch.int64, device="cuda")
    q.decode(pair.cache, w.q[0].cuda(), w.top_k, pair.ws, q.opts(trace=tr))
    H.assert_status_ok(pair.ws)
    rec = tr[1:].view(cap, 2).cpu().numpy()
    rec = rec[rec[:, 0] != 0]
    assert len(rec) > 0
    t, info = rec[:, 0], rec[:, 1].astype(np.uint64)
    ev = (info >> np.uint64(24)) & np.uint64(0xff)
    kinds = set(int(e) for e in ev)
    assert {1, 2, 20, 21, 22, 23, 24, 25, 26} <= kinds
    # one selection and one merge per (b, g), by the leader of its cluster
    assert int((ev == 22).sum()) == w.batch * w.num_kv_heads
    assert int((ev == 26).sum()) == w.batch * w.num_kv_heads
    assert (t.max() - t.min()) < 1e9


def test_stream_trace_records_a_timeline():
    """The stream kernel's timeline: every CTA starts and exits; one selection and one
    merge per (b, g), each by some CTA's selector team."""
    w = small(lens=(3000, 700), batch=2, budget=256)
    pair = H.on_device(w)
    cap = 256 * 160  # 256 records per CTA, at most one CTA per SM
    tr = torch.zeros(1 + 2 * cap, dtype=torch.int64, device="cuda")
    q.decode(pair.cache, w.q[0].cuda(), w.top_k, pair.ws,
             q.opts(trace=tr, path=q.QUEST_PATH_STREAM))
    H.assert_status_ok(pair.ws)
    rec = tr[1:].view(cap, 2).cpu().numpy()
    rec = rec[rec[:, 0] != 0]
    t, info = rec[:, 0], rec[:, 1].astype(np.uint64)
    ev = (info >> np.uint64(24)) & np.uint64(0xff)
    ctas = (info >> np.uint64(32)) & np.uint64(0xffff)
    n_ctas = len(set(int(c) for c in ctas[ev == 1]))
    assert n_ctas >= 1 and int((ev == 2).sum()) == n_ctas
    assert int((ev == 8).sum()) == w.batch * w.num_kv_heads    # selections done
    assert int((ev == 10).sum()) == w.batch * w.num_kv_heads   # merges done
    assert (t.max() - t.min()) < 1e9


def test_fused_equals_chain():
    """The fused step and the three-call chain select the same pages (same score
    arithmetic) and agree up to split-merge rounding."""
    w = small(lens=(3000, 700), batch=2, hq=8, hkv=4, budget=256, outliers=4)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    i1 = torch.empty((2, 4, w.top_k), dtype=torch.int32, device="cuda")
    c1 = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    o1, l1 = q.decode(pair.cache, qd, w.top_k, pair.ws, idx_out=i1, count_out=c1)
    s = q.estimate(pair.cache, qd, pair.ws)
    idx, cnt = q.topk(pair.cache, s, w.top_k, pair.ws)
    o2, l2 = q.sparse_decode(pair.cache, qd, idx, cnt, w.top_k, pair.ws)
    H.assert_status_ok(pair.ws)
    assert torch.equal(i1, idx) and torch.equal(c1, cnt)
    torch.testing.assert_close(o1.float(), o2.float(), atol=2e-3, rtol=0)
    torch.testing.assert_close(l1, l2, atol=1e-4, rtol=0)


def test_split_invariance_and_repeatability():
    w = small(lens=(5000, 2100), batch=2, hq=8, hkv=2, budget=1024, outliers=4)
    pair = H.on_device(w, top_k=w.top_k, opts=q.opts(pages_per_split=1))
    qd = w.q[0].cuda()
    base, base_lse = q.decode(pair.cache, qd, w.top_k, pair.ws)
    again, again_lse = q.decode(pair.cache, qd, w.top_k, pair.ws)
    assert torch.equal(base, again) and torch.equal(base_lse, again_lse)
    for pps, stp in [(1, 16), (3, 64), (8, 128), (32, 1000), (64, 7)]:
        o = q.opts(pages_per_split=pps, score_tile_pages=stp)
        out, lse = q.decode(pair.cache, qd, w.top_k, pair.ws, o)
        torch.testing.assert_close(out.float(), base.float(), atol=2e-3, rtol=0)
        torch.testing.assert_close(lse, base_lse, atol=1e-4, rtol=0)
    H.assert_status_ok(pair.ws)


def test_workspace_reuse_many_calls():
    w = small(lens=(4000, 100, 2500), budget=512)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    first, _ = q.decode(pair.cache, qd, w.top_k, pair.ws)
    for _ in range(50):
        out, _ = q.decode(pair.cache, qd, w.top_k, pair.ws)
    H.assert_status_ok(pair.ws)
    assert torch.equal(first, out)
    # the header counters are back to zero
    hdr = pair.ws[:32].view(torch.int32).cpu().tolist()
    assert hdr[4] == 0 and hdr[5] == 0
    # so they are after one-launch steps through the cluster kernel and the stream kernel
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, one_launch=True)
    so = q.opts(path=q.QUEST_PATH_STREAM)
    for _ in range(5):
        out_s, _ = q.decode(pair.cache, qd, w.top_k, pair.ws, so)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=so, one_launch=True)
    H.assert_status_ok(pair.ws)
    hdr = pair.ws[:32].view(torch.int32).cpu().tolist()
    assert hdr[4] == 0 and hdr[5] == 0
    # and so are the per-pair arrival counters and selection flags (the first three
    # arrays after the header)
    nbg = w.batch * w.num_kv_heads
    ctr = pair.ws[256:256 + 3 * 256 + 4 * nbg].view(torch.int32).cpu().numpy()
    assert not ctr.any()


def test_planted_needles_selected_on_gpu():
    w = wl.build("needles", batch=2, num_q_heads=8, num_kv_heads=8, page_size=16,
                 prefill_lens=[8192, 5000], steps=4, budget=512, seed=3, outliers=4,
                 needles_per_head=8, needle_mode="direction")
    pair = H.on_device(w)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, check_needles=True)


@pytest.mark.parametrize("path", ALL_PATHS, ids=ALL_PATH_IDS)
def test_empty_and_single_token_sequences(path):
    w = small(lens=(0, 1, 0), steps=2)
    pair = H.on_device(w)
    qd = w.q[0].cuda()
    o = q.opts(path=path)
    idx = torch.empty((3, w.num_kv_heads, w.top_k), dtype=torch.int32, device="cuda")
    cnt = torch.empty((3, w.num_kv_heads), dtype=torch.int32, device="cuda")
    out, lse = q.decode(pair.cache, qd, w.top_k, pair.ws, o, idx_out=idx, count_out=cnt)
    H.assert_status_ok(pair.ws)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    assert torch.all(cnt[0] == 0) and torch.all(idx[0] == -1) and torch.all(cnt[1] == 1)
    ro, rl = oracle.dense(pair.ref, w.q[0].numpy())
    H.assert_attention_close(out, lse, ro, rl)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o)
    for t in range(w.steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o, one_launch=True, check_cache=True)


# ---------------------------------------------------------------- device-side faults
# Every fault below is caught by the kernels' own bounds checks (they skip the access and
# record a status); nothing here faults, traps or hangs the GPU.

def test_bad_block_table_entry_is_reported():
    # sequence 1 has 7 pages and top-K keeps 8, so every page (and the bad entry) is read
    w = small(lens=(300, 100), batch=2)
    bt = w.block_table.clone()
    bt[1, 3] = w.num_phys + 5          # out of the pool
    w.block_table = bt
    pair = H.on_device(w, build_meta=False)
    q.build_meta(pair.cache, pair.ws)
    rc, detail = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_PAGE and detail[0] == 1 and detail[1] == 3
    for path in ALL_PATHS:
        q.workspace_init(pair.ws)
        q.decode(pair.cache, w.q[0].cuda(), w.top_k, pair.ws, q.opts(path=path))
        rc, detail = q.read_status(pair.ws)
        assert rc == q.QUEST_ERR_BAD_PAGE, path


def test_bad_lengths_are_reported():
    w = small(lens=(300,), batch=1, steps=1)
    pair = H.on_device(w)
    cap = w.block_table.shape[1] * w.page_size
    pair.cache.seq_lens.fill_(cap)                 # full row: append has no room
    q.append(pair.cache, w.q[0, :, :4].contiguous().cuda(), w.q[0, :, :4].contiguous().cuda(),
             pair.ws)
    rc, _ = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_LENGTH
    assert int(pair.cache.seq_lens[0]) == cap      # untouched
    pair.cache.seq_lens.fill_(cap + 1)             # beyond the row
    for path in ALL_PATHS:
        q.workspace_init(pair.ws)
        q.decode(pair.cache, w.q[0].cuda(), w.top_k, pair.ws, q.opts(path=path))
        rc, _ = q.read_status(pair.ws)
        assert rc == q.QUEST_ERR_BAD_LENGTH, path


@pytest.mark.parametrize("path", ALL_PATHS, ids=ALL_PATH_IDS)
def test_step_without_room_or_page_is_reported(path):
    """A decode step whose token has no room (full row) or whose next page is unmapped
    reports it and leaves the length alone, through either path."""
    o = q.opts(path=path)
    w = small(lens=(32,), batch=1, steps=1)
    pair = H.on_device(w)
    cap = pair.cache.max_pages * w.page_size
    kn, vn = w.k_new[0].cuda(), w.v_new[0].cuda()
    pair.cache.seq_lens.fill_(cap)                      # full row
    q.decode_step(pair.cache, w.q[0].cuda(), kn, vn, w.top_k, pair.ws, o)
    rc, _ = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_LENGTH
    assert int(pair.cache.seq_lens[0]) == cap
    q.workspace_init(pair.ws)
    pair.cache.seq_lens.fill_(32)                       # next token opens page 2 ...
    pair.cache.block_table[0, 2] = w.num_phys + 7       # ... which points outside the pool
    q.decode_step(pair.cache, w.q[0].cuda(), kn, vn, w.top_k, pair.ws, o)
    rc, detail = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_PAGE and detail[0] == 0 and detail[1] == 2
    assert int(pair.cache.seq_lens[0]) == 32


def test_bad_selection_is_reported():
    w = small(lens=(300,), batch=1)
    pair = H.on_device(w)
    idx = torch.full((1, 4, w.top_k), 2, dtype=torch.int32, device="cuda")
    idx[0, 1, 0] = 1000                            # past the sequence's pages
    cnt = torch.full((1, 4), 3, dtype=torch.int32, device="cuda")
    q.sparse_decode(pair.cache, w.q[0].cuda(), idx, cnt, w.top_k, pair.ws)
    rc, detail = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_SELECTION and detail[1] == 1000
    cnt.fill_(w.top_k + 1)                         # count above top_k
    q.workspace_init(pair.ws)
    q.sparse_decode(pair.cache, w.q[0].cuda(), idx, cnt, w.top_k, pair.ws)
    rc, _ = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_BAD_SELECTION


@pytest.mark.parametrize("path", [q.QUEST_PATH_FUSED, q.QUEST_PATH_STREAM], ids=["fused", "stream"])
def test_withheld_selection_times_out_and_context_survives(path):
    """A flag that nothing sets: every decode item's bounded wait runs out (20 ms), the
    call reports QUEST_ERR_TIMEOUT, and the next normal call works."""
    w = small(lens=(3000, 2000), batch=2, budget=256)
    pair = H.on_device(w)
    o = q.opts(debug_flags=q.QUEST_DEBUG_WITHHOLD_SELECTION, wait_limit_ns=20_000_000, path=path)
    q.decode(pair.cache, w.q[0].cuda(), w.top_k, pair.ws, o)
    rc, detail = q.read_status(pair.ws)
    assert rc == q.QUEST_ERR_TIMEOUT
    q.workspace_init(pair.ws)
    H.run_step_and_compare(pair, 0, w.top_k, opts=q.opts(path=path))


@pytest.mark.parametrize("path", [q.QUEST_PATH_AUTO, q.QUEST_PATH_STREAM], ids=["auto", "stream"])
def test_decode_plan_matches_calls(path):
    """A DecodePlan (arguments checked once) issues the same C calls as decode_step /
    decode: two copies of one workload stepped side by side give bit-identical outputs,
    selections, boxes and lengths; a q of the wrong shape is refused before any launch."""
    w = small(lens=(3000, 700, 1), batch=3, hq=8, hkv=4, budget=256, outliers=4, steps=3)
    a, b = H.on_device(w), H.on_device(w)
    o = q.opts(path=path)
    shape_i, shape_c = (3, 4, w.top_k), (3, 4)
    ia = torch.empty(shape_i, dtype=torch.int32, device="cuda")
    ca = torch.empty(shape_c, dtype=torch.int32, device="cuda")
    ib = torch.empty_like(ia)
    cb = torch.empty_like(ca)
    plan = q.DecodePlan(b.cache, w.top_k, b.ws, o, idx_out=ib, count_out=cb)
    for t in range(w.steps):
        qd, kn, vn = w.q[t].cuda(), w.k_new[t].cuda(), w.v_new[t].cuda()
        oa, la = q.decode_step(a.cache, qd, kn, vn, w.top_k, a.ws, o, idx_out=ia, count_out=ca)
        ob, lb = plan.step(qd, kn, vn)
        assert torch.equal(oa, ob) and torch.equal(la, lb), t
        assert torch.equal(ia, ib) and torch.equal(ca, cb), t
    oa, la = q.decode(a.cache, w.q[0].cuda(), w.top_k, a.ws, o)
    ob, lb = plan.decode(w.q[0].cuda())
    assert torch.equal(oa, ob) and torch.equal(la, lb)
    H.assert_status_ok(a.ws)
    H.assert_status_ok(b.ws)
    assert torch.equal(a.cache.meta, b.cache.meta)
    assert torch.equal(a.cache.seq_lens, b.cache.seq_lens)
    with pytest.raises(ValueError):
        plan.decode(torch.zeros((3, 4, 128), dtype=torch.float16, device="cuda"))


@pytest.mark.parametrize("cs", [1, 2])
@pytest.mark.parametrize("ctas", [1, 3])
def test_cluster_pair_loop_with_few_clusters(cs, ctas):
    """The one-launch cluster kernel is persistent over pairs.  With max_ctas capping the
    grid at 1 or 3 clusters of 1 or 2 CTAs, the 12 (sequence, kv head) pairs run through
    each cluster's pair loop: two appending steps match the oracle (selection, attention,
    and on the last step boxes, rows and lengths), and the capped launch gives the same
    selections and outputs, bit for bit, as the uncapped one."""
    w = small(lens=(3000, 700, 1), batch=3, hq=8, hkv=4, budget=256, outliers=4, steps=2)
    a, b = H.on_device(w), H.on_device(w)
    o_cap = q.opts(path=q.QUEST_PATH_FUSED, cluster_size=cs, max_ctas=ctas)
    o_all = q.opts(path=q.QUEST_PATH_FUSED, cluster_size=cs)
    for t in range(w.steps):
        H.run_step_and_compare(a, t, w.top_k, opts=o_cap, one_launch=True,
                               check_cache=(t == w.steps - 1))
        H.run_step_and_compare(b, t, w.top_k, opts=o_all, one_launch=True)
    assert torch.equal(a.cache.meta, b.cache.meta)
    assert torch.equal(a.cache.seq_lens, b.cache.seq_lens)
    qd = w.q[0].cuda()
    ia = torch.empty((3, 4, w.top_k), dtype=torch.int32, device="cuda")
    ca = torch.empty((3, 4), dtype=torch.int32, device="cuda")
    ib, cb = torch.empty_like(ia), torch.empty_like(ca)
    oa, la = q.decode(a.cache, qd, w.top_k, a.ws, o_cap, idx_out=ia, count_out=ca)
    ob, lb = q.decode(b.cache, qd, w.top_k, b.ws, o_all, idx_out=ib, count_out=cb)
    H.assert_status_ok(a.ws)
    assert torch.equal(ia, ib) and torch.equal(ca, cb)
    assert torch.equal(oa, ob) and torch.equal(la, lb)


def test_chain_launch_count_follows_the_work_item_rule():
    """On the chain, a call on short MHA rows with few decode work items selects inside the
    sparse decode (two launches); GQA, or many work items, keep the top-K kernel (three).
    All match the oracle."""
    few = small(lens=(3000, 700), batch=2, hq=4, hkv=4, budget=256, outliers=4, steps=1)
    gqa = small(lens=(3000, 700), batch=2, hq=8, hkv=4, budget=256, outliers=4, steps=1)
    many = wl.build("many_pairs", batch=8, num_q_heads=64, num_kv_heads=64, page_size=16,
                    prefill_lens=[2000 + 37 * i for i in range(8)], steps=1, budget=1024, seed=3)
    o = q.opts(path=q.QUEST_PATH_CHAIN)
    for w, launches in ((few, 2), (gqa, 3), (many, 3)):
        pair = H.on_device(w)
        assert q.decode_launches(pair.cache, w.top_k, o) == launches
        H.run_step_and_compare(pair, 0, w.top_k, opts=o, one_launch=True, check_cache=True)


@pytest.mark.parametrize("hq,hkv,max_pages,chain_launches",
                         [(4, 4, 4096, 2), (4, 4, 4097, 3), (8, 4, 4096, 3)],
                         ids=["mha_4096", "mha_4097", "gqa_4096"])
def test_exact_ties_on_every_path_go_to_the_lower_page(hq, hkv, max_pages, chain_launches):
    """Every page's keys are one vector per kv head scaled by one of four factors, so the
    page scores take four values, each shared by hundreds of pages, and the rule that ties
    go to the lower page alone fixes the selection.  Each decode path (the top-K inside
    the decode's work items on MHA rows of up to 4096 pages, the top-K kernel on longer
    rows and on GQA, the cluster kernel, the stream kernel) returns the oracle's pages bit
    for bit, and the oracle's attention over them."""
    B, P, K = 2, 16, 128
    w = wl.build("ties", batch=B, num_q_heads=hq, num_kv_heads=hkv, page_size=P,
                 prefill_lens=[P * 3000 + 5, P * 900], steps=1, budget=K * P, seed=11,
                 max_pages=max_pages)
    gen = torch.Generator().manual_seed(5)
    u = torch.randn(hkv, 128, generator=gen)
    u = 4.0 * u / u.norm(dim=1, keepdim=True)
    for b in range(B):
        n = int((w.block_table[b] >= 0).sum())
        p = torch.arange(n).unsqueeze(1)
        c = 1 + (7 * p + 3 * torch.arange(hkv).unsqueeze(0) + b) % 4          # [n][Hkv]
        w.k_pool[w.block_table[b, :n].long()] = (
            (c[:, :, None, None] * u[None, :, None, :]).expand(n, hkv, P, 128).to(torch.float16))
    G = hq // hkv
    for h in range(hq):
        sign = 1.0 if (h // G) % 2 == 0 else -1.0                 # the top or the bottom class
        w.q[0, :, h] = (sign * u[h // G]).to(torch.float16)

    qh = w.q[0].numpy().astype(np.float32)
    ref = H.on_device(w).ref
    ref_scores = oracle.score(ref, qh)
    ref_idx, ref_cnt = oracle.topk(ref, ref_scores, K)
    for b in range(B):
        for g in range(hkv):
            s = np.sort(ref_scores[b, g][np.isfinite(ref_scores[b, g])])[::-1]
            assert s[K - 1] == s[K], "the K-th and the next page must tie"
    want = np.sort(ref_idx, axis=2)
    out_ref, lse_ref = oracle.attend(ref, qh, want, ref_cnt)

    ran = []
    for path in (q.QUEST_PATH_AUTO, q.QUEST_PATH_CHAIN, q.QUEST_PATH_FUSED,
                 q.QUEST_PATH_STREAM):
        o = q.opts(path=path)
        pair = H.on_device(w, opts=o)
        try:
            q.decode_path(pair.cache, K, o)
        except q.QuestError:
            continue                            # a one-launch kernel this shape does not fit
        if path == q.QUEST_PATH_CHAIN:
            assert q.decode_launches(pair.cache, K, o) == chain_launches
        idx = torch.empty((B, hkv, K), dtype=torch.int32, device="cuda")
        cnt = torch.empty((B, hkv), dtype=torch.int32, device="cuda")
        out, lse = q.decode(pair.cache, w.q[0].cuda(), K, pair.ws, o, idx_out=idx,
                            count_out=cnt)
        H.assert_status_ok(pair.ws)
        np.testing.assert_array_equal(cnt.cpu().numpy(), ref_cnt)
        np.testing.assert_array_equal(idx.cpu().numpy(), want)
        H.assert_attention_close(out, lse, out_ref, lse_ref)
        ran.append(path)
    assert q.QUEST_PATH_AUTO in ran and q.QUEST_PATH_CHAIN in ran, ran


@pytest.mark.parametrize("append", [False, True], ids=["decode", "step"])
def test_fused_union_form_matches_separate_calls_and_oracle(append):
    """quest_decode / quest_decode_step with gqa_union (the chain: per-head bounds, union
    top-K, sparse decode over the union) gives the same union, counts and outputs, bit for
    bit, as the separate calls, and matches the oracle's attention over that union."""
    w = small(lens=(3000, 700, 16 * 9), batch=3, hq=8, hkv=2, budget=256, outliers=4,
              steps=1)
    a, b = H.on_device(w), H.on_device(w)
    K, G = w.top_k, 4
    o = q.opts(gqa_union=True)
    cap = min(G * K, a.cache.max_pages)
    ws_a = q.workspace(a.cache, K, o)
    idx = torch.empty((3, 2, cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((3, 2), dtype=torch.int32, device="cuda")
    qd, kn, vn = w.q[0].cuda(), w.k_new[0].cuda(), w.v_new[0].cuda()
    assert q.decode_path(a.cache, K, o) == q.QUEST_PATH_CHAIN
    if append:
        out, lse = q.decode_step(a.cache, qd, kn, vn, K, ws_a, o, idx_out=idx, count_out=cnt)
        q.append(b.cache, kn, vn, b.ws)
    else:
        out, lse = q.decode(a.cache, qd, K, ws_a, o, idx_out=idx, count_out=cnt)
    sh = q.estimate_heads(b.cache, qd, b.ws)
    i2, c2 = q.topk(b.cache, sh, K, b.ws, o)
    ws_u = q.workspace(b.cache, cap)
    o2, l2 = q.sparse_decode(b.cache, qd, i2, c2, cap, ws_u)
    H.assert_status_ok(ws_a)
    H.assert_status_ok(b.ws)
    assert torch.equal(idx, i2) and torch.equal(cnt, c2)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert torch.equal(a.cache.meta, b.cache.meta) and torch.equal(a.cache.seq_lens, b.cache.seq_lens)
    if append:
        oracle.append(a.ref, w.k_new[0].numpy(), w.v_new[0].numpy())
    qh = w.q[0].numpy().astype(np.float32)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    out_ref, lse_ref = oracle.attend(a.ref, qh, gi, gc)
    H.assert_attention_close(out, lse, out_ref, lse_ref)
    with pytest.raises(q.QuestError):
        q.decode(a.cache, qd, K, ws_a, q.opts(gqa_union=True, sink_pages=1, local_pages=1))
