"""Pins of the CPU oracle to what the Quest pages and mathematics fix (no GPU).

Each test checks the oracle against something other than itself: an invariant the pages
state, a closed form, a hand-worked fixture, or brute force on tiny inputs.  Citations:
  [Guide]   "Guide to Quest: Query-Aware KV Cache Sparsity for LLMs"
  [Summary] "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference" (Tang 2024)
"""
import math
import os

import numpy as np
import pytest

import oracle
from query_aware_kv_gb300 import workloads as wl

pytestmark = pytest.mark.usefixtures("oracle_built")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def make(batch=2, hq=4, hkv=4, P=16, lens=(70, 33), steps=0, d=128, seed=0, **kw):
    w = wl.build("pin", batch=batch, num_q_heads=hq, num_kv_heads=hkv, page_size=P,
                 prefill_lens=list(lens), steps=steps, budget=4 * P, seed=seed, head_dim=d,
                 **kw)
    c = oracle.Cache.from_arrays(w.k_pool.numpy(), w.v_pool.numpy(), w.block_table.numpy(),
                                 w.seq_lens.numpy(), hq)
    return w, c


def logical_keys(c, b, g, p):
    """Keys of logical page p of sequence b (valid tokens only), float64 [n][d]."""
    P = c.k_pool.shape[2]
    L = int(c.seq_lens[b])
    n = min(P, L - p * P)
    phys = int(c.block_table[b, p])
    return c.k_pool[phys, g, :n].astype(np.float64)


def fp32_sum_tol(terms):
    """Bound on the rounding error of a float32 sum of len(terms) exact terms."""
    return len(terms) * 2.0 ** -24 * float(np.sum(np.abs(terms))) + 1e-30


# ----------------------------------------------------------------------------------
# bounding boxes ([Guide] Solution step 1)
# ----------------------------------------------------------------------------------

def test_meta_box_contains_and_is_attained():
    w, c = make(lens=(70, 33, 16, 1), batch=4)
    P = c.k_pool.shape[2]
    # junk in the slots past each sequence end must not enter a box
    for b in range(4):
        L = int(c.seq_lens[b])
        p = (L - 1) // P
        phys = int(c.block_table[b, p])
        for t in range(L - p * P, P):
            c.k_pool[phys, :, t, :] = 1e4 if t % 2 else -1e4
    meta = oracle.build_meta(c).astype(np.float64)
    for b in range(4):
        L = int(c.seq_lens[b])
        for p in range(wl.pages_for(L, P)):
            phys = int(c.block_table[b, p])
            for g in range(c.k_pool.shape[1]):
                keys = logical_keys(c, b, g, p)
                lo, hi = meta[phys, g, 0], meta[phys, g, 1]
                assert np.all(keys >= lo) and np.all(keys <= hi)
                # every bound is attained by a valid token in its dimension
                assert np.all(np.any(keys == lo, axis=0))
                assert np.all(np.any(keys == hi, axis=0))


def test_meta_matches_vectorised_reduction_and_leaves_other_pages():
    w, c = make(lens=(100, 47, 5), batch=3, hq=2, hkv=2, P=32, spare_pages=3)
    meta = oracle.build_meta(c)
    P = 32
    touched = set()
    for b in range(3):
        L = int(c.seq_lens[b])
        for p in range(wl.pages_for(L, P)):
            phys = int(c.block_table[b, p])
            touched.add(phys)
            n = min(P, L - p * P)
            slab = c.k_pool[phys, :, :n, :]           # [Hkv][n][d]
            np.testing.assert_array_equal(meta[phys, :, 0].astype(np.float32), slab.min(axis=1))
            np.testing.assert_array_equal(meta[phys, :, 1].astype(np.float32), slab.max(axis=1))
    for phys in range(c.k_pool.shape[0]):
        if phys not in touched:
            assert np.all(np.isnan(c.meta[phys]))


def test_meta_single_token_page_is_the_key():
    w, c = make(lens=(17,), batch=1)
    meta = oracle.build_meta(c)
    phys = int(c.block_table[0, 1])
    np.testing.assert_array_equal(meta[phys, :, 0].astype(np.float32), c.k_pool[phys, :, 0])
    np.testing.assert_array_equal(meta[phys, :, 1].astype(np.float32), c.k_pool[phys, :, 0])


def _golden():
    rows = {}
    keys, kmin, kmax, bound, maxqk = [], {}, {}, {}, {}
    with open(os.path.join(GOLDEN, "score_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tag, *vals = line.split()
            if tag == "key":
                keys.append([float(v) for v in vals])
            elif tag in ("kmin", "kmax"):
                (kmin if tag == "kmin" else kmax)[int(vals[0])] = [float(v) for v in vals[1:]]
            elif tag in ("bound", "max_qk"):
                (bound if tag == "bound" else maxqk)[int(vals[0])] = float(vals[1])
            elif tag == "query":
                rows["query"] = [float(v) for v in vals]
            else:
                rows[tag] = int(vals[0])
    return rows, np.array(keys), kmin, kmax, bound, maxqk


def test_score_hand_worked_example():
    rows, keys, kmin, kmax, bound, maxqk = _golden()
    d, P, L = rows["head_dim"], rows["page_size"], rows["seq_len"]
    n_pages = len(keys) // P
    k_pool = keys.reshape(n_pages, 1, P, d).astype(np.float32)
    bt = np.arange(n_pages, dtype=np.int32)[None, :]
    c = oracle.Cache.from_arrays(k_pool, np.zeros_like(k_pool), bt, [L], 1)
    meta = oracle.build_meta(c).astype(np.float64)
    for p in range(n_pages):
        np.testing.assert_array_equal(meta[p, 0, 0], kmin[p])
        np.testing.assert_array_equal(meta[p, 0, 1], kmax[p])
    q = np.array(rows["query"], np.float32).reshape(1, 1, d)
    s = oracle.score(c, q)
    for p in range(n_pages):
        assert s[0, 0, p] == bound[p]
        assert maxqk[p] <= bound[p]
    idx, cnt = oracle.topk(c, s, 1)
    assert idx[0, 0, 0] == rows["top1"] and cnt[0, 0] == 1


# ----------------------------------------------------------------------------------
# criticality bound ([Guide] Solution step 2)
# ----------------------------------------------------------------------------------

@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_score_upper_bounds_every_key(hq, hkv):
    w, c = make(hq=hq, hkv=hkv, lens=(150, 64, 9), batch=3, outliers=2)
    oracle.build_meta(c)
    q = w.q if w.q.shape[0] else None
    rng = np.random.default_rng(1)
    q = rng.standard_normal((3, hq, 128)).astype(np.float16).astype(np.float32)
    s = oracle.score(c, q)
    G = hq // hkv
    for b in range(3):
        for g in range(hkv):
            for p in range(wl.pages_for(int(c.seq_lens[b]), 16)):
                keys = logical_keys(c, b, g, p)
                best = -np.inf
                tol = 0.0
                phys = int(c.block_table[b, p])
                for h in range(g * G, (g + 1) * G):
                    qd = q[b, h].astype(np.float64)
                    best = max(best, float((keys @ qd).max()))
                    terms = np.maximum(qd * c.meta[phys, g, 0], qd * c.meta[phys, g, 1])
                    tol = max(tol, fp32_sum_tol(terms))
                assert s[b, g, p] >= best - tol


@pytest.mark.parametrize("sign", [+1, -1])
def test_score_single_signed_query_uses_one_side(sign):
    """q >= 0 gives sum q_i*Kmax_i; q <= 0 gives sum q_i*Kmin_i ([Guide] Solution step 2)."""
    w, c = make(lens=(90,), batch=1)
    oracle.build_meta(c)
    rng = np.random.default_rng(2)
    q = (sign * np.abs(rng.standard_normal((1, 4, 128)))).astype(np.float16).astype(np.float32)
    s = oracle.score(c, q)
    side = 1 if sign > 0 else 0
    for g in range(4):
        for p in range(wl.pages_for(90, 16)):
            phys = int(c.block_table[0, p])
            terms = q[0, g].astype(np.float64) * c.meta[phys, g, side]
            assert abs(s[0, g, p] - terms.sum()) <= fp32_sum_tol(terms)


def test_score_exact_for_one_token_and_corner_pages():
    """A one-token page scores q.k; a page holding its own corner key scores max_t q.k_t."""
    w, c = make(lens=(33,), batch=1)  # page 2 holds a single token
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 128)).astype(np.float16).astype(np.float32)
    # plant the corner of page 0's box as its token 5, per head
    phys0 = int(c.block_table[0, 0])
    for g in range(4):
        keys = c.k_pool[phys0, g, :16]
        c.k_pool[phys0, g, 5] = np.where(q[0, g] > 0, keys.max(axis=0), keys.min(axis=0))
    oracle.build_meta(c)
    s = oracle.score(c, q)
    for g in range(4):
        qd = q[0, g].astype(np.float64)
        one = logical_keys(c, 0, g, 2)
        assert one.shape[0] == 1
        terms = qd * one[0]
        assert abs(s[0, g, 2] - terms.sum()) <= fp32_sum_tol(terms)
        keys = logical_keys(c, 0, g, 0)
        qk = keys @ qd
        assert abs(s[0, g, 0] - qk.max()) <= fp32_sum_tol(qd * keys[5])


def test_score_gqa_is_max_over_the_group():
    """Group score = max over the group's query heads; query head h reads kv head h // G."""
    hq, hkv = 8, 2
    w, c = make(hq=hq, hkv=hkv, lens=(80, 40), batch=2)
    oracle.build_meta(c)
    rng = np.random.default_rng(4)
    q = rng.standard_normal((2, hq, 128)).astype(np.float16).astype(np.float32)
    s = oracle.score(c, q)
    # MHA cache whose kv head h carries kv head h // G of the GQA cache
    G = hq // hkv
    rep = oracle.Cache.from_arrays(np.repeat(c.k_pool, G, axis=1), np.repeat(c.v_pool, G, axis=1),
                                   c.block_table, c.seq_lens, hq)
    oracle.build_meta(rep)
    s_rep = oracle.score(rep, q)
    np.testing.assert_array_equal(s, s_rep.reshape(2, hkv, G, -1).max(axis=2))


def test_score_past_end_is_neg_inf():
    w, c = make(lens=(20, 100), batch=2)
    oracle.build_meta(c)
    s = oracle.score(c, np.ones((2, 4, 128), np.float32))
    assert np.all(np.isneginf(s[0, :, 2:])) and np.all(np.isfinite(s[0, :, :2]))
    assert np.all(np.isfinite(s[1, :, :7]))


# ----------------------------------------------------------------------------------
# top-K ([Guide] Solution step 3)
# ----------------------------------------------------------------------------------

def test_topk_matches_bruteforce_sort():
    rng = np.random.default_rng(5)
    w, c = make(lens=(400, 250, 30), batch=3)
    n = [wl.pages_for(int(L), 16) for L in c.seq_lens]
    scores = np.full((3, 4, c.block_table.shape[1]), -np.inf, np.float32)
    for b in range(3):
        scores[b, :, :n[b]] = rng.standard_normal((4, n[b])).astype(np.float32)
    for K in (1, 5, 16, 40):
        idx, cnt = oracle.topk(c, scores, K)
        for b in range(3):
            for g in range(4):
                ref = sorted(range(n[b]), key=lambda p: (-float(scores[b, g, p]), p))[:K]
                assert cnt[b, g] == len(ref) == min(K, n[b])
                assert idx[b, g, :cnt[b, g]].tolist() == ref
                assert np.all(idx[b, g, cnt[b, g]:] == -1)


def test_topk_ties_go_to_lower_index():
    w, c = make(lens=(16 * 40,), batch=1, hq=1, hkv=1)
    scores = np.full((1, 1, c.block_table.shape[1]), -np.inf, np.float32)
    vals = np.array([3.0, 1.0, 2.0, 2.0, 1.0, 2.0, 5.0, 2.0] * 5, np.float32)
    scores[0, 0, :40] = vals
    idx, cnt = oracle.topk(c, scores, 12)
    # 5 fives, then 7 of the 20 twos (the lowest pages among them)... sorted by rank
    fives = [p for p in range(40) if vals[p] == 5.0]
    threes = [p for p in range(40) if vals[p] == 3.0]
    twos = [p for p in range(40) if vals[p] == 2.0][:2]
    assert idx[0, 0].tolist() == fives + threes + twos


def test_topk_keeps_everything_when_short():
    w, c = make(lens=(40, 16 * 9), batch=2)
    s = np.zeros((2, 4, c.block_table.shape[1]), np.float32)
    idx, cnt = oracle.topk(c, s, 16)
    assert cnt.tolist() == [[3] * 4, [9] * 4]
    assert idx[0, 0, :3].tolist() == [0, 1, 2] and np.all(idx[0, 0, 3:] == -1)


def test_topk_window_keeps_sinks_and_local_pages():
    """[Guide] Solution step 3 / Implementation step 2: the first `sink` and last `local`
    pages are always kept; the other K - sink - local pages are the best of the rest, by
    brute force; a sequence of at most K pages keeps everything."""
    rng = np.random.default_rng(9)
    w, c = make(lens=(16 * 60, 16 * 7, 16 * 30 - 5), batch=3)
    n = [wl.pages_for(int(L), 16) for L in c.seq_lens]
    scores = np.full((3, 4, c.block_table.shape[1]), -np.inf, np.float32)
    for b in range(3):
        scores[b, :, :n[b]] = rng.standard_normal((4, n[b])).astype(np.float32)
        scores[b, 0, :n[b]] = np.round(scores[b, 0, :n[b]])  # ties
    scores[0, 1, :2] = 100.0  # a sink that would win anyway
    for K, sink, local in [(16, 2, 2), (16, 0, 3), (16, 4, 0), (10, 5, 5), (9, 0, 0)]:
        idx, cnt = oracle.topk(c, scores, K, sink, local)
        for b in range(3):
            for g in range(4):
                got = idx[b, g, :cnt[b, g]].tolist()
                if n[b] <= K:
                    assert sorted(got) == list(range(n[b]))
                    continue
                mand = list(range(sink)) + list(range(n[b] - local, n[b]))
                rest = sorted(range(sink, n[b] - local), key=lambda p: (-float(scores[b, g, p]), p))
                assert got == mand + rest[:K - sink - local]
                assert cnt[b, g] == K and len(set(got)) == K
                assert np.all(idx[b, g, K:] == -1)


def test_topk_window_zero_is_plain_topk_and_local_zero_keeps_no_tail():
    rng = np.random.default_rng(10)
    w, c = make(lens=(16 * 50,), batch=1)
    scores = np.full((1, 4, c.block_table.shape[1]), -np.inf, np.float32)
    scores[0, :, :50] = rng.standard_normal((4, 50)).astype(np.float32)
    scores[0, :, 49] = 1e6  # the last page: kept on merit only
    a, _ = oracle.topk(c, scores, 8)
    b, _ = oracle.topk(c, scores, 8, 0, 0)
    assert np.array_equal(a, b)
    idx, cnt = oracle.topk(c, scores, 8, 3, 0)
    for g in range(4):
        got = idx[0, g, :8].tolist()
        assert got[:3] == [0, 1, 2] and 49 in got  # no page is masked by local = 0
    with pytest.raises(oracle.OracleError):
        oracle.topk(c, scores, 4, 3, 2)  # the window does not fit the budget


def test_score_heads_are_the_per_head_bounds_whose_group_max_is_the_score():
    """The per-query-head bound, by a float64 brute force over the page's boxes, and its
    maximum over each group is the kv-head score."""
    w, c = make(lens=(300, 40), batch=2, hq=8, hkv=2)
    oracle.build_meta(c)
    rng = np.random.default_rng(12)
    qh = rng.standard_normal((2, 8, 128)).astype(np.float16).astype(np.float32)
    sh = oracle.score_heads(c, qh)
    sk = oracle.score(c, qh)
    for b in range(2):
        n = wl.pages_for(int(c.seq_lens[b]), 16)
        assert np.all(np.isneginf(sh[b, :, n:]))
        for h in range(8):
            g = h // 4
            for p in range(n):
                ph = int(c.block_table[b, p])
                mn = c.meta[ph, g, 0].astype(np.float64)
                mx = c.meta[ph, g, 1].astype(np.float64)
                qq = qh[b, h].astype(np.float64)
                ref = np.maximum(qq * mn, qq * mx).sum()
                assert abs(sh[b, h, p] - ref) <= 1e-4 * max(1.0, abs(ref))
        for g in range(2):
            np.testing.assert_array_equal(sh[b, 4 * g:4 * g + 4, :n].max(axis=0), sk[b, g, :n])


def test_topk_union_is_the_union_of_per_head_topk():
    """[Guide] Best Practices step 2 (GQA, union form): brute force per query head, union
    per group, ascending; at most G * K pages; a group of one head is plain top-K; short
    sequences keep every page."""
    rng = np.random.default_rng(13)
    w, c = make(lens=(16 * 90, 16 * 5, 16 * 33), batch=3, hq=8, hkv=2)
    mp = c.block_table.shape[1]
    n = [wl.pages_for(int(L), 16) for L in c.seq_lens]
    sh = np.full((3, 8, mp), -np.inf, np.float32)
    for b in range(3):
        sh[b, :, :n[b]] = rng.standard_normal((8, n[b])).astype(np.float32)
        sh[b, 1, :n[b]] = np.round(sh[b, 1, :n[b]])  # ties inside one head
    for K in (1, 7, 20):
        idx, cnt = oracle.topk_union(c, sh, K)
        assert idx.shape[2] == min(4 * K, mp)
        for b in range(3):
            for g in range(2):
                if n[b] <= K:
                    want = list(range(n[b]))
                else:
                    want = set()
                    for h in range(4 * g, 4 * g + 4):
                        want |= set(sorted(range(n[b]), key=lambda p: (-float(sh[b, h, p]), p))[:K])
                    want = sorted(want)
                assert idx[b, g, :cnt[b, g]].tolist() == want
                assert cnt[b, g] <= 4 * K and np.all(idx[b, g, cnt[b, g]:] == -1)
    # one head per group: the union is the plain top-K set
    w1, c1 = make(lens=(16 * 90,), batch=1, hq=2, hkv=2)
    s1 = np.full((1, 2, c1.block_table.shape[1]), -np.inf, np.float32)
    s1[0, :, :90] = rng.standard_normal((2, 90)).astype(np.float32)
    iu, cu = oracle.topk_union(c1, s1, 9)
    ip, cp = oracle.topk(c1, s1, 9)
    for g in range(2):
        assert iu[0, g, :cu[0, g]].tolist() == sorted(ip[0, g, :cp[0, g]].tolist())


def test_planted_needles_are_selected():
    """[Guide] Evaluation: a page holding a key aligned with the query gets an elevated
    bound and is kept by the top-K."""
    w = wl.build("needles", batch=1, num_q_heads=4, num_kv_heads=4, page_size=16,
                 prefill_lens=[4096], steps=3, budget=256, seed=11, outliers=4,
                 needles_per_head=8, needle_mode="direction")
    c = oracle.Cache.from_arrays(w.k_pool.numpy(), w.v_pool.numpy(), w.block_table.numpy(),
                                 w.seq_lens.numpy(), 4)
    oracle.build_meta(c)
    for t in range(w.steps):
        s, idx, cnt, out, lse = oracle.decode_step(c, w.q[t].numpy(), w.top_k,
                                                   w.k_new[t].numpy(), w.v_new[t].numpy())
        for (b, g, p, slot) in w.needles:
            assert p in idx[b, g, :cnt[b, g]].tolist()


# ----------------------------------------------------------------------------------
# attention over the kept pages ([Summary]; [Guide] Solution step 3, Implementation step 3)
# ----------------------------------------------------------------------------------

def dense_bruteforce(c, q):
    """softmax(q K^T / sqrt(d)) V over the logical token sequence, float64, vectorised."""
    B, Hq, d = q.shape
    hkv = c.k_pool.shape[1]
    P = c.k_pool.shape[2]
    G = Hq // hkv
    out = np.zeros((B, Hq, d))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(c.seq_lens[b])
        t = np.arange(L)
        phys = c.block_table[b, t // P]
        for h in range(Hq):
            K = c.k_pool[phys, h // G, t % P].astype(np.float64)
            V = c.v_pool[phys, h // G, t % P].astype(np.float64)
            z = K @ q[b, h].astype(np.float64) / math.sqrt(d)
            m = z.max()
            w = np.exp(z - m)
            out[b, h] = (w / w.sum()) @ V
            lse[b, h] = m + math.log(w.sum())
    return out, lse


@pytest.mark.parametrize("hq,hkv,P", [(4, 4, 16), (8, 2, 32)])
def test_all_pages_equals_dense_bruteforce(hq, hkv, P):
    w, c = make(hq=hq, hkv=hkv, P=P, lens=(130, 64, 7), batch=3)
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, hq, 128)).astype(np.float16).astype(np.float32)
    out, lse = oracle.dense(c, q)
    ref, ref_lse = dense_bruteforce(c, q)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12)
    # the same through score -> top-K with K >= every page count
    oracle.build_meta(c)
    s = oracle.score(c, q)
    idx, cnt = oracle.topk(c, s, 9)
    out2, lse2 = oracle.attend(c, q, idx, cnt)
    np.testing.assert_allclose(out2, ref, rtol=1e-10, atol=1e-12)


def test_single_token_selection_returns_its_value():
    w, c = make(lens=(33,), batch=1)
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 4, 128)).astype(np.float16).astype(np.float32)
    idx = np.full((1, 4, 1), 2, np.int32)
    cnt = np.ones((1, 4), np.int32)
    out, lse = oracle.attend(c, q, idx, cnt)
    phys = int(c.block_table[0, 2])
    for g in range(4):
        np.testing.assert_array_equal(out[0, g], c.v_pool[phys, g, 0].astype(np.float64))
        z = float(c.k_pool[phys, g, 0].astype(np.float64) @ q[0, g].astype(np.float64)) / math.sqrt(128)
        assert abs(lse[0, g] - z) <= 1e-12 * max(1.0, abs(z))


def test_identical_keys_average_the_values():
    w, c = make(lens=(40,), batch=1)
    c.k_pool[:] = c.k_pool[0, 0, 0]
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 4, 128)).astype(np.float16).astype(np.float32)
    out, lse = oracle.dense(c, q)
    for g in range(4):
        vals = np.concatenate([c.v_pool[int(c.block_table[0, p]), g, :min(16, 40 - 16 * p)]
                               for p in range(3)]).astype(np.float64)
        np.testing.assert_allclose(out[0, g], vals.mean(axis=0), rtol=1e-12, atol=1e-12)
        z = float(c.k_pool[0, 0, 0].astype(np.float64) @ q[0, g].astype(np.float64)) / math.sqrt(128)
        assert abs(lse[0, g] - (z + math.log(40))) <= 1e-12 * abs(z + math.log(40))


def test_disjoint_selections_merge_by_logsumexp():
    """Attention over A u B equals the lse-weighted mix of attention over A and over B."""
    w, c = make(lens=(160,), batch=1, hq=8, hkv=2)
    rng = np.random.default_rng(9)
    q = rng.standard_normal((1, 8, 128)).astype(np.float16).astype(np.float32)
    A = np.array([[[0, 3, 7], [1, 2, 9]]], np.int32)
    Bs = np.array([[[1, 5, 9], [0, 4, 8]]], np.int32)
    cnt = np.full((1, 2), 3, np.int32)
    oa, la = oracle.attend(c, q, A, cnt)
    ob, lb = oracle.attend(c, q, Bs, cnt)
    ou, lu = oracle.attend(c, q, np.concatenate([A, Bs], axis=2), cnt * 2)
    m = np.maximum(la, lb)
    wa, wb = np.exp(la - m), np.exp(lb - m)
    np.testing.assert_allclose(lu, m + np.log(wa + wb), rtol=1e-12)
    mix = (wa[..., None] * oa + wb[..., None] * ob) / (wa + wb)[..., None]
    np.testing.assert_allclose(ou, mix, rtol=1e-10, atol=1e-12)


def test_placement_and_junk_do_not_matter():
    """Moving pages to other physical slots, or junk past the end, leaves the result."""
    w, c = make(lens=(75,), batch=1, spare_pages=4)
    rng = np.random.default_rng(10)
    q = rng.standard_normal((1, 4, 128)).astype(np.float16).astype(np.float32)
    out, lse = oracle.dense(c, q)
    perm = rng.permutation(c.k_pool.shape[0]).astype(np.int32)
    k2 = np.empty_like(c.k_pool)
    v2 = np.empty_like(c.v_pool)
    k2[perm] = c.k_pool
    v2[perm] = c.v_pool
    bt2 = np.where(c.block_table >= 0, perm[np.maximum(c.block_table, 0)], -1).astype(np.int32)
    last = int(bt2[0, 4])
    k2[last, :, 75 - 64:] = np.nan
    v2[last, :, 75 - 64:] = np.nan
    c2 = oracle.Cache.from_arrays(k2, v2, bt2, c.seq_lens, 4)
    out2, lse2 = oracle.dense(c2, q)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


def test_dominant_key_wins():
    w, c = make(lens=(64,), batch=1)
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 4, 128)).astype(np.float16).astype(np.float32)
    phys = int(c.block_table[0, 1])
    for g in range(4):
        c.k_pool[phys, g, 3] = (q[0, g] * 8.0).astype(np.float16)
    out, lse = oracle.dense(c, q)
    for g in range(4):
        np.testing.assert_allclose(out[0, g], c.v_pool[phys, g, 3], atol=1e-6)


def test_empty_sequence():
    w, c = make(lens=(0, 20), batch=2, steps=1)
    q = np.ones((2, 4, 128), np.float32)
    out, lse = oracle.dense(c, q)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ----------------------------------------------------------------------------------
# decode-time append ([Guide] Solution step 1: boxes formed during token generation)
# ----------------------------------------------------------------------------------

def test_append_incremental_equals_rebuild():
    w, c = make(lens=(30, 47), batch=2, steps=40, hq=4, hkv=2)
    oracle.build_meta(c)
    for t in range(w.steps):
        oracle.append(c, w.k_new[t].numpy(), w.v_new[t].numpy())
    assert c.seq_lens.tolist() == [70, 87]
    rebuilt = oracle.Cache.from_arrays(c.k_pool, c.v_pool, c.block_table, c.seq_lens, 4)
    oracle.build_meta(rebuilt)
    for b in range(2):
        for p in range(wl.pages_for(int(c.seq_lens[b]), 16)):
            phys = int(c.block_table[b, p])
            np.testing.assert_array_equal(c.meta[phys], rebuilt.meta[phys])
    # the appended tokens sit at their positions
    t = 12
    pos = 30 + t
    phys = int(c.block_table[0, pos // 16])
    np.testing.assert_array_equal(c.k_pool[phys, :, pos % 16], w.k_new[t, 0].float().numpy())
    np.testing.assert_array_equal(c.v_pool[phys, :, pos % 16], w.v_new[t, 0].float().numpy())


def test_append_opening_a_page_starts_a_fresh_box():
    w, c = make(lens=(32,), batch=1, steps=1)
    oracle.build_meta(c)
    phys = int(c.block_table[0, 2])
    c.meta[phys] = 1e4 * np.sign(np.arange(2)[:, None] - 0.5)  # stale box: [-1e4, 1e4]
    oracle.append(c, w.k_new[0].numpy(), w.v_new[0].numpy())
    np.testing.assert_array_equal(c.meta[phys, :, 0], w.k_new[0, 0].float().numpy())
    np.testing.assert_array_equal(c.meta[phys, :, 1], w.k_new[0, 0].float().numpy())


def test_append_past_capacity_is_an_error():
    w, c = make(lens=(32,), batch=1, steps=0)
    assert c.block_table.shape[1] == 2
    with pytest.raises(oracle.OracleError):
        oracle.append(c, np.zeros((1, 4, 128)), np.zeros((1, 4, 128)))


def test_chunked_prefill_boxes_are_the_prompt_boxes():
    """Chunks of 5, 16 and 40 tokens from lengths 0 and 7: every page's box is the
    per-dimension min / max of its keys (numpy reduction over the final pool), stale
    boxes of fresh pages are replaced, and each token sits at its position."""
    w, c = make(lens=(0, 7), batch=2, steps=61, hq=4, hkv=2)
    c.meta[...] = 1e4  # stale boxes on every page that holds no token yet
    oracle.build_meta(c)  # boxes the 7 rows sequence 1 holds before the chunks
    kc = w.k_new.permute(1, 0, 2, 3).float().numpy()  # [B][61][Hkv][d]
    vc = w.v_new.permute(1, 0, 2, 3).float().numpy()
    done = 0
    for n in (5, 16, 40):
        oracle.prefill(c, kc[:, done:done + n], vc[:, done:done + n])
        done += n
    assert c.seq_lens.tolist() == [61, 68]
    for b, L0 in ((0, 0), (1, 7)):
        for t in (0, 4, 5, 20, 60):
            pos = L0 + t
            phys = int(c.block_table[b, pos // 16])
            np.testing.assert_array_equal(c.k_pool[phys, :, pos % 16], kc[b, t])
            np.testing.assert_array_equal(c.v_pool[phys, :, pos % 16], vc[b, t])
        for p in range(wl.pages_for(int(c.seq_lens[b]), 16)):
            phys = int(c.block_table[b, p])
            for g in range(2):
                keys = logical_keys(c, b, g, p)
                np.testing.assert_array_equal(c.meta[phys, g, 0], keys.min(axis=0))
                np.testing.assert_array_equal(c.meta[phys, g, 1], keys.max(axis=0))
