"""Every layer of a decode step in one call (quest_decode_layers: one launch, or the layers
as separate kernels): the layers share the batch, block table and lengths, each has its own
pools, boxes, query and new token.
Checked against the oracle per layer (acceptance rules of tests/harness.py) and against
one quest_decode_step call per layer with the same cluster size (bit-exact: the same pairs
are computed by the same code)."""
import numpy as np
import pytest
import torch

import oracle
import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

import harness as H

pytestmark = pytest.mark.gpu


def _layers(n, lens, hq=8, hkv=4, P=16, budget=256, seed=0):
    ws_ = [wl.build(f"layer{i}", batch=len(lens), num_q_heads=hq, num_kv_heads=hkv, page_size=P,
                    prefill_lens=list(lens), steps=1, budget=budget, seed=seed + i, outliers=4)
           for i in range(n)]
    return ws_


def _shared_cache(ws_, layer):
    """Layer `layer`'s pools under layer 0's block table and lengths (device + oracle)."""
    w0, w = ws_[0], ws_[layer]
    dev = torch.device("cuda")
    bt = w0.block_table.to(dev)
    sl = w0.seq_lens.to(dev)
    c = q.PagedCache.allocate_meta(w.k_pool.to(dev), w.v_pool.to(dev), bt, sl, w.num_q_heads)
    ref = oracle.Cache.from_arrays(w.k_pool.numpy(), w.v_pool.numpy(), w0.block_table.numpy(),
                                   w0.seq_lens.numpy(), w.num_q_heads)
    return c, ref


@pytest.mark.parametrize("path", ["cluster4", "chain"])
@pytest.mark.parametrize("append", [False, True])
def test_layers_match_oracle_and_single_calls(append, path):
    n = 4
    ws_ = _layers(n, lens=(2500, 700, 16 * 40 + 3))
    K = ws_[0].top_k
    caches, refs = zip(*[_shared_cache(ws_, i) for i in range(n)])
    base = caches[0]
    # the layers share block table and lengths: point every layer's descriptor at them
    layers = [q.PagedCache(c.k_pool, c.v_pool, c.meta, base.block_table, base.seq_lens,
                           ws_[0].num_q_heads) for c in caches]
    ws = q.workspace(base, K)
    for lay in layers:
        q.build_meta(lay, ws)
    for r in refs:
        oracle.build_meta(r)
    meta0 = [lay.meta.clone() for lay in layers]
    len0 = base.seq_lens.clone()
    qs = [w.q[0].cuda() for w in ws_]
    kn = [w.k_new[0].cuda() for w in ws_] if append else None
    vn = [w.v_new[0].cuda() for w in ws_] if append else None
    o = q.opts(cluster_size=4) if path == "cluster4" else q.opts(path=q.QUEST_PATH_CHAIN)
    outs, lses = q.decode_layers(base, layers, qs, K, ws, o, k_new=kn, v_new=vn)
    H.assert_status_ok(ws)
    assert base.seq_lens.cpu().tolist() == [int(x) + (1 if append else 0) for x in len0.cpu()]
    for i in range(n):
        if append:
            oracle.append(refs[i], ws_[i].k_new[0].numpy(), ws_[i].v_new[0].numpy())
        qh = ws_[i].q[0].numpy().astype(np.float32)
        rs = oracle.score(refs[i], qh)
        ri, rc = oracle.topk(refs[i], rs, K)
        # the selection is not returned by the multi-layer call: compare the output with the
        # oracle's attention over the oracle's own selection (no near-ties in these inputs)
        out_ref, lse_ref = oracle.attend(refs[i], qh, ri, rc)
        H.assert_attention_close(outs[i], lses[i], out_ref, lse_ref)
    # one quest_decode_step / quest_decode per layer, same cluster size or the same chain of
    # kernels: bit-exact
    multi_out = [x.clone() for x in outs]
    multi_meta = [lay.meta.clone() for lay in layers]
    for i, lay in enumerate(layers):
        lay.meta.copy_(meta0[i])
    for i, lay in enumerate(layers):
        base.seq_lens.copy_(len0)
        if append:
            out, lse = q.decode_step(lay, qs[i], kn[i], vn[i], K, ws, o)
        else:
            out, lse = q.decode(lay, qs[i], K, ws, o)
        assert torch.equal(out, multi_out[i]), i
        assert torch.equal(lay.meta, multi_meta[i]), i
    H.assert_status_ok(ws)


def _on_block_table(w, bt0):
    """w's pools laid out under the block table bt0: logical page p of sequence b goes to
    physical page bt0[b, p] (the layers of a model share one block table; each layer's
    workload draws its own)."""
    src, dst = w.block_table.long(), bt0.long()
    m = (src >= 0) & (dst >= 0)
    k = torch.zeros_like(w.k_pool)
    v = torch.zeros_like(w.v_pool)
    k[dst[m]] = w.k_pool[src[m]]
    v[dst[m]] = w.v_pool[src[m]]
    return k, v


N_LAYERS_128K = 32
BUDGETS_128K = (1024, 2048)


@pytest.fixture(scope="module")
def model_128k():
    """The 32 layers of the 128K-context model (1 sequence of 131 072 tokens, 32 MHA heads,
    8192 pages of 16 per head, one needle page per head and layer) on one shared block table,
    with the oracle's selection and attention of every layer at both budgets."""
    dev = torch.device("cuda")
    w0 = wl.yarn_128k_layer(0, seed=0, device="cuda", budget=2048)
    bt0, sl0 = w0.block_table, w0.seq_lens
    Hq = w0.num_q_heads
    base = q.PagedCache.allocate_meta(w0.k_pool, w0.v_pool, bt0, sl0.clone(), Hq)
    layers, qs, needles = [base], [w0.q[0]], [w0.needles]
    for i in range(1, N_LAYERS_128K):
        w = wl.yarn_128k_layer(i, seed=0, device="cuda", budget=2048)
        k, v = _on_block_table(w, bt0)
        layers.append(q.PagedCache.allocate_meta(k, v, base.block_table, base.seq_lens, Hq))
        qs.append(w.q[0])
        needles.append(w.needles)
        del w, k, v
    ws = {b: q.workspace(base, b // 16) for b in BUDGETS_128K}
    for lay in layers:
        q.build_meta(lay, ws[BUDGETS_128K[0]])
    torch.cuda.synchronize()
    bt, sl = bt0.cpu().numpy(), sl0.cpu().numpy()
    ref = {}
    for i, lay in enumerate(layers):
        r = oracle.Cache.from_arrays(lay.k_pool.cpu().numpy(), lay.v_pool.cpu().numpy(), bt, sl,
                                     Hq)
        oracle.build_meta(r)
        qh = qs[i].cpu().numpy().astype(np.float32)
        rs = oracle.score(r, qh)
        for budget in BUDGETS_128K:
            ri, rc = oracle.topk(r, rs, budget // 16)
            for (b, g, p, slot) in needles[i]:  # the workload plants what the method must find
                assert p in ri[b, g, :rc[b, g]].tolist(), ("oracle misses a needle", i, g)
            ref[(i, budget)] = oracle.attend(r, qh, ri, rc)
        del r
    return dict(base=base, layers=layers, qs=qs, needles=needles, ws=ws, ref=ref, dev=dev)


@pytest.mark.parametrize("budget", BUDGETS_128K)
@pytest.mark.parametrize("path", [q.QUEST_PATH_AUTO, q.QUEST_PATH_FUSED], ids=["auto", "fused"])
def test_layers_of_the_128k_model(model_128k, path, budget):
    """All 32 layers of the 128K-context model in one quest_decode_layers call (1024
    (layer, kv head) pairs), through the automatic choice and in one launch of the cluster
    kernel (more pairs than resident clusters: every cluster loops over pairs).  Every
    layer's outputs must match the oracle's attention over the oracle's selection, and in
    every layer every head's needle page must be among the pages the GPU selects: the
    selection is read from a single-layer quest_decode of the same layer (its scores and
    top-K are the same arithmetic as the multi-layer call's; the outputs of the two agree)."""
    m = model_128k
    base, layers, qs, ws = m["base"], m["layers"], m["qs"], m["ws"][budget]
    K = budget // 16
    o = q.opts(path=path)
    outs, lses = q.decode_layers(base, layers, qs, K, ws, o)
    H.assert_status_ok(ws)
    idx = torch.empty((1, 32, K), dtype=torch.int32, device="cuda")
    cnt = torch.empty((1, 32), dtype=torch.int32, device="cuda")
    for i, lay in enumerate(layers):
        out_ref, lse_ref = m["ref"][(i, budget)]
        H.assert_attention_close(outs[i], lses[i], out_ref, lse_ref)
        one, one_lse = q.decode(lay, qs[i], K, ws, o, idx_out=idx, count_out=cnt)
        gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
        for (b, g, p, slot) in m["needles"][i]:
            assert p in gi[b, g, :gc[b, g]].tolist(), ("needle page not selected", i, g, p)
        torch.testing.assert_close(one.float(), outs[i].float(), atol=2e-3, rtol=0)
    H.assert_status_ok(ws)
