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


@pytest.mark.parametrize("path", [q.QUEST_PATH_AUTO, q.QUEST_PATH_FUSED], ids=["auto", "fused"])
def test_layers_of_the_128k_model(path):
    """Four layers of the 128K-context shape (8192 pages per head), through the automatic
    choice (the layers as separate kernels here) and in one launch; every head's needle
    page must be in the oracle's selection and the outputs must match."""
    n = 4
    ws_ = [wl.yarn_128k_layer(layer, seed=0, device="cuda", budget=2048) for layer in range(n)]
    w0 = ws_[0]
    K = w0.top_k
    dev = torch.device("cuda")
    base = q.PagedCache.allocate_meta(w0.k_pool, w0.v_pool, w0.block_table, w0.seq_lens.clone(),
                                      w0.num_q_heads)
    layers = [base] + [q.PagedCache.allocate_meta(w.k_pool, w.v_pool, base.block_table,
                                                   base.seq_lens, w.num_q_heads)
                       for w in ws_[1:]]
    ws = q.workspace(base, K)
    for lay in layers:
        q.build_meta(lay, ws)
    qs = [w.q[0] for w in ws_]
    outs, lses = q.decode_layers(base, layers, qs, K, ws, q.opts(path=path))
    H.assert_status_ok(ws)
    bt = w0.block_table.cpu().numpy()
    sl = w0.seq_lens.cpu().numpy()
    for i, w in enumerate(ws_):
        ref = oracle.Cache.from_arrays(w.k_pool.cpu().numpy(), w.v_pool.cpu().numpy(), bt, sl,
                                       w.num_q_heads)
        oracle.build_meta(ref)
        qh = w.q[0].cpu().numpy().astype(np.float32)
        rs = oracle.score(ref, qh)
        ri, rc = oracle.topk(ref, rs, K)
        out_ref, lse_ref = oracle.attend(ref, qh, ri, rc)
        H.assert_attention_close(outs[i], lses[i], out_ref, lse_ref)
        del ref
