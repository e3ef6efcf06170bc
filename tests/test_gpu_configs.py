"""Parity of the fused decode step at the full sizes of the five workloads, in the launch
configuration the benchmark uses (automatic cluster size, quest_decode_step), against the
CPU oracle on the same seeded inputs.  Acceptance rules as in tests/harness.py:

* selection: exactly K_b distinct valid pages; swaps only inside the oracle's 1e-5
  relative tie window around its K_b-th score;
* attention: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| against the oracle's attention over
  the GPU's selected pages;
* lengths, appended rows and boxes: bit-exact (checked on the last step);
* planted needle pages are selected.

The decode calls choose between the one-launch kernel and the chain of separate kernels
(QUEST_PATH_AUTO); the larger workloads run both through that choice and through the
one-launch kernel.
"""
import pytest
import torch

import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

import harness as H

pytestmark = pytest.mark.gpu


PATHS = [q.QUEST_PATH_AUTO, q.QUEST_PATH_FUSED, q.QUEST_PATH_STREAM]
PATH_IDS = ["auto", "fused", "stream"]


def _run(w, steps, check_needles=True, path=q.QUEST_PATH_AUTO):
    pair = H.on_device(w)
    o = q.opts(path=path)
    for t in range(steps):
        H.run_step_and_compare(pair, t, w.top_k, opts=o, one_launch=True,
                               check_needles=check_needles, check_cache=(t == steps - 1))


@pytest.mark.parametrize("path", [q.QUEST_PATH_AUTO, q.QUEST_PATH_STREAM], ids=["auto", "stream"])
def test_longchat_32k_every_step(path):
    """The benchmark workload: 32768 prefilled tokens, then all 64 decode steps (each
    appends a token: 2049 -> 2052 pages), 32 MHA heads, budget 2048."""
    w = wl.longchat_32k(seed=0, device="cuda")
    _run(w, w.steps, path=path)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("budget", [256, 512, 1024, 2048, 4096])
def test_batched_ragged(budget, path):
    """8 sequences of 8K-32K tokens, 32 heads, the five budgets; four decode steps, through
    the automatic path choice and through the one-launch kernel."""
    w = wl.batched_ragged(seed=0, device="cuda", budget=budget, steps=4)
    _run(w, w.steps, check_needles=False, path=path)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("layer,budget", [(0, 1024), (13, 2048), (31, 2048)])
def test_yarn_128k_layers(layer, budget, path):
    """Single layers of the 128K-context model (8192 pages per head); each head's needle
    page must be kept."""
    w = wl.yarn_128k_layer(layer, seed=0, device="cuda", budget=budget)
    _run(w, 1, path=path)


@pytest.mark.parametrize("path", PATHS, ids=PATH_IDS)
@pytest.mark.parametrize("page_size", [16, 32])
def test_gqa_llama31(page_size, path):
    """4 sequences of 64K tokens, 32 query / 8 kv heads, budget 4096, page 16 and 32."""
    w = wl.gqa_llama31(seed=0, device="cuda", page_size=page_size)
    _run(w, 1, check_needles=False, path=path)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("page_size", [16, 32])
def test_gqa_llama31_union_form(page_size):
    """The full-size GQA workload through quest_decode_step in the union form (gqa_union):
    every query head's top-K pages, their union per kv head, attention over the union.
    The union is compared with the oracle's (swaps only inside some head's tie window around
    its K-th score) and the attention with the oracle's over the GPU's union."""
    import numpy as np
    import oracle
    w = wl.gqa_llama31(seed=0, device="cuda", page_size=page_size)
    pair = H.on_device(w)
    K, G = w.top_k, w.num_q_heads // w.num_kv_heads
    o = q.opts(gqa_union=True)
    cap = min(G * K, pair.cache.max_pages)
    ws = q.workspace(pair.cache, K, o)
    idx = torch.empty((w.batch, w.num_kv_heads, cap), dtype=torch.int32, device="cuda")
    cnt = torch.empty((w.batch, w.num_kv_heads), dtype=torch.int32, device="cuda")
    out, lse = q.decode_step(pair.cache, w.q[0], w.k_new[0], w.v_new[0], K, ws, o,
                             idx_out=idx, count_out=cnt)
    H.assert_status_ok(ws)
    oracle.append(pair.ref, w.k_new[0].cpu().numpy(), w.v_new[0].cpu().numpy())
    assert pair.cache.seq_lens.cpu().numpy().tolist() == pair.ref.seq_lens.tolist()
    qh = w.q[0].cpu().numpy().astype(np.float32)
    ref_sh = oracle.score_heads(pair.ref, qh)
    ri, rc = oracle.topk_union(pair.ref, ref_sh, K)
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    for b in range(w.batch):
        n = wl.pages_for(int(pair.ref.seq_lens[b]), page_size)
        for g in range(w.num_kv_heads):
            got = set(gi[b, g, :gc[b, g]].tolist())
            want = set(ri[b, g, :rc[b, g]].tolist())
            window = set()
            for h in range(g * G, (g + 1) * G):
                row = ref_sh[b, h, :n]
                sk = float(np.sort(row)[::-1][K - 1])
                window |= {p for p in range(n) if abs(float(row[p]) - sk) <= H.TIE_REL * abs(sk)}
            assert got - window == want - window, (b, g)
    out_ref, lse_ref = oracle.attend(pair.ref, qh, gi, gc)
    H.assert_attention_close(out, lse, out_ref, lse_ref)
    torch.cuda.empty_cache()
