"""Helpers of the GPU parity tests: put a workload on the device, mirror it in the CPU
oracle, and compare the two under the acceptance rules of the decode path.

Rules (also stated in the test files):
* bounding boxes, appended tokens, lengths: bit-exact;
* scores: |gpu - oracle| <= 2 * d * 2^-24 * sum_i |corner term_i| (two fp32 summation
  orders of the same exact products);
* selection: exactly K_b distinct valid pages; with s_K the oracle's K_b-th score and
  W = {p : |s_p - s_K| <= 1e-5 |s_K|}, GPU \\ W == oracle \\ W (swaps only among near-ties);
* attention: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise (fp16 output vs the
  double oracle), against the oracle's attention over the GPU's selected pages.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

import oracle
import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import workloads as wl

ATOL = 2e-3
RTOL = 1e-2
TIE_REL = 1e-5


@dataclass
class Pair:
    w: wl.Workload
    cache: q.PagedCache
    ws: torch.Tensor
    ref: oracle.Cache


def on_device(w: wl.Workload, top_k: Optional[int] = None, opts=None, build_meta=True) -> Pair:
    """Device copy of the workload (meta built by the library), plus the oracle mirror
    (meta built by the oracle from the same keys)."""
    dev = torch.device("cuda")
    k = w.k_pool.to(dev).contiguous()
    v = w.v_pool.to(dev).contiguous()
    bt = w.block_table.to(dev).contiguous()
    sl = w.seq_lens.to(dev).contiguous()
    cache = q.PagedCache.allocate_meta(k, v, bt, sl, w.num_q_heads)
    ws = q.workspace(cache, top_k or w.top_k, opts)
    if build_meta:
        q.build_meta(cache, ws)
    ref = oracle.Cache.from_arrays(w.k_pool.cpu().numpy(), w.v_pool.cpu().numpy(),
                                   w.block_table.cpu().numpy(), w.seq_lens.cpu().numpy(),
                                   w.num_q_heads)
    if build_meta:
        oracle.build_meta(ref)
    return Pair(w, cache, ws, ref)


def assert_status_ok(ws: torch.Tensor) -> None:
    rc, detail = q.read_status(ws)
    assert rc == 0, f"device status {rc} detail {detail}"


def valid_pages(ref: oracle.Cache):
    P = ref.k_pool.shape[2]
    for b in range(ref.block_table.shape[0]):
        for p in range(wl.pages_for(int(ref.seq_lens[b]), P)):
            yield b, p, int(ref.block_table[b, p])


def assert_meta_equal(pair: Pair) -> None:
    """GPU machines [B][Hkv][max_pages][2][d] (logical order) vs the oracle's boxes
    [num_phys][Hkv][2][d] (physical order), bit-exact for every existing page."""
    gpu = pair.cache.meta.cpu().numpy()
    ref16 = pair.ref.meta.astype(np.float16)
    for b, p, ph in valid_pages(pair.ref):
        np.testing.assert_array_equal(gpu[b, :, p].view(np.uint16), ref16[ph].view(np.uint16),
                                      err_msg=f"box of sequence {b} page {p}")


def score_tolerance(ref: oracle.Cache, qh: np.ndarray) -> np.ndarray:
    """[B][Hkv][max_pages] bound on fp32 reordering error of the scores."""
    B, max_pages = ref.block_table.shape
    hkv = ref.k_pool.shape[1]
    G = ref.num_q_heads // hkv
    tol = np.zeros((B, hkv, max_pages))
    d = ref.k_pool.shape[3]
    for b, p, ph in valid_pages(ref):
        for g in range(hkv):
            qq = qh[b, g * G:(g + 1) * G].astype(np.float64)              # [G][d]
            corner = np.maximum(np.abs(qq * ref.meta[ph, g, 0]), np.abs(qq * ref.meta[ph, g, 1]))
            tol[b, g, p] = 2.0 * d * 2.0 ** -24 * corner.sum(axis=1).max() + 1e-30
    return tol


def assert_scores_close(gpu: np.ndarray, ref_scores: np.ndarray, tol: np.ndarray) -> None:
    finite = np.isfinite(ref_scores)
    assert np.array_equal(np.isneginf(gpu), np.isneginf(ref_scores))
    err = np.abs(gpu[finite].astype(np.float64) - ref_scores[finite])
    bad = err > tol[finite]
    assert not bad.any(), f"{bad.sum()} scores beyond tolerance, worst {err.max()}"


def assert_selection(gpu_idx: np.ndarray, gpu_cnt: np.ndarray, ref_scores: np.ndarray,
                     ref_idx: np.ndarray, ref_cnt: np.ndarray) -> int:
    """Tie-window rule; returns how many (b, g) rows differ only inside the window."""
    B, hkv, K = ref_idx.shape
    swapped = 0
    for b in range(B):
        for g in range(hkv):
            kb = int(ref_cnt[b, g])
            assert int(gpu_cnt[b, g]) == kb, (b, g, int(gpu_cnt[b, g]), kb)
            got = gpu_idx[b, g, :kb].tolist()
            assert len(set(got)) == kb, "duplicate pages"
            assert got == sorted(got), "selection must be in ascending page order"
            assert np.all(gpu_idx[b, g, kb:] == -1)
            want = set(ref_idx[b, g, :kb].tolist())
            if set(got) == want:
                continue
            sk = float(ref_scores[b, g, ref_idx[b, g, kb - 1]])
            row = ref_scores[b, g]
            window = {p for p in range(len(row))
                      if np.isfinite(row[p]) and abs(float(row[p]) - sk) <= TIE_REL * abs(sk)}
            assert set(got) - window == want - window, (b, g)
            swapped += 1
    return swapped


def assert_attention_close(out_gpu: torch.Tensor, lse_gpu: Optional[torch.Tensor],
                           out_ref: np.ndarray, lse_ref: np.ndarray) -> None:
    o = out_gpu.float().cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(o, out_ref, atol=ATOL, rtol=RTOL)
    if lse_gpu is not None:
        l = lse_gpu.cpu().numpy().astype(np.float64)
        inf = np.isneginf(lse_ref)
        assert np.array_equal(np.isneginf(l), inf)
        np.testing.assert_allclose(l[~inf], lse_ref[~inf], atol=ATOL, rtol=RTOL)


def oracle_selection_arrays(gpu_idx: np.ndarray, gpu_cnt: np.ndarray):
    return gpu_idx.astype(np.int32), gpu_cnt.astype(np.int32)


def run_step_and_compare(pair: Pair, step: int, top_k: int, opts=None, fused: bool = True,
                         check_needles: bool = False, one_launch: bool = False,
                         check_cache: bool = False, sink: int = 0, local: int = 0) -> int:
    """One decode step on both sides (append + score + select + attend); compares
    scores (unfused only), selection and attention; with check_cache also the boxes,
    pools and lengths.  one_launch: quest_decode_step (append folded into the fused
    kernel) instead of quest_append + quest_decode."""
    w = pair.w
    qd = w.q[step].to("cuda").contiguous()
    kn = w.k_new[step].to("cuda").contiguous()
    vn = w.v_new[step].to("cuda").contiguous()
    if not one_launch:
        q.append(pair.cache, kn, vn, pair.ws)
    oracle.append(pair.ref, w.k_new[step].cpu().numpy(), w.v_new[step].cpu().numpy())
    qh = w.q[step].cpu().numpy().astype(np.float32)
    ref_scores = oracle.score(pair.ref, qh)
    ref_idx, ref_cnt = oracle.topk(pair.ref, ref_scores, top_k, sink, local)
    if one_launch:
        idx = torch.empty((w.batch, w.num_kv_heads, top_k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((w.batch, w.num_kv_heads), dtype=torch.int32, device="cuda")
        out, lse = q.decode_step(pair.cache, qd, kn, vn, top_k, pair.ws, opts, idx_out=idx,
                                 count_out=cnt)
    elif fused:
        idx = torch.empty((w.batch, w.num_kv_heads, top_k), dtype=torch.int32, device="cuda")
        cnt = torch.empty((w.batch, w.num_kv_heads), dtype=torch.int32, device="cuda")
        out, lse = q.decode(pair.cache, qd, top_k, pair.ws, opts, idx_out=idx, count_out=cnt)
    else:
        scores = q.estimate(pair.cache, qd, pair.ws)
        assert_scores_close(scores.cpu().numpy(), ref_scores, score_tolerance(pair.ref, qh))
        idx, cnt = q.topk(pair.cache, scores, top_k, pair.ws, opts)
        out, lse = q.sparse_decode(pair.cache, qd, idx, cnt, top_k, pair.ws, opts)
    assert_status_ok(pair.ws)
    assert pair.cache.seq_lens.cpu().numpy().tolist() == pair.ref.seq_lens.tolist()
    gi, gc = idx.cpu().numpy(), cnt.cpu().numpy()
    swapped = assert_selection(gi, gc, ref_scores, ref_idx, ref_cnt)
    out_ref, lse_ref = oracle.attend(pair.ref, qh, gi, gc)
    assert_attention_close(out, lse, out_ref, lse_ref)
    if check_needles:
        for (b, g, p, slot) in w.needles:
            assert p in gi[b, g, :gc[b, g]].tolist(), ("needle page not selected", b, g, p)
    if check_cache:
        assert_meta_equal(pair)
        kp = pair.cache.k_pool.cpu().numpy()
        vp = pair.cache.v_pool.cpu().numpy()
        P = w.page_size
        for b, p, ph in valid_pages(pair.ref):
            n = min(P, int(pair.ref.seq_lens[b]) - p * P)
            np.testing.assert_array_equal(kp[ph, :, :n].astype(np.float32), pair.ref.k_pool[ph, :, :n])
            np.testing.assert_array_equal(vp[ph, :, :n].astype(np.float32), pair.ref.v_pool[ph, :, :n])
    return swapped
