"""CPU oracle of Quest's decode path - TEST INFRASTRUCTURE ONLY.

Plain C loops (``quest_oracle.c``) behind a numpy interface.  Only the tests, the
package smoke check and the benchmark's CPU-baseline / reference leg may import this
package.  It shares no code with the CUDA library and never imports it.

fp16 inputs are widened to float32 (exact) before the C code sees them; bounding boxes
come back as fp16 (exact: each is one of the inputs).  Attention outputs are float64.

Parity status: every function here is pinned by CPU tests (tests/test_oracle_pins.py)
against invariants, closed forms, brute force and hand-worked fixtures; none is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "quest_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no contraction of a*b+c into FMA)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "max_pages",
        "num_phys")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            D = ctypes.POINTER(_Dims)
            lib.oq_build_meta.argtypes = [D, P, P, P, P]
            lib.oq_append.argtypes = [D, P, P, P, P, P, P, P]
            lib.oq_score.argtypes = [D, P, P, P, P, P]
            lib.oq_topk.argtypes = [D, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P]
            lib.oq_score_heads.argtypes = [D, P, P, P, P, P]
            lib.oq_topk_union.argtypes = [D, P, P, ctypes.c_int, ctypes.c_int, P, P]
            lib.oq_attend.argtypes = [D, P, P, P, P, P, P, P, ctypes.c_int, P, P]
            for f in (lib.oq_build_meta, lib.oq_append, lib.oq_score, lib.oq_topk,
                      lib.oq_score_heads, lib.oq_topk_union,
                      lib.oq_attend):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.float32)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=np.int32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class OracleError(RuntimeError):
    pass


@dataclass
class Cache:
    """Host copy of one paged cache (one layer).  Arrays are float32 / int32."""
    k_pool: np.ndarray       # [num_phys][Hkv][P][d] float32 (fp16 values)
    v_pool: np.ndarray
    meta: np.ndarray         # [num_phys][Hkv][2][d] float32 (fp16 values)
    block_table: np.ndarray  # [B][max_pages] int32
    seq_lens: np.ndarray     # [B] int32
    num_q_heads: int

    @staticmethod
    def from_arrays(k_pool, v_pool, block_table, seq_lens, num_q_heads: int,
                    meta=None) -> "Cache":
        k = _f32(k_pool).copy()
        v = _f32(v_pool).copy()
        if meta is None:
            meta = np.full((k.shape[0], k.shape[1], 2, k.shape[3]), np.nan, np.float32)
        return Cache(k, v, _f32(meta).copy(), _i32(block_table).copy(), _i32(seq_lens).copy(),
                     int(num_q_heads))

    def dims(self) -> _Dims:
        num_phys, hkv, P, d = self.k_pool.shape
        B, max_pages = self.block_table.shape
        return _Dims(B, self.num_q_heads, hkv, d, P, max_pages, num_phys)


def build_meta(c: Cache) -> np.ndarray:
    """Bounding boxes of every page of every sequence; updates ``c.meta`` in place and
    returns it as fp16."""
    dims = c.dims()
    rc = _load().oq_build_meta(ctypes.byref(dims), _ptr(c.k_pool), _ptr(c.block_table),
                               _ptr(c.seq_lens), _ptr(c.meta))
    if rc:
        raise OracleError("build_meta: bad block table entry or length")
    return c.meta.astype(np.float16)


def append(c: Cache, k_new, v_new) -> None:
    """Append one token per sequence ([B][Hkv][d]) at seq_lens[b]; seq_lens grows by 1."""
    dims = c.dims()
    kn, vn = _f32(k_new), _f32(v_new)
    rc = _load().oq_append(ctypes.byref(dims), _ptr(c.k_pool), _ptr(c.v_pool), _ptr(c.meta),
                           _ptr(c.block_table), _ptr(c.seq_lens), _ptr(kn), _ptr(vn))
    if rc:
        raise OracleError("append: page not allocated or cache full")


def prefill(c: Cache, k, v) -> None:
    """Chunked prefill: n tokens per sequence ([B][n][Hkv][d]) written in token order, each
    one exactly as ``append`` places it and widens its page's box ("Guide to Quest",
    Solution step 1: boxes are formed as pages fill, in prefill as in generation)."""
    kk, vv = _f32(k), _f32(v)
    for j in range(kk.shape[1]):
        append(c, kk[:, j], vv[:, j])


def score(c: Cache, q) -> np.ndarray:
    """Page scores [B][Hkv][max_pages] float32 (-inf past the last page)."""
    dims = c.dims()
    qq = _f32(q)
    out = np.empty((dims.batch, dims.num_kv_heads, dims.max_pages), np.float32)
    rc = _load().oq_score(ctypes.byref(dims), _ptr(qq), _ptr(c.meta), _ptr(c.block_table),
                          _ptr(c.seq_lens), _ptr(out))
    if rc:
        raise OracleError("score: bad block table entry or length")
    return out


def topk(c: Cache, scores, K: int, sink: int = 0, local: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Kept pages [B][Hkv][K] (-1 padded) and counts [B][Hkv]: with sink = local = 0 in
    rank order; otherwise the first `sink` and last `local` pages of every sequence longer
    than K pages, then the best of the others in rank order."""
    dims = c.dims()
    sc = _f32(scores)
    idx = np.empty((dims.batch, dims.num_kv_heads, K), np.int32)
    cnt = np.empty((dims.batch, dims.num_kv_heads), np.int32)
    rc = _load().oq_topk(ctypes.byref(dims), _ptr(sc), _ptr(c.seq_lens), int(K), int(sink),
                         int(local), _ptr(idx), _ptr(cnt))
    if rc:
        raise OracleError("topk: bad K, window or length")
    return idx, cnt


def score_heads(c: Cache, q) -> np.ndarray:
    """Per-query-head page scores [B][Hq][max_pages] float32 (-inf past the last page)."""
    dims = c.dims()
    qq = _f32(q)
    out = np.empty((dims.batch, dims.num_q_heads, dims.max_pages), np.float32)
    rc = _load().oq_score_heads(ctypes.byref(dims), _ptr(qq), _ptr(c.meta), _ptr(c.block_table),
                                _ptr(c.seq_lens), _ptr(out))
    if rc:
        raise OracleError("score_heads: bad block table entry or length")
    return out


def topk_union(c: Cache, scores_h, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """Union over each group's query heads of their top-K pages: idx [B][Hkv][min(G*K,
    max_pages)] ascending (-1 padded) and counts [B][Hkv]."""
    dims = c.dims()
    G = dims.num_q_heads // dims.num_kv_heads
    cap = min(G * K, dims.max_pages)
    sc = _f32(scores_h)
    idx = np.empty((dims.batch, dims.num_kv_heads, cap), np.int32)
    cnt = np.empty((dims.batch, dims.num_kv_heads), np.int32)
    rc = _load().oq_topk_union(ctypes.byref(dims), _ptr(sc), _ptr(c.seq_lens), int(K), int(cap),
                               _ptr(idx), _ptr(cnt))
    if rc:
        raise OracleError("topk_union: bad K or length")
    return idx, cnt


def attend(c: Cache, q, idx, count) -> Tuple[np.ndarray, np.ndarray]:
    """Exact attention over the kept pages: out [B][Hq][d] and lse [B][Hq], float64."""
    dims = c.dims()
    qq = _f32(q)
    ii, cc = _i32(idx), _i32(count)
    K = ii.shape[-1]
    out = np.empty((dims.batch, dims.num_q_heads, dims.head_dim), np.float64)
    lse = np.empty((dims.batch, dims.num_q_heads), np.float64)
    rc = _load().oq_attend(ctypes.byref(dims), _ptr(qq), _ptr(c.k_pool), _ptr(c.v_pool),
                           _ptr(c.block_table), _ptr(c.seq_lens), _ptr(ii), _ptr(cc), int(K),
                           _ptr(out), _ptr(lse))
    if rc:
        raise OracleError("attend: bad selection, block table entry or length")
    return out, lse


def all_pages(c: Cache) -> Tuple[np.ndarray, np.ndarray]:
    """A selection that keeps every page (used for dense attention)."""
    dims = c.dims()
    P = dims.page_size
    n = (c.seq_lens.astype(np.int64) + P - 1) // P
    K = max(1, int(n.max()) if n.size else 1)
    idx = np.full((dims.batch, dims.num_kv_heads, K), -1, np.int32)
    cnt = np.zeros((dims.batch, dims.num_kv_heads), np.int32)
    for b in range(dims.batch):
        idx[b, :, :n[b]] = np.arange(n[b], dtype=np.int32)
        cnt[b, :] = n[b]
    return idx, cnt


def dense(c: Cache, q) -> Tuple[np.ndarray, np.ndarray]:
    """Full-context attention (every page kept)."""
    idx, cnt = all_pages(c)
    return attend(c, q, idx, cnt)


def decode_step(c: Cache, q, K: int, k_new=None, v_new=None, sink: int = 0, local: int = 0):
    """One decode step: optional append, then score, select and attend.
    Returns (scores, idx, count, out, lse)."""
    if k_new is not None:
        append(c, k_new, v_new)
    s = score(c, q)
    idx, cnt = topk(c, s, K, sink, local)
    out, lse = attend(c, q, idx, cnt)
    return s, idx, cnt, out, lse
