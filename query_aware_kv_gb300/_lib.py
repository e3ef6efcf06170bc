"""ctypes binding of libquest.so (C ABI in include/quest.h).

Argument marshalling only: tensors are checked for device, dtype, shape and contiguity,
their device pointers and the current CUDA stream are handed to the library, and a
non-zero status becomes a ``QuestError``.  Every step of the decode path runs in the
library's kernels; there is no fallback.  The library must have been built
(``__graft_entry__.build()`` or ``python -m query_aware_kv_gb300.build``); if it is
missing, loading fails with an error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Sequence, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libquest.so")

QUEST_OK = 0
QUEST_ERR_INVALID_ARG = 1
QUEST_ERR_UNSUPPORTED = 2
QUEST_ERR_WORKSPACE = 3
QUEST_ERR_CUDA = 4
QUEST_ERR_TIMEOUT = 5
QUEST_ERR_BAD_PAGE = 6
QUEST_ERR_BAD_LENGTH = 7
QUEST_ERR_BAD_SELECTION = 8
QUEST_MAX_PAGES = 16384
QUEST_DEBUG_WITHHOLD_SELECTION = 1
QUEST_PATH_AUTO, QUEST_PATH_FUSED, QUEST_PATH_CHAIN, QUEST_PATH_STREAM = 0, 1, 2, 3
HEAD_DIM = 128

# Every symbol include/quest.h declares.
EXPORTS = (
    "quest_workspace_size", "quest_workspace_init", "quest_build_meta", "quest_append",
    "quest_prefill",
    "quest_estimate", "quest_estimate_heads", "quest_topk", "quest_sparse_decode",
    "quest_decode", "quest_decode_layers", "quest_decode_path", "quest_decode_launches",
    "quest_decode_step", "quest_dense_decode", "quest_decode_static", "quest_read_status",
    "quest_last_error", "quest_status_string", "quest_version",
)


class QuestError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class QuestCacheDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
        ("num_phys", ctypes.c_int32),
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("meta", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
    ]


class QuestLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("k_pool", "v_pool", "meta", "q", "k_new", "v_new", "out", "lse")]


class QuestOpts(ctypes.Structure):
    _fields_ = [
        ("pages_per_split", ctypes.c_int32), ("score_tile_pages", ctypes.c_int32),
        ("max_ctas", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
        ("wait_limit_ns", ctypes.c_int64), ("reserved", ctypes.c_int32),
        ("trace_capacity", ctypes.c_int32), ("trace", ctypes.c_void_p),
        ("cluster_size", ctypes.c_int32), ("sink_pages", ctypes.c_int32),
        ("local_pages", ctypes.c_int32), ("gqa_union", ctypes.c_int32),
        ("path", ctypes.c_int32),
    ]


_lib = None
_lock = threading.Lock()


def load() -> ctypes.CDLL:
    """Load libquest.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                "(the Quest kernels have no fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        V, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        C = ctypes.POINTER(QuestCacheDesc)
        O = ctypes.POINTER(QuestOpts)
        sig = {
            "quest_workspace_size": (SZ, [C, I32, O]),
            "quest_workspace_init": (ctypes.c_int, [V, SZ, V]),
            "quest_build_meta": (ctypes.c_int, [C, V, SZ, V]),
            "quest_append": (ctypes.c_int, [C, V, V, V, SZ, V]),
            "quest_prefill": (ctypes.c_int, [C, V, V, I32, V, SZ, V]),
            "quest_estimate": (ctypes.c_int, [C, V, V, V, SZ, V]),
            "quest_estimate_heads": (ctypes.c_int, [C, V, V, V, SZ, V]),
            "quest_topk": (ctypes.c_int, [C, V, I32, V, V, V, SZ, O, V]),
            "quest_sparse_decode": (ctypes.c_int, [C, V, V, V, I32, V, V, V, SZ, O, V]),
            "quest_decode": (ctypes.c_int, [C, V, I32, V, V, V, V, V, SZ, O, V]),
            "quest_decode_step": (ctypes.c_int, [C, V, V, V, I32, V, V, V, V, V, SZ, O, V]),
            "quest_decode_layers": (ctypes.c_int, [C, ctypes.POINTER(QuestLayer), I32, I32, V,
                                                   SZ, O, V]),
            "quest_decode_path": (ctypes.c_int, [C, I32, O, I32]),
            "quest_decode_launches": (ctypes.c_int, [C, I32, O]),
            "quest_dense_decode": (ctypes.c_int, [C, V, V, V, V, SZ, O, V]),
            "quest_read_status": (ctypes.c_int, [V, SZ, V, ctypes.POINTER(I32)]),
            "quest_last_error": (ctypes.c_char_p, []),
            "quest_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "quest_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(rc: int) -> None:
    if rc != QUEST_OK:
        lib = load()
        raise QuestError(rc, lib.quest_last_error().decode() or lib.quest_status_string(rc).decode())


def _stream(stream: Optional[torch.cuda.Stream]) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def opts(pages_per_split: int = 0, score_tile_pages: int = 0, max_ctas: int = 0,
         debug_flags: int = 0, wait_limit_ns: int = 0, trace: Optional[torch.Tensor] = None,
         cluster_size: int = 0, sink_pages: int = 0, local_pages: int = 0,
         gqa_union: bool = False, path: int = 0) -> QuestOpts:
    """Launch tuning (0 = default).  ``trace``: int64 CUDA tensor of 1 + 2n elements whose
    first element is zero; receives up to n timeline records of a one-launch kernel.
    ``sink_pages`` / ``local_pages``: pages always kept at the start / end of a sequence
    longer than top_k pages.  ``path``: QUEST_PATH_AUTO / _FUSED / _CHAIN / _STREAM for the
    decode calls."""
    cap, ptr = 0, None
    if trace is not None:
        _need(trace, "trace", torch.int64)
        cap, ptr = (trace.numel() - 1) // 2, trace.data_ptr()
    o = QuestOpts(pages_per_split, score_tile_pages, max_ctas, debug_flags, wait_limit_ns,
                  0, cap, ptr, cluster_size, sink_pages, local_pages, int(gqa_union),
                  int(path))
    o._trace_ref = trace  # keep the buffer alive with the options
    return o


def _opts_ref(o: Optional[QuestOpts]):
    return None if o is None else ctypes.byref(o)


def _sel_row(cache, top_k: int, o: Optional[QuestOpts]) -> int:
    """Entries of a selection row of the decode calls: top_k, or min(G * top_k, max_pages)
    in the union form (o.gqa_union)."""
    if o is not None and o.gqa_union:
        G = cache.desc.num_q_heads // cache.num_kv_heads
        return min(G * int(top_k), cache.max_pages)
    return int(top_k)


@dataclass
class PagedCache:
    """One layer's paged fp16 KV cache with per-page key min/max (device tensors).

    k_pool, v_pool: [num_phys][Hkv][P][128] fp16; meta: [B][Hkv][max_pages][2][128] fp16
    (boxes per sequence, logical page order); block_table: [B][max_pages] int32;
    seq_lens: [B] int32 (advanced by ``append`` / ``decode_step``).
    """
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    meta: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    num_q_heads: int

    def __post_init__(self):
        num_phys, hkv, P, d = self.k_pool.shape
        B, max_pages = self.block_table.shape
        _need(self.k_pool, "k_pool", torch.float16)
        _need(self.v_pool, "v_pool", torch.float16, self.k_pool.shape)
        _need(self.meta, "meta", torch.float16, (B, hkv, max_pages, 2, d))
        _need(self.block_table, "block_table", torch.int32)
        _need(self.seq_lens, "seq_lens", torch.int32, (B,))
        self.desc = QuestCacheDesc(B, int(self.num_q_heads), hkv, d, P, max_pages, num_phys,
                                   self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                                   self.meta.data_ptr(), self.block_table.data_ptr(),
                                   self.seq_lens.data_ptr())

    @classmethod
    def allocate_meta(cls, k_pool, v_pool, block_table, seq_lens, num_q_heads):
        num_phys, hkv, P, d = k_pool.shape
        B, max_pages = block_table.shape
        meta = torch.zeros((B, hkv, max_pages, 2, d), dtype=torch.float16, device=k_pool.device)
        return cls(k_pool, v_pool, meta, block_table, seq_lens, num_q_heads)

    @property
    def batch(self) -> int:
        return self.desc.batch

    @property
    def num_kv_heads(self) -> int:
        return self.desc.num_kv_heads

    @property
    def max_pages(self) -> int:
        return self.desc.max_pages

    @property
    def page_size(self) -> int:
        return self.desc.page_size


def workspace_size(cache: PagedCache, top_k: int, o: Optional[QuestOpts] = None) -> int:
    lib = load()
    n = lib.quest_workspace_size(ctypes.byref(cache.desc), int(top_k), _opts_ref(o))
    if n == 0:
        raise QuestError(QUEST_ERR_INVALID_ARG, lib.quest_last_error().decode())
    return int(n)


def workspace(cache: PagedCache, top_k: int, o: Optional[QuestOpts] = None) -> torch.Tensor:
    """A zeroed workspace for every call on this cache with this top_k / opts."""
    n = workspace_size(cache, top_k, o)
    return torch.zeros(n, dtype=torch.uint8, device=cache.k_pool.device)


def workspace_init(ws: torch.Tensor, stream=None) -> None:
    _check(load().quest_workspace_init(ws.data_ptr(), ws.numel(), _stream(stream)))


def build_meta(cache: PagedCache, ws: torch.Tensor, stream=None) -> None:
    _check(load().quest_build_meta(ctypes.byref(cache.desc), ws.data_ptr(), ws.numel(),
                                   _stream(stream)))


def append(cache: PagedCache, k_new: torch.Tensor, v_new: torch.Tensor, ws: torch.Tensor,
           stream=None) -> None:
    shape = (cache.batch, cache.num_kv_heads, HEAD_DIM)
    _need(k_new, "k_new", torch.float16, shape)
    _need(v_new, "v_new", torch.float16, shape)
    _check(load().quest_append(ctypes.byref(cache.desc), k_new.data_ptr(), v_new.data_ptr(),
                               ws.data_ptr(), ws.numel(), _stream(stream)))


def prefill(cache: PagedCache, k: torch.Tensor, v: torch.Tensor, ws: torch.Tensor,
            stream=None) -> None:
    """Write a chunk of n tokens per sequence ([B][n][Hkv][128] fp16) at seq_lens and fold
    it into the page boxes; seq_lens grows by n."""
    if k.dim() != 4:
        raise ValueError("k must be [batch][n_tokens][num_kv_heads][128]")
    shape = (cache.batch, k.shape[1], cache.num_kv_heads, HEAD_DIM)
    _need(k, "k", torch.float16, shape)
    _need(v, "v", torch.float16, shape)
    _check(load().quest_prefill(ctypes.byref(cache.desc), k.data_ptr(), v.data_ptr(),
                                int(k.shape[1]), ws.data_ptr(), ws.numel(), _stream(stream)))


def estimate(cache: PagedCache, q: torch.Tensor, ws: torch.Tensor,
             scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    shape = (cache.batch, cache.num_kv_heads, cache.max_pages)
    if scores is None:
        scores = torch.empty(shape, dtype=torch.float32, device=q.device)
    _need(scores, "scores", torch.float32, shape)
    _check(load().quest_estimate(ctypes.byref(cache.desc), q.data_ptr(), scores.data_ptr(),
                                 ws.data_ptr(), ws.numel(), _stream(stream)))
    return scores


def estimate_heads(cache: PagedCache, q: torch.Tensor, ws: torch.Tensor,
                   scores: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Per-query-head page bounds [B][Hq][max_pages] (input of the union selection)."""
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    shape = (cache.batch, cache.desc.num_q_heads, cache.max_pages)
    if scores is None:
        scores = torch.empty(shape, dtype=torch.float32, device=q.device)
    _need(scores, "scores", torch.float32, shape)
    _check(load().quest_estimate_heads(ctypes.byref(cache.desc), q.data_ptr(), scores.data_ptr(),
                                       ws.data_ptr(), ws.numel(), _stream(stream)))
    return scores


def topk(cache: PagedCache, scores: torch.Tensor, top_k: int, ws: torch.Tensor,
         o: Optional[QuestOpts] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Kept pages (ascending, -1 padded) and counts.  With o.gqa_union the scores are per
    query head and the rows hold min(G * top_k, max_pages) entries."""
    union = o is not None and bool(o.gqa_union)
    rows = cache.desc.num_q_heads if union else cache.num_kv_heads
    _need(scores, "scores", torch.float32, (cache.batch, rows, cache.max_pages))
    G = cache.desc.num_q_heads // cache.num_kv_heads
    cap = min(G * top_k, cache.max_pages) if union else top_k
    idx = torch.empty((cache.batch, cache.num_kv_heads, cap), dtype=torch.int32,
                      device=scores.device)
    cnt = torch.empty((cache.batch, cache.num_kv_heads), dtype=torch.int32, device=scores.device)
    _check(load().quest_topk(ctypes.byref(cache.desc), scores.data_ptr(), int(top_k),
                             idx.data_ptr(), cnt.data_ptr(), ws.data_ptr(), ws.numel(),
                             _opts_ref(o), _stream(stream)))
    return idx, cnt


def _out(cache: PagedCache, q: torch.Tensor, out, lse, want_lse: bool):
    B, Hq = cache.batch, cache.desc.num_q_heads
    if out is None:
        out = torch.empty((B, Hq, HEAD_DIM), dtype=torch.float16, device=q.device)
    _need(out, "out", torch.float16, (B, Hq, HEAD_DIM))
    if lse is None and want_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, "lse", torch.float32, (B, Hq))
    return out, lse


def sparse_decode(cache: PagedCache, q: torch.Tensor, idx: torch.Tensor, count: torch.Tensor,
                  top_k: int, ws: torch.Tensor, o: Optional[QuestOpts] = None, out=None,
                  lse=None, want_lse: bool = True, stream=None):
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    _need(idx, "idx", torch.int32, (cache.batch, cache.num_kv_heads, top_k))
    _need(count, "count", torch.int32, (cache.batch, cache.num_kv_heads))
    out, lse = _out(cache, q, out, lse, want_lse)
    _check(load().quest_sparse_decode(ctypes.byref(cache.desc), q.data_ptr(), idx.data_ptr(),
                                      count.data_ptr(), int(top_k), out.data_ptr(), _ptr(lse),
                                      ws.data_ptr(), ws.numel(), _opts_ref(o), _stream(stream)))
    return out, lse


def decode(cache: PagedCache, q: torch.Tensor, top_k: int, ws: torch.Tensor,
           o: Optional[QuestOpts] = None, out=None, lse=None, want_lse: bool = True,
           idx_out: Optional[torch.Tensor] = None, count_out: Optional[torch.Tensor] = None,
           stream=None):
    """Estimate + top-K + sparse decode: one launch of the cluster or the stream kernel, or
    a chain of kernels (o.path; automatic by default, see decode_path).  With o.gqa_union
    the selection is the union of every query head's top-K (rows of min(G * top_k,
    max_pages) in idx_out), on the chain."""
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    out, lse = _out(cache, q, out, lse, want_lse)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32,
              (cache.batch, cache.num_kv_heads, _sel_row(cache, top_k, o)))
    if count_out is not None:
        _need(count_out, "count_out", torch.int32, (cache.batch, cache.num_kv_heads))
    _check(load().quest_decode(ctypes.byref(cache.desc), q.data_ptr(), int(top_k), out.data_ptr(),
                               _ptr(lse), _ptr(idx_out), _ptr(count_out), ws.data_ptr(),
                               ws.numel(), _opts_ref(o), _stream(stream)))
    return out, lse


def decode_step(cache: PagedCache, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                top_k: int, ws: torch.Tensor, o: Optional[QuestOpts] = None, out=None, lse=None,
                want_lse: bool = True, idx_out: Optional[torch.Tensor] = None,
                count_out: Optional[torch.Tensor] = None, stream=None):
    """Append (k_new, v_new) and run the decode step over the cache that holds them: one
    launch, or the chain with the append folded into its estimate (o.path)."""
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    shape = (cache.batch, cache.num_kv_heads, HEAD_DIM)
    _need(k_new, "k_new", torch.float16, shape)
    _need(v_new, "v_new", torch.float16, shape)
    out, lse = _out(cache, q, out, lse, want_lse)
    if idx_out is not None:
        _need(idx_out, "idx_out", torch.int32,
              (cache.batch, cache.num_kv_heads, _sel_row(cache, top_k, o)))
    if count_out is not None:
        _need(count_out, "count_out", torch.int32, (cache.batch, cache.num_kv_heads))
    _check(load().quest_decode_step(ctypes.byref(cache.desc), q.data_ptr(), k_new.data_ptr(),
                                    v_new.data_ptr(), int(top_k), out.data_ptr(), _ptr(lse),
                                    _ptr(idx_out), _ptr(count_out), ws.data_ptr(), ws.numel(),
                                    _opts_ref(o), _stream(stream)))
    return out, lse


class DecodePlan:
    """quest_decode / quest_decode_step bound to one cache, top_k, workspace, options, stream
    and set of output buffers, for a decode loop.  Everything but the step's own tensors is
    checked once, here; each call then only checks that q (and k_new, v_new) have the shape,
    dtype and device fixed here and are contiguous, and goes straight to the C entry point
    (the argument checks of ``decode`` / ``decode_step`` cost the host several microseconds
    a call).  ``stream``: the stream every call is issued on (default: the current stream at
    construction).  The outputs (``out``, ``lse``, ``idx_out``, ``count_out``) are
    overwritten by every call and returned by it."""

    def __init__(self, cache: PagedCache, top_k: int, ws: torch.Tensor,
                 o: Optional[QuestOpts] = None, out=None, lse=None, want_lse: bool = True,
                 idx_out: Optional[torch.Tensor] = None,
                 count_out: Optional[torch.Tensor] = None, stream=None):
        B, Hq, Hkv = cache.batch, cache.desc.num_q_heads, cache.num_kv_heads
        self._qshape = torch.Size((B, Hq, HEAD_DIM))
        self._kvshape = torch.Size((B, Hkv, HEAD_DIM))
        self._dev = cache.k_pool.get_device()
        probe = torch.empty(0, dtype=torch.float16, device=cache.k_pool.device)
        self.out, self.lse = _out(cache, probe, out, lse, want_lse)
        if idx_out is not None:
            _need(idx_out, "idx_out", torch.int32, (B, Hkv, _sel_row(cache, top_k, o)))
        if count_out is not None:
            _need(count_out, "count_out", torch.int32, (B, Hkv))
        _need(ws, "ws", torch.uint8)
        self.idx_out, self.count_out = idx_out, count_out
        self._keep = (cache, ws, o)  # alive as long as the plan
        self._lib = load()
        self._desc = ctypes.byref(cache.desc)
        # the arguments after q (and k_new, v_new), in C order
        self._tail = (int(top_k), self.out.data_ptr(), _ptr(self.lse), _ptr(idx_out),
                      _ptr(count_out), ws.data_ptr(), ws.numel(), _opts_ref(o), _stream(stream))

    def _ok(self, t, shape) -> bool:
        return (type(t) is torch.Tensor and t.dtype is torch.float16 and t.shape == shape and
                t.get_device() == self._dev and t.is_contiguous())

    def decode(self, q: torch.Tensor):
        """quest_decode of this step's queries; returns (out, lse)."""
        if not self._ok(q, self._qshape):
            _need(q, "q", torch.float16, self._qshape)
            raise ValueError("q is on another device than the cache")
        rc = self._lib.quest_decode(self._desc, q.data_ptr(), *self._tail)
        if rc:
            _check(rc)
        return self.out, self.lse

    def step(self, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor):
        """quest_decode_step: append (k_new, v_new), then decode q; returns (out, lse)."""
        if not (self._ok(q, self._qshape) and self._ok(k_new, self._kvshape) and
                self._ok(v_new, self._kvshape)):
            _need(q, "q", torch.float16, self._qshape)
            _need(k_new, "k_new", torch.float16, self._kvshape)
            _need(v_new, "v_new", torch.float16, self._kvshape)
            raise ValueError("q / k_new / v_new are on another device than the cache")
        t = self._tail
        rc = self._lib.quest_decode_step(self._desc, q.data_ptr(), k_new.data_ptr(),
                                         v_new.data_ptr(), *t)
        if rc:
            _check(rc)
        return self.out, self.lse


def decode_layers(cache: PagedCache, layers: Sequence[PagedCache], q: Sequence[torch.Tensor],
                  top_k: int, ws: torch.Tensor, o: Optional[QuestOpts] = None,
                  k_new: Optional[Sequence[torch.Tensor]] = None,
                  v_new: Optional[Sequence[torch.Tensor]] = None, out=None, lse=None,
                  want_lse: bool = True, stream=None):
    """The step of every layer in one call (one launch, or the layers as chains: o.path).
    `cache` holds the shared shape, block table and lengths; `layers[i]` holds layer i's
    pools and boxes (same shape); with k_new / v_new every layer appends its token and the
    lengths advance once."""
    n = len(layers)
    if len(q) != n or (k_new is not None and (len(k_new) != n or len(v_new) != n)):
        raise ValueError("one q (and k_new, v_new) per layer")
    outs = list(out) if out is not None else [None] * n
    lses = list(lse) if lse is not None else [None] * n
    arr = (QuestLayer * max(n, 1))()
    keep = []
    for i, lay in enumerate(layers):
        if (lay.k_pool.shape != cache.k_pool.shape or lay.meta.shape != cache.meta.shape):
            raise ValueError(f"layer {i}: pools / boxes differ in shape from the cache")
        _need(q[i], "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
        outs[i], lses[i] = _out(cache, q[i], outs[i], lses[i], want_lse)
        kn = vn = None
        if k_new is not None:
            shape = (cache.batch, cache.num_kv_heads, HEAD_DIM)
            _need(k_new[i], "k_new", torch.float16, shape)
            _need(v_new[i], "v_new", torch.float16, shape)
            kn, vn = k_new[i].data_ptr(), v_new[i].data_ptr()
        arr[i] = QuestLayer(lay.k_pool.data_ptr(), lay.v_pool.data_ptr(), lay.meta.data_ptr(),
                            q[i].data_ptr(), kn, vn, outs[i].data_ptr(), _ptr(lses[i]))
    keep.append(arr)
    _check(load().quest_decode_layers(ctypes.byref(cache.desc), arr, int(n), int(top_k),
                                      ws.data_ptr(), ws.numel(), _opts_ref(o), _stream(stream)))
    return outs, lses


def dense_decode(cache: PagedCache, q: torch.Tensor, ws: torch.Tensor,
                 o: Optional[QuestOpts] = None, out=None, lse=None, want_lse: bool = True,
                 stream=None):
    _need(q, "q", torch.float16, (cache.batch, cache.desc.num_q_heads, HEAD_DIM))
    out, lse = _out(cache, q, out, lse, want_lse)
    _check(load().quest_dense_decode(ctypes.byref(cache.desc), q.data_ptr(), out.data_ptr(),
                                     _ptr(lse), ws.data_ptr(), ws.numel(), _opts_ref(o),
                                     _stream(stream)))
    return out, lse


def decode_path(cache: PagedCache, top_k: int, o: Optional[QuestOpts] = None,
                n_layers: int = 1) -> int:
    """QUEST_PATH_FUSED, _CHAIN or _STREAM: the path the decode calls take for this cache,
    top_k and options."""
    lib = load()
    r = lib.quest_decode_path(ctypes.byref(cache.desc), int(top_k), _opts_ref(o), int(n_layers))
    if r < 0:
        raise QuestError(-r, lib.quest_last_error().decode())
    return int(r)


def decode_launches(cache: PagedCache, top_k: int, o: Optional[QuestOpts] = None) -> int:
    """Kernel launches of one decode / decode_step call for this cache, top_k and options."""
    lib = load()
    r = lib.quest_decode_launches(ctypes.byref(cache.desc), int(top_k), _opts_ref(o))
    if r < 0:
        raise QuestError(-r, lib.quest_last_error().decode())
    return int(r)


def read_status(ws: torch.Tensor, stream=None) -> Tuple[int, Tuple[int, int, int]]:
    """Synchronise, return (device status, (sequence, page, site)) and clear the status."""
    detail = (ctypes.c_int32 * 3)()
    rc = load().quest_read_status(ws.data_ptr(), ws.numel(), _stream(stream), detail)
    return int(rc), (int(detail[0]), int(detail[1]), int(detail[2]))
