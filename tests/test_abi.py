"""The C-ABI library builds, loads and exports every symbol include/quest.h declares; its
host-side argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import os
import re

import pytest

import query_aware_kv_gb300 as q
from query_aware_kv_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return q.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "quest.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quest_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(q.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.quest_version() == 1


def test_status_strings(lib):
    assert lib.quest_status_string(0) == b"QUEST_OK"
    assert lib.quest_status_string(q.QUEST_ERR_TIMEOUT) == b"QUEST_ERR_TIMEOUT"
    assert lib.quest_status_string(99) == b"QUEST_ERR_UNKNOWN"


def desc(**kw):
    base = dict(batch=1, num_q_heads=4, num_kv_heads=4, head_dim=128, page_size=16,
                max_pages=64, num_phys=64, k_pool=16, v_pool=32, meta=48, block_table=64,
                seq_lens=80)
    base.update(kw)
    return q.QuestCacheDesc(*[base[f] for f, _ in q.QuestCacheDesc._fields_])


@pytest.mark.parametrize("kw,needle", [
    (dict(head_dim=64), "head_dim"),
    (dict(page_size=8), "page_size"),
    (dict(num_q_heads=12, num_kv_heads=4), "group size"),
    (dict(num_q_heads=6, num_kv_heads=4), "multiple"),
    (dict(max_pages=q.QUEST_MAX_PAGES + 1), "max_pages"),
    (dict(k_pool=0), "NULL"),
    (dict(meta=40), "aligned"),
])
def test_workspace_size_rejects_bad_descriptors(lib, kw, needle):
    d = desc(**kw)
    assert lib.quest_workspace_size(ctypes.byref(d), 16, None) == 0
    assert needle in lib.quest_last_error().decode()


def test_workspace_size_grows_with_top_k(lib):
    d = desc()
    a = lib.quest_workspace_size(ctypes.byref(d), 16, None)
    b = lib.quest_workspace_size(ctypes.byref(d), 64, None)
    assert 0 < a < b
    assert lib.quest_workspace_size(ctypes.byref(d), 0, None) == 0


def test_calls_reject_bad_arguments_without_launching(lib):
    d = desc()
    assert lib.quest_decode(None, 16, 16, 16, None, None, None, 256, 1 << 20, None, None) == \
        q.QUEST_ERR_INVALID_ARG
    # NULL workspace
    assert lib.quest_decode(ctypes.byref(d), 16, 16, 16, None, None, None, None, 0, None,
                            None) == q.QUEST_ERR_WORKSPACE
    # workspace too small for this top_k
    assert lib.quest_sparse_decode(ctypes.byref(d), 16, 16, 16, 16, 16, None, 256, 1024, None,
                                   None) == q.QUEST_ERR_WORKSPACE
    assert "needs" in lib.quest_last_error().decode()
    # misaligned query
    assert lib.quest_estimate(ctypes.byref(d), 18, 16, 256, 1 << 20, None) == \
        q.QUEST_ERR_INVALID_ARG
    # top_k out of range
    assert lib.quest_topk(ctypes.byref(d), 16, 0, 16, 16, 256, 1 << 20, None, None) == \
        q.QUEST_ERR_INVALID_ARG
    # a sink / local window larger than the budget, or negative
    for sink, local in ((3, 2), (-1, 0), (0, -2)):
        o = q.opts(sink_pages=sink, local_pages=local)
        assert lib.quest_topk(ctypes.byref(d), 16, 4, 16, 16, 256, 1 << 20, ctypes.byref(o),
                              None) == q.QUEST_ERR_INVALID_ARG
        assert lib.quest_decode(ctypes.byref(d), 16, 4, 16, None, None, None, 256, 1 << 20,
                                ctypes.byref(o), None) == q.QUEST_ERR_INVALID_ARG
        assert "sink_pages" in lib.quest_last_error().decode()
    # the union selection does not combine with a sink / local window
    ou2 = q.opts(gqa_union=True, sink_pages=1)
    assert lib.quest_decode(ctypes.byref(d), 16, 4, 16, None, None, None, 256, 1 << 20,
                            ctypes.byref(ou2), None) == q.QUEST_ERR_INVALID_ARG
    assert lib.quest_topk(ctypes.byref(d), 16, 4, 16, 16, 256, 1 << 20, ctypes.byref(ou2),
                          None) == q.QUEST_ERR_INVALID_ARG
    # multi-layer call: layer count out of range, k_new for some layers only
    lay = (q.QuestLayer * 2)()
    for i in range(2):
        lay[i] = q.QuestLayer(16, 16, 16, 16, None, None, 16, None)
    assert lib.quest_decode_layers(ctypes.byref(d), lay, 0, 4, 256, 1 << 20, None, None) == \
        q.QUEST_ERR_INVALID_ARG
    assert lib.quest_decode_layers(ctypes.byref(d), lay, 33, 4, 256, 1 << 20, None, None) == \
        q.QUEST_ERR_INVALID_ARG
    lay[1].k_new, lay[1].v_new = 16, 16
    assert lib.quest_decode_layers(ctypes.byref(d), lay, 2, 4, 256, 1 << 20, None, None) == \
        q.QUEST_ERR_INVALID_ARG
    assert "k_new" in lib.quest_last_error().decode()
    # unsupported geometry
    d2 = desc(page_size=64)
    assert lib.quest_build_meta(ctypes.byref(d2), 256, 1 << 20, None) == q.QUEST_ERR_UNSUPPORTED
    # an empty batch is a no-op
    d3 = desc(batch=0)
    assert lib.quest_append(ctypes.byref(d3), 16, 16, 256, 1 << 20, None) == q.QUEST_OK


def test_decode_rejects_unknown_path(lib):
    d = desc()
    o = q.opts(path=4)
    ws = ctypes.c_void_p(1 << 20)  # never dereferenced: the call fails before any launch
    assert lib.quest_decode(ctypes.byref(d), 16, 16, 16, 256, 256, 256, ws,
                            1 << 40, ctypes.byref(o), None) == q.QUEST_ERR_INVALID_ARG
    assert "path" in lib.quest_last_error().decode()


def test_stream_path_is_chosen_on_request_and_bounded(lib):
    """QUEST_PATH_STREAM is taken when asked for (no device query needed); shapes beyond its
    on-chip tables (more than 1024 sequences, top_k above 2048) are refused."""
    d = desc()
    o = q.opts(path=q.QUEST_PATH_STREAM)
    assert lib.quest_decode_path(ctypes.byref(d), 16, ctypes.byref(o), 1) == q.QUEST_PATH_STREAM
    assert lib.quest_decode_path(ctypes.byref(d), 4096, ctypes.byref(o), 1) == \
        -q.QUEST_ERR_UNSUPPORTED
    big = desc(batch=2000, num_q_heads=1, num_kv_heads=1)
    assert lib.quest_decode_path(ctypes.byref(big), 16, ctypes.byref(o), 1) == \
        -q.QUEST_ERR_UNSUPPORTED
    assert "stream" in lib.quest_last_error().decode()


def test_decode_path_rejects_bad_arguments_without_querying(lib):
    d = desc()
    assert lib.quest_decode_path(ctypes.byref(d), 16, None, 0) == -q.QUEST_ERR_INVALID_ARG
    assert lib.quest_decode_path(ctypes.byref(d), 0, None, 1) == -q.QUEST_ERR_INVALID_ARG
    o = q.opts(path=5)
    assert lib.quest_decode_path(ctypes.byref(d), 16, ctypes.byref(o), 1) == \
        -q.QUEST_ERR_INVALID_ARG
    assert "path" in lib.quest_last_error().decode()


def test_prefill_rejects_bad_arguments_without_launching(lib):
    d = desc()
    ws = ctypes.create_string_buffer(1 << 12)
    assert lib.quest_prefill(ctypes.byref(d), 16, 16, -1, ws, 1 << 12, None) == \
        q.QUEST_ERR_INVALID_ARG
    assert lib.quest_prefill(ctypes.byref(d), 16, 16, 64 * 16 + 1, ws, 1 << 12, None) == \
        q.QUEST_ERR_INVALID_ARG
    assert lib.quest_prefill(ctypes.byref(d), 16, 24, 8, ws, 1 << 12, None) == \
        q.QUEST_ERR_INVALID_ARG
    assert "aligned" in lib.quest_last_error().decode()
    assert lib.quest_prefill(ctypes.byref(d), 16, 16, 8, None, 0, None) == q.QUEST_ERR_WORKSPACE
    # an empty chunk is a no-op, so it touches nothing
    assert lib.quest_prefill(ctypes.byref(d), 16, 16, 0, None, 0, None) == q.QUEST_OK


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from query_aware_kv_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load()


def _c_layout(tmp_path, struct, fields):
    """sizeof and offsetof of a quest.h struct as the C compiler lays it out."""
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "quest.h"', 'int main(void) {',
             f'  printf("%zu\\n", sizeof({struct}));']
    lines += [f'  printf("%zu\\n", offsetof({struct}, {f}));' for f in fields]
    lines += ['  return 0;', '}']
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    import subprocess
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                           str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split()
    return int(out[0]), [int(x) for x in out[1:]]


@pytest.mark.parametrize("struct,ctype", [("quest_cache_t", q.QuestCacheDesc),
                                          ("quest_opts_t", q.QuestOpts),
                                          ("quest_layer_t", q.QuestLayer)])
def test_binding_structs_match_the_header(tmp_path, struct, ctype):
    """The ctypes mirrors of the header's structs have the C compiler's size and field
    offsets, field by field."""
    fields = [f for f, _ in ctype._fields_]
    size, offsets = _c_layout(tmp_path, struct, fields)
    assert ctypes.sizeof(ctype) == size
    assert [getattr(ctype, f).offset for f in fields] == offsets


def test_binding_constants_match_the_header():
    """Every QUEST_* constant of the header that the binding mirrors has the header's value
    (read from the header text, so no compiler is involved)."""
    text = open(os.path.join(ROOT, "include", "quest.h")).read()
    defines = dict(re.findall(r"#define (QUEST_[A-Z_]+) (\d+)", text))
    mirrored = [n for n in dir(q) if n.startswith("QUEST_") and isinstance(getattr(q, n), int)]
    assert len(mirrored) >= 15
    for name in mirrored:
        assert name in defines, name
        assert int(defines[name]) == getattr(q, name), name


def test_decode_launches_without_a_device_query(lib):
    """One launch on the one-launch paths (asked for: no device query); bad arguments are
    refused as by quest_decode_path."""
    d = desc()
    for path in (q.QUEST_PATH_STREAM, q.QUEST_PATH_FUSED):
        o = q.opts(path=path)
        assert lib.quest_decode_launches(ctypes.byref(d), 16, ctypes.byref(o)) == 1
    assert lib.quest_decode_launches(ctypes.byref(d), 0, None) == -q.QUEST_ERR_INVALID_ARG
    o = q.opts(path=7)
    assert lib.quest_decode_launches(ctypes.byref(d), 16, ctypes.byref(o)) == \
        -q.QUEST_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(num_q_heads=16, num_kv_heads=4),
                                dict(max_pages=4097, num_phys=4097)],
                         ids=["gqa", "mha_4097_pages"])
def test_chain_keeps_the_topk_kernel_on_gqa_and_long_rows(lib, kw):
    """On GQA rows, and on rows longer than 4096 pages, the chain selects in a top-K kernel
    of its own whatever the GPU (three launches)."""
    d = desc(**kw)
    o = q.opts(path=q.QUEST_PATH_CHAIN)
    assert lib.quest_decode_path(ctypes.byref(d), 16, ctypes.byref(o), 1) == q.QUEST_PATH_CHAIN
    assert lib.quest_decode_launches(ctypes.byref(d), 16, ctypes.byref(o)) == 3


def test_union_form_runs_on_the_chain(lib):
    """gqa_union on the fused calls: the chain (no device query), three launches, a larger
    workspace (per-head scores, union rows); the one-launch paths refuse it."""
    d = desc(num_q_heads=16, num_kv_heads=4)
    o = q.opts(gqa_union=True)
    assert lib.quest_decode_path(ctypes.byref(d), 8, ctypes.byref(o), 1) == q.QUEST_PATH_CHAIN
    assert lib.quest_decode_launches(ctypes.byref(d), 8, ctypes.byref(o)) == 3
    assert lib.quest_workspace_size(ctypes.byref(d), 8, ctypes.byref(o)) > \
        lib.quest_workspace_size(ctypes.byref(d), 8, None)
    for path in (q.QUEST_PATH_FUSED, q.QUEST_PATH_STREAM):
        o = q.opts(gqa_union=True, path=path)
        assert lib.quest_decode_path(ctypes.byref(d), 8, ctypes.byref(o), 1) == \
            -q.QUEST_ERR_UNSUPPORTED
    o = q.opts(gqa_union=True)
    assert lib.quest_decode_path(ctypes.byref(d), 8, ctypes.byref(o), 2) == \
        -q.QUEST_ERR_UNSUPPORTED
