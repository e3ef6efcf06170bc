// quest_api.cu - the C ABI of libquest.so (declared in include/quest.h): host-side
// argument checks, work decomposition, workspace layout and kernel dispatch.  No call
// allocates memory or synchronises, except quest_read_status.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "quest_internal.h"

using namespace quest;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(QUEST_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

size_t up256(size_t x) { return (x + 255) / 256 * 256; }

int check_cache(const quest_cache_t* c) {
  if (!c) return fail(QUEST_ERR_INVALID_ARG, "cache descriptor is NULL");
  if (c->head_dim != kHeadDim)
    return fail(QUEST_ERR_UNSUPPORTED, "head_dim %d: only 128 is supported", c->head_dim);
  if (c->page_size != 16 && c->page_size != 32)
    return fail(QUEST_ERR_UNSUPPORTED, "page_size %d: only 16 and 32 are supported", c->page_size);
  if (c->batch < 0 || c->num_q_heads < 1 || c->num_kv_heads < 1 || c->max_pages < 1 ||
      c->num_phys < 1)
    return fail(QUEST_ERR_INVALID_ARG,
                "bad sizes: batch %d, num_q_heads %d, num_kv_heads %d, max_pages %d, num_phys %d",
                c->batch, c->num_q_heads, c->num_kv_heads, c->max_pages, c->num_phys);
  if (c->num_q_heads % c->num_kv_heads)
    return fail(QUEST_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                c->num_q_heads, c->num_kv_heads);
  const int G = c->num_q_heads / c->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8)
    return fail(QUEST_ERR_UNSUPPORTED, "group size %d: only 1, 2, 4, 8 are supported", G);
  if (c->max_pages > QUEST_MAX_PAGES)
    return fail(QUEST_ERR_UNSUPPORTED, "max_pages %d exceeds %d", c->max_pages, QUEST_MAX_PAGES);
  if ((long long)c->batch * c->num_kv_heads > 65535)
    return fail(QUEST_ERR_UNSUPPORTED, "batch * num_kv_heads exceeds 65535");
  if (c->batch == 0) return QUEST_OK;
  if (!c->k_pool || !c->v_pool || !c->meta || !c->block_table || !c->seq_lens)
    return fail(QUEST_ERR_INVALID_ARG, "a cache pointer is NULL");
  if (!aligned(c->k_pool, 16) || !aligned(c->v_pool, 16) || !aligned(c->meta, 16) ||
      !aligned(c->block_table, 4) || !aligned(c->seq_lens, 4))
    return fail(QUEST_ERR_INVALID_ARG, "pools and meta must be 16-byte aligned");
  return QUEST_OK;
}

int check_topk(int top_k) {
  if (top_k < 1 || top_k > QUEST_MAX_PAGES)
    return fail(QUEST_ERR_INVALID_ARG, "top_k %d outside [1, %d]", top_k, QUEST_MAX_PAGES);
  return QUEST_OK;
}

int check_window(const quest_opts_t* o, int top_k) {
  if (!o) return QUEST_OK;
  if (o->sink_pages < 0 || o->local_pages < 0 ||
      (long long)o->sink_pages + o->local_pages > (long long)top_k)
    return fail(QUEST_ERR_INVALID_ARG,
                "sink_pages %d and local_pages %d must be >= 0 with a sum <= top_k %d",
                o->sink_pages, o->local_pages, top_k);
  return QUEST_OK;
}

Tiling make_tiling(const quest_cache_t* c, int top_k, const quest_opts_t* o) {
  Tiling t{};
  t.topk_cap = top_k;
  t.score_rows = 1;
  if (o && o->gqa_union) {  // a fused call in the union form: per-head scores, union rows
    const int G = c->num_kv_heads > 0 ? c->num_q_heads / c->num_kv_heads : 1;
    t.topk_cap = (int)std::min<long long>((long long)G * top_k, c->max_pages);
    t.score_rows = G;
  }
  int stp = (o && o->score_tile_pages > 0) ? o->score_tile_pages : kDefaultScoreTilePages;
  if (stp > c->max_pages) stp = c->max_pages;
  t.score_tile_pages = stp;
  t.n_score_tiles = (int)cdiv(c->max_pages, stp);
  const int user_pps = (o && o->pages_per_split > 0) ? o->pages_per_split : 0;
  const int pps = user_pps ? user_pps : kDefaultPagesPerSplit;
  const int kcap = t.topk_cap < c->max_pages ? t.topk_cap : c->max_pages;
  // by default about 8 sparse work items per (sequence, kv head), of at least 16 pages: a
  // work item of a few pages spends most of its time filling its ring and merging
  t.pps_sparse = user_pps ? (int)std::max<long long>(user_pps, cdiv(kcap, kMaxSplits))
                          : (int)std::max<long long>(kMinSparsePagesPerSplit, cdiv(kcap, 8));
  t.n_splits_sparse = (int)cdiv(kcap, t.pps_sparse);
  t.pps_dense = (int)std::max<long long>(pps, cdiv(c->max_pages, 64));
  t.n_splits_dense = (int)cdiv(c->max_pages, t.pps_dense);
  t.max_splits = std::max(t.n_splits_sparse, t.n_splits_dense);
  // the stream kernel writes one partial per decode piece of kStreamPiecePages kept pages
  t.max_splits = std::max<int>(t.max_splits, (int)cdiv(kcap, kStreamPiecePages));
  return t;
}

WsLayout make_layout(const quest_cache_t* c, const Tiling& t) {
  WsLayout L{};
  const size_t nbg = (size_t)c->batch * c->num_kv_heads;
  const size_t nbh = (size_t)c->batch * c->num_q_heads;
  size_t off = sizeof(WsHeader);
  L.score_arrive = off;  off = up256(off + nbg * 4);
  L.ready = off;         off = up256(off + nbg * 4);
  L.decode_arrive = off; off = up256(off + nbg * 4);
  L.seq_done = off;      off = up256(off + (size_t)c->batch * 4);
  L.skeys = off;         off = up256(off + nbg * c->max_pages * 4);
  L.scores = off;        off = up256(off + nbg * t.score_rows * c->max_pages * 4);
  L.sel_idx = off;       off = up256(off + nbg * (size_t)t.topk_cap * 4);
  L.sel_count = off;     off = up256(off + nbg * 4);
  L.part_ml = off;       off = up256(off + nbh * t.max_splits * 2 * 4);
  L.part_acc = off;      off = up256(off + nbh * t.max_splits * kHeadDim * 4);
  L.sel_pair = off;      off = up256(off + nbg * (size_t)t.topk_cap * 8);
  L.total = off;
  return L;
}

Params make_params(const quest_cache_t* c, void* ws, const WsLayout& L, const Tiling& t,
                   const quest_opts_t* o) {
  Params p{};
  p.B = c->batch;
  p.Hq = c->num_q_heads;
  p.Hkv = c->num_kv_heads;
  p.P = c->page_size;
  p.max_pages = c->max_pages;
  p.num_phys = c->num_phys;
  p.k_pool = static_cast<__half*>(c->k_pool);
  p.v_pool = static_cast<__half*>(c->v_pool);
  p.meta = static_cast<__half*>(c->meta);
  p.block_table = c->block_table;
  p.seq_lens = c->seq_lens;
  unsigned char* w = static_cast<unsigned char*>(ws);
  WsHeader* h = reinterpret_cast<WsHeader*>(w);
  p.status = &h->status;
  p.exited = &h->exited;
  p.score_arrive = reinterpret_cast<unsigned*>(w + L.score_arrive);
  p.ready = reinterpret_cast<unsigned*>(w + L.ready);
  p.decode_arrive = reinterpret_cast<unsigned*>(w + L.decode_arrive);
  p.seq_done = reinterpret_cast<unsigned*>(w + L.seq_done);
  p.scores = reinterpret_cast<float*>(w + L.scores);
  p.sel_idx = reinterpret_cast<int*>(w + L.sel_idx);
  p.sel_count = reinterpret_cast<int*>(w + L.sel_count);
  p.part_ml = reinterpret_cast<float*>(w + L.part_ml);
  p.part_acc = reinterpret_cast<float*>(w + L.part_acc);
  p.sel_pair = reinterpret_cast<int*>(w + L.sel_pair);
  p.skeys = reinterpret_cast<unsigned*>(w + L.skeys);
  p.started = &h->started;
  p.top_k = t.topk_cap;
  p.score_tile_pages = t.score_tile_pages;
  p.n_score_tiles = t.n_score_tiles;
  p.wait_limit_ns = (o && o->wait_limit_ns > 0) ? o->wait_limit_ns : kDefaultWaitNs;
  p.debug_flags = o ? o->debug_flags : 0;
  p.sink_pages = o ? o->sink_pages : 0;
  p.local_pages = o ? o->local_pages : 0;
  p.qscale = (float)(1.4426950408889634 / std::sqrt((double)kHeadDim));
  return p;
}

// Common checks of the workspace; `need` = bytes this call requires.
int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(QUEST_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(QUEST_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(QUEST_ERR_WORKSPACE, "workspace has %zu bytes, this call needs %zu", ws_bytes, need);
  return QUEST_OK;
}

int launched(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  return QUEST_OK;
}

int group_of(const quest_cache_t* c) { return c->num_q_heads / c->num_kv_heads; }

}  // namespace

namespace quest {

int decode_workspace_requirement(const quest_cache_t* cache, int top_k, size_t* total,
                                 size_t* zeroed) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_topk(top_k))) return rc;
  const WsLayout L = make_layout(cache, make_tiling(cache, top_k, nullptr));
  *total = L.total;
  *zeroed = L.scores;
  return QUEST_OK;
}

int set_last_error(int code, const char* message) { return fail(code, "%s", message); }

}  // namespace quest

extern "C" {

int quest_version(void) { return QUEST_VERSION; }

const char* quest_last_error(void) { return g_err.c_str(); }

const char* quest_status_string(int code) {
  switch (code) {
    case QUEST_OK: return "QUEST_OK";
    case QUEST_ERR_INVALID_ARG: return "QUEST_ERR_INVALID_ARG";
    case QUEST_ERR_UNSUPPORTED: return "QUEST_ERR_UNSUPPORTED";
    case QUEST_ERR_WORKSPACE: return "QUEST_ERR_WORKSPACE";
    case QUEST_ERR_CUDA: return "QUEST_ERR_CUDA";
    case QUEST_ERR_TIMEOUT: return "QUEST_ERR_TIMEOUT";
    case QUEST_ERR_BAD_PAGE: return "QUEST_ERR_BAD_PAGE";
    case QUEST_ERR_BAD_LENGTH: return "QUEST_ERR_BAD_LENGTH";
    case QUEST_ERR_BAD_SELECTION: return "QUEST_ERR_BAD_SELECTION";
    default: return "QUEST_ERR_UNKNOWN";
  }
}

size_t quest_workspace_size(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts) {
  if (check_cache(cache) != QUEST_OK || check_topk(top_k) != QUEST_OK) return 0;
  return make_layout(cache, make_tiling(cache, top_k, opts)).total;
}

int quest_workspace_init(void* ws, size_t ws_bytes, quest_stream_t stream) {
  if (!ws) return fail(QUEST_ERR_WORKSPACE, "workspace is NULL");
  return launched(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)),
                  "cudaMemsetAsync(workspace)");
}

int quest_build_meta(const quest_cache_t* cache, void* ws, size_t ws_bytes, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, 1, nullptr);
  const Params p = make_params(cache, ws, make_layout(cache, t), t, nullptr);
  return launched(launch_build_meta(p, static_cast<cudaStream_t>(stream)), "quest_build_meta");
}

int quest_append(const quest_cache_t* cache, const void* k_new, const void* v_new, void* ws,
                 size_t ws_bytes, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(QUEST_ERR_INVALID_ARG, "k_new / v_new must be non-NULL and 16-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, 1, nullptr);
  const Params p = make_params(cache, ws, make_layout(cache, t), t, nullptr);
  return launched(launch_append(p, static_cast<const __half*>(k_new),
                                static_cast<const __half*>(v_new),
                                static_cast<cudaStream_t>(stream)),
                  "quest_append");
}

int quest_prefill(const quest_cache_t* cache, const void* k, const void* v, int32_t n_tokens,
                  void* ws, size_t ws_bytes, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (n_tokens < 0) return fail(QUEST_ERR_INVALID_ARG, "n_tokens must be >= 0");
  if (cache->batch == 0 || n_tokens == 0) return QUEST_OK;
  if ((long long)n_tokens > (long long)cache->max_pages * cache->page_size)
    return fail(QUEST_ERR_INVALID_ARG, "n_tokens exceeds max_pages * page_size");
  if (!k || !v || !aligned(k, 16) || !aligned(v, 16))
    return fail(QUEST_ERR_INVALID_ARG, "k / v must be non-NULL and 16-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, 1, nullptr);
  const Params p = make_params(cache, ws, make_layout(cache, t), t, nullptr);
  return launched(launch_prefill(p, static_cast<const __half*>(k), static_cast<const __half*>(v),
                                 n_tokens, static_cast<cudaStream_t>(stream)),
                  "quest_prefill");
}

int quest_estimate(const quest_cache_t* cache, const void* q, float* scores, void* ws,
                   size_t ws_bytes, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!q || !scores || !aligned(q, 16) || !aligned(scores, 4))
    return fail(QUEST_ERR_INVALID_ARG, "q must be 16-byte aligned, scores 4-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, 1, nullptr);
  Params p = make_params(cache, ws, make_layout(cache, t), t, nullptr);
  p.q = static_cast<const __half*>(q);
  p.scores = scores;
  return launched(launch_estimate(p, group_of(cache), false, static_cast<cudaStream_t>(stream)),
                  "quest_estimate");
}

int quest_estimate_heads(const quest_cache_t* cache, const void* q, float* scores, void* ws,
                         size_t ws_bytes, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!q || !scores || !aligned(q, 16) || !aligned(scores, 4))
    return fail(QUEST_ERR_INVALID_ARG, "q must be 16-byte aligned, scores 4-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, 1, nullptr);
  Params p = make_params(cache, ws, make_layout(cache, t), t, nullptr);
  p.q = static_cast<const __half*>(q);
  p.scores = scores;
  return launched(launch_estimate(p, group_of(cache), true, static_cast<cudaStream_t>(stream)),
                  "quest_estimate_heads");
}

int quest_topk(const quest_cache_t* cache, const float* scores, int32_t top_k, int32_t* idx,
               int32_t* count, void* ws, size_t ws_bytes, const quest_opts_t* opts,
               quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_topk(top_k))) return rc;
  if ((rc = check_window(opts, top_k))) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!scores || !idx || !count || !aligned(scores, 4) || !aligned(idx, 4) || !aligned(count, 4))
    return fail(QUEST_ERR_INVALID_ARG, "scores / idx / count must be non-NULL and 4-byte aligned");
  if ((rc = check_ws(ws, ws_bytes, sizeof(WsHeader)))) return rc;
  const Tiling t = make_tiling(cache, top_k, nullptr);
  Params p = make_params(cache, ws, make_layout(cache, t), t, opts);
  p.scores = const_cast<float*>(scores);
  p.sel_idx = idx;
  p.sel_count = count;
  p.top_k = top_k;
  if (opts && opts->gqa_union) {
    if (opts->sink_pages || opts->local_pages)
      return fail(QUEST_ERR_INVALID_ARG, "gqa_union does not combine with sink / local pages");
    const long long cap = std::min((long long)group_of(cache) * top_k, (long long)cache->max_pages);
    return launched(launch_topk_union(p, (int)cap, static_cast<cudaStream_t>(stream)),
                    "quest_topk");
  }
  return launched(launch_topk(p, static_cast<cudaStream_t>(stream)), "quest_topk");
}

int quest_sparse_decode(const quest_cache_t* cache, const void* q, const int32_t* idx,
                        const int32_t* count, int32_t top_k, void* out, float* lse, void* ws,
                        size_t ws_bytes, const quest_opts_t* opts, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_topk(top_k))) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!q || !idx || !count || !out || !aligned(q, 16) || !aligned(out, 16) || !aligned(idx, 4) ||
      !aligned(count, 4) || !aligned(lse, 4))
    return fail(QUEST_ERR_INVALID_ARG, "q / idx / count / out must be non-NULL and aligned");
  const Tiling t = make_tiling(cache, top_k, opts);
  const WsLayout L = make_layout(cache, t);
  if ((rc = check_ws(ws, ws_bytes, L.total))) return rc;
  Params p = make_params(cache, ws, L, t, opts);
  p.q = static_cast<const __half*>(q);
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  p.sel_idx = const_cast<int*>(idx);
  p.sel_count = const_cast<int*>(count);
  p.top_k = top_k;
  p.pps = t.pps_sparse;
  p.n_splits = t.n_splits_sparse;
  p.dense = 0;
  return launched(launch_decode(p, group_of(cache), static_cast<cudaStream_t>(stream)),
                  "quest_sparse_decode");
}

// The automatic choice between the one-launch cluster kernel and the chain depends only on
// the device and the shape; it takes occupancy queries, so it is made once per device and
// shape and remembered.
static cudaError_t auto_path_fused(int G, int P, int max_pages, int top_k, int nbg,
                                   bool* fused) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, bool> memo;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, G, P, max_pages, top_k, nbg);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = memo.find(key);
    if (it != memo.end()) {
      *fused = it->second;
      return cudaSuccess;
    }
  }
  bool f = false;
  if (cluster_any_fits(G, P, max_pages, top_k) &&
      (e = cluster_preferred(G, P, max_pages, top_k, nbg, &f)) != cudaSuccess)
    return e;
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = f;
  *fused = f;
  return cudaSuccess;
}

// Where a chain decode call selects its pages.  For MHA rows of at most 4096 pages whose
// decode work items fit on the GPU about twice over, every work item takes its pair's top-K
// itself (the redundant selections run on SMs that would otherwise idle, and the top-K
// kernel, its launch and the selection's round trip through global memory drop out of the
// step); otherwise the top-K kernel selects once per pair, with 16 warps, and also resolves
// every kept page's physical page for the decode kernel.  Measured on GB300 (quest_decode,
// L2 flushed): 32K MHA 31.5 against 32.2 us, 8 ragged 8K-32K sequences at budget 256 54.0
// against 56.4; but the 128K row (8192 pages) 54.1 against 50.9 and GQA-4 at page 32 62.8
// against 60.7, where the longer selection or the heavier decode work item makes the
// redundant top-K the longer path.
static void set_chain_selection(Params& p) {
  static std::mutex mu;
  static int sms[64] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    std::lock_guard<std::mutex> lock(mu);
    if (!sms[dev & 63]) cudaDeviceGetAttribute(&sms[dev & 63], cudaDevAttrMultiProcessorCount, dev);
    n = sms[dev & 63];
  }
  const long long items = (long long)p.B * p.Hkv * p.n_splits;
  p.chain_select = (n > 0 && items <= 2LL * n && p.Hq == p.Hkv && p.max_pages <= 4096) ? 1 : 0;
  p.chain_pairs = 1 - p.chain_select;
}

// The path of a decode call (QUEST_PATH_FUSED, _CHAIN or _STREAM in quest.h).
static int decide_path(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts,
                       int n_layers, int* path_out) {
  const int cs = opts ? opts->cluster_size : 0;
  if (cs < 0 || cs > kMaxClusterSize)
    return fail(QUEST_ERR_INVALID_ARG, "cluster_size %d: use 0 (automatic) or 1..%d", cs,
                kMaxClusterSize);
  const int path = opts ? opts->path : QUEST_PATH_AUTO;
  if (path < QUEST_PATH_AUTO || path > QUEST_PATH_STREAM)
    return fail(QUEST_ERR_INVALID_ARG, "path %d: use QUEST_PATH_AUTO, _FUSED, _CHAIN or _STREAM",
                path);
  const int G = group_of(cache);
  if (opts && opts->gqa_union) {  // the union form runs as a chain of kernels only
    if (path == QUEST_PATH_FUSED || path == QUEST_PATH_STREAM || cs > 0)
      return fail(QUEST_ERR_UNSUPPORTED, "gqa_union runs on the chain path only (its one-launch "
                  "kernels select per kv head)");
    if (n_layers > 1)
      return fail(QUEST_ERR_UNSUPPORTED, "gqa_union: quest_decode_layers selects per kv head");
    *path_out = QUEST_PATH_CHAIN;
    return QUEST_OK;
  }
  if (path == QUEST_PATH_STREAM) {
    if (stream_slots(G, cache->page_size, cache->max_pages, top_k, cache->batch,
                     cache->num_q_heads) <= 0)
      return fail(QUEST_ERR_UNSUPPORTED,
                  "the stream kernel does not fit this shape (batch %d, max_pages %d, top_k %d)",
                  cache->batch, cache->max_pages, top_k);
    *path_out = QUEST_PATH_STREAM;
    return QUEST_OK;
  }
  *path_out = path == QUEST_PATH_CHAIN ? QUEST_PATH_CHAIN : QUEST_PATH_FUSED;
  if (path == QUEST_PATH_AUTO && cs == 0 && !(opts && (opts->trace || opts->debug_flags))) {
    bool fused = false;
    const long long nbg = (long long)n_layers * cache->batch * cache->num_kv_heads;
    const cudaError_t e = auto_path_fused(G, cache->page_size, cache->max_pages, top_k,
                                          (int)std::min<long long>(nbg, 0x7fffffff), &fused);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy of the one-launch kernel");
    *path_out = fused ? QUEST_PATH_FUSED : QUEST_PATH_CHAIN;
  }
  return QUEST_OK;
}

static int decode_impl(const quest_cache_t* cache, const void* q, const void* k_new,
                       const void* v_new, int32_t top_k, void* out, float* lse, int32_t* idx_out,
                       int32_t* count_out, void* ws, size_t ws_bytes, const quest_opts_t* opts,
                       quest_stream_t stream, const char* what) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_topk(top_k))) return rc;
  if ((rc = check_window(opts, top_k))) return rc;
  const bool uni = opts && opts->gqa_union;
  if (uni && (opts->sink_pages || opts->local_pages))
    return fail(QUEST_ERR_INVALID_ARG, "gqa_union does not combine with sink / local pages");
  if (cache->batch == 0) return QUEST_OK;
  if (!q || !out || !aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(idx_out, 4) || !aligned(count_out, 4))
    return fail(QUEST_ERR_INVALID_ARG, "q / out must be non-NULL and aligned");
  if ((k_new == nullptr) != (v_new == nullptr) || !aligned(k_new, 16) || !aligned(v_new, 16))
    return fail(QUEST_ERR_INVALID_ARG, "k_new and v_new must both be NULL or both 16-byte aligned");
  if (opts && opts->trace && (opts->trace_capacity < 0 || !aligned(opts->trace, 8)))
    return fail(QUEST_ERR_INVALID_ARG, "trace must be 8-byte aligned with trace_capacity >= 0");
  const Tiling t = make_tiling(cache, top_k, opts);
  const WsLayout L = make_layout(cache, t);
  if ((rc = check_ws(ws, ws_bytes, L.total))) return rc;
  Params p = make_params(cache, ws, L, t, opts);
  p.q = static_cast<const __half*>(q);
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  if (idx_out) p.sel_idx = idx_out;
  if (count_out) p.sel_count = count_out;
  p.top_k = top_k;
  p.pps = t.pps_sparse;
  p.n_splits = t.n_splits_sparse;
  p.dense = 0;
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.trace = opts ? reinterpret_cast<unsigned long long*>(opts->trace) : nullptr;
  p.trace_capacity = opts ? opts->trace_capacity : 0;
  const int cs = opts ? opts->cluster_size : 0;  // 0: the library picks
  const int G = group_of(cache);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  int path = QUEST_PATH_FUSED;
  if ((rc = decide_path(cache, top_k, opts, 1, &path))) return rc;
  if (path == QUEST_PATH_STREAM) {
    // one persistent launch over the whole GPU; the selection is written out only when asked
    p.chain_append = p.k_new != nullptr ? 1 : 0;
    p.n_splits = (int)cdiv(std::min(top_k, cache->max_pages), kStreamPiecePages);
    p.sel_idx = idx_out;
    p.sel_count = count_out;
    const LayerPtrs lay{p.k_pool, p.v_pool, p.meta, p.q, p.k_new, p.v_new, p.out, p.lse};
    return launched(launch_stream(p, lay, G, opts ? opts->max_ctas : 0, s), what);
  }
  if (path == QUEST_PATH_CHAIN && uni) {
    // the union form of the group-level selection ("Guide to Quest", Best Practices step
    // 2): the new token first (the lengths advance with it), then every query head's
    // bounds, each head's top-K and their union per kv head (rows of topk_cap), and the
    // sparse decode over the union; the selection goes to idx_out / count_out (rows of
    // topk_cap) if given
    const int cap = t.topk_cap;
    cudaError_t e = cudaSuccess;
    if (k_new) e = launch_append(p, p.k_new, p.v_new, s, true);
    p.chain_append = 0;
    p.k_new = p.v_new = nullptr;
    if (e == cudaSuccess) e = launch_estimate(p, G, true, s);
    if (e == cudaSuccess) e = launch_topk_union(p, cap, s);
    Params d = p;
    d.top_k = cap;  // row stride of the union selection
    if (e == cudaSuccess) e = launch_decode(d, G, s);
    return launched(e, what);
  }
  if (path == QUEST_PATH_CHAIN) {
    // the same step as separate kernels: estimate (which also writes the new token's row
    // and widens its box), top-K (its own kernel, or inside every decode work item: see
    // set_chain_selection), sparse decode (which advances the lengths at its end); the
    // selection goes to idx_out / count_out if given, else to the workspace
    p.chain_append = p.k_new != nullptr ? 1 : 0;
    set_chain_selection(p);
    cudaError_t e = launch_estimate(p, G, false, s);
    if (e == cudaSuccess && !p.chain_select) e = launch_topk(p, s);
    if (e == cudaSuccess) e = launch_decode(p, G, s);
    return launched(e, what);
  }
  if (!cluster_any_fits(G, cache->page_size, cache->max_pages, top_k))
    return fail(QUEST_ERR_UNSUPPORTED, "max_pages %d needs more shared memory than a CTA has",
                cache->max_pages);
  if (cs > 0 && cluster_smem_bytes(G, cache->page_size, cache->max_pages, cs, top_k) > kMaxSmem)
    return fail(QUEST_ERR_UNSUPPORTED, "cluster_size %d needs more shared memory than a CTA has",
                cs);
  p.sel_idx = idx_out;     // the cluster kernel writes the selection only when asked
  p.sel_count = count_out;
  LayerTable lt{};
  lt.n = 1;
  lt.l[0] = LayerPtrs{p.k_pool, p.v_pool, p.meta, p.q, p.k_new, p.v_new, p.out, p.lse};
  return launched(launch_cluster(p, lt, G, cs, opts ? opts->max_ctas : 0, s), what);
}

int quest_decode_launches(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts) {
  int rc = check_cache(cache);
  if (rc) return -rc;
  if ((rc = check_topk(top_k))) return -rc;
  int path = QUEST_PATH_FUSED;
  if ((rc = decide_path(cache, top_k, opts, 1, &path))) return -rc;
  if (path != QUEST_PATH_CHAIN) return 1;
  if (opts && opts->gqa_union) return 3;  // per-head bounds, union top-K, sparse decode
  const Tiling t = make_tiling(cache, top_k, opts);
  Params p{};
  p.B = cache->batch;
  p.Hq = cache->num_q_heads;
  p.Hkv = cache->num_kv_heads;
  p.max_pages = cache->max_pages;
  p.n_splits = t.n_splits_sparse;
  set_chain_selection(p);
  return p.chain_select ? 2 : 3;
}

int quest_decode_path(const quest_cache_t* cache, int32_t top_k, const quest_opts_t* opts,
                      int32_t n_layers) {
  int rc = check_cache(cache);
  if (rc) return -rc;
  if ((rc = check_topk(top_k))) return -rc;
  if (n_layers < 1 || n_layers > QUEST_MAX_LAYERS)
    return -fail(QUEST_ERR_INVALID_ARG, "n_layers %d: use 1..%d", n_layers, QUEST_MAX_LAYERS);
  int path = QUEST_PATH_FUSED;
  if ((rc = decide_path(cache, top_k, opts, n_layers, &path))) return -rc;
  return path;
}

int quest_decode(const quest_cache_t* cache, const void* q, int32_t top_k, void* out, float* lse,
                 int32_t* idx_out, int32_t* count_out, void* ws, size_t ws_bytes,
                 const quest_opts_t* opts, quest_stream_t stream) {
  return decode_impl(cache, q, nullptr, nullptr, top_k, out, lse, idx_out, count_out, ws,
                     ws_bytes, opts, stream, "quest_decode");
}

int quest_decode_step(const quest_cache_t* cache, const void* q, const void* k_new,
                      const void* v_new, int32_t top_k, void* out, float* lse, int32_t* idx_out,
                      int32_t* count_out, void* ws, size_t ws_bytes, const quest_opts_t* opts,
                      quest_stream_t stream) {
  if (!k_new || !v_new)
    return fail(QUEST_ERR_INVALID_ARG, "quest_decode_step needs k_new and v_new");
  return decode_impl(cache, q, k_new, v_new, top_k, out, lse, idx_out, count_out, ws, ws_bytes,
                     opts, stream, "quest_decode_step");
}

static_assert(kMaxLayers == QUEST_MAX_LAYERS, "layer table size");

int quest_decode_layers(const quest_cache_t* cache, const quest_layer_t* layers, int32_t n_layers,
                        int32_t top_k, void* ws, size_t ws_bytes, const quest_opts_t* opts,
                        quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_topk(top_k))) return rc;
  if ((rc = check_window(opts, top_k))) return rc;
  if (opts && opts->gqa_union)
    return fail(QUEST_ERR_UNSUPPORTED, "gqa_union: the fused step selects per kv head");
  if (!layers || n_layers < 1 || n_layers > QUEST_MAX_LAYERS)
    return fail(QUEST_ERR_INVALID_ARG, "n_layers %d: use 1..%d layers", n_layers, QUEST_MAX_LAYERS);
  if (cache->batch == 0) return QUEST_OK;
  if ((long long)n_layers * cache->batch * cache->num_kv_heads > 0x7fffffffLL)
    return fail(QUEST_ERR_UNSUPPORTED, "too many (layer, sequence, kv head) pairs");
  const bool append = layers[0].k_new != nullptr;
  LayerTable lt{};
  lt.n = n_layers;
  for (int i = 0; i < n_layers; ++i) {
    const quest_layer_t& L = layers[i];
    if (!L.k_pool || !L.v_pool || !L.meta || !L.q || !L.out || !aligned(L.k_pool, 16) ||
        !aligned(L.v_pool, 16) || !aligned(L.meta, 16) || !aligned(L.q, 16) ||
        !aligned(L.out, 16) || !aligned(L.lse, 4))
      return fail(QUEST_ERR_INVALID_ARG, "layer %d: pools, boxes, q and out must be non-NULL "
                  "and 16-byte aligned", i);
    if ((L.k_new != nullptr) != append || (L.v_new != nullptr) != append ||
        !aligned(L.k_new, 16) || !aligned(L.v_new, 16))
      return fail(QUEST_ERR_INVALID_ARG, "layer %d: k_new / v_new must be given (16-byte "
                  "aligned) for every layer or for none", i);
    lt.l[i] = LayerPtrs{static_cast<__half*>(L.k_pool), static_cast<__half*>(L.v_pool),
                        static_cast<__half*>(L.meta), static_cast<const __half*>(L.q),
                        static_cast<const __half*>(L.k_new), static_cast<const __half*>(L.v_new),
                        static_cast<__half*>(L.out), L.lse};
  }
  const Tiling t = make_tiling(cache, top_k, opts);
  const WsLayout Lw = make_layout(cache, t);
  if ((rc = check_ws(ws, ws_bytes, Lw.total))) return rc;
  Params p = make_params(cache, ws, Lw, t, opts);
  p.top_k = top_k;
  p.dense = 0;
  p.q = lt.l[0].q;
  p.out = lt.l[0].out;
  p.lse = lt.l[0].lse;
  p.k_new = lt.l[0].k_new;  // non-NULL: every layer appends, lengths advance once
  p.v_new = lt.l[0].v_new;
  p.sel_idx = nullptr;
  p.sel_count = nullptr;
  p.trace = opts ? reinterpret_cast<unsigned long long*>(opts->trace) : nullptr;
  p.trace_capacity = opts ? opts->trace_capacity : 0;
  const int cs = opts ? opts->cluster_size : 0;
  const int G = group_of(cache);
  int path = QUEST_PATH_FUSED;
  if ((rc = decide_path(cache, top_k, opts, n_layers, &path))) return rc;
  const bool fits = cluster_any_fits(G, cache->page_size, cache->max_pages, top_k);
  if (path == QUEST_PATH_STREAM) {
    // one stream launch per layer; every layer appends its token at the same position and
    // only the last launch advances the lengths
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    Params c = make_params(cache, ws, Lw, t, opts);
    c.top_k = top_k;
    c.dense = 0;
    c.n_splits = (int)cdiv(std::min(top_k, cache->max_pages), kStreamPiecePages);
    c.chain_append = append ? 1 : 0;
    c.sel_idx = nullptr;
    c.sel_count = nullptr;
    c.trace = p.trace;
    c.trace_capacity = p.trace_capacity;
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
      Params l = c;
      l.k_pool = lt.l[i].k_pool;
      l.v_pool = lt.l[i].v_pool;
      l.meta = lt.l[i].meta;
      l.hold_lengths = i + 1 < n_layers ? 1 : 0;
      e = launch_stream(l, lt.l[i], G, opts ? opts->max_ctas : 0, s);
    }
    return launched(e, "quest_decode_layers");
  }
  if (path == QUEST_PATH_CHAIN) {
    // layer after layer as separate kernels: every layer's token row and box first (at the
    // same position), the lengths advanced once, then each layer's estimate, top-K and
    // sparse decode over the cache that holds the new token
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    Params c = make_params(cache, ws, Lw, t, opts);
    c.top_k = top_k;
    c.pps = t.pps_sparse;
    c.n_splits = t.n_splits_sparse;
    c.dense = 0;
    set_chain_selection(c);
    auto at = [&](int i) {
      Params l = c;
      l.k_pool = lt.l[i].k_pool;
      l.v_pool = lt.l[i].v_pool;
      l.meta = lt.l[i].meta;
      l.q = lt.l[i].q;
      l.out = lt.l[i].out;
      l.lse = lt.l[i].lse;
      return l;
    };
    cudaError_t e = cudaSuccess;
    if (append) {
      for (int i = 0; i < n_layers && e == cudaSuccess; ++i)
        e = launch_append(at(i), lt.l[i].k_new, lt.l[i].v_new, s, false);
      if (e == cudaSuccess) e = launch_advance_lengths(c, 1, s);
    }
    for (int i = 0; i < n_layers && e == cudaSuccess; ++i) {
      const Params l = at(i);
      e = launch_estimate(l, G, false, s);
      if (e == cudaSuccess && !l.chain_select) e = launch_topk(l, s);
      if (e == cudaSuccess) e = launch_decode(l, G, s);
    }
    return launched(e, "quest_decode_layers");
  }
  if (!fits)
    return fail(QUEST_ERR_UNSUPPORTED, "max_pages %d needs more shared memory than a CTA has",
                cache->max_pages);
  if (cs > 0 &&
      cluster_smem_bytes(G, cache->page_size, cache->max_pages, cs, top_k) > kMaxSmem)
    return fail(QUEST_ERR_UNSUPPORTED, "cluster_size %d needs more shared memory than a CTA has",
                cs);
  return launched(launch_cluster(p, lt, G, cs, opts ? opts->max_ctas : 0,
                                 static_cast<cudaStream_t>(stream)),
                  "quest_decode_layers");
}

int quest_dense_decode(const quest_cache_t* cache, const void* q, void* out, float* lse, void* ws,
                       size_t ws_bytes, const quest_opts_t* opts, quest_stream_t stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->batch == 0) return QUEST_OK;
  if (!q || !out || !aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return fail(QUEST_ERR_INVALID_ARG, "q / out must be non-NULL and aligned");
  const Tiling t = make_tiling(cache, 1, opts);
  const WsLayout L = make_layout(cache, t);
  if ((rc = check_ws(ws, ws_bytes, L.total))) return rc;
  Params p = make_params(cache, ws, L, t, opts);
  p.q = static_cast<const __half*>(q);
  p.out = static_cast<__half*>(out);
  p.lse = lse;
  p.top_k = cache->max_pages;
  p.pps = t.pps_dense;
  p.n_splits = t.n_splits_dense;
  p.dense = 1;
  return launched(launch_decode(p, group_of(cache), static_cast<cudaStream_t>(stream)),
                  "quest_dense_decode");
}

int quest_read_status(void* ws, size_t ws_bytes, quest_stream_t stream, int32_t* detail) {
  if (!ws || ws_bytes < sizeof(WsHeader)) return fail(QUEST_ERR_WORKSPACE, "workspace too small");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int h[4] = {0, 0, 0, 0};
  e = cudaMemcpy(h, ws, sizeof(h), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status)");
  if (detail) {
    detail[0] = h[1];
    detail[1] = h[2];
    detail[2] = h[3];
  }
  if (h[0] != QUEST_OK) {
    e = cudaMemset(ws, 0, sizeof(h));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
    fail(h[0], "device reported %s (sequence %d, page %d, site %d)", quest_status_string(h[0]),
         h[1], h[2], h[3]);
  }
  return h[0];
}

}  // extern "C"
