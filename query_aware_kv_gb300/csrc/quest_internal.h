// quest_internal.h - declarations shared by the CUDA translation units of libquest.so.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "quest.h"

namespace quest {

constexpr int kHeadDim = 128;
constexpr int kConsumerWarps = 8;           // warps that compute
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kDecodeThreads = kConsumerThreads + 32;  // + one copy-producer warp
constexpr int kStages = 8;                  // smem ring depth (pages in flight per CTA)
constexpr int kMaxSplits = 256;             // split-K partials per (sequence, q head)
constexpr int kDefaultPagesPerSplit = 8;    // dense decode work items (at least)
constexpr int kMinSparsePagesPerSplit = 16;  // sparse decode work items, by default
constexpr int kDefaultScoreTilePages = 128;
constexpr long long kDefaultWaitNs = 1000000000LL;

// Places in the code that record a device fault (third detail word).
enum FaultSite : int {
  kSiteMeta = 1, kSiteAppend = 2, kSiteScore = 3, kSiteTopk = 4, kSiteDecode = 5,
  kSiteWaitSelection = 6, kSiteWaitStage = 7, kSiteWaitSlot = 8, kSiteSelection = 9,
};

// First 256 bytes of the workspace.
struct WsHeader {
  int status;        // QUEST_OK or the first QUEST_ERR_* the device saw
  int detail[3];     // sequence, logical page, fault site
  unsigned exited;   // cluster kernel: CTAs that have left (the last advances the lengths)
  unsigned started;  // stream kernel: CTAs that have read the lengths of an appending step
  unsigned pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct Tiling {
  int topk_cap;          // slots per selection row: top_k (min(G * top_k, max_pages) for the
                         // union form of a fused call)
  int score_rows;        // score rows per (b, kv head): 1, or G for the union form
  int score_tile_pages;  // pages per scoring work item
  int n_score_tiles;     // scoring work items per (b, g)
  int pps_sparse, n_splits_sparse;  // selected pages per decode item, items per (b, g)
  int pps_dense, n_splits_dense;
  int max_splits;
};

struct WsLayout {
  size_t score_arrive, ready, decode_arrive;  // u32 [B*Hkv] each
  size_t seq_done;                            // u32 [B]
  size_t skeys;                               // u32 [B*Hkv*max_pages] stream kernel's key
                                              // rows (0 = not written yet; kept zero)
  size_t scores;                              // f32 [B*Hkv*score_rows*max_pages]
  size_t sel_idx, sel_count;                  // i32 [B*Hkv*topk_cap], [B*Hkv]
  size_t part_ml, part_acc;                   // f32 [B*Hq*max_splits*2], [..*128]
  size_t sel_pair;                            // i32x2 [B*Hkv*topk_cap] (logical, physical)
  size_t total;
};

// Everything a kernel needs, passed by value.
struct Params {
  int B, Hq, Hkv, P, max_pages, num_phys;
  __half* k_pool;
  __half* v_pool;
  __half* meta;
  const int* block_table;
  int* seq_lens;

  const __half* q;       // [B][Hq][128]
  __half* out;           // [B][Hq][128]
  float* lse;            // [B][Hq] or null
  float* scores;         // [B][Hkv][max_pages]
  int* sel_idx;          // [B][Hkv][top_k]
  int* sel_count;        // [B][Hkv]
  int top_k;             // row length of sel_idx (= requested K, capped at max_pages)
  int sink_pages, local_pages;  // pages always kept at the start / end of a long sequence

  int score_tile_pages, n_score_tiles;
  int pps, n_splits;     // decode work-item size and count per (b, g)
  int dense;             // decode every page instead of a selection

  int* status;           // -> WsHeader::status (detail follows it)
  unsigned* exited;
  unsigned* score_arrive;
  unsigned* ready;
  unsigned* decode_arrive;
  float* part_ml;        // [B][Hq][n_splits][2]  (running max in log2 units, sum)
  float* part_acc;       // [B][Hq][n_splits][128]

  long long wait_limit_ns;
  int debug_flags;
  float qscale;          // log2(e) / sqrt(128)

  unsigned* seq_done;    // chain decode: kv heads of a sequence merged so far
  int chain_append;      // chain and stream kernel: the step appends k_new; every kernel
                         // sees seq_lens + 1 (when there is room) and the last step of the
                         // call advances seq_lens
  int* sel_pair;         // stream kernel and chain: [B][Hkv][top_k] (logical, physical page)
  int chain_pairs;       // chain: topk_kernel also writes sel_pair, decode_kernel reads it
  int chain_select;      // chain: every decode work item takes its pair's top-K itself
  unsigned* skeys;       // stream kernel: [B][Hkv][max_pages] page keys, 0 until written
  unsigned* started;     // stream kernel: CTAs that have read the lengths
  int hold_lengths;      // stream kernel: append, but leave seq_lens to a later launch
  int sel_ctas;          // stream kernel: the last sel_ctas CTAs of the grid select and merge
  int ring_slots;        // stream kernel: stages in each streaming CTA's ring
                         // (every layer but the last of a multi-layer step)
  const __half* k_new;   // fused step: token appended per (b, g) before scoring, or null
  const __half* v_new;
  unsigned long long* trace;  // one-launch kernels: optional timeline (quest_opts_t.trace)
  int trace_capacity;
};

// Launch with programmatic dependent launch allowed: the kernel may start while the
// previous kernel on the stream finishes; every kernel calls griddepcontrol.wait before
// touching memory an earlier kernel wrote.
inline cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// Dynamic shared memory of the decode-capable kernels (bytes), see quest_device.cuh.
size_t decode_smem_bytes(int G, int P, int topk_keys, int score_tile_pages);
// Raise a kernel's dynamic shared-memory cap (once per device and kernel).
// Per-layer tensors of a multi-layer fused step (the shape, block table and lengths are
// shared by every layer).  Passed by value as a kernel parameter.
struct LayerPtrs {
  __half* k_pool;
  __half* v_pool;
  __half* meta;
  const __half* q;
  const __half* k_new;
  const __half* v_new;
  __half* out;
  float* lse;
};
constexpr int kMaxLayers = 32;
struct LayerTable {
  int n;
  int pad;
  LayerPtrs l[kMaxLayers];
};

cudaError_t ensure_smem(const void* fn, size_t bytes);

// Host-side checks of quest_decode's cache / top_k arguments (status code, error text
// set), and the workspace bytes it needs: `total`, of which the first `zeroed` bytes
// (header, arrival counters, ready flags, key rows) must be zero when a call starts.
int decode_workspace_requirement(const quest_cache_t* cache, int top_k, size_t* total,
                                 size_t* zeroed);
// Record a failure for quest_last_error(); returns `code`.
int set_last_error(int code, const char* message);

cudaError_t launch_build_meta(const Params& p, cudaStream_t s);
cudaError_t launch_append(const Params& p, const __half* k_new, const __half* v_new,
                          cudaStream_t s, bool advance = true);
// seq_lens[b] += n for every sequence with room whose touched pages are mapped.
cudaError_t launch_advance_lengths(const Params& p, int n, cudaStream_t s);
cudaError_t launch_estimate(const Params& p, int G, bool per_head, cudaStream_t s);
cudaError_t launch_topk_union(const Params& p, int row_cap, cudaStream_t s);
cudaError_t launch_prefill(const Params& p, const __half* k, const __half* v, int n,
                           cudaStream_t s);
// Whether QUEST_PATH_AUTO takes the one-launch cluster kernel for this step (see quest.h).
cudaError_t cluster_preferred(int G, int P, int max_pages, int top_k, int nbg, bool* out);
cudaError_t launch_topk(const Params& p, cudaStream_t s);
cudaError_t launch_decode(const Params& p, int G, cudaStream_t s);
size_t cluster_smem_bytes(int G, int P, int max_pages, int cs, int top_k);
bool cluster_any_fits(int G, int P, int max_pages, int top_k);
cudaError_t launch_cluster(const Params& p, const LayerTable& lt, int G, int cs, int max_clusters,
                           cudaStream_t s);
constexpr int kMaxClusterSize = 16;
// The stream kernel (one persistent launch, every CTA on every pair): ring slots for this
// shape (0 if it does not fit), its shared memory, and its launch.
int stream_slots(int G, int P, int max_pages, int top_k, int batch, int hq);
size_t stream_smem_bytes(int G, int P, int max_pages, int top_k, int batch, int hq);
cudaError_t launch_stream(const Params& p, const LayerPtrs& lay, int G, int max_ctas,
                          cudaStream_t s);
constexpr int kStreamPiecePages = 8;  // kept pages per decode piece of the stream kernel
constexpr size_t kMaxSmem = 227 * 1024;  // dynamic shared memory of one CTA

}  // namespace quest
