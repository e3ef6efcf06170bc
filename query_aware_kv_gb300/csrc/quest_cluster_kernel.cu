// quest_cluster_kernel.cu - the whole Quest decode step in thread-block clusters: (optional)
// append, page scoring, top-K, split-K sparse decode and the log-sum-exp merge, with every
// cross-CTA step in distributed shared memory.
//
// "Guide to Quest", Best Practices step 3 asks for the bound estimation to be fused with
// the page gather.  On GB300 the unit for that is a cluster of CS CTAs per (sequence, kv
// head) pair; a cluster takes the pairs c, c + #clusters, ... one after the other:
//   1. every CTA scores a contiguous share of the pair's pages (boxes streamed by 1-D bulk
//      copies through an mbarrier ring by a producer warp), then stores the scores, as
//      order-preserving keys, and the share's key range into rank 0's shared memory and
//      arrives on rank 0's barrier;
//   2. rank 0 picks the top-K pages ("Guide to Quest", Solution step 3) and arrives on
//      every CTA's selection barrier;
//   3. each CTA's producer reads its share of the selection from rank 0, resolves the pages
//      through the block table and streams their K / V chunks; the consumer warps run
//      flash-decode over them (exact attention over the kept pages only: "Quest:
//      Query-Aware Sparsity for Efficient Long-Context LLM Inference", Summary) and store
//      the partial (max, sum, accumulator) into rank 0;
//   4. rank 0 merges the partials by log-sum-exp and writes the output.
// Rank 0's buffers alternate between consecutive pairs, so the other CTAs can start scoring
// the next pair while rank 0 still merges.  No global atomics, flags or work queue sit on
// the critical path; every wait is bounded.
#include <map>
#include <mutex>
#include <tuple>

#include "quest_device.cuh"

namespace quest {

namespace {

enum ClusterTraceEvent : int {
  kCtStart = 1, kCtExit = 2, kCtScoreDone = 20, kCtTopkBegin = 21, kCtTopkEnd = 22,
  kCtSelReady = 23, kCtDecodeDone = 24, kCtMergeBegin = 25, kCtMergeEnd = 26,
  kCtIssueFirst = 27, kCtIssueLast = 28, kCtProdSel = 29, kCtFirstStage = 30,
};

// Timeline record without atomics: CTA c owns records [c * kTraceSlots, (c + 1) *
// kTraceSlots) of the trace buffer; `slot` is the caller's running count: the consumer's
// thread 0 counts from 0, the producer's lane 0 from kProducerSlot0.
constexpr int kTraceSlots = 64;
constexpr int kProducerSlot0 = 40;
__device__ __forceinline__ void ctrace(const Params& p, int* slot, int ev, int item,
                                       int limit = kProducerSlot0) {
  if (p.trace == nullptr) return;
  if (*slot >= limit) return;
  const long long i = (long long)blockIdx.x * kTraceSlots + (*slot)++;
  if (i >= p.trace_capacity) return;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  p.trace[1 + 2 * i] = (unsigned long long)global_ns();
  p.trace[2 + 2 * i] = ((unsigned long long)smid << 48) |
                       ((unsigned long long)(blockIdx.x & 0xffff) << 32) |
                       ((unsigned long long)(ev & 0xff) << 24) | (unsigned)(item & 0xffffff);
}

// ---------------------------------------------------------------- cluster PTX
__device__ __forceinline__ uint32_t cta_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Address of `local` (this CTA's shared memory) in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t remote(const void* local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(local)), "r"(rank));
  return a;
}
__device__ __forceinline__ uint32_t ld_remote_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_remote_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_remote_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Arrive on an mbarrier of another CTA (release: this CTA's earlier writes, to shared or
// global memory, are visible to the waiter that acquires the phase).
__device__ __forceinline__ void arrive_remote(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ bool wait_cluster_bounded(const Params& p, uint64_t* bar, uint32_t parity, int site) {
  if (try_wait_cluster(bar, parity)) return true;
  const long long t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (try_wait_cluster(bar, parity)) return true;
    if (global_ns() - t0 > p.wait_limit_ns) {
      report(p, QUEST_ERR_TIMEOUT, -1, -1, site);
      return false;
    }
  }
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Start pulling [p, p + bytes) into L2 (no destination in the CTA).  p and bytes: multiples
// of 16.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_count(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

struct StageInfo {
  int n;       // decode: valid tokens of the staged page
  int first;   // scoring: first page of the stage
  int count;   // scoring: pages in the stage (0 if the copy was not issued)
  int pad;
};

template <int P>
struct CShape {
  static constexpr int kStage = 2 * P * kHeadDim * 2;            // one page's K + V chunks
  static constexpr int kBoxesPerStage = kStage / (2 * kHeadDim * 2);  // 16 or 32 boxes
};

// Shared memory.  Buffers indexed [2] alternate between consecutive pairs of a cluster.
struct CSmem {
  uint64_t *full, *empty;  // stage ring: [kStages] each
  uint64_t* bar_scores;    // rank 0 [2]: every CTA's keys of pair j are in place (count CS)
  uint64_t* bar_sel;       // every CTA [2]: the selection of pair j is in place (count 1)
  uint64_t* bar_part;      // rank 0 [2]: every CTA's partial of pair j is in place (count CS)
  uint64_t* prod_ok;       // every CTA [2]: its producer has passed the wait for selection j
  int* lens;
  int* scratch;            // [256]
  int* misc;               // [16]
  // streaming (every CTA)
  unsigned char* ring;
  StageInfo* stage;
  float* wsc;
  float* st;
  float* red;              // [warp][G][128] warp merge
  uint32_t* mykeys;        // [ceil(max_pages / CS)] this CTA's keys, before they go to rank 0
  // selection (rank 0)
  uint32_t* keys;          // [2][keys_stride(max_pages)] score keys, stored by every CTA
  uint32_t* ranges;        // [2][CS][2] key range of each CTA's share
  int* sel;                // [2][kcap] kept pages, ascending
  float* parts;            // [2][CS][G * (128 + 2)] partials M[G], L[G], A[G][128]
  int* hist;               // [kFastBins], at the start of the ring: rank 0's ring is idle
                           // while it selects
};

constexpr int kLenCache = 1024;

// Row stride of the selector's key buffers: a multiple of 4 keys, so that both rows start on
// 16 bytes (the selection reads keys four at a time).
__host__ __device__ inline int keys_stride(int max_pages) { return (max_pages + 3) & ~3; }

// Every CTA of a cluster streams; rank 0 also selects and merges.
__host__ __device__ inline int streamers_of(int cs) { return cs; }

// One layout for every CTA of the launch: the streaming region, then rank 0's selection
// region (allocated, unused, in the other ranks so that addresses agree across the cluster).
__host__ __device__ inline size_t cluster_smem_layout(int G, int P, int max_pages, int cs,
                                                      int top_k, CSmem* s, unsigned char* base) {
  const int S = streamers_of(cs);
  const int kcap = top_k < max_pages ? top_k : max_pages;
  const size_t part_floats = (size_t)G * (kHeadDim + 2);
  size_t o = 0;
  const size_t full = o;     o += kStages * 8;
  const size_t empty = o;    o += kStages * 8;
  const size_t bars = o;     o += 8 * 8;
  const size_t lens = o;     o += kLenCache * 4;
  const size_t scratch = o;  o += 256 * 4;
  const size_t misc = o;     o = align_up(o + 16 * 4, 128);
  // streaming region
  size_t a = o;
  const size_t ring = a;     a = align_up(a + (size_t)kStages * 2 * P * kHeadDim * 2, 16);
  static_assert((size_t)kStages * 2 * 16 * kHeadDim * 2 >= (size_t)kFastBins * 4,
                "the ring holds the selection's histogram");
  const size_t sdesc = a;    a = align_up(a + kStages * sizeof(StageInfo), 16);
  const size_t wsc = a;      a = align_up(a + (size_t)kConsumerWarps * G * P * 4, 16);
  const size_t st = a;       a = align_up(a + (size_t)kConsumerWarps * G * 3 * 4, 16);
  const size_t red = a;      a = align_up(a + (size_t)kConsumerWarps * G * kHeadDim * 4, 16);
  const size_t mykeys = a;   a = align_up(a + (size_t)(cs > 1 ? (max_pages + S - 1) / S : 0) * 4, 128);
  // selection region
  size_t b = a;
  const size_t keys = b;     b = align_up(b + (size_t)2 * keys_stride(max_pages) * 4, 16);
  const size_t ranges = b;   b = align_up(b + (size_t)2 * S * 2 * 4, 16);
  const size_t sel = b;      b = align_up(b + (size_t)2 * kcap * 4, 16);
  const size_t parts = b;    b = align_up(b + (size_t)2 * S * part_floats * 4, 16);
  const size_t total = b;
  if (s) {
    s->full = reinterpret_cast<uint64_t*>(base + full);
    s->empty = reinterpret_cast<uint64_t*>(base + empty);
    s->bar_scores = reinterpret_cast<uint64_t*>(base + bars);
    s->bar_sel = s->bar_scores + 2;
    s->bar_part = s->bar_scores + 4;
    s->prod_ok = s->bar_scores + 6;
    s->lens = reinterpret_cast<int*>(base + lens);
    s->scratch = reinterpret_cast<int*>(base + scratch);
    s->misc = reinterpret_cast<int*>(base + misc);
    s->ring = base + ring;
    s->stage = reinterpret_cast<StageInfo*>(base + sdesc);
    s->wsc = reinterpret_cast<float*>(base + wsc);
    s->st = reinterpret_cast<float*>(base + st);
    s->red = reinterpret_cast<float*>(base + red);
    s->mykeys = reinterpret_cast<uint32_t*>(base + mykeys);
    s->keys = reinterpret_cast<uint32_t*>(base + keys);
    s->ranges = reinterpret_cast<uint32_t*>(base + ranges);
    s->sel = reinterpret_cast<int*>(base + sel);
    s->parts = reinterpret_cast<float*>(base + parts);
    s->hist = reinterpret_cast<int*>(base + ring);
  }
  return total;
}

// The cluster's j-th pair and its roles.
struct Role {
  int rank, cs, S, si;  // S: CTAs that stream (all of them), si: this CTA's index among them
  bool selector;
  int cid, ncl, nbg, npairs;
};

__device__ __forceinline__ Role make_role(const Params& p, int cs, int n_layers) {
  Role r;
  r.rank = (int)cta_rank();
  r.cs = cs;
  r.S = streamers_of(cs);
  r.selector = r.rank == 0;
  r.si = r.rank;
  r.cid = (int)cluster_index();
  r.ncl = (int)cluster_count();
  r.nbg = n_layers * p.B * p.Hkv;
  r.npairs = r.cid < r.nbg ? (r.nbg - 1 - r.cid) / r.ncl + 1 : 0;
  return r;
}

struct Pair {
  const LayerPtrs* lay;    // this pair's layer: pools, boxes, q, new token, output
  int b, g, L, N, count;
  int p_lo, p_hi;          // this streamer's scoring share
  int q_lo, q_hi;          // this streamer's decode share (ranks of the selection)
  int buf;                 // alternating buffer of this pair
  int append_page;         // page receiving the appended token, or -1
};

__device__ __forceinline__ Pair pair_geometry(const Params& p, const LayerTable& lt,
                                              const CSmem& s, const Role& r, int j) {
  Pair q;
  const int pair = r.cid + j * r.ncl;  // layer-major over (layer, sequence, kv head)
  const int nbg1 = p.B * p.Hkv;
  const int layer = pair / nbg1, bg = pair - layer * nbg1;
  q.lay = &lt.l[layer];
  q.b = bg / p.Hkv;
  q.g = bg % p.Hkv;
  q.buf = j & 1;
  const int L0 = q.b < kLenCache ? s.lens[q.b] : p.seq_lens[q.b];
  const long long cap = (long long)p.max_pages * p.P;
  int L = L0;
  if (L0 < 0 || (long long)L0 > cap) {
    if (r.rank == 0 && q.g == 0 && threadIdx.x == 0) report(p, QUEST_ERR_BAD_LENGTH, q.b, -1, kSiteScore);
    L = 0;
  }
  q.append_page = -1;
  if (p.k_new != nullptr && L0 >= 0 && (long long)L0 + 1 <= cap) {
    L = L0 + 1;
    q.append_page = L0 / p.P;
  }
  q.L = L;
  q.N = (L + p.P - 1) / p.P;
  q.count = min(p.top_k, q.N);
  const int si = r.si;
  const int share = (q.N + r.S - 1) / r.S;
  q.p_lo = min(q.N, si * share);
  q.p_hi = min(q.N, q.p_lo + share);
  q.q_lo = (int)((long long)q.count * si / r.S);
  q.q_hi = (int)((long long)q.count * (si + 1) / r.S);
  return q;
}

// ---------------------------------------------------------------- producer warp
template <int G, int P>
__device__ void c_produce_score(const Params& p, const CSmem& s, const Pair& q, uint32_t& stage_seq,
                                int* pslot) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  const int lane = threadIdx.x & 31;
  // contiguous boxes, one bulk copy per stage
  const int n_live = q.p_hi - q.p_lo;
  if (lane == 0) {
    const __half* box0 = q.lay->meta + box_offset(p, q.b, q.g, q.p_lo);
    for (int u0 = 0; u0 < n_live; u0 += kSP) {
      const uint32_t kk = stage_seq + (uint32_t)(u0 / kSP);
      const int st = (int)(kk % kStages);
      const bool free_ok =
          mbar_wait_bounded(p, &s.empty[st], ((kk / kStages) & 1u) ^ 1u, kSiteWaitSlot);
      const int n = min(kSP, n_live - u0);
      s.stage[st].first = q.p_lo + u0;
      s.stage[st].count = free_ok ? n : 0;
      s.stage[st].n = 0;
      if (free_ok) {
        mbar_arrive_expect_tx(&s.full[st], (uint32_t)n * 2 * kHeadDim * 2);
        bulk_g2s(s.ring + (size_t)st * kStage, box0 + (size_t)u0 * 2 * kHeadDim,
                 (uint32_t)n * 2 * kHeadDim * 2, &s.full[st]);
      } else {
        mbar_arrive(&s.full[st]);
      }
      if (u0 == 0) ctrace(p, pslot, kCtIssueFirst, q.b * p.Hkv + q.g, kTraceSlots - 1);
    }
    if (n_live > 0) ctrace(p, pslot, kCtIssueLast, q.b * p.Hkv + q.g, kTraceSlots - 1);
  }
  stage_seq += (uint32_t)((n_live + kSP - 1) / kSP);
  __syncwarp();
}

// The decode share of pair j, once the selector has published the selection.  The wait is
// made for every pair, even with nothing to decode: a phase parity names the right phase
// only while the waiter is at most one phase behind.
template <int G, int P>
__device__ void c_produce_decode(const Params& p, const CSmem& s, const Pair& q, int j,
                                 uint32_t& stage_seq, int* pslot) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr uint32_t kChunk = P * kHeadDim * 2;
  const int lane = threadIdx.x & 31;
  const int n_dec = q.q_hi - q.q_lo;
  bool ok = true;
  if (lane == 0 && q.N > 0) {
    // while the selection is being made: the pair's block-table row into L2, so that the
    // page lookups after it hit L2 (whole 16-byte units inside the row only)
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(p.block_table + (size_t)q.b * p.max_pages);
    const uintptr_t a1 = reinterpret_cast<uintptr_t>(p.block_table + (size_t)q.b * p.max_pages + q.N);
    const uintptr_t lo16 = (a0 + 15) & ~(uintptr_t)15, hi16 = a1 & ~(uintptr_t)15;
    if (hi16 > lo16) prefetch_l2(reinterpret_cast<const void*>(lo16), (uint32_t)(hi16 - lo16));
  }
  if (lane == 0) {
    ok = wait_cluster_bounded(p, &s.bar_sel[q.buf], (uint32_t)(j >> 1) & 1u, kSiteWaitSelection);
    mbar_arrive(&s.prod_ok[q.buf]);
    ctrace(p, pslot, kCtProdSel, q.b * p.Hkv + q.g, kTraceSlots - 1);
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (n_dec <= 0) return;
  if (p.k_new != nullptr) fence_proxy_async_global();  // appended rows: generic writes
  const int kcap = min(p.top_k, p.max_pages);
  const uint32_t sel0 = remote(s.sel + q.buf * kcap, 0);
  const size_t chunk_elems = (size_t)P * kHeadDim;
  for (int c = 0; c < n_dec; c += 32) {
    const int rr = c + lane;
    int nv = 0, lp = -1;
    const __half* ksrc = nullptr;
    const __half* vsrc = nullptr;
    if (ok && rr < n_dec) {
      lp = (int)ld_remote_u32(sel0 + 4u * (uint32_t)(q.q_lo + rr));
      if (lp < 0 || lp >= q.N) {
        report(p, QUEST_ERR_BAD_SELECTION, q.b, lp, kSiteSelection);
      } else {
        const int phys = p.block_table[(size_t)q.b * p.max_pages + lp];
        if (phys < 0 || phys >= p.num_phys) {
          report(p, QUEST_ERR_BAD_PAGE, q.b, lp, kSiteDecode);
        } else {
          nv = min(P, q.L - lp * P);
          const size_t off = ((size_t)phys * p.Hkv + q.g) * chunk_elems;
          ksrc = q.lay->k_pool + off;
          vsrc = q.lay->v_pool + off;
        }
      }
    }
    const int cnt = min(32, n_dec - c);
    for (int jj = 0; jj < cnt; ++jj) {
      if (lane == jj) {
        const uint32_t kk = stage_seq + (uint32_t)jj;
        const int st = (int)(kk % kStages);
        const bool free_ok =
            mbar_wait_bounded(p, &s.empty[st], ((kk / kStages) & 1u) ^ 1u, kSiteWaitSlot);
        s.stage[st].n = free_ok ? nv : 0;
        s.stage[st].first = lp;
        if (free_ok && nv > 0) {
          unsigned char* dst = s.ring + (size_t)st * kStage;
          mbar_arrive_expect_tx(&s.full[st], 2 * kChunk);
          bulk_g2s(dst, ksrc, kChunk, &s.full[st]);
          bulk_g2s(dst + kChunk, vsrc, kChunk, &s.full[st]);
        } else {
          mbar_arrive(&s.full[st]);
        }
      }
      __syncwarp();
    }
    stage_seq += (uint32_t)cnt;
  }
  if (lane == 0) ctrace(p, pslot, kCtIssueLast, q.b * p.Hkv + q.g, kTraceSlots - 1);
}

// Work order, pair after pair: score, then on rank 0 select, then decode, then on rank 0
// merge.  Every step sits behind one call site, so the kernel's code stays small (its first
// execution in a launch waits for instruction fetches from memory).
enum Task : int { kTaskScore = 0, kTaskDecode = 1, kTaskSelect = 2, kTaskMerge = 3 };

__device__ __forceinline__ int task_count(const Role& r, bool producer) {
  return r.npairs * ((r.selector && !producer) ? 4 : 2);
}

__device__ __forceinline__ int task_at(const Role& r, bool producer, int t, int* j) {
  if (r.selector && !producer) {
    *j = t >> 2;
    const int k = t & 3;
    return k == 0 ? kTaskScore : k == 1 ? kTaskSelect : k == 2 ? kTaskDecode : kTaskMerge;
  }
  *j = t >> 1;
  return (t & 1) ? kTaskDecode : kTaskScore;
}

template <int G, int P>
__device__ void c_produce(const Params& p, const LayerTable& lt, const CSmem& s, const Role& r) {
  uint32_t stage_seq = 0;
  int pslot = kProducerSlot0;
  const int n = task_count(r, true);
  for (int t = 0; t < n; ++t) {
    int j;
    const int kind = task_at(r, true, t, &j);
    const Pair q = pair_geometry(p, lt, s, r, j);
    if (kind == kTaskScore)
      c_produce_score<G, P>(p, s, q, stage_seq, &pslot);
    else
      c_produce_decode<G, P>(p, s, q, j, stage_seq, &pslot);
  }
}

// ---------------------------------------------------------------- consumer warps
// Score this streamer's share of pair q; the keys and the share's key range go straight
// into the selector's shared memory.  Folds the appended token into its page's box and
// writes its K / V row.
template <int G, int P>
__device__ void c_score_share(const Params& p, const CSmem& s, const Role& r, const Pair& q,
                              uint32_t stage_base, int* tslot) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  const int tid = threadIdx.x, lane = tid & 31;
  const int hw = tid >> 4, c = tid & 15;
  const int n_live = q.p_hi - q.p_lo;
  const int S = r.S;
  const uint32_t range0 = remote(s.ranges + (q.buf * S + r.si) * 2, 0);
  if (n_live <= 0) {
    if (tid == 0) {
      st_remote_u32(range0, 0xffffffffu);
      st_remote_u32(range0 + 4u, 0u);
    }
    return;
  }
  // keys land in this CTA's shared memory (the selector's buffer itself in a cluster of one)
  // and go to the selector in one pass at the end: a store to another CTA inside the loop
  // would hold up every stage's release of its ring slot
  uint32_t* kout = r.selector ? s.keys + (size_t)q.buf * keys_stride(p.max_pages) + q.p_lo : s.mykeys;
  uint32_t lo = 0xffffffffu, hi = 0u;
  QueryFrag<G> f;
  load_query_frag<G>(q.lay->q, p.Hq, q.b, q.g, c, f);
  uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
  const bool mine_append = q.append_page >= q.p_lo && q.append_page < q.p_hi;
  const int slot_a = (q.L - 1) % P;
  int append_phys = -1;
  if (mine_append) {
    const size_t o = ((size_t)q.b * p.Hkv + q.g) * kHeadDim + 8 * c;
    knew = *reinterpret_cast<const uint4*>(q.lay->k_new + o);
    vnew = *reinterpret_cast<const uint4*>(q.lay->v_new + o);
    const int phys = p.block_table[(size_t)q.b * p.max_pages + q.append_page];
    append_phys = (phys >= 0 && phys < p.num_phys) ? phys : -1;
  }
  const int n_units = (n_live + kSP - 1) / kSP;
  for (int u = 0; u < n_units; ++u) {
    const uint32_t k = stage_base + (uint32_t)u;
    const int st = (int)(k % kStages);
    mbar_wait_bounded(p, &s.full[st], (k / kStages) & 1u, kSiteWaitStage);
    if (u == 0 && tid == 0) ctrace(p, tslot, kCtFirstStage, q.b * p.Hkv + q.g);
    const StageInfo sd = s.stage[st];
#pragma unroll
    for (int rep = 0; rep < kSP / 16; ++rep) {
      const int j = hw + 16 * rep;
      if (j >= kSP) break;
      const int page = sd.first + j;
      const bool have = j < sd.count;
      const unsigned char* rec = s.ring + (size_t)st * kStage + (size_t)j * 2 * kHeadDim * 2;
      uint4 mn = make_uint4(0, 0, 0, 0), mx = make_uint4(0, 0, 0, 0);
      if (have) {
        mn = *reinterpret_cast<const uint4*>(rec + 16 * c);
        mx = *reinterpret_cast<const uint4*>(rec + 2 * kHeadDim + 16 * c);
      }
      if (have && page == q.append_page) {
        if (append_phys >= 0) {
          if (slot_a == 0) {
            mn = knew;
            mx = knew;
          } else {
            const uint32_t a[4] = {mn.x, mn.y, mn.z, mn.w};
            const uint32_t z[4] = {mx.x, mx.y, mx.z, mx.w};
            const uint32_t n[4] = {knew.x, knew.y, knew.z, knew.w};
            uint32_t ra[4], rz[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const __half2 hn = *reinterpret_cast<const __half2*>(&n[w]);
              const __half2 l2 = __hmin2(*reinterpret_cast<const __half2*>(&a[w]), hn);
              const __half2 h2 = __hmax2(*reinterpret_cast<const __half2*>(&z[w]), hn);
              ra[w] = *reinterpret_cast<const uint32_t*>(&l2);
              rz[w] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            mn = make_uint4(ra[0], ra[1], ra[2], ra[3]);
            mx = make_uint4(rz[0], rz[1], rz[2], rz[3]);
          }
          __half* box = q.lay->meta + box_offset(p, q.b, q.g, page);
          *reinterpret_cast<uint4*>(box + 8 * c) = mn;
          *reinterpret_cast<uint4*>(box + kHeadDim + 8 * c) = mx;
          const size_t kv = (((size_t)append_phys * p.Hkv + q.g) * P + slot_a) * kHeadDim + 8 * c;
          *reinterpret_cast<uint4*>(q.lay->k_pool + kv) = knew;
          *reinterpret_cast<uint4*>(q.lay->v_pool + kv) = vnew;
        } else if (c == 0) {
          report(p, QUEST_ERR_BAD_PAGE, q.b, page, kSiteAppend);
        }
      }
      float best = -CUDART_INF_F;
#pragma unroll
      for (int jh = 0; jh < G; ++jh) {
        float sc = corner_dot<G>(f, jh, mn, mx);
        sc += __shfl_xor_sync(0xffffffffu, sc, 8);
        sc += __shfl_xor_sync(0xffffffffu, sc, 4);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        best = fmaxf(best, sc);
      }
      if (c == 0 && page < q.p_hi) {
        // pages of the sink / local window of a long sequence get the largest key
        const bool forced =
            q.N > q.count && (page < p.sink_pages || page >= q.N - p.local_pages);
        const uint32_t key = forced ? 0xffffffffu : score_key(have ? best : -CUDART_INF_F);
        kout[page - q.p_lo] = key;
        lo = min(lo, key);
        hi = max(hi, key);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
  }
  if (mine_append) fence_proxy_async_global();  // appended rows, before the scores are released
  // this share's key range, to the selector
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    s.scratch[tid >> 5] = (int)lo;
    s.scratch[8 + (tid >> 5)] = (int)hi;
  }
  bsync<kConsumerThreads, true>();
  if (tid == 0) {
    uint32_t l = 0xffffffffu, h = 0u;
    for (int w = 0; w < kConsumerWarps; ++w) {
      l = min(l, (uint32_t)s.scratch[w]);
      h = max(h, (uint32_t)s.scratch[8 + w]);
    }
    st_remote_u32(range0, l);
    st_remote_u32(range0 + 4u, h);
  }
  if (!r.selector) {
    const uint32_t keys0 = remote(s.keys + (size_t)q.buf * keys_stride(p.max_pages) + q.p_lo, 0);
    for (int i = tid; i < n_live; i += kConsumerThreads) st_remote_u32(keys0 + 4u * (uint32_t)i, s.mykeys[i]);
  }
}

// Rank 0: the top-K of pair q's N keys (in s.keys[buf]) into s.sel[buf], ascending.
__device__ void c_select(const Params& p, const CSmem& s, const Role& r, const Pair& q) {
  const int tid = threadIdx.x;
  const int kcap = min(p.top_k, p.max_pages);
  int* sel = s.sel + q.buf * kcap;
  int* cnt_slot = s.misc + 8;
  if (q.N <= q.count) {
    for (int i = tid; i < q.count; i += kConsumerThreads) sel[i] = i;
    if (tid == 0) *cnt_slot = q.N;
    return;
  }
  const uint32_t* rg = s.ranges + q.buf * r.S * 2;
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = 0; i < r.S; ++i) {
    lo = min(lo, rg[2 * i]);
    hi = max(hi, rg[2 * i + 1]);
  }
  // the histogram lives in the ring, which bulk copies wrote last: clear it first
  for (int i = tid; i < kFastBins / 4; i += kConsumerThreads)
    reinterpret_cast<int4*>(s.hist)[i] = make_int4(0, 0, 0, 0);
  bsync<kConsumerThreads, true>();
  topk_fast<kConsumerThreads, true>(s.keys + (size_t)q.buf * keys_stride(p.max_pages), q.N,
                                    q.count, lo, hi, sel, s.hist, s.scratch);
  if (tid == 0) *cnt_slot = q.count;
  // the ring goes back to bulk copies (async proxy) after these generic writes
  fence_proxy_async_smem();
}

// Selector: the selection, for the caller, if asked for (after it was released).
__device__ void c_publish_selection(const Params& p, const CSmem& s, const Pair& q) {
  if (p.sel_idx == nullptr) return;
  const int tid = threadIdx.x;
  const int kcap = min(p.top_k, p.max_pages);
  const int* sel = s.sel + q.buf * kcap;
  const int bg = q.b * p.Hkv + q.g;
  int* row = p.sel_idx + (size_t)bg * p.top_k;
  for (int i = tid; i < p.top_k; i += kConsumerThreads) row[i] = i < q.count ? sel[i] : -1;
  if (tid == 0 && p.sel_count != nullptr) p.sel_count[bg] = q.count;
}

// Flash-decode over this streamer's share of the selection; the partial goes to the
// selector's slot parts[buf][si].
template <int G, int P>
__device__ void c_decode_share(const Params& p, const CSmem& s, const Role& r, const Pair& q,
                               uint32_t stage_base) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr int PF = G * (kHeadDim + 2);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = q.q_hi - q.q_lo;
  const uint32_t slot = remote(s.parts + (size_t)(q.buf * r.S + r.si) * PF, 0);
  if (n <= 0) {
    if (tid < G) {
      st_remote_f32(slot + 4u * (uint32_t)tid, -CUDART_INF_F);
      st_remote_f32(slot + 4u * (uint32_t)(G + tid), 0.f);
    }
    return;
  }
  float qf[G][4];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint2 raw =
        *reinterpret_cast<const uint2*>(q.lay->q + ((size_t)q.b * p.Hq + q.g * G + j) * kHeadDim + 4 * lane);
    const float2 a = h2f(raw.x), c = h2f(raw.y);
    qf[j][0] = a.x * p.qscale;
    qf[j][1] = a.y * p.qscale;
    qf[j][2] = c.x * p.qscale;
    qf[j][3] = c.y * p.qscale;
  }
  float acc[G][4];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;
  float* sc = s.wsc + warp * G * P;
  float* st = s.st + warp * G * 3;
  if (lane < G) {
    st[lane * 3 + 0] = -CUDART_INF_F;
    st[lane * 3 + 1] = 0.f;
    st[lane * 3 + 2] = 1.f;
  }
  __syncwarp();
  for (int rr = warp; rr < n; rr += kConsumerWarps) {
    const uint32_t k = stage_base + (uint32_t)rr;
    const int stg = (int)(k % kStages);
    const bool ok = mbar_wait_bounded(p, &s.full[stg], (k / kStages) & 1u, kSiteWaitStage);
    const int nv = ok ? s.stage[stg].n : 0;
    if (nv > 0) {
      const __half* Ks = reinterpret_cast<const __half*>(s.ring + (size_t)stg * kStage);
      page_update<G, P>(qf, acc, Ks, Ks + P * kHeadDim, nv, sc, st, lane);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive_count(&s.empty[stg], kConsumerWarps);
  }
  // merge the 8 warps into this streamer's partial
#pragma unroll
  for (int j = 0; j < G; ++j)
    *reinterpret_cast<float4*>(s.red + ((size_t)warp * G + j) * kHeadDim + 4 * lane) =
        make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
  bsync<kConsumerThreads, true>();
  for (int o = tid; o < G * kHeadDim; o += kConsumerThreads) {
    const int j = o / kHeadDim, i = o % kHeadDim;
    float Mx = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) Mx = fmaxf(Mx, s.st[(w * G + j) * 3]);
    float a = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = s.st[(w * G + j) * 3];
      if (mw != -CUDART_INF_F) {
        const float f = exp2f(mw - Mx);
        a = fmaf(s.red[((size_t)w * G + j) * kHeadDim + i], f, a);
        l = fmaf(s.st[(w * G + j) * 3 + 1], f, l);
      }
    }
    st_remote_f32(slot + 4u * (uint32_t)(2 * G + j * kHeadDim + i), a);
    if (i == 0) {
      st_remote_f32(slot + 4u * (uint32_t)j, Mx);
      st_remote_f32(slot + 4u * (uint32_t)(G + j), l);
    }
  }
}

// Selector: merge the streamers' partials of pair q into out / lse.
template <int G>
__device__ void c_merge(const Params& p, const CSmem& s, const Role& r, const Pair& q) {
  constexpr int PF = G * (kHeadDim + 2);
  const int tid = threadIdx.x;
  const float* parts = s.parts + (size_t)q.buf * r.S * PF;
  for (int o = tid; o < G * kHeadDim; o += kConsumerThreads) {
    const int j = o / kHeadDim, i = o % kHeadDim;
    float Mx = -CUDART_INF_F;
    for (int u = 0; u < r.S; ++u) Mx = fmaxf(Mx, parts[u * PF + j]);
    float acc = 0.f, ls = 0.f;
    for (int u = 0; u < r.S; ++u) {
      const float m = parts[u * PF + j];
      if (m != -CUDART_INF_F) {
        const float f = exp2f(m - Mx);
        acc = fmaf(parts[u * PF + 2 * G + j * kHeadDim + i], f, acc);
        ls = fmaf(parts[u * PF + G + j], f, ls);
      }
    }
    const int h = q.g * G + j;
    q.lay->out[((size_t)q.b * p.Hq + h) * kHeadDim + i] = __float2half_rn(ls > 0.f ? acc / ls : 0.f);
    if (i == 0 && q.lay->lse)
      q.lay->lse[(size_t)q.b * p.Hq + h] =
          ls > 0.f ? (Mx + log2f(ls)) * 0.69314718055994531f : -CUDART_INF_F;
  }
}

// Selector of pair j: wait for the keys, select, release every streamer, publish.
__device__ void c_selector_step(const Params& p, const CSmem& s, const Role& r, const Pair& q,
                                int j, int* tslot) {
  const int tid = threadIdx.x;
  const int bg = q.b * p.Hkv + q.g;
  if (tid == 0) wait_cluster_bounded(p, &s.bar_scores[q.buf], (uint32_t)(j >> 1) & 1u, kSiteWaitSelection);
  bsync<kConsumerThreads, true>();
  if (tid == 0) ctrace(p, tslot, kCtTopkBegin, bg);
  c_select(p, s, r, q);
  bsync<kConsumerThreads, true>();
  if (tid == 0) ctrace(p, tslot, kCtTopkEnd, bg);
  if (tid < r.S && !(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION))
    arrive_remote(remote(&s.bar_sel[q.buf], (uint32_t)tid));
  c_publish_selection(p, s, q);
}

__device__ void c_selector_merge_wait(const Params& p, const CSmem& s, const Pair& q, int j,
                                      int* tslot) {
  const int tid = threadIdx.x;
  if (tid == 0) wait_cluster_bounded(p, &s.bar_part[q.buf], (uint32_t)(j >> 1) & 1u, kSiteWaitSlot);
  bsync<kConsumerThreads, true>();
  if (tid == 0) ctrace(p, tslot, kCtMergeBegin, q.b * p.Hkv + q.g);
}

// Scores of pair j.  Before they are released, this CTA's producer must have passed its
// wait for selection j - 2: selection j cannot complete before these scores arrive, so the
// producer is never two phases behind on a selection barrier (a parity wait would then
// miss its phase), even when this CTA's shares are empty and its consumers run ahead.
template <int G, int P>
__device__ void c_stream_score(const Params& p, const CSmem& s, const Role& r, const Pair& q,
                               int j, uint32_t& stage_seq, int* tslot) {
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  c_score_share<G, P>(p, s, r, q, stage_seq, tslot);
  stage_seq += (uint32_t)((q.p_hi - q.p_lo + kSP - 1) / kSP);
  bsync<kConsumerThreads, true>();
  if (threadIdx.x == 0) {
    if (j >= 2) mbar_wait_bounded(p, &s.prod_ok[q.buf], (uint32_t)((j - 2) >> 1) & 1u, kSiteWaitSlot);
    ctrace(p, tslot, kCtScoreDone, q.b * p.Hkv + q.g);
    arrive_remote(remote(&s.bar_scores[q.buf], 0));
  }
}

template <int G, int P>
__device__ void c_stream_decode(const Params& p, const CSmem& s, const Role& r, const Pair& q,
                                int j, uint32_t& stage_seq, int* tslot) {
  const int tid = threadIdx.x;
  const int bg = q.b * p.Hkv + q.g;
  if (!r.selector) {
    // the selection of this pair is out: the selector is done with its keys, and with
    // every earlier pair's partials
    if (tid == 0) wait_cluster_bounded(p, &s.bar_sel[q.buf], (uint32_t)(j >> 1) & 1u, kSiteWaitSelection);
    bsync<kConsumerThreads, true>();
  }
  if (tid == 0) ctrace(p, tslot, kCtSelReady, bg);
  c_decode_share<G, P>(p, s, r, q, stage_seq);
  stage_seq += (uint32_t)max(0, q.q_hi - q.q_lo);
  bsync<kConsumerThreads, true>();
  if (tid == 0) {
    ctrace(p, tslot, kCtDecodeDone, bg);
    arrive_remote(remote(&s.bar_part[q.buf], 0));
  }
}

template <int G, int P>
__device__ void c_consume(const Params& p, const LayerTable& lt, const CSmem& s, const Role& r) {
  uint32_t stage_seq = 0;
  int tslot = 1;  // slot 0: the CTA's start record
  const int n = task_count(r, false);
  for (int t = 0; t < n; ++t) {
    int j;
    const int kind = task_at(r, false, t, &j);
    const Pair q = pair_geometry(p, lt, s, r, j);
    if (kind == kTaskScore) {
      c_stream_score<G, P>(p, s, r, q, j, stage_seq, &tslot);
    } else if (kind == kTaskDecode) {
      c_stream_decode<G, P>(p, s, r, q, j, stage_seq, &tslot);
    } else if (kind == kTaskSelect) {
      c_selector_step(p, s, r, q, j, &tslot);
    } else {
      c_selector_merge_wait(p, s, q, j, &tslot);
      c_merge<G>(p, s, r, q);
      bsync<kConsumerThreads, true>();
      if (threadIdx.x == 0) ctrace(p, &tslot, kCtMergeEnd, q.b * p.Hkv + q.g);
    }
  }
}

}  // namespace

template <int G, int P>
__global__ void __launch_bounds__(kDecodeThreads, (P == 16 && G <= 4) ? 2 : 1)
    cluster_kernel(Params p, int cs, const __grid_constant__ LayerTable lt) {
  extern __shared__ __align__(128) unsigned char smem[];
  CSmem s;
  cluster_smem_layout(G, P, p.max_pages, cs, p.top_k, &s, smem);
  const Role r = make_role(p, cs, lt.n);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.bar_scores[i], (uint32_t)r.S);
      mbar_init(&s.bar_sel[i], 1);
      mbar_init(&s.bar_part[i], (uint32_t)r.S);
      mbar_init(&s.prod_ok[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive
  pdl_wait();
  for (int b = threadIdx.x; b < min(p.B, kLenCache); b += blockDim.x) s.lens[b] = p.seq_lens[b];
  __syncthreads();
  if (threadIdx.x == 0) {
    int slot0 = 0;
    ctrace(p, &slot0, kCtStart, r.rank);
  }
  if (threadIdx.x >= kConsumerThreads) {
    c_produce<G, P>(p, lt, s, r);
  } else {
    c_consume<G, P>(p, lt, s, r);
  }
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another may still read its shared memory
  if (threadIdx.x == 0) {
    int slot_last = kTraceSlots - 1;
    ctrace(p, &slot_last, kCtExit, r.rank, kTraceSlots);
  }
  // With an appended token, the last CTA to leave advances the lengths (pairs past the
  // shared-memory cache read seq_lens as they go), one sequence per lane of its warp 0.
  if (p.k_new != nullptr && threadIdx.x < 32) {
    unsigned last = 0;
    if (threadIdx.x == 0) {
      __threadfence();
      last = atomicAdd(p.exited, 1u) == gridDim.x - 1u;
    }
    if (__shfl_sync(0xffffffffu, last, 0)) {
      for (int b = threadIdx.x; b < p.B; b += 32) {
        const int L0 = p.seq_lens[b];
        if (L0 < 0 || (long long)L0 + 1 > (long long)p.max_pages * p.P) {
          report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);
          continue;
        }
        const int phys = p.block_table[(size_t)b * p.max_pages + L0 / p.P];
        if (phys >= 0 && phys < p.num_phys) p.seq_lens[b] = L0 + 1;
      }
      if (threadIdx.x == 0) *p.exited = 0u;
    }
  }
}


template <int G, int P>
static const void* cluster_fn() { return (const void*)cluster_kernel<G, P>; }

static const void* pick_cluster(int G, int P) {
  if (P == 16) {
    switch (G) {
      case 1: return cluster_fn<1, 16>();
      case 2: return cluster_fn<2, 16>();
      case 4: return cluster_fn<4, 16>();
      default: return cluster_fn<8, 16>();
    }
  }
  switch (G) {
    case 1: return cluster_fn<1, 32>();
    case 2: return cluster_fn<2, 32>();
    case 4: return cluster_fn<4, 32>();
    default: return cluster_fn<8, 32>();
  }
}

size_t cluster_smem_bytes(int G, int P, int max_pages, int cs, int top_k) {
  return cluster_smem_layout(G, P, max_pages, cs, top_k, nullptr, nullptr);
}

namespace {

constexpr int kAutoClusterMax = 8;

cudaLaunchConfig_t cluster_config(int cs, int ncl, size_t smem, cudaStream_t s,
                                  cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(cs * ncl));
  cfg.blockDim = dim3(kDecodeThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// How many clusters of `cs` CTAs can be resident at once (cached per device and shape).
cudaError_t resident_clusters(int G, int P, int max_pages, int top_k, int cs, int* out) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int, int, int, int>, int> memo;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const auto key = std::make_tuple(dev, G, P, max_pages, top_k, cs);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = memo.find(key);
    if (it != memo.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  const void* fn = pick_cluster(G, P);
  const size_t smem = cluster_smem_bytes(G, P, max_pages, cs, top_k);
  if ((e = ensure_smem(fn, smem)) != cudaSuccess) return e;
  if (cs > 8 && (e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                          1)) != cudaSuccess)
    return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(cs, 1, smem, nullptr, attr);
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  memo[key] = n;
  *out = n;
  return cudaSuccess;
}

// Automatic cluster size: the largest portable size (up to 8) at which the clusters of all
// pairs are resident together, so every pair runs at once over as many SMs as possible; with
// more pairs than that, one CTA per pair.  (Measured on the 32-pair LongChat layer: clusters
// of 8 beat 4, 9-16 and 1.)
cudaError_t choose_cluster_size(int G, int P, int max_pages, int top_k, int nbg, int* cs_out) {
  cudaError_t e;
  for (int cs = kAutoClusterMax; cs > 1; --cs) {
    if (cluster_smem_bytes(G, P, max_pages, cs, top_k) > kMaxSmem) continue;
    int n = 0;
    if ((e = resident_clusters(G, P, max_pages, top_k, cs, &n)) != cudaSuccess) return e;
    if (n >= nbg) {
      *cs_out = cs;
      return cudaSuccess;
    }
  }
  *cs_out = 1;
  return cluster_smem_bytes(G, P, max_pages, 1, top_k) <= kMaxSmem ? cudaSuccess
                                                                     : cudaErrorInvalidConfiguration;
}

}  // namespace

constexpr int kFusedMaxPages = 1024;

cudaError_t cluster_preferred(int G, int P, int max_pages, int top_k, int nbg, bool* out) {
  int cs = 0;
  cudaError_t e = choose_cluster_size(G, P, max_pages, top_k, nbg, &cs);
  if (e != cudaSuccess) return e;
  const void* fn = pick_cluster(G, P);
  const size_t smem = cluster_smem_bytes(G, P, max_pages, cs, top_k);
  if ((e = ensure_smem(fn, smem)) != cudaSuccess) return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kDecodeThreads, smem)) !=
      cudaSuccess)
    return e;
  // rows of a thousand pages or more: the chain's whole-GPU scoring and decode kernels win
  // over the pair's cluster (measured: equal near 16K tokens per sequence at page 16)
  *out = per_sm >= 2 && cs >= 2 && max_pages < kFusedMaxPages;
  return cudaSuccess;
}

bool cluster_any_fits(int G, int P, int max_pages, int top_k) {
  for (int cs = 1; cs <= kMaxClusterSize; ++cs)
    if (cluster_smem_bytes(G, P, max_pages, cs, top_k) <= kMaxSmem) return true;
  return false;
}

cudaError_t launch_cluster(const Params& p, const LayerTable& lt, int G, int cs, int max_clusters,
                           cudaStream_t s) {
  const int nbg = lt.n * p.B * p.Hkv;
  cudaError_t e;
  if (cs <= 0 && (e = choose_cluster_size(G, p.P, p.max_pages, p.top_k, nbg, &cs)) != cudaSuccess)
    return e;
  const void* fn = pick_cluster(G, p.P);
  const size_t smem = cluster_smem_bytes(G, p.P, p.max_pages, cs, p.top_k);
  int resident = 0;
  if ((e = resident_clusters(G, p.P, p.max_pages, p.top_k, cs, &resident)) != cudaSuccess)
    return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  // as many clusters as can be resident at once (they loop over the pairs)
  long long ncl = nbg;
  if (ncl > resident) ncl = resident;
  if (max_clusters > 0 && ncl > max_clusters) ncl = max_clusters;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(cs, (int)ncl, smem, s, attr);
  Params pp = p;
  int c = cs;
  LayerTable tt = lt;
  void* args[] = {&pp, &c, &tt};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace quest
