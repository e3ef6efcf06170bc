// quest_cluster_kernel.cu - the whole Quest decode step of one (sequence, kv head) in one
// thread-block cluster: (optional) append, page scoring, top-K, split-K sparse decode and
// the log-sum-exp merge, with every cross-CTA step in distributed shared memory.
//
// "Guide to Quest", Best Practices step 3 asks for the bound estimation to be fused with
// the page gather.  On GB300 the natural unit for that is a cluster of CS CTAs (8 by
// default) per (b, g) pair:
//   1. each CTA scores a contiguous share of the pair's pages (boxes streamed by 1-D bulk
//      copies through an mbarrier ring by a producer warp) and stores the scores, as
//      order-preserving keys, straight into the leader's (rank 0) shared memory;
//   2. each CTA signals the leader with a remote mbarrier arrive; the leader selects the
//      top-K pages ("Guide to Quest", Solution step 3) from its local copy of the keys into
//      its shared memory, then arrives on every CTA's selection barrier;
//   3. each CTA's producer reads its share of the selection from the leader, resolves the
//      pages through the block table and streams their K / V chunks; the consumer warps
//      run flash-decode over them (Tang 2024 summary: exact attention over the Top-K);
//   4. each CTA stores its partial (max, sum, accumulator) into the leader's shared memory
//      and signals it; the leader merges the partials by log-sum-exp and writes the output.
// No global atomics, flags or work queue sit on the critical path.  Clusters are
// persistent: cluster c handles pairs c, c + #clusters, ...  Every wait is bounded.
#include <map>
#include <mutex>
#include <tuple>

#include "quest_device.cuh"

namespace quest {

namespace {

enum ClusterTraceEvent : int {
  kCtStart = 1, kCtExit = 2, kCtScoreDone = 20, kCtTopkBegin = 21, kCtTopkEnd = 22,
  kCtSelReady = 23, kCtDecodeDone = 24, kCtMergeBegin = 25, kCtMergeEnd = 26,
};

// Timeline record without atomics: CTA c owns records [c * kTraceSlots, (c + 1) *
// kTraceSlots) of the trace buffer; `slot` is the caller's running count (thread 0 only).
constexpr int kTraceSlots = 64;
__device__ __forceinline__ void ctrace(const Params& p, int* slot, int ev, int item) {
  if (p.trace == nullptr) return;
  const long long i = (long long)blockIdx.x * kTraceSlots + (*slot)++;
  if (*slot > kTraceSlots || i >= p.trace_capacity) return;
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

struct CSmem {
  unsigned char* ring;
  uint64_t *full, *empty;
  uint64_t* bar_scores;  // leader: every CTA's scores are in place (count CS)
  uint64_t* bar_sel;     // every CTA: the leader's selection is in place (count 1)
  uint64_t* bar_part;    // leader: every CTA's partial is in place (count CS)
  StageInfo* stage;
  uint32_t* keys;        // leader: score keys of the pair's pages (stored by every CTA)
  uint32_t* ranges;      // leader: [CS][2] key range of each CTA's share
  int* sel;              // leader: the kept pages, ascending
  float* parts;          // leader: [CS][G*(128+2)] partials M[G], L[G], A[G][128]
  float* wsc;
  float* st;
  unsigned char* aux;    // leader top-K histogram / candidates, or the warp merge buffer
  int* lens;
  int* scratch;
  int* misc;
};

constexpr int kLenCache = 1024;

__host__ __device__ inline size_t cluster_smem_layout(int G, int P, int max_pages, int cs,
                                                      int top_k, CSmem* s, unsigned char* base) {
  const size_t stage = (size_t)2 * P * kHeadDim * 2;
  const int kcap = top_k < max_pages ? top_k : max_pages;
  const size_t red = (size_t)kConsumerWarps * G * kHeadDim * 4;
  const size_t tk = (size_t)kTopkBins * 4 + (size_t)kTopkCand * 8 +
                    align_up((size_t)((max_pages + 31) / 32) * 4, 16);
  const size_t aux = red > tk ? red : tk;
  const size_t part_floats = (size_t)G * (kHeadDim + 2);
  size_t o = 0;
  const size_t ring = o;     o = align_up(o + kStages * stage, 128);
  const size_t full = o;     o += kStages * 8;
  const size_t empty = o;    o += kStages * 8;
  const size_t bars = o;     o += 3 * 8;
  const size_t sdesc = o;    o = align_up(o + kStages * sizeof(StageInfo), 16);
  const size_t keys = o;     o = align_up(o + (size_t)max_pages * 4, 16);
  const size_t ranges = o;   o = align_up(o + (size_t)cs * 2 * 4, 16);
  const size_t sel = o;      o = align_up(o + (size_t)kcap * 4, 16);
  const size_t parts = o;    o = align_up(o + (size_t)cs * part_floats * 4, 16);
  const size_t wsc = o;      o = align_up(o + (size_t)kConsumerWarps * G * P * 4, 16);
  const size_t st = o;       o = align_up(o + (size_t)kConsumerWarps * G * 3 * 4, 16);
  const size_t auxo = o;     o = align_up(o + aux, 16);
  const size_t lens = o;     o += kLenCache * 4;
  const size_t scratch = o;  o += 64 * 4;
  const size_t misc = o;     o += 16 * 4;
  if (s) {
    s->ring = base + ring;
    s->full = reinterpret_cast<uint64_t*>(base + full);
    s->empty = reinterpret_cast<uint64_t*>(base + empty);
    s->bar_scores = reinterpret_cast<uint64_t*>(base + bars);
    s->bar_sel = s->bar_scores + 1;
    s->bar_part = s->bar_scores + 2;
    s->stage = reinterpret_cast<StageInfo*>(base + sdesc);
    s->keys = reinterpret_cast<uint32_t*>(base + keys);
    s->ranges = reinterpret_cast<uint32_t*>(base + ranges);
    s->sel = reinterpret_cast<int*>(base + sel);
    s->parts = reinterpret_cast<float*>(base + parts);
    s->wsc = reinterpret_cast<float*>(base + wsc);
    s->st = reinterpret_cast<float*>(base + st);
    s->aux = base + auxo;
    s->lens = reinterpret_cast<int*>(base + lens);
    s->scratch = reinterpret_cast<int*>(base + scratch);
    s->misc = reinterpret_cast<int*>(base + misc);
  }
  return o;
}

// Geometry of pair bg as this launch sees it (identical in every CTA and warp).
struct Pair {
  int b, g, L, N, count;   // tokens (after the append), pages, kept pages
  int p_lo, p_hi;          // this CTA's scoring share
  int q_lo, q_hi;          // this CTA's decode share (ranks of the selection)
  int share;               // pages per scoring share
  int append_page, append_phys;
};

__device__ __forceinline__ Pair pair_geometry(const Params& p, const CSmem& s, int bg, int rank,
                                              int cs) {
  Pair q;
  q.b = bg / p.Hkv;
  q.g = bg % p.Hkv;
  const int L0 = q.b < kLenCache ? s.lens[q.b] : p.seq_lens[q.b];
  const long long cap = (long long)p.max_pages * p.P;
  int L = L0;
  if (L0 < 0 || (long long)L0 > cap) {
    if (rank == 0 && q.g == 0 && threadIdx.x == 0) report(p, QUEST_ERR_BAD_LENGTH, q.b, -1, kSiteScore);
    L = 0;
  }
  q.append_page = -1;
  q.append_phys = -1;
  if (p.k_new != nullptr && L0 >= 0 && (long long)L0 + 1 <= cap) {
    L = L0 + 1;
    q.append_page = L0 / p.P;
    const int phys = p.block_table[(size_t)q.b * p.max_pages + q.append_page];
    q.append_phys = (phys >= 0 && phys < p.num_phys) ? phys : -1;
  }
  q.L = L;
  q.N = (L + p.P - 1) / p.P;
  q.count = min(p.top_k, q.N);
  q.share = (q.N + cs - 1) / cs;
  q.p_lo = min(q.N, rank * q.share);
  q.p_hi = min(q.N, q.p_lo + q.share);
  q.q_lo = (int)((long long)q.count * rank / cs);
  q.q_hi = (int)((long long)q.count * (rank + 1) / cs);
  return q;
}

// ---------------------------------------------------------------- producer warp
template <int G, int P>
__device__ void c_produce(const Params& p, const CSmem& s, int rank, int cs) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  constexpr uint32_t kChunk = P * kHeadDim * 2;
  const int lane = threadIdx.x & 31;
  const int nbg = p.B * p.Hkv;
  const int cid = (int)cluster_index(), ncl = (int)cluster_count();
  uint32_t stage_seq = 0;
  int it = 0;
  for (int bg = cid; bg < nbg; bg += ncl, ++it) {
    const Pair q = pair_geometry(p, s, bg, rank, cs);
    // 1. this CTA's scoring share: contiguous boxes, one bulk copy per stage
    const int n_live = q.p_hi - q.p_lo;
    if (lane == 0) {
      const __half* box0 = p.meta + box_offset(p, q.b, q.g, q.p_lo);
      for (int u0 = 0; u0 < n_live; u0 += kSP) {
        const uint32_t k = stage_seq + (uint32_t)(u0 / kSP);
        const int st = (int)(k % kStages);
        const bool free_ok =
            mbar_wait_bounded(p, &s.empty[st], ((k / kStages) & 1u) ^ 1u, kSiteWaitSlot);
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
      }
    }
    stage_seq += (uint32_t)((n_live + kSP - 1) / kSP);
    __syncwarp();
    // 2. this CTA's share of the selection, once the leader has published it.  The wait
    //    is made for every pair, even with nothing to decode: a phase parity names the
    //    right phase only while the waiter is at most one phase behind.
    const int n_dec = q.q_hi - q.q_lo;
    bool ok = true;
    if (lane == 0) ok = wait_cluster_bounded(p, s.bar_sel, (uint32_t)it & 1u, kSiteWaitSelection);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (n_dec > 0) {
      if (p.k_new != nullptr) fence_proxy_async_global();  // appended rows: generic writes
      const uint32_t sel0 = remote(s.sel, 0);
      const size_t chunk_elems = (size_t)P * kHeadDim;
      for (int c = 0; c < n_dec; c += 32) {
        const int r = c + lane;
        int nv = 0, lp = -1;
        const __half* ksrc = nullptr;
        const __half* vsrc = nullptr;
        if (ok && r < n_dec) {
          lp = (int)ld_remote_u32(sel0 + 4u * (uint32_t)(q.q_lo + r));
          if (lp < 0 || lp >= q.N) {
            report(p, QUEST_ERR_BAD_SELECTION, q.b, lp, kSiteSelection);
          } else {
            const int phys = p.block_table[(size_t)q.b * p.max_pages + lp];
            if (phys < 0 || phys >= p.num_phys) {
              report(p, QUEST_ERR_BAD_PAGE, q.b, lp, kSiteDecode);
            } else {
              nv = min(P, q.L - lp * P);
              const size_t off = ((size_t)phys * p.Hkv + q.g) * chunk_elems;
              ksrc = p.k_pool + off;
              vsrc = p.v_pool + off;
            }
          }
        }
        const int cnt = min(32, n_dec - c);
        for (int j = 0; j < cnt; ++j) {
          if (lane == j) {
            const uint32_t k = stage_seq + (uint32_t)j;
            const int st = (int)(k % kStages);
            const bool free_ok =
                mbar_wait_bounded(p, &s.empty[st], ((k / kStages) & 1u) ^ 1u, kSiteWaitSlot);
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
    }
  }
}

// ---------------------------------------------------------------- consumer warps
template <int G, int P>
__device__ void c_score_share(const Params& p, const CSmem& s, const Pair& q, uint32_t stage_base,
                              int rank) {
  constexpr int kStage = CShape<P>::kStage;
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  const int tid = threadIdx.x, lane = tid & 31;
  const int hw = tid >> 4, c = tid & 15;
  const int n_live = q.p_hi - q.p_lo;
  if (n_live <= 0) {
    if (tid == 0) {
      const uint32_t r0 = remote(s.ranges, 0) + 8u * (uint32_t)rank;
      st_remote_u32(r0, 0xffffffffu);
      st_remote_u32(r0 + 4u, 0u);
    }
    return;
  }
  const uint32_t keys0 = remote(s.keys, 0);
  uint32_t lo = 0xffffffffu, hi = 0u;
  QueryFrag<G> f;
  load_query_frag<G>(p, q.b, q.g, c, f);
  uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
  const bool mine_append = q.append_page >= q.p_lo && q.append_page < q.p_hi;
  const int slot_a = (q.L - 1) % P;
  if (mine_append) {
    const size_t o = ((size_t)q.b * p.Hkv + q.g) * kHeadDim + 8 * c;
    knew = *reinterpret_cast<const uint4*>(p.k_new + o);
    vnew = *reinterpret_cast<const uint4*>(p.v_new + o);
  }
  const int n_units = (n_live + kSP - 1) / kSP;
  for (int u = 0; u < n_units; ++u) {
    const uint32_t k = stage_base + (uint32_t)u;
    const int st = (int)(k % kStages);
    mbar_wait_bounded(p, &s.full[st], (k / kStages) & 1u, kSiteWaitStage);
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
        if (q.append_phys >= 0) {
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
              const __half2 lo = __hmin2(*reinterpret_cast<const __half2*>(&a[w]), hn);
              const __half2 hi = __hmax2(*reinterpret_cast<const __half2*>(&z[w]), hn);
              ra[w] = *reinterpret_cast<const uint32_t*>(&lo);
              rz[w] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            mn = make_uint4(ra[0], ra[1], ra[2], ra[3]);
            mx = make_uint4(rz[0], rz[1], rz[2], rz[3]);
          }
          __half* box = p.meta + box_offset(p, q.b, q.g, page);
          *reinterpret_cast<uint4*>(box + 8 * c) = mn;
          *reinterpret_cast<uint4*>(box + kHeadDim + 8 * c) = mx;
          const size_t kv = (((size_t)q.append_phys * p.Hkv + q.g) * P + slot_a) * kHeadDim + 8 * c;
          *reinterpret_cast<uint4*>(p.k_pool + kv) = knew;
          *reinterpret_cast<uint4*>(p.v_pool + kv) = vnew;
        } else if (c == 0) {
          report(p, QUEST_ERR_BAD_PAGE, q.b, page, kSiteAppend);
        }
      }
      float best = -CUDART_INF_F;
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        float v = corner_dot<G>(f, jj, mn, mx);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        best = fmaxf(best, v);
      }
      if (c == 0 && page < q.p_hi) {
        const uint32_t key = score_key(have ? best : -CUDART_INF_F);
        st_remote_u32(keys0 + 4u * (uint32_t)page, key);
        lo = min(lo, key);
        hi = max(hi, key);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
  }
  if (mine_append) fence_proxy_async_global();  // appended rows, before the scores are released
  // this share's key range, to the leader
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
    const uint32_t r0 = remote(s.ranges, 0) + 8u * (uint32_t)rank;
    st_remote_u32(r0, l);
    st_remote_u32(r0 + 4u, h);
  }
}

// Leader: select the top-K of the pair's N keys (already in s.keys) into s.sel.
__device__ void c_select(const Params& p, const CSmem& s, const Pair& q, int cs) {
  const int tid = threadIdx.x;
  int* cnt_slot = s.misc + 8;
  if (q.N <= q.count) {
    for (int r = tid; r < q.count; r += kConsumerThreads) s.sel[r] = r;
    if (tid == 0) *cnt_slot = q.N;
    return;
  }
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int r = 0; r < cs; ++r) {
    lo = min(lo, s.ranges[2 * r]);
    hi = max(hi, s.ranges[2 * r + 1]);
  }
  TopkSmem t;
  t.keys = s.keys;
  t.hist = reinterpret_cast<int*>(s.aux);
  t.cand_key = reinterpret_cast<uint32_t*>(s.aux + (size_t)kTopkBins * 4);
  t.cand_idx = reinterpret_cast<int*>(s.aux + (size_t)kTopkBins * 4 + kTopkCand * 4);
  t.kept = reinterpret_cast<uint32_t*>(s.aux + (size_t)kTopkBins * 4 + kTopkCand * 8);
  topk_core<kConsumerThreads, true>(q.N, q.count, s.sel, cnt_slot, t, s.scratch, lo, hi);
}

// Leader: the selection, for the caller, if asked for (after it was released).
__device__ void c_publish_selection(const Params& p, const CSmem& s, const Pair& q) {
  if (p.sel_idx == nullptr) return;
  const int tid = threadIdx.x;
  const int bg = q.b * p.Hkv + q.g;
  int* row = p.sel_idx + (size_t)bg * p.top_k;
  for (int r = tid; r < p.top_k; r += kConsumerThreads) row[r] = r < q.count ? s.sel[r] : -1;
  if (tid == 0 && p.sel_count != nullptr) p.sel_count[bg] = q.count;
}

template <int G, int P>
__device__ void c_decode_share(const Params& p, const CSmem& s, const Pair& q, uint32_t stage_base,
                               int rank) {
  constexpr int kStage = CShape<P>::kStage;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = q.q_hi - q.q_lo;
  // this CTA's partial goes to the leader's slot `rank`: M[G], L[G], A[G][128]
  const uint32_t slot = remote(s.parts, 0) + 4u * (uint32_t)(rank * G * (kHeadDim + 2));
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
        *reinterpret_cast<const uint2*>(p.q + ((size_t)q.b * p.Hq + q.g * G + j) * kHeadDim + 4 * lane);
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
  for (int r = warp; r < n; r += kConsumerWarps) {
    const uint32_t k = stage_base + (uint32_t)r;
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
  bsync<kConsumerThreads, true>();
  // merge the 8 warps into this CTA's partial
  float* red = reinterpret_cast<float*>(s.aux);
#pragma unroll
  for (int j = 0; j < G; ++j)
    *reinterpret_cast<float4*>(red + ((size_t)warp * G + j) * kHeadDim + 4 * lane) =
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
        a = fmaf(red[((size_t)w * G + j) * kHeadDim + i], f, a);
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

// Leader: merge the cluster's partials (in its shared memory) into out / lse.
template <int G>
__device__ void c_merge(const Params& p, const CSmem& s, const Pair& q, int cs) {
  const int tid = threadIdx.x;
  const int stride = G * (kHeadDim + 2);
  for (int o = tid; o < G * kHeadDim; o += kConsumerThreads) {
    const int j = o / kHeadDim, i = o % kHeadDim;
    float Mx = -CUDART_INF_F;
    for (int r = 0; r < cs; ++r) Mx = fmaxf(Mx, s.parts[r * stride + j]);
    float acc = 0.f, ls = 0.f;
    for (int r = 0; r < cs; ++r) {
      const float m = s.parts[r * stride + j];
      if (m != -CUDART_INF_F) {
        const float f = exp2f(m - Mx);
        acc = fmaf(s.parts[r * stride + 2 * G + j * kHeadDim + i], f, acc);
        ls = fmaf(s.parts[r * stride + G + j], f, ls);
      }
    }
    const int h = q.g * G + j;
    p.out[((size_t)q.b * p.Hq + h) * kHeadDim + i] = __float2half_rn(ls > 0.f ? acc / ls : 0.f);
    if (i == 0 && p.lse)
      p.lse[(size_t)q.b * p.Hq + h] =
          ls > 0.f ? (Mx + log2f(ls)) * 0.69314718055994531f : -CUDART_INF_F;
  }
}

template <int G, int P>
__device__ void c_consume(const Params& p, const CSmem& s, int rank, int cs) {
  constexpr int kSP = CShape<P>::kBoxesPerStage;
  const int tid = threadIdx.x;
  const int nbg = p.B * p.Hkv;
  const int cid = (int)cluster_index(), ncl = (int)cluster_count();
  uint32_t stage_seq = 0;
  int it = 0;
  int tslot = 1;  // slot 0: the CTA's start record
  for (int bg = cid; bg < nbg; bg += ncl, ++it) {
    const Pair q = pair_geometry(p, s, bg, rank, cs);
    const uint32_t par = (uint32_t)it & 1u;
    // 1. scoring share -> this CTA's shared memory; tell the leader
    c_score_share<G, P>(p, s, q, stage_seq, rank);
    stage_seq += (uint32_t)((q.p_hi - q.p_lo + kSP - 1) / kSP);
    bsync<kConsumerThreads, true>();
    if (tid == 0) {
      ctrace(p, &tslot, kCtScoreDone, bg);
      arrive_remote(remote(s.bar_scores, 0));
    }
    // 2. leader: select, then publish to every CTA
    if (rank == 0) {
      if (tid == 0) s.misc[6] = wait_cluster_bounded(p, s.bar_scores, par, kSiteWaitSelection) ? 1 : 0;
      bsync<kConsumerThreads, true>();
      if (tid == 0) ctrace(p, &tslot, kCtTopkBegin, bg);
      c_select(p, s, q, cs);
      bsync<kConsumerThreads, true>();
      if (tid == 0) ctrace(p, &tslot, kCtTopkEnd, bg);
      if (tid < cs && !(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION))
        arrive_remote(remote(s.bar_sel, (uint32_t)tid));
      c_publish_selection(p, s, q);
    }
    // no CTA writes its next scores before the leader has read these
    if (tid == 0) s.misc[7] = wait_cluster_bounded(p, s.bar_sel, par, kSiteWaitSelection) ? 1 : 0;
    bsync<kConsumerThreads, true>();
    if (tid == 0) ctrace(p, &tslot, kCtSelReady, bg);
    // 3. decode share -> this CTA's partial; tell the leader
    c_decode_share<G, P>(p, s, q, stage_seq, rank);
    stage_seq += (uint32_t)max(0, q.q_hi - q.q_lo);
    bsync<kConsumerThreads, true>();
    if (tid == 0) {
      ctrace(p, &tslot, kCtDecodeDone, bg);
      arrive_remote(remote(s.bar_part, 0));
    }
    // 4. leader: merge
    if (rank == 0) {
      if (tid == 0) s.misc[6] = wait_cluster_bounded(p, s.bar_part, par, kSiteWaitSlot) ? 1 : 0;
      bsync<kConsumerThreads, true>();
      if (tid == 0) ctrace(p, &tslot, kCtMergeBegin, bg);
      c_merge<G>(p, s, q, cs);
      bsync<kConsumerThreads, true>();
      if (tid == 0) ctrace(p, &tslot, kCtMergeEnd, bg);
    }
  }
}

}  // namespace

template <int G, int P>
__global__ void __launch_bounds__(kDecodeThreads, (P == 16 && G <= 4) ? 2 : 1)
    cluster_kernel(Params p, int cs) {
  extern __shared__ __align__(128) unsigned char smem[];
  CSmem s;
  cluster_smem_layout(G, P, p.max_pages, cs, p.top_k, &s, smem);
  const int rank = (int)cta_rank();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    mbar_init(s.bar_scores, (uint32_t)cs);
    mbar_init(s.bar_sel, 1);
    mbar_init(s.bar_part, (uint32_t)cs);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive
  pdl_wait();
  for (int b = threadIdx.x; b < min(p.B, kLenCache); b += blockDim.x) s.lens[b] = p.seq_lens[b];
  __syncthreads();
  if (threadIdx.x == 0) {
    int slot0 = 0;
    ctrace(p, &slot0, kCtStart, rank);
  }
  if (threadIdx.x >= kConsumerThreads)
    c_produce<G, P>(p, s, rank, cs);
  else
    c_consume<G, P>(p, s, rank, cs);
  __syncthreads();
  cluster_sync_all();  // no CTA leaves while another may still read its shared memory
  if (threadIdx.x == 0) {
    int slot_last = kTraceSlots - 1;
    ctrace(p, &slot_last, kCtExit, rank);
    __threadfence();
    if (atomicAdd(p.exited, 1u) == gridDim.x - 1u) {
      // every CTA is done: advance the lengths of the sequences that received a token
      if (p.k_new != nullptr) {
        for (int b = 0; b < p.B; ++b) {
          const int L0 = p.seq_lens[b];
          if (L0 < 0 || (long long)L0 + 1 > (long long)p.max_pages * p.P) {
            report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);
            continue;
          }
          const int phys = p.block_table[(size_t)b * p.max_pages + L0 / p.P];
          if (phys >= 0 && phys < p.num_phys) p.seq_lens[b] = L0 + 1;
        }
      }
      *p.exited = 0u;
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

// Automatic cluster size: the largest size (up to kMaxClusterSize) at which the clusters of
// all pairs are resident together, so every pair runs at once over as many SMs as possible;
// with more pairs than that, one CTA per pair.
cudaError_t choose_cluster_size(int G, int P, int max_pages, int top_k, int nbg, int* cs_out) {
  for (int cs = kMaxClusterSize; cs > 1; --cs) {
    if (cluster_smem_bytes(G, P, max_pages, cs, top_k) > 227 * 1024) continue;
    int n = 0;
    cudaError_t e = resident_clusters(G, P, max_pages, top_k, cs, &n);
    if (e != cudaSuccess) return e;
    if (n >= nbg) {
      *cs_out = cs;
      return cudaSuccess;
    }
  }
  *cs_out = 1;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_cluster(const Params& p, int G, int cs, int max_clusters, cudaStream_t s) {
  const int nbg = p.B * p.Hkv;
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
  void* args[] = {&pp, &c};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace quest
