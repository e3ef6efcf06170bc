// quest_fused_kernel.cu - a whole Quest decode step in one persistent, warp-specialised
// launch: (optional) append of the new token, page scoring, top-K selection and split-K
// sparse flash-decode.
//
// "Guide to Quest", Best Practices step 3 suggests fusing the bound estimation with the
// page gather so that nothing sits between the phases.  Structure of one CTA:
//
//   producer warp (warp 8)  takes work items from a queue in the workspace, resolves
//       their pages through the block table and streams their data into a shared-memory
//       ring with 1-D bulk copies (TMA): for a scoring item, the 512 B box records of 16
//       (P=16) or 32 (P=32) pages per stage; for a decode item, the K and V chunks of one
//       kept page per stage.  It runs ahead of the consumers by up to kStages stages and
//       kQueue items, so the latency of tickets, block-table rows and copies overlaps the
//       consumers' work on earlier items.
//   consumer warps (0..7)   take the items in the same order and compute: scores of the
//       staged boxes (half-warp per page), or flash-decode of the staged pages (warp per
//       page); per-item steps (top-K, warp merge, split merge) sync on a named barrier
//       that the producer does not join.
//
// Queue order: the scoring items of (b, g) come before its decode items, which follow
// the scoring items of `decode_lag` later (b, g) pairs, so HBM sees both streams at once
// and a (b, g)'s selection is usually ready when its decode items are taken.  The CTA
// that finishes the last scoring item of a (b, g) selects its pages and publishes them
// (flag = launch epoch + 1); a producer holding a decode item of that (b, g) waits for
// the flag (bounded).  A waiting producer only waits on items handed out earlier to
// running CTAs whose consumers never wait on producers of other CTAs, so the queue cannot
// deadlock.  The CTA that finishes the last decode item of a (b, g) merges its partials.
#include "quest_device.cuh"

namespace quest {

namespace {

constexpr int kQueue = 4;  // item descriptors in flight per CTA
constexpr int kKindScore = 0, kKindDecode = 1, kKindEnd = 2;

// Trace events (see quest_opts_t::trace).
enum TraceEvent : int {
  kEvCtaStart = 1, kEvCtaExit = 2, kEvTicket = 3, kEvReadyWait = 4, kEvReadyDone = 5,
  kEvItemBegin = 6, kEvItemEnd = 7, kEvTopkBegin = 8, kEvTopkEnd = 9, kEvMergeBegin = 10,
  kEvMergeEnd = 11, kEvPushed = 13, kEvFirstStage = 14, kEvStagesDone = 15, kEvArrived = 16,
};

__device__ __forceinline__ void trace(const Params& p, int ev, int item) {
  if (p.trace == nullptr) return;
  const unsigned long long i = atomicAdd(p.trace, 1ull);
  if (i < (unsigned long long)p.trace_capacity) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    p.trace[1 + 2 * i] = (unsigned long long)global_ns();
    p.trace[2 + 2 * i] = ((unsigned long long)smid << 48) |
                         ((unsigned long long)(blockIdx.x & 0xffff) << 32) |
                         ((unsigned long long)(ev & 0xff) << 24) | (unsigned)(item & 0xffffff);
  }
}

struct ItemDesc {
  int kind;
  int b, g, bg;
  int sub;          // scoring tile or decode split
  int first;        // first page (scoring) or first rank (decode)
  int n_units;      // stages the producer pushes for this item
  int n_live;       // scoring: pages of the tile that exist
  int L, N, count;  // tokens (after the append), pages, kept pages
  unsigned stage_base;
  int append_page;  // scoring: logical page that receives the appended token, else -1
  int append_phys;  // its physical page
  int pad[2];
};
static_assert(sizeof(ItemDesc) == 64, "item descriptor is 64 B");

struct StageDesc {
  int n;       // decode: valid tokens of the staged page; scoring: unused
  int first;   // scoring: logical page of slot 0
  unsigned mask;  // scoring: slots that hold a record
  int pad;
};

template <int P>
struct FusedShape {
  static constexpr int kStageBytes = 2 * P * kHeadDim * 2;  // one page's K + V chunks
  static constexpr int kBoxesPerStage = kStageBytes / (2 * kHeadDim * 2);  // 16 or 32
};

struct FusedSmem {
  unsigned char* ring;
  uint64_t *full, *empty, *item_full, *item_empty;
  StageDesc* stage;
  ItemDesc* item;
  float* wsc;
  float* st;
  float* red;     // warp merge of a decode item       } these three share memory:
  float* mscale;  // split merge                        } a consumer uses one at a time
  unsigned char* topk;  // top-K keys / histogram      }
  int* lens;      // seq_lens[0 .. min(B, kLenCache)) read once per CTA
  int* scratch;
  int* misc;
};

constexpr int kLenCache = 1024;   // sequence lengths cached in shared memory

__host__ __device__ inline size_t fused_smem_layout(int G, int P, int max_pages, FusedSmem* s,
                                                    unsigned char* base) {
  const size_t stage = (size_t)2 * P * kHeadDim * 2;
  const size_t red = (size_t)kConsumerWarps * G * kHeadDim * 4;
  const size_t msc = (size_t)G * (kMaxSplits + 2) * 4;
  const size_t keys = topk_smem_bytes(max_pages);
  const size_t aux = (red + msc > keys) ? red + msc : keys;
  size_t o = 0;
  const size_t ring = o;       o = align_up(o + kStages * stage, 128);
  const size_t full = o;       o += kStages * 8;
  const size_t empty = o;      o += kStages * 8;
  const size_t ifull = o;      o += kQueue * 8;
  const size_t iempty = o;     o += kQueue * 8;
  const size_t sdesc = o;      o = align_up(o + kStages * sizeof(StageDesc), 16);
  const size_t idesc = o;      o = align_up(o + kQueue * sizeof(ItemDesc), 16);
  const size_t wsc = o;        o = align_up(o + (size_t)kConsumerWarps * G * P * 4, 16);
  const size_t st = o;         o = align_up(o + (size_t)kConsumerWarps * G * 3 * 4, 16);
  const size_t auxo = o;       o = align_up(o + aux, 16);
  const size_t lens = o;       o += kLenCache * 4;
  const size_t scratch = o;    o += 64 * 4;
  const size_t misc = o;       o += 16 * 4;
  if (s) {
    s->ring = base + ring;
    s->full = reinterpret_cast<uint64_t*>(base + full);
    s->empty = reinterpret_cast<uint64_t*>(base + empty);
    s->item_full = reinterpret_cast<uint64_t*>(base + ifull);
    s->item_empty = reinterpret_cast<uint64_t*>(base + iempty);
    s->stage = reinterpret_cast<StageDesc*>(base + sdesc);
    s->item = reinterpret_cast<ItemDesc*>(base + idesc);
    s->wsc = reinterpret_cast<float*>(base + wsc);
    s->st = reinterpret_cast<float*>(base + st);
    s->red = reinterpret_cast<float*>(base + auxo);
    s->mscale = reinterpret_cast<float*>(base + auxo + red);
    s->topk = base + auxo;
    s->lens = reinterpret_cast<int*>(base + lens);
    s->scratch = reinterpret_cast<int*>(base + scratch);
    s->misc = reinterpret_cast<int*>(base + misc);
  }
  return o;
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Ticket -> (kind, b*Hkv + g, tile or split).  Rounds i = 0 .. nbg-1+lag: round i holds
// the scoring items of pair i (if i < nbg), then the decode items of pair i - lag (if
// i >= lag).
__device__ __forceinline__ void map_ticket(unsigned t, int nbg, int S, int D, int lag, int* kind,
                                           int* bg, int* sub) {
  const int A = min(lag, nbg);
  const long long a_items = (long long)A * S;
  if ((long long)t < a_items) {
    *kind = kKindScore; *bg = t / S; *sub = t % S;
    return;
  }
  long long r = (long long)t - a_items;
  const long long b_items = (long long)(nbg - A) * (S + D);
  if (r < b_items) {
    const int round = (int)(r / (S + D)), o = (int)(r % (S + D));
    if (o < S) {
      *kind = kKindScore; *bg = A + round; *sub = o;
    } else {
      *kind = kKindDecode; *bg = round; *sub = o - S;
    }
    return;
  }
  r -= b_items;
  *kind = kKindDecode;
  *bg = (nbg - A) + (int)(r / D);
  *sub = (int)(r % D);
}

// Length of sequence b as this launch sees it: seq_lens[b], plus one when a token is
// appended and it fits.  *append_ok tells whether the append applies.
__device__ __forceinline__ int step_len(const Params& p, const int* lens, int b, bool* append_ok) {
  const int L0 = b < kLenCache ? lens[b] : p.seq_lens[b];
  *append_ok = false;
  if (L0 < 0 || (long long)L0 > (long long)p.max_pages * p.P) return -1;
  if (p.k_new != nullptr && (long long)L0 + 1 <= (long long)p.max_pages * p.P) {
    *append_ok = true;
    return L0 + 1;
  }
  return L0;
}

// ------------------------------------------------------------------------------------
// producer warp
// ------------------------------------------------------------------------------------
template <int G, int P>
__device__ void produce(const Params& p, const FusedSmem& s, unsigned target) {
  constexpr int kStage = FusedShape<P>::kStageBytes;
  constexpr int kSP = FusedShape<P>::kBoxesPerStage;
  constexpr uint32_t kChunk = P * kHeadDim * 2;
  const int lane = threadIdx.x & 31;
  const int nbg = p.B * p.Hkv;
  const unsigned n_items = (unsigned)nbg * (unsigned)(p.n_score_tiles + p.n_splits);
  uint32_t item_seq = 0, stage_seq = 0;
  unsigned t_next = 0;
  if (lane == 0) t_next = atomicAdd(p.ticket, 1u);
  while (true) {
    // the next ticket is requested one item ahead, so its latency overlaps this item
    unsigned t = __shfl_sync(0xffffffffu, t_next, 0);
    if (lane == 0 && t < n_items) t_next = atomicAdd(p.ticket, 1u);
    const int slot = (int)(item_seq % kQueue);
    bool ok = true;
    if (lane == 0) {
      trace(p, kEvTicket, (int)t);
      ok = mbar_wait_bounded(p, &s.item_empty[slot], ((item_seq / kQueue) & 1u) ^ 1u, kSiteWaitSlot);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) return;
    ItemDesc d;
    d.kind = kKindEnd;
    d.n_units = 0;
    d.stage_base = stage_seq;
    d.append_page = -1;
    d.append_phys = -1;
    if (t < n_items) {
      int kind, bg, sub;
      map_ticket(t, nbg, p.n_score_tiles, p.n_splits, p.decode_lag, &kind, &bg, &sub);
      const int b = bg / p.Hkv, g = bg % p.Hkv;
      bool append_ok;
      int L = step_len(p, s.lens, b, &append_ok);
      if (L < 0) {
        if (lane == 0) report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteScore);
        L = 0;
      }
      const int N = (L + P - 1) / P;
      d.kind = kind; d.b = b; d.g = g; d.bg = bg; d.sub = sub; d.L = L; d.N = N;
      d.count = min(p.top_k, N);
      if (kind == kKindScore) {
        const int p0 = sub * p.score_tile_pages;
        const int n_live = max(0, min(N - p0, min(p.score_tile_pages, p.max_pages - p0)));
        d.first = p0;
        d.n_live = n_live;
        d.n_units = (n_live + kSP - 1) / kSP;
        if (append_ok) {
          const int pa = (L - 1) / P;
          if (pa >= p0 && pa < p0 + n_live) {
            const int phys = p.block_table[(size_t)b * p.max_pages + pa];
            d.append_page = pa;
            d.append_phys = (phys >= 0 && phys < p.num_phys) ? phys : -1;
          }
        }
      } else {
        const int r0 = sub * p.pps;
        const int n_tile = max(0, min(d.count - r0, p.pps));
        d.first = r0;
        d.n_live = n_tile;
        d.n_units = n_tile;
        if (n_tile > 0) {
          bool ready = true;
          if (lane == 0) {
            trace(p, kEvReadyWait, (int)t);
            ready = wait_flag_bounded(p, &p.ready[bg], target, b, kSiteWaitSelection);
            trace(p, kEvReadyDone, (int)t);
          }
          ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
          if (!ready) d.n_units = 0;
          // a page's appended K/V row was written by generic stores in this launch
          if (p.k_new != nullptr) fence_proxy_async_global();
        }
      }
    }
    if (lane == 0) {
      s.item[slot] = d;
      mbar_arrive(&s.item_full[slot]);
    }
    __syncwarp();
    if (d.kind == kKindEnd) return;

    if (d.kind == kKindScore) {
      // the item's boxes are contiguous: one bulk copy of up to kSP records per stage
      if (lane == 0) {
        const __half* box0 = p.meta + box_offset(p, d.b, d.g, d.first);
        for (int u0 = 0; u0 < d.n_live; u0 += kSP) {
          const uint32_t k = stage_seq + (uint32_t)(u0 / kSP);
          const int st = (int)(k % kStages);
          const bool free_ok =
              mbar_wait_bounded(p, &s.empty[st], ((k / kStages) & 1u) ^ 1u, kSiteWaitSlot);
          const int n = min(kSP, d.n_live - u0);
          s.stage[st].first = d.first + u0;
          s.stage[st].mask = free_ok ? (n == 32 ? 0xffffffffu : ((1u << n) - 1u)) : 0u;
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
      stage_seq += (uint32_t)d.n_units;
      __syncwarp();
    } else if (d.n_units > 0) {
      const int* sel_row = p.sel_idx + (size_t)d.bg * p.top_k;
      const size_t chunk_elems = (size_t)P * kHeadDim;
      for (int c = 0; c < d.n_units; c += 32) {
        const int r = c + lane;
        int nv = 0;
        const __half* ksrc = nullptr;
        const __half* vsrc = nullptr;
        int lp = -1;
        if (r < d.n_units) {
          lp = __ldcg(sel_row + d.first + r);
          if (lp < 0 || lp >= d.N) {
            report(p, QUEST_ERR_BAD_SELECTION, d.b, lp, kSiteSelection);
          } else {
            const int phys = p.block_table[(size_t)d.b * p.max_pages + lp];
            if (phys < 0 || phys >= p.num_phys) {
              report(p, QUEST_ERR_BAD_PAGE, d.b, lp, kSiteDecode);
            } else {
              nv = min(P, d.L - lp * P);
              const size_t off = ((size_t)phys * p.Hkv + d.g) * chunk_elems;
              ksrc = p.k_pool + off;
              vsrc = p.v_pool + off;
            }
          }
        }
        const int cnt = min(32, d.n_units - c);
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
    if (lane == 0) trace(p, kEvPushed, (int)t);
    ++item_seq;
  }
}

// ------------------------------------------------------------------------------------
// consumer warps
// ------------------------------------------------------------------------------------
// Scores of one scoring item; applies the appended token to its page's box first.
template <int G, int P>
__device__ void consume_score(const Params& p, const FusedSmem& s, const ItemDesc& d,
                              unsigned target) {
  constexpr int kStage = FusedShape<P>::kStageBytes;
  constexpr int kSP = FusedShape<P>::kBoxesPerStage;
  const int tid = threadIdx.x, lane = tid & 31;
  const int hw = tid >> 4, c = tid & 15;
  QueryFrag<G> f;
  load_query_frag<G>(p, d.b, d.g, c, f);
  float* row = p.scores + (size_t)d.bg * p.max_pages;
  // the appended token (its key widens, or opens, the box of page append_page)
  uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
  const int slot_a = (d.L - 1) % P;
  if (d.append_page >= 0) {
    const size_t o = ((size_t)d.b * p.Hkv + d.g) * kHeadDim + 8 * c;
    knew = *reinterpret_cast<const uint4*>(p.k_new + o);
    vnew = *reinterpret_cast<const uint4*>(p.v_new + o);
  }
  for (int u = 0; u < d.n_units; ++u) {
    const uint32_t k = d.stage_base + (uint32_t)u;
    const int st = (int)(k % kStages);
    mbar_wait_bounded(p, &s.full[st], (k / kStages) & 1u, kSiteWaitStage);
    if (u == 0 && tid == 0) trace(p, kEvFirstStage, d.bg);
    const StageDesc sd = s.stage[st];
#pragma unroll
    for (int rep = 0; rep < kSP / 16; ++rep) {
      const int j = hw + 16 * rep;
      const int page = sd.first + j;
      const bool live = page < d.first + d.n_live;
      const bool have = (sd.mask >> j) & 1u;
      const unsigned char* rec = s.ring + (size_t)st * kStage + (size_t)j * 2 * kHeadDim * 2;
      uint4 mn = *reinterpret_cast<const uint4*>(rec + 16 * c);
      uint4 mx = *reinterpret_cast<const uint4*>(rec + 2 * kHeadDim + 16 * c);
      if (page == d.append_page && have) {
        if (d.append_phys >= 0) {
          if (slot_a == 0) {
            mn = knew;
            mx = knew;
          } else {
            const uint32_t a[4] = {mn.x, mn.y, mn.z, mn.w};
            const uint32_t z[4] = {mx.x, mx.y, mx.z, mx.w};
            const uint32_t n[4] = {knew.x, knew.y, knew.z, knew.w};
            uint32_t ra[4], rz[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const __half2 hn = *reinterpret_cast<const __half2*>(&n[q]);
              const __half2 lo = __hmin2(*reinterpret_cast<const __half2*>(&a[q]), hn);
              const __half2 hi = __hmax2(*reinterpret_cast<const __half2*>(&z[q]), hn);
              ra[q] = *reinterpret_cast<const uint32_t*>(&lo);
              rz[q] = *reinterpret_cast<const uint32_t*>(&hi);
            }
            mn = make_uint4(ra[0], ra[1], ra[2], ra[3]);
            mx = make_uint4(rz[0], rz[1], rz[2], rz[3]);
          }
          const size_t ph = (size_t)d.append_phys;
          __half* box = p.meta + box_offset(p, d.b, d.g, page);
          *reinterpret_cast<uint4*>(box + 8 * c) = mn;
          *reinterpret_cast<uint4*>(box + kHeadDim + 8 * c) = mx;
          const size_t kv = ((ph * p.Hkv + d.g) * P + slot_a) * kHeadDim + 8 * c;
          *reinterpret_cast<uint4*>(p.k_pool + kv) = knew;
          *reinterpret_cast<uint4*>(p.v_pool + kv) = vnew;
        } else if (c == 0) {
          report(p, QUEST_ERR_BAD_PAGE, d.b, page, kSiteAppend);
        }
      }
      float best = -CUDART_INF_F;
#pragma unroll
      for (int jj = 0; jj < G; ++jj) {
        float sc = corner_dot<G>(f, jj, mn, mx);
        sc += __shfl_xor_sync(0xffffffffu, sc, 8);
        sc += __shfl_xor_sync(0xffffffffu, sc, 4);
        sc += __shfl_xor_sync(0xffffffffu, sc, 2);
        sc += __shfl_xor_sync(0xffffffffu, sc, 1);
        best = fmaxf(best, sc);
      }
      if (c == 0 && live) row[page] = have ? best : -CUDART_INF_F;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s.empty[st]);
  }
  if (tid == 0) trace(p, kEvStagesDone, d.bg);
  if (d.append_page >= 0) fence_proxy_async_global();  // appended rows, before the selection
  const bool last = arrive_last<kConsumerThreads, true>(&p.score_arrive[d.bg],
                                                        (unsigned)p.n_score_tiles, s.misc + 1);
  if (tid == 0) trace(p, kEvArrived, d.bg);
  if (last) {
    if (tid == 0) trace(p, kEvTopkBegin, d.bg);
    topk_row<kConsumerThreads, true>(row, d.N, p.top_k, p.sink_pages, p.local_pages,
                                     p.sel_idx + (size_t)d.bg * p.top_k,
                                        p.sel_count + d.bg, topk_smem_at(s.topk, p.max_pages),
                                        s.scratch);
    bsync<kConsumerThreads, true>();  // every thread's selection writes precede the release
    if (tid == 0) {
      p.score_arrive[d.bg] = 0u;
      if (!(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION)) st_release_u32(&p.ready[d.bg], target);
      trace(p, kEvTopkEnd, d.bg);
    }
  }
}

// Flash-decode of one decode item; writes its partial and merges if it is the last.
template <int G, int P>
__device__ void consume_decode(const Params& p, const FusedSmem& s, const ItemDesc& d) {
  constexpr int kStage = FusedShape<P>::kStageBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (d.n_units > 0) {
    float qf[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint2 raw = *reinterpret_cast<const uint2*>(
          p.q + ((size_t)d.b * p.Hq + d.g * G + j) * kHeadDim + 4 * lane);
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
    for (int r = warp; r < d.n_units; r += kConsumerWarps) {
      const uint32_t k = d.stage_base + (uint32_t)r;
      const int stg = (int)(k % kStages);
      const bool ok = mbar_wait_bounded(p, &s.full[stg], (k / kStages) & 1u, kSiteWaitStage);
      const int nv = ok ? s.stage[stg].n : 0;
      if (nv > 0) {
        const __half* Ks = reinterpret_cast<const __half*>(s.ring + (size_t)stg * kStage);
        page_update<G, P>(qf, acc, Ks, Ks + P * kHeadDim, nv, sc, st, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&s.empty[stg], kConsumerWarps);
    }
    bsync<kConsumerThreads, true>();
    // merge the 8 warps' states into this item's partial
#pragma unroll
    for (int j = 0; j < G; ++j)
      *reinterpret_cast<float4*>(s.red + ((size_t)warp * G + j) * kHeadDim + 4 * lane) =
          make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
    bsync<kConsumerThreads, true>();
    for (int o = tid; o < G * kHeadDim; o += kConsumerThreads) {
      const int j = o / kHeadDim, i = o % kHeadDim;
      float M = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s.st[(w * G + j) * 3]);
      float A = 0.f, Ls = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = s.st[(w * G + j) * 3];
        if (mw != -CUDART_INF_F) {
          const float f = exp2f(mw - M);
          A = fmaf(s.red[((size_t)w * G + j) * kHeadDim + i], f, A);
          Ls = fmaf(s.st[(w * G + j) * 3 + 1], f, Ls);
        }
      }
      const size_t slot = (size_t)(d.b * p.Hq + d.g * G + j) * p.n_splits + d.sub;
      p.part_acc[slot * kHeadDim + i] = A;
      if (i == 0) {
        p.part_ml[slot * 2] = M;
        p.part_ml[slot * 2 + 1] = Ls;
      }
    }
  }
  if (arrive_last<kConsumerThreads, true>(&p.decode_arrive[d.bg], (unsigned)p.n_splits,
                                          s.misc + 3)) {
    if (tid == 0) trace(p, kEvMergeBegin, d.bg);
    merge_splits<G, kConsumerThreads, true>(p, s.mscale, d.b, d.g, (d.count + p.pps - 1) / p.pps);
    if (tid == 0) {
      p.decode_arrive[d.bg] = 0u;
      trace(p, kEvMergeEnd, d.bg);
    }
  }
}

template <int G, int P>
__device__ void consume(const Params& p, const FusedSmem& s, unsigned target) {
  const int tid = threadIdx.x;
  uint32_t item_seq = 0;
  while (true) {
    const int slot = (int)(item_seq % kQueue);
    // one thread waits and the others follow its outcome, so that all consumer warps
    // always reach the same named barriers
    if (tid == 0)
      s.misc[5] = mbar_wait_bounded(p, &s.item_full[slot], (item_seq / kQueue) & 1u, kSiteWaitSlot);
    bsync<kConsumerThreads, true>();
    if (!s.misc[5]) return;
    const ItemDesc d = s.item[slot];
    bsync<kConsumerThreads, true>();
    if (tid == 0) mbar_arrive(&s.item_empty[slot]);
    if (d.kind == kKindEnd) return;
    if (tid == 0) trace(p, kEvItemBegin, d.kind * 0x100000 + d.bg * 0x400 + d.sub);
    if (d.kind == kKindScore)
      consume_score<G, P>(p, s, d, target);
    else
      consume_decode<G, P>(p, s, d);
    if (tid == 0) trace(p, kEvItemEnd, d.kind * 0x100000 + d.bg * 0x400 + d.sub);
    ++item_seq;
  }
}

}  // namespace

template <int G, int P>
__global__ void __launch_bounds__(kDecodeThreads, (P == 16 && G <= 4) ? 2 : 1)
    fused_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  FusedSmem s;
  fused_smem_layout(G, P, p.max_pages, &s, smem);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(&s.item_full[i], 1);
      mbar_init(&s.item_empty[i], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  for (int b = threadIdx.x; b < min(p.B, kLenCache); b += blockDim.x) s.lens[b] = p.seq_lens[b];
  __syncthreads();
  const unsigned target = *p.epoch + 1u;
  if (threadIdx.x == 0) trace(p, kEvCtaStart, 0);
  if (threadIdx.x >= kConsumerThreads)
    produce<G, P>(p, s, target);
  else
    consume<G, P>(p, s, target);
  __syncthreads();
  if (threadIdx.x == 0) {
    trace(p, kEvCtaExit, 0);
    __threadfence();
    if (atomicAdd(p.exited, 1u) == gridDim.x - 1u) {
      // every CTA is done: reset the queue, advance the epoch and the lengths
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
      *p.ticket = 0u;
      *p.exited = 0u;
      *p.epoch = target;
    }
  }
}

template <int G, int P>
static const void* fused_fn() { return (const void*)fused_kernel<G, P>; }

static const void* pick_fused(int G, int P) {
  if (P == 16) {
    switch (G) {
      case 1: return fused_fn<1, 16>();
      case 2: return fused_fn<2, 16>();
      case 4: return fused_fn<4, 16>();
      default: return fused_fn<8, 16>();
    }
  }
  switch (G) {
    case 1: return fused_fn<1, 32>();
    case 2: return fused_fn<2, 32>();
    case 4: return fused_fn<4, 32>();
    default: return fused_fn<8, 32>();
  }
}

size_t fused_smem_bytes(int G, int P, int max_pages) {
  return fused_smem_layout(G, P, max_pages, nullptr, nullptr);
}

cudaError_t launch_fused(const Params& p, int G, int max_ctas, cudaStream_t s) {
  const void* fn = pick_fused(G, p.P);
  const size_t smem = fused_smem_bytes(G, p.P, p.max_pages);
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, per_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kDecodeThreads, smem)) !=
      cudaSuccess)
    return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long n_items =
      (long long)p.B * p.Hkv * (p.n_score_tiles + (long long)p.n_splits);
  long long grid = (long long)sms * per_sm;
  if (max_ctas > 0 && grid > max_ctas) grid = max_ctas;
  if (grid > n_items) grid = n_items;
  if (grid < 1) grid = 1;
  Params pp = p;
  void* args[] = {&pp};
  return launch_pdl(fn, dim3((unsigned)grid), dim3(kDecodeThreads), smem, s, args);
}

}  // namespace quest
