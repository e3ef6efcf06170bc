// quest_stream_kernel.cu - the whole Quest decode step in one persistent launch that keeps
// HBM streaming from start to end: page scoring of every (sequence, kv head) pair, the
// top-K of each pair as soon as its last box is scored, and split-K sparse decode of the
// kept pages, with the selection of one pair overlapping the streaming of the others.
//
// "Guide to Quest", Best Practices step 3 asks for the bound estimation to be fused with
// the page gather.  The three steps of a pair depend on one another (all of a pair's
// bounds before its top-K, its top-K before its pages are read), so a pair alone leaves
// HBM idle while it selects.  Here every CTA (one per SM) works on every pair:
//
//   producer warp (12)     walks this CTA's share of the work in a fixed order and
//       streams it into a shared-memory ring with 1-D bulk copies (TMA): first its scoring
//       pieces (the boxes of up to P pages of one pair, "Guide to Quest", Solution
//       step 1), then its decode pieces (the K and V chunks of up to 8 kept pages of one
//       pair, once that pair's selection is published).  The query of the pair rides
//       along in every stage.
//   consumer warps (4..11) stage s belongs to consumer s mod 8.  Scoring stage: the
//       bound of each page (Solution step 2) becomes an order-preserving key in global
//       memory; the warp then counts the piece on the pair's arrival counter, and the
//       warp that completes a pair hands its selection to this CTA's selector team.
//       Decode stage: flash-decode of one kept page (Tang 2024 summary: exact attention
//       over the Top-K pages); the 8 warps' states of a piece are combined in shared
//       memory into one split-K partial, and the warp that completes a pair's last piece
//       hands its merge to the selector team.
//   selector team (0..3)   runs the jobs handed to it: the exact top-K of a pair's keys
//       (Solution step 3; ties to the lower page), published with the physical page of
//       every kept page, or the log-sum-exp merge of a pair's partials into the output.
//
// Work is split in global order over all CTAs (piece q goes to CTA q mod gridDim), pairs
// in order, so the GPU scores pair 0 first and pair 31 last: pairs complete, and are
// selected, one after another while the boxes of later pairs still stream, and the
// decode pieces (taken in the same pair order) find their selection published.  Every
// CTA must be resident at once (cooperative launch); every wait is bounded.
#include <mutex>

#include "quest_device.cuh"

namespace quest {

namespace {

constexpr int kSelWarps = 4;                       // selector team: warps 0..3
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSWarps = kConsumerWarps;            // consumers: warps 4..11
constexpr int kPiecePages = kStreamPiecePages;     // kept pages per decode piece
static_assert(kPiecePages == kSWarps, "page i of a decode piece goes to consumer i");
constexpr int kProducerWarp = kSelWarps + kSWarps;  // warp 12
constexpr int kStreamThreads = (kProducerWarp + 1) * 32;
constexpr int kJobs = 64;                          // job queue of the selector team
constexpr int kStreamMaxBatch = 1024;              // sequences whose lengths are kept on chip
constexpr int kStreamMaxTopk = 2048;               // kept pages per pair (256 decode pieces)
constexpr int kStreamTrace = 64;                   // timeline records per CTA

enum : int { kStEmpty = 0, kStScore = 1, kStDecode = 2 };
enum : int { kJobSelect = 1, kJobMerge = 2 };
// control words in shared memory
enum : int { kCtlComb = 0, kCtlFree = 2, kCtlTail = 4, kCtlDone = 5, kCtlWords = 8 };

enum StreamTraceEvent : int {
  kSeStart = 1, kSeExit = 2, kSeFirstScore = 3, kSeLastScore = 4, kSeFirstDecode = 5,
  kSeLastDecode = 6, kSeSelBegin = 7, kSeSelEnd = 8, kSeMergeBegin = 9, kSeMergeEnd = 10,
  kSeIssueDecode = 11, kSeIssueLast = 12,
};

struct SInfo {
  int kind;  // kStEmpty / kStScore / kStDecode
  int j;     // pair
  int a;     // scoring: first page; decode: piece of the pair
  int n;     // scoring: boxes; decode: valid tokens of the page (0: nothing staged)
};

struct SSmem {
  unsigned char* ring;  // [S][slot]: data (P boxes, or a page's K then V chunk), then q
  uint64_t* full;       // [S]
  uint64_t* empty;      // [S]
  SInfo* info;          // [S]
  float* wsc;           // [kSWarps][G * P] logits, then weights, of the page in hand
  float* st;            // [kSWarps][G * 3] running max (log2 units), sum, rescale
  float* cbuf;          // [2][kSWarps][G * (2 + 128)]: per warp m[G], l[G], acc[G][128]
  int* ctl;             // [kCtlWords]
  int* jobs;            // [kJobs]
  int* lens;            // [B] tokens of each sequence in this step (after its append)
  int* sb;              // [B + 1] scoring pieces before sequence b (all its kv heads)
  int* db;              // [B + 1] decode pieces before sequence b
  uint32_t* keys;       // [keys_stride(max_pages)] selector: the pair's keys
  int* hist;            // [2 * kTopkBins]
  uint32_t* kept;       // [2 * ceil(max_pages / 32)]
  int* scratch;         // [256]
  int* sel;             // [kcap] kept pages, ascending
  float* msc;           // [G][npc_max + 2] merge: scale of each partial, max, sum
};

__host__ __device__ inline int s_keys_stride(int max_pages) { return (max_pages + 3) & ~3; }

__host__ __device__ inline size_t s_slot_bytes(int G, int P) {
  return align_up((size_t)2 * P * kHeadDim * 2 + (size_t)G * kHeadDim * 2, 128);
}

// Everything but the ring, then as many ring slots as fit in `budget` bytes (0 if fewer
// than kSWarps fit).  Writes the layout into s when given.
__host__ __device__ inline size_t stream_smem_layout(int G, int P, int max_pages, int top_k,
                                                     int batch, size_t budget, int* slots,
                                                     SSmem* s, unsigned char* base) {
  const int kcap = top_k < max_pages ? top_k : max_pages;
  const int npc = (kcap + kPiecePages - 1) / kPiecePages;
  size_t o = 0;
  const size_t wsc = o;      o = align_up(o + (size_t)kSWarps * G * P * 4, 16);
  const size_t st = o;       o = align_up(o + (size_t)kSWarps * G * 3 * 4, 16);
  const size_t cbuf = o;     o = align_up(o + (size_t)2 * kSWarps * G * (2 + kHeadDim) * 4, 16);
  const size_t ctl = o;      o = align_up(o + kCtlWords * 4, 16);
  const size_t jobs = o;     o = align_up(o + kJobs * 4, 16);
  const size_t lens = o;     o = align_up(o + (size_t)batch * 4, 16);
  const size_t sb = o;       o = align_up(o + (size_t)(batch + 1) * 4, 16);
  const size_t db = o;       o = align_up(o + (size_t)(batch + 1) * 4, 16);
  const size_t keys = o;     o = align_up(o + (size_t)s_keys_stride(max_pages) * 4, 16);
  const size_t hist = o;     o = align_up(o + (size_t)2 * kTopkBins * 4, 16);
  const size_t kept = o;     o = align_up(o + (size_t)2 * ((max_pages + 31) / 32) * 4, 16);
  const size_t scr = o;      o = align_up(o + 256 * 4, 16);
  const size_t sel = o;      o = align_up(o + (size_t)kcap * 4, 16);
  const size_t msc = o;      o = align_up(o + (size_t)G * (npc + 2) * 4, 128);
  const size_t fixed = o;
  const size_t per_slot = s_slot_bytes(G, P) + 2 * 8 + sizeof(SInfo);
  // a multiple of kSWarps: stage s sits in slot s mod S and belongs to consumer s mod 8, so
  // every slot keeps one consumer, which waits on its phases in order (a parity wait that
  // ran two phases ahead of the slot would be satisfied by the wrong phase)
  int S = 0;
  if (budget > fixed + 256) S = (int)((budget - fixed - 256) / per_slot);
  if (S > 64) S = 64;
  S -= S % kSWarps;
  if (slots) *slots = S;
  const size_t ring = align_up(fixed, 128);
  size_t e = ring + (size_t)S * s_slot_bytes(G, P);
  const size_t full = e;     e += (size_t)S * 8;
  const size_t empty = e;    e += (size_t)S * 8;
  const size_t infoo = e;    e = align_up(e + (size_t)S * sizeof(SInfo), 16);
  if (s) {
    s->ring = base + ring;
    s->full = reinterpret_cast<uint64_t*>(base + full);
    s->empty = reinterpret_cast<uint64_t*>(base + empty);
    s->info = reinterpret_cast<SInfo*>(base + infoo);
    s->wsc = reinterpret_cast<float*>(base + wsc);
    s->st = reinterpret_cast<float*>(base + st);
    s->cbuf = reinterpret_cast<float*>(base + cbuf);
    s->ctl = reinterpret_cast<int*>(base + ctl);
    s->jobs = reinterpret_cast<int*>(base + jobs);
    s->lens = reinterpret_cast<int*>(base + lens);
    s->sb = reinterpret_cast<int*>(base + sb);
    s->db = reinterpret_cast<int*>(base + db);
    s->keys = reinterpret_cast<uint32_t*>(base + keys);
    s->hist = reinterpret_cast<int*>(base + hist);
    s->kept = reinterpret_cast<uint32_t*>(base + kept);
    s->scratch = reinterpret_cast<int*>(base + scr);
    s->sel = reinterpret_cast<int*>(base + sel);
    s->msc = reinterpret_cast<float*>(base + msc);
  }
  return e;
}

// ---------------------------------------------------------------- geometry of one call
struct PairGeo {
  int b, g, L, N, K;
  int npc;  // scoring pieces (ceil(N / P))
  int ndc;  // decode pieces (ceil(K / 8))
};

__device__ __forceinline__ PairGeo pair_geo(const Params& p, const SSmem& s, int j) {
  PairGeo q;
  q.b = j / p.Hkv;
  q.g = j - q.b * p.Hkv;
  q.L = s.lens[q.b];
  q.N = (q.L + p.P - 1) / p.P;
  q.K = min(p.top_k, q.N);
  q.npc = (q.N + p.P - 1) / p.P;  // a scoring piece holds the boxes of P pages
  q.ndc = (q.K + kPiecePages - 1) / kPiecePages;
  return q;
}

// Largest b with pre[b] <= r (pre: B + 1 non-decreasing entries, pre[0] = 0 <= r <
// pre[B]): the sequence that holds global piece r.
__device__ __forceinline__ int seq_of_piece(const int* pre, int B, int r) {
  int lo = 0, hi = B;  // pre[lo] <= r < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// Global piece r -> pair j and the piece's index within the pair; per sequence b the
// pieces are [pre[b], pre[b+1]), kv head after kv head.
__device__ __forceinline__ void piece_of(const Params& p, const int* pre, int r, int* j, int* u) {
  const int b = seq_of_piece(pre, p.B, r);
  const int per_head = (pre[b + 1] - pre[b]) / p.Hkv;
  const int off = r - pre[b];
  const int g = off / per_head;
  *u = off - g * per_head;
  *j = b * p.Hkv + g;
}

__device__ __forceinline__ void strace(const Params& p, int* slot, int ev, int item) {
  if (p.trace == nullptr || *slot >= kStreamTrace) return;
  const long long i = (long long)blockIdx.x * kStreamTrace + (*slot)++;
  if (i >= p.trace_capacity) return;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  p.trace[1 + 2 * i] = (unsigned long long)global_ns();
  p.trace[2 + 2 * i] = ((unsigned long long)smid << 48) |
                       ((unsigned long long)(blockIdx.x & 0xffff) << 32) |
                       ((unsigned long long)(ev & 0xff) << 24) | (unsigned)(item & 0xffffff);
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ int ld_volatile_s32(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

// Hand a job to this CTA's selector team (one lane).
__device__ void push_job(const Params& p, const SSmem& s, int kind, int j) {
  const int slot = atomicAdd(&s.ctl[kCtlTail], 1) % kJobs;
  // the slot's previous job (kJobs pushes ago) must have been taken
  if (ld_volatile_s32(&s.jobs[slot]) != 0) {
    const long long t0 = global_ns();
    while (ld_volatile_s32(&s.jobs[slot]) != 0) {
      __nanosleep(64);
      if (global_ns() - t0 > p.wait_limit_ns) {
        report(p, QUEST_ERR_TIMEOUT, -1, j, kSiteWaitSlot);
        return;
      }
    }
  }
  __threadfence_block();
  atomicExch(&s.jobs[slot], (kind << 28) | (j + 1));
}

// ---------------------------------------------------------------- producer warp
template <int G, int P>
__device__ void s_produce(const Params& p, const LayerPtrs& lay, const SSmem& s, int S,
                          int TS, int TD, int nS_pad) {
  constexpr uint32_t kChunk = (uint32_t)P * kHeadDim * 2;  // one page of K (or V), one kv head
  constexpr uint32_t kBox = 2 * kHeadDim * 2;              // one page's box (min, max)
  constexpr uint32_t kQ = (uint32_t)G * kHeadDim * 2;
  const size_t slot_bytes = s_slot_bytes(G, P);
  const int lane = threadIdx.x & 31;
  const int C = (int)gridDim.x, c = (int)blockIdx.x;
  int tslot = kStreamTrace / 2;
  uint32_t stage = 0;
  auto slot_free = [&](uint32_t st_idx) -> bool {
    const int sl = (int)(st_idx % (uint32_t)S);
    return mbar_wait_bounded(p, &s.empty[sl], ((st_idx / (uint32_t)S) & 1u) ^ 1u, kSiteWaitSlot);
  };
  // ---- scoring pieces: the boxes of up to P pages of one pair (P boxes fill one stage)
  if (lane == 0) {
    for (int r = c; r < TS; r += C, ++stage) {
      int j, u;
      piece_of(p, s.sb, r, &j, &u);
      const PairGeo q = pair_geo(p, s, j);
      const int p0 = u * P;
      const int n = min(P, q.N - p0);
      const int sl = (int)(stage % (uint32_t)S);
      const bool ok = slot_free(stage);
      s.info[sl] = SInfo{kStScore, j, p0, ok ? n : 0};
      if (ok) {
        unsigned char* dst = s.ring + (size_t)sl * slot_bytes;
        mbar_arrive_expect_tx(&s.full[sl], (uint32_t)n * kBox + kQ);
        bulk_g2s(dst, lay.meta + box_offset(p, q.b, q.g, p0), (uint32_t)n * kBox, &s.full[sl]);
        bulk_g2s(dst + 2 * kChunk, lay.q + ((size_t)q.b * p.Hq + (size_t)q.g * G) * kHeadDim, kQ,
                 &s.full[sl]);
      } else {
        mbar_arrive(&s.full[sl]);
      }
    }
    for (; stage < (uint32_t)nS_pad; ++stage) {  // round up to whole rounds of kSWarps
      const int sl = (int)(stage % (uint32_t)S);
      const bool ok = slot_free(stage);
      s.info[sl] = SInfo{kStEmpty, 0, 0, 0};
      (void)ok;
      mbar_arrive(&s.full[sl]);
    }
    if (TS > c) strace(p, &tslot, kSeIssueLast, 0);
  }
  stage = __shfl_sync(0xffffffffu, stage, 0);
  // ---- decode pieces: up to 8 kept pages of one pair, page i to consumer i
  bool first = true;
  for (int r = c; r < TD; r += C) {
    int j, v;
    piece_of(p, s.db, r, &j, &v);
    const PairGeo q = pair_geo(p, s, j);
    const int n = min(kPiecePages, q.K - v * kPiecePages);
    bool ok = true;
    if (lane == 0) ok = wait_flag_bounded(p, p.ready + j, 1u, q.b, kSiteWaitSelection);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) (void)ld_acquire_u32(p.ready + j);  // every lane acquires the selection
    if (first && lane == 0) strace(p, &tslot, kSeIssueDecode, j);
    first = false;
    // the selection's kept pages (written with their physical page by the selector); the
    // appended token's row was written by a generic store: order it before the bulk copy
    fence_proxy_async_global();
    int nv = 0;
    const __half* ksrc = nullptr;
    const __half* vsrc = nullptr;
    if (ok && lane < n) {
      const int2 e = __ldcg(reinterpret_cast<const int2*>(p.sel_pair) +
                            (size_t)j * p.top_k + v * kPiecePages + lane);
      if (e.x >= 0 && e.x < q.N && e.y >= 0 && e.y < p.num_phys) {
        nv = min(P, q.L - e.x * P);
        const size_t off = ((size_t)e.y * p.Hkv + q.g) * (size_t)P * kHeadDim;
        ksrc = lay.k_pool + off;
        vsrc = lay.v_pool + off;
      }
    }
    for (int i = 0; i < kPiecePages; ++i) {
      if (lane == i) {
        const int sl = (int)(stage % (uint32_t)S);
        const bool fr = slot_free(stage);
        const int nvs = fr ? nv : 0;
        s.info[sl] = SInfo{kStDecode, j, v, nvs};
        if (nvs > 0) {
          unsigned char* dst = s.ring + (size_t)sl * slot_bytes;
          mbar_arrive_expect_tx(&s.full[sl], 2 * kChunk + kQ);
          bulk_g2s(dst, ksrc, kChunk, &s.full[sl]);
          bulk_g2s(dst + kChunk, vsrc, kChunk, &s.full[sl]);
          bulk_g2s(dst + 2 * kChunk, lay.q + ((size_t)q.b * p.Hq + (size_t)q.g * G) * kHeadDim,
                   kQ, &s.full[sl]);
        } else {
          mbar_arrive(&s.full[sl]);
        }
      }
      ++stage;
      __syncwarp();
    }
  }
  if (TD > c && lane == 0) strace(p, &tslot, kSeIssueLast, 1);
}

// ---------------------------------------------------------------- consumer warps
// Bound of every page of a scoring stage (half-warp per page); the keys go to global
// memory.  The page of the step's new token first takes the token: its box opens or widens
// in registers, is scored, and is written back with the token's K and V rows.
template <int G, int P>
__device__ void s_score_stage(const Params& p, const LayerPtrs& lay, const SSmem& s,
                              const unsigned char* slot, const SInfo& in, const PairGeo& q) {
  const int lane = threadIdx.x & 31;
  const int hw = lane >> 4, c = lane & 15;
  QueryFrag<G> f;
  load_query_frag<G>(reinterpret_cast<const __half*>(slot + 2 * (size_t)P * kHeadDim * 2), 0, 0,
                     0, c, f);
  // the appended token (tokens L-1 of a step that appends)
  const bool appends = lay.k_new != nullptr && p.chain_append;  // set per call on the host
  const int ap = appends && q.L > 0 ? (q.L - 1) / P : -1;
  const bool mine = ap >= in.a && ap < in.a + in.n;
  uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
  int aphys = -1;
  if (mine) {
    const size_t o = ((size_t)q.b * p.Hkv + q.g) * kHeadDim + 8 * c;
    knew = *reinterpret_cast<const uint4*>(lay.k_new + o);
    vnew = *reinterpret_cast<const uint4*>(lay.v_new + o);
    const int ph = p.block_table[(size_t)q.b * p.max_pages + ap];
    aphys = (ph >= 0 && ph < p.num_phys) ? ph : -1;
  }
  uint32_t* krow = reinterpret_cast<uint32_t*>(p.scores) + (size_t)(q.b * p.Hkv + q.g) * p.max_pages;
  const bool windowed = q.N > q.K && (p.sink_pages > 0 || p.local_pages > 0);
  for (int r0 = 0; r0 < in.n; r0 += 2) {
    const int r = r0 + hw;
    const int page = in.a + r;
    uint4 mn = make_uint4(0, 0, 0, 0), mx = make_uint4(0, 0, 0, 0);
    if (r < in.n) {
      const unsigned char* rec = slot + (size_t)r * 2 * kHeadDim * 2;
      mn = *reinterpret_cast<const uint4*>(rec + 16 * c);
      mx = *reinterpret_cast<const uint4*>(rec + 2 * kHeadDim + 16 * c);
    }
    if (mine && r < in.n && page == ap) {
      if (aphys >= 0) {
        const int slot_a = (q.L - 1) % P;
        if (slot_a == 0) {
          mn = knew;
          mx = knew;
        } else {
          const uint32_t a[4] = {mn.x, mn.y, mn.z, mn.w};
          const uint32_t z[4] = {mx.x, mx.y, mx.z, mx.w};
          const uint32_t nw[4] = {knew.x, knew.y, knew.z, knew.w};
          uint32_t ra[4], rz[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const __half2 hn = *reinterpret_cast<const __half2*>(&nw[w]);
            const __half2 l2 = __hmin2(*reinterpret_cast<const __half2*>(&a[w]), hn);
            const __half2 h2 = __hmax2(*reinterpret_cast<const __half2*>(&z[w]), hn);
            ra[w] = *reinterpret_cast<const uint32_t*>(&l2);
            rz[w] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          mn = make_uint4(ra[0], ra[1], ra[2], ra[3]);
          mx = make_uint4(rz[0], rz[1], rz[2], rz[3]);
        }
        __half* box = lay.meta + box_offset(p, q.b, q.g, page);
        *reinterpret_cast<uint4*>(box + 8 * c) = mn;
        *reinterpret_cast<uint4*>(box + kHeadDim + 8 * c) = mx;
        const size_t kv = (((size_t)aphys * p.Hkv + q.g) * P + slot_a) * kHeadDim + 8 * c;
        *reinterpret_cast<uint4*>(lay.k_pool + kv) = knew;
        *reinterpret_cast<uint4*>(lay.v_pool + kv) = vnew;
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
    if (c == 0 && r < in.n) {
      // pages of the sink / local window of a long sequence get the largest key
      const bool forced = windowed && (page < p.sink_pages || page >= q.N - p.local_pages);
      __stcg(krow + page, forced ? 0xffffffffu : score_key(best));
    }
  }
  if (mine) fence_proxy_async_global();  // the appended row, before the pair is released
}

// Flash-decode of the one kept page of a decode stage; this warp's state of the piece goes
// to the piece's combine buffer.  Returns with the slot released.
template <int G, int P>
__device__ void s_decode_stage(const Params& p, const SSmem& s, const unsigned char* slot,
                               const SInfo& in, int w, uint64_t* empty_bar, float* cb,
                               const int* free_word, int k) {
  const int lane = threadIdx.x & 31;
  float* sc = s.wsc + w * G * P;
  float* st = s.st + w * G * 3;
  float acc[G][4];
#pragma unroll
  for (int jh = 0; jh < G; ++jh)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[jh][k] = 0.f;
  if (lane < G) {
    st[lane * 3 + 0] = -CUDART_INF_F;
    st[lane * 3 + 1] = 0.f;
    st[lane * 3 + 2] = 1.f;
  }
  __syncwarp();
  if (in.n > 0) {
    const __half* Ks = reinterpret_cast<const __half*>(slot);
    const __half* qs = Ks + 2 * P * kHeadDim;
    float qf[G][4];
#pragma unroll
    for (int jh = 0; jh < G; ++jh) {
      const uint2 raw = lds_u2(qs + jh * kHeadDim + 4 * lane);
      const float2 a = h2f(raw.x), cc = h2f(raw.y);
      qf[jh][0] = a.x * p.qscale;
      qf[jh][1] = a.y * p.qscale;
      qf[jh][2] = cc.x * p.qscale;
      qf[jh][3] = cc.y * p.qscale;
    }
    page_update<G, P>(qf, acc, Ks, Ks + P * kHeadDim, in.n, sc, st, lane);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(empty_bar);
  // the combine buffer of this piece's parity must be done with piece k - 2
  if (ld_volatile_s32(free_word) != k) {
    const long long t0 = global_ns();
    while (ld_volatile_s32(free_word) != k) {
      __nanosleep(32);
      if (global_ns() - t0 > p.wait_limit_ns) {
        if (lane == 0) report(p, QUEST_ERR_TIMEOUT, -1, k, kSiteWaitSlot);
        break;
      }
    }
  }
  // this warp's state: m[G], l[G], acc[G][128]
  if (lane < G) {
    cb[lane] = st[lane * 3 + 0];
    cb[G + lane] = st[lane * 3 + 1];
  }
#pragma unroll
  for (int jh = 0; jh < G; ++jh)
    *reinterpret_cast<float4*>(cb + 2 * G + jh * kHeadDim + 4 * lane) =
        make_float4(acc[jh][0], acc[jh][1], acc[jh][2], acc[jh][3]);
}

// Combine the 8 warps' states of a piece into its split-K partial (one warp).
template <int G>
__device__ void s_combine(const Params& p, const float* cbase, const PairGeo& q, int v) {
  const int lane = threadIdx.x & 31;
  constexpr int WF = 2 * G + G * kHeadDim;  // floats per warp state
#pragma unroll
  for (int jh = 0; jh < G; ++jh) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) M = fmaxf(M, cbase[w * WF + jh]);
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) {
      const float m = cbase[w * WF + jh];
      const float f = (m == -CUDART_INF_F) ? 0.f : exp2f(m - M);
      const float4 a = *reinterpret_cast<const float4*>(cbase + w * WF + 2 * G + jh * kHeadDim + 4 * lane);
      A.x = fmaf(a.x, f, A.x);
      A.y = fmaf(a.y, f, A.y);
      A.z = fmaf(a.z, f, A.z);
      A.w = fmaf(a.w, f, A.w);
      Ls = fmaf(cbase[w * WF + G + jh], f, Ls);
    }
    const size_t slotp = ((size_t)q.b * p.Hq + (size_t)q.g * G + jh) * p.n_splits + v;
    *reinterpret_cast<float4*>(p.part_acc + slotp * kHeadDim + 4 * lane) = A;
    if (lane == 0) {
      p.part_ml[slotp * 2] = M;
      p.part_ml[slotp * 2 + 1] = Ls;
    }
  }
}

template <int G, int P>
__device__ void s_consume(const Params& p, const LayerPtrs& lay, const SSmem& s, int S,
                          int total_stages, int nS_pad) {
  const int lane = threadIdx.x & 31;
  const int w = (threadIdx.x >> 5) - kSelWarps;
  const size_t slot_bytes = s_slot_bytes(G, P);
  constexpr int WF = 2 * G + G * kHeadDim;
  int tslot = 1 + 2 * w;
  bool first_score = true, first_decode = true;
  for (int stg = w; stg < total_stages; stg += kSWarps) {
    const int sl = stg % S;
    const bool ok = mbar_wait_bounded(p, &s.full[sl], (uint32_t)(stg / S) & 1u, kSiteWaitStage);
    SInfo in = s.info[sl];
    if (!ok) in.n = 0;
    const unsigned char* slot = s.ring + (size_t)sl * slot_bytes;
    if (in.kind == kStScore) {
      if (first_score && lane == 0 && w == 0) strace(p, &tslot, kSeFirstScore, in.j);
      first_score = false;
      const PairGeo q = pair_geo(p, s, in.j);
      if (in.n > 0) s_score_stage<G, P>(p, lay, s, slot, in, q);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s.empty[sl]);
        // the piece is counted on the pair; the warp that completes the pair selects it
        const unsigned old = atom_add_acq_rel(p.score_arrive + in.j, 1u);
        if (old + 1u == (unsigned)q.npc) push_job(p, s, kJobSelect, in.j);
      }
    } else if (in.kind == kStDecode) {
      if (first_decode && lane == 0 && w == 0) strace(p, &tslot, kSeFirstDecode, in.j);
      first_decode = false;
      const int k = (stg - nS_pad) / kSWarps;  // this CTA's decode piece
      const int par = k & 1;
      float* cbase = s.cbuf + (size_t)par * kSWarps * WF;
      s_decode_stage<G, P>(p, s, slot, in, w, &s.empty[sl], cbase + w * WF,
                           &s.ctl[kCtlFree + par], k);
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        __threadfence_block();
        last = atomicAdd(&s.ctl[kCtlComb + par], 1) == kSWarps - 1;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last) {
        __threadfence_block();
        const PairGeo q = pair_geo(p, s, in.j);
        s_combine<G>(p, cbase, q, in.a);
        __syncwarp();
        if (lane == 0) {
          s.ctl[kCtlComb + par] = 0;
          __threadfence_block();
          atomicExch(&s.ctl[kCtlFree + par], k + 2);
          const unsigned old = atom_add_acq_rel(p.decode_arrive + in.j, 1u);
          if (old + 1u == (unsigned)q.ndc) push_job(p, s, kJobMerge, in.j);
        }
      }
      if (lane == 0 && stg + kSWarps >= total_stages && w == 0)
        strace(p, &tslot, kSeLastDecode, in.j);
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[sl]);
    }
  }
  __syncwarp();
  if (lane == 0) {
    __threadfence_block();
    atomicAdd(&s.ctl[kCtlDone], 1);
  }
}

// ---------------------------------------------------------------- selector team
// Exact top-K of pair j's keys; the kept pages (ascending) go out with their physical
// pages, then the pair is released to the decode pieces.
__device__ void s_select(const Params& p, const SSmem& s, const PairGeo& q, int j) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* sel = s.sel;
  int* cnt_slot = s.scratch + 200;
  if (q.N <= q.K) {
    for (int r = tid; r < q.K; r += kSelThreads) sel[r] = r;
  } else {
    const uint32_t* krow = reinterpret_cast<const uint32_t*>(p.scores) + (size_t)j * p.max_pages;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int i0 = 0; i0 < q.N; i0 += 16 * kSelThreads) {
      uint32_t v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        v[u] = i < q.N ? __ldcg(krow + i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        if (i < q.N) {
          s.keys[i] = v[u];
          lo = min(lo, v[u]);
          hi = max(hi, v[u]);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      s.scratch[100 + warp] = (int)lo;
      s.scratch[110 + warp] = (int)hi;
    }
    bsync<kSelThreads, true>();
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      lo = min(lo, (uint32_t)s.scratch[100 + w]);
      hi = max(hi, (uint32_t)s.scratch[110 + w]);
    }
    topk_keys<kSelThreads, true>(s.keys, q.N, q.K, lo, hi, sel, cnt_slot, s.hist, s.kept,
                                 s.scratch);
  }
  bsync<kSelThreads, true>();
  // kept pages with their physical page, for the decode producers; the caller's copy
  int2* out = reinterpret_cast<int2*>(p.sel_pair) + (size_t)j * p.top_k;
  int* idx_row = p.sel_idx ? p.sel_idx + (size_t)j * p.top_k : nullptr;
  for (int r = tid; r < q.K; r += kSelThreads) {
    const int lp = sel[r];
    int phys = p.block_table[(size_t)q.b * p.max_pages + lp];
    if (phys < 0 || phys >= p.num_phys) {
      report(p, QUEST_ERR_BAD_PAGE, q.b, lp, kSiteDecode);
      phys = -1;
    }
    __stcg(out + r, make_int2(lp, phys));
    if (idx_row) idx_row[r] = lp;
  }
  if (idx_row)
    for (int r = q.K + tid; r < p.top_k; r += kSelThreads) idx_row[r] = -1;
  if (tid == 0 && p.sel_count) p.sel_count[j] = q.K;
  __threadfence();
  bsync<kSelThreads, true>();
  if (tid == 0) {
    p.score_arrive[j] = 0u;  // every piece of the pair has arrived: ready for the next call
    if (!(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION)) st_release_u32(p.ready + j, 1u);
  }
}

// Log-sum-exp merge of pair j's piece partials into out / lse.
template <int G>
__device__ void s_merge(const Params& p, const LayerPtrs& lay, const SSmem& s, const PairGeo& q,
                        int j) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = q.ndc;
  const int stride = n + 2;
  float* msc = s.msc;  // [G][n + 2]: m of each piece, then scale; M; sum
  const size_t h0 = (size_t)q.b * p.Hq + (size_t)q.g * G;
  for (int jh = warp; jh < G; jh += kSelWarps) {
    const float* ml = p.part_ml + (h0 + jh) * p.n_splits * 2;
    float M = -CUDART_INF_F;
    for (int v = lane; v < n; v += 32) M = fmaxf(M, __ldcg(ml + 2 * v));
    M = warp_max(M);
    float Ls = 0.f;
    for (int v = lane; v < n; v += 32) {
      const float m = __ldcg(ml + 2 * v);
      const float f = (m == -CUDART_INF_F) ? 0.f : exp2f(m - M);
      msc[jh * stride + v] = f;
      Ls = fmaf(__ldcg(ml + 2 * v + 1), f, Ls);
    }
    Ls = warp_sum(Ls);
    if (lane == 0) {
      msc[jh * stride + n] = M;
      msc[jh * stride + n + 1] = Ls;
    }
  }
  bsync<kSelThreads, true>();
  for (int o = tid; o < G * kHeadDim; o += kSelThreads) {
    const int jh = o / kHeadDim, i = o - jh * kHeadDim;
    const float* row = msc + jh * stride;
    const float* accp = p.part_acc + (h0 + jh) * p.n_splits * kHeadDim + i;
    float A0 = 0.f, A1 = 0.f, A2 = 0.f, A3 = 0.f;
    int v = 0;
    for (; v + 4 <= n; v += 4) {
      const float a0 = __ldcg(accp + (size_t)v * kHeadDim);
      const float a1 = __ldcg(accp + (size_t)(v + 1) * kHeadDim);
      const float a2 = __ldcg(accp + (size_t)(v + 2) * kHeadDim);
      const float a3 = __ldcg(accp + (size_t)(v + 3) * kHeadDim);
      A0 = fmaf(a0, row[v], A0);
      A1 = fmaf(a1, row[v + 1], A1);
      A2 = fmaf(a2, row[v + 2], A2);
      A3 = fmaf(a3, row[v + 3], A3);
    }
    for (; v < n; ++v) A0 = fmaf(__ldcg(accp + (size_t)v * kHeadDim), row[v], A0);
    const float A = (A0 + A1) + (A2 + A3);
    const float Ls = row[n + 1];
    const size_t h = h0 + jh;
    lay.out[h * kHeadDim + i] = __float2half_rn(Ls > 0.f ? A / Ls : 0.f);
    if (i == 0 && lay.lse)
      lay.lse[h] = Ls > 0.f ? (row[n] + log2f(Ls)) * 0.69314718055994531f : -CUDART_INF_F;
  }
  bsync<kSelThreads, true>();
  if (tid == 0) {
    p.decode_arrive[j] = 0u;  // the next call starts from zero
    p.ready[j] = 0u;
  }
}

// A pair with no token: out = 0, lse = -inf, nothing kept.
template <int G>
__device__ void s_empty_pair(const Params& p, const LayerPtrs& lay, const PairGeo& q, int j) {
  const int tid = threadIdx.x;
  const size_t h0 = (size_t)q.b * p.Hq + (size_t)q.g * G;
  for (int o = tid; o < G * kHeadDim; o += kSelThreads) lay.out[h0 * kHeadDim + o] = __float2half_rn(0.f);
  if (tid < G && lay.lse) lay.lse[h0 + tid] = -CUDART_INF_F;
  if (p.sel_idx)
    for (int r = tid; r < p.top_k; r += kSelThreads) p.sel_idx[(size_t)j * p.top_k + r] = -1;
  if (tid == 0 && p.sel_count) p.sel_count[j] = 0;
}

template <int G>
__device__ void s_selector(const Params& p, const LayerPtrs& lay, const SSmem& s, int NP) {
  const int tid = threadIdx.x;
  int tslot = kStreamTrace / 2 + 8;
  // pairs without a token are finished here
  for (int j = (int)blockIdx.x; j < NP; j += (int)gridDim.x) {
    const PairGeo q = pair_geo(p, s, j);
    if (q.N == 0) s_empty_pair<G>(p, lay, q, j);
  }
  int* bc = s.scratch + 240;  // broadcast of the job
  for (int head = 0;; ++head) {
    const int sl = head % kJobs;
    if (tid == 0) {
      int job = ld_volatile_s32(&s.jobs[sl]);
      const long long t0 = global_ns();
      while (job == 0) {
        if (ld_volatile_s32(&s.ctl[kCtlDone]) == kSWarps) {
          job = ld_volatile_s32(&s.jobs[sl]);  // a job pushed before the last warp finished
          if (job == 0) job = -1;
          break;
        }
        __nanosleep(64);
        job = ld_volatile_s32(&s.jobs[sl]);
        if (global_ns() - t0 > 4 * p.wait_limit_ns) {
          report(p, QUEST_ERR_TIMEOUT, -1, -1, kSiteWaitSelection);
          job = -1;
          break;
        }
      }
      if (job > 0) {
        s.jobs[sl] = 0;
        __threadfence();  // acquire side of the pair's completion, for the whole team
      }
      *bc = job;
    }
    bsync<kSelThreads, true>();
    const int job = *bc;
    bsync<kSelThreads, true>();
    if (job < 0) break;
    const int kind = job >> 28, j = (job & 0x0fffffff) - 1;
    const PairGeo q = pair_geo(p, s, j);
    if (kind == kJobSelect) {
      if (tid == 0) strace(p, &tslot, kSeSelBegin, j);
      s_select(p, s, q, j);
      if (tid == 0) strace(p, &tslot, kSeSelEnd, j);
    } else {
      if (tid == 0) strace(p, &tslot, kSeMergeBegin, j);
      s_merge<G>(p, lay, s, q, j);
      if (tid == 0) strace(p, &tslot, kSeMergeEnd, j);
    }
    bsync<kSelThreads, true>();
  }
}

}  // namespace

// One CTA per SM, all resident (cooperative launch).  Single layer: `lay` holds the pools,
// boxes, query, new token and outputs.
template <int G, int P>
__global__ void __launch_bounds__(kStreamThreads, 1)
    stream_kernel(Params p, const __grid_constant__ LayerPtrs lay) {
  extern __shared__ __align__(128) unsigned char smem[];
  SSmem s;
  int S = 0;  // ring slots: the host launched with the same layout
  stream_smem_layout(G, P, p.max_pages, p.top_k, p.B, kMaxSmem, &S, &s, smem);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    fence_mbar_init();
  }
  if (tid < kCtlWords) s.ctl[tid] = (tid == kCtlFree + 1) ? 1 : 0;
  if (tid < kJobs) s.jobs[tid] = 0;
  for (int i = tid; i < 2 * kTopkBins; i += blockDim.x) s.hist[i] = 0;
  pdl_wait();
  // this step's length of every sequence (the new token counts when there is room)
  const long long cap = (long long)p.max_pages * p.P;
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int L0 = p.seq_lens[b];
    int L = L0;
    if (L0 < 0 || (long long)L0 > cap) {
      if (blockIdx.x == 0) report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteScore);
      L = 0;
    } else if (p.chain_append) {
      if ((long long)L0 + 1 <= cap) {
        L = L0 + 1;
      } else if (blockIdx.x == 0) {
        report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);  // no room for the new token
      }
    }
    s.lens[b] = L;
  }
  __syncthreads();
  if (p.chain_append && !p.hold_lengths && tid == 0) red_add_release(p.started, 1u);
  // piece prefixes over the sequences (warp 0, 32 sequences at a time)
  if (tid < 32) {
    int sb = 0, db = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int b = b0 + tid;
      int ns = 0, nd = 0;
      if (b < p.B) {
        const int N = (s.lens[b] + p.P - 1) / p.P;
        const int K = min(p.top_k, N);
        ns = (N + p.P - 1) / p.P * p.Hkv;
        nd = (K + kPiecePages - 1) / kPiecePages * p.Hkv;
      }
      int is = ns, id = nd;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, is, o);
        const int d = __shfl_up_sync(0xffffffffu, id, o);
        if (tid >= o) {
          is += a;
          id += d;
        }
      }
      if (b < p.B) {
        s.sb[b] = sb + is - ns;
        s.db[b] = db + id - nd;
      }
      sb += __shfl_sync(0xffffffffu, is, 31);
      db += __shfl_sync(0xffffffffu, id, 31);
    }
    if (tid == 0) {
      s.sb[p.B] = sb;
      s.db[p.B] = db;
    }
  }
  __syncthreads();
  const int TS = s.sb[p.B], TD = s.db[p.B];
  const int C = (int)gridDim.x, c = (int)blockIdx.x;
  const int nS = c < TS ? (TS - 1 - c) / C + 1 : 0;
  const int nD = c < TD ? (TD - 1 - c) / C + 1 : 0;
  const int nS_pad = (nS + kSWarps - 1) / kSWarps * kSWarps;
  const int total = nS_pad + nD * kSWarps;
  if (tid == 0) {
    int t0 = 0;
    strace(p, &t0, kSeStart, TS);
  }
  const int warp = tid >> 5;
  if (warp == kProducerWarp) {
    s_produce<G, P>(p, lay, s, S, TS, TD, nS_pad);
  } else if (warp >= kSelWarps) {
    s_consume<G, P>(p, lay, s, S, total, nS_pad);
  } else {
    s_selector<G>(p, lay, s, p.B * p.Hkv);
  }
  __syncthreads();
  // a wait that gave up may leave copies in flight: let them land before the CTA leaves
  if (tid == kProducerWarp * 32 && ld_relaxed_s32(p.status) != QUEST_OK) {
    const int last = total;
    for (int st = max(0, last - S); st < last; ++st)
      mbar_wait_bounded(p, &s.full[st % S], (uint32_t)(st / S) & 1u, kSiteWaitStage);
  }
  if (tid == 0) {
    int tl = kStreamTrace - 1;
    strace(p, &tl, kSeExit, 0);
  }
  // With an appended token, CTA 0 advances the lengths once every CTA has read them.
  if (p.chain_append && !p.hold_lengths && c == 0 && tid < 32) {
    bool ok = true;
    if (tid == 0) ok = wait_flag_bounded(p, p.started, (unsigned)C, -1, kSiteWaitSlot);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (ok) {
      for (int b = tid; b < p.B; b += 32) {
        const int L0 = p.seq_lens[b];
        if (L0 < 0 || (long long)L0 + 1 > cap) continue;  // reported at the start
        const int phys = p.block_table[(size_t)b * p.max_pages + L0 / p.P];
        if (phys >= 0 && phys < p.num_phys) p.seq_lens[b] = L0 + 1;
      }
    }
    __syncwarp();
    if (tid == 0) *p.started = 0u;
  }
}

template <int G, int P>
static const void* stream_fn() { return (const void*)stream_kernel<G, P>; }

static const void* pick_stream(int G, int P) {
  if (P == 16) {
    switch (G) {
      case 1: return stream_fn<1, 16>();
      case 2: return stream_fn<2, 16>();
      case 4: return stream_fn<4, 16>();
      default: return stream_fn<8, 16>();
    }
  }
  switch (G) {
    case 1: return stream_fn<1, 32>();
    case 2: return stream_fn<2, 32>();
    case 4: return stream_fn<4, 32>();
    default: return stream_fn<8, 32>();
  }
}

// Ring slots of the stream kernel for this shape (0: it does not fit).
int stream_slots(int G, int P, int max_pages, int top_k, int batch) {
  if (batch > kStreamMaxBatch || top_k > kStreamMaxTopk) return 0;
  int S = 0;
  stream_smem_layout(G, P, max_pages, top_k, batch, kMaxSmem, &S, nullptr, nullptr);
  return S;
}

namespace {

struct DevInfo {
  int sms = 0;
  bool coop = false;
};

cudaError_t device_info(DevInfo* out) {
  static std::mutex mu;
  static DevInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev & 63]) {
    DevInfo d;
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    int coop = 0;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess)
      return e;
    d.coop = coop != 0;
    cache[dev & 63] = d;
    have[dev & 63] = true;
  }
  *out = cache[dev & 63];
  return cudaSuccess;
}

}  // namespace

size_t stream_smem_bytes(int G, int P, int max_pages, int top_k, int batch) {
  return stream_smem_layout(G, P, max_pages, top_k, batch, kMaxSmem, nullptr, nullptr, nullptr);
}

// CTAs of a stream launch: one per SM, fewer for a small step (about 64 KB of stream per
// CTA at least), at most max_ctas when given.
cudaError_t stream_grid(const Params& p, int max_ctas, int* ctas) {
  DevInfo d;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return e;
  if (!d.coop) return cudaErrorNotSupported;
  const long long kcap = std::min<long long>(p.top_k, p.max_pages);
  const long long bytes = (long long)p.B * p.Hkv *
                          ((long long)p.max_pages * 2 * kHeadDim * 2 + kcap * p.P * kHeadDim * 4);
  long long n = (bytes + (64 << 10) - 1) / (64 << 10);
  if (n > d.sms) n = d.sms;
  if (n < 1) n = 1;
  if (max_ctas > 0 && n > max_ctas) n = max_ctas;
  *ctas = (int)n;
  return cudaSuccess;
}

cudaError_t launch_stream(const Params& p, const LayerPtrs& lay, int G, int max_ctas,
                          cudaStream_t s) {
  const int S = stream_slots(G, p.P, p.max_pages, p.top_k, p.B);
  if (S < kSWarps) return cudaErrorInvalidConfiguration;
  const size_t smem = stream_smem_layout(G, p.P, p.max_pages, p.top_k, p.B, kMaxSmem, nullptr,
                                         nullptr, nullptr);
  const void* fn = pick_stream(G, p.P);
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int ctas = 0;
  if ((e = stream_grid(p, max_ctas, &ctas)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)ctas);
  cfg.blockDim = dim3(kStreamThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  Params pp = p;
  LayerPtrs ll = lay;
  void* args[] = {&pp, &ll};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace quest
