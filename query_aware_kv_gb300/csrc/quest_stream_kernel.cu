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
//   producer warp (8)      walks this CTA's share of the work in a fixed order and
//       streams it into a shared-memory ring: first its scoring pieces (the boxes of up
//       to P pages of one pair, "Guide to Quest", Solution step 1, one 1-D bulk copy
//       (TMA) each), then its decode pieces (the K and V chunks of up to 8 kept pages of
//       one pair, once that pair's selection is published: scattered 4 KB chunks, copied
//       by the whole warp 16 bytes a lane with cp.async).
//   consumer warps (0..7)  stage s belongs to consumer s mod 8.  Scoring stage: the
//       bound of each page (Solution step 2) becomes an order-preserving key in global
//       memory, and the piece is counted on its pair (a release reduction).  Decode
//       stage: flash-decode of one kept page (exact attention over the kept pages only:
//       "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference", Summary);
//       the 8 warps' states of a piece are combined in shared memory into
//       one split-K partial, which is counted on its pair.
//   selector CTAs          the last few CTAs of the grid stream nothing: each owns every
//       sel_ctas-th pair and, with 12 warps, takes the exact top-K of a pair's keys as
//       soon as they are all in (Solution step 3; ties to the lower page), publishes it
//       with the physical page of every kept page, and, once all of the pair's decode
//       pieces are in, merges their partials by log-sum-exp into the output.  Selection is
//       a chain of short dependent steps: on an SM of its own it is not slowed by the
//       streaming warps.
//
// Work is split in global order over the streaming CTAs (piece q goes to CTA q mod C), pairs
// in order, so the GPU scores pair 0 first and pair 31 last: pairs complete, and are
// selected, one after another while the boxes of later pairs still stream, and the
// decode pieces (taken in the same pair order) find their selection published.  Every
// CTA must be resident at once (cooperative launch); every wait is bounded.
#include <mutex>

#include "quest_device.cuh"

namespace quest {

namespace {

constexpr int kSelWarps = 12;                      // a selector CTA's team: warps 0..11
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSWarps = kConsumerWarps;            // a streaming CTA's consumers: warps 0..7
constexpr int kPiecePages = kStreamPiecePages;     // kept pages per decode piece
static_assert(kPiecePages == kSWarps, "page i of a decode piece goes to consumer i");
constexpr int kProducerWarp = kSWarps;             // warp 8
constexpr int kStreamThreads = (kSelWarps + 1) * 32;  // both roles launch 13 warps
constexpr int kStreamMaxBatch = 1024;              // sequences whose lengths are kept on chip
constexpr int kStreamMaxTopk = 2048;               // kept pages per pair (256 decode pieces)
constexpr int kStreamTrace = 256;                  // timeline records per CTA
// record slots of a CTA: 0 start; streaming CTA: consumer w [8 + 24w, 32 + 24w), producer
// [200, 255); selector CTA: [8, 255); 255 exit
constexpr int kTrProducer = 200, kTrSelector = 8, kTrLast = kStreamTrace - 1;

enum : int { kStEmpty = 0, kStScore = 1, kStDecode = 2 };
// control words in shared memory
enum : int { kCtlComb = 0, kCtlFree = 2, kCtlWords = 8 };

enum StreamTraceEvent : int {
  kSeStart = 1, kSeExit = 2, kSeFirstScore = 3, kSeLastScore = 4, kSeFirstDecode = 5,
  kSeLastDecode = 6, kSeSelBegin = 7, kSeSelEnd = 8, kSeMergeBegin = 9, kSeMergeEnd = 10,
  kSeIssueDecode = 11, kSeIssueLast = 12, kSeStageDone = 13, kSeIssue = 14, kSeSelLoaded = 15,
  kSeStageLanded = 16, kSeSelTopk = 17, kSeSelWritten = 18, kSeSelFenced = 19,
};

struct SInfo {
  int kind;  // kStEmpty / kStScore / kStDecode
  int j;     // pair
  int a;     // scoring: first page; decode: piece of the pair
  int n;     // scoring: boxes; decode: valid tokens of the page (0: nothing staged)
  int b, g;  // the pair's sequence and kv head
  int L, N;  // the sequence's tokens (after this step's append) and pages
};

struct SSmem {
  unsigned char* ring;  // [S][slot]: data (P boxes, or a page's K then V chunk), then q
  uint64_t* full;       // [S]
  uint64_t* empty;      // [S]
  SInfo* info;          // [S]
  float* wsc;           // [kSWarps][G * P] logits, then weights, of the page in hand
  float* st;            // [kSWarps][G * 3] running max (log2 units), sum, rescale
  float* cbuf;          // [nb][kSWarps][cbuf_floats(G)]: per warp acc[G][128], m[G], l[G]
  int* ctl;             // [kCtlWords]
  int* lens;            // [B] tokens of each sequence in this step (after its append)
  int* sb;              // [B + 1] scoring pieces before sequence b (all its kv heads)
  int* db;              // [B + 1] decode pieces before sequence b
  uint32_t* keys;       // [keys_stride(max_pages)] selector: the pair's keys
  int* hist;            // [kFastBins] selection histogram (zero between uses)
  int* scratch;         // [256]
  int* sel;             // [kcap] kept pages, ascending
  float* msc;           // [G][npc_max + 2] merge: scale of each partial, max, sum
  int nb;               // combine buffers (decode piece k uses buffer k mod nb)
  __half* qall;         // [B][Hq][128] every query, or null (each stage carries its own)
  uint64_t* qbar;       // completes when qall has landed
};

__host__ __device__ inline int s_keys_stride(int max_pages) { return (max_pages + 3) & ~3; }

// Floats of one warp's state in the combine buffer: acc[G][128], then m[G] and l[G], padded
// to whole 16-byte units so that every warp's acc starts on 16 bytes (float4 accesses).
__host__ __device__ constexpr int cbuf_floats(int G) { return G * kHeadDim + ((2 * G + 3) & ~3); }

// The queries of every pair (B * Hq * 256 bytes) are staged in shared memory once when they
// fit in kQAllBytes; otherwise every stage carries its pair's query after its data.
constexpr size_t kQAllBytes = 32 << 10;
__host__ __device__ inline bool q_all(int batch, int hq) {
  return (size_t)batch * hq * kHeadDim * 2 <= kQAllBytes;
}
__host__ __device__ inline size_t s_slot_bytes(int G, int P, bool qall) {
  return align_up((size_t)2 * P * kHeadDim * 2 + (qall ? 0 : (size_t)G * kHeadDim * 2), 128);
}

// Bytes a selector CTA keeps in shared memory (in the space a streaming CTA gives its ring).
__host__ __device__ inline size_t selector_bytes(int G, int max_pages, int kcap) {
  const int npc = (kcap + kPiecePages - 1) / kPiecePages;
  return align_up((size_t)s_keys_stride(max_pages) * 4, 16) + (size_t)kFastBins * 4 +
         256 * 4 + align_up((size_t)kcap * 4, 16) + align_up((size_t)G * (npc + 2) * 4, 16);
}

// The fixed part, the ring barriers and descriptors, then one region that is the ring in a
// streaming CTA and the selection buffers in a selector CTA; as many ring slots as fit in
// `budget` bytes (a multiple of kSWarps; 0 if the shape does not fit).  Writes the layout
// into s when given.
__host__ __device__ inline size_t stream_smem_layout_nb(int G, int P, int max_pages, int top_k,
                                                        int batch, int hq, size_t budget,
                                                        int max_slots, int nb, int* slots, SSmem* s,
                                                        unsigned char* base) {
  const int kcap = top_k < max_pages ? top_k : max_pages;
  const bool qall = q_all(batch, hq);
  const int npc = (kcap + kPiecePages - 1) / kPiecePages;
  size_t o = 0;
  const size_t wsc = o;      o = align_up(o + (size_t)kSWarps * G * P * 4, 16);
  const size_t st = o;       o = align_up(o + (size_t)kSWarps * G * 3 * 4, 16);
  const size_t cbuf = o;     o = align_up(o + (size_t)nb * kSWarps * cbuf_floats(G) * 4, 16);
  const size_t ctl = o;      o = align_up(o + kCtlWords * 4, 16);
  const size_t lens = o;     o = align_up(o + (size_t)batch * 4, 16);
  const size_t sb = o;       o = align_up(o + (size_t)(batch + 1) * 4, 16);
  const size_t db = o;       o = align_up(o + (size_t)(batch + 1) * 4, 16);
  const size_t qa = o;       o = align_up(o + (qall ? (size_t)batch * hq * kHeadDim * 2 : 0), 128);
  const size_t qbar = o;     o += 16;
  const size_t fixed = o;
  const size_t per_slot = s_slot_bytes(G, P, qall) + 2 * 8 + sizeof(SInfo);
  // a multiple of kSWarps: stage s sits in slot s mod S and belongs to consumer s mod 8, so
  // every slot keeps one consumer, which waits on its phases in order (a parity wait that
  // ran two phases ahead of the slot would be satisfied by the wrong phase)
  int S = 0;
  if (budget > fixed + 512) S = (int)((budget - fixed - 512) / per_slot);
  if (S > max_slots) S = max_slots;
  S -= S % kSWarps;
  const size_t bars = fixed;
  size_t e = bars + (size_t)S * 16;
  const size_t infoo = e;    e = align_up(e + (size_t)S * sizeof(SInfo), 128);
  const size_t region = e;
  const size_t ring_bytes = (size_t)S * s_slot_bytes(G, P, qall);
  const size_t sel_bytes = selector_bytes(G, max_pages, kcap);
  e = region + (ring_bytes > sel_bytes ? ring_bytes : sel_bytes);
  if (e > budget) S = 0;
  if (slots) *slots = S;
  if (s) {
    s->ring = base + region;
    s->full = reinterpret_cast<uint64_t*>(base + bars);
    s->empty = s->full + S;
    s->info = reinterpret_cast<SInfo*>(base + infoo);
    s->wsc = reinterpret_cast<float*>(base + wsc);
    s->st = reinterpret_cast<float*>(base + st);
    s->cbuf = reinterpret_cast<float*>(base + cbuf);
    s->ctl = reinterpret_cast<int*>(base + ctl);
    s->lens = reinterpret_cast<int*>(base + lens);
    s->sb = reinterpret_cast<int*>(base + sb);
    s->db = reinterpret_cast<int*>(base + db);
    size_t r = region;
    s->keys = reinterpret_cast<uint32_t*>(base + r);  r += align_up((size_t)s_keys_stride(max_pages) * 4, 16);
    s->hist = reinterpret_cast<int*>(base + r);       r += (size_t)kFastBins * 4;
    s->scratch = reinterpret_cast<int*>(base + r);    r += 256 * 4;
    s->sel = reinterpret_cast<int*>(base + r);        r += align_up((size_t)kcap * 4, 16);
    s->msc = reinterpret_cast<float*>(base + r);
    (void)npc;
    s->nb = nb;
    s->qall = qall ? reinterpret_cast<__half*>(base + qa) : nullptr;
    s->qbar = reinterpret_cast<uint64_t*>(base + qbar);
  }
  return e;
}

// The layout with two combine buffers (a piece's warps need not wait for the previous
// piece's combine) if the ring still gets kSWarps slots, else with one.
__host__ __device__ inline size_t stream_smem_layout(int G, int P, int max_pages, int top_k,
                                                     int batch, int hq, size_t budget,
                                                     int max_slots, int* slots, SSmem* s,
                                                     unsigned char* base) {
  int S = 0;
  stream_smem_layout_nb(G, P, max_pages, top_k, batch, hq, budget, max_slots, 2, &S, nullptr,
                        nullptr);
  const int nb = S >= kSWarps ? 2 : 1;
  return stream_smem_layout_nb(G, P, max_pages, top_k, batch, hq, budget, max_slots, nb, slots,
                               s, base);
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

// The geometry a consumer needs, from its stage's descriptor (no division).
__device__ __forceinline__ PairGeo geo_of(const Params& p, const SInfo& in) {
  PairGeo q;
  q.b = in.b;
  q.g = in.g;
  q.L = in.L;
  q.N = in.N;
  q.K = min(p.top_k, in.N);
  q.npc = 0;
  q.ndc = 0;
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

// A timeline record (out of line: it is off the hot path unless a trace was asked for).
__device__ __noinline__ void strace_rec(const Params& p, int* slot, int ev, int item) {
  const long long i = (long long)blockIdx.x * kStreamTrace + (*slot)++;
  if (i >= p.trace_capacity) return;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  p.trace[1 + 2 * i] = (unsigned long long)global_ns();
  p.trace[2 + 2 * i] = ((unsigned long long)smid << 48) |
                       ((unsigned long long)(blockIdx.x & 0xffff) << 32) |
                       ((unsigned long long)(ev & 0xff) << 24) | (unsigned)(item & 0xffffff);
}
__device__ __forceinline__ void strace(const Params& p, int* slot, int limit, int ev, int item) {
  if (p.trace != nullptr && *slot < limit) strace_rec(p, slot, ev, item);
}

__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_volatile_s32(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

// True in every thread of the selector team if `pred` holds in any of them (named barrier 1).
template <int NT>
__device__ __forceinline__ bool bany(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.or.pred po, 1, %2, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NT)
      : "memory");
  return r != 0;
}

// ---------------------------------------------------------------- producer warp
// The ring position of stage `stage`: slot and phase parity, advanced without a division.
struct RingPos {
  int slot;
  uint32_t phase;
  __device__ __forceinline__ void step(int by, int S) {
    slot += by;
    if (slot >= S) {
      slot -= S;
      phase ^= 1u;
    }
  }
};

// Stages are issued in order, one lane at a time; each lane first works out, in parallel
// with the others, where its stage's data comes from (the mapping of pieces to pairs takes
// integer divisions: done serially they would make the producer the bottleneck).
template <int G, int P>
__device__ void s_produce(const Params& p, const LayerPtrs& lay, const SSmem& s, int S, int C,
                          int TS, int TD, int nS, int nS_pad) {
  constexpr uint32_t kChunk = (uint32_t)P * kHeadDim * 2;  // one page of K (or V), one kv head
  constexpr uint32_t kBox = 2 * kHeadDim * 2;              // one page's box (min, max)
  const bool qall = s.qall != nullptr;
  const uint32_t kQ = qall ? 0u : (uint32_t)G * kHeadDim * 2;
  const size_t slot_bytes = s_slot_bytes(G, P, qall);
  const int lane = threadIdx.x & 31;
  const int c = (int)blockIdx.x;
  int tslot = kTrProducer;
  RingPos pos{0, 0u};
  if (qall && lane == 0) {  // every query of the call, once
    const uint32_t qb = (uint32_t)((size_t)p.B * p.Hq * kHeadDim * 2);
    mbar_arrive_expect_tx(s.qbar, qb);
    bulk_g2s(s.qall, lay.q, qb, s.qbar);
  }
  // ---- scoring pieces (the boxes of up to P pages of one pair fill one stage), then
  // empty stages up to a whole round of kSWarps
  for (int k0 = 0; k0 < nS_pad; k0 += 32) {
    const int k = k0 + lane;
    int j = 0, p0 = 0, n = 0;
    PairGeo q{};
    const __half* box = nullptr;
    const __half* qsrc = nullptr;
    if (k < nS) {
      int u;
      piece_of(p, s.sb, c + k * C, &j, &u);
      q = pair_geo(p, s, j);
      p0 = u * P;
      n = min(P, q.N - p0);
      box = lay.meta + box_offset(p, q.b, q.g, p0);
      qsrc = lay.q + ((size_t)q.b * p.Hq + (size_t)q.g * G) * kHeadDim;
    }
    const int cnt = min(32, nS_pad - k0);
#pragma unroll 1
    for (int i = 0; i < cnt; ++i) {
      if (lane == i) {
        const bool ok = mbar_wait_bounded(p, &s.empty[pos.slot], pos.phase ^ 1u, kSiteWaitSlot);
        uint64_t* bar = &s.full[pos.slot];
        strace(p, &tslot, kTrLast - 2, kSeIssue, k);
        if (k < nS) {
          s.info[pos.slot] = SInfo{kStScore, j, p0, ok ? n : 0, q.b, q.g, q.L, q.N};
          if (ok) {
            unsigned char* dst = s.ring + (size_t)pos.slot * slot_bytes;
            mbar_arrive_expect_tx(bar, (uint32_t)n * kBox + kQ);
            bulk_g2s(dst, box, (uint32_t)n * kBox, bar);
            if (!qall) bulk_g2s(dst + 2 * kChunk, qsrc, kQ, bar);
          } else {
            mbar_arrive(bar);
          }
        } else {
          s.info[pos.slot] = SInfo{kStEmpty, 0, 0, 0, 0, 0, 0, 0};
          mbar_arrive(bar);
        }
      }
      pos.step(1, S);
      __syncwarp();
    }
  }
  if (lane == 0 && TS > c) strace(p, &tslot, kTrLast, kSeIssueLast, 0);
  // ---- decode pieces: up to 8 kept pages of one pair, page i to consumer i.  Lane l
  // works out piece k0 + l's pair; the kept pages of the next piece are fetched while the
  // current piece's copies are being issued, when its selection is already out.  A page's
  // K and V chunks are scattered over the pool: the whole warp copies them, 16 bytes a lane
  // per instruction, and the stage completes on its full barrier through the copies' own
  // arrivals (each lane's, plus one plain arrival of lane 0).
  bool first = true;
  const int nD = c < TD ? (TD - 1 - c) / C + 1 : 0;
  int2 e_next = make_int2(-1, -1);
  bool have_next = false;
  for (int k0 = 0; k0 < nD; k0 += 32) {
    int dj = 0, dv = 0;
    if (k0 + lane < nD) piece_of(p, s.db, c + (k0 + lane) * C, &dj, &dv);
    const int cnt = min(32, nD - k0);
#pragma unroll 1
    for (int i = 0; i < cnt; ++i) {
      const int j = __shfl_sync(0xffffffffu, dj, i), v = __shfl_sync(0xffffffffu, dv, i);
      const PairGeo q = pair_geo(p, s, j);
      const int n = min(kPiecePages, q.K - v * kPiecePages);
      bool ok = true;
      int2 e = make_int2(-1, -1);
      if (have_next) {
        e = e_next;
      } else {
        if (lane == 0) ok = wait_flag_bounded(p, p.ready + j, 1u, q.b, kSiteWaitSelection);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok) {
          (void)ld_acquire_u32(p.ready + j);  // every lane acquires the selection
          if (lane < n)
            e = __ldcg(reinterpret_cast<const int2*>(p.sel_pair) + (size_t)j * p.top_k +
                       v * kPiecePages + lane);
        }
      }
      if (first && lane == 0) strace(p, &tslot, kTrLast, kSeIssueDecode, j);
      first = false;
      int nv = 0, ph = 0;
      if (ok && lane < n && e.x >= 0 && e.x < q.N && e.y >= 0 && e.y < p.num_phys) {
        nv = min(P, q.L - e.x * P);
        ph = e.y;
      }
      // the next piece's kept pages, if its pair is already selected
      have_next = false;
      if (i + 1 < cnt || k0 + 32 < nD) {  // warp-uniform
        int jn, vn;
        if (i + 1 < cnt) {
          jn = __shfl_sync(0xffffffffu, dj, i + 1);
          vn = __shfl_sync(0xffffffffu, dv, i + 1);
        } else {
          int a = 0, b2 = 0;
          if (lane == 0) piece_of(p, s.db, c + (k0 + 32) * C, &a, &b2);
          jn = __shfl_sync(0xffffffffu, a, 0);
          vn = __shfl_sync(0xffffffffu, b2, 0);
        }
        int rdy = 0;
        if (lane == 0) rdy = ld_acquire_u32(p.ready + jn) == 1u;
        rdy = __shfl_sync(0xffffffffu, rdy, 0);
        if (rdy) {
          const PairGeo qn = pair_geo(p, s, jn);
          const int nn = min(kPiecePages, qn.K - vn * kPiecePages);
          (void)ld_acquire_u32(p.ready + jn);  // every lane acquires the selection
          if (lane < nn)
            e_next = __ldcg(reinterpret_cast<const int2*>(p.sel_pair) + (size_t)jn * p.top_k +
                            vn * kPiecePages + lane);
          have_next = true;
        }
      }
      const unsigned char* qsrc = reinterpret_cast<const unsigned char*>(
          lay.q + ((size_t)q.b * p.Hq + (size_t)q.g * G) * kHeadDim);
#pragma unroll 1
      for (int t = 0; t < kPiecePages; ++t) {
        const int nvt = __shfl_sync(0xffffffffu, nv, t);
        const int pht = __shfl_sync(0xffffffffu, ph, t);
        int fr = 1;
        if (lane == 0) fr = mbar_wait_bounded(p, &s.empty[pos.slot], pos.phase ^ 1u, kSiteWaitSlot);
        fr = __shfl_sync(0xffffffffu, fr, 0);
        __syncwarp();  // the slot's last reads happen before any lane's copy into it
        const int nvs = fr ? nvt : 0;
        uint64_t* bar = &s.full[pos.slot];
        if (lane == 0) s.info[pos.slot] = SInfo{kStDecode, j, v, nvs, q.b, q.g, q.L, q.N};
        if (nvs > 0) {  // warp-uniform
          unsigned char* dst = s.ring + (size_t)pos.slot * slot_bytes + 16 * lane;
          const size_t off = (((size_t)pht * p.Hkv + q.g) * (size_t)P * kHeadDim) * 2 + 16 * lane;
          const unsigned char* ks = reinterpret_cast<const unsigned char*>(lay.k_pool) + off;
          const unsigned char* vs = reinterpret_cast<const unsigned char*>(lay.v_pool) + off;
#pragma unroll
          for (int u = 0; u < (int)kChunk / 512; ++u) cp_async16(dst + 512 * u, ks + 512 * u);
#pragma unroll
          for (int u = 0; u < (int)kChunk / 512; ++u)
            cp_async16(dst + kChunk + 512 * u, vs + 512 * u);
          if (!qall)  // the pair's G query rows, 16 G units of 16 bytes
            for (int u = lane; u < (int)kQ / 16; u += 32)
              cp_async16(dst - 16 * lane + 2 * kChunk + 16 * u, qsrc + 16 * u);
          cp_async_arrive(bar);
          __syncwarp();  // every lane's pending arrival is counted before lane 0's
        }
        if (lane == 0) mbar_arrive(bar);
        pos.step(1, S);
        __syncwarp();
      }
    }
  }
  if (TD > c && lane == 0) strace(p, &tslot, kTrLast, kSeIssueLast, 1);
}

// ---------------------------------------------------------------- consumer warps
// The query heads of a stage's pair: in the shared copy of every query, or after the data.
template <int G, int P>
__device__ __forceinline__ const __half* stage_q(const Params& p, const SSmem& s,
                                                 const unsigned char* slot, const PairGeo& q) {
  if (s.qall) return s.qall + ((size_t)q.b * p.Hq + (size_t)q.g * G) * kHeadDim;
  return reinterpret_cast<const __half*>(slot + 2 * (size_t)P * kHeadDim * 2);
}

// Bound of every page of a scoring stage (half-warp per page); the keys go to the pair's
// key row in global memory, where the pair's selector polls for them (a written key is
// never 0).  The page of the step's new token first takes the token: its box opens or
// widens (in the staged copy too), is written back with the token's K and V rows, and those
// writes are made visible before any key of the stage (the selection that follows releases
// the page to the decode pieces, which read the rows).  Returns true (in the whole warp) if
// the stage wrote into its slot.
template <int G, int P>
__device__ bool s_score_stage(const Params& p, const LayerPtrs& lay, const SSmem& s,
                              unsigned char* slot, const SInfo& in, const PairGeo& q) {
  const int lane = threadIdx.x & 31;
  const int hw = lane >> 4, c = lane & 15;
  QueryFrag<G> f;
  load_query_frag<G>(stage_q<G, P>(p, s, slot, q), 0, 0, 0, c, f);
  const int ap = (lay.k_new != nullptr && p.chain_append && q.L > 0) ? (q.L - 1) / P : -1;
  const bool takes_token = ap >= in.a && ap < in.a + in.n;  // warp-uniform
  if (takes_token) {
    if (hw == 0) {
      const int ph = p.block_table[(size_t)q.b * p.max_pages + ap];
      if (ph >= 0 && ph < p.num_phys) {
        const size_t o = ((size_t)q.b * p.Hkv + q.g) * kHeadDim + 8 * c;
        const uint4 knew = *reinterpret_cast<const uint4*>(lay.k_new + o);
        const uint4 vnew = *reinterpret_cast<const uint4*>(lay.v_new + o);
        const int slot_a = (q.L - 1) % P;
        unsigned char* rec = slot + (size_t)(ap - in.a) * 2 * kHeadDim * 2;
        uint4 mn = knew, mx = knew;
        if (slot_a != 0) {
          const uint4 a0 = *reinterpret_cast<const uint4*>(rec + 16 * c);
          const uint4 z0 = *reinterpret_cast<const uint4*>(rec + 2 * kHeadDim + 16 * c);
          const uint32_t a[4] = {a0.x, a0.y, a0.z, a0.w};
          const uint32_t z[4] = {z0.x, z0.y, z0.z, z0.w};
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
        *reinterpret_cast<uint4*>(rec + 16 * c) = mn;  // the staged box, for the scoring below
        *reinterpret_cast<uint4*>(rec + 2 * kHeadDim + 16 * c) = mx;
        __half* box = lay.meta + box_offset(p, q.b, q.g, ap);
        *reinterpret_cast<uint4*>(box + 8 * c) = mn;
        *reinterpret_cast<uint4*>(box + kHeadDim + 8 * c) = mx;
        const size_t kv = (((size_t)ph * p.Hkv + q.g) * P + slot_a) * kHeadDim + 8 * c;
        *reinterpret_cast<uint4*>(lay.k_pool + kv) = knew;
        *reinterpret_cast<uint4*>(lay.v_pool + kv) = vnew;
      } else if (c == 0) {
        report(p, QUEST_ERR_BAD_PAGE, q.b, ap, kSiteAppend);
      }
    }
    __threadfence();  // the new rows and box, before this stage's keys
    __syncwarp();
  }
  unsigned* krow = p.skeys + (size_t)(q.b * p.Hkv + q.g) * p.max_pages;
  const bool windowed = q.N > q.K && (p.sink_pages > 0 || p.local_pages > 0);
  // half-warp hw scores boxes hw, hw + 2, ...: UB of them at a time, every load issued
  // before any arithmetic and the half-warp sums interleaved, so that the stage is not one
  // long chain of dependent steps
  constexpr int UB = G <= 2 ? 4 : 2;
#pragma unroll 1
  for (int r0 = 0; 2 * r0 < in.n; r0 += UB) {
    uint4 mn[UB], mx[UB];
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      const int r = 2 * (r0 + u) + hw;
      mn[u] = make_uint4(0, 0, 0, 0);
      mx[u] = make_uint4(0, 0, 0, 0);
      if (r < in.n) {
        const unsigned char* rec = slot + (size_t)r * 2 * kHeadDim * 2;
        mn[u] = *reinterpret_cast<const uint4*>(rec + 16 * c);
        mx[u] = *reinterpret_cast<const uint4*>(rec + 2 * kHeadDim + 16 * c);
      }
    }
    float sc[UB][G];
#pragma unroll
    for (int u = 0; u < UB; ++u)
#pragma unroll
      for (int jh = 0; jh < G; ++jh) sc[u][jh] = corner_dot<G>(f, jh, mn[u], mx[u]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
#pragma unroll
      for (int u = 0; u < UB; ++u)
#pragma unroll
        for (int jh = 0; jh < G; ++jh) sc[u][jh] += __shfl_xor_sync(0xffffffffu, sc[u][jh], o);
    // lane c < UB of half-warp hw writes the key of box 2 (r0 + c) + hw: the warp's keys
    // of this group are one contiguous run
    uint32_t key = 0u;
#pragma unroll
    for (int u = 0; u < UB; ++u) {
      float best = sc[u][0];
#pragma unroll
      for (int jh = 1; jh < G; ++jh) best = fmaxf(best, sc[u][jh]);
      const int page = in.a + 2 * (r0 + u) + hw;
      // pages of the sink / local window of a long sequence get the largest key; no score
      // key is 0 (that would take a NaN with every bit set), so 0 can mean "not written"
      const bool forced = windowed && (page < p.sink_pages || page >= q.N - p.local_pages);
      const uint32_t k = forced ? 0xffffffffu : max(score_key(best), 1u);
      if (c == u) key = k;
    }
    const int r = 2 * (r0 + c) + hw;
    if (c < UB && r < in.n) __stcg(krow + in.a + r, key);
  }
  return takes_token;
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
    const __half* qs = stage_q<G, P>(p, s, slot, geo_of(p, in));
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
  // the combine buffer of this piece must be done with piece k - nb
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
  // this warp's state: acc[G][128], m[G], l[G]
  if (lane < G) {
    cb[G * kHeadDim + lane] = st[lane * 3 + 0];
    cb[G * kHeadDim + G + lane] = st[lane * 3 + 1];
  }
#pragma unroll
  for (int jh = 0; jh < G; ++jh)
    *reinterpret_cast<float4*>(cb + jh * kHeadDim + 4 * lane) =
        make_float4(acc[jh][0], acc[jh][1], acc[jh][2], acc[jh][3]);
}

// Combine the 8 warps' states of a piece into its split-K partial (one warp).
template <int G>
__device__ void s_combine(const Params& p, const float* cbase, const PairGeo& q, int v) {
  const int lane = threadIdx.x & 31;
  constexpr int WF = cbuf_floats(G);  // floats per warp state
  constexpr int MO = G * kHeadDim;    // offset of m[G]; l[G] follows
#pragma unroll
  for (int jh = 0; jh < G; ++jh) {
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) M = fmaxf(M, cbase[w * WF + MO + jh]);
    float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
    float Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kSWarps; ++w) {
      const float m = cbase[w * WF + MO + jh];
      const float f = (m == -CUDART_INF_F) ? 0.f : exp2f(m - M);
      const float4 a = *reinterpret_cast<const float4*>(cbase + w * WF + jh * kHeadDim + 4 * lane);
      A.x = fmaf(a.x, f, A.x);
      A.y = fmaf(a.y, f, A.y);
      A.z = fmaf(a.z, f, A.z);
      A.w = fmaf(a.w, f, A.w);
      Ls = fmaf(cbase[w * WF + MO + G + jh], f, Ls);
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
  const int w = threadIdx.x >> 5;
  const size_t slot_bytes = s_slot_bytes(G, P, s.qall != nullptr);
  constexpr int WF = cbuf_floats(G);
  if (s.qall) mbar_wait_bounded(p, s.qbar, 0u, kSiteWaitStage);  // the queries have landed
  static_assert(WF % 4 == 0, "each warp's state starts on 16 bytes");
  int tslot = 8 + 24 * w;
  RingPos pos{w, 0u};  // S is a multiple of kSWarps: this warp's slots are w, w + 8, ...
  for (int stg = w; stg < total_stages; stg += kSWarps, pos.step(kSWarps, S)) {
    const int sl = pos.slot;
    const bool ok = mbar_wait_bounded(p, &s.full[sl], pos.phase, kSiteWaitStage);
    if (lane == 0) strace(p, &tslot, 32 + 24 * w, kSeStageLanded, stg);
    SInfo in = s.info[sl];
    if (!ok) in.n = 0;
    unsigned char* slot = s.ring + (size_t)sl * slot_bytes;
    if (in.kind == kStScore) {
      const PairGeo q = geo_of(p, in);
      // a stage that took the new token wrote into its slot: generic writes, ordered before
      // the slot goes back to bulk copies (the other stages only read their slot)
      if (in.n > 0 && s_score_stage<G, P>(p, lay, s, slot, in, q)) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[sl]);
    } else if (in.kind == kStDecode) {
      const int k = (stg - nS_pad) / kSWarps;  // this CTA's decode piece
      const int par = k % s.nb;
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
        const PairGeo q = geo_of(p, in);
        s_combine<G>(p, cbase, q, in.a);
        __syncwarp();
        if (lane == 0) {
          s.ctl[kCtlComb + par] = 0;
          __threadfence_block();
          atomicExch(&s.ctl[kCtlFree + par], k + s.nb);
          red_add_release(p.decode_arrive + in.j, 1u);  // after the partial
        }
      }
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.empty[sl]);
    }
    if (lane == 0 && in.kind != kStEmpty)
      strace(p, &tslot, 32 + 24 * w, kSeStageDone, (stg & 0xfffff) | (in.kind << 20));
  }
}

// ---------------------------------------------------------------- selector team
// Exact top-K of pair j's keys; the kept pages (ascending) go out with their physical
// pages, then the pair is released to the decode pieces.  The keys arrive in the pair's
// key row from every CTA's consumers: the row is read until none of its N keys is 0 (not
// written yet), then cleared for the next call.
__device__ void s_select(const Params& p, const SSmem& s, const PairGeo& q, int j) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* sel = s.sel;
  unsigned* krow = p.skeys + (size_t)j * p.max_pages;
  uint32_t lo = 0xffffffffu, hi = 0u;
  const long long t0 = global_ns();
  while (true) {
    int missing = 0;
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll 1
    for (int i0 = 0; i0 < q.N; i0 += 4 * kSelThreads) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        v[u] = i < q.N ? __ldcg(krow + i) : 1u;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kSelThreads + tid;
        if (i < q.N) {
          s.keys[i] = v[u];
          missing |= v[u] == 0u;
          lo = min(lo, v[u]);
          hi = max(hi, v[u]);
        }
      }
    }
    if (!bany<kSelThreads>(missing != 0)) break;
    // thread 0 decides when to give up, for the whole team
    if (bany<kSelThreads>(tid == 0 && global_ns() - t0 > p.wait_limit_ns)) {
      if (tid == 0) report(p, QUEST_ERR_TIMEOUT, q.b, -1, kSiteWaitSelection);
      break;
    }
    __nanosleep(200);
  }
  // the keys are in shared memory: clear the row for the next call
  for (int i = tid; i < q.N; i += kSelThreads) __stcg(krow + i, 0u);
  if (q.N <= q.K) {
    for (int r = tid; r < q.K; r += kSelThreads) sel[r] = r;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      s.scratch[100 + warp] = (int)lo;
      s.scratch[120 + warp] = (int)hi;
    }
    bsync<kSelThreads, true>();
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll
    for (int w = 0; w < kSelWarps; ++w) {
      lo = min(lo, (uint32_t)s.scratch[100 + w]);
      hi = max(hi, (uint32_t)s.scratch[120 + w]);
    }
    if (tid == 0) {
      int* ts = s.scratch + 250;  // the team's trace slot, kept by the team's loop
      strace(p, ts, kTrLast, kSeSelLoaded, j);
    }
    topk_fast<kSelThreads, true>(s.keys, q.N, q.K, lo, hi, sel, s.hist, s.scratch);
    if (tid == 0) strace(p, s.scratch + 250, kTrLast, kSeSelTopk, j);
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
  if (tid == 0) strace(p, s.scratch + 250, kTrLast, kSeSelWritten, j);
  __threadfence();
  bsync<kSelThreads, true>();
  if (tid == 0) strace(p, s.scratch + 250, kTrLast, kSeSelFenced, j);
  if (tid == 0 && !(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION))
    st_release_u32(p.ready + j, 1u);
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

// Selector CTA sc of Cs owns pairs sc, sc + Cs, ...: pairs finish scoring roughly in
// order, so consecutive pairs go to different selector CTAs and are selected side by side.
// For each of its pairs, in order, the team waits until all of the pair's keys are in and
// selects; then, pair by pair again, it waits until every decode piece has been combined
// (counted by the streaming CTAs' consumers with release reductions, polled with acquire
// loads; all CTAs are resident, so every count completes) and merges.
template <int G>
__device__ void s_selector(const Params& p, const LayerPtrs& lay, const SSmem& s, int NP,
                           int sc, int Cs) {
  const int tid = threadIdx.x;
  int* tslot = s.scratch + 250;  // the team's next trace record (thread 0 only)
  if (tid == 0) *tslot = kTrSelector;
  for (int j = sc; j < NP; j += Cs) {
    const PairGeo q = pair_geo(p, s, j);
    if (q.N == 0) {
      s_empty_pair<G>(p, lay, q, j);
      continue;
    }
    if (tid == 0) strace(p, tslot, kTrLast, kSeSelBegin, j);
    s_select(p, s, q, j);
    if (tid == 0) strace(p, tslot, kTrLast, kSeSelEnd, j);
    bsync<kSelThreads, true>();
  }
  for (int j = sc; j < NP; j += Cs) {
    const PairGeo q = pair_geo(p, s, j);
    if (q.N == 0) continue;
    if (tid == 0) wait_flag_bounded(p, p.decode_arrive + j, (unsigned)q.ndc, q.b, kSiteWaitSlot);
    bsync<kSelThreads, true>();
    (void)ld_acquire_u32(p.decode_arrive + j);  // every thread acquires the pair's partials
    if (tid == 0) strace(p, tslot, kTrLast, kSeMergeBegin, j);
    s_merge<G>(p, lay, s, q, j);
    if (tid == 0) strace(p, tslot, kTrLast, kSeMergeEnd, j);
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
  stream_smem_layout(G, P, p.max_pages, p.top_k, p.B, p.Hq, kMaxSmem, p.ring_slots, &S, &s,
                     smem);
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(s.qbar, 1);
    fence_mbar_init();
  }
  const int Cs = p.sel_ctas, C = (int)gridDim.x - Cs, c = (int)blockIdx.x;
  const bool selector = c >= C;  // the last Cs CTAs select and merge, the others stream
  if (tid < kCtlWords) s.ctl[tid] = (tid == kCtlFree + 1) ? 1 : 0;
  if (selector)
    for (int i = tid; i < kFastBins; i += blockDim.x) s.hist[i] = 0;
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
  const int nS = !selector && c < TS ? (TS - 1 - c) / C + 1 : 0;
  const int nD = !selector && c < TD ? (TD - 1 - c) / C + 1 : 0;
  const int nS_pad = (nS + kSWarps - 1) / kSWarps * kSWarps;
  const int total = nS_pad + nD * kSWarps;
  if (tid == 0) {
    int t0 = 0;
    strace(p, &t0, 1, kSeStart, TS);
  }
  const int warp = tid >> 5;
  if (selector) {
    if (warp < kSelWarps) s_selector<G>(p, lay, s, p.B * p.Hkv, c - C, Cs);
  } else if (warp == kProducerWarp) {
    s_produce<G, P>(p, lay, s, S, C, TS, TD, nS, nS_pad);
  } else if (warp < kSWarps) {
    s_consume<G, P>(p, lay, s, S, total, nS_pad);
  }
  __syncthreads();
  // a wait that gave up may leave copies in flight: let them land before the CTA leaves
  if (!selector && tid == kProducerWarp * 32 && ld_relaxed_s32(p.status) != QUEST_OK) {
    const int last = total;
    for (int st = max(0, last - S); st < last; ++st)
      mbar_wait_bounded(p, &s.full[st % S], (uint32_t)(st / S) & 1u, kSiteWaitStage);
  }
  if (tid == 0) {
    int tl = kStreamTrace - 1;
    strace(p, &tl, kStreamTrace, kSeExit, 0);
  }
  // With an appended token, CTA 0 advances the lengths once every CTA has read them.
  if (p.chain_append && !p.hold_lengths && c == 0 && tid < 32) {
    bool ok = true;
    if (tid == 0) ok = wait_flag_bounded(p, p.started, gridDim.x, -1, kSiteWaitSlot);
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

// Ring slots at most (the shared memory left after the rest usually holds fewer: ~24 slots
// of 8 KB at page 16; a shallower ring measured no faster).
constexpr int kStreamMaxSlots = 64;

// Ring slots of the stream kernel for this shape (0: it does not fit).
int stream_slots(int G, int P, int max_pages, int top_k, int batch, int hq) {
  // (the selection packs per-thread counts of keys in 16 bits)
  if (batch > kStreamMaxBatch || top_k > kStreamMaxTopk || max_pages >= 65536)
    return 0;
  int S = 0;
  stream_smem_layout(G, P, max_pages, top_k, batch, hq, kMaxSmem, kStreamMaxSlots, &S,
                     nullptr, nullptr);
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

size_t stream_smem_bytes(int G, int P, int max_pages, int top_k, int batch, int hq) {
  const int S = stream_slots(G, P, max_pages, top_k, batch, hq);
  return stream_smem_layout(G, P, max_pages, top_k, batch, hq, kMaxSmem, S, nullptr, nullptr,
                            nullptr);
}

// CTAs of a stream launch: selector CTAs, one for every two pairs (at most 16, at most a
// quarter of the grid, at least one), and streaming CTAs, one per remaining SM, fewer for a
// small step (about 64 KB of stream per CTA at least).  max_ctas, when given, caps the
// whole grid (which keeps at least one CTA of each kind).
cudaError_t stream_grid(const Params& p, int max_ctas, int* ctas, int* sel_ctas) {
  DevInfo d;
  cudaError_t e = device_info(&d);
  if (e != cudaSuccess) return e;
  if (!d.coop) return cudaErrorNotSupported;
  const long long kcap = std::min<long long>(p.top_k, p.max_pages);
  const long long pairs = (long long)p.B * p.Hkv;
  const long long bytes =
      pairs * ((long long)p.max_pages * 2 * kHeadDim * 2 + kcap * p.P * kHeadDim * 4);
  const long long want_sel = std::max<long long>(1, std::min<long long>(16, (pairs + 1) / 2));
  long long n = (bytes + (64 << 10) - 1) / (64 << 10) + want_sel;
  if (n > d.sms) n = d.sms;
  if (max_ctas > 0 && n > max_ctas) n = max_ctas;
  if (n < 2) n = 2;
  const long long sel = std::max<long long>(1, std::min<long long>(want_sel, n / 4));
  *ctas = (int)n;
  *sel_ctas = (int)sel;
  return cudaSuccess;
}

cudaError_t launch_stream(const Params& p, const LayerPtrs& lay, int G, int max_ctas,
                          cudaStream_t s) {
  const int S = stream_slots(G, p.P, p.max_pages, p.top_k, p.B, p.Hq);
  if (S < kSWarps) return cudaErrorInvalidConfiguration;
  const size_t smem = stream_smem_bytes(G, p.P, p.max_pages, p.top_k, p.B, p.Hq);
  const void* fn = pick_stream(G, p.P);
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int ctas = 0, sel = 0;
  if ((e = stream_grid(p, max_ctas, &ctas, &sel)) != cudaSuccess) return e;
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
  pp.sel_ctas = sel;
  pp.ring_slots = S;
  LayerPtrs ll = lay;
  void* args[] = {&pp, &ll};
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace quest
