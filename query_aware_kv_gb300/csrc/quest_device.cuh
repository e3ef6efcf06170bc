// quest_device.cuh - device building blocks of the Quest decode path (sm_103a).
//
//   score_tile    : criticality bound of a run of pages for one (sequence, kv head)
//                   ("Guide to Quest", Solution step 2).
//   topk_fast     : exact top-K of a row of score keys, ties to the lower page index
//   topk_row        ("Guide to Quest", Solution step 3); topk_row loads the row first.
//   decode_tile   : flash-decode over a run of kept pages, staged into shared memory by
//                   per-lane 16-byte cp.async copies into an mbarrier ring; writes one
//                   split-K partial (exact attention over the kept pages only: "Quest:
//                   Query-Aware Sparsity for Efficient Long-Context LLM Inference",
//                   Summary).
//   merge_splits  : log-sum-exp merge of the partials of one (sequence, kv head).
#pragma once

#include <math_constants.h>

#include "quest_internal.h"

namespace quest {

// ------------------------------------------------------------------------------------
// shared-memory map of the decode-capable kernels
// ------------------------------------------------------------------------------------
__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct SmemMap {
  size_t ring, full, empty, nvalid, wsc, st, mscale, hist, scratch, misc, bt, total;
};

// ring      : kStages x (K chunk + V chunk) of one stage of one kv head (a page, or half a
//             page at page size 32); also reused, when idle,
//             for the warp-merge buffer and for the top-K keys
// full/empty: mbarriers of the ring
// wsc       : per consumer warp, G x PS logits then weights of the stage in hand (PS
//             tokens a stage)
// st        : per consumer warp and head: running max (log2 units), running sum, rescale
// mscale    : per head, the merge scale of every split, then the merged max and sum
// Pages of a decode ring stage: a page at page size 16, half a page at 32.
__host__ __device__ constexpr int decode_sub(int P) { return P >= 32 ? P / 16 : 1; }

__host__ __device__ inline SmemMap make_smem_map(int G, int P, int topk_keys, int stp) {
  SmemMap m{};
  const int PS = P / decode_sub(P);  // tokens of a stage
  const size_t ring = (size_t)kStages * 2 * PS * kHeadDim * 2;
  const size_t red = (size_t)kConsumerWarps * G * kHeadDim * 4;
  const size_t keys = (size_t)topk_keys * 4;
  size_t a = ring;
  if (red > a) a = red;
  if (keys > a) a = keys;
  size_t o = 0;
  m.ring = o;    o = align_up(o + a, 128);
  m.full = o;    o += kStages * 8;
  m.empty = o;   o += kStages * 8;
  m.nvalid = o;  o = align_up(o + kStages * 4, 16);
  m.wsc = o;     o = align_up(o + (size_t)kConsumerWarps * G * PS * 4, 16);
  m.st = o;      o = align_up(o + (size_t)kConsumerWarps * G * 3 * 4, 16);
  m.mscale = o;  o = align_up(o + (size_t)G * (kMaxSplits + 2) * 4, 16);
  m.hist = o;    o += 256 * 4;
  m.scratch = o; o += 64 * 4;
  m.misc = o;    o += 16 * 4;
  m.bt = o;      o = align_up(o + (size_t)stp * 4, 16);
  m.total = o;
  return m;
}

// ------------------------------------------------------------------------------------
// PTX helpers
// ------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return (long long)t;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// The waiting thread may be suspended until the phase completes or a short system-defined
// time passes.  (An explicit suspend-time hint made the fused step about 3 us slower end to
// end on GB300.)
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 16-byte copy global -> shared through the load path (L2 only).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
// An arrival on `bar` once this thread's earlier cp.async copies have landed; the pending
// count is raised by one now, so the phase cannot complete before that arrival.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ uint4 ld_stream_v4(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Offset (in halves) of the box record of logical page `page` of (sequence b, kv head g):
// boxes are kept per sequence in logical page order, [B][Hkv][max_pages][2][128].
__device__ __forceinline__ size_t box_offset(const Params& p, int b, int g, int page) {
  return (((size_t)b * p.Hkv + g) * p.max_pages + page) * 2 * kHeadDim;
}

__device__ __forceinline__ uint2 lds_u2(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ float2 h2f(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// First device fault wins; later ones are dropped.
static __device__ __noinline__ void report(const Params& p, int code, int b, int page, int site) {
  if (atomicCAS(p.status, 0, code) == 0) {
    p.status[1] = b;
    p.status[2] = page;
    p.status[3] = site;
  }
}

// Tokens present in sequence b, or 0 (and a report) if seq_lens[b] is out of range.
__device__ __forceinline__ int check_len(const Params& p, int b, int L, int site) {
  if (L < 0 || (long long)L > (long long)p.max_pages * p.P) {
    report(p, QUEST_ERR_BAD_LENGTH, b, -1, site);
    return 0;
  }
  return L;
}
__device__ __forceinline__ int load_len(const Params& p, int b, int site) {
  return check_len(p, b, p.seq_lens[b], site);
}
// The step's length of sequence b from its stored length L0 (already loaded): with an
// appending chain step the new token counts if the sequence has room for it.
__device__ __forceinline__ int step_len(const Params& p, int b, int L0, int site) {
  const int L = check_len(p, b, L0, site);
  const bool app = p.chain_append && (long long)L + 1 <= (long long)p.max_pages * p.P && L == L0;
  return app ? L + 1 : L;
}

// load_len for the kernels of a chain step: when the step appends (p.chain_append), the new
// token counts if the sequence has room for it; *appended then says so.
__device__ __forceinline__ int load_len_step(const Params& p, int b, int site,
                                             bool* appended = nullptr) {
  const int L = load_len(p, b, site);
  const bool app = p.chain_append && (long long)L + 1 <= (long long)p.max_pages * p.P &&
                   L == p.seq_lens[b];
  if (appended) *appended = app;
  return app ? L + 1 : L;
}

// Bounded wait on an mbarrier phase; false (and a report) once wait_limit_ns has passed.
// The polling loop is out of line: every wait site shares one copy of it.
static __device__ __noinline__ bool mbar_wait_slow(const Params& p, uint64_t* bar, uint32_t parity,
                                            int site) {
  const long long t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > p.wait_limit_ns) {
      report(p, QUEST_ERR_TIMEOUT, -1, -1, site);
      return false;
    }
  }
}
__device__ __forceinline__ bool mbar_wait_bounded(const Params& p, uint64_t* bar,
                                                  uint32_t parity, int site) {
  return mbar_try_wait(bar, parity) || mbar_wait_slow(p, bar, parity, site);
}

// Bounded wait until *flag == target (acquire).  Gives up early once another CTA timed out.
static __device__ __noinline__ bool wait_flag_slow(const Params& p, const unsigned* flag,
                                            unsigned target, int b, int site) {
  const long long t0 = global_ns();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_u32(flag) == target) return true;
    if (ld_relaxed_s32(p.status) == QUEST_ERR_TIMEOUT) return false;
    if (global_ns() - t0 > p.wait_limit_ns) {
      report(p, QUEST_ERR_TIMEOUT, b, -1, site);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_flag_bounded(const Params& p, const unsigned* flag,
                                                  unsigned target, int b, int site) {
  return ld_acquire_u32(flag) == target || wait_flag_slow(p, flag, target, b, site);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Barrier over the NT threads that run a block-wide step: the whole CTA (__syncthreads)
// or, inside the fused kernel, the consumer warps only (named barrier 1), so that the
// producer warp keeps running ahead.
template <int NT, bool kNamed>
__device__ __forceinline__ void bsync() {
  if constexpr (kNamed) {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
  } else {
    __syncthreads();
  }
}

// Inclusive prefix sum over the NT participating threads (NT a multiple of 32, threads
// 0..NT-1).  scratch >= 32 ints.
template <int NT, bool kNamed>
__device__ __forceinline__ int block_incl_scan(int v, int* scratch) {
  constexpr int nw = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  bsync<NT, kNamed>();
  if (warp == 0) {
    int t = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    if (lane < nw) scratch[lane] = t;
  }
  bsync<NT, kNamed>();
  const int add = warp > 0 ? scratch[warp - 1] : 0;
  bsync<NT, kNamed>();
  return v + add;
}

// Arrival on a per-(b, g) counter; true in the one CTA that arrives last.  The last CTA
// sees every write the others made before arriving.
template <int NT, bool kNamed>
__device__ __forceinline__ bool arrive_last(unsigned* counter, unsigned target, int* s_flag) {
  bsync<NT, kNamed>();  // every thread's writes happen before thread 0's release
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    *s_flag = (old == target - 1u) ? 1 : 0;
  }
  bsync<NT, kNamed>();  // ... and the last one's acquire happens before every thread's reads
  const bool last = *s_flag != 0;
  bsync<NT, kNamed>();
  return last;
}

// ------------------------------------------------------------------------------------
// scoring: U(q, p) = sum_i max(q_i Kmin_i, q_i Kmax_i)  ("Guide to Quest", Solution
// step 2), evaluated in its sign-split form: per dimension the box corner that the sign of
// q_i picks (Kmax for q_i > 0, Kmin otherwise) is selected with one bitwise op on packed
// halves, widened, and multiplied (exact) into an fp32 sum.
// ------------------------------------------------------------------------------------
template <int G>
struct QueryFrag {
  float qf[G][8];   // q of each head of the group, dims [8c, 8c+8)
  uint32_t neg[G][4];  // per packed pair, 0xFFFF in the halves whose q is negative
};

template <int G>
__device__ __forceinline__ void load_query_frag(const __half* qry, int Hq, int b, int g, int c,
                                                QueryFrag<G>& f) {
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint4 raw =
        *reinterpret_cast<const uint4*>(qry + ((size_t)b * Hq + g * G + j) * kHeadDim + 8 * c);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f.neg[j][k] = ((w[k] >> 15) & 0x00010001u) * 0xFFFFu;
      const float2 v = h2f(w[k]);
      f.qf[j][2 * k] = v.x;
      f.qf[j][2 * k + 1] = v.y;
    }
  }
}

template <int G>
__device__ __forceinline__ void load_query_frag(const Params& p, int b, int g, int c,
                                                QueryFrag<G>& f) {
  load_query_frag<G>(p.q, p.Hq, b, g, c, f);
}

template <int G>
__device__ __forceinline__ float corner_dot(const QueryFrag<G>& f, int j, const uint4& mn,
                                            const uint4& mx) {
  const uint32_t a[4] = {mn.x, mn.y, mn.z, mn.w};
  const uint32_t c[4] = {mx.x, mx.y, mx.z, mx.w};
  float s = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t sel = (a[k] & f.neg[j][k]) | (c[k] & ~f.neg[j][k]);
    const float2 v = h2f(sel);
    s = fmaf(f.qf[j][2 * k], v.x, s);
    s = fmaf(f.qf[j][2 * k + 1], v.y, s);
  }
  return s;
}

// The step's new token into page ap of (b, g), by the 16 threads c = 0..15 of one half-warp
// (16 bytes of the row each): its K / V rows go to slot `aslot` of physical page `aphys`
// (-1: unmapped, reported, nothing written) and its box opens (slot 0) or widens with the
// new key.
__device__ __forceinline__ void append_token_box(const Params& p, int b, int g, int ap,
                                                 int aslot, int aphys, int c) {
  if (aphys < 0) {
    if (c == 0) report(p, QUEST_ERR_BAD_PAGE, b, ap, kSiteAppend);
    return;
  }
  const size_t o = ((size_t)b * p.Hkv + g) * kHeadDim + 8 * c;
  const uint4 knew = *reinterpret_cast<const uint4*>(p.k_new + o);
  const uint4 vnew = *reinterpret_cast<const uint4*>(p.v_new + o);
  __half* box = p.meta + box_offset(p, b, g, ap) + 8 * c;
  uint4 mn = knew, mx = knew;
  if (aslot != 0) {
    const uint4 a0 = __ldcg(reinterpret_cast<const uint4*>(box));
    const uint4 z0 = __ldcg(reinterpret_cast<const uint4*>(box + kHeadDim));
    const uint32_t a[4] = {a0.x, a0.y, a0.z, a0.w};
    const uint32_t z[4] = {z0.x, z0.y, z0.z, z0.w};
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
  *reinterpret_cast<uint4*>(box) = mn;
  *reinterpret_cast<uint4*>(box + kHeadDim) = mx;
  const size_t kv = (((size_t)aphys * p.Hkv + g) * p.P + aslot) * kHeadDim + 8 * c;
  *reinterpret_cast<uint4*>(p.k_pool + kv) = knew;
  *reinterpret_cast<uint4*>(p.v_pool + kv) = vnew;
}

// Scores of pages [p0, p0 + n_live) of (b, g) into dst.  The boxes of those pages are
// contiguous (logical page order).  Half-warp per page, 16 B of the min row and 16 B of the
// max row per lane, 4 pages in flight per half-warp.  Called by the whole block.
// PerHead: dst is query head (g * G)'s row of a [B][Hq][max_pages] array and every head of
// the group writes its own bound (rows `stride` floats apart) instead of the group maximum.
// Append (a chain step, not PerHead): page ap, if in this tile, first takes the step's new
// token (append_token_box, by the block's first half-warp, before a block barrier), and the
// boxes are then read through L2 (the read-only path may not see a box written during the
// kernel), so the page is scored with its new box, as in the one-launch kernels.
template <int G, bool PerHead = false, bool Append = false>
__device__ void score_tile(const Params& p, int b, int g, int p0, int n_live, float* dst,
                           size_t stride = 0, int ap = -1, int aslot = 0, int aphys = -1) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int hw = tid >> 4, c = tid & 15, nhw = nthr >> 4;
  if constexpr (Append && !PerHead) {
    if (ap >= p0 && ap < p0 + n_live) {  // block-uniform
      if (tid < 16) append_token_box(p, b, g, ap, aslot, aphys, c);
      __syncthreads();
    }
  }
  QueryFrag<G> f;
  load_query_frag<G>(p, b, g, c, f);
  const __half* box0 = p.meta + box_offset(p, b, g, p0) + 8 * c;
  constexpr int U = 4;
  for (int base = 0; base < n_live; base += U * nhw) {
    uint4 mn[U], mx[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = base + u * nhw + hw;
      mn[u] = make_uint4(0, 0, 0, 0);
      mx[u] = make_uint4(0, 0, 0, 0);
      if (r < n_live) {
        const __half* src = box0 + (size_t)r * 2 * kHeadDim;
        if constexpr (Append && !PerHead) {
          mn[u] = __ldcg(reinterpret_cast<const uint4*>(src));
          mx[u] = __ldcg(reinterpret_cast<const uint4*>(src + kHeadDim));
        } else {
          mn[u] = ld_stream_v4(src);
          mx[u] = ld_stream_v4(src + kHeadDim);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float best = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < G; ++j) {
        float s = corner_dot<G>(f, j, mn[u], mx[u]);
        s += __shfl_xor_sync(0xffffffffu, s, 8);
        s += __shfl_xor_sync(0xffffffffu, s, 4);
        s += __shfl_xor_sync(0xffffffffu, s, 2);
        s += __shfl_xor_sync(0xffffffffu, s, 1);
        best = fmaxf(best, s);
        if (PerHead) {
          const int r = base + u * nhw + hw;
          if (c == 0 && r < n_live) dst[(size_t)j * stride + r] = s;
        }
      }
      const int r = base + u * nhw + hw;
      if (!PerHead && c == 0 && r < n_live) dst[r] = best;
    }
  }
}

// ------------------------------------------------------------------------------------
// top-K: "Guide to Quest", Solution step 3.  Scores become order-preserving unsigned keys
// (sign flip), so the K largest scores are the K largest keys; see topk_fast below.
// ------------------------------------------------------------------------------------
constexpr int kFastBins = 4096;  // histogram bins of one selection level (12-bit digits)

__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t u = __float_as_uint(s + 0.0f);  // -0 -> +0
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Shared memory of one selection over a row of up to max_pages scores.
struct TopkSmem {
  uint32_t* keys;      // [max_pages]
  int* hist;           // [kFastBins]
};

__host__ __device__ inline size_t topk_smem_bytes(int max_pages) {
  return align_up((size_t)max_pages * 4, 16) + (size_t)kFastBins * 4;
}

// Ints of the decode ring's region that a selection inside the decode kernel needs: its
// keys and histogram, then 256 ints of scratch.
__host__ __device__ inline int select_ring_ints(int max_pages) {
  return (int)((topk_smem_bytes(max_pages) + 256 * 4) / 4);
}

__device__ inline TopkSmem topk_smem_at(unsigned char* base, int max_pages) {
  TopkSmem t;
  t.keys = reinterpret_cast<uint32_t*>(base);
  base += align_up((size_t)max_pages * 4, 16);
  t.hist = reinterpret_cast<int*>(base);
  return t;
}


// Inclusive / exclusive sum over NT threads with warp shuffles and one barrier; tot: shared
// [NW] ints of the caller's choosing.
template <int NT, bool kNamed>
__device__ __forceinline__ int block_excl_sum(int v, int* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) tot[warp] = x;
  bsync<NT, kNamed>();
  int pre = lane < warp ? tot[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
  return pre + x - v;
}


// ------------------------------------------------------------------------------------
// Exact selection of the K largest of N keys in shared memory ("Guide to Quest", Solution
// step 3; ties to the lower index), the kept indices written in ascending order.  With
// d = key - lo, the bits of d are resolved 12 at a time from the span's leading bit: each
// level builds one 4096-bin histogram of the digit of the keys still tied with the
// threshold, and one block scan from the top bin finds the bin that holds the K-th largest
// key.  The search ends when that bin is taken whole, when d is exhausted, or when the bin
// holds at most 32 keys: one warp gathers those and finds the K-th largest value among them
// by counting.  Every step is a short pass with few barriers; a shared-memory histogram of
// 4096 bins spreads the keys of a score row thinly, so its atomics rarely collide.
// hist: kFastBins ints, zero on entry (left zero); scratch: 2 * (NT / 32) + 40 ints.
// Called by threads 0..NT-1 with K < N < 65536.
// ------------------------------------------------------------------------------------
constexpr int kFewKeys = 32;  // a threshold bin this small is resolved by one warp

template <int NT, bool kNamed>
__device__ void topk_fast(const uint32_t* keys, int N, int K, uint32_t lo, uint32_t hi,
                          int* idx_out, int* hist, int* scratch) {
  constexpr int NW = NT / 32;
  constexpr int BPT = (kFastBins + NT - 1) / NT;  // bins per thread in the scan
  static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int* found = scratch + 2 * NW;  // [0] bin, [1] keys above it, [2] keys in it, [3] gathered,
                                  // [4] threshold key, [5] candidates above it
  uint32_t* cand = reinterpret_cast<uint32_t*>(found + 8);  // [kFewKeys]
  const uint32_t span = hi - lo;
  int top = span ? 32 - __clz(span) : 0;  // bits of d below `top` are not resolved yet
  uint32_t pref = 0;                      // d >> top of the keys tied with the threshold
  int need = K;                           // keys still to take among those tied
  bool whole = false, first = true;
  while (top > 0) {
    const int sh = top > 12 ? top - 12 : 0;
    const uint32_t mask = (1u << (top - sh)) - 1u;
#pragma unroll 1
    for (int i = tid; i < N; i += NT) {
      const uint32_t d = keys[i] - lo;
      if (first || (d >> top) == pref) atomicAdd(&hist[(d >> sh) & mask], 1);
    }
    bsync<NT, kNamed>();
    // thread t holds bins [low, low + BPT), low = kFastBins - (t + 1) * BPT (read, cleared)
    const int low = kFastBins - (tid + 1) * BPT;
    int c[BPT];
    if constexpr (BPT % 4 == 0) {
#pragma unroll
      for (int q4 = 0; q4 < BPT / 4; ++q4) {
        int4* h4 = reinterpret_cast<int4*>(hist + low) + q4;
        const int4 x = *h4;
        c[4 * q4] = x.x;
        c[4 * q4 + 1] = x.y;
        c[4 * q4 + 2] = x.z;
        c[4 * q4 + 3] = x.w;
        *h4 = make_int4(0, 0, 0, 0);
      }
    } else {
#pragma unroll
      for (int k = 0; k < BPT; ++k) {
        c[k] = 0;
        if (low + k >= 0) {
          c[k] = hist[low + k];
          hist[low + k] = 0;
        }
      }
    }
    int tot = 0;
#pragma unroll
    for (int k = 0; k < BPT; ++k) tot += c[k];
    const int excl = block_excl_sum<NT, kNamed>(tot, scratch);
    if (excl < need && need <= excl + tot) {
      int acc = excl;
#pragma unroll
      for (int k = BPT - 1; k >= 0; --k) {
        if (acc < need && acc + c[k] >= need) {
          found[0] = low + k;
          found[1] = acc;
          found[2] = c[k];
        }
        acc += c[k];
      }
    }
    if (tid == 0) found[3] = 0;
    bsync<NT, kNamed>();
    // (found[] is next written after the next level's histogram and its barrier)
    const int bstar = found[0], above = found[1], cnt = found[2];
    need -= above;
    pref = (pref << (top - sh)) | (uint32_t)bstar;
    top = sh;
    first = false;
    if (cnt == need) {
      whole = true;
      break;
    }
    if (top == 0) break;
    if (cnt <= kFewKeys) {
#pragma unroll 1
      for (int i = tid; i < N; i += NT) {
        const uint32_t v = keys[i];
        if (((v - lo) >> top) == pref) cand[atomicAdd(&found[3], 1)] = v;
      }
      bsync<NT, kNamed>();
      if (warp == 0) {
        const uint32_t x = lane < cnt ? cand[lane] : 0u;
        int gt = 0, eq = 0;
        for (int q = 0; q < cnt; ++q) {
          const uint32_t y = __shfl_sync(0xffffffffu, x, q);
          gt += y > x;
          eq += y == x;
        }
        if (lane < cnt && gt < need && need <= gt + eq) {  // x is the need-th largest value
          found[4] = (int)x;
          found[5] = gt;
        }
      }
      bsync<NT, kNamed>();
      need -= found[5];
      pref = (uint32_t)found[4] - lo;
      top = 0;
      break;
    }
  }
  // kept: (d >> top) > pref; tied: == pref, the `need` lowest indices of them (all if whole).
  // Thread t takes indices [t*R, t*R + R) (R odd, so that a warp's 32 runs fall in 32
  // different shared-memory banks): it counts its kept and tied keys, one block scan gives
  // its place in the output and its share of the ties, and a second look at its run writes
  // them out in ascending order.  Short loops, no unrolling: this runs once per selection
  // and its code is fetched cold.
  const int R = ((N + NT - 1) / NT) | 1;
  const int i0 = min(N, tid * R), i1 = min(N, i0 + R);
  const uint32_t tsh = top >= 32 ? 31u : (uint32_t)top;  // top < 32 here; keeps the shift defined
  int nk = 0, nt = 0;
#pragma unroll 1
  for (int i = i0; i < i1; ++i) {
    const uint32_t h = (keys[i] - lo) >> tsh;
    nk += h > pref;
    nt += h == pref;
  }
  // packed counts: both are below 2^16 (N < 65536).  Ties are taken in index order, so the
  // threads before this one took min(their ties, need) of them: one scan places everything.
  const int pre = block_excl_sum<NT, kNamed>((nk << 16) | nt, scratch);
  const int tie_before = pre & 0xffff;
  int take = whole ? nt : max(0, min(nt, need - tie_before));
  int pos = (pre >> 16) + (whole ? tie_before : min(tie_before, need));
#pragma unroll 1
  for (int i = i0; i < i1; ++i) {
    const uint32_t h = (keys[i] - lo) >> tsh;
    bool keep = h > pref;
    if (h == pref && take > 0) {
      keep = true;
      --take;
    }
    if (keep) idx_out[pos++] = i;
  }
  bsync<NT, kNamed>();
}

// One row of N scores in global memory (possibly written by another CTA): keys into shared
// memory with their range, then topk_fast.  N <= 64 * NT.  In a row longer than K, the
// first `sink` and last `local` pages get the largest key, so they are always kept.
template <int NT, bool kNamed>
__device__ void topk_row(const float* row, int N, int K, int sink, int local, int* idx_out,
                         int* count_out, const TopkSmem& t, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  if (N <= K) {
    for (int r = tid; r < K; r += NT) idx_out[r] = r < N ? r : -1;
    if (tid == 0) *count_out = N;
    return;
  }
  uint32_t lo = 0xffffffffu, hi = 0u;
  const int rounds = (N + NT - 1) / NT;
  for (int r0 = 0; r0 < rounds; r0 += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = (r0 + u) * NT + tid;
      v[u] = i < N ? __ldcg(row + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = (r0 + u) * NT + tid;
      if (i < N) {
        const bool forced = N > K && (i < sink || i >= N - local);
        const uint32_t k = forced ? 0xffffffffu : score_key(v[u]);
        t.keys[i] = k;
        lo = min(lo, k);
        hi = max(hi, k);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  if (lane == 0) {
    scratch[warp] = (int)lo;
    scratch[NW + warp] = (int)hi;
  }
  for (int i = tid; i < kFastBins / 4; i += NT)
    reinterpret_cast<int4*>(t.hist)[i] = make_int4(0, 0, 0, 0);
  bsync<NT, kNamed>();
  lo = 0xffffffffu;
  hi = 0u;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    lo = min(lo, (uint32_t)scratch[w]);
    hi = max(hi, (uint32_t)scratch[NW + w]);
  }
  topk_fast<NT, kNamed>(t.keys, N, K, lo, hi, idx_out, t.hist, scratch);
  if (tid == 0) *count_out = K;
}



// ------------------------------------------------------------------------------------
// decode: one ring stage (P tokens here: a page, or half a page at page size 32) of one
// kv head against the G query heads of its group, in one warp.
// Lane l owns dims [4l, 4l+4).  Logits: 16 (head, token) partial dot products per chunk
// are summed across the warp with a transposing butterfly (15 shuffles leave each lane
// pair holding one full logit).  Softmax: running max / sum per head (log2 domain).
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float transpose_reduce16(float (&v)[16], int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 16;
    const float send = hi ? v[i] : v[i + 8];
    const float keep = hi ? v[i + 8] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 8;
    const float send = hi ? v[i] : v[i + 4];
    const float keep = hi ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 4;
    const float send = hi ? v[i] : v[i + 2];
    const float keep = hi ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  {
    const bool hi = lane & 2;
    const float send = hi ? v[0] : v[1];
    const float keep = hi ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  return v[0];
}
// Which of the 16 values lane `lane` holds after transpose_reduce16.
__device__ __forceinline__ int reduced_index(int lane) {
  return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

template <int G, int P>
__device__ __forceinline__ void page_update(const float (&qf)[G][4], float (&acc)[G][4],
                                            const __half* Ks, const __half* Vs, int nv,
                                            float* sc, float* st, int lane) {
  constexpr int TC = 16 / G;  // tokens per chunk of 16 (head, token) values
  constexpr int NCH = P / TC;
  // 1. logits (log2 units; q was pre-scaled by log2(e)/sqrt(d)) into sc[G][P]
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    float v[16];
#pragma unroll
    for (int tj = 0; tj < TC; ++tj) {
      const int t = ch * TC + tj;
      const uint2 raw = lds_u2(Ks + t * kHeadDim + 4 * lane);
      const float2 k01 = h2f(raw.x), k23 = h2f(raw.y);
#pragma unroll
      for (int j = 0; j < G; ++j)
        v[j * TC + tj] =
            fmaf(qf[j][0], k01.x, fmaf(qf[j][1], k01.y, fmaf(qf[j][2], k23.x, qf[j][3] * k23.y)));
    }
    const float r = transpose_reduce16(v, lane);
    const int vi = reduced_index(lane);
    const int j = vi / TC, t = ch * TC + vi % TC;
    if ((lane & 1) == 0) sc[j * P + t] = (t < nv) ? r : -CUDART_INF_F;
  }
  __syncwarp();
  // 2. per head: tile max, new running max, weights, tile sum
  constexpr int GP = G * P;
  constexpr int NV = GP >= 32 ? GP / 32 : 1;
  constexpr int SEG = P < 32 ? P : 32;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int vidx = GP >= 32 ? lane + 32 * i : (lane % GP);
    const int j = vidx / P, t = vidx % P;
    const float x = sc[j * P + t];
    float mt = x;
#pragma unroll
    for (int o = SEG / 2; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
    const float m_old = st[j * 3 + 0];
    const float m_new = fmaxf(m_old, mt);
    const float w = (x == -CUDART_INF_F) ? 0.f : exp2f(x - m_new);
    float sum = w;
#pragma unroll
    for (int o = SEG / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    __syncwarp();
    sc[j * P + t] = w;
    if (t == 0 && (GP >= 32 || lane < GP)) {
      const float alpha = (m_new == -CUDART_INF_F) ? 1.f : exp2f(m_old - m_new);
      st[j * 3 + 1] = st[j * 3 + 1] * alpha + sum;
      st[j * 3 + 0] = m_new;
      st[j * 3 + 2] = alpha;
    }
    __syncwarp();
  }
  // 3. acc = acc * alpha + sum_t w_t v_t  (tokens past the end contribute nothing, even junk)
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const float a = st[j * 3 + 2];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] *= a;
  }
#pragma unroll
  for (int t4 = 0; t4 < P / 4; ++t4) {
    float vv[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = 4 * t4 + u;
      const uint2 raw = lds_u2(Vs + t * kHeadDim + 4 * lane);
      const float2 a = h2f(raw.x), c = h2f(raw.y);
      const bool live = t < nv;
      vv[u][0] = live ? a.x : 0.f;
      vv[u][1] = live ? a.y : 0.f;
      vv[u][2] = live ? c.x : 0.f;
      vv[u][3] = live ? c.y : 0.f;
    }
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float4 w4 = *reinterpret_cast<const float4*>(sc + j * P + 4 * t4);
      const float ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[j][k] = fmaf(ws[u], vv[u][k], acc[j][k]);
    }
  }
  __syncwarp();
}

// Flash-decode over kept pages r0 .. r0 + n_tile - 1 of (b, g) (ranks in sel_row, or
// logical pages r0.. when sel_row is null) and write this work item's split-K partial.
// pc: pages this CTA has already pushed through its ring (mbarrier phase bookkeeping).
// Called by the whole block (kDecodeThreads threads): warps 0..7 compute, warp 8 issues
// the copies.  n_tile >= 1.
template <int G, int P>
__device__ void decode_tile(const Params& p, unsigned char* smem, const SmemMap& m, int b,
                            int g, int split, int r0, int n_tile, int L, int N_b,
                            const int* sel_row, uint32_t pc) {
  // A ring stage holds PS tokens of K and of V: a whole page at page size 16, half a page
  // at 32 (each page then fills SUB consecutive stages), so that the ring stays 64 KiB and
  // three CTAs share an SM at either page size.
  constexpr int SUB = decode_sub(P), PS = P / SUB;
  constexpr uint32_t kChunk = PS * kHeadDim * 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  unsigned char* ring = smem + m.ring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.full);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + m.empty);
  int* nvalid_s = reinterpret_cast<int*>(smem + m.nvalid);
  float* st_all = reinterpret_cast<float*>(smem + m.st);
  float acc[G][4];
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[j][k] = 0.f;

  if (warp == kConsumerWarps) {
    // ---- producer warp: resolve pages 32 at a time, then fill their stages in order.  A
    // page's K and V chunks lie anywhere in the pool: the whole warp copies them, 16 bytes a
    // lane per instruction (the same rate as one bulk copy per chunk measured here, with no
    // byte count to arm), and the stage completes on its full barrier through the copies'
    // own arrivals (each lane's, plus one plain arrival of lane 0).
    const size_t chunk_elems = (size_t)P * kHeadDim;
    for (int base = 0; base < n_tile; base += 32) {
      const int r = base + lane;
      int nv = 0, phys = 0;
      if (r < n_tile) {
        int lp;
        if (p.chain_pairs) {  // the top-K kernel resolved the physical page already
          const int2 e = __ldcg(reinterpret_cast<const int2*>(p.sel_pair) +
                                ((size_t)b * p.Hkv + g) * p.top_k + r0 + r);
          lp = e.x;
          phys = e.y;
        } else {
          lp = sel_row ? sel_row[r0 + r] : r0 + r;  // (global, or this CTA's shared memory)
        }
        if (lp < 0 || lp >= N_b) {
          report(p, QUEST_ERR_BAD_SELECTION, b, lp, kSiteSelection);
        } else {
          if (!p.chain_pairs) phys = p.block_table[(size_t)b * p.max_pages + lp];
          if (phys < 0 || phys >= p.num_phys) {
            report(p, QUEST_ERR_BAD_PAGE, b, lp, kSiteDecode);
            phys = 0;
          } else {
            nv = min(P, L - lp * P);
          }
        }
      }
      const int cnt = min(32, n_tile - base);
#pragma unroll 1
      for (int j = 0; j < cnt; ++j) {
        const int nvj0 = __shfl_sync(0xffffffffu, nv, j);
        const int phj = __shfl_sync(0xffffffffu, phys, j);
#pragma unroll 1
        for (int h = 0; h < SUB; ++h) {
          const int nvj = max(0, min(PS, nvj0 - h * PS));
          const uint32_t k = pc + (uint32_t)((base + j) * SUB + h);
          const int stage = (int)(k % kStages);
          const uint32_t par = ((k / kStages) & 1u) ^ 1u;
          int ok = 1;
          if (lane == 0) ok = mbar_wait_bounded(p, &empty[stage], par, kSiteWaitSlot);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          __syncwarp();  // the stage's last reads happen before any lane's copy into it
          const int nvs = ok ? nvj : 0;
          if (lane == 0) nvalid_s[stage] = nvs;
          if (nvs > 0) {  // warp-uniform
            const size_t off = (((size_t)phj * p.Hkv + g) * chunk_elems +
                                (size_t)h * PS * kHeadDim) * 2 + 16 * lane;
            const unsigned char* ks = reinterpret_cast<const unsigned char*>(p.k_pool) + off;
            const unsigned char* vs = reinterpret_cast<const unsigned char*>(p.v_pool) + off;
            unsigned char* dst = ring + (size_t)stage * 2 * kChunk + 16 * lane;
#pragma unroll
            for (int u = 0; u < (int)kChunk / 512; ++u) cp_async16(dst + 512 * u, ks + 512 * u);
#pragma unroll
            for (int u = 0; u < (int)kChunk / 512; ++u)
              cp_async16(dst + kChunk + 512 * u, vs + 512 * u);
            cp_async_arrive(&full[stage]);
            __syncwarp();  // every lane's pending arrival is counted before lane 0's
          }
          if (lane == 0) mbar_arrive(&full[stage]);
          __syncwarp();
        }
      }
    }
  } else {
    // ---- consumer warps
    float qf[G][4];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint2 raw = *reinterpret_cast<const uint2*>(
          p.q + ((size_t)b * p.Hq + g * G + j) * kHeadDim + 4 * lane);
      const float2 a = h2f(raw.x), c = h2f(raw.y);
      qf[j][0] = a.x * p.qscale;
      qf[j][1] = a.y * p.qscale;
      qf[j][2] = c.x * p.qscale;
      qf[j][3] = c.y * p.qscale;
    }
    float* sc = reinterpret_cast<float*>(smem + m.wsc) + warp * G * PS;
    float* st = st_all + warp * G * 3;
    if (lane < G) {
      st[lane * 3 + 0] = -CUDART_INF_F;
      st[lane * 3 + 1] = 0.f;
      st[lane * 3 + 2] = 1.f;
    }
    __syncwarp();
    for (int r = warp; r < n_tile * SUB; r += kConsumerWarps) {
      const uint32_t k = pc + (uint32_t)r;
      const int stage = (int)(k % kStages);
      const uint32_t par = (k / kStages) & 1u;
      const bool ok = mbar_wait_bounded(p, &full[stage], par, kSiteWaitStage);
      const int nv = ok ? nvalid_s[stage] : 0;
      if (nv > 0) {
        const __half* Ks = reinterpret_cast<const __half*>(ring + (size_t)stage * 2 * kChunk);
        page_update<G, PS>(qf, acc, Ks, Ks + PS * kHeadDim, nv, sc, st, lane);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
  }
  __syncthreads();  // ring idle: every copy of this tile has landed and been read

  // ---- merge the 8 warps' states into this work item's partial
  float* red = reinterpret_cast<float*>(ring);  // [warp][G][128]
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int j = 0; j < G; ++j)
      *reinterpret_cast<float4*>(red + ((size_t)warp * G + j) * kHeadDim + 4 * lane) =
          make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
  }
  __syncthreads();
  for (int o = tid; o < G * kHeadDim; o += blockDim.x) {
    const int j = o / kHeadDim, i = o % kHeadDim;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, st_all[(w * G + j) * 3]);
    float A = 0.f, Ls = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = st_all[(w * G + j) * 3];
      if (mw != -CUDART_INF_F) {
        const float s = exp2f(mw - M);
        A = fmaf(red[((size_t)w * G + j) * kHeadDim + i], s, A);
        Ls = fmaf(st_all[(w * G + j) * 3 + 1], s, Ls);
      }
    }
    const size_t slot = (size_t)(b * p.Hq + g * G + j) * p.n_splits + split;
    p.part_acc[slot * kHeadDim + i] = A;
    if (i == 0) {
      p.part_ml[slot * 2] = M;
      p.part_ml[slot * 2 + 1] = Ls;
    }
  }
  fence_proxy_async_smem();  // generic use of the ring (the merge buffer) is ordered before
                             // any later bulk copy into it
}

// Log-sum-exp merge of the first n_live partials of every head of (b, g) into out / lse.
// msc: shared [G][kMaxSplits + 2] floats.  Called by threads 0..NT-1.
template <int G, int NT, bool kNamed>
__device__ void merge_splits(const Params& p, float* msc, int b, int g, int n_live) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp < G) {
    const int h = g * G + warp;
    const float* ml = p.part_ml + (size_t)(b * p.Hq + h) * p.n_splits * 2;
    float* row = msc + warp * (kMaxSplits + 2);
    float M = -CUDART_INF_F;
    for (int s = lane; s < n_live; s += 32) M = fmaxf(M, __ldcg(ml + 2 * s));
    M = warp_max(M);
    float Ls = 0.f;
    for (int s = lane; s < n_live; s += 32) {
      const float ms = __ldcg(ml + 2 * s);
      const float f = (ms == -CUDART_INF_F) ? 0.f : exp2f(ms - M);
      row[s] = f;
      Ls = fmaf(__ldcg(ml + 2 * s + 1), f, Ls);
    }
    Ls = warp_sum(Ls);
    if (lane == 0) {
      row[kMaxSplits] = M;
      row[kMaxSplits + 1] = Ls;
    }
  }
  bsync<NT, kNamed>();
  for (int o = tid; o < G * kHeadDim; o += NT) {
    const int j = o / kHeadDim, i = o % kHeadDim;
    const int h = g * G + j;
    const float* row = msc + j * (kMaxSplits + 2);
    const float Ls = row[kMaxSplits + 1];
    const float* accp = p.part_acc + (size_t)(b * p.Hq + h) * p.n_splits * kHeadDim + i;
    float A = 0.f;
    int s = 0;
    for (; s + 8 <= n_live; s += 8) {  // 8 independent loads in flight
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = row[s + u] != 0.f ? __ldcg(accp + (size_t)(s + u) * kHeadDim) : 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) A = fmaf(v[u], row[s + u], A);
    }
    for (; s < n_live; ++s) {
      const float f = row[s];
      if (f != 0.f) A = fmaf(__ldcg(accp + (size_t)s * kHeadDim), f, A);
    }
    p.out[(size_t)(b * p.Hq + h) * kHeadDim + i] = __float2half_rn(Ls > 0.f ? A / Ls : 0.f);
    if (i == 0 && p.lse)
      p.lse[b * p.Hq + h] =
          Ls > 0.f ? (row[kMaxSplits] + log2f(Ls)) * 0.69314718055994531f : -CUDART_INF_F;
  }
  bsync<NT, kNamed>();
}

// Shared prologue of the decode-capable kernels: ring barriers.
__device__ __forceinline__ void init_ring(unsigned char* smem, const SmemMap& m) {
  if (threadIdx.x == 0) {
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + m.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + m.empty);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
}

}  // namespace quest
