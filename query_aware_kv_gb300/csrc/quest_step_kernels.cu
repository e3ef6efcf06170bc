// quest_step_kernels.cu - the three steps of a Quest decode step as separate launches:
// page scoring, top-K selection, split-K sparse (or dense) flash-decode, whose work items
// can also take their pair's top-K themselves (two launches per step).
#include <mutex>
#include <unordered_map>

#include "quest_device.cuh"

namespace quest {

size_t decode_smem_bytes(int G, int P, int topk_keys, int score_tile_pages) {
  return make_smem_map(G, P, topk_keys, score_tile_pages).total;
}

// Raise the dynamic shared-memory cap of `fn` once per device.
cudaError_t ensure_smem(const void* fn, size_t bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, size_t> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  auto& m = done[dev & 63];
  auto it = m.find(fn);
  if (it != m.end() && it->second >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) m[fn] = bytes;
  return e;
}

// ---------------------------------------------------------------- scoring
// grid (n_score_tiles, B*Hkv), 256 threads.
// PerHead: scores is [B][Hq][max_pages], one row per query head (quest_estimate_heads).
// Append: a chain step that also writes its new token (a variant of its own, so that the
// plain estimate keeps its registers).
template <int G, bool PerHead, bool Append>
__global__ void __launch_bounds__(kConsumerThreads) estimate_kernel(Params p) {
  pdl_wait();
  const int tile = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  bool appended = false;
  const int L = Append ? load_len_step(p, b, kSiteScore, &appended) : load_len(p, b, kSiteScore);
  const int N = (L + p.P - 1) / p.P;
  const int p0 = tile * p.score_tile_pages;
  const int np = min(p.score_tile_pages, p.max_pages - p0);
  const int n_live = max(0, min(N - p0, np));
  const size_t first_row = PerHead ? (size_t)b * p.Hq + (size_t)g * G : (size_t)bg;
  float* row = p.scores + first_row * p.max_pages + p0;
  for (int j = 0; j < (PerHead ? G : 1); ++j)
    for (int i = n_live + (int)threadIdx.x; i < np; i += blockDim.x)
      row[(size_t)j * p.max_pages + i] = -CUDART_INF_F;
  // a chain step's new token goes in with the scoring of its page
  int ap = -1, aslot = 0, aphys = -1;
  if (Append && appended) {
    ap = (L - 1) / p.P;
    aslot = (L - 1) % p.P;
    if (ap >= p0 && ap < p0 + n_live) {
      const int phys = p.block_table[(size_t)b * p.max_pages + ap];
      aphys = (phys >= 0 && phys < p.num_phys) ? phys : -1;
    }
  } else if (Append && (long long)L == (long long)p.max_pages * p.P && tile == 0 && g == 0 &&
             threadIdx.x == 0) {
    report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);  // no room for the new token
  }
  if (n_live > 0) {
    if constexpr (Append)
      score_tile<G, false, true>(p, b, g, p0, n_live, row, (size_t)p.max_pages, ap, aslot, aphys);
    else
      score_tile<G, PerHead>(p, b, g, p0, n_live, row, (size_t)p.max_pages);
  }
}

// ---------------------------------------------------------------- top-K
// grid (B*Hkv), kTopkThreads threads; dynamic smem: keys of one score row + histogram +
// scratch.  The selection is bound by instruction latency (dependent steps per key, block
// barriers between passes), so a row gets 16 warps: fewer keys per thread, and four warps
// per scheduler to hide each other's waits.
constexpr int kTopkThreads = 512;

// chain_pairs (a chain decode call): the kept pages also go out with their physical pages
// ((logical, physical) in sel_pair, physical -1 if unmapped), so that the decode kernel
// starts its copies one dependent load earlier; the block table row is read into shared
// memory alongside the length and the scores.  Dynamic smem: topk_smem_bytes(max_pages)
// + 256 ints, + max_pages + top_k ints with chain_pairs.
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char sm[];
  pdl_wait();
  const int bg = blockIdx.x, b = bg / p.Hkv;
  const int tid = threadIdx.x;
  int* scratch = reinterpret_cast<int*>(sm + topk_smem_bytes(p.max_pages));  // [256]
  int* bt_s = scratch + 256;                                                  // [max_pages]
  int* sel_s = bt_s + p.max_pages;                                            // [top_k]
  const int L0 = p.seq_lens[b];
  if (p.chain_pairs)
    for (int i = tid; i < p.max_pages; i += kTopkThreads)
      bt_s[i] = p.block_table[(size_t)b * p.max_pages + i];
  const int L = step_len(p, b, L0, kSiteTopk);
  const int N = (L + p.P - 1) / p.P;
  int* idx_g = p.sel_idx + (size_t)bg * p.top_k;
  topk_row<kTopkThreads, false>(p.scores + (size_t)bg * p.max_pages, N, p.top_k,
                                p.sink_pages, p.local_pages, p.chain_pairs ? sel_s : idx_g,
                                p.sel_count + bg, topk_smem_at(sm, p.max_pages), scratch);
  if (p.chain_pairs) {
    __syncthreads();  // the selection and the block table row are in shared memory
    int2* pr = reinterpret_cast<int2*>(p.sel_pair) + (size_t)bg * p.top_k;
    for (int r = tid; r < p.top_k; r += kTopkThreads) {
      const int lp = sel_s[r];
      int ph = -1;
      if (lp >= 0 && lp < N) {
        ph = bt_s[lp];
        if (ph < 0 || ph >= p.num_phys) ph = -1;
      }
      idx_g[r] = lp;
      pr[r] = make_int2(lp, ph);
    }
  }
}

// Group-level selection, union form ("Guide to Quest", Best Practices step 2): each query
// head of the group keeps its own top-K pages (the selection above, one row of the
// per-head scores at a time), the kv head keeps their union, written in ascending order
// into a row of `row_cap` entries.  grid (B*Hkv), 256 threads.
__global__ void __launch_bounds__(kConsumerThreads) topk_union_kernel(Params p, int row_cap) {
  extern __shared__ __align__(16) unsigned char sm[];
  pdl_wait();
  const int tid = threadIdx.x;
  const int bg = blockIdx.x, b = bg / p.Hkv, g = bg % p.Hkv;
  const int G = p.Hq / p.Hkv, K = p.top_k;
  const int L = load_len(p, b, kSiteTopk);
  const int N = (L + p.P - 1) / p.P;
  int* idx_out = p.sel_idx + (size_t)bg * row_cap;
  if (N <= K) {
    for (int r = tid; r < row_cap; r += kConsumerThreads) idx_out[r] = r < N ? r : -1;
    if (tid == 0) p.sel_count[bg] = N;
    return;
  }
  const TopkSmem t = topk_smem_at(sm, p.max_pages);
  int* scratch = reinterpret_cast<int*>(sm + topk_smem_bytes(p.max_pages));  // [256]
  int* list = scratch + 256;                                                   // [K]
  uint32_t* ubits = reinterpret_cast<uint32_t*>(list + K);                     // [nw]
  const int nw = (N + 31) >> 5;
  for (int i = tid; i < nw; i += kConsumerThreads) ubits[i] = 0u;
  for (int j = 0; j < G; ++j) {
    __syncthreads();
    const float* row = p.scores + ((size_t)b * p.Hq + (size_t)g * G + j) * p.max_pages;
    topk_row<kConsumerThreads, false>(row, N, K, 0, 0, list, scratch + 255, t, scratch);
    __syncthreads();
    for (int r = tid; r < K; r += kConsumerThreads)
      atomicOr(&ubits[list[r] >> 5], 1u << (list[r] & 31));
  }
  __syncthreads();
  // the union in ascending order: per-thread word counts, one block scan, then the bits
  const int wpt = (nw + kConsumerThreads - 1) / kConsumerThreads;
  const int w0 = min(nw, tid * wpt), w1 = min(nw, w0 + wpt);
  int n = 0;
  for (int w = w0; w < w1; ++w) n += __popc(ubits[w]);
  int pos = block_excl_sum<kConsumerThreads, false>(n, scratch + 32);
  for (int w = w0; w < w1; ++w) {
    uint32_t A = ubits[w];
    while (A) {
      const int bit = __ffs(A) - 1;
      A &= A - 1u;
      idx_out[pos++] = w * 32 + bit;
    }
  }
  __syncthreads();
  if (tid == kConsumerThreads - 1) scratch[48] = pos;  // the last thread ends at the total
  __syncthreads();
  const int total = scratch[48];
  for (int r = total + tid; r < row_cap; r += kConsumerThreads) idx_out[r] = -1;
  if (tid == 0) p.sel_count[bg] = total;
}

// ---------------------------------------------------------------- decode
// grid (n_splits, B*Hkv), kDecodeThreads threads.  Work item `split` of (b, g) attends
// over kept pages [split*pps, split*pps + pps); the last work item of (b, g) to finish
// merges the partials.
template <int G, int P>
__global__ void __launch_bounds__(kDecodeThreads) decode_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemMap m = make_smem_map(G, P, p.chain_select ? select_ring_ints(p.max_pages) : 0, 0);
  init_ring(smem, m);
  pdl_wait();
  const int split = blockIdx.x, bg = blockIdx.y;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  // the length and the selection's count are independent: both loads go out together
  const int L0 = p.seq_lens[b];
  const int c0 = (p.dense || p.chain_select) ? 0 : p.sel_count[bg];
  const int L = step_len(p, b, L0, kSiteDecode);
  const int N = (L + P - 1) / P;
  int count = N;
  const int* sel_row = nullptr;
  if (p.chain_select) {
    // A chain step without a top-K kernel: every work item of the pair takes the pair's
    // top-K over the scores itself (the same arithmetic, so the same pages in every one),
    // in the ring's space before the ring is used, and keeps the kept pages in shared
    // memory; work item 0 also writes the caller's copy.
    int* sel_s = reinterpret_cast<int*>(smem + m.total);  // [top_k]
    int* cnt_s = reinterpret_cast<int*>(smem + m.misc) + 8;
    unsigned char* ring = smem + m.ring;
    topk_row<kDecodeThreads, false>(p.scores + (size_t)bg * p.max_pages, N, p.top_k,
                                    p.sink_pages, p.local_pages, sel_s, cnt_s,
                                    topk_smem_at(ring, p.max_pages),
                                    reinterpret_cast<int*>(ring + topk_smem_bytes(p.max_pages)));
    __syncthreads();
    count = *cnt_s;
    sel_row = sel_s;
    if (split == 0) {
      for (int r = threadIdx.x; r < p.top_k; r += kDecodeThreads)
        p.sel_idx[(size_t)bg * p.top_k + r] = sel_s[r];
      if (threadIdx.x == 0) p.sel_count[bg] = count;
    }
  } else if (!p.dense) {
    count = c0;
    const int cap = min(p.top_k, N);
    if (count < 0 || count > cap) {
      if (threadIdx.x == 0 && split == 0) report(p, QUEST_ERR_BAD_SELECTION, b, count, kSiteSelection);
      count = max(0, min(count, cap));
    }
    sel_row = p.sel_idx + (size_t)bg * p.top_k;
  }
  const int r0 = split * p.pps;
  const int n_tile = max(0, min(count - r0, p.pps));
  if (n_tile > 0) decode_tile<G, P>(p, smem, m, b, g, split, r0, n_tile, L, N, sel_row, 0u);
  int* misc = reinterpret_cast<int*>(smem + m.misc);
  if (arrive_last<kDecodeThreads, false>(&p.decode_arrive[bg], (unsigned)p.n_splits, misc)) {
    merge_splits<G, kDecodeThreads, false>(p, reinterpret_cast<float*>(smem + m.mscale), b, g,
                                           (count + p.pps - 1) / p.pps);
    if (threadIdx.x == 0) {
      p.decode_arrive[bg] = 0u;
      // a chain step that appended: once every kv head of the sequence has merged (so every
      // work item of it has read its length), the length takes the new token
      if (p.chain_append) {
        __threadfence();
        if (atomicAdd(&p.seq_done[b], 1u) == (unsigned)p.Hkv - 1u) {
          p.seq_done[b] = 0u;
          const int L0 = p.seq_lens[b];
          if (L0 >= 0 && (long long)L0 + 1 <= (long long)p.max_pages * P) {
            const int phys = p.block_table[(size_t)b * p.max_pages + L0 / P];
            if (phys >= 0 && phys < p.num_phys) p.seq_lens[b] = L0 + 1;
          }
        }
      }
    }
  }
}

template <int G>
static const void* estimate_fn(bool per_head, bool append) {
  if (per_head) return (const void*)estimate_kernel<G, true, false>;
  return append ? (const void*)estimate_kernel<G, false, true>
                : (const void*)estimate_kernel<G, false, false>;
}

template <int G, int P>
static const void* decode_fn() { return (const void*)decode_kernel<G, P>; }

static const void* pick_estimate(int G, bool per_head, bool append) {
  switch (G) {
    case 1: return estimate_fn<1>(per_head, append);
    case 2: return estimate_fn<2>(per_head, append);
    case 4: return estimate_fn<4>(per_head, append);
    default: return estimate_fn<8>(per_head, append);
  }
}

static const void* pick_decode(int G, int P) {
  if (P == 16) {
    switch (G) {
      case 1: return decode_fn<1, 16>();
      case 2: return decode_fn<2, 16>();
      case 4: return decode_fn<4, 16>();
      default: return decode_fn<8, 16>();
    }
  }
  switch (G) {
    case 1: return decode_fn<1, 32>();
    case 2: return decode_fn<2, 32>();
    case 4: return decode_fn<4, 32>();
    default: return decode_fn<8, 32>();
  }
}

cudaError_t launch_estimate(const Params& p, int G, bool per_head, cudaStream_t s) {
  const void* fn = pick_estimate(G, per_head, !per_head && p.chain_append);
  const size_t smem = 0;
  Params pp = p;
  void* args[] = {&pp};
  return launch_pdl(fn, dim3(p.n_score_tiles, p.B * p.Hkv), dim3(kConsumerThreads), smem, s,
                    args);
}

cudaError_t launch_topk_union(const Params& p, int row_cap, cudaStream_t s) {
  const void* fn = (const void*)topk_union_kernel;
  const size_t smem = topk_smem_bytes(p.max_pages) + 256 * 4 + (size_t)p.top_k * 4 +
                      (size_t)((p.max_pages + 31) / 32) * 4;
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  Params pp = p;
  int rc = row_cap;
  void* args[] = {&pp, &rc};
  return launch_pdl(fn, dim3(p.B * p.Hkv), dim3(kConsumerThreads), smem, s, args);
}

cudaError_t launch_topk(const Params& p, cudaStream_t s) {
  const void* fn = (const void*)topk_kernel;
  const size_t smem = topk_smem_bytes(p.max_pages) + 256 * 4 +
                      (p.chain_pairs ? ((size_t)p.max_pages + p.top_k) * 4 : 0);
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  Params pp = p;
  void* args[] = {&pp};
  return launch_pdl(fn, dim3(p.B * p.Hkv), dim3(kTopkThreads), smem, s, args);
}

cudaError_t launch_decode(const Params& p, int G, cudaStream_t s) {
  const void* fn = pick_decode(G, p.P);
  const size_t smem = p.chain_select ? decode_smem_bytes(G, p.P, select_ring_ints(p.max_pages), 0) +
                                           align_up((size_t)p.top_k * 4, 16)
                                     : decode_smem_bytes(G, p.P, 0, 0);
  cudaError_t e = ensure_smem(fn, smem);
  if (e != cudaSuccess) return e;
  Params pp = p;
  void* args[] = {&pp};
  return launch_pdl(fn, dim3(p.n_splits, p.B * p.Hkv), dim3(kDecodeThreads), smem, s, args);
}

}  // namespace quest
