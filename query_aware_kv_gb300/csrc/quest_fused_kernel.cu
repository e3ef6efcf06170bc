// quest_fused_kernel.cu - a whole Quest decode step (score, select, attend) in one
// persistent launch.
//
// "Guide to Quest", Best Practices step 3 suggests fusing the bound estimation with the
// page gather so that no host orchestration sits between the phases.  Here every resident
// CTA takes work items from a queue in the workspace:
//   items [0, B*Hkv*n_score_tiles)   scoring tiles, (b, g)-major
//   items [.., + B*Hkv*n_splits)     split-K decode items, (b, g)-major
// The CTA that finishes the last scoring tile of (b, g) runs that (b, g)'s top-K and
// publishes it (flag = launch epoch + 1); a decode item of (b, g) waits, with a time
// bound, for that flag.  Every item a decode item can wait on was handed out earlier to a
// running CTA that never waits itself, so the queue cannot deadlock whatever the
// residency.  The CTA that finishes the last decode item of (b, g) merges its partials.
// Counters return to zero before the launch ends; the epoch makes old flags stale.
#include "quest_device.cuh"

namespace quest {

template <int G, int P>
__global__ void __launch_bounds__(kDecodeThreads, (P == 16 && G <= 4) ? 2 : 1)
    fused_kernel(Params p, int topk_keys) {
  extern __shared__ __align__(128) unsigned char smem[];
  const SmemMap m = make_smem_map(G, P, topk_keys, p.score_tile_pages);
  init_ring(smem, m);
  pdl_wait();
  int* misc = reinterpret_cast<int*>(smem + m.misc);
  const unsigned target = *p.epoch + 1u;
  const int nbg = p.B * p.Hkv;
  const int n_score = nbg * p.n_score_tiles;
  const int n_items = n_score + nbg * p.n_splits;
  uint32_t pc = 0;  // pages pushed through this CTA's ring so far
  while (true) {
    if (threadIdx.x == 0) misc[0] = (int)atomicAdd(p.ticket, 1u);
    __syncthreads();
    const int item = misc[0];
    __syncthreads();
    if (item >= n_items) break;
    if (item < n_score) {
      // ---------------- scoring tile (+ top-K by the last tile of the (b, g))
      const int bg = item / p.n_score_tiles, tile = item % p.n_score_tiles;
      const int b = bg / p.Hkv, g = bg % p.Hkv;
      const int L = load_len(p, b, kSiteScore);
      const int N = (L + P - 1) / P;
      const int p0 = tile * p.score_tile_pages;
      const int n_live = max(0, min(N - p0, min(p.score_tile_pages, p.max_pages - p0)));
      float* row = p.scores + (size_t)bg * p.max_pages;
      if (n_live > 0)
        score_tile<G>(p, b, g, p0, n_live, row + p0, reinterpret_cast<int*>(smem + m.bt));
      if (arrive_last(&p.score_arrive[bg], (unsigned)p.n_score_tiles, misc + 1)) {
        topk_select(row, N, p.top_k, p.sel_idx + (size_t)bg * p.top_k, p.sel_count + bg,
                    reinterpret_cast<uint32_t*>(smem + m.ring),
                    reinterpret_cast<int*>(smem + m.hist), reinterpret_cast<int*>(smem + m.scratch));
        fence_proxy_async_smem();  // the keys used the ring's memory
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
          p.score_arrive[bg] = 0u;
          if (!(p.debug_flags & QUEST_DEBUG_WITHHOLD_SELECTION)) st_release_u32(&p.ready[bg], target);
        }
      }
    } else {
      // ---------------- split-K decode item (+ merge by the last item of the (b, g))
      const int d = item - n_score;
      const int bg = d / p.n_splits, split = d % p.n_splits;
      const int b = bg / p.Hkv, g = bg % p.Hkv;
      const int L = load_len(p, b, kSiteDecode);
      const int N = (L + P - 1) / P;
      const int count = min(p.top_k, N);
      const int r0 = split * p.pps;
      const int n_tile = max(0, min(count - r0, p.pps));
      if (n_tile > 0) {
        if (threadIdx.x == 0)
          misc[2] = wait_flag_bounded(p, &p.ready[bg], target, b, kSiteWaitSelection) ? 1 : 0;
        __syncthreads();
        const bool ok = misc[2] != 0;
        __syncthreads();
        if (ok) {
          decode_tile<G, P>(p, smem, m, b, g, split, r0, n_tile, L, N,
                            p.sel_idx + (size_t)bg * p.top_k, pc);
          pc += (uint32_t)n_tile;
        }
      }
      if (arrive_last(&p.decode_arrive[bg], (unsigned)p.n_splits, misc + 3)) {
        merge_splits<G>(p, smem, m, b, g, (count + p.pps - 1) / p.pps);
        if (threadIdx.x == 0) p.decode_arrive[bg] = 0u;
      }
    }
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.exited, 1u) == gridDim.x - 1u) {
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

cudaError_t launch_fused(const Params& p, int G, int max_ctas, cudaStream_t s) {
  const void* fn = pick_fused(G, p.P);
  const int topk_keys = p.max_pages;
  const size_t smem = decode_smem_bytes(G, p.P, topk_keys, p.score_tile_pages);
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
  int tk = topk_keys;
  void* args[] = {&pp, &tk};
  return launch_pdl(fn, dim3((unsigned)grid), dim3(kDecodeThreads), smem, s, args);
}

}  // namespace quest
