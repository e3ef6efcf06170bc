// quest_cache_kernels.cu - page bounding boxes after prefill, the chunked-prefill write that
// forms them on the fly, and the decode-time append.
//
// "Guide to Quest: Query-Aware KV Cache Sparsity for LLMs", Solution step 1: each page
// is summarised by the per-dimension minimum and maximum of its keys, formed while the
// page is filled during prompt prefill or token generation.
#include "quest_device.cuh"

namespace quest {

// One warp per (sequence, logical page, kv head).  Half-warp hw takes rows hw, hw+2, ...;
// lane c of the half-warp owns dims [8c, 8c+8) (16 B), so a half-warp reads one 256 B key
// row per load and a warp keeps P/2 x 16 B loads in flight.  min/max in packed fp16 is
// exact.  Slots past the sequence end are never read into the box.
template <int P>
__global__ void __launch_bounds__(256) build_meta_kernel(Params p) {
  pdl_wait();
  const long long unit = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31, hw = lane >> 4, c = lane & 15;
  const long long units = (long long)p.B * p.max_pages * p.Hkv;
  if (unit >= units) return;  // warp-uniform; this kernel has no block barrier
  const int g = (int)(unit % p.Hkv);
  const long long bp = unit / p.Hkv;
  const int pg = (int)(bp % p.max_pages);
  const int b = (int)(bp / p.max_pages);
  const int L = load_len(p, b, kSiteMeta);
  if (pg * P >= L) return;
  const int phys = p.block_table[(size_t)b * p.max_pages + pg];
  if (phys < 0 || phys >= p.num_phys) {
    if (lane == 0) report(p, QUEST_ERR_BAD_PAGE, b, pg, kSiteMeta);
    return;
  }
  const int nv = min(P, L - pg * P);
  const __half* src = p.k_pool + ((size_t)phys * p.Hkv + g) * P * kHeadDim + 8 * c;
  uint4 rows[P / 2];
#pragma unroll
  for (int r = 0; r < P / 2; ++r) {
    const int t = hw + 2 * r;
    rows[r] = ld_stream_v4(src + (size_t)(t < nv ? t : 0) * kHeadDim);  // row 0 is always valid
  }
  __half2 mn[4], mx[4];
  {
    const uint32_t w[4] = {rows[0].x, rows[0].y, rows[0].z, rows[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) mn[k] = mx[k] = *reinterpret_cast<const __half2*>(&w[k]);
  }
#pragma unroll
  for (int r = 1; r < P / 2; ++r) {
    const uint32_t w[4] = {rows[r].x, rows[r].y, rows[r].z, rows[r].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const __half2 v = *reinterpret_cast<const __half2*>(&w[k]);
      mn[k] = __hmin2(mn[k], v);
      mx[k] = __hmax2(mx[k], v);
    }
  }
  // combine the two half-warps (even and odd rows)
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t a = *reinterpret_cast<uint32_t*>(&mn[k]);
    uint32_t z = *reinterpret_cast<uint32_t*>(&mx[k]);
    a = __shfl_xor_sync(0xffffffffu, a, 16);
    z = __shfl_xor_sync(0xffffffffu, z, 16);
    mn[k] = __hmin2(mn[k], *reinterpret_cast<const __half2*>(&a));
    mx[k] = __hmax2(mx[k], *reinterpret_cast<const __half2*>(&z));
  }
  __half2* dst = reinterpret_cast<__half2*>(p.meta + box_offset(p, b, g, pg) +
                                            (hw ? kHeadDim : 0) + 8 * c);
  const __half2* v = hw ? mx : mn;
  uint4 o;
  o.x = *reinterpret_cast<const uint32_t*>(&v[0]);
  o.y = *reinterpret_cast<const uint32_t*>(&v[1]);
  o.z = *reinterpret_cast<const uint32_t*>(&v[2]);
  o.w = *reinterpret_cast<const uint32_t*>(&v[3]);
  *reinterpret_cast<uint4*>(dst) = o;
}

// One CTA per sequence; warps loop over kv heads.  Lanes 0-15 move the key row and own
// the box minimum, lanes 16-31 move the value row and own the maximum.  The new token
// opens a fresh box in slot 0 and widens the existing one otherwise.  The length grows
// once every head is written (unless `advance` is 0: a caller appending the same position
// in several layers advances the lengths once, afterwards).
template <int P>
__global__ void __launch_bounds__(256) append_kernel(Params p, const __half* k_new,
                                                     const __half* v_new, int advance) {
  pdl_wait();
  pdl_trigger();  // the decode step that follows may start its prologue
  __shared__ int s_len, s_phys;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) {
    int L = p.seq_lens[b];
    int phys = -1;
    if (L < 0 || (long long)L + 1 > (long long)p.max_pages * P) {
      report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);
      L = -1;
    } else {
      phys = p.block_table[(size_t)b * p.max_pages + L / P];
      if (phys < 0 || phys >= p.num_phys) {
        report(p, QUEST_ERR_BAD_PAGE, b, L / P, kSiteAppend);
        L = -1;
      }
    }
    s_len = L;
    s_phys = phys;
  }
  __syncthreads();
  const int L = s_len;
  if (L < 0) return;  // block-uniform
  const int phys = s_phys, slot = L % P;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, c = lane & 15;
  const bool upper = lane >= 16;
  for (int g = warp; g < p.Hkv; g += 8) {
    const size_t row = ((size_t)b * p.Hkv + g) * kHeadDim + 8 * c;
    const uint4 kk = *reinterpret_cast<const uint4*>(k_new + row);
    const uint4 mine = upper ? *reinterpret_cast<const uint4*>(v_new + row) : kk;
    const size_t kv_off = (((size_t)phys * p.Hkv + g) * P + slot) * kHeadDim + 8 * c;
    *reinterpret_cast<uint4*>((upper ? p.v_pool : p.k_pool) + kv_off) = mine;
    uint4* box = reinterpret_cast<uint4*>(p.meta + box_offset(p, b, g, L / P) +
                                          (upper ? kHeadDim : 0) + 8 * c);
    uint4 res = kk;
    if (slot != 0) {
      const uint4 cur = *box;
      const uint32_t a[4] = {cur.x, cur.y, cur.z, cur.w};
      const uint32_t n[4] = {kk.x, kk.y, kk.z, kk.w};
      uint32_t r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 x = *reinterpret_cast<const __half2*>(&a[k]);
        const __half2 y = *reinterpret_cast<const __half2*>(&n[k]);
        const __half2 z = upper ? __hmax2(x, y) : __hmin2(x, y);
        r[k] = *reinterpret_cast<const uint32_t*>(&z);
      }
      res = make_uint4(r[0], r[1], r[2], r[3]);
    }
    *box = res;
  }
  __syncthreads();
  if (advance && threadIdx.x == 0) p.seq_lens[b] = L + 1;
}

// Chunked prefill: n new tokens per sequence are written at slots [L, L + n) and folded
// into their pages' boxes in the same pass ("Guide to Quest", Solution step 1: the boxes
// are formed while pages are filled during prefill).  grid (ceil(Hkv / 4), pages a chunk
// can touch, B), 128 threads: block (z, j, b) owns logical page L / P + j of sequence b,
// warp w its kv head 4z + w.  Heads vary fastest across blocks, so that the blocks in
// flight read whole token rows of the chunk and write whole physical pages.  Half-warp hw takes the page's new rows hw, hw + 2, ... and
// lane c dims [8c, 8c + 8); all of a half-warp's rows (8 at a time) are loaded before any
// is stored, so that a warp keeps 8 KB in flight.  The box of a page that already held
// tokens is widened, otherwise replaced.  k, v: fp16 [B][n][Hkv][128].  Lengths advance
// in prefill_lens_kernel.
constexpr int kPrefillWarps = 4;

template <int P>
__global__ void __launch_bounds__(32 * kPrefillWarps) prefill_kernel(Params p, const __half* k,
                                                                     const __half* v, int n) {
  pdl_wait();
  const int b = blockIdx.z;
  const int g = blockIdx.x * kPrefillWarps + (threadIdx.x >> 5);
  const int L = p.seq_lens[b];
  if (L < 0 || (long long)L + n > (long long)p.max_pages * P) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      report(p, QUEST_ERR_BAD_LENGTH, b, -1, kSiteAppend);
    return;
  }
  const int page = L / P + (int)blockIdx.y;
  const int t0 = max(page * P, L), t1 = min(page * P + P, L + n);  // new tokens of this page
  if (t0 >= t1 || g >= p.Hkv) return;  // warp-uniform; no block barrier below
  const int phys = p.block_table[(size_t)b * p.max_pages + page];
  if (phys < 0 || phys >= p.num_phys) {
    if ((threadIdx.x & 31) == 0 && g == 0) report(p, QUEST_ERR_BAD_PAGE, b, page, kSiteAppend);
    return;
  }
  const int lane = threadIdx.x & 31, hw = lane >> 4, c = lane & 15;
  const size_t in_stride = (size_t)p.Hkv * kHeadDim;  // one token of the chunk
  const __half* kin = k + ((size_t)b * n * p.Hkv + g) * kHeadDim + 8 * c;
  const __half* vin = v + ((size_t)b * n * p.Hkv + g) * kHeadDim + 8 * c;
  __half* kout = p.k_pool + ((size_t)phys * p.Hkv + g) * P * kHeadDim + 8 * c;
  __half* vout = p.v_pool + ((size_t)phys * p.Hkv + g) * P * kHeadDim + 8 * c;
  __half2 mn[4], mx[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) mn[e] = mx[e] = __float2half2_rn(0.f);
  bool any = false;
  constexpr int R = 8;
#pragma unroll 1
  for (int tb = t0 + hw; tb < t1; tb += 2 * R) {
    uint4 kk[R], vv[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = tb + 2 * r;
      if (t < t1) {
        kk[r] = __ldcs(reinterpret_cast<const uint4*>(kin + (size_t)(t - L) * in_stride));
        vv[r] = __ldcs(reinterpret_cast<const uint4*>(vin + (size_t)(t - L) * in_stride));
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const int t = tb + 2 * r;
      if (t < t1) {
        __stcs(reinterpret_cast<uint4*>(kout + (size_t)(t % P) * kHeadDim), kk[r]);
        __stcs(reinterpret_cast<uint4*>(vout + (size_t)(t % P) * kHeadDim), vv[r]);
        const uint32_t w[4] = {kk[r].x, kk[r].y, kk[r].z, kk[r].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 h = *reinterpret_cast<const __half2*>(&w[e]);
          mn[e] = any ? __hmin2(mn[e], h) : h;
          mx[e] = any ? __hmax2(mx[e], h) : h;
        }
        any = true;
      }
    }
  }
  // combine the two half-warps (the upper one has no row when the page gets one token)
  const bool other = __shfl_xor_sync(0xffffffffu, any ? 1 : 0, 16) != 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t a = *reinterpret_cast<uint32_t*>(&mn[e]), z = *reinterpret_cast<uint32_t*>(&mx[e]);
    const uint32_t oa = __shfl_xor_sync(0xffffffffu, a, 16);
    const uint32_t oz = __shfl_xor_sync(0xffffffffu, z, 16);
    if (other) {
      const __half2 ha = *reinterpret_cast<const __half2*>(&oa);
      const __half2 hz = *reinterpret_cast<const __half2*>(&oz);
      mn[e] = any ? __hmin2(mn[e], ha) : ha;
      mx[e] = any ? __hmax2(mx[e], hz) : hz;
    }
  }
  if (hw == 0) {
    uint4* bmin = reinterpret_cast<uint4*>(p.meta + box_offset(p, b, g, page) + 8 * c);
    uint4* bmax = reinterpret_cast<uint4*>(p.meta + box_offset(p, b, g, page) + kHeadDim + 8 * c);
    if (page * P < L) {  // the page already held tokens: widen its box
      const uint4 cmn = *bmin, cmx = *bmax;
      const uint32_t a[4] = {cmn.x, cmn.y, cmn.z, cmn.w};
      const uint32_t z[4] = {cmx.x, cmx.y, cmx.z, cmx.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        mn[e] = __hmin2(mn[e], *reinterpret_cast<const __half2*>(&a[e]));
        mx[e] = __hmax2(mx[e], *reinterpret_cast<const __half2*>(&z[e]));
      }
    }
    *bmin = make_uint4(*reinterpret_cast<uint32_t*>(&mn[0]), *reinterpret_cast<uint32_t*>(&mn[1]),
                       *reinterpret_cast<uint32_t*>(&mn[2]), *reinterpret_cast<uint32_t*>(&mn[3]));
    *bmax = make_uint4(*reinterpret_cast<uint32_t*>(&mx[0]), *reinterpret_cast<uint32_t*>(&mx[1]),
                       *reinterpret_cast<uint32_t*>(&mx[2]), *reinterpret_cast<uint32_t*>(&mx[3]));
  }
}

// Advances the lengths of the sequences the chunk fitted into (the same tests as above).
// One block per sequence; its threads check the block-table entries of the touched pages
// side by side (a serial scan of a long chunk's pages by one thread cost ~150 us).
__global__ void __launch_bounds__(256) prefill_lens_kernel(Params p, int n) {
  pdl_wait();
  const int b = blockIdx.x;
  const int L = p.seq_lens[b];
  const bool fits = L >= 0 && (long long)L + n <= (long long)p.max_pages * p.P;
  int bad = 0;
  if (fits) {
    const int first = L / p.P, last = (L + n - 1) / p.P;
    for (int pg = first + (int)threadIdx.x; pg <= last; pg += blockDim.x) {
      const int phys = p.block_table[(size_t)b * p.max_pages + pg];
      bad |= phys < 0 || phys >= p.num_phys;  // reported by the write kernel
    }
  }
  bad = __syncthreads_or(bad);
  if (fits && !bad && threadIdx.x == 0) p.seq_lens[b] = L + n;
}

cudaError_t launch_advance_lengths(const Params& p, int n, cudaStream_t s) {
  Params pp = p;
  int nn = n;
  void* args[] = {&pp, &nn};
  return launch_pdl((const void*)prefill_lens_kernel, dim3(p.B), dim3(256), 0, s, args);
}

cudaError_t launch_prefill(const Params& p, const __half* k, const __half* v, int n,
                           cudaStream_t s) {
  Params pp = p;
  const __half* kk = k;
  const __half* vv = v;
  int nn = n;
  void* args[] = {&pp, &kk, &vv, &nn};
  const unsigned pages = (unsigned)((n + p.P - 1) / p.P + 1);
  const void* fn = p.P == 16 ? (const void*)prefill_kernel<16> : (const void*)prefill_kernel<32>;
  cudaError_t e = launch_pdl(fn, dim3((p.Hkv + kPrefillWarps - 1) / kPrefillWarps, pages, p.B),
                             dim3(32 * kPrefillWarps), 0, s, args);
  if (e != cudaSuccess) return e;
  return launch_advance_lengths(p, n, s);
}

cudaError_t launch_build_meta(const Params& p, cudaStream_t s) {
  const long long units = (long long)p.B * p.max_pages * p.Hkv;
  const unsigned blocks = (unsigned)((units + 7) / 8);
  Params pp = p;
  void* args[] = {&pp};
  const void* fn = p.P == 16 ? (const void*)build_meta_kernel<16> : (const void*)build_meta_kernel<32>;
  return launch_pdl(fn, dim3(blocks), dim3(256), 0, s, args);
}

cudaError_t launch_append(const Params& p, const __half* k_new, const __half* v_new,
                          cudaStream_t s, bool advance) {
  Params pp = p;
  const __half* kn = k_new;
  const __half* vn = v_new;
  int adv = advance ? 1 : 0;
  void* args[] = {&pp, &kn, &vn, &adv};
  const void* fn = p.P == 16 ? (const void*)append_kernel<16> : (const void*)append_kernel<32>;
  return launch_pdl(fn, dim3(p.B), dim3(256), 0, s, args);
}

}  // namespace quest
