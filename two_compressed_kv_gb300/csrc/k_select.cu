// Decode step, second part: exact top-k token selection per KV head.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction, prior-work paragraph:
// query-aware selection of the tokens to attend (as in Quest); here the
// min(top_k, T) highest scores, ties to the lower token index.
#include <cooperative_groups.h>

#include "decode_common.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// select: exact top-k of one stream by a cluster of R CTAs (R = 1..8).  CTA r
// owns the token range [r * per, (r + 1) * per) and its warp w a contiguous
// sub-range (a "block" (r, w)); blocks in (r, w) order cover the tokens in
// order.  The score kernel left the level-1 bin b1 of the k-th largest key and
// the number k1 of keys still needed from that bin.
//   1. one pass over the scores: each warp lists, in token order, its "sure"
//      tokens (key bin above b1: all selected) and its candidates (key bin
//      b1, with the key), in its own part of the stream's scratch area;
//   2. cluster barrier; every CTA reads the per-block counts of all ranks
//      (distributed shared memory) and the candidates of the whole stream
//      (in token order), and selects the same threshold: the key thr of the
//      k1-th largest candidate (two more 10-bit radix digits), then among
//      keys equal to thr the lowest tokens (radix on 0x7fffffff - t): t_cut;
//   3. the selected candidates B (token order) and the sure tokens are merged
//      by position: sure token j of the stream lands at j + |{b in B : b < t}|,
//      B[i] at i + |{sure tokens < B[i]}|; each warp places its own block.
// With more than SEL_CAP candidates the threshold is found the same way from
// the scratch area and step 3 re-reads the scores instead.  Deterministic:
// candidates are only counted, never summed.
// grid: (R, BH), cluster (R, 1, 1), block 1024, dynamic smem SEL_CAP * 12
// ---------------------------------------------------------------------------
constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;
constexpr int SEL_CAP = 8192;                 // candidates kept in shared memory
constexpr size_t SEL_SMEM = (size_t)SEL_CAP * (sizeof(uint2) + sizeof(int32_t));

// exclusive scan of one value per thread over SEL_THREADS threads
__device__ __forceinline__ uint32_t sel_excl_scan(uint32_t v, uint32_t* sh, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = sh[lane];
    uint32_t x = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += o;
    }
    sh[32 + lane] = x - w;                    // exclusive warp offsets
    if (lane == 31) sh[64] = x;
  }
  __syncthreads();
  const uint32_t before = sh[32 + warp];
  if (total) *total = sh[64];
  __syncthreads();
  return before + inc - v;
}

// first index i in [0, n) with a[i] >= x (n if none); a ascending
__device__ __forceinline__ uint32_t lower_bound_i32(const int32_t* a, uint32_t n, int64_t x) {
  uint32_t lo = 0, hi = n;
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if ((int64_t)a[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

struct SelShared {
  uint32_t ws[SEL_WARPS], wc[SEL_WARPS];     // this CTA: sure / candidate count per warp
  uint32_t Sp[8 * SEL_WARPS + 1];            // exclusive prefix over blocks (q, w): sure
  uint32_t Cp[8 * SEL_WARPS + 1];            // same for candidates
  uint32_t scan[72];
  uint32_t hist[2048];
  uint32_t warp8[8], res[2];
};

struct SelGeom {
  int64_t per, T;
  __device__ int64_t rank_lo(int q) const { return (int64_t)q * per; }
  __device__ int64_t rank_hi(int q) const {
    const int64_t h = (int64_t)(q + 1) * per;
    return h < T ? h : T;
  }
  __device__ int64_t wlen(int q) const {
    const int64_t len = rank_hi(q) - rank_lo(q);
    return len > 0 ? (len + SEL_WARPS * 128 - 1) / (SEL_WARPS * 128) * 128 : 0;
  }
  __device__ int64_t block_lo(int q, int w) const {
    const int64_t x = rank_lo(q) + (int64_t)w * wlen(q);
    return x < rank_hi(q) ? x : rank_hi(q);
  }
  __device__ int64_t block_hi(int q, int w) const {
    const int64_t x = rank_lo(q) + (int64_t)(w + 1) * wlen(q);
    return x < rank_hi(q) ? x : rank_hi(q);
  }
};

__device__ __forceinline__ void select_kernel_body(const DecodeParams& p) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  uint2* cbuf = reinterpret_cast<uint2*>(sel_dyn);                        // [SEL_CAP]
  int32_t* bbuf = reinterpret_cast<int32_t*>(sel_dyn + SEL_CAP * sizeof(uint2));  // [SEL_CAP]
  __shared__ SelShared sh;
  const int R = (int)cl.num_blocks(), r = (int)cl.block_rank();
  const int s = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();     // scores and the level-1 state come from the score kernel
  if (p.pdl_trigger) griddep_launch();
  SelGeom geo;
  geo.per = (((p.Tp + R - 1) / R) + 15) / 16 * 16;
  geo.T = p.T;
  const float* sc = p.scores + (size_t)s * p.Tp;
  uint2* cs = p.cand + (size_t)s * p.Tp;             // the stream's scratch area
  const uint32_t b1 = p.state[s].b1;
  const int64_t w_lo = geo.block_lo(r, warp), w_hi = geo.block_hi(r, warp);
  // block (q, w): candidates at cs[lo + i]; sure tokens at int32 slot
  // 2 * (hi - lo) - 1 - j of the same area (2 nc + ns <= 2 (hi - lo))
  uint2* cand_w = cs + w_lo;
  int32_t* sure_w = reinterpret_cast<int32_t*>(cand_w);
  const int64_t L_w = w_hi - w_lo;

  // ---- 1. sure tokens and candidates of this warp's block, in token order --
  // Lane l takes the 32 consecutive tokens at b0 + 32 l of each 1024-token
  // step.  bin(key) > b1 and bin(key) == b1 are tested as float compares
  // against the smallest floats of bins b1 and b1 + 1 (the key map is
  // monotone; both zeros fall in the same bin and compare equal).
  uint32_t ns_w = 0, nc_w = 0;
  // bins 0 and >= 4088 also hold infinities and NaNs: those compare by key
  const bool by_key = b1 == 0u || b1 >= 4088u;
  const float f_lo = by_key ? 0.f : key2f(b1 << 20);
  const float f_hi = by_key ? 0.f : key2f((b1 + 1u) << 20);
  for (int64_t b0 = w_lo; b0 < w_hi; b0 += 32 * 32) {
    const int64_t t0 = b0 + 32 * lane;
    float4 f[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      f[j] = t0 + 4 * j < w_hi ? __ldcg(reinterpret_cast<const float4*>(sc + t0) + j)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    const int nv = t0 >= w_hi ? 0 : (w_hi - t0 >= 32 ? 32 : (int)(w_hi - t0));
    uint32_t sm = 0, cm = 0;        // bit i: token t0 + i is sure / a candidate
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float v4[4] = {f[j].x, f[j].y, f[j].z, f[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sm |= (uint32_t)(v4[e] >= f_hi) << (4 * j + e);
        cm |= (uint32_t)(v4[e] >= f_lo && v4[e] < f_hi) << (4 * j + e);
      }
    }
    if (by_key) {
      sm = 0;
      cm = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float v4[4] = {f[j].x, f[j].y, f[j].z, f[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t bin = f2key(v4[e]) >> 20;
          sm |= (uint32_t)(bin > b1) << (4 * j + e);
          cm |= (uint32_t)(bin == b1) << (4 * j + e);
        }
      }
    }
    const uint32_t valid = nv >= 32 ? 0xffffffffu : ((1u << nv) - 1u);
    sm &= valid;
    cm &= valid;
    const uint32_t packed = (uint32_t)__popc(sm) | ((uint32_t)__popc(cm) << 16);
    uint32_t inc = packed;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += o;
    }
    const uint32_t excl = inc - packed, tot = __shfl_sync(0xffffffffu, inc, 31);
    int32_t* sp = sure_w + (2 * L_w - 1 - (int64_t)(ns_w + (excl & 0xffffu)));
    uint2* cp = cand_w + (nc_w + (excl >> 16));
    while (sm) {
      const int i = __ffs(sm) - 1;
      sm &= sm - 1;
      *sp-- = (int32_t)(t0 + i);
    }
    while (cm) {
      const int i = __ffs(cm) - 1;
      cm &= cm - 1;
      *cp++ = make_uint2(f2key(__ldcg(sc + t0 + i)), (uint32_t)(t0 + i));
    }
    ns_w += tot & 0xffffu;
    nc_w += tot >> 16;
  }
  if (lane == 0) {
    sh.ws[warp] = ns_w;
    sh.wc[warp] = nc_w;
  }
  cl.sync();

  // ---- 2. counts of every block of the stream, then the threshold ----------
  {
    uint32_t sv = 0, cv = 0;
    if (tid < R * SEL_WARPS) {
      const SelShared* rs = cl.map_shared_rank(&sh, tid / SEL_WARPS);
      sv = rs->ws[tid % SEL_WARPS];
      cv = rs->wc[tid % SEL_WARPS];
    }
    uint32_t st, ct;
    const uint32_t se = sel_excl_scan(sv, sh.scan, &st);
    const uint32_t ce = sel_excl_scan(cv, sh.scan, &ct);
    if (tid < R * SEL_WARPS) {
      sh.Sp[tid] = se;
      sh.Cp[tid] = ce;
    }
    if (tid == 0) {
      sh.Sp[R * SEL_WARPS] = st;
      sh.Cp[R * SEL_WARPS] = ct;
    }
  }
  cl.sync();   // no remote shared-memory reads past this point
  const int NB = R * SEL_WARPS;
  const uint32_t N = sh.Cp[NB];
  const bool fast = N <= (uint32_t)SEL_CAP;
  if (fast) {
    for (int b = warp; b < NB; b += SEL_WARPS) {
      const uint32_t c0 = sh.Cp[b], cnt = sh.Cp[b + 1] - c0;
      const uint2* src = cs + geo.block_lo(b / SEL_WARPS, b % SEL_WARPS);
      for (uint32_t i = lane; i < cnt; i += 32) cbuf[c0 + i] = __ldcg(src + i);
    }
    __syncthreads();
  }
  auto cand_at = [&](uint32_t i) -> uint2 {
    if (fast) return cbuf[i];
    int lo = 0, hi = NB - 1;                  // last block b with Cp[b] <= i
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (sh.Cp[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return __ldcg(cs + geo.block_lo(lo / SEL_WARPS, lo % SEL_WARPS) + (i - sh.Cp[lo]));
  };
  const uint32_t need = p.state[s].k1;
  for (int x = tid; x < 1024; x += SEL_THREADS) sh.hist[x] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < N; i += SEL_THREADS) atomicAdd(&sh.hist[(cand_at(i).x >> 10) & 1023u], 1u);
  __syncthreads();
  find_bin<1024>(sh.hist, need, sh.res, sh.warp8);
  const uint32_t bA = sh.res[0] & 1023u, needA = sh.res[1];
  __syncthreads();
  for (int x = tid; x < 1024; x += SEL_THREADS) sh.hist[x] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < N; i += SEL_THREADS) {
    const uint32_t key = cand_at(i).x;
    if (((key >> 10) & 1023u) == bA) atomicAdd(&sh.hist[key & 1023u], 1u);
  }
  __syncthreads();
  find_bin<1024>(sh.hist, needA, sh.res, sh.warp8);
  const uint32_t bB = sh.res[0] & 1023u, need_eq = sh.res[1];
  const uint32_t n_eq = sh.hist[bB];
  const uint32_t thr = (b1 << 20) | (bA << 10) | bB;
  __syncthreads();
  int32_t t_cut = 0x7fffffff;
  if (need_eq < n_eq) {
    // the need_eq lowest token ids among keys equal to thr
    uint32_t prefix = 0, krem = need_eq;
    for (int lev = 0; lev < 3; ++lev) {
      const int nb = lev == 0 ? 2048 : 1024;
      const int shift = lev == 0 ? 20 : (lev == 1 ? 10 : 0);
      for (int x = tid; x < nb; x += SEL_THREADS) sh.hist[x] = 0u;
      __syncthreads();
      for (uint32_t i = tid; i < N; i += SEL_THREADS) {
        const uint2 cv = cand_at(i);
        if (cv.x != thr) continue;
        const uint32_t u = 0x7fffffffu - cv.y;
        if (lev > 0 && (u >> (shift + 10)) != prefix) continue;
        atomicAdd(&sh.hist[(u >> shift) & (uint32_t)(nb - 1)], 1u);
      }
      __syncthreads();
      if (lev == 0) find_bin<2048>(sh.hist, krem, sh.res, sh.warp8);
      else find_bin<1024>(sh.hist, krem, sh.res, sh.warp8);
      prefix = (prefix << (lev == 0 ? 0 : 10)) | (sh.res[0] & (uint32_t)(nb - 1));
      krem = sh.res[1];
      __syncthreads();
    }
    t_cut = (int32_t)(0x7fffffffu - prefix);
  }
  if (r == 0 && tid == 0) {
    p.state[s].thr = thr;
    p.state[s].t_cut = t_cut;
  }
  auto chosen = [&](uint32_t key, int64_t t) -> bool {
    return key > thr || (key == thr && t <= (int64_t)t_cut);
  };
  int32_t* out = p.sel + (size_t)s * p.kk;
  int32_t* out2 = p.sel_user ? p.sel_user + (size_t)s * p.kk : nullptr;
  auto put = [&](uint32_t pos, int32_t t) {
    if (pos < (uint32_t)p.kk) {
      out[pos] = t;
      if (out2) out2[pos] = t;
    }
  };

  if (fast) {
    // ---- 3. B = selected candidates in token order; merge with sure tokens -
    uint32_t cnt = 0;
    const uint32_t i0 = (uint32_t)tid * (SEL_CAP / SEL_THREADS);
#pragma unroll
    for (int e = 0; e < SEL_CAP / SEL_THREADS; ++e) {
      const uint32_t i = i0 + e;
      if (i < N && chosen(cbuf[i].x, cbuf[i].y)) ++cnt;
    }
    uint32_t nB;
    uint32_t pos = sel_excl_scan(cnt, sh.scan, &nB);
#pragma unroll
    for (int e = 0; e < SEL_CAP / SEL_THREADS; ++e) {
      const uint32_t i = i0 + e;
      if (i < N && chosen(cbuf[i].x, cbuf[i].y)) bbuf[pos++] = (int32_t)cbuf[i].y;
    }
    __syncthreads();
    const uint32_t gS = sh.Sp[r * SEL_WARPS + warp];
    const uint32_t bl = lower_bound_i32(bbuf, nB, w_lo), bh = lower_bound_i32(bbuf, nB, w_hi);
    for (uint32_t bg = bl;; bg += 32) {
      const uint32_t b = bg + lane;
      const int32_t tb = b < bh ? bbuf[b] : -1;
      uint32_t below = 0;
      for (uint32_t j0 = 0; j0 < ns_w; j0 += 32) {
        const uint32_t j = j0 + lane;
        const int32_t t = j < ns_w ? sure_w[2 * L_w - 1 - (int64_t)j] : 0x7fffffff;
        if (bg == bl && j < ns_w) put(gS + j + lower_bound_i32(bbuf, nB, t), t);
        if (bh > bl) {
          const int nk = ns_w - j0 < 32u ? (int)(ns_w - j0) : 32;
          for (int k = 0; k < nk; ++k) below += __shfl_sync(0xffffffffu, t, k) < tb;
        }
      }
      if (b < bh) put(b + gS + below, tb);
      if (bg + 32 >= bh) break;
    }
  } else {
    // ---- 3'. many candidates: count, then write, re-reading the scores -----
    auto is_sel = [&](float x, int64_t t) -> uint32_t {
      return (t < w_hi && chosen(f2key(x), t)) ? 1u : 0u;
    };
    uint32_t offset = 0;
    {
      // selected tokens of every earlier block: sure ones plus chosen candidates
      uint32_t c = 0;
      const uint32_t lim = sh.Cp[r * SEL_WARPS];
      for (uint32_t i = tid; i < lim; i += SEL_THREADS) {
        const uint2 cv = cand_at(i);
        c += chosen(cv.x, cv.y);
      }
      uint32_t tot;
      sel_excl_scan(c, sh.scan, &tot);
      offset = sh.Sp[r * SEL_WARPS] + tot;
    }
    uint32_t wcount = 0;
    for (int64_t b0 = w_lo; b0 < w_hi; b0 += 128) {
      const int64_t t0 = b0 + 4 * lane;
      const float4 f = t0 < w_hi ? __ldcg(reinterpret_cast<const float4*>(sc + t0))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      wcount += is_sel(f.x, t0) + is_sel(f.y, t0 + 1) + is_sel(f.z, t0 + 2) + is_sel(f.w, t0 + 3);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wcount += __shfl_xor_sync(0xffffffffu, wcount, off);
    uint32_t wbase = offset + sel_excl_scan(lane == 0 ? wcount : 0u, sh.scan, nullptr);
    wbase = __shfl_sync(0xffffffffu, wbase, 0);
    for (int64_t b0 = w_lo; b0 < w_hi; b0 += 128) {
      const int64_t t0 = b0 + 4 * lane;
      const float4 f = t0 < w_hi ? __ldcg(reinterpret_cast<const float4*>(sc + t0))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t m = is_sel(f.x, t0) | (is_sel(f.y, t0 + 1) << 1) |
                         (is_sel(f.z, t0 + 2) << 2) | (is_sel(f.w, t0 + 3) << 3);
      const uint32_t n = __popc(m);
      uint32_t inc = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t o = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += o;
      }
      uint32_t q = wbase + inc - n;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if ((m >> e) & 1u) put(q++, (int32_t)(t0 + e));
      wbase += __shfl_sync(0xffffffffu, inc, 31);
    }
  }
}

// one layer (parameters by value), and several layers in one launch (layer = blockIdx.z)
__global__ void __launch_bounds__(SEL_THREADS, 1) select_kernel(DecodeParams p) { select_kernel_body(p); }
__global__ void __launch_bounds__(SEL_THREADS, 1) select_kernel_layers(const __grid_constant__ LayerParams lp) {
  select_kernel_body(lp.p[blockIdx.z]);
}

int select_cluster_size(int n_streams, int64_t T, int G) {
  int R = 1;
  while (R < 8 && (int64_t)n_streams * R * 2 <= G && T / (2 * R) >= 4096) R *= 2;
  return R;
}

cudaError_t prepare_select_kernels() {
  const cudaError_t e = cudaFuncSetAttribute(select_kernel_layers,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SEL_SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)SEL_SMEM);
}

cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st, const LayerParams* lp, int n) {
  const bool pdl = ((p.pdl >> MKV_KERNEL_TOPK) & 1) != 0;
  if (lp)
    return launch_kernel(select_kernel_layers, dim3(p.sel_R, p.B * p.H, n), dim3(SEL_THREADS),
                         SEL_SMEM, st, pdl, p.sel_R, *lp);
  return launch_kernel(select_kernel, dim3(p.sel_R, p.B * p.H, 1), dim3(SEL_THREADS), SEL_SMEM,
                       st, pdl, p.sel_R, p);
}

}  // namespace mkv
