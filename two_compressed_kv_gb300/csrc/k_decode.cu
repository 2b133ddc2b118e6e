// Decode-step kernels: attention over the packed two-D compressed cache.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction: query-aware token selection
// (prior-work paragraph) and attention computed on the packed dense format
// with CUDA cores, without unpacking ("Observation & Method 2").
//
// Launch order per step: qrot -> score -> topk (4 launches) -> attn -> merge.
// No kernel waits on another CTA; every cross-CTA combination is either an
// integer atomic (histograms: order-independent) or a later launch.
#include "mkv_internal.cuh"

namespace mkv {

// Order-preserving map of fp32 to uint32 (larger float -> larger key);
// -0 and +0 map to the same key so that equal scores tie.
__device__ __forceinline__ uint32_t f2key(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void h8_to_f(const uint4& raw, float v[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 f = __half22float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

// ---------------------------------------------------------------------------
// qrot: q~_i = q_i R_K for the g query heads of a KV head; q_bar = sum_i q~_i.
// Also clears the stream's selection histograms for this step.
// grid: BH, block: 128 (thread j = output channel)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) qrot_kernel(DecodeParams p) {
  const int s = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int j = threadIdx.x;
  __shared__ float qs[MAX_G][D];
  const __half* q = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * D;
  for (int i = 0; i < p.g; ++i) qs[i][j] = __half2float(q[i * D + j]);
  uint32_t* hist = p.hist + (size_t)s * HIST_WORDS;
  for (int x = j; x < HIST_WORDS; x += 128) hist[x] = 0u;
  __syncthreads();
  const float* R = p.RK + (size_t)s * D * D;
  float acc[MAX_G];
#pragma unroll
  for (int i = 0; i < MAX_G; ++i) acc[i] = 0.f;
  for (int r = 0; r < D; ++r) {
    const float rv = R[r * D + j];
#pragma unroll
    for (int i = 0; i < MAX_G; ++i)
      if (i < p.g) acc[i] = fmaf(qs[i][r], rv, acc[i]);
  }
  float sum = 0.f;
  float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * p.g) * D;
#pragma unroll
  for (int i = 0; i < MAX_G; ++i) {
    if (i < p.g) {
      qt[i * D + j] = acc[i];
      sum += acc[i];
    }
  }
  p.qbar[(size_t)s * D + j] = sum;
}

// ---------------------------------------------------------------------------
// score: s_t = q_bar . k^_t for every cached token of a stream, read straight
// from the packed segments with 16-byte loads.  A warp walks one segment at a
// time; each lane owns one 16-byte chunk (8 channels) of a row, so a warp
// covers floor(32 / chunks_per_row) consecutive rows per load and the bytes a
// warp reads are contiguous.  Also builds the first radix histogram (key bits
// 31..21) of the stream's scores.
// grid: (ctas_per_stream, BH), block: 256
// ---------------------------------------------------------------------------
constexpr int SCORE_WARPS = 8;
constexpr int SCORE_UNROLL = 4;

template <int STRAT>
__device__ __forceinline__ void score_segment(const uint8_t* base, int rows, int c, int lane,
                                              const float* qb, const float* qrep,
                                              const float* qm, float* out, uint32_t* hist) {
  const int cpr = (STRAT == MKV_STRATEGY_DENSE) ? 16 : (c >> 3);   // 16-B chunks per row
  const int rpi = 32 / cpr;                                          // rows per warp load
  const int active = rpi * cpr;
  const int my_row = lane / cpr;
  const int my_chunk = lane - my_row * cpr;
  const uint8_t* vals = base + ((STRAT == MKV_STRATEGY_SM) ? pad16((uint32_t)c) : 0u);
  const uint8_t* idxs = base + 2u * (uint32_t)c * (uint32_t)rows;    // PV index block
  for (int r0 = 0; r0 < rows; r0 += rpi * SCORE_UNROLL) {
    uint4 raw[SCORE_UNROLL];
    uint2 ix[SCORE_UNROLL];
    bool ok[SCORE_UNROLL];
#pragma unroll
    for (int u = 0; u < SCORE_UNROLL; ++u) {
      const int row = r0 + u * rpi + my_row;
      ok[u] = (lane < active) && (row < rows);
      const uint32_t chunk = (uint32_t)row * cpr + my_chunk;
      if (ok[u]) {
        raw[u] = __ldg(reinterpret_cast<const uint4*>(vals) + chunk);
        if (STRAT == MKV_STRATEGY_PV) ix[u] = __ldg(reinterpret_cast<const uint2*>(idxs) + chunk);
      } else {
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        ix[u] = make_uint2(0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < SCORE_UNROLL; ++u) {
      float v[8];
      h8_to_f(raw[u], v);
      float part = 0.f;
      if (STRAT == MKV_STRATEGY_PV) {
        const uint32_t w0 = ix[u].x, w1 = ix[u].y;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t ch = ((e < 4 ? w0 : w1) >> (8 * (e & 3))) & 0x7fu;
          part = fmaf(v[e], qrep[ch * 32 + lane], part);
        }
      } else {
        const float* qq = (STRAT == MKV_STRATEGY_SM ? qm : qb) + my_chunk * 8;
        const float4 a = *reinterpret_cast<const float4*>(qq);
        const float4 b = *reinterpret_cast<const float4*>(qq + 4);
        part = fmaf(v[0], a.x, part);
        part = fmaf(v[1], a.y, part);
        part = fmaf(v[2], a.z, part);
        part = fmaf(v[3], a.w, part);
        part = fmaf(v[4], b.x, part);
        part = fmaf(v[5], b.y, part);
        part = fmaf(v[6], b.z, part);
        part = fmaf(v[7], b.w, part);
      }
      // the row's leader (chunk 0) adds the row's chunks in channel order
      float sum = part;
      for (int off = 1; off < cpr; ++off) {
        const float o = __shfl_down_sync(0xffffffffu, part, off);
        if (my_chunk == 0) sum += o;
      }
      if (ok[u] && my_chunk == 0) {
        const int row = r0 + u * rpi + my_row;
        out[row] = sum;
        atomicAdd(&hist[f2key(sum) >> 21], 1u);
      }
    }
  }
}

__global__ void __launch_bounds__(256) score_kernel(DecodeParams p) {
  const int s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ __align__(16) float qb[D];
  __shared__ __align__(16) float qrep[D * 32];
  __shared__ uint32_t hist[HIST1];
  __shared__ __align__(16) float qm[SCORE_WARPS][D];
  for (int x = threadIdx.x; x < D; x += blockDim.x) qb[x] = p.qbar[(size_t)s * D + x];
  for (int x = threadIdx.x; x < HIST1; x += blockDim.x) hist[x] = 0u;
  __syncthreads();
  for (int x = threadIdx.x; x < D * 32; x += blockDim.x) qrep[x] = qb[x >> 5];
  __syncthreads();

  const int seg0 = blockIdx.x * p.score_segs_per_cta;
  const int seg1 = min(p.n_seg, seg0 + p.score_segs_per_cta);
  const mkv_segment_header* hdr = p.hdrK + (size_t)s * p.n_seg;
  float* scores = p.scores + (size_t)s * p.T;
  for (int sg = seg0 + warp; sg < seg1; sg += SCORE_WARPS) {
    const mkv_segment_header hd = hdr[sg];
    const uint8_t* base = p.pool + (size_t)hd.off16 * 16u;
    float* out = scores + (int64_t)sg * p.S;
    if (hd.strategy == MKV_STRATEGY_SM) {
      for (int j = lane; j < p.c; j += 32) qm[warp][j] = qb[base[j] & 127];
      __syncwarp();
      score_segment<MKV_STRATEGY_SM>(base, hd.rows, p.c, lane, qb, qrep, qm[warp], out, hist);
      __syncwarp();
    } else if (hd.strategy == MKV_STRATEGY_PV) {
      score_segment<MKV_STRATEGY_PV>(base, hd.rows, p.c, lane, qb, qrep, qm[warp], out, hist);
    } else {
      score_segment<MKV_STRATEGY_DENSE>(base, hd.rows, p.c, lane, qb, qrep, qm[warp], out, hist);
    }
  }
  __syncthreads();
  uint32_t* gh = p.hist + (size_t)s * HIST_WORDS;
  for (int x = threadIdx.x; x < HIST1; x += blockDim.x)
    if (hist[x]) atomicAdd(&gh[x], hist[x]);
}

// ---------------------------------------------------------------------------
// Top-k selection: exact radix select on the ordered keys of the fp32 scores,
// 11 + 11 + 10 bits, ties to the lower token index, output in ascending
// token order.  Each launch re-derives the digits chosen so far from the
// (complete) histograms of the earlier levels.
// ---------------------------------------------------------------------------
constexpr int TK_THREADS = 256;

// Block-wide: the bin holding the krem-th largest key of histogram h[nbins]
// (counting from the top), and how many keys of that bin are still needed.
__device__ void find_bin(const uint32_t* h, int nbins, uint32_t krem, uint32_t* out_bin,
                         uint32_t* out_krem, uint32_t* sh_warp) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int per = nbins / TK_THREADS;
  const int lo = t * per;
  uint32_t mine = 0;
  for (int i = 0; i < per; ++i) mine += h[lo + i];
  // suffix sum over threads (higher thread = higher bins): inclusive within warp
  uint32_t suf = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_down_sync(0xffffffffu, suf, off);
    if (lane + off < 32) suf += o;
  }
  if (lane == 0) sh_warp[warp] = suf;     // warp total
  __syncthreads();
  uint32_t above_warps = 0;
  for (int w = warp + 1; w < TK_THREADS / 32; ++w) above_warps += sh_warp[w];
  uint32_t running = above_warps + (suf - mine);   // keys in bins above this thread's
  for (int i = per - 1; i >= 0; --i) {
    const uint32_t c = h[lo + i];
    if (running < krem && krem <= running + c) {
      *out_bin = (uint32_t)(lo + i);
      *out_krem = krem - running;
    }
    running += c;
  }
  __syncthreads();
}

// Digits chosen by the levels before `level` (1-based); fills pre[] and krem.
struct Sel {
  uint32_t b1, b2, b3, k1, k2, k3;
};

__device__ void resolve(const uint32_t* gh, int levels, uint32_t kk, Sel* sel) {
  __shared__ uint32_t sh_warp[TK_THREADS / 32];
  __shared__ uint32_t hs[HIST1];
  __shared__ Sel r;
  if (threadIdx.x == 0) r = Sel{0u, 0u, 0u, 1u, 1u, 1u};
  for (int x = threadIdx.x; x < HIST1; x += TK_THREADS) hs[x] = gh[x];
  __syncthreads();
  find_bin(hs, HIST1, kk, &r.b1, &r.k1, sh_warp);
  if (levels >= 2) {
    for (int x = threadIdx.x; x < HIST2; x += TK_THREADS) hs[x] = gh[HIST1 + x];
    __syncthreads();
    find_bin(hs, HIST2, r.k1, &r.b2, &r.k2, sh_warp);
  }
  if (levels >= 3) {
    for (int x = threadIdx.x; x < HIST3; x += TK_THREADS) hs[x] = gh[HIST1 + HIST2 + x];
    __syncthreads();
    find_bin(hs, HIST3, r.k2, &r.b3, &r.k3, sh_warp);
  }
  *sel = r;
  __syncthreads();
}

// level 2 or 3 histogram of the keys that match the digits chosen so far
template <int LEVEL>
__global__ void __launch_bounds__(TK_THREADS) topk_hist_kernel(DecodeParams p) {
  const int s = blockIdx.y;
  __shared__ uint32_t hl[HIST2];
  uint32_t* gh = p.hist + (size_t)s * HIST_WORDS;
  Sel r;
  resolve(gh, LEVEL - 1, (uint32_t)p.kk, &r);
  const int nb = LEVEL == 2 ? HIST2 : HIST3;
  for (int x = threadIdx.x; x < nb; x += TK_THREADS) hl[x] = 0u;
  __syncthreads();
  const int64_t t0 = (int64_t)blockIdx.x * TOPK_CHUNK;
  const int64_t t1 = imin64(p.T, t0 + TOPK_CHUNK);
  const float* sc = p.scores + (size_t)s * p.T;
  for (int64_t t = t0 + threadIdx.x; t < t1; t += TK_THREADS) {
    const uint32_t key = f2key(sc[t]);
    if (LEVEL == 2) {
      if ((key >> 21) == r.b1) atomicAdd(&hl[(key >> 10) & 2047u], 1u);
    } else {
      if ((key >> 10) == ((r.b1 << 11) | r.b2)) atomicAdd(&hl[key & 1023u], 1u);
    }
  }
  __syncthreads();
  uint32_t* dst = gh + (LEVEL == 2 ? HIST1 : HIST1 + HIST2);
  for (int x = threadIdx.x; x < nb; x += TK_THREADS)
    if (hl[x]) atomicAdd(&dst[x], hl[x]);
}

// per chunk: keys above the threshold and keys equal to it
__global__ void __launch_bounds__(TK_THREADS) topk_count_kernel(DecodeParams p) {
  const int s = blockIdx.y;
  Sel r;
  resolve(p.hist + (size_t)s * HIST_WORDS, 3, (uint32_t)p.kk, &r);
  const uint32_t thr = (r.b1 << 21) | (r.b2 << 10) | r.b3;
  const int64_t t0 = (int64_t)blockIdx.x * TOPK_CHUNK;
  const int64_t t1 = imin64(p.T, t0 + TOPK_CHUNK);
  const float* sc = p.scores + (size_t)s * p.T;
  int gt = 0, eq = 0;
  for (int64_t t = t0 + threadIdx.x; t < t1; t += TK_THREADS) {
    const uint32_t key = f2key(sc[t]);
    gt += key > thr;
    eq += key == thr;
  }
  __shared__ int sg[TK_THREADS / 32], se[TK_THREADS / 32];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gt += __shfl_xor_sync(0xffffffffu, gt, off);
    eq += __shfl_xor_sync(0xffffffffu, eq, off);
  }
  if ((threadIdx.x & 31) == 0) {
    sg[threadIdx.x >> 5] = gt;
    se[threadIdx.x >> 5] = eq;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int G = 0, E = 0;
    for (int w = 0; w < TK_THREADS / 32; ++w) {
      G += sg[w];
      E += se[w];
    }
    p.cnt[(size_t)s * p.topk_chunks + blockIdx.x] = make_int2(G, E);
    if (blockIdx.x == 0) p.res[s] = make_int2((int)thr, (int)r.k3);
  }
}

// writes the selected token ids in ascending order
__global__ void __launch_bounds__(TK_THREADS) topk_write_kernel(DecodeParams p) {
  const int s = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int2 rs = p.res[s];
  const uint32_t thr = (uint32_t)rs.x;
  const int need_eq = rs.y;
  __shared__ int sh[2][TK_THREADS / 32];
  __shared__ int before[2];
  // keys above / equal to the threshold in all earlier chunks of the stream
  int gb = 0, eb = 0;
  for (int c = tid; c < (int)blockIdx.x; c += TK_THREADS) {
    const int2 v = p.cnt[(size_t)s * p.topk_chunks + c];
    gb += v.x;
    eb += v.y;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    gb += __shfl_xor_sync(0xffffffffu, gb, off);
    eb += __shfl_xor_sync(0xffffffffu, eb, off);
  }
  if (lane == 0) {
    sh[0][warp] = gb;
    sh[1][warp] = eb;
  }
  __syncthreads();
  if (tid == 0) {
    int G = 0, E = 0;
    for (int w = 0; w < TK_THREADS / 32; ++w) {
      G += sh[0][w];
      E += sh[1][w];
    }
    before[0] = G;
    before[1] = E;
  }
  __syncthreads();
  // each thread owns TOPK_CHUNK / TK_THREADS consecutive tokens
  constexpr int PER = TOPK_CHUNK / TK_THREADS;
  const int64_t t0 = (int64_t)blockIdx.x * TOPK_CHUNK + (int64_t)tid * PER;
  const float* sc = p.scores + (size_t)s * p.T;
  uint32_t keys[PER];
  int lg = 0, le = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int64_t t = t0 + i;
    keys[i] = (t < p.T) ? f2key(sc[t]) : 0u;
    const bool valid = t < p.T;
    lg += valid && keys[i] > thr;
    le += valid && keys[i] == thr;
  }
  // exclusive scan of the packed (gt, eq) counts over the block
  uint32_t v = (uint32_t)lg | ((uint32_t)le << 16);
  uint32_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  __shared__ uint32_t wsum[TK_THREADS / 32];
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  uint32_t wbefore = 0;
  for (int w = 0; w < warp; ++w) wbefore += wsum[w];
  const uint32_t excl = wbefore + inc - v;
  int g_prior = before[0] + (int)(excl & 0xffffu);
  int e_prior = before[1] + (int)(excl >> 16);
  int32_t* out = p.sel + (size_t)s * p.kk;
  int32_t* out2 = p.sel_user ? p.sel_user + (size_t)s * p.kk : nullptr;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int64_t t = t0 + i;
    if (t >= p.T) break;
    const bool isg = keys[i] > thr, ise = keys[i] == thr;
    if (isg || (ise && e_prior < need_eq)) {
      const int pos = g_prior + min(e_prior, need_eq);
      if (pos >= p.kk) break;   // cannot happen with consistent histograms
      out[pos] = (int32_t)t;
      if (out2) out2[pos] = (int32_t)t;
    }
    g_prior += isg;
    e_prior += ise;
  }
}

// ---------------------------------------------------------------------------
// attn: split-K attention of the g query heads over a chunk of selected tokens,
// reading the packed K/V rows in place (values + channel indices).
// Partials per (stream, chunk, head): max logit m, sum of exp l, and the
// unnormalised output in the rotated V basis.
// grid: (attn_chunks, BH), block: 128 (4 warps)
// ---------------------------------------------------------------------------
constexpr int ATTN_WARPS = 4;

__device__ __forceinline__ int64_t clamp_t(int32_t t, int64_t T) {
  return t < 0 ? 0 : (t >= T ? T - 1 : (int64_t)t);
}

struct RowRef {
  const __half* vals;
  const uint8_t* idx;   // nullptr for dense rows
  int nnz;
};

__device__ __forceinline__ RowRef row_ref(const uint8_t* pool, const mkv_segment_header* hdr,
                                          int64_t t, int S, int c) {
  const int64_t sg = t / S;   // t is clamped to [0, T) by the caller
  const int r = (int)(t - sg * S);
  const mkv_segment_header hd = hdr[sg];
  const uint8_t* base = pool + (size_t)hd.off16 * 16u;
  RowRef rr;
  if (hd.strategy == MKV_STRATEGY_SM) {
    rr.idx = base;
    rr.vals = reinterpret_cast<const __half*>(base + pad16((uint32_t)c) + 2u * (uint32_t)c * r);
    rr.nnz = c;
  } else if (hd.strategy == MKV_STRATEGY_PV) {
    rr.vals = reinterpret_cast<const __half*>(base + 2u * (uint32_t)c * r);
    rr.idx = base + 2u * (uint32_t)c * hd.rows + (uint32_t)c * r;
    rr.nnz = c;
  } else {
    rr.vals = reinterpret_cast<const __half*>(base + 256u * r);
    rr.idx = nullptr;
    rr.nnz = D;
  }
  return rr;
}

__global__ void __launch_bounds__(128) attn_kernel(DecodeParams p) {
  extern __shared__ __align__(16) float sm[];
  const int s = blockIdx.y, ch = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* qs = sm;                                  // [g][128]
  float* acc = qs + g * D;                         // [4][g][128]
  float* lg = acc + ATTN_WARPS * g * D;            // [chunk][g]
  float* ml = lg + p.attn_chunk * g;               // [g][2]
  const float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * g) * D;
  for (int x = threadIdx.x; x < g * D; x += blockDim.x) qs[x] = qt[x];
  for (int x = threadIdx.x; x < ATTN_WARPS * g * D; x += blockDim.x) acc[x] = 0.f;
  __syncthreads();
  const int j0 = ch * p.attn_chunk;
  const int n = min(p.attn_chunk, p.kk - j0);
  const int32_t* sel = p.sel + (size_t)s * p.kk + j0;
  const mkv_segment_header* hK = p.hdrK + (size_t)s * p.n_seg;
  const mkv_segment_header* hV = p.hdrV + (size_t)s * p.n_seg;
  const float scale = 0.08838834764831845f;   // 1 / sqrt(128)

  // logits
  for (int i = warp; i < n; i += ATTN_WARPS) {
    const RowRef rr = row_ref(p.pool, hK, clamp_t(sel[i], p.T), p.S, p.c);
    float part[MAX_G];
#pragma unroll
    for (int hh = 0; hh < MAX_G; ++hh) part[hh] = 0.f;
    for (int j = lane; j < rr.nnz; j += 32) {
      const float v = __half2float(rr.vals[j]);
      const int chn = rr.idx ? (rr.idx[j] & 127) : j;
#pragma unroll
      for (int hh = 0; hh < MAX_G; ++hh)
        if (hh < g) part[hh] = fmaf(qs[hh * D + chn], v, part[hh]);
    }
#pragma unroll
    for (int hh = 0; hh < MAX_G; ++hh) {
      if (hh < g) {
        float x = part[hh];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) lg[i * g + hh] = x * scale;
      }
    }
  }
  __syncthreads();
  // softmax statistics of the chunk (one thread per head, token order)
  if ((int)threadIdx.x < g) {
    const int hh = threadIdx.x;
    float m = -INFINITY;
    for (int i = 0; i < n; ++i) m = fmaxf(m, lg[i * g + hh]);
    float l = 0.f;
    for (int i = 0; i < n; ++i) {
      const float e = expf(lg[i * g + hh] - m);
      lg[i * g + hh] = e;
      l += e;
    }
    ml[hh * 2] = m;
    ml[hh * 2 + 1] = l;
  }
  __syncthreads();
  // sum_t p_t v^_t into per-warp accumulators (channels of one row are distinct)
  float* myacc = acc + warp * g * D;
  for (int i = warp; i < n; i += ATTN_WARPS) {
    const RowRef rr = row_ref(p.pool, hV, clamp_t(sel[i], p.T), p.S, p.c);
    for (int j = lane; j < rr.nnz; j += 32) {
      const float v = __half2float(rr.vals[j]);
      const int chn = rr.idx ? (rr.idx[j] & 127) : j;
      for (int hh = 0; hh < g; ++hh) myacc[hh * D + chn] = fmaf(lg[i * g + hh], v, myacc[hh * D + chn]);
    }
    __syncwarp();
  }
  __syncthreads();
  const size_t pbase = ((size_t)s * p.attn_chunks + ch) * g;
  for (int x = threadIdx.x; x < g * D; x += blockDim.x) {
    float o = 0.f;
#pragma unroll
    for (int w = 0; w < ATTN_WARPS; ++w) o += acc[w * g * D + x];
    p.part_o[pbase * D + x] = o;
  }
  if ((int)threadIdx.x < 2 * g) p.part_ml[pbase * 2 + threadIdx.x] = ml[threadIdx.x];
}

// ---------------------------------------------------------------------------
// merge: log-sum-exp merge of the chunk partials, then o = o~ R_V^T.
// grid: BH, block: 128
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) merge_kernel(DecodeParams p) {
  const int s = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g;
  const int x = threadIdx.x, warp = x >> 5, lane = x & 31;
  __shared__ __align__(16) float ot[MAX_G][D];
  for (int hh = 0; hh < g; ++hh) {
    float M = -INFINITY;
    for (int c = 0; c < p.attn_chunks; ++c)
      M = fmaxf(M, p.part_ml[(((size_t)s * p.attn_chunks + c) * g + hh) * 2]);
    float L = 0.f, o = 0.f;
    for (int c = 0; c < p.attn_chunks; ++c) {
      const size_t pi = ((size_t)s * p.attn_chunks + c) * g + hh;
      const float w = expf(p.part_ml[pi * 2] - M);
      L = fmaf(p.part_ml[pi * 2 + 1], w, L);
      o = fmaf(p.part_o[pi * D + x], w, o);
    }
    ot[hh][x] = o / L;
  }
  __syncthreads();
  const float* RV = p.RV + (size_t)s * D * D;
  float* out = p.out + ((size_t)b * p.Hq + (size_t)h * g) * D;
  for (int r = warp; r < D; r += 4) {
    float rv[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) rv[m] = RV[r * D + lane + 32 * m];
    for (int hh = 0; hh < g; ++hh) {
      float d = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) d = fmaf(rv[m], ot[hh][lane + 32 * m], d);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
      if (lane == 0) out[hh * D + r] = d;
    }
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_qrot(const DecodeParams& p, cudaStream_t st) {
  qrot_kernel<<<p.B * p.H, 128, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_score(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.score_ctas_per_stream, p.B * p.H);
  score_kernel<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.topk_chunks, p.B * p.H);
  topk_hist_kernel<2><<<grid, TK_THREADS, 0, st>>>(p);
  topk_hist_kernel<3><<<grid, TK_THREADS, 0, st>>>(p);
  topk_count_kernel<<<grid, TK_THREADS, 0, st>>>(p);
  topk_write_kernel<<<grid, TK_THREADS, 0, st>>>(p);
  return cudaGetLastError();
}

size_t attn_smem_bytes(int g, int chunk) {
  return sizeof(float) * ((size_t)g * D + (size_t)ATTN_WARPS * g * D + (size_t)chunk * g + 2 * g);
}

cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st) {
  const size_t smem = attn_smem_bytes(p.g, p.attn_chunk);
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.attn_chunks, p.B * p.H);
  attn_kernel<<<grid, 128, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st) {
  merge_kernel<<<p.B * p.H, 128, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mkv
