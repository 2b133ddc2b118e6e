// Decode step, last part: attention over the selected tokens, read in place
// from the packed cache, and the output rotation back to the original basis.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction, "Observation & Method 2":
// attention computed on the packed dense format without unpacking.
#include "decode_common.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// attn: split-K attention of the g query heads over a chunk of <= 128
// selected tokens, reading the packed K/V rows in place (fp16 values + uint8
// channel indices).  Row addresses of the chunk are resolved first.  Then a
// group of 8 lanes serves a token, one 16-byte chunk (8 stored values) per
// lane, and every thread fetches the chunks of its tokens together: K chunks
// give partial logits (summed over the 8 lanes by a fixed butterfly), V
// chunks are copied into a zeroed fp16 tile V[token][channel].  The softmax
// weights p (fp32) are split into fp16 hi + 2^11 * lo parts, stored
// transposed P[head][token], and o~ = P V runs on tensor cores (mma.sync,
// fp32 accumulation, one accumulator per part): warp w owns channels
// [32w, 32w + 32).  Partials per (stream, chunk, head): max logit m, sum of
// exp l and the unnormalised output in the rotated V basis.
// grid: (attn_chunks, BH), block 128, dynamic smem
// ---------------------------------------------------------------------------
constexpr int ATTN_THREADS = 128;
constexpr int VLD = 136;            // halves per V tile row (272 B: ldmatrix without conflicts)
constexpr int PLD = 136;            // halves per P row

constexpr int32_t NO_IDX = (int32_t)0x80000000;

// Row of token t in one stream: pool offset of its stored values / 16, and
// the byte distance / 8 from the values to the row's channel list (the
// segment mask for SM, the row's own indices for PV; NO_IDX for dense rows).
__device__ __forceinline__ uint2 row_meta(const mkv_segment_header* hdr, int64_t t, int S, int c) {
  const int64_t sg = t / S;
  const uint32_t r = (uint32_t)(t - sg * S);
  const mkv_segment_header hd = hdr[sg];
  const uint32_t c2 = 2u * (uint32_t)c;
  if (hd.strategy == MKV_STRATEGY_SM) {
    const uint32_t dv = pad16((uint32_t)c) + c2 * r;       // values after the mask
    return make_uint2(hd.off16 + dv / 16u, (uint32_t)(-(int32_t)(dv / 8u)));
  }
  if (hd.strategy == MKV_STRATEGY_PV) {
    const uint32_t dv = c2 * r;
    return make_uint2(hd.off16 + dv / 16u, (uint32_t)c * (2u * hd.rows - r) / 8u);
  }
  return make_uint2(hd.off16 + 16u * r, (uint32_t)NO_IDX);
}

// One past the last pool byte that the row (values and channel list) spans.
__device__ __forceinline__ uint64_t row_end(const uint2& m, int c) {
  const uint64_t v0 = (uint64_t)m.x * 16u;
  if ((int32_t)m.y == NO_IDX) return v0 + 256u;
  const uint64_t vend = v0 + 2u * (uint32_t)c;
  const uint64_t iend = (uint64_t)((int64_t)v0 + 8 * (int64_t)(int32_t)m.y) + (uint32_t)c;
  return vend > iend ? vend : iend;
}

// tokens of a chunk rounded up to the mma K step
__host__ __device__ constexpr int attn_rows16(int chunk) { return (chunk + 15) & ~15; }

size_t attn_smem_bytes(int g, int chunk) {
  const int gp = (g + 3) & ~3;
  return (size_t)attn_rows16(chunk) * VLD * 2 + 2 * MAX_G * PLD * 2 + (size_t)chunk * 16 +
         sizeof(float) * ((size_t)D * gp + (size_t)chunk * gp + 2 * g);
}

__device__ __forceinline__ int chan_of(const uint2& x, int e) {
  return (int)(((e < 4 ? x.x : x.y) >> (8 * (e & 3))) & 0x7fu);
}

// everything after the row addresses; GM = heads per instantiation (4 or 16)
template <int GM>
__device__ __forceinline__ void attn_body(const DecodeParams& p, int s, int chk, int n,
                                          const uint4* __restrict__ meta,
                                          __half* __restrict__ Vd, __half* __restrict__ Pt,
                                          const float* __restrict__ qs, float* __restrict__ lg,
                                          float* __restrict__ ml) {
  const int g = p.g, gp = (g + 3) & ~3;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cl = tid & 7, tg = tid >> 3;
  const int c = p.c;
  constexpr int U = 4;                          // tokens per thread per batch
  const float scale = 0.08838834764831845f;     // 1 / sqrt(128)
  // ---- logits and V tile: 8 lanes per token, 8 tokens per thread ---------
  for (int base = 0; base < ATTN_THREADS / 16 && 16 * base < n; base += U) {
    uint4 mt[U], kvv[U], vvv[U];
    uint2 kix[U], vix[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = tg + 16 * (base + u);
      mt[u] = i < n ? meta[i] : make_uint4(0u, (uint32_t)NO_IDX, 0u, (uint32_t)NO_IDX);
      kvv[u] = vvv[u] = make_uint4(0u, 0u, 0u, 0u);
      kix[u] = vix[u] = make_uint2(0u, 0u);
      if (i < n) {
        const bool kd = (int32_t)mt[u].y == NO_IDX, vd = (int32_t)mt[u].w == NO_IDX;
        const uint8_t* kp = p.pool + (uint64_t)mt[u].x * 16u;
        const uint8_t* vp = p.pool + (uint64_t)mt[u].z * 16u;
        if (8 * cl < (kd ? D : c)) {
          kvv[u] = ld_cg_u4(kp + 16 * cl);
          if (!kd) kix[u] = ld_cg_u2(kp + 8 * (int64_t)(int32_t)mt[u].y + 8 * cl);
        }
        if (8 * cl < (vd ? D : c)) {
          vvv[u] = ld_cg_u4(vp + 16 * cl);
          if (!vd) vix[u] = ld_cg_u2(vp + 8 * (int64_t)(int32_t)mt[u].w + 8 * cl);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = tg + 16 * (base + u);
      const bool kd = (int32_t)mt[u].y == NO_IDX, vd = (int32_t)mt[u].w == NO_IDX;
      const int kn = kd ? D : c, vn = vd ? D : c;
      float part[GM];
#pragma unroll
      for (int hh = 0; hh < GM; ++hh) part[hh] = 0.f;
      if (i < n) {
        // rows with more than 64 stored values (dense, or c > 64) have chunks 8..15
        for (int ck = cl; ck < 16; ck += 8) {
          uint4 kr = kvv[u], vr = vvv[u];
          uint2 kx = kix[u], vx = vix[u];
          if (ck >= 8) {
            if (8 * ck >= kn && 8 * ck >= vn) break;
            const uint8_t* kp = p.pool + (uint64_t)mt[u].x * 16u;
            const uint8_t* vp = p.pool + (uint64_t)mt[u].z * 16u;
            kr = vr = make_uint4(0u, 0u, 0u, 0u);
            kx = vx = make_uint2(0u, 0u);
            if (8 * ck < kn) {
              kr = ld_cg_u4(kp + 16 * ck);
              if (!kd) kx = ld_cg_u2(kp + 8 * (int64_t)(int32_t)mt[u].y + 8 * ck);
            }
            if (8 * ck < vn) {
              vr = ld_cg_u4(vp + 16 * ck);
              if (!vd) vx = ld_cg_u2(vp + 8 * (int64_t)(int32_t)mt[u].w + 8 * ck);
            }
          }
          if (8 * ck < vn) {
            const __half* hv = reinterpret_cast<const __half*>(&vr);
            __half* vrow = Vd + (size_t)i * VLD;
#pragma unroll
            for (int e = 0; e < 8; ++e) vrow[vd ? 8 * ck + e : chan_of(vx, e)] = hv[e];
          }
          if (8 * ck < kn) {
            float v[8];
            h8_to_f(kr, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float* qq = qs + (kd ? 8 * ck + e : chan_of(kx, e)) * gp;
#pragma unroll
              for (int h4 = 0; h4 < GM; h4 += 4) {
                if (h4 < g) {
                  const float4 q4 = *reinterpret_cast<const float4*>(qq + h4);
                  part[h4] = fmaf(q4.x, v[e], part[h4]);
                  part[h4 + 1] = fmaf(q4.y, v[e], part[h4 + 1]);
                  part[h4 + 2] = fmaf(q4.z, v[e], part[h4 + 2]);
                  part[h4 + 3] = fmaf(q4.w, v[e], part[h4 + 3]);
                }
              }
            }
          }
        }
      }
      // sum over the token's 8 lanes (fixed butterfly order)
#pragma unroll
      for (int hh = 0; hh < GM; ++hh) {
        if (hh < gp) {
          float x = part[hh];
          x += __shfl_xor_sync(0xffffffffu, x, 1);
          x += __shfl_xor_sync(0xffffffffu, x, 2);
          x += __shfl_xor_sync(0xffffffffu, x, 4);
          if (cl == 0 && i < n) lg[i * gp + hh] = x * scale;
        }
      }
    }
  }
  __syncthreads();
  // ---- softmax per head (warp per head, fixed-order reductions); weights go
  // to P[head][token] as fp16 hi and 2^11 * (p - hi) ----------------------
  __half* Ph = Pt;
  __half* Pl = Pt + MAX_G * PLD;
  for (int hh = warp; hh < g; hh += ATTN_THREADS / 32) {
    float m = -INFINITY;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, lg[i * gp + hh]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float e = expf(lg[i * gp + hh] - m);
      const __half hi = __float2half_rn(e);
      Ph[hh * PLD + i] = hi;
      Pl[hh * PLD + i] = __float2half_rn((e - __half2float(hi)) * 2048.f);
      l += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
    if (lane == 0) {
      ml[hh * 2] = m;
      ml[hh * 2 + 1] = l;
    }
  }
  __syncthreads();
  // ---- o~ = P V on tensor cores: warp w, channels [32w, 32w + 32) ----------
  float ch_[4][4], cl_[4][4];
#pragma unroll
  for (int a = 0; a < 4; ++a)
#pragma unroll
    for (int e = 0; e < 4; ++e) ch_[a][e] = cl_[a][e] = 0.f;
  const int mm = lane >> 3, r8 = lane & 7;
  const uint32_t ph = smem_u32(Ph), pl = smem_u32(Pl), vd = smem_u32(Vd);
  const int ksteps = (n + 15) >> 4;
  for (int ks = 0; ks < ksteps; ++ks) {
    const int k0 = ks * 16;
    uint32_t ah[4], al[4];
    const uint32_t aoff = (uint32_t)(((r8 + (mm & 1) * 8) * PLD + k0 + (mm >> 1) * 8) * 2);
    ldsm_x4(ph + aoff, ah);
    ldsm_x4(pl + aoff, al);
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      uint32_t bb[4];
      const int row = k0 + (mm & 1) * 8 + r8;
      const int col = warp * 32 + np * 16 + (mm >> 1) * 8;
      ldsm_x4_t(vd + (uint32_t)((row * VLD + col) * 2), bb);
      mma16816(ch_[2 * np], ah, bb[0], bb[1]);
      mma16816(ch_[2 * np + 1], ah, bb[2], bb[3]);
      mma16816(cl_[2 * np], al, bb[0], bb[1]);
      mma16816(cl_[2 * np + 1], al, bb[2], bb[3]);
    }
  }
  const size_t pbase = ((size_t)s * p.attn_chunks + chk) * g;
  const int h0 = lane >> 2, c0 = warp * 32 + 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int chn = c0 + nt * 8;
    if (h0 < g)
      *reinterpret_cast<float2*>(p.part_o + (pbase + h0) * D + chn) =
          make_float2(fmaf(cl_[nt][0], 1.f / 2048.f, ch_[nt][0]),
                      fmaf(cl_[nt][1], 1.f / 2048.f, ch_[nt][1]));
    if (h0 + 8 < g)
      *reinterpret_cast<float2*>(p.part_o + (pbase + h0 + 8) * D + chn) =
          make_float2(fmaf(cl_[nt][2], 1.f / 2048.f, ch_[nt][2]),
                      fmaf(cl_[nt][3], 1.f / 2048.f, ch_[nt][3]));
  }
  if (tid < 2 * g) p.part_ml[pbase * 2 + tid] = ml[tid];
}

// GM: heads per instantiation (4 or 16); MINB: resident CTAs per SM asked of
// the register allocator (6 for chunks of <= 64 tokens and g <= 4).
template <int GM, int MINB>
__global__ void __launch_bounds__(ATTN_THREADS, MINB) attn_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t asm_[];
  const int s = blockIdx.y, chk = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g, gp = (g + 3) & ~3;
  const int tid = threadIdx.x;
  const int CH = p.attn_chunk;
  const int R16 = attn_rows16(CH);
  __half* Vd = reinterpret_cast<__half*>(asm_);                                // [R16][VLD]
  __half* Pt = Vd + (size_t)R16 * VLD;                                         // [2][16][PLD]
  uint4* meta = reinterpret_cast<uint4*>(Pt + 2 * MAX_G * PLD);               // [CH]
  float* qs = reinterpret_cast<float*>(meta + CH);                             // [128][gp]
  float* lg = qs + D * gp;                                                     // [CH][gp]
  float* ml = lg + CH * gp;                                                    // [g][2]
  const float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * g) * D;
  for (int x = tid; x < D * gp; x += ATTN_THREADS) {
    const int chn = x / gp, hh = x % gp;
    qs[x] = hh < g ? qt[hh * D + chn] : 0.f;
  }
  {
    // the V tile and both P parts start at zero (rows past n, heads past g)
    uint4* z = reinterpret_cast<uint4*>(Vd);
    const int nz = (R16 * VLD + 2 * MAX_G * PLD) / 8;
    for (int x = tid; x < nz; x += ATTN_THREADS) z[x] = make_uint4(0u, 0u, 0u, 0u);
  }
  const int j0 = chk * CH;
  const int n = min(CH, p.kk - j0);
  // q~ (from the rotation kernel, two launches back) and the ctx's headers
  // are ready; the selection is not
  griddep_wait();
  griddep_launch();
  if (tid < n) {
    const int64_t t = clamp_t(p.sel[(size_t)s * p.kk + j0 + tid], p.T);
    uint2 km = row_meta(p.hdrK + (size_t)s * p.n_seg, t, p.S, p.c);
    uint2 vm = row_meta(p.hdrV + (size_t)s * p.n_seg, t, p.S, p.c);
    if (row_end(km, p.c) > p.pool_check || row_end(vm, p.c) > p.pool_check) {
      // outside the checked pool extent: report it and read a dense row at
      // offset 0 instead (inside every pool)
      atomicOr(p.err, DEV_ERR_CHECK);
      km = vm = make_uint2(0u, (uint32_t)NO_IDX);
    }
    meta[tid] = make_uint4(km.x, km.y, vm.x, vm.y);
  }
  __syncthreads();
  attn_body<GM>(p, s, chk, n, meta, Vd, Pt, qs, lg, ml);
}

// ---------------------------------------------------------------------------
// merge: log-sum-exp merge of the chunk partials, then o = o~ R_V^T.  CTA
// (s, q) writes output rows [32q, 32q + 32) of every head of stream s; the
// weights and the merged o~ are recomputed by each of the four CTAs (from
// L2), and the 32 rows of R_V are staged transposed in shared memory.
// grid: (BH, 4), block 128, dynamic smem: chunk weights
// ---------------------------------------------------------------------------
constexpr int MG_THREADS = 128;
constexpr int MG_ROWS = 32;
constexpr int MG_LD = MG_ROWS + 1;

__global__ void __launch_bounds__(MG_THREADS) merge_kernel(DecodeParams p) {
  extern __shared__ __align__(16) float wsm[];     // [attn_chunks][g] weights
  __shared__ float Rt[D * MG_LD];                  // Rt[j][rr] = R_V[32q + rr][j]
  __shared__ __align__(16) float ot[MAX_G][D];
  __shared__ float Linv[MAX_G];
  const int s = blockIdx.x, r0 = blockIdx.y * MG_ROWS;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g, nc = p.attn_chunks;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    const float4* R4 = reinterpret_cast<const float4*>(p.RV + ((size_t)s * D + r0) * D);
#pragma unroll
    for (int x = 0; x < MG_ROWS * D / 4 / MG_THREADS; ++x) {
      const int f = tid + x * MG_THREADS;           // float4 index within the 32 rows
      const int rr = f >> 5, j = (f & 31) * 4;
      const float4 v = __ldg(R4 + f);
      Rt[(j + 0) * MG_LD + rr] = v.x;
      Rt[(j + 1) * MG_LD + rr] = v.y;
      Rt[(j + 2) * MG_LD + rr] = v.z;
      Rt[(j + 3) * MG_LD + rr] = v.w;
    }
  }
  griddep_wait();     // the partials come from the attention kernel
  griddep_launch();
  // weights exp(m_c - M) and 1 / L per head: warp per head, lanes over chunks
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml + (size_t)s * nc * g * 2);
  for (int hh = warp; hh < g; hh += MG_THREADS / 32) {
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldg(ml + c * g + hh).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int c = lane; c < nc; c += 32) {
      const float2 v = __ldg(ml + c * g + hh);
      const float w = expf(v.x - M);
      wsm[c * g + hh] = w;
      L = fmaf(v.y, w, L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) Linv[hh] = 1.f / L;
  }
  __syncthreads();
  const float* po = p.part_o + (size_t)s * nc * g * D;
  for (int x = tid; x < g * D; x += MG_THREADS) {
    const int hh = x / D;
    float o = 0.f;
#pragma unroll 32
    for (int c = 0; c < nc; ++c) o = fmaf(__ldg(po + (size_t)c * g * D + x), wsm[c * g + hh], o);
    ot[hh][x % D] = o * Linv[hh];
  }
  __syncthreads();
  // thread (rr, hq): out[hh][r0 + rr] for hh = hq, hq + 4, ...
  float* out = p.out + ((size_t)b * p.Hq + (size_t)h * g) * D;
  const int rr = tid & 31, hq = tid >> 5;
  for (int hh = hq; hh < g; hh += MG_THREADS / 32) {
    float d0 = 0.f, d1 = 0.f;
#pragma unroll 8
    for (int j = 0; j < D; j += 2) {
      d0 = fmaf(Rt[j * MG_LD + rr], ot[hh][j], d0);
      d1 = fmaf(Rt[(j + 1) * MG_LD + rr], ot[hh][j + 1], d1);
    }
    out[hh * D + r0 + rr] = d0 + d1;
  }
}

cudaError_t prepare_attn_kernels() {
  const int mx = (int)attn_smem_bytes(MAX_G, ATTN_MAX_CHUNK);
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<4, 6>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_kernel<4, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_kernel<MAX_G, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              48 * 1024 + 4 * 1024);
}

cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.attn_chunks, p.B * p.H);
  const size_t smem = attn_smem_bytes(p.g, p.attn_chunk);
  const bool pdl = p.pdl != 0;
  if (p.g <= 4 && p.attn_chunk <= 64)
    return launch_kernel(attn_kernel<4, 6>, grid, dim3(ATTN_THREADS), smem, st, pdl, 0, p);
  if (p.g <= 4) return launch_kernel(attn_kernel<4, 4>, grid, dim3(ATTN_THREADS), smem, st, pdl, 0, p);
  return launch_kernel(attn_kernel<MAX_G, 4>, grid, dim3(ATTN_THREADS), smem, st, pdl, 0, p);
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st) {
  return launch_kernel(merge_kernel, dim3(p.B * p.H, D / MG_ROWS), dim3(MG_THREADS),
                       sizeof(float) * (size_t)p.attn_chunks * p.g, st, p.pdl != 0, 0, p);
}

}  // namespace mkv
