// Prefill compression kernels.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction, "Observation & Method 1":
// rotate each KV head's vectors into an SVD basis, pick important elements per
// vector, split the cache into segments and give each segment a strategy;
// "Observation & Method 2": pack the sparse result into a dense format.
//
// Per stream (b, h, X in {K, V}):
//   gram     G = X^T X over all tokens (tensor cores, fp16 in, fp32 accumulate),
//            split over CTAs; partial Grams are summed in a fixed order later.
//   eig      cyclic Jacobi on G in fp32 (one CTA per stream), then sort by
//            descending eigenvalue, fix column signs, write R and lambda.
//   analyze  x~ = x R on tensor cores with R split into fp16 hi + lo parts
//            (lo scaled by 2^11 so it stays a normal fp16, own accumulator),
//            per-token top-c channels, per-segment energies and strategy.
//   scan     exclusive scan of the packed segment sizes -> headers, total.
//   pack     same rotation and selection again, writes the packed payload.
#include "mkv_internal.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// PTX helpers (sm_80+ instructions that sm_103a keeps)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A [rows][128] fp16 tile in shared memory: 256-byte rows of 16 chunks of 16 B,
// chunk index XOR (row & 7) so that 8 rows at one logical chunk hit 8
// different bank groups.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 256 + ((chunk ^ (row & 7)) << 4));
}

// Loads tokens [t0, t0+64) of a stream into a swizzled tile; rows at or past T
// are zero-filled.
__device__ __forceinline__ void load_tile(uint32_t tile, const __half* X, int64_t t0, int64_t T) {
  for (int i = threadIdx.x; i < TILE_T * 16; i += blockDim.x) {
    const int row = i >> 4, chunk = i & 15;
    const int64_t t = t0 + row;
    const bool ok = t < T;
    const __half* src = X + (ok ? t : 0) * D + chunk * 8;
    cp_async16(tile + swz(row, chunk), src, ok ? 16u : 0u);
  }
}

// ---------------------------------------------------------------------------
// gram: partial G over one chunk of tokens.  8 warps; warp w owns the 32 x 64
// block G[i0:i0+32, j0:j0+64].  A = X^T and B = X both come from the token-major
// tile through ldmatrix.trans.  The tensor-core accumulators take GR_FLUSH
// tiles at a time and are then added into a separate fp32 sum: tensor-core
// accumulation does not round to nearest, so its error grows with the number
// of products summed in one accumulator; flushing keeps G good to a few 1e-6
// relative at any context length.
// grid: (gram_chunks, BH, 2), block 256, dynamic smem 3 x 16 KB
// ---------------------------------------------------------------------------
constexpr int GR_STAGES = 3;
constexpr int GR_FLUSH = 2;     // tiles (of 64 tokens) per accumulator flush

__global__ void __launch_bounds__(256) gram_kernel(CompressParams p) {
  extern __shared__ __align__(128) uint8_t gsm[];
  const int chunk = blockIdx.x, s = blockIdx.y, x = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const __half* X = p.X[x] + (size_t)s * p.T * D;
  const int64_t tb = (int64_t)chunk * p.gram_chunk_tokens;
  const int64_t te = imin64(p.T, tb + p.gram_chunk_tokens);
  const int n_tiles = te > tb ? (int)((te - tb + TILE_T - 1) / TILE_T) : 0;
  const uint32_t base = smem_u32(gsm);
  const int i0 = (warp & 3) * 32, j0 = (warp >> 2) * 64;

  float acc[2][8][4], tot[2][8][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[a][b][e] = tot[a][b][e] = 0.f;

  for (int st = 0; st < GR_STAGES - 1; ++st) {
    if (st < n_tiles) load_tile(base + st * 16384u, X, tb + (int64_t)st * TILE_T, te);
    cp_async_commit();
  }
  const int mm = lane >> 3, r8 = lane & 7;
  for (int it = 0; it < n_tiles; ++it) {
    cp_async_wait<GR_STAGES - 2>();
    __syncthreads();
    const int nxt = it + GR_STAGES - 1;
    if (nxt < n_tiles) load_tile(base + (nxt % GR_STAGES) * 16384u, X, tb + (int64_t)nxt * TILE_T, te);
    cp_async_commit();
    const uint32_t tile = base + (it % GR_STAGES) * 16384u;
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const int kt0 = ks * 16;
      uint32_t a[2][4];
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int row = kt0 + (mm >> 1) * 8 + r8;
        const int ch = (i0 + mi * 16 + (mm & 1) * 8) >> 3;
        ldsm_x4_t(tile + swz(row, ch), a[mi]);
      }
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t bb[4];
        const int row = kt0 + (mm & 1) * 8 + r8;
        const int ch = (j0 + np * 16 + (mm >> 1) * 8) >> 3;
        ldsm_x4_t(tile + swz(row, ch), bb);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
          mma16816(acc[mi][2 * np], a[mi], bb[0], bb[1]);
          mma16816(acc[mi][2 * np + 1], a[mi], bb[2], bb[3]);
        }
      }
    }
    if ((it + 1) % GR_FLUSH == 0 || it + 1 == n_tiles) {
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            tot[a][b][e] += acc[a][b][e];
            acc[a][b][e] = 0.f;
          }
    }
  }
  cp_async_wait<0>();
  float* out = p.gram_part + (((size_t)x * p.BH + s) * p.gram_chunks + chunk) * (D * D);
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 8; ++ni) {
      const int i = i0 + mi * 16 + g, j = j0 + ni * 8 + 2 * q;
      *reinterpret_cast<float2*>(out + i * D + j) = make_float2(tot[mi][ni][0], tot[mi][ni][1]);
      *reinterpret_cast<float2*>(out + (i + 8) * D + j) = make_float2(tot[mi][ni][2], tot[mi][ni][3]);
    }
}

// ---------------------------------------------------------------------------
// eig: symmetric eigendecomposition of one stream's G (fp32 cyclic Jacobi with
// the round-robin parallel ordering: 64 disjoint rotations per round, 127
// rounds per sweep).  Refinement: after the first solve the accumulated
// rotations V are re-orthonormalised (one Newton-Schulz step) and A = V^T G V
// is formed afresh from the original G, then swept again; this removes the
// rounding drift that in-place updates leave in A, so the eigen-residual is
// set by the fp32 rounding of the products (about sqrt(n) eps_32 of ||G||).
// Eigenvalues are sorted descending (ties to the lower index), and each
// column's largest-magnitude entry is made positive (ties to the lower row).
// grid: 2 * BH, block 512, dynamic smem 3 x 128 x 129 floats
// ---------------------------------------------------------------------------
constexpr int EIG_THREADS = 512;
constexpr int LDA = D + 1;
constexpr int EIG_MAX_SWEEPS = 16;
constexpr int EIG_REFINE_SWEEPS = 6;

__device__ __forceinline__ int rr_player(int pos, int round) {
  return pos == 0 ? 0 : 1 + (pos - 1 + round) % (D - 1);
}

struct EigShared {
  float cs[64], sn[64], tt[64];
  int top[64], bot[64];
  int rotated;
};

// Jacobi sweeps on A (in place), accumulating the rotations into V, until a
// sweep rotates nothing or max_sweeps have run.  Block-wide.
__device__ void jacobi_sweeps(float* A, float* V, int max_sweeps, EigShared& sh) {
  const int tid = threadIdx.x;
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    if (tid == 0) sh.rotated = 0;
    __syncthreads();
    for (int round = 0; round < D - 1; ++round) {
      if (tid < 64) {
        int a = rr_player(tid, round), b = rr_player(D - 1 - tid, round);
        const int pp = min(a, b), qq = max(a, b);
        const float app = A[pp * LDA + pp], aqq = A[qq * LDA + qq], apq = A[pp * LDA + qq];
        float c = 1.f, s = 0.f, t = 0.f;
        if (apq != 0.f && fabsf(apq) > 1e-7f * sqrtf(fabsf(app * aqq))) {
          const float th = (aqq - app) / (2.f * apq);
          t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(1.f + th * th));
          c = 1.f / sqrtf(1.f + t * t);
          s = t * c;
          sh.rotated = 1;
        }
        sh.cs[tid] = c;
        sh.sn[tid] = s;
        sh.tt[tid] = t;
        sh.top[tid] = pp;
        sh.bot[tid] = qq;
      }
      __syncthreads();
      for (int blk = tid; blk < 64 * 64; blk += EIG_THREADS) {
        const int P = blk >> 6, Q = blk & 63;
        const int p1 = sh.top[P], p2 = sh.bot[P];
        if (P == Q) {
          const float apq = A[p1 * LDA + p2], t = sh.tt[P];
          A[p1 * LDA + p1] -= t * apq;
          A[p2 * LDA + p2] += t * apq;
          A[p1 * LDA + p2] = 0.f;
          A[p2 * LDA + p1] = 0.f;
        } else {
          const int q1 = sh.top[Q], q2 = sh.bot[Q];
          const float cP = sh.cs[P], sP = sh.sn[P], cQ = sh.cs[Q], sQ = sh.sn[Q];
          const float b11 = A[p1 * LDA + q1], b12 = A[p1 * LDA + q2];
          const float b21 = A[p2 * LDA + q1], b22 = A[p2 * LDA + q2];
          const float u11 = cP * b11 - sP * b21, u12 = cP * b12 - sP * b22;
          const float u21 = sP * b11 + cP * b21, u22 = sP * b12 + cP * b22;
          A[p1 * LDA + q1] = cQ * u11 - sQ * u12;
          A[p1 * LDA + q2] = sQ * u11 + cQ * u12;
          A[p2 * LDA + q1] = cQ * u21 - sQ * u22;
          A[p2 * LDA + q2] = sQ * u21 + cQ * u22;
        }
      }
      for (int e = tid; e < D * 64; e += EIG_THREADS) {
        const int r = e >> 6, k = e & 63;
        const int pp = sh.top[k], qq = sh.bot[k];
        const float c = sh.cs[k], s = sh.sn[k];
        const float vp = V[r * LDA + pp], vq = V[r * LDA + qq];
        V[r * LDA + pp] = c * vp - s * vq;
        V[r * LDA + qq] = s * vp + c * vq;
      }
      __syncthreads();
    }
    const int any = sh.rotated;
    __syncthreads();
    if (!any) break;
  }
}

// C = op(X) Y for 128 x 128 matrices in shared memory (row stride LDA), with
// op(X) = X^T when TRANS_X.  Each thread owns D * D / EIG_THREADS entries of
// C; C must not alias X or Y.  Block-wide.
template <bool TRANS_X>
__device__ void smem_matmul(const float* X, const float* Y, float* C) {
  const int tid = threadIdx.x;
#pragma unroll 1
  for (int k = 0; k < D * D / EIG_THREADS; ++k) {
    const int e = tid + k * EIG_THREADS;
    const int r = e >> 7, cc = e & 127;
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i)
      acc = fmaf(TRANS_X ? X[i * LDA + r] : X[r * LDA + i], Y[i * LDA + cc], acc);
    C[r * LDA + cc] = acc;
  }
  __syncthreads();
}

// One Newton-Schulz step V <- V (1.5 I - 0.5 V^T V); W is scratch.
__device__ void newton_schulz(float* V, float* W) {
  const int tid = threadIdx.x;
  smem_matmul<true>(V, V, W);
  float nv[D * D / EIG_THREADS];
#pragma unroll
  for (int k = 0; k < D * D / EIG_THREADS; ++k) {
    const int e = tid + k * EIG_THREADS;
    const int r = e >> 7, a = e & 127;
    float acc = 0.f;
    for (int b = 0; b < D; ++b) acc = fmaf(V[r * LDA + b], W[b * LDA + a], acc);
    nv[k] = 1.5f * V[r * LDA + a] - 0.5f * acc;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < D * D / EIG_THREADS; ++k) {
    const int e = tid + k * EIG_THREADS;
    V[(e >> 7) * LDA + (e & 127)] = nv[k];
  }
  __syncthreads();
}

__global__ void __launch_bounds__(EIG_THREADS) eig_kernel(CompressParams p) {
  extern __shared__ __align__(16) float esm[];
  float* A = esm;
  float* V = esm + D * LDA;
  float* Gs = esm + 2 * D * LDA;
  __shared__ EigShared sh;
  __shared__ float lam[D];
  __shared__ int rank[D];
  __shared__ float sgn[D];
  const int sx = blockIdx.x;   // X * BH + s
  const int tid = threadIdx.x;
  const float* part = p.gram_part + (size_t)sx * p.gram_chunks * (D * D);
  for (int e = tid; e < D * D; e += EIG_THREADS) {
    float a = 0.f;
    for (int c = 0; c < p.gram_chunks; ++c) a += part[(size_t)c * D * D + e];
    const int i = e >> 7, j = e & 127;
    A[i * LDA + j] = a;
    V[i * LDA + j] = (i == j) ? 1.f : 0.f;
  }
  __syncthreads();
  // symmetrise: each (i, j), i < j, pair is owned by one thread; keep G
  for (int e = tid; e < D * D; e += EIG_THREADS) {
    const int i = e >> 7, j = e & 127;
    if (i < j) {
      const float v = 0.5f * (A[i * LDA + j] + A[j * LDA + i]);
      A[i * LDA + j] = v;
      A[j * LDA + i] = v;
      Gs[i * LDA + j] = v;
      Gs[j * LDA + i] = v;
    } else if (i == j) {
      Gs[i * LDA + i] = A[i * LDA + i];
    }
  }
  __syncthreads();

  jacobi_sweeps(A, V, EIG_MAX_SWEEPS, sh);
  // refinement: orthonormal V, then A = V^T G V from the original G
  newton_schulz(V, A);
  smem_matmul<false>(Gs, V, A);     // A = G V
  smem_matmul<true>(V, A, Gs);      // Gs = V^T G V
  float* Ar = Gs;
  float* W = A;
  for (int e = tid; e < D * D; e += EIG_THREADS) {
    const int i = e >> 7, j = e & 127;
    if (i < j) {
      const float v = 0.5f * (Ar[i * LDA + j] + Ar[j * LDA + i]);
      Ar[i * LDA + j] = v;
      Ar[j * LDA + i] = v;
    }
  }
  __syncthreads();
  jacobi_sweeps(Ar, V, EIG_REFINE_SWEEPS, sh);
  if (tid < D) lam[tid] = Ar[tid * LDA + tid];
  __syncthreads();
  newton_schulz(V, W);
  if (tid < D) {
    const int j = tid;
    const float lj = lam[j];
    int rk = 0;
    for (int i = 0; i < D; ++i) rk += (lam[i] > lj) || (lam[i] == lj && i < j);
    rank[j] = rk;
    int best = 0;
    float bv = fabsf(V[j]);
    for (int r = 1; r < D; ++r) {
      const float a = fabsf(V[r * LDA + j]);
      if (a > bv) {
        bv = a;
        best = r;
      }
    }
    sgn[j] = V[best * LDA + j] < 0.f ? -1.f : 1.f;
  }
  __syncthreads();
  float* R = p.R + (size_t)sx * D * D;
  for (int e = tid; e < D * D; e += EIG_THREADS) {
    const int r = e >> 7, j = e & 127;
    R[r * D + rank[j]] = sgn[j] * V[r * LDA + j];
  }
  if (tid < D) p.lam[(size_t)sx * D + rank[tid]] = lam[tid];
}

// ---------------------------------------------------------------------------
// Warp-level top-c of 128 non-negative keys (lane holds channels lane + 32m),
// ties to the lower channel.  Binary search on the key bits for the c-th
// largest key; stops early once exactly c keys are >= the candidate.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void warp_topc(const uint32_t key[4], int c, bool sel[4]) {
  const int lane = threadIdx.x & 31;
  if (c >= D) {
#pragma unroll
    for (int m = 0; m < 4; ++m) sel[m] = true;
    return;
  }
  uint32_t thr = 0;
  int cnt_ge = D;
  for (int bit = 30; bit >= 0; --bit) {
    const uint32_t cand = thr | (1u << bit);
    const int local = (key[0] >= cand) + (key[1] >= cand) + (key[2] >= cand) + (key[3] >= cand);
    const int cnt = __reduce_add_sync(0xffffffffu, local);
    if (cnt >= c) {
      thr = cand;
      cnt_ge = cnt;
      if (cnt == c) break;
    }
  }
  if (cnt_ge == c) {
#pragma unroll
    for (int m = 0; m < 4; ++m) sel[m] = key[m] >= thr;
    return;
  }
  const int gt = __reduce_add_sync(0xffffffffu, (key[0] > thr) + (key[1] > thr) + (key[2] > thr) +
                                                     (key[3] > thr));
  const int need = c - gt;
  int before = 0;
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t eqb = __ballot_sync(0xffffffffu, key[m] == thr);
    const int rk = before + __popc(eqb & lt);
    sel[m] = key[m] > thr || (key[m] == thr && rk < need);
    before += __popc(eqb);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// ---------------------------------------------------------------------------
// analyze (PACK = false) / pack (PACK = true).
// One CTA covers whole segments [sg0, sg1) of one stream, in 64-token tiles.
// Warp w computes rows 16*(w&3).. and columns 64*(w>>2).. of x~ = x R_hi + x R_lo.
// grid: (ctas_per_stream, BH, 2), block 256, dynamic smem ~131 KB
// ---------------------------------------------------------------------------
constexpr int XT_LD = D + 4;
constexpr size_t AN_SMEM = 2 * 32768 + 2 * 16384 + (size_t)TILE_T * XT_LD * 4 + TILE_T * 16 +
                           TILE_T * 4 + D * 4 + 64;

template <bool PACK>
__global__ void __launch_bounds__(256, 1) analyze_kernel(CompressParams p) {
  extern __shared__ __align__(128) uint8_t asmem[];
  uint8_t* Rhi = asmem;
  uint8_t* Rlo = asmem + 32768;
  uint8_t* Xs = asmem + 65536;                                  // 2 x 16 KB
  float* Xt = reinterpret_cast<float*>(asmem + 65536 + 32768);  // [64][XT_LD]
  uint32_t* tokmask = reinterpret_cast<uint32_t*>(Xt + TILE_T * XT_LD);  // [64][4]
  float* tokkept = reinterpret_cast<float*>(tokmask + TILE_T * 4);       // [64]
  float* colacc = tokkept + TILE_T;                                      // [128]
  float* segkept = colacc + D;                                           // [1]

  const int x = blockIdx.z, s = blockIdx.y;
  const int sx = x * p.BH + s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int sg0 = blockIdx.x * p.segs_per_cta;
  const int sg1 = min(p.n_seg, sg0 + p.segs_per_cta);
  if (sg0 >= sg1) return;
  const int64_t tb = (int64_t)sg0 * p.S;
  const int64_t te = imin64(p.T, (int64_t)sg1 * p.S);
  const __half* X = p.X[x] + (size_t)s * p.T * D;
  const uint32_t xs_base = smem_u32(Xs);

  // first tile in flight while R is split and transposed
  load_tile(xs_base, X, tb, p.T);
  cp_async_commit();
  {
    const float* R = p.R + (size_t)sx * D * D;
    for (int e = tid; e < D * D; e += blockDim.x) {
      const int i = e >> 7, j = e & 127;      // R[i][j]: input channel i, basis vector j
      const float r = R[e];
      const __half hi = __float2half_rn(r);
      const __half lo = __float2half_rn((r - __half2float(hi)) * 2048.f);   // kept normal
      const uint32_t off = swz(j, i >> 3) + (i & 7) * 2;
      *reinterpret_cast<__half*>(Rhi + off) = hi;
      *reinterpret_cast<__half*>(Rlo + off) = lo;
    }
  }
  if (!PACK) {
    for (int j = tid; j < D; j += blockDim.x) colacc[j] = 0.f;
    if (tid == 0) segkept[0] = 0.f;
  }
  const uint32_t rhi = smem_u32(Rhi), rlo = smem_u32(Rlo);
  const SegInfo* seginfo = p.seg + (size_t)sx * p.n_seg;
  const mkv_segment_header* hdr = p.hdr + (size_t)sx * p.n_seg;
  const int m0 = (warp & 3) * 16, n0 = (warp >> 2) * 64;
  const int mm = lane >> 3, r8 = lane & 7;
  const int n_tiles = (int)((te - tb + TILE_T - 1) / TILE_T);

  for (int it = 0; it < n_tiles; ++it) {
    const int64_t t0 = tb + (int64_t)it * TILE_T;
    const int rows = (int)imin64(TILE_T, te - t0);
    if (it + 1 < n_tiles) load_tile(xs_base + ((it + 1) & 1) * 16384u, X, t0 + TILE_T, p.T);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t tile = xs_base + (it & 1) * 16384u;
    // ---- x~ tile on tensor cores -------------------------------------------
    float acc[8][4], accl[8][4];
#pragma unroll
    for (int ni = 0; ni < 8; ++ni)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[ni][e] = accl[ni][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      ldsm_x4(tile + swz(m0 + (mm & 1) * 8 + r8, 2 * ks + (mm >> 1)), a);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int jr = n0 + np * 16 + (mm >> 1) * 8 + r8;
        const uint32_t off = swz(jr, 2 * ks + (mm & 1));
        uint32_t bh[4], bl[4];
        ldsm_x4(rhi + off, bh);
        ldsm_x4(rlo + off, bl);
        mma16816(acc[2 * np], a, bh[0], bh[1]);
        mma16816(acc[2 * np + 1], a, bh[2], bh[3]);
        mma16816(accl[2 * np], a, bl[0], bl[1]);
        mma16816(accl[2 * np + 1], a, bl[2], bl[3]);
      }
    }
    {
      const int g = lane >> 2, q = lane & 3;
      constexpr float kLo = 1.f / 2048.f;
#pragma unroll
      for (int ni = 0; ni < 8; ++ni) {
        const int col = n0 + ni * 8 + 2 * q;
        *reinterpret_cast<float2*>(Xt + (m0 + g) * XT_LD + col) =
            make_float2(fmaf(accl[ni][0], kLo, acc[ni][0]), fmaf(accl[ni][1], kLo, acc[ni][1]));
        *reinterpret_cast<float2*>(Xt + (m0 + g + 8) * XT_LD + col) =
            make_float2(fmaf(accl[ni][2], kLo, acc[ni][2]), fmaf(accl[ni][3], kLo, acc[ni][3]));
      }
    }
    __syncthreads();
    // ---- per-token selection (and packing) ---------------------------------
    for (int r = warp; r < rows; r += 8) {
      const int64_t t = t0 + r;
      float v[4];
      uint32_t key[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[m] = Xt[r * XT_LD + lane + 32 * m];
        key[m] = __float_as_uint(v[m]) & 0x7fffffffu;
      }
      if (!PACK) {
        bool sel[4];
        warp_topc(key, p.c, sel);
        float kept = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) kept += sel[m] ? v[m] * v[m] : 0.f;
        kept = warp_sum(kept);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t w = __ballot_sync(0xffffffffu, sel[m]);
          if (lane == 0) tokmask[r * 4 + m] = w;
        }
        if (lane == 0) tokkept[r] = kept;
      } else {
        const int sg = (int)(t / p.S);
        const int rl = (int)(t - (int64_t)sg * p.S);
        const SegInfo si = seginfo[sg];
        if ((uint64_t)hdr[sg].off16 * 16u + si.size > p.pool_check) {
          // the segment would end past the checked pool extent: report, skip
          if (lane == 0) atomicOr(p.err, DEV_ERR_CHECK);
          continue;
        }
        uint8_t* seg = p.pool + (size_t)hdr[sg].off16 * 16u;
        const uint32_t c = (uint32_t)p.c;
        if (si.strategy == MKV_STRATEGY_DENSE) {
          __half* row = reinterpret_cast<__half*>(seg + 256u * rl);
#pragma unroll
          for (int m = 0; m < 4; ++m) row[lane + 32 * m] = __float2half_rn(v[m]);
        } else {
          uint32_t w[4];
          if (si.strategy == MKV_STRATEGY_SM) {
#pragma unroll
            for (int m = 0; m < 4; ++m) w[m] = si.mask[m];
          } else {
            bool sel[4];
            warp_topc(key, p.c, sel);
#pragma unroll
            for (int m = 0; m < 4; ++m) w[m] = __ballot_sync(0xffffffffu, sel[m]);
          }
          __half* vrow;
          uint8_t* irow;
          if (si.strategy == MKV_STRATEGY_SM) {
            vrow = reinterpret_cast<__half*>(seg + pad16(c) + 2u * c * rl);
            irow = (rl == 0) ? seg : nullptr;
          } else {
            vrow = reinterpret_cast<__half*>(seg + 2u * c * rl);
            irow = seg + 2u * c * si.rows + c * rl;
          }
          const uint32_t lt = (1u << lane) - 1u;
          int before = 0;
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if ((w[m] >> lane) & 1u) {
              const int pos = before + __popc(w[m] & lt);
              vrow[pos] = __float2half_rn(v[m]);
              if (irow) irow[pos] = (uint8_t)(lane + 32 * m);
            }
            before += __popc(w[m]);
          }
          // zero the padding after the index bytes
          if (si.strategy == MKV_STRATEGY_SM && rl == 0) {
            for (uint32_t z = c + lane; z < pad16(c); z += 32) seg[z] = 0;
          }
          if (si.strategy == MKV_STRATEGY_PV && rl == si.rows - 1) {
            uint8_t* ib = seg + 2u * c * si.rows;
            for (uint32_t z = c * si.rows + lane; z < pad16(c * si.rows); z += 32) ib[z] = 0;
          }
        }
      }
    }
    __syncthreads();
    if (!PACK) {
      // ---- segment statistics: walk the segments that intersect this tile ----
      int64_t a = t0;
      const int64_t tend = t0 + rows;
      while (a < tend) {
        const int sg = (int)(a / p.S);
        const int64_t segend = imin64(p.T, (int64_t)(sg + 1) * p.S);
        const int64_t b = imin64(tend, segend);
        if (tid < D) {
          float cacc = colacc[tid];
          for (int64_t t = a; t < b; ++t) {
            const float val = Xt[(int)(t - t0) * XT_LD + tid];
            cacc = fmaf(val, val, cacc);
          }
          colacc[tid] = cacc;
        } else if (tid == D) {
          float k = segkept[0];
          for (int64_t t = a; t < b; ++t) k += tokkept[(int)(t - t0)];
          segkept[0] = k;
        }
        __syncthreads();
        if (b == segend) {
          if (warp == 0) {
            float cv[4];
            uint32_t key[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              cv[m] = colacc[lane + 32 * m];
              key[m] = __float_as_uint(cv[m]) & 0x7fffffffu;
            }
            const float etot = warp_sum(cv[0] + cv[1] + cv[2] + cv[3]);
            bool sel[4];
            warp_topc(key, p.c, sel);
            float smk = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) smk += sel[m] ? cv[m] : 0.f;
            smk = warp_sum(smk);
            uint32_t w[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) w[m] = __ballot_sync(0xffffffffu, sel[m]);
            if (lane == 0) {
              const int rws = (int)(segend - (int64_t)sg * p.S);
              const float fsm = etot > 0.f ? smk / etot : 1.f;
              const float fpv = etot > 0.f ? segkept[0] / etot : 1.f;
              uint32_t best = segment_bytes(MKV_STRATEGY_DENSE, rws, p.c);
              int strat = MKV_STRATEGY_DENSE;
              const uint32_t cpv = segment_bytes(MKV_STRATEGY_PV, rws, p.c);
              const uint32_t csm = segment_bytes(MKV_STRATEGY_SM, rws, p.c);
              if (fpv >= p.tau && cpv <= best) {
                best = cpv;
                strat = MKV_STRATEGY_PV;
              }
              if (fsm >= p.tau && csm <= best) {
                best = csm;
                strat = MKV_STRATEGY_SM;
              }
              SegInfo si;
              si.size = best;
              si.strategy = (uint8_t)strat;
              si.pad = 0;
              si.rows = (uint16_t)rws;
#pragma unroll
              for (int m = 0; m < 4; ++m) si.mask[m] = w[m];
              si.f_sm = fsm;
              si.f_pv = fpv;
              p.seg[(size_t)sx * p.n_seg + sg] = si;
            }
          }
          __syncthreads();
          if (tid < D) colacc[tid] = 0.f;
          if (tid == D) segkept[0] = 0.f;
          __syncthreads();
        }
        a = b;
      }
    }
  }
  cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// scan: offsets of every segment of every stream (K streams first, then V),
// segment headers and the total packed size.  One CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) scan_kernel(CompressParams p) {
  const int64_t n = (int64_t)2 * p.BH * p.n_seg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (n + 1023) / 1024;
  const int64_t lo = imin64(n, tid * per), hi = imin64(n, lo + per);
  unsigned long long mine = 0;
  for (int64_t e = lo; e < hi; ++e) mine += p.seg[e].size;
  unsigned long long inc = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  __shared__ unsigned long long ws[32];
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  unsigned long long wb = 0;
  for (int w = 0; w < warp; ++w) wb += ws[w];
  unsigned long long off = wb + inc - mine;
  __shared__ unsigned int n_dense[2];
  if (tid < 2) n_dense[tid] = 0u;
  __syncthreads();
  const int64_t per_x = (int64_t)p.BH * p.n_seg;
  for (int64_t e = lo; e < hi; ++e) {
    const SegInfo si = p.seg[e];
    if (si.strategy == MKV_STRATEGY_DENSE) atomicAdd(&n_dense[e >= per_x ? 1 : 0], 1u);
    mkv_segment_header h;
    h.off16 = (uint32_t)(off >> 4);
    h.strategy = si.strategy;
    h.reserved = 0;
    h.rows = si.rows;
    p.hdr[e] = h;
    off += si.size;
  }
  __syncthreads();
  if (tid == 1023) p.total[0] = wb + inc;
  if (tid < 2) p.total[1 + tid] = n_dense[tid];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_gram(const CompressParams& p, cudaStream_t st) {
  const int smem = GR_STAGES * 16384;
  dim3 grid(p.gram_chunks, p.BH, 2);
  gram_kernel<<<grid, 256, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_eig(const CompressParams& p, cudaStream_t st) {
  const int smem = 3 * D * LDA * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  eig_kernel<<<2 * p.BH, EIG_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

template <bool PACK>
static cudaError_t launch_an(const CompressParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(analyze_kernel<PACK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)AN_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.ctas_per_stream, p.BH, 2);
  analyze_kernel<PACK><<<grid, 256, AN_SMEM, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_analyze(const CompressParams& p, cudaStream_t st) { return launch_an<false>(p, st); }
cudaError_t launch_pack(const CompressParams& p, cudaStream_t st) { return launch_an<true>(p, st); }

cudaError_t launch_scan(const CompressParams& p, cudaStream_t st) {
  scan_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mkv
