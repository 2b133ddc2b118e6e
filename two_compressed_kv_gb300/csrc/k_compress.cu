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
#include "block_scan.cuh"
#include "tc05.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// cp.async with a source size: bytes past src_bytes are filled with zeros
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(dst), "l"(src));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// ---------------------------------------------------------------------------
// X tiles for the fifth-generation tensor cores: 128 tokens x 128 channels of
// fp16 in the 128-byte swizzled layout, as two 16 KB atoms columns (channels
// 0-63, 64-127); in each, token r is the 128-byte row r and its 16-byte chunk
// c sits at chunk c ^ (r mod 8).  The same tile is a K-major operand with
// tokens as M (the rotation X R) and an MN-major operand with channels as M
// or N and tokens as K (the Gram X^T X).
// ---------------------------------------------------------------------------
constexpr int TC_T = GRAM_TILE;              // tokens per tile
constexpr uint32_t TC_TILE = 32768;          // bytes per tile
constexpr uint32_t TC_ATOMS = 16384;         // bytes per 64-channel half

// Loads tokens [t0, t0 + 128) of a stream (rows at or past t_end read as
// zeros); 128 threads, 16 copies each.
__device__ __forceinline__ void tc_load_tile(uint32_t tile, const __half* X, int64_t t0,
                                             int64_t t_end) {
#pragma unroll 4
  for (int q = threadIdx.x; q < TC_T * 16; q += 128) {
    const int row = q >> 4, c16 = q & 15;
    const int64_t t = t0 + row;
    const bool ok = t < t_end;
    const __half* src = X + (ok ? t : 0) * D + c16 * 8;
    const uint32_t dst = tile + (uint32_t)(c16 >> 3) * TC_ATOMS + (uint32_t)row * 128u +
                         ((uint32_t)((c16 & 7) ^ (row & 7)) << 4);
    cp_async16(dst, src, ok ? 16u : 0u);
  }
}

// MN-major descriptor of a tile used with channels as M (or N): 64-channel
// atoms 16 KB apart (leading byte offset), groups of 8 tokens 1024 B apart
// (stride byte offset), 128-byte swizzle.  K (tokens) advances by 16 tokens
// = 2048 B per MMA.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(TC_ATOMS >> 4) << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// kind::f16 instruction descriptor with both operands MN-major (bits 15, 16)
__host__ __device__ constexpr uint32_t idesc_f16_f32_mn(int M, int N) {
  return idesc_f16_f32(M, N) | (1u << 15) | (1u << 16);
}

// Waits on an mbarrier phase with the library's bounded wait; records a
// timeout in the status word and returns false if it gives up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_wait(bar, parity)) return true;
  atomicOr(err, DEV_ERR_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// gram: partial G = X^T X over one chunk of tokens on the tensor cores
// (tcgen05, fp16 operands, fp32 accumulators in tensor memory).  Tiles of 128
// tokens are double-buffered (cp.async); thread 0 issues the 8 MMAs of a tile
// (M = N = 128 channels, K = 16 tokens each) into one of two TMEM
// accumulators and commits them to that accumulator's mbarrier; meanwhile
// the 128 threads add the other accumulator into fp32 registers (thread i
// holds row i of G).  Flushing after every tile keeps the tensor-core
// accumulation to 128 products, so G is good to a few 1e-6 relative at any
// context length.
// grid: (gram_chunks, BH, 2), block 128, dynamic smem 2 tiles + alignment
// ---------------------------------------------------------------------------
constexpr int GT_THREADS = 128;
constexpr size_t GT_SMEM = 2 * TC_TILE + 1024 + 16384;   // +16 KB: at most two CTAs per SM

__global__ void __launch_bounds__(GT_THREADS, 1) gram_kernel(CompressParams p) {
  extern __shared__ uint8_t gsm_raw[];
  __shared__ uint64_t mma_done[2];
  __shared__ uint32_t tbase_sh;
  const int chunk = blockIdx.x, s = blockIdx.y, x = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const __half* X = p.X[x] + (size_t)s * p.T * D;
  const int64_t tb = (int64_t)chunk * p.gram_chunk_tokens;
  const int64_t te = imin64(p.T, tb + p.gram_chunk_tokens);
  const int n_tiles = te > tb ? (int)((te - tb + TC_T - 1) / TC_T) : 0;
  const uint32_t base = (smem_u32(gsm_raw) + 1023u) & ~1023u;     // 1024-byte aligned tiles

  if (warp == 0) {
    tmem_alloc(&tbase_sh, 256);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    mbar_init_fence();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tbase_sh;
  const uint32_t idesc = idesc_f16_f32_mn(128, 128);
  float tot[D];
#pragma unroll
  for (int j = 0; j < D; ++j) tot[j] = 0.f;
  bool ok = true;

  // adds accumulator b (its use-th completion) into tot
  auto flush = [&](int b, int use) {
    if (!tc_wait(&mma_done[b], (uint32_t)(use & 1), p.err)) {
      ok = false;
      return;
    }
    tc_fence_after();
    const uint32_t ta = tbase + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * 128);
#pragma unroll
    for (int q = 0; q < D / 16; ++q) {
      uint32_t r[16];
      tmem_ld16(ta + 16 * q, r);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 16; ++j) tot[16 * q + j] += __uint_as_float(r[j]);
    }
  };

  if (n_tiles > 0) tc_load_tile(base, X, tb, te);
  cp_async_commit();
  for (int it = 0; it < n_tiles && ok; ++it) {
    const int b = it & 1;
    // the other buffer's MMAs (tile it - 1) must be done before its smem is
    // refilled and its accumulator read
    if (it >= 1) flush(b ^ 1, (it - 1) >> 1);
    tc_fence_before();
    __syncthreads();
    if (it + 1 < n_tiles) tc_load_tile(base + (b ^ 1) * TC_TILE, X, tb + (int64_t)(it + 1) * TC_T, te);
    cp_async_commit();
    cp_async_wait<1>();
    fence_proxy_async();          // the tile's generic-proxy writes, before the MMAs read it
    __syncthreads();
    if (tid == 0) {
      tc_fence_after();
      const uint32_t tile = base + b * TC_TILE;
#pragma unroll
      for (int k = 0; k < TC_T / 16; ++k) {
        const uint64_t dsc = sdesc_mn_sw128(tile + (uint32_t)k * 2048u);
        tc_mma_f16(tbase + (uint32_t)(b * 128), dsc, dsc, idesc, k > 0 ? 1u : 0u);
      }
      tc_commit(&mma_done[b]);
    }
  }
  if (ok && n_tiles > 0) flush((n_tiles - 1) & 1, (n_tiles - 1) >> 1);
  cp_async_wait<0>();
  float* out = p.gram_part + (((size_t)x * p.BH + s) * p.gram_chunks + chunk) * (D * D) +
               (size_t)tid * D;
#pragma unroll
  for (int j = 0; j < D; j += 4) *reinterpret_cast<float4*>(out + j) = make_float4(tot[j], tot[j + 1], tot[j + 2], tot[j + 3]);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 256);
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
// During the sweeps A keeps only its upper triangle (entry (i, j) at
// (min, max)) and V is held column-major, so that a rotation of two columns
// of V moves whole rows of 16-byte vectors.
// grid: 2 * BH, block 1024, dynamic smem 2 x 128 x 129 + 128 x 132 floats
// ---------------------------------------------------------------------------
constexpr int EIG_THREADS = 1024;
constexpr int LDA = D + 1;
constexpr int LDV = D + 4;            // column-major V: 16-byte aligned columns
constexpr int EIG_MAX_SWEEPS = 16;
constexpr int EIG_REFINE_SWEEPS = 6;

__device__ __forceinline__ int rr_player(int pos, int round) {
  return pos == 0 ? 0 : 1 + (pos - 1 + round) % (D - 1);
}

struct EigShared {
  float cs[64], sn[64];
  int top[64], bot[64];
  int rotated;
  float floor;
};

__device__ __forceinline__ int upper(int i, int j) { return i < j ? i * LDA + j : j * LDA + i; }

// Jacobi sweeps on the upper triangle of A (in place), accumulating the
// rotations into the column-major Vt (column k of V at Vt + k LDV), until a
// sweep rotates nothing or max_sweeps have run.  A pair (p, q) is rotated
// when |a_pq| > tol sqrt(|a_pp a_qq|) and |a_pq| > floor_rel max_i |a_ii|
// (floor_rel = 0: no floor); blocks and columns whose rotations are all
// identities are left untouched.  Block-wide.
//
// A round's 64 rotations split A into 64 x 64 blocks of 2 x 2.  The thread
// that computes rotation P also updates the diagonal block (P, P); by
// symmetry only the 2016 off-diagonal blocks (P, Q), Q = P + d (mod 64),
// d = 1 .. 31, and d = 32 for P < 32, are formed: warp w takes P = w and
// P = w + 32, lane l the offset d = l (lane 0: d = 32 for P = w only), so
// that a warp's accesses share their row and spread over the banks.  Thread
// t updates rows 4 (t / 64) .. +3 and 4 (t / 64 + 16) .. +3 of the two
// columns of V that rotation t mod 64 mixes.
__device__ void jacobi_sweeps(float* A, float* Vt, int max_sweeps, float tol, float floor_rel,
                              EigShared& sh) {
  static_assert(EIG_THREADS == 1024, "two blocks and two row groups of V per thread");
  const int tid = threadIdx.x;
  float floor_abs = 0.f;
  if (floor_rel > 0.f) {
    // the largest diagonal entry (warp 0), read by every thread
    if (tid < 32) {
      float mx = 0.f;
      for (int i = tid; i < D; i += 32) mx = fmaxf(mx, fabsf(A[i * LDA + i]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (tid == 0) sh.floor = floor_rel * mx;
    }
    __syncthreads();
    floor_abs = sh.floor;
  }
  const int w = tid >> 5, l = tid & 31;
  const int R = tid & 63, g = tid >> 6;
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    if (tid == 0) sh.rotated = 0;
    __syncthreads();
    for (int round = 0; round < D - 1; ++round) {
      if (tid < 64) {
        int a = rr_player(tid, round), b = rr_player(D - 1 - tid, round);
        const int pp = min(a, b), qq = max(a, b);
        const float app = A[pp * LDA + pp], aqq = A[qq * LDA + qq], apq = A[pp * LDA + qq];
        float c = 1.f, s = 0.f;
        if (apq != 0.f && fabsf(apq) > tol * sqrtf(fabsf(app * aqq)) && fabsf(apq) > floor_abs) {
          const float th = (aqq - app) / (2.f * apq);
          const float t = (th >= 0.f ? 1.f : -1.f) / (fabsf(th) + sqrtf(1.f + th * th));
          c = 1.f / sqrtf(1.f + t * t);
          s = t * c;
          sh.rotated = 1;
          // the diagonal block: no other update of this round touches it
          A[pp * LDA + pp] = app - t * apq;
          A[qq * LDA + qq] = aqq + t * apq;
          A[pp * LDA + qq] = 0.f;
        }
        sh.cs[tid] = c;
        sh.sn[tid] = s;
        sh.top[tid] = pp;
        sh.bot[tid] = qq;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int P = w + 32 * k;
        if (k == 1 && l == 0) break;   // (w + 32, w) is lane 0's block (w, w + 32)
        const int Q = (P + (l == 0 ? 32 : l)) & 63;
        const float sP = sh.sn[P], sQ = sh.sn[Q];
        if (sP == 0.f && sQ == 0.f) continue;   // both rotations are identities
        const float cP = sh.cs[P], cQ = sh.cs[Q];
        const int p1 = sh.top[P], p2 = sh.bot[P], q1 = sh.top[Q], q2 = sh.bot[Q];
        const int i11 = upper(p1, q1), i12 = upper(p1, q2), i21 = upper(p2, q1), i22 = upper(p2, q2);
        const float b11 = A[i11], b12 = A[i12], b21 = A[i21], b22 = A[i22];
        const float u11 = cP * b11 - sP * b21, u12 = cP * b12 - sP * b22;
        const float u21 = sP * b11 + cP * b21, u22 = sP * b12 + cP * b22;
        A[i11] = cQ * u11 - sQ * u12;
        A[i12] = sQ * u11 + cQ * u12;
        A[i21] = cQ * u21 - sQ * u22;
        A[i22] = sQ * u21 + cQ * u22;
      }
      {
        const float sR = sh.sn[R];
        if (sR != 0.f) {
          const float cR = sh.cs[R];
          float4* vp = reinterpret_cast<float4*>(Vt + sh.top[R] * LDV);
          float4* vq = reinterpret_cast<float4*>(Vt + sh.bot[R] * LDV);
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int r4 = g + 16 * k;
            const float4 x = vp[r4], y = vq[r4];
            vp[r4] = make_float4(cR * x.x - sR * y.x, cR * x.y - sR * y.y, cR * x.z - sR * y.z,
                                 cR * x.w - sR * y.w);
            vq[r4] = make_float4(sR * x.x + cR * y.x, sR * x.y + cR * y.y, sR * x.z + cR * y.z,
                                 sR * x.w + cR * y.w);
          }
        }
      }
      __syncthreads();
    }
    const int any = sh.rotated;
    __syncthreads();
    if (!any) break;
  }
}

// V between its row-major (row stride LDA) and column-major (column stride
// LDV) forms, in place through registers.  Block-wide.
template <bool TO_COLUMNS>
__device__ void v_relayout(float* V) {
  const int tid = threadIdx.x;
  float v[D * D / EIG_THREADS];
#pragma unroll
  for (int k = 0; k < D * D / EIG_THREADS; ++k) {
    const int e = tid + k * EIG_THREADS, r = e >> 7, c = e & 127;
    v[k] = TO_COLUMNS ? V[r * LDA + c] : V[c * LDV + r];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < D * D / EIG_THREADS; ++k) {
    const int e = tid + k * EIG_THREADS, r = e >> 7, c = e & 127;
    if (TO_COLUMNS) V[c * LDV + r] = v[k];
    else V[r * LDA + c] = v[k];
  }
  __syncthreads();
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
  float* V = esm + D * LDA;          // row-major (LDA) or, during the sweeps, column-major (LDV)
  float* Gs = V + D * LDV;
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
    V[i * LDV + j] = (i == j) ? 1.f : 0.f;   // column-major for the sweeps
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

  // the first solve only has to bring A close to diagonal (pairs at or
  // below 1e-6 of the largest diagonal entry are left): the refinement below
  // re-forms V^T G V and finishes the convergence
  jacobi_sweeps(A, V, EIG_MAX_SWEEPS, 1e-5f, 1e-6f, sh);
  v_relayout<false>(V);
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
  v_relayout<true>(V);
  jacobi_sweeps(Ar, V, EIG_REFINE_SWEEPS, 1e-7f, 0.f, sh);
  v_relayout<false>(V);
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
// 32 x 32 bit-matrix transpose in registers: on entry w[r] bit c is entry
// (r, c), on exit w[c] bit r.  Block swaps of 16 and 8 (one byte transpose
// by byte permutes), then of 4, 2 and 1.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void transpose32(uint32_t w[32]) {
  // the 16- and 8-bit levels together: in each group w[r], w[r + 8],
  // w[r + 16], w[r + 24] byte j of word i trades places with byte i of word j
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const uint32_t lo01 = __byte_perm(w[r], w[r + 8], 0x5140), hi01 = __byte_perm(w[r], w[r + 8], 0x7362);
    const uint32_t lo23 = __byte_perm(w[r + 16], w[r + 24], 0x5140);
    const uint32_t hi23 = __byte_perm(w[r + 16], w[r + 24], 0x7362);
    w[r] = __byte_perm(lo01, lo23, 0x5410);
    w[r + 8] = __byte_perm(lo01, lo23, 0x7632);
    w[r + 16] = __byte_perm(hi01, hi23, 0x5410);
    w[r + 24] = __byte_perm(hi01, hi23, 0x7632);
  }
#pragma unroll
  for (int sft = 4, lvl = 0; sft >= 1; sft >>= 1, ++lvl) {
    const uint32_t m = lvl == 0 ? 0x0f0f0f0fu : lvl == 1 ? 0x33333333u : 0x55555555u;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      if (r & sft) continue;
      const uint32_t t = ((w[r] >> sft) ^ w[r + sft]) & m;
      w[r + sft] ^= t;
      w[r] ^= t << sft;
    }
  }
}

// ---------------------------------------------------------------------------
// Per-token top-c of 128 magnitudes held by a group of four lanes (32 each:
// lane 4k + i has channels 32 i .. 32 i + 31), ties to the lower channel.
// The magnitudes' bit patterns (non-negative floats order like their bits)
// are transposed into bit planes; a radix select from the top bit, two bits
// a step, keeps, per lane, the set A of keys that match the threshold's bits
// so far and the set G of keys already above it, with group counts
// (shuffles whose mask is the group alone: groups leave the loop at
// different steps).  It stops once G and A hold exactly c keys; otherwise A
// ends as the keys equal to the threshold, of which the lowest channels are
// taken, lower lanes' first.
// Returns this lane's 32 mask bits; the kept energy is summed by the caller.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quad_topc(uint32_t w[32], int c) {
  const int lane = threadIdx.x & 31;
  const unsigned gm = 15u << (lane & ~3);       // the four lanes of this token
  const int sub = lane & 3;
  if (c >= D) return 0xffffffffu;
  transpose32(w);                               // w[b] bit j: bit b of key j
  uint32_t A = 0xffffffffu, G = 0u;
  int nG = 0, nA = D;                           // group counts of G and A
  // two bit planes per step (plane 31 is zero): the group counts of the keys
  // of A whose two bits are 11, 10 and 01, packed 8 bits apart, in one sum
#pragma unroll
  for (int b = 31; b >= 1; b -= 2) {
    const uint32_t hi = w[b], lo = w[b - 1];
    const uint32_t a1 = A & hi, x11 = a1 & lo, x10 = a1 & ~lo, x01 = A & ~hi & lo;
    uint32_t pk = (uint32_t)__popc(x11) | ((uint32_t)__popc(x10) << 8) | ((uint32_t)__popc(x01) << 16);
    pk += __shfl_xor_sync(gm, pk, 1);
    pk += __shfl_xor_sync(gm, pk, 2);
    const int n11 = (int)(pk & 255u), n10 = (int)((pk >> 8) & 255u), n01 = (int)(pk >> 16);
    if (nG + n11 >= c) {
      A = x11;
      nA = n11;
    } else if (nG + n11 + n10 >= c) {
      G |= x11;
      nG += n11;
      A = x10;
      nA = n10;
    } else if (nG + n11 + n10 + n01 >= c) {
      G |= a1;
      nG += n11 + n10;
      A = x01;
      nA = n01;
    } else {
      G |= A & (hi | lo);
      nG += n11 + n10 + n01;
      A &= ~(hi | lo);
      nA -= n11 + n10 + n01;
    }
    if (nG + nA == c) break;
  }
  // take all of G and the lowest (c - nG) keys of A, lower lanes first
  const int na = __popc(A);
  int incl = na;
  int o = __shfl_up_sync(gm, incl, 1, 4);
  if (sub >= 1) incl += o;
  o = __shfl_up_sync(gm, incl, 2, 4);
  if (sub >= 2) incl += o;
  const int take = min(na, max(0, (c - nG) - (incl - na)));
  uint32_t t = 0u, a = A;
  for (int q = 0; q < take; ++q) {
    t |= a & (0u - a);
    a &= a - 1u;
  }
  return G | t;
}

// ---------------------------------------------------------------------------
// rotate: the statistics pass (PACK = false) and the packing pass (PACK =
// true).  One CTA (16 warps) covers whole segments [sg0, sg1) of one stream in
// tiles of 128 tokens.  x~ = x R_hi + 2^-11 (x R_lo) on the tensor cores
// (tcgen05, M = 128 tokens, N = 128 basis vectors, K = 128 channels; R split
// into an fp16 part and a remainder scaled by 2^11 so that it stays a normal
// fp16, one TMEM accumulator each).  Warp w reads TMEM lanes 32 (w mod 4)
// .. +31 (one token each), channels 32 (w / 4) .. +31.
//   statistics: the readback goes to an fp32 tile in shared memory; per token
//     the c channels of largest |x~| (quad_topc: four lanes per token), its
//     kept energy and channel mask (the mask also goes to global scratch for
//     the packing pass); per segment the column energies and the kept energy,
//     stored for the strategy kernel.
//   packing: with the segment data and the tokens' stored masks staged in
//     shared memory, each thread compacts its 32 channels of one token from
//     the readback registers into a shared-memory image of the packed row
//     (values, and index bytes for PV): the segment mask for SM, the token's
//     mask for PV, every channel for dense segments.  The images are then
//     written out in aligned 16- and 8-byte pieces (c is a multiple of 8, so
//     every packed value row starts on 16 bytes and every index row on 8).
// grid: (ctas_per_stream, BH, 2), block 512, dynamic smem rt_smem(PACK)
// ---------------------------------------------------------------------------
constexpr int RT_THREADS = 512;
static_assert(RT_THREADS == 4 * D, "four lanes per token and four column partial sums");
// fp32 x~ rows: channel ch at column ch + 8 (ch / 32), row stride 161 (= 1 mod
// 32): conflict-free by column, by row, and for the four lanes of a token
// that read its four 32-channel quarters at once
constexpr int XT_LD = D + 3 * 8 + 9;
static_assert(XT_LD % 32 == 1, "row stride");
__device__ __forceinline__ int xt_col(int ch) { return ch + 8 * (ch >> 5); }
constexpr int RT_MAXSEG = TC_T / 16 + 1;   // segments a tile can touch (S >= 16)
constexpr int ST_V = 2 * D + 16;      // staged value row bytes (16-byte pieces, banks spread)
constexpr int ST_I = D + 8;           // staged index row bytes (8-byte pieces)
// statistics: the fp32 tile; packing: the staged value and index rows
constexpr size_t rt_smem(bool pack) {
  return 1024 + 4 * (size_t)TC_TILE +
         (pack ? (size_t)TC_T * (ST_V + ST_I) + 2 * TC_T * 16 : (size_t)TC_T * XT_LD * 4) +
         TC_T * 16 + TC_T * 4 + D * 4 + 64;
}
static_assert(rt_smem(false) <= 227 * 1024 && rt_smem(true) <= 227 * 1024, "shared memory");

// The 16 MMAs of one tile: x~ hi part into columns tacc .. +127, lo part
// into tacc + 128 .. +255; committed to bar.  One thread.
__device__ __forceinline__ void rt_issue_mma(uint32_t xt, uint32_t Bhi, uint32_t Blo, uint32_t tacc,
                                             uint64_t* bar) {
  const uint32_t idesc = idesc_f16_f32(128, 128);
  tc_fence_after();
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t ko = (uint32_t)(k >> 2) * TC_ATOMS + (uint32_t)(k & 3) * 32u;
    const uint64_t a = sdesc_k_sw128(xt + ko);
    tc_mma_f16(tacc, a, sdesc_k_sw128(Bhi + ko), idesc, k > 0 ? 1u : 0u);
    tc_mma_f16(tacc + 128, a, sdesc_k_sw128(Blo + ko), idesc, k > 0 ? 1u : 0u);
  }
  tc_commit(bar);
}

template <bool PACK>
__global__ void __launch_bounds__(RT_THREADS, 1) rotate_kernel(CompressParams p) {
  extern __shared__ uint8_t rt_raw[];
  __shared__ uint64_t mma_bar[2];
  __shared__ uint32_t tbase_sh;
  // packing: segment data of three tiles (the current one, the next, and the
  // one being loaded)
  __shared__ __align__(16) SegInfo seg3[3][RT_MAXSEG];
  __shared__ __align__(8) mkv_segment_header hdr3[3][RT_MAXSEG];
  __shared__ float colpart[RT_THREADS / D][D];   // column-energy partial sums
  __shared__ uint32_t rowinfo[TC_T];             // packing: segment slot << 16 | row in segment
  const uint32_t raw = smem_u32(rt_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;            // tiles on 1024-byte boundaries
  uint8_t* gbase = rt_raw + (base - raw);
  const uint32_t Bhi = base, Blo = base + TC_TILE, Xs = base + 2 * TC_TILE;
  float* Xt = reinterpret_cast<float*>(gbase + 4 * TC_TILE);             // [128][XT_LD]
  uint8_t* stv = gbase + 4 * TC_TILE;                                     // [128][ST_V]
  uint8_t* sti = stv + TC_T * ST_V;                                       // [128][ST_I]
  // statistics: [128][4]; packing: [3][128][4] (three tiles, like the segment data)
  uint32_t* tokmask = reinterpret_cast<uint32_t*>(
      PACK ? sti + TC_T * ST_I : reinterpret_cast<uint8_t*>(Xt + TC_T * XT_LD));
  float* tokkept = reinterpret_cast<float*>(tokmask + (PACK ? 3 : 1) * TC_T * 4);   // [128]
  float* colacc = tokkept + TC_T;                                        // [128]
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
  const int n_tiles = (int)((te - tb + TC_T - 1) / TC_T);

  uint32_t* gmask = p.tokmask + (size_t)sx * p.T * 4;
  // packing: tile j's token masks and segment data into buffer j mod 3, in
  // the same cp.async group as its X tile (threads 0..127)
  auto load_meta = [&](int j) {
    const int offj = j * TC_T;                      // past the CTA's first token (32-bit)
    const int64_t t0j = tb + offj;
    const int rowsj = (int)imin64(TC_T, te - t0j);
    const int sgfj = sg0 + offj / p.S;
    const int nsgj = sg0 + (offj + rowsj - 1) / p.S - sgfj + 1;
    const int mbj = j % 3;
    const bool live = tid < rowsj;
    cp_async16(smem_u32(tokmask + (mbj * TC_T + tid) * 4),
               gmask + (size_t)(live ? t0j + tid : t0j) * 4, live ? 16u : 0u);
    if (tid < nsgj) {
      const size_t e = (size_t)sx * p.n_seg + sgfj + tid;
      const uint8_t* src = reinterpret_cast<const uint8_t*>(p.seg + e);
      cp_async16(smem_u32(&seg3[mbj][tid]), src, 16u);
      cp_async16(smem_u32(&seg3[mbj][tid]) + 16u, src + 16, 16u);
      cp_async8(smem_u32(&hdr3[mbj][tid]), p.hdr + e);
    }
  };

  // two TMEM accumulator pairs: the MMAs of tile it + 1 run while tile it is
  // read back
  if (warp == 0) {
    tmem_alloc(&tbase_sh, 512);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&mma_bar[0], 1);
    mbar_init(&mma_bar[1], 1);
    mbar_init_fence();
  }
  // tiles 0 and 1 in flight while R is split into the two B operands
  if (tid < 128) {
    tc_load_tile(Xs, X, tb, te);
    if (PACK) load_meta(0);
  }
  cp_async_commit();
  if (n_tiles > 1 && tid < 128) {
    tc_load_tile(Xs + TC_TILE, X, tb + TC_T, te);
    if (PACK) load_meta(1);
  }
  cp_async_commit();
  {
    // B = R^T, K-major: row j (basis vector) holds R[0..127][j] along K
    const float* R = p.R + (size_t)sx * D * D;
    for (int e = tid; e < D * D; e += RT_THREADS) {
      const int i = e >> 7, j = e & 127;      // R[i][j]: input channel i, basis vector j
      const float r = R[e];
      const __half hi = __float2half_rn(r);
      const __half lo = __float2half_rn((r - __half2float(hi)) * 2048.f);   // kept normal
      const uint32_t off = (uint32_t)(i >> 6) * TC_ATOMS + (uint32_t)j * 128u +
                           ((uint32_t)(((i & 63) >> 3) ^ (j & 7)) << 4) + (uint32_t)(i & 7) * 2u;
      *reinterpret_cast<__half*>(gbase + off) = hi;
      *reinterpret_cast<__half*>(gbase + TC_TILE + off) = lo;
    }
  }
  if (!PACK) {
    if (tid < D) colacc[tid] = 0.f;
    if (tid == 0) segkept[0] = 0.f;
  }
  cp_async_wait<1>();             // tile 0
  fence_proxy_async();            // tile and B operands: generic-proxy writes before the MMAs
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tbase_sh;
  if (tid == 0) rt_issue_mma(Xs, Bhi, Blo, tbase, &mma_bar[0]);
  bool ok = true;

  for (int it = 0; it < n_tiles && ok; ++it) {
    const int64_t t0 = tb + (int64_t)it * TC_T;
    const int rows = (int)imin64(TC_T, te - t0);
    const int b = it & 1;
    const int mb = it % 3;
    const SegInfo* seg_sh = seg3[mb];
    const mkv_segment_header* hdr_sh = hdr3[mb];
    const uint32_t* tmask = tokmask + (PACK ? mb * TC_T * 4 : 0);
    if (it + 1 < n_tiles) {
      cp_async_wait<0>();         // this thread's part of tile it + 1 (and its segment data)
      fence_proxy_async();
    }
    // row r of the tile is row lr0 + r past the start of segment sgf (32-bit:
    // a CTA covers whole segments from sg0 on)
    const int sgf = sg0 + (it * TC_T) / p.S;
    const int lr0 = it * TC_T - (sgf - sg0) * p.S;
    // one decision for the whole block; past it tile it + 1 has landed and
    // the previous tile's shared-memory reads are done
    if (__syncthreads_or(!tc_wait(&mma_bar[b], (uint32_t)((it >> 1) & 1), p.err))) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (it + 1 < n_tiles && tid == 0)   // tile it + 1's MMAs into the other pair
      rt_issue_mma(Xs + (uint32_t)(b ^ 1) * TC_TILE, Bhi, Blo, tbase + (uint32_t)(b ^ 1) * 256u,
                   &mma_bar[b ^ 1]);
    // X buffer b is free: tile it + 2 in flight from here
    if (it + 2 < n_tiles && tid < 128) {
      tc_load_tile(Xs + (uint32_t)b * TC_TILE, X, t0 + 2 * TC_T, te);
      if (PACK) load_meta(it + 2);
    }
    cp_async_commit();
    if (PACK) {
      // ---- compaction: thread = (token, 32 channels) -----------------------------
      const int tok = 32 * (warp & 3) + lane, qt = warp >> 2, c0 = 32 * qt;
      const uint32_t ta = tbase + (uint32_t)b * 256u + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0;
      const bool live = tok < rows;
      int strat = MKV_STRATEGY_DENSE, pos = 0;
      uint32_t m = 0xffffffffu;
      uint8_t* sm_idx = nullptr;     // SM index bytes of a segment's first row go straight out
      if (live) {
        const int q = (lr0 + tok) / p.S;
        const int rl = lr0 + tok - q * p.S;
        const SegInfo& si = seg_sh[q];
        strat = si.strategy;
        if (strat != MKV_STRATEGY_DENSE) {
          const uint32_t* mw = strat == MKV_STRATEGY_SM ? si.mask : tmask + 4 * tok;
          m = mw[qt];
          for (int z = 0; z < qt; ++z) pos += __popc(mw[z]);
        }
        if (qt == 0) rowinfo[tok] = ((uint32_t)q << 16) | (uint32_t)rl;
        if (strat == MKV_STRATEGY_SM && rl == 0 &&
            (uint64_t)hdr_sh[q].off16 * 16u + si.size <= p.pool_check)
          sm_idx = p.pool + (size_t)hdr_sh[q].off16 * 16u;
      }
      __half* vrow = reinterpret_cast<__half*>(stv + tok * ST_V);
      uint8_t* irow = strat == MKV_STRATEGY_PV ? sti + tok * ST_I : nullptr;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[16], l[16];
        __syncwarp();
        tmem_ld16(ta + 16 * q, h);
        tmem_ld16(ta + 128 + 16 * q, l);
        tmem_ld_wait();
        __half2 hv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          hv[j] = __floats2half2_rn(fmaf(__uint_as_float(l[2 * j]), 1.f / 2048.f, __uint_as_float(h[2 * j])),
                                    fmaf(__uint_as_float(l[2 * j + 1]), 1.f / 2048.f,
                                         __uint_as_float(h[2 * j + 1])));
        if (live) {
          if (strat == MKV_STRATEGY_DENSE) {
            uint4* dst = reinterpret_cast<uint4*>(stv + tok * ST_V + 2 * (c0 + 16 * q));
            const uint32_t* hw = reinterpret_cast<const uint32_t*>(hv);
            dst[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            dst[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
          } else {
            // each kept channel's slot from a prefix count: independent stores
            const uint32_t mm = (m >> (16 * q)) & 0xffffu;
            const int ch0 = c0 + 16 * q;
            if (irow) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if ((mm >> j) & 1u) {
                  const int pj = pos + __popc(mm & ((1u << j) - 1u));
                  vrow[pj] = (j & 1) ? __high2half(hv[j >> 1]) : __low2half(hv[j >> 1]);
                  irow[pj] = (uint8_t)(ch0 + j);
                }
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if ((mm >> j) & 1u)
                  vrow[pos + __popc(mm & ((1u << j) - 1u))] =
                      (j & 1) ? __high2half(hv[j >> 1]) : __low2half(hv[j >> 1]);
              }
            }
            if (sm_idx) {
              for (uint32_t a = mm, n = 0; a; a &= a - 1u, ++n)
                sm_idx[pos + n] = (uint8_t)(ch0 + __ffs(a) - 1);
            }
            pos += __popc(mm);
          }
        }
      }
    } else {
      // warp w: token 32 (w mod 4) + lane (its TMEM lane quarter), channels
      // 32 (w / 4) .. 32 (w / 4) + 31
      const int tok = 32 * (warp & 3) + lane, c0 = 32 * (warp >> 2);
      const uint32_t ta = tbase + (uint32_t)b * 256u + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)c0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        uint32_t h[16], l[16];
        tmem_ld16(ta + 16 * q, h);
        tmem_ld16(ta + 128 + 16 * q, l);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          Xt[tok * XT_LD + xt_col(c0) + 16 * q + j] =
              fmaf(__uint_as_float(l[j]), 1.f / 2048.f, __uint_as_float(h[j]));
      }
    }
    tc_fence_before();
    __syncthreads();
    if (!PACK) {
      // ---- per-token channels: four lanes per token ----------------------------
      const int tok = tid >> 2, quarter = tid & 3;
      const float* xrow = Xt + tok * XT_LD + xt_col(32 * quarter);
      uint32_t k[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) k[j] = __float_as_uint(xrow[j]) & 0x7fffffffu;
      const uint32_t m = quad_topc(k, p.c);
      // this lane's kept energy, in channel order
      float kept = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float f = xrow[j];
        kept = ((m >> j) & 1u) ? fmaf(f, f, kept) : kept;
      }
      // the group's parts in channel order: (0 + 1) + (2 + 3)
      kept += __shfl_xor_sync(0xffffffffu, kept, 1);
      kept += __shfl_xor_sync(0xffffffffu, kept, 2);
      if (tok < rows) {
        tokmask[4 * tok + quarter] = m;
        gmask[(size_t)(t0 + tok) * 4 + quarter] = m;
        if (!quarter) tokkept[tok] = kept;
      }
      __syncthreads();
      // ---- per segment: column energies and kept energy, for the strategy -------
      // pieces of the tile by segment, in tile rows: segment sgf + q ends at
      // row (q + 1) S - lr0, or at the end of the stream
      const bool at_end = t0 + rows == p.T;
      for (int q = 0, r0 = 0, qend = p.S - lr0; r0 < rows; ++q, r0 = qend, qend += p.S) {
        const int r1 = min(rows, qend);
        const int sg = sgf + q;
        const bool complete = r1 == qend || (r1 == rows && at_end);
        // every thread: column tid mod 128 over rows r0 + part, r0 + part + 4, ...
        // (part = tid / 128); warp 4 also sums the tokens' kept energies
        {
          const int col = tid & (D - 1), part = tid >> 7;
          float q = 0.f;
          for (int r = r0 + part; r < r1; r += RT_THREADS / D) {
            const float val = Xt[r * XT_LD + xt_col(col)];
            q = fmaf(val, val, q);
          }
          colpart[part][col] = q;
        }
        float kq = 0.f;
        if (warp == 4) {
          for (int r = r0 + lane; r < r1; r += 32) kq += tokkept[r];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, o);
        }
        __syncthreads();
        if (tid < D) {
          float cacc = colacc[tid] + ((colpart[0][tid] + colpart[1][tid]) +
                                      (colpart[2][tid] + colpart[3][tid]));
          if (complete) {
            p.colE[((size_t)sx * p.n_seg + sg) * D + tid] = cacc;
            cacc = 0.f;
          }
          colacc[tid] = cacc;
        } else if (tid == 4 * 32) {
          float kk = segkept[0] + kq;
          if (complete) {
            p.segK[(size_t)sx * p.n_seg + sg] = kk;
            kk = 0.f;
          }
          segkept[0] = kk;
        }
        __syncthreads();          // colpart is rewritten by the next piece
      }
    } else {
      // ---- copy-out: four threads per row, 16-byte pieces k = sub, sub + 4, ... ----
      const uint32_t c = (uint32_t)p.c;
      const int r = tid >> 2, sub = tid & 3;
      if (r < rows) {
        const uint32_t ri = rowinfo[r];
        const int q = (int)(ri >> 16);
        const uint32_t rl = ri & 0xffffu;
        const SegInfo& si = seg_sh[q];
        const uint32_t off16 = hdr_sh[q].off16;
        if ((uint64_t)off16 * 16u + si.size > p.pool_check) {
          // the segment would end past the checked pool extent: report, skip
          if (sub == 0) atomicOr(p.err, DEV_ERR_CHECK);
        } else {
          uint8_t* seg = p.pool + (size_t)off16 * 16u;
          const int strat = si.strategy;
          const uint32_t srows = si.rows;
          const uint4* src = reinterpret_cast<const uint4*>(stv + r * ST_V);
          if (strat == MKV_STRATEGY_DENSE) {
            uint4* dst = reinterpret_cast<uint4*>(seg + 256u * rl);
#pragma unroll
            for (int k = sub; k < 16; k += 4) dst[k] = src[k];
          } else {
            uint4* dst = reinterpret_cast<uint4*>(
                seg + (strat == MKV_STRATEGY_SM ? pad16(c) : 0u) + 2u * c * rl);
            const int nck = (int)(c >> 3);
            for (int k = sub; k < nck; k += 4) dst[k] = src[k];
            if (strat == MKV_STRATEGY_PV) {
              uint2* idst = reinterpret_cast<uint2*>(seg + 2u * c * srows + c * rl);
              const uint2* isrc = reinterpret_cast<const uint2*>(sti + r * ST_I);
              for (int k = sub; k < nck; k += 4) idst[k] = isrc[k];
            }
            if (sub == 0) {
              if (strat == MKV_STRATEGY_PVB)
                *reinterpret_cast<uint4*>(seg + 2u * c * srows + 16u * rl) =
                    *reinterpret_cast<const uint4*>(tmask + 4 * r);
              // zero padding after the index bytes (c and c * rows are multiples of 8)
              if (strat == MKV_STRATEGY_SM && rl == 0 && (c & 15u))
                *reinterpret_cast<uint2*>(seg + c) = make_uint2(0u, 0u);
              if (strat == MKV_STRATEGY_PV && rl == srows - 1 && ((c * srows) & 15u))
                *reinterpret_cast<uint2*>(seg + 3u * c * srows) = make_uint2(0u, 0u);
            }
          }
        }
      }
    }
    // the fp32 tile and staged data are rewritten only past the next tile's
    // first barrier
  }
  cp_async_wait<0>();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------------------
// strategy: one warp per segment (all segments of all streams).  From the
// segment's column energies and kept energy: e_tot, the shared mask (top-c
// column energies, ties to the lower channel), f_SM, f_PV, and the cheapest
// strategy whose fraction reaches tau (dense always allowed; cost ties
// resolve SM, PV, dense).
// grid: ceil(2 BH n_seg / 8), block 256
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) strategy_kernel(CompressParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t e = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t n = (int64_t)2 * p.BH * p.n_seg;
  if (e >= n) return;
  const int sg = (int)(e % p.n_seg);
  float cv[4];
  uint32_t key[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    cv[m] = p.colE[(size_t)e * D + lane + 32 * m];
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
    const int rws = (int)(imin64(p.T, (int64_t)(sg + 1) * p.S) - (int64_t)sg * p.S);
    const float kept = p.segK[e];
    const float fsm = etot > 0.f ? smk / etot : 1.f;
    const float fpv = etot > 0.f ? kept / etot : 1.f;
    uint32_t best = segment_bytes(MKV_STRATEGY_DENSE, rws, p.c);
    int strat = MKV_STRATEGY_DENSE;
    const uint32_t cpv = segment_bytes(MKV_STRATEGY_PV, rws, p.c);
    const uint32_t csm = segment_bytes(MKV_STRATEGY_SM, rws, p.c);
    const uint32_t cpb = segment_bytes(MKV_STRATEGY_PVB, rws, p.c);
    // cost ties resolve SM, PV, PVB, dense: later checks win ties
    if (p.bitmask_pv && fpv >= p.tau && cpb <= best) {
      best = cpb;
      strat = MKV_STRATEGY_PVB;
    }
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
    p.seg[e] = si;
  }
}

// ---------------------------------------------------------------------------
// scan: offsets of every segment of every stream (K streams first, then V),
// segment headers and the total packed size.  One CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) scan_kernel(CompressParams p) {
  // steps of 8192 consecutive segments, thread tid taking segments 8 tid ..
  // 8 tid + 7 of the step (the 8-byte head of each segment record: size,
  // strategy, rows), a block-wide exclusive scan per step and a running carry
  const int64_t n = (int64_t)2 * p.BH * p.n_seg;
  const int tid = threadIdx.x;
  const int64_t per_x = (int64_t)p.BH * p.n_seg;
  __shared__ unsigned long long ws[65];
  __shared__ unsigned int n_dense[2];
  if (tid < 2) n_dense[tid] = 0u;
  unsigned long long carry = 0;     // bytes of all earlier steps (same in every thread)
  unsigned int dense_lo = 0, dense_hi = 0;
  for (int64_t s0 = 0; s0 < n; s0 += 8192) {
    const int64_t e0 = s0 + 8 * (int64_t)tid;
    uint2 hd[8];                     // x: size, y: strategy | rows << 16
    unsigned long long mine = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      hd[u] = e0 + u < n ? *reinterpret_cast<const uint2*>(&p.seg[e0 + u]) : make_uint2(0u, 0u);
      mine += hd[u].x;
    }
    unsigned long long tot;
    unsigned long long off = carry + block_excl_scan64(mine, ws, tot);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (e0 + u < n) {
        const uint32_t strat = hd[u].y & 0xffu;
        if (strat == MKV_STRATEGY_DENSE) {
          if (e0 + u >= per_x) ++dense_hi; else ++dense_lo;
        }
        mkv_segment_header h;
        h.off16 = (uint32_t)(off >> 4);
        h.strategy = (uint8_t)strat;
        h.reserved = 0;
        h.rows = (uint16_t)(hd[u].y >> 16);
        p.hdr[e0 + u] = h;
        off += hd[u].x;
      }
    }
    carry += tot;
  }
  if (dense_lo) atomicAdd(&n_dense[0], dense_lo);
  if (dense_hi) atomicAdd(&n_dense[1], dense_hi);
  __syncthreads();
  if (tid == 0) p.total[0] = carry;
  if (tid < 2) p.total[1 + tid] = n_dense[tid];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_gram(const CompressParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)GT_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.gram_chunks, p.BH, 2);
  gram_kernel<<<grid, GT_THREADS, GT_SMEM, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_eig(const CompressParams& p, cudaStream_t st) {
  const int smem = (2 * D * LDA + D * LDV) * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(eig_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  eig_kernel<<<2 * p.BH, EIG_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

template <bool PACK>
static cudaError_t launch_rot(const CompressParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(rotate_kernel<PACK>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)rt_smem(PACK));
  if (e != cudaSuccess) return e;
  dim3 grid(p.ctas_per_stream, p.BH, 2);
  rotate_kernel<PACK><<<grid, RT_THREADS, rt_smem(PACK), st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_analyze(const CompressParams& p, cudaStream_t st) {
  cudaError_t e = launch_rot<false>(p, st);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)2 * p.BH * p.n_seg;
  strategy_kernel<<<(unsigned)((n + 7) / 8), 256, 0, st>>>(p);
  return cudaGetLastError();
}
cudaError_t launch_pack(const CompressParams& p, cudaStream_t st) { return launch_rot<true>(p, st); }

cudaError_t launch_scan(const CompressParams& p, cudaStream_t st) {
  scan_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mkv
