// Decode-step kernels: attention over the packed two-D compressed cache.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction: query-aware token selection
// (prior-work paragraph) and attention computed on the packed dense format
// with CUDA cores, without unpacking ("Observation & Method 2").
//
// Launch order per step: qrot -> score -> topk_pass2 -> topk_write -> attn -> merge.
// No kernel waits on another CTA.  Cross-CTA results are combined with
// integer atomics (order-independent), "last CTA finishes" tickets, or a
// later launch; every floating-point sum runs in a fixed order, so a decode is
// bit-for-bit repeatable.
#include "mkv_internal.cuh"
#include "ptx.cuh"

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
    const float2 f = __half22float2(h[e]);
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

__device__ __forceinline__ int64_t clamp_t(int32_t t, int64_t T) {
  return t < 0 ? 0 : (t >= T ? T - 1 : (int64_t)t);
}

// Block-wide (the first 256 threads compute; every thread must call it): the
// bin of histogram h[NB] (shared memory) holding the krem-th largest key,
// counting from the top bin, and how many keys of that bin are still needed.
// Results land in res[0] (bin) and res[1] (remaining count).
// If no bin holds the krem-th key (an inconsistent histogram), the result is
// bin 0 with krem: wrong but safe, since every caller masks bins to [0, NB).
template <int NB>
__device__ void find_bin(const uint32_t* h, uint32_t krem, uint32_t* res, uint32_t* sh_warp) {
  constexpr int PER = NB / 256;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  if (t == 0) {
    res[0] = 0u;
    res[1] = krem;
  }
  uint32_t mine = 0, suf = 0;
  if (t < 256) {
#pragma unroll
    for (int i = 0; i < PER; ++i) mine += h[t * PER + i];
    suf = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t o = __shfl_down_sync(0xffffffffu, suf, off);
      if (lane + off < 32) suf += o;
    }
    if (lane == 0) sh_warp[warp] = suf;
  }
  __syncthreads();
  if (t < 256) {
    uint32_t above = 0;
    for (int w = warp + 1; w < 8; ++w) above += sh_warp[w];
    uint32_t running = above + (suf - mine);
    for (int i = PER - 1; i >= 0; --i) {
      const uint32_t c = h[t * PER + i];
      if (running < krem && krem <= running + c) {
        res[0] = (uint32_t)(t * PER + i);
        res[1] = krem - running;
      }
      running += c;
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// qrot: q~_i = q_i R_K for the g query heads of a KV head, q_bar = sum_i q~_i.
// R_K is staged in shared memory with 16-byte loads.  Also clears the stream's
// histogram, tickets and candidate counter for this step.
// grid: BH, block: 512 (column j = tid % 128, heads tid / 128 + 4n), dynamic
// smem 64 KB
// ---------------------------------------------------------------------------
constexpr int QR_THREADS = 512;

__global__ void __launch_bounds__(QR_THREADS) qrot_kernel(DecodeParams p) {
  extern __shared__ __align__(16) float Rs[];   // [128][128]
  __shared__ float qs[MAX_G][D];
  __shared__ float psum[4][D];
  const int s = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int tid = threadIdx.x, j = tid & 127, hq = tid >> 7;
  const float4* R4 = reinterpret_cast<const float4*>(p.RK + (size_t)s * D * D);
  float4* Rs4 = reinterpret_cast<float4*>(Rs);
#pragma unroll
  for (int x = 0; x < D * D / 4 / QR_THREADS; ++x) Rs4[tid + x * QR_THREADS] = __ldg(R4 + tid + x * QR_THREADS);
  const __half* q = p.q + ((size_t)b * p.Hq + (size_t)h * p.g) * D;
  for (int x = tid; x < p.g * D; x += QR_THREADS) qs[x / D][x % D] = __half2float(q[x]);
  uint4* hz = reinterpret_cast<uint4*>(p.hist + (size_t)s * HIST1);
  for (int x = tid; x < HIST1 / 4; x += QR_THREADS) hz[x] = make_uint4(0u, 0u, 0u, 0u);
  if (tid == 0) {
    p.tick1[s] = 0u;
    p.tick2[s] = 0u;
    p.cand_n[s] = 0u;
  }
  __syncthreads();
  float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * p.g) * D;
  float mine = 0.f;
  for (int i = hq; i < p.g; i += 4) {
    float acc = 0.f;
#pragma unroll 8
    for (int r = 0; r < D; ++r) acc = fmaf(qs[i][r], Rs[r * D + j], acc);
    qt[i * D + j] = acc;
    mine += acc;
  }
  psum[hq][j] = mine;
  __syncthreads();
  if (tid < D) p.qbar[(size_t)s * D + j] = ((psum[0][j] + psum[1][j]) + psum[2][j]) + psum[3][j];
}

// ---------------------------------------------------------------------------
// score: s_t = q_bar . k^_t for every cached token, straight from the packed
// segments.  Persistent: CTA i streams the flattened K segments
// [part[i], part[i+1]) (balanced by bytes at compression time).  One producer
// warp groups runs of whole, contiguous segments into stages of about 52 KB
// and moves each with one bulk copy (whole 128-byte lines, L2 evict-first)
// into a ring of shared-memory slots; it also lists the stage's 32-row blocks.
// 20 consumer warps take those blocks round-robin and score one row per
// lane from shared memory.  Scores go to global memory with an L2 evict-last
// hint for the selection passes; the level-1 radix histogram (key bits
// 31..20) is built on the way, and the CTA that finishes a stream last turns
// it into the level-1 bin of the k-th largest score.
// grid: G, block: 21 warps, dynamic smem n_stages * (stage_bytes + 256)
// ---------------------------------------------------------------------------
constexpr int SC_CONS = 20;
constexpr int SC_THREADS = (SC_CONS + 1) * 32;
constexpr int SC_NSLOT = 2;
constexpr int SC_MAX_STAGES = 6;
constexpr int SC_MAX_SEGS = 64;                  // segments per stage
constexpr int SC_HDR_SLOT = SC_MAX_SEGS + 2;     // header entries per stage (even start)
constexpr int SC_STAGE_TARGET = 52 * 1024;
constexpr int SC_STATIC_SMEM = SC_NSLOT * HIST1 * 4 + SC_NSLOT * D * 4 + SC_CONS * D * 4 +
                               SC_MAX_STAGES * SC_HDR_SLOT * 8 + 2048;

// shared-memory bytes of one stage slot: the stage plus slack for line alignment
__host__ __device__ constexpr size_t sc_slot(int stage_bytes) { return (size_t)stage_bytes + 256; }

// header i of the flattened K segments as two words, or zeros past the end
__device__ __forceinline__ uint2 load_hdr(const mkv_segment_header* h, int i, int end) {
  return i < end ? __ldg(reinterpret_cast<const uint2*>(h) + i) : make_uint2(0u, 0u);
}

struct StageMeta {
  int32_t seg0;        // first segment, or -1 for the end marker
  int32_t nseg;
  uint64_t byte0;      // pool offset of the slot's first byte (128-byte aligned)
};

// Dot product of one packed row with q_bar, from shared memory; one row per
// thread, CPR = 16-byte chunks per row (c / 8, or 16 for dense rows).  Lane i
// starts at chunk (i % 8) / P with P = 8 / gcd(CPR, 8): the 8 lanes of a
// quarter-warp then read 8 different 16-byte bank groups whatever the row
// stride (16 * CPR bytes), and for odd CPR every lane reads the same chunk of
// q_bar (a broadcast).  q_bar values come from the segment's gathered mask
// (SM), q_bar indexed by the stored channel (PV) or q_bar itself (dense).
// Four independent accumulators, summed in a fixed order.
template <int STRAT, int CPR>
__device__ __forceinline__ float row_dot(const uint8_t* base, int rows, int row, int lane,
                                         const float* qsrc, const float* qm) {
  constexpr uint32_t C = 8u * CPR;
  constexpr int G8 = (CPR % 8 == 0) ? 8 : ((CPR % 4 == 0) ? 4 : ((CPR % 2 == 0) ? 2 : 1));
  constexpr int P = 8 / G8;
  constexpr int NB = CPR > 5 ? 4 : CPR;      // chunks loaded ahead of the arithmetic
  const uint8_t* rowp = (STRAT == MKV_STRATEGY_SM)   ? base + pad16(C) + 2u * C * row
                        : (STRAT == MKV_STRATEGY_PV) ? base + 2u * C * row
                                                     : base + 256u * row;
  const uint8_t* idxp = base + 2u * C * (uint32_t)rows + C * (uint32_t)row;
  const int rot = (lane & 7) / P;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j0 = 0; j0 < CPR; j0 += NB) {
    uint4 raw[NB];
    uint2 ixs[NB];
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      if (j0 + jj < CPR) {
        int k = j0 + jj + rot;
        k = k >= CPR ? k - CPR : k;
        raw[jj] = *reinterpret_cast<const uint4*>(rowp + 16 * k);
        if (STRAT == MKV_STRATEGY_PV) ixs[jj] = *reinterpret_cast<const uint2*>(idxp + 8 * k);
      }
    }
#pragma unroll
    for (int jj = 0; jj < NB; ++jj) {
      if (j0 + jj < CPR) {
        int k = j0 + jj + rot;
        k = k >= CPR ? k - CPR : k;
        float v[8];
        h8_to_f(raw[jj], v);
        if (STRAT == MKV_STRATEGY_PV) {
          const uint2 ix = ixs[jj];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t ch = ((e < 4 ? ix.x : ix.y) >> (8 * (e & 3))) & 0x7fu;
            acc[e & 3] = fmaf(v[e], qsrc[ch], acc[e & 3]);
          }
        } else {
          const float* qq = (STRAT == MKV_STRATEGY_SM ? qm : qsrc) + 8 * k;
          const float4 a = *reinterpret_cast<const float4*>(qq);
          const float4 b = *reinterpret_cast<const float4*>(qq + 4);
          acc[0] = fmaf(v[0], a.x, acc[0]);
          acc[1] = fmaf(v[1], a.y, acc[1]);
          acc[2] = fmaf(v[2], a.z, acc[2]);
          acc[3] = fmaf(v[3], a.w, acc[3]);
          acc[0] = fmaf(v[4], b.x, acc[0]);
          acc[1] = fmaf(v[5], b.y, acc[1]);
          acc[2] = fmaf(v[6], b.z, acc[2]);
          acc[3] = fmaf(v[7], b.w, acc[3]);
        }
      }
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

// scores of rows [r0, r0 + 32) of one segment: one row per lane
template <int STRAT, int CPR>
__device__ __forceinline__ void score_block(const uint8_t* base, int rows, int r0, int lane,
                                            const float* qsrc, const float* qm, float* out,
                                            uint32_t* hs, uint64_t pol) {
  const int row = r0 + lane;
  if (row < rows) {
    const float sc = row_dot<STRAT, CPR>(base, rows, row, lane, qsrc, qm);
    st_f32_hint(out + row, sc, pol);
    atomicAdd(&hs[f2key(sc) >> 20], 1u);
  }
}

template <int STRAT>
__device__ __forceinline__ void score_block_c(int cpr, const uint8_t* base, int rows, int r0,
                                              int lane, const float* qsrc, const float* qm,
                                              float* out, uint32_t* hs, uint64_t pol) {
#define MKV_CASE(N) \
  case N: score_block<STRAT, N>(base, rows, r0, lane, qsrc, qm, out, hs, pol); break;
  switch (cpr) {
    MKV_CASE(1) MKV_CASE(2) MKV_CASE(3) MKV_CASE(4) MKV_CASE(5) MKV_CASE(6) MKV_CASE(7)
    MKV_CASE(8) MKV_CASE(9) MKV_CASE(10) MKV_CASE(11) MKV_CASE(12) MKV_CASE(13) MKV_CASE(14)
    MKV_CASE(15) MKV_CASE(16)
    default: break;
  }
#undef MKV_CASE
}

__global__ void __launch_bounds__(SC_THREADS, 1) score_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ uint64_t full_bar[SC_MAX_STAGES], empty_bar[SC_MAX_STAGES];
  __shared__ StageMeta meta[SC_MAX_STAGES];
  __shared__ __align__(16) uint2 shdr[SC_MAX_STAGES][SC_HDR_SLOT];   // each stage's headers
  __shared__ __align__(16) float qb[SC_NSLOT][D];
  __shared__ uint32_t hist[SC_NSLOT][HIST1];
  __shared__ __align__(16) float qm[SC_CONS][D];
  __shared__ uint32_t sh_warp[8], sh_res[2];
  __shared__ int sh_flag, sh_issued, sh_consumed;

  const int a = p.part[blockIdx.x], b = p.part[blockIdx.x + 1];
  if (a >= b) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s_first = a / p.n_seg, s_last = (b - 1) / p.n_seg;
  const int NST = p.n_stages;
  const size_t slot_bytes = sc_slot(p.stage_bytes);
  for (int x = tid; x < SC_NSLOT * HIST1; x += SC_THREADS) (&hist[0][0])[x] = 0u;
  for (int x = tid; x < SC_NSLOT * D; x += SC_THREADS) {
    const int s = s_first + x / D;
    (&qb[0][0])[x] = (s <= s_last) ? p.qbar[(size_t)s * D + (x % D)] : 0.f;
  }
  if (tid == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(&full_bar[st], 1);
      mbar_init(&empty_bar[st], SC_CONS);
    }
    mbar_init_fence();
    sh_issued = 0;
    sh_consumed = 0;
  }
  __syncthreads();

  if (warp == SC_CONS) {
    // ---- producer warp --------------------------------------------------------
    // The stages were planned at compression; plan entries come 32 at a time
    // (one per lane), the next batch already in flight.  Per stage: one bulk
    // copy of the segments' lines and one of their headers.
    const uint64_t pol = policy_evict_first();
    const int n_st = p.plan_n[blockIdx.x];
    const uint4* pl = reinterpret_cast<const uint4*>(p.plan + a);
    uint4 cur = lane < n_st ? __ldg(pl + lane) : make_uint4(0u, 0u, 0u, 0u);
    uint4 nxt = 32 + lane < n_st ? __ldg(pl + 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
    bool ok = true;
    int k = 0;
    for (; k <= n_st; ++k) {
      const int slot = k % NST, use = k / NST;
      if (use > 0) {
        bool got = true;
        if (lane == 0) got = mbar_wait(&empty_bar[slot], (use - 1) & 1);
        if (!__shfl_sync(0xffffffffu, (int)got, 0)) {
          ok = false;
          break;
        }
      }
      if (k == n_st) {          // end marker: a phase with no bytes
        if (lane == 0) {
          meta[slot].seg0 = -1;
          mbar_arrive(&full_bar[slot]);
        }
        ++k;
        break;
      }
      if (k > 0 && (k & 31) == 0) {
        cur = nxt;
        nxt = k + 32 + lane < n_st ? __ldg(pl + k + 32 + lane) : make_uint4(0u, 0u, 0u, 0u);
      }
      uint4 e;
      e.x = __shfl_sync(0xffffffffu, cur.x, k & 31);
      e.y = __shfl_sync(0xffffffffu, cur.y, k & 31);
      e.z = __shfl_sync(0xffffffffu, cur.z, k & 31);
      e.w = __shfl_sync(0xffffffffu, cur.w, k & 31);
      const StagePlan sp = *reinterpret_cast<const StagePlan*>(&e);
      if (lane == 0) {
        const uint32_t nb = sp.nlines * 128u, hb = (uint32_t)sp.nhdr2 * 16u;
        meta[slot].seg0 = (int32_t)sp.seg0;
        meta[slot].nseg = sp.nseg;
        meta[slot].byte0 = (uint64_t)sp.line0 * 128u;
        fence_proxy_async();
        mbar_arrive_expect_tx(&full_bar[slot], nb + hb);
        bulk_g2s(stage_mem + (size_t)slot * slot_bytes, p.pool + (uint64_t)sp.line0 * 128u, nb,
                 &full_bar[slot], pol);
        bulk_g2s(&shdr[slot][0], p.hdrK + (sp.seg0 & ~1u), hb, &full_bar[slot], pol);
      }
    }
    if (lane == 0) {
      if (!ok) atomicExch(p.err, DEV_ERR_TIMEOUT);
      sh_issued = k;
    }
    __syncwarp();   // the whole producer warp reaches the block barrier together
  } else {
    // ---- consumers ----------------------------------------------------------
    const uint64_t pol = policy_evict_last();
    const int bps = (p.S + 31) >> 5;      // 32-row blocks per segment
    int k = 0, last_sm = -1;
    while (true) {
      const int slot = k % NST, use = k / NST;
      // one lane polls the barrier for the warp
      int got = 1;
      if (lane == 0) got = mbar_wait(&full_bar[slot], use & 1);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) {
        if (lane == 0) atomicExch(p.err, DEV_ERR_TIMEOUT);
        break;
      }
      const StageMeta m = meta[slot];
      if (m.seg0 < 0) {
        ++k;
        break;
      }
      const uint8_t* sbase = stage_mem + (size_t)slot * slot_bytes;
      const int n_items = m.nseg * bps, hofs = m.seg0 & 1;
      for (int it = warp; it < n_items; it += SC_CONS) {
        const int ls = it / bps, blk = it - ls * bps;
        const uint2 hw = shdr[slot][ls + hofs];
        const mkv_segment_header hd = *reinterpret_cast<const mkv_segment_header*>(&hw);
        const int sg = m.seg0 + ls;
        const int rows = hd.rows, strat = hd.strategy;
        if (blk * 32 >= rows) continue;
        const uint8_t* base = sbase + ((uint64_t)hd.off16 * 16u - m.byte0);
        const int s = sg / p.n_seg;
        const int sl = s - s_first;
        const float* qsrc = sl < SC_NSLOT ? qb[sl] : p.qbar + (size_t)s * D;
        uint32_t* hs = sl < SC_NSLOT ? hist[sl] : p.hist + (size_t)s * HIST1;
        float* out = p.scores + (size_t)s * p.Tp + (int64_t)(sg - s * p.n_seg) * p.S;
        if (strat == MKV_STRATEGY_SM) {
          if (last_sm != sg) {
            __syncwarp();
            for (int jj = lane; jj < p.c; jj += 32) qm[warp][jj] = qsrc[base[jj] & 127];
            __syncwarp();
            last_sm = sg;
          }
          score_block_c<MKV_STRATEGY_SM>(p.c >> 3, base, rows, blk * 32, lane, qsrc, qm[warp],
                                         out, hs, pol);
        } else if (strat == MKV_STRATEGY_PV) {
          score_block_c<MKV_STRATEGY_PV>(p.c >> 3, base, rows, blk * 32, lane, qsrc, qm[warp],
                                         out, hs, pol);
        } else {
          score_block<MKV_STRATEGY_DENSE, 16>(base, rows, blk * 32, lane, qsrc, qm[warp], out, hs,
                                              pol);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
      ++k;
    }
    if (warp == 0 && lane == 0) sh_consumed = k;
  }
  __syncthreads();
  // after a timeout, wait (bounded) for copies still landing in shared memory
  if (tid == 0) {
    for (int k = sh_consumed; k < sh_issued; ++k) mbar_wait(&full_bar[k % NST], (k / NST) & 1);
  }
  __syncthreads();
  // ---- level-1 histogram: merge into the stream's global histogram ----------
  for (int sl = 0; sl < SC_NSLOT; ++sl) {
    const int s = s_first + sl;
    if (s > s_last) break;
    uint32_t* gh = p.hist + (size_t)s * HIST1;
    for (int x = tid; x < HIST1; x += SC_THREADS)
      if (hist[sl][x]) atomicAdd(&gh[x], hist[sl][x]);
  }
  __threadfence();
  __syncthreads();
  for (int s = s_first; s <= s_last; ++s) {
    if (tid == 0) sh_flag = (atomicAdd(&p.tick1[s], 1u) == (uint32_t)p.cta_cnt[s] - 1u);
    __syncthreads();
    if (sh_flag) {
      __threadfence();
      uint32_t* h = &hist[0][0];
      for (int x = tid; x < HIST1; x += SC_THREADS) h[x] = __ldcg(&p.hist[(size_t)s * HIST1 + x]);
      __syncthreads();
      find_bin<HIST1>(h, (uint32_t)p.kk, sh_res, sh_warp);
      if (tid == 0) {
        p.state[s].b1 = sh_res[0] & (HIST1 - 1);
        p.state[s].k1 = sh_res[1];
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// topk_pass2: per 4096-token chunk, counts the tokens whose key lies above
// the level-1 bin (all selected) and appends the tokens of that bin to the
// stream's candidate list.  The CTA that finishes a stream last selects
// exactly among the candidates (keys by two more radix digits, then equal
// keys by lowest token index), then turns the per-chunk counts into output
// offsets.
// grid: (topk_chunks, BH), block 256, 16 tokens per thread
// ---------------------------------------------------------------------------
constexpr int TK_THREADS = 256;
constexpr int TK_PER = TOPK_CHUNK / TK_THREADS;   // 16

__device__ __forceinline__ void load16(const float* sc, int64_t t0, int64_t T, float v[TK_PER],
                                       bool hint_first, uint64_t pol) {
  if (t0 + TK_PER <= T) {
#pragma unroll
    for (int i = 0; i < TK_PER / 4; ++i) {
      const float4 f = hint_first ? ld_f4_hint(sc + t0 + 4 * i, pol)
                                  : __ldcg(reinterpret_cast<const float4*>(sc + t0) + i);
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < TK_PER; ++i) v[i] = (t0 + i < T) ? __ldcg(sc + t0 + i) : 0.f;
  }
}

// exclusive scan of one value per thread over the block (TK_THREADS threads)
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  uint32_t before = 0, all = 0;
  for (int w = 0; w < TK_THREADS / 32; ++w) {
    if (w < warp) before += sh[w];
    all += sh[w];
  }
  __syncthreads();
  if (total) *total = all;
  return before + inc - v;
}

__global__ void __launch_bounds__(TK_THREADS) topk_pass2_kernel(DecodeParams p) {
  const int s = blockIdx.y, ch = blockIdx.x, tid = threadIdx.x;
  __shared__ uint32_t sh_scan[TK_THREADS / 32], sh_warp[8], sh_res[2];
  __shared__ uint32_t hbuf[2048];
  __shared__ int sh_last;
  __shared__ uint32_t sh_base;
  const uint32_t b1 = p.state[s].b1;
  const int64_t t0 = (int64_t)ch * TOPK_CHUNK + (int64_t)tid * TK_PER;
  const float* sc = p.scores + (size_t)s * p.Tp;
  float v[TK_PER];
  load16(sc, t0, p.T, v, false, 0);
  uint32_t sure = 0, ncand = 0, keys[TK_PER];
#pragma unroll
  for (int i = 0; i < TK_PER; ++i) {
    keys[i] = f2key(v[i]);
    const bool valid = t0 + i < p.T;
    const uint32_t bin = keys[i] >> 20;
    sure += valid && bin > b1;
    ncand += valid && bin == b1;
  }
  uint32_t sure_all, ncand_all;
  block_excl_scan(sure, sh_scan, &sure_all);
  const uint32_t my_off = block_excl_scan(ncand, sh_scan, &ncand_all);
  if (tid == 0) {
    p.cnt[(size_t)s * p.topk_chunks + ch] = (int32_t)sure_all;
    sh_base = ncand_all ? atomicAdd(&p.cand_n[s], ncand_all) : 0u;
  }
  __syncthreads();
  uint2* cand = p.cand + (size_t)s * p.Tp;
  uint32_t pos = sh_base + my_off;
#pragma unroll
  for (int i = 0; i < TK_PER; ++i) {
    if (t0 + i < p.T && (keys[i] >> 20) == b1) cand[pos++] = make_uint2(keys[i], (uint32_t)(t0 + i));
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = (atomicAdd(&p.tick2[s], 1u) == gridDim.x - 1u);
  __syncthreads();
  if (!sh_last) return;
  __threadfence();

  // ---- last CTA of the stream: exact threshold among the candidates --------
  const uint32_t N = __ldcg(&p.cand_n[s]);
  const uint32_t need = p.state[s].k1;
  // key bits 19..10
  for (int x = tid; x < 1024; x += TK_THREADS) hbuf[x] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < N; i += TK_THREADS) atomicAdd(&hbuf[(__ldcg(&cand[i].x) >> 10) & 1023u], 1u);
  __syncthreads();
  find_bin<1024>(hbuf, need, sh_res, sh_warp);
  const uint32_t bA = sh_res[0] & 1023u, needA = sh_res[1];
  // key bits 9..0 among keys in bin bA
  for (int x = tid; x < 1024; x += TK_THREADS) hbuf[x] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < N; i += TK_THREADS) {
    const uint32_t key = __ldcg(&cand[i].x);
    if (((key >> 10) & 1023u) == bA) atomicAdd(&hbuf[key & 1023u], 1u);
  }
  __syncthreads();
  find_bin<1024>(hbuf, needA, sh_res, sh_warp);
  const uint32_t bB = sh_res[0] & 1023u, need_eq = sh_res[1];
  const uint32_t n_eq = hbuf[bB];
  const uint32_t thr = (b1 << 20) | (bA << 10) | bB;
  __syncthreads();
  int32_t t_cut = 0x7fffffff;
  if (need_eq < n_eq) {
    // the need_eq lowest token indices among keys equal to thr: radix select
    // on u = 0x7fffffff - t (largest u = lowest t), bits 30..20, 19..10, 9..0
    uint32_t prefix = 0, krem = need_eq;
    for (int lev = 0; lev < 3; ++lev) {
      const int nb = lev == 0 ? 2048 : 1024;
      const int shift = lev == 0 ? 20 : (lev == 1 ? 10 : 0);
      for (int x = tid; x < nb; x += TK_THREADS) hbuf[x] = 0u;
      __syncthreads();
      for (uint32_t i = tid; i < N; i += TK_THREADS) {
        const uint2 cv = __ldcg(&cand[i]);
        if (cv.x != thr) continue;
        const uint32_t u = 0x7fffffffu - cv.y;
        if (lev > 0 && (u >> (shift + 10)) != prefix) continue;
        atomicAdd(&hbuf[(u >> shift) & (uint32_t)(nb - 1)], 1u);
      }
      __syncthreads();
      if (lev == 0) find_bin<2048>(hbuf, krem, sh_res, sh_warp);
      else find_bin<1024>(hbuf, krem, sh_res, sh_warp);
      prefix = (prefix << (lev == 0 ? 0 : 10)) | (sh_res[0] & (uint32_t)(nb - 1));
      krem = sh_res[1];
    }
    t_cut = (int32_t)(0x7fffffffu - prefix);
  }
  if (tid == 0) {
    p.state[s].thr = thr;
    p.state[s].t_cut = t_cut;
  }
  // per-chunk counts of the selected candidates, then exclusive offsets
  int32_t* cnt = p.cnt + (size_t)s * p.topk_chunks;
  for (uint32_t i = tid; i < N; i += TK_THREADS) {
    const uint2 cv = __ldcg(&cand[i]);
    if (cv.x > thr || (cv.x == thr && (int32_t)cv.y <= t_cut)) atomicAdd(&cnt[cv.y / TOPK_CHUNK], 1);
  }
  __threadfence();
  __syncthreads();
  const int nch = p.topk_chunks;
  const int per = (nch + TK_THREADS - 1) / TK_THREADS;
  const int lo = min(nch, tid * per), hi = min(nch, lo + per);
  uint32_t mine = 0;
  for (int x = lo; x < hi; ++x) mine += (uint32_t)__ldcg(&cnt[x]);
  uint32_t off = block_excl_scan(mine, sh_scan, nullptr);
  for (int x = lo; x < hi; ++x) {
    const uint32_t c = (uint32_t)__ldcg(&cnt[x]);
    cnt[x] = (int32_t)off;
    off += c;
  }
}

// writes the selected token ids of one chunk in ascending order
__global__ void __launch_bounds__(TK_THREADS) topk_write_kernel(DecodeParams p) {
  const int s = blockIdx.y, ch = blockIdx.x, tid = threadIdx.x;
  __shared__ uint32_t sh_scan[TK_THREADS / 32];
  const uint32_t thr = p.state[s].thr;
  const int32_t t_cut = p.state[s].t_cut;
  const int base = p.cnt[(size_t)s * p.topk_chunks + ch];
  const int64_t t0 = (int64_t)ch * TOPK_CHUNK + (int64_t)tid * TK_PER;
  float v[TK_PER];
  load16(p.scores + (size_t)s * p.Tp, t0, p.T, v, true, policy_evict_first());
  uint32_t n = 0;
  bool selv[TK_PER];
#pragma unroll
  for (int i = 0; i < TK_PER; ++i) {
    const uint32_t key = f2key(v[i]);
    const int64_t t = t0 + i;
    selv[i] = t < p.T && (key > thr || (key == thr && t <= t_cut));
    n += selv[i];
  }
  int pos = base + (int)block_excl_scan(n, sh_scan, nullptr);
  int32_t* out = p.sel + (size_t)s * p.kk;
  int32_t* out2 = p.sel_user ? p.sel_user + (size_t)s * p.kk : nullptr;
#pragma unroll
  for (int i = 0; i < TK_PER; ++i) {
    if (selv[i] && pos >= 0 && pos < p.kk) {
      out[pos] = (int32_t)(t0 + i);
      if (out2) out2[pos] = (int32_t)(t0 + i);
    }
    pos += selv[i];
  }
}

// ---------------------------------------------------------------------------
// attn: split-K attention of the g query heads over a chunk of <= 128
// selected tokens, reading the packed K/V rows in place (fp16 values + uint8
// channel indices).  Row addresses of the chunk are resolved first.  Then a
// group of 8 lanes serves a token, one 16-byte chunk (8 stored values) per
// lane, and every thread fetches the chunks of its tokens together: K chunks
// give partial logits (summed over the 8 lanes by a fixed butterfly), V
// chunks are copied into a zeroed fp16 tile V[token][channel] (rows padded to
// 65 words).  After the softmax statistics, thread j sums p_t,i * V[t][j] over
// the tokens in order.  Partials per (stream, chunk, head): max logit m, sum
// of exp l and the unnormalised output in the rotated V basis.
// grid: (attn_chunks, BH), block 128, dynamic smem
// ---------------------------------------------------------------------------
constexpr int ATTN_THREADS = 128;
constexpr int VD_LD = 130;          // halves per V tile row
constexpr uint64_t NO_IDX = ~0ull;

__device__ __forceinline__ void row_addr(const mkv_segment_header* hdr, int64_t t, int S, int c,
                                         uint64_t* vals, uint64_t* idx, int* nnz) {
  const int64_t sg = t / S;
  const uint32_t r = (uint32_t)(t - sg * S);
  const mkv_segment_header hd = hdr[sg];
  const uint64_t base = (uint64_t)hd.off16 * 16u;
  if (hd.strategy == MKV_STRATEGY_SM) {
    *vals = base + pad16((uint32_t)c) + 2u * (uint32_t)c * r;
    *idx = base;
    *nnz = c;
  } else if (hd.strategy == MKV_STRATEGY_PV) {
    *vals = base + 2u * (uint32_t)c * r;
    *idx = base + 2u * (uint32_t)c * hd.rows + (uint32_t)c * r;
    *nnz = c;
  } else {
    *vals = base + 256u * r;
    *idx = NO_IDX;
    *nnz = D;
  }
}

size_t attn_smem_bytes(int g, int chunk) {
  const int gp = (g + 3) & ~3;
  return (size_t)chunk * VD_LD * 2 + (size_t)chunk * (4 * 8 + 2 * 4) +
         sizeof(float) * ((size_t)D * gp + (size_t)chunk * gp + 2 * g);
}

__device__ __forceinline__ int chan_of(const uint2& x, int e) {
  return (int)(((e < 4 ? x.x : x.y) >> (8 * (e & 3))) & 0x7fu);
}

// everything after the row addresses; GM = heads per instantiation (4 or 16)
template <int GM>
__device__ __forceinline__ void attn_body(const DecodeParams& p, int s, int chk, int n,
                                          const uint64_t* kv_, const uint64_t* ki_,
                                          const int* kn_, const uint64_t* vv_,
                                          const uint64_t* vi_, const int* vn_, __half* Vd,
                                          const float* qs, float* lg, float* ml) {
  const int g = p.g, gp = (g + 3) & ~3;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cl = tid & 7, tg = tid >> 3;
  constexpr int U = 4;                          // tokens per thread per batch
  const float scale = 0.08838834764831845f;     // 1 / sqrt(128)
  // ---- logits and V tile: 8 lanes per token, 8 tokens per thread ---------
  for (int base = 0; base < ATTN_THREADS / 16; base += U) {
    uint4 kvv[U], vvv[U];
    uint2 kix[U], vix[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = tg + 16 * (base + u);
      kvv[u] = vvv[u] = make_uint4(0u, 0u, 0u, 0u);
      kix[u] = vix[u] = make_uint2(0u, 0u);
      if (i < n) {
        if (8 * cl < kn_[i]) {
          kvv[u] = __ldg(reinterpret_cast<const uint4*>(p.pool + kv_[i]) + cl);
          if (ki_[i] != NO_IDX) kix[u] = __ldg(reinterpret_cast<const uint2*>(p.pool + ki_[i]) + cl);
        }
        if (8 * cl < vn_[i]) {
          vvv[u] = __ldg(reinterpret_cast<const uint4*>(p.pool + vv_[i]) + cl);
          if (vi_[i] != NO_IDX) vix[u] = __ldg(reinterpret_cast<const uint2*>(p.pool + vi_[i]) + cl);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = tg + 16 * (base + u);
      float part[GM];
#pragma unroll
      for (int hh = 0; hh < GM; ++hh) part[hh] = 0.f;
      if (i < n) {
        // rows with more than 64 stored values (dense, or c > 64) have chunks 8..15
        for (int ck = cl; ck < 16; ck += 8) {
          uint4 kr = kvv[u], vr = vvv[u];
          uint2 kx = kix[u], vx = vix[u];
          if (ck >= 8) {
            if (8 * ck >= kn_[i] && 8 * ck >= vn_[i]) break;
            kr = vr = make_uint4(0u, 0u, 0u, 0u);
            kx = vx = make_uint2(0u, 0u);
            if (8 * ck < kn_[i]) {
              kr = __ldg(reinterpret_cast<const uint4*>(p.pool + kv_[i]) + ck);
              if (ki_[i] != NO_IDX) kx = __ldg(reinterpret_cast<const uint2*>(p.pool + ki_[i]) + ck);
            }
            if (8 * ck < vn_[i]) {
              vr = __ldg(reinterpret_cast<const uint4*>(p.pool + vv_[i]) + ck);
              if (vi_[i] != NO_IDX) vx = __ldg(reinterpret_cast<const uint2*>(p.pool + vi_[i]) + ck);
            }
          }
          if (8 * ck < vn_[i]) {
            const __half* hv = reinterpret_cast<const __half*>(&vr);
            __half* vrow = Vd + (size_t)i * VD_LD;
            const bool dense = vi_[i] == NO_IDX;
#pragma unroll
            for (int e = 0; e < 8; ++e) vrow[dense ? 8 * ck + e : chan_of(vx, e)] = hv[e];
          }
          if (8 * ck < kn_[i]) {
            float v[8];
            h8_to_f(kr, v);
            const bool dense = ki_[i] == NO_IDX;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float* qq = qs + (dense ? 8 * ck + e : chan_of(kx, e)) * gp;
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
  // ---- softmax statistics per head (warp per head, fixed-order reductions) --
  for (int hh = warp; hh < g; hh += ATTN_THREADS / 32) {
    float m = -INFINITY;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, lg[i * gp + hh]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float l = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float e = expf(lg[i * gp + hh] - m);
      lg[i * gp + hh] = e;
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
  // ---- o~_i[j] = sum_t p_t,i V[t][j]: thread j, tokens in order ------------
  const int jc = tid;   // channel
  float o[GM];
#pragma unroll
  for (int hh = 0; hh < GM; ++hh) o[hh] = 0.f;
  for (int i = 0; i < n; ++i) {
    const float v = __half2float(Vd[(size_t)i * VD_LD + jc]);
#pragma unroll
    for (int h4 = 0; h4 < GM; h4 += 4) {
      if (h4 < g) {
        const float4 p4 = *reinterpret_cast<const float4*>(lg + i * gp + h4);
        o[h4] = fmaf(p4.x, v, o[h4]);
        o[h4 + 1] = fmaf(p4.y, v, o[h4 + 1]);
        o[h4 + 2] = fmaf(p4.z, v, o[h4 + 2]);
        o[h4 + 3] = fmaf(p4.w, v, o[h4 + 3]);
      }
    }
  }
  const size_t pbase = ((size_t)s * p.attn_chunks + chk) * g;
#pragma unroll
  for (int hh = 0; hh < GM; ++hh)
    if (hh < g) p.part_o[(pbase + hh) * D + jc] = o[hh];
  if (tid < 2 * g) p.part_ml[pbase * 2 + tid] = ml[tid];
}

__global__ void __launch_bounds__(ATTN_THREADS, 4) attn_kernel(DecodeParams p) {
  extern __shared__ __align__(16) uint8_t asm_[];
  const int s = blockIdx.y, chk = blockIdx.x;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g, gp = (g + 3) & ~3;
  const int tid = threadIdx.x;
  const int CH = p.attn_chunk;
  __half* Vd = reinterpret_cast<__half*>(asm_);                                // [CH][VD_LD]
  uint64_t* kv_ = reinterpret_cast<uint64_t*>(asm_ + (size_t)CH * VD_LD * 2);  // [CH]
  uint64_t* ki_ = kv_ + CH;
  uint64_t* vv_ = ki_ + CH;
  uint64_t* vi_ = vv_ + CH;
  int* kn_ = reinterpret_cast<int*>(vi_ + CH);
  int* vn_ = kn_ + CH;
  float* qs = reinterpret_cast<float*>(vn_ + CH);                              // [128][gp]
  float* lg = qs + D * gp;                                                     // [CH][gp]
  float* ml = lg + CH * gp;                                                    // [g][2]
  const float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * g) * D;
  for (int x = tid; x < D * gp; x += ATTN_THREADS) {
    const int chn = x / gp, hh = x % gp;
    qs[x] = hh < g ? qt[hh * D + chn] : 0.f;
  }
  {
    uint32_t* z = reinterpret_cast<uint32_t*>(Vd);
    for (int x = tid; x < CH * VD_LD / 2; x += ATTN_THREADS) z[x] = 0u;
  }
  const int j0 = chk * CH;
  const int n = min(CH, p.kk - j0);
  if (tid < n) {
    const int64_t t = clamp_t(p.sel[(size_t)s * p.kk + j0 + tid], p.T);
    row_addr(p.hdrK + (size_t)s * p.n_seg, t, p.S, p.c, &kv_[tid], &ki_[tid], &kn_[tid]);
    row_addr(p.hdrV + (size_t)s * p.n_seg, t, p.S, p.c, &vv_[tid], &vi_[tid], &vn_[tid]);
  }
  __syncthreads();
  if (g <= 4) attn_body<4>(p, s, chk, n, kv_, ki_, kn_, vv_, vi_, vn_, Vd, qs, lg, ml);
  else attn_body<MAX_G>(p, s, chk, n, kv_, ki_, kn_, vv_, vi_, vn_, Vd, qs, lg, ml);
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

// ---------------------------------------------------------------------------
// partition of the K segments over the score kernel's CTAs (compression time):
// CTA i starts at the first segment whose payload starts at or after
// i * total / G bytes of the K payload.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) partition_kernel(const mkv_segment_header* hdrK,
                                                         int n_streams, int n_seg, int c, int G,
                                                         int32_t* part, int32_t* cta_cnt) {
  const int64_t n = (int64_t)n_streams * n_seg;
  const mkv_segment_header last = hdrK[n - 1];
  const uint64_t first = (uint64_t)hdrK[0].off16 * 16u;
  const uint64_t total =
      (uint64_t)last.off16 * 16u + segment_bytes(last.strategy, last.rows, c) - first;
  for (int s = threadIdx.x; s < n_streams; s += blockDim.x) cta_cnt[s] = 0;
  for (int i = threadIdx.x; i <= G; i += blockDim.x) {
    const uint64_t target = (uint64_t)(((double)i / (double)G) * (double)total);
    int64_t lo = 0, hi = n;   // first segment whose start >= target
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if ((uint64_t)hdrK[mid].off16 * 16u - first >= target) hi = mid; else lo = mid + 1;
    }
    part[i] = (int32_t)(i == 0 ? 0 : (i == G ? n : lo));
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G; i += blockDim.x) {
    const int a = part[i], b = part[i + 1];
    if (a >= b) continue;
    for (int s = a / n_seg; s <= (b - 1) / n_seg; ++s) atomicAdd(&cta_cnt[s], 1);
  }
}

// ---------------------------------------------------------------------------
// plan: the score kernel's stages for CTA i (one warp per CTA, compression
// time).  Whole segments are grouped in order while the stage's line-aligned
// span stays within stage_bytes (at least one segment per stage) and it holds
// at most SC_MAX_SEGS segments.  A stage never has more entries than its CTA
// has segments, so CTA i's plan fits in plan[part[i] .. part[i + 1]).
// ---------------------------------------------------------------------------
__device__ __forceinline__ StagePlan make_stage(int seg0, int nseg, uint64_t off0, uint64_t end) {
  StagePlan sp;
  sp.seg0 = (uint32_t)seg0;
  sp.nseg = (uint16_t)nseg;
  sp.nhdr2 = (uint16_t)(((uint32_t)(seg0 + nseg) + 1u) / 2u - (uint32_t)seg0 / 2u);
  sp.line0 = (uint32_t)(off0 >> 7);
  sp.nlines = (uint32_t)(((end + 127u) >> 7) - (off0 >> 7));
  return sp;
}

__global__ void __launch_bounds__(32) plan_kernel(const mkv_segment_header* hdrK, int c,
                                                  int stage_bytes, const int32_t* part,
                                                  StagePlan* plan, int32_t* plan_n) {
  const int i = blockIdx.x, lane = threadIdx.x;
  const int a = part[i], b = part[i + 1];
  int k = 0, seg0 = a, nseg = 0;
  uint64_t off0 = 0, end = 0;
  for (int base = a; base < b; base += 32) {
    const uint2 w = load_hdr(hdrK, base + lane, b);
    const mkv_segment_header hd = *reinterpret_cast<const mkv_segment_header*>(&w);
    const uint64_t st = (uint64_t)hd.off16 * 16u;
    const uint64_t se = st + segment_bytes(hd.strategy, hd.rows, c);
    const int nb = min(32, b - base);
    for (int j = 0; j < nb; ++j) {
      const uint64_t sj = __shfl_sync(0xffffffffu, st, j);
      const uint64_t ej = __shfl_sync(0xffffffffu, se, j);
      if (nseg > 0 && (nseg == SC_MAX_SEGS || ((ej + 127u) & ~127ull) - (off0 & ~127ull) >
                                                  (uint64_t)stage_bytes + 128u)) {
        if (lane == 0) plan[a + k] = make_stage(seg0, nseg, off0, end);
        ++k;
        seg0 = base + j;
        nseg = 0;
      }
      if (nseg == 0) off0 = sj;
      end = ej;
      ++nseg;
    }
  }
  if (nseg > 0) {
    if (lane == 0) plan[a + k] = make_stage(seg0, nseg, off0, end);
    ++k;
  }
  if (lane == 0) plan_n[i] = k;
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
void score_stage_plan(int S, int c, int* stage_bytes, int* n_stages) {
  uint32_t mx = 0;
  for (int st = 0; st < 3; ++st) {
    const uint32_t b = segment_bytes(st, S, c);
    mx = mx > b ? mx : b;
  }
  const int sb = (int)(mx > (uint32_t)SC_STAGE_TARGET ? mx : (uint32_t)SC_STAGE_TARGET);
  const int budget = 227 * 1024 - SC_STATIC_SMEM;
  int ns = budget / (int)sc_slot(sb);
  ns = ns > SC_MAX_STAGES ? SC_MAX_STAGES : ns;
  *stage_bytes = sb;
  *n_stages = ns;
}

cudaError_t prepare_decode_kernels() {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)attn_smem_bytes(MAX_G, ATTN_MAX_CHUNK));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           48 * 1024 + 4 * 1024);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qrot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, D * D * 4);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              227 * 1024 - SC_STATIC_SMEM);
}

cudaError_t launch_partition(const mkv_segment_header* hdrK, int n_streams, int n_seg, int c,
                             int G, int stage_bytes, int32_t* part, int32_t* cta_cnt,
                             StagePlan* plan, int32_t* plan_n, cudaStream_t st) {
  partition_kernel<<<1, 1024, 0, st>>>(hdrK, n_streams, n_seg, c, G, part, cta_cnt);
  plan_kernel<<<G, 32, 0, st>>>(hdrK, c, stage_bytes, part, plan, plan_n);
  return cudaGetLastError();
}

cudaError_t launch_qrot(const DecodeParams& p, cudaStream_t st) {
  qrot_kernel<<<p.B * p.H, QR_THREADS, D * D * 4, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_score(const DecodeParams& p, cudaStream_t st) {
  score_kernel<<<p.G, SC_THREADS, sc_slot(p.stage_bytes) * p.n_stages, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.topk_chunks, p.B * p.H);
  topk_pass2_kernel<<<grid, TK_THREADS, 0, st>>>(p);
  topk_write_kernel<<<grid, TK_THREADS, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.attn_chunks, p.B * p.H);
  attn_kernel<<<grid, ATTN_THREADS, attn_smem_bytes(p.g, p.attn_chunk), st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.B * p.H, D / MG_ROWS);
  merge_kernel<<<grid, MG_THREADS, sizeof(float) * (size_t)p.attn_chunks * p.g, st>>>(p);
  return cudaGetLastError();
}

}  // namespace mkv
