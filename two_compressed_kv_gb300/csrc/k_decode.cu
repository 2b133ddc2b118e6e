// Decode-step kernels: attention over the packed two-D compressed cache.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction: query-aware token selection
// (prior-work paragraph) and attention computed on the packed dense format
// with CUDA cores, without unpacking ("Observation & Method 2").
//
// Launch order per step: qrot -> score -> select -> attn -> merge.
// No kernel waits on another CTA.  Cross-CTA results are combined with
// integer atomics (order-independent), "last CTA finishes" tickets, or a
// later launch; every floating-point sum runs in a fixed order, so a decode is
// bit-for-bit repeatable.
#include <cooperative_groups.h>

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

// Inverse of f2key for keys of finite floats (key 0x80000000 gives +0).
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
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
  if (tid == 0) p.tick1[s] = 0u;
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

// CPR = c / 8 is a template parameter of the whole kernel (one instantiation
// per c), so the per-item dispatch is only on the segment's strategy.
template <int CPR>
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
    const int bps = (p.S + 31) >> 5;      // 32-row blocks per segment (1..8)
    // it / bps = (it * bps_inv) >> 16, exact for it < 512
    const uint32_t bps_inv = (65536u + (uint32_t)bps - 1u) / (uint32_t)bps;
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
      // stream of the stage's first segment; later segments step over stream
      // boundaries (at most a few per stage)
      int s_cur = m.seg0 / p.n_seg, s_end = (s_cur + 1) * p.n_seg;
      for (int it = warp; it < n_items; it += SC_CONS) {
        const int ls = (int)(((uint32_t)it * bps_inv) >> 16), blk = it - ls * bps;
        const uint2 hw = shdr[slot][ls + hofs];
        const mkv_segment_header hd = *reinterpret_cast<const mkv_segment_header*>(&hw);
        const int sg = m.seg0 + ls;
        const int rows = hd.rows, strat = hd.strategy;
        if (blk * 32 >= rows) continue;
        const uint8_t* base = sbase + ((uint64_t)hd.off16 * 16u - m.byte0);
        while (sg >= s_end) {
          ++s_cur;
          s_end += p.n_seg;
        }
        const int s = s_cur;
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
          score_block<MKV_STRATEGY_SM, CPR>(base, rows, blk * 32, lane, qsrc, qm[warp], out, hs,
                                            pol);
        } else if (strat == MKV_STRATEGY_PV) {
          score_block<MKV_STRATEGY_PV, CPR>(base, rows, blk * 32, lane, qsrc, qm[warp], out, hs,
                                            pol);
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

__global__ void __launch_bounds__(SEL_THREADS, 1) select_kernel(DecodeParams p) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t sel_dyn[];
  uint2* cbuf = reinterpret_cast<uint2*>(sel_dyn);                        // [SEL_CAP]
  int32_t* bbuf = reinterpret_cast<int32_t*>(sel_dyn + SEL_CAP * sizeof(uint2));  // [SEL_CAP]
  __shared__ SelShared sh;
  const int R = (int)cl.num_blocks(), r = (int)cl.block_rank();
  const int s = blockIdx.y, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  for (int base = 0; base < ATTN_THREADS / 16; base += U) {
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

__global__ void __launch_bounds__(ATTN_THREADS, 4) attn_kernel(DecodeParams p) {
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
  if (tid < n) {
    const int64_t t = clamp_t(p.sel[(size_t)s * p.kk + j0 + tid], p.T);
    const uint2 km = row_meta(p.hdrK + (size_t)s * p.n_seg, t, p.S, p.c);
    const uint2 vm = row_meta(p.hdrV + (size_t)s * p.n_seg, t, p.S, p.c);
    meta[tid] = make_uint4(km.x, km.y, vm.x, vm.y);
  }
  __syncthreads();
  if (g <= 4) attn_body<4>(p, s, chk, n, meta, Vd, Pt, qs, lg, ml);
  else attn_body<MAX_G>(p, s, chk, n, meta, Vd, Pt, qs, lg, ml);
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
  e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)SEL_SMEM);
  if (e != cudaSuccess) return e;
#define MKV_SCORE_ATTR(N)                                                                   \
  e = cudaFuncSetAttribute(score_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                           227 * 1024 - SC_STATIC_SMEM);                                  \
  if (e != cudaSuccess) return e;
  MKV_SCORE_ATTR(1) MKV_SCORE_ATTR(2) MKV_SCORE_ATTR(3) MKV_SCORE_ATTR(4) MKV_SCORE_ATTR(5)
  MKV_SCORE_ATTR(6) MKV_SCORE_ATTR(7) MKV_SCORE_ATTR(8) MKV_SCORE_ATTR(9) MKV_SCORE_ATTR(10)
  MKV_SCORE_ATTR(11) MKV_SCORE_ATTR(12) MKV_SCORE_ATTR(13) MKV_SCORE_ATTR(14)
  MKV_SCORE_ATTR(15) MKV_SCORE_ATTR(16)
#undef MKV_SCORE_ATTR
  return cudaSuccess;
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
  const size_t smem = sc_slot(p.stage_bytes) * p.n_stages;
  switch (p.c >> 3) {
#define MKV_SCORE_CASE(N) \
  case N: score_kernel<N><<<p.G, SC_THREADS, smem, st>>>(p); break;
    MKV_SCORE_CASE(1) MKV_SCORE_CASE(2) MKV_SCORE_CASE(3) MKV_SCORE_CASE(4) MKV_SCORE_CASE(5)
    MKV_SCORE_CASE(6) MKV_SCORE_CASE(7) MKV_SCORE_CASE(8) MKV_SCORE_CASE(9) MKV_SCORE_CASE(10)
    MKV_SCORE_CASE(11) MKV_SCORE_CASE(12) MKV_SCORE_CASE(13) MKV_SCORE_CASE(14)
    MKV_SCORE_CASE(15) MKV_SCORE_CASE(16)
#undef MKV_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int select_cluster_size(int n_streams, int64_t T, int G) {
  int R = 1;
  while (R < 8 && (int64_t)n_streams * R * 2 <= G && T / (2 * R) >= 4096) R *= 2;
  return R;
}

cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.sel_R, p.B * p.H, 1);
  cfg.blockDim = dim3(SEL_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SEL_SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.sel_R;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, select_kernel, p);
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
