// Decode step, first part: query rotation and the score pass.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction: query-aware token selection
// (prior-work paragraph) over the packed two-D compressed keys, computed on
// the packed dense format without unpacking ("Observation & Method 2").
//
// Launch order per step: qrot -> score -> select -> attn -> merge.  No kernel
// waits on another CTA.  Cross-CTA results are combined with integer atomics
// (order-independent), "last CTA finishes" tickets, or a later launch; every
// floating-point sum runs in a fixed order, so a decode is bit-for-bit
// repeatable.  This file also holds the compression-time partition of the
// score work (partition and plan kernels).
#include "block_scan.cuh"
#include "decode_common.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// qrot: q~_i = q_i R_K for the g query heads of a KV head, q_bar = sum_i q~_i.
// R_K is staged in shared memory with 16-byte loads.  Also clears the stream's
// histogram and ticket for this step.
// grid: BH, block: 512 (column j = tid % 128, heads tid / 128 + 4n), dynamic
// smem 64 KB
// ---------------------------------------------------------------------------
constexpr int QR_THREADS = 512;

__device__ __forceinline__ void qrot_kernel_body(const DecodeParams& p) {
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
  // R_K belongs to the ctx; q and the step's buffers may still be in use by
  // the kernel before this one
  griddep_wait();
  if (p.pdl_trigger) griddep_launch();
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
  const int n_tail = (int)(p.T - p.T_packed);
  if (tid < D) {
    const float qb = ((psum[0][j] + psum[1][j]) + psum[2][j]) + psum[3][j];
    p.qbar[(size_t)s * D + j] = qb;
    qs[0][j] = qb;
  }
  if (n_tail > 0) {
    // scores of the tail's tokens (dense rotated rows) and their histogram
    __syncthreads();
    const __half* rows = reinterpret_cast<const __half*>(p.pool + (uint64_t)p.tail_k16 * 16u) +
                         (size_t)s * p.S * D;
    for (int t = tid; t < n_tail; t += QR_THREADS) {
      const __half2* r2 = reinterpret_cast<const __half2*>(rows + (size_t)t * D);
      float acc = 0.f;
#pragma unroll 8
      for (int x = 0; x < D / 2; ++x) {
        const float2 f = __half22float2(r2[x]);
        acc = fmaf(f.x, qs[0][2 * x], acc);
        acc = fmaf(f.y, qs[0][2 * x + 1], acc);
      }
      p.scores[(size_t)s * p.Tp + p.T_packed + t] = acc;
      atomicAdd(&p.hist[(size_t)s * HIST1 + (f2key(acc) >> 20)], 1u);
    }
  }
}

// one layer (parameters by value), and several layers in one launch (layer = blockIdx.z)
__global__ void __launch_bounds__(QR_THREADS) qrot_kernel(DecodeParams p) { qrot_kernel_body(p); }
__global__ void __launch_bounds__(QR_THREADS) qrot_kernel_layers(const __grid_constant__ LayerParams lp) {
  qrot_kernel_body(lp.p[blockIdx.z]);
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
// PVB rows: the c stored values in channel order and the row's 128-bit
// channel bitmask; value i belongs to the i-th set bit.  Chunks are taken in
// order (no rotation) and the bits walked with find-first-set.
template <int CPR>
__device__ __forceinline__ float row_dot_bitmask(const uint8_t* base, int rows, int row,
                                                 const float* qsrc) {
  constexpr uint32_t C = 8u * CPR;
  const uint8_t* rowp = base + 2u * C * row;
  const uint4 mk = *reinterpret_cast<const uint4*>(base + 2u * C * (uint32_t)rows + 16u * row);
  uint32_t cur = mk.x, nxt1 = mk.y, nxt2 = mk.z, nxt3 = mk.w;
  int wbase = 0;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int k = 0; k < CPR; ++k) {
    float v[8];
    h8_to_f(*reinterpret_cast<const uint4*>(rowp + 16 * k), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      while (cur == 0u && wbase < 96) {   // at most three words to skip
        cur = nxt1;
        nxt1 = nxt2;
        nxt2 = nxt3;
        nxt3 = 0u;
        wbase += 32;
      }
      const int ch = wbase + __ffs(cur) - 1;
      cur &= cur - 1u;
      acc[e & 3] = fmaf(v[e], qsrc[ch & 127], acc[e & 3]);
    }
  }
  return (acc[0] + acc[1]) + (acc[2] + acc[3]);
}

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
    float sc;
    if constexpr (STRAT == MKV_STRATEGY_PVB) sc = row_dot_bitmask<CPR>(base, rows, row, qsrc);
    else sc = row_dot<STRAT, CPR>(base, rows, row, lane, qsrc, qm);
    st_f32_hint(out + row, sc, pol);
    atomicAdd(&hs[f2key(sc) >> 20], 1u);
  }
}

// CPR = c / 8 is a template parameter of the whole kernel (one instantiation
// per c), so the per-item dispatch is only on the segment's strategy.
template <int CPR>
__device__ __forceinline__ void score_kernel_body(const DecodeParams& p) {
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
  if (a >= b) {
    griddep_wait();
    if (p.pdl_trigger) griddep_launch();
    return;
  }
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int s_first = a / p.n_seg, s_last = (b - 1) / p.n_seg;
  const int NST = p.n_stages;
  const size_t slot_bytes = sc_slot(p.stage_bytes);
  for (int x = tid; x < SC_NSLOT * HIST1; x += SC_THREADS) (&hist[0][0])[x] = 0u;
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

  // The producer starts copying packed keys (ctx data) at once; q_bar, the
  // histograms, tickets and scores are touched only after griddep_wait, which
  // the consumers pass before their loop and the producer after its own.
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
      if ((uint64_t)(sp.line0 + sp.nlines) * 128u > p.pool_check) {
        // the stage would read past the checked pool extent: report it and
        // end the pass here (consumers see the end marker)
        if (lane == 0) {
          atomicOr(p.err, DEV_ERR_CHECK);
          meta[slot].seg0 = -1;
          mbar_arrive(&full_bar[slot]);
        }
        ++k;
        break;
      }
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
    griddep_wait();
    if (lane == 0) {
      if (!ok) atomicOr(p.err, DEV_ERR_TIMEOUT);
      sh_issued = k;
    }
    __syncwarp();   // the whole producer warp reaches the block barrier together
  } else {
    // ---- consumers ----------------------------------------------------------
    griddep_wait();
    if (warp == 0 && p.pdl_trigger) griddep_launch();
    for (int x = tid; x < SC_NSLOT * D; x += SC_CONS * 32) {
      const int s = s_first + x / D;
      (&qb[0][0])[x] = (s <= s_last) ? p.qbar[(size_t)s * D + (x % D)] : 0.f;
    }
    named_barrier_sync(1, SC_CONS * 32);
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
        if (lane == 0) atomicOr(p.err, DEV_ERR_TIMEOUT);
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
        float* out = p.scores + (size_t)s * p.Tp + seg_start(sg - s * p.n_seg, p.S, p.nseg0, p.T0);
        // the common case reads q_bar and counts into this CTA's shared copies;
        // keeping the two cases apart lets both compile to shared-memory
        // loads and atomics instead of generic ones
        auto item = [&](const float* qsrc, uint32_t* hs) {
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
          } else if (strat == MKV_STRATEGY_PVB) {
            score_block<MKV_STRATEGY_PVB, CPR>(base, rows, blk * 32, lane, qsrc, qm[warp], out, hs,
                                               pol);
          } else {
            score_block<MKV_STRATEGY_DENSE, 16>(base, rows, blk * 32, lane, qsrc, qm[warp], out,
                                                hs, pol);
          }
        };
        if (sl == 0) item(qb[0], hist[0]);
        else if (sl == 1) item(qb[1], hist[1]);
        else item(p.qbar + (size_t)s * D, p.hist + (size_t)s * HIST1);
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

// one layer (parameters by value), and several layers in one launch (layer = blockIdx.z)
template <int CPR>
__global__ void __launch_bounds__(SC_THREADS, 1) score_kernel(DecodeParams p) { score_kernel_body<CPR>(p); }
template <int CPR>
__global__ void __launch_bounds__(SC_THREADS, 1) score_kernel_layers(const __grid_constant__ LayerParams lp) {
  score_kernel_body<CPR>(lp.p[blockIdx.z]);
}

// ---------------------------------------------------------------------------
// partition of the K segments over the score kernel's CTAs (compression time
// and after each commit): CTA i starts at the first segment (in stream,
// segment order) whose cumulative size before it reaches i * total / G.
// prefix[] receives the cumulative sizes (one CTA of 1024 threads).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) partition_kernel(const mkv_segment_header* hdrK,
                                                         int n_streams, int n_seg, int c, int G,
                                                         int32_t* part, int32_t* cta_cnt,
                                                         int64_t* prefix) {
  __shared__ unsigned long long wsum[65];
  const int64_t n = (int64_t)n_streams * n_seg;
  const int tid = threadIdx.x;
  // steps of 8192 consecutive segments, thread tid taking 8 tid .. 8 tid + 7
  // of the step (coalesced loads), a block-wide exclusive scan per step and
  // a running carry
  unsigned long long carry = 0;
  for (int64_t s0 = 0; s0 < n; s0 += 8192) {
    const int64_t e0 = s0 + 8 * (int64_t)tid;
    uint32_t sz[8];
    unsigned long long mine = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      sz[u] = 0u;
      if (e0 + u < n) {
        const mkv_segment_header h = hdrK[e0 + u];
        sz[u] = segment_bytes(h.strategy, h.rows, c);
      }
      mine += sz[u];
    }
    unsigned long long tot;
    unsigned long long acc = carry + block_excl_scan64(mine, wsum, tot);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (e0 + u < n) prefix[e0 + u] = (int64_t)acc;
      acc += sz[u];
    }
    carry += tot;
  }
  if (tid == 0) prefix[n] = (int64_t)carry;
  for (int s = tid; s < n_streams; s += blockDim.x) cta_cnt[s] = 0;
  __syncthreads();
  const int64_t total = prefix[n];
  for (int i = tid; i <= G; i += blockDim.x) {
    const int64_t target = (int64_t)(((double)i / (double)G) * (double)total);
    int64_t a = 0, b = n;   // first segment whose cumulative start >= target
    while (a < b) {
      const int64_t mid = (a + b) >> 1;
      if (prefix[mid] >= target) b = mid; else a = mid + 1;
    }
    part[i] = (int32_t)(i == 0 ? 0 : (i == G ? n : a));
  }
  __syncthreads();
  for (int i = tid; i < G; i += blockDim.x) {
    const int a = part[i], b = part[i + 1];
    if (a >= b) continue;
    for (int s = a / n_seg; s <= (b - 1) / n_seg; ++s) atomicAdd(&cta_cnt[s], 1);
  }
}

// ---------------------------------------------------------------------------
// plan: the score kernel's stages for CTA i (one warp per CTA, compression
// time).  Whole segments are grouped in order while each starts where the
// previous one ends in the pool (committed segments do not), the stage's
// line-aligned span stays within stage_bytes (at least one segment per stage)
// and it holds at most SC_MAX_SEGS segments.  A stage never has more entries than its CTA
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
      if (nseg > 0 && (nseg == SC_MAX_SEGS || sj != end ||
                       ((ej + 127u) & ~127ull) - (off0 & ~127ull) > (uint64_t)stage_bytes + 128u)) {
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

cudaError_t prepare_score_kernels() {
  cudaError_t e = cudaFuncSetAttribute(qrot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, D * D * 4);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(qrot_kernel_layers, cudaFuncAttributeMaxDynamicSharedMemorySize, D * D * 4);
  if (e != cudaSuccess) return e;
#define MKV_SCORE_ATTR(N)                                                                        \
  e = cudaFuncSetAttribute(score_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize,        \
                           227 * 1024 - SC_STATIC_SMEM);                                       \
  if (e != cudaSuccess) return e;                                                               \
  e = cudaFuncSetAttribute(score_kernel_layers<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                           227 * 1024 - SC_STATIC_SMEM);                                       \
  if (e != cudaSuccess) return e;
  MKV_SCORE_ATTR(1) MKV_SCORE_ATTR(2) MKV_SCORE_ATTR(3) MKV_SCORE_ATTR(4) MKV_SCORE_ATTR(5)
  MKV_SCORE_ATTR(6) MKV_SCORE_ATTR(7) MKV_SCORE_ATTR(8) MKV_SCORE_ATTR(9) MKV_SCORE_ATTR(10)
  MKV_SCORE_ATTR(11) MKV_SCORE_ATTR(12) MKV_SCORE_ATTR(13) MKV_SCORE_ATTR(14)
  MKV_SCORE_ATTR(15) MKV_SCORE_ATTR(16)
#undef MKV_SCORE_ATTR
  return cudaSuccess;
}

cudaError_t prepare_decode_kernels() {
  cudaError_t e = prepare_score_kernels();
  if (e == cudaSuccess) e = prepare_select_kernels();
  if (e == cudaSuccess) e = prepare_attn_kernels();
  return e;
}

cudaError_t launch_partition(const mkv_segment_header* hdrK, int n_streams, int n_seg, int c,
                             int G, int stage_bytes, int32_t* part, int32_t* cta_cnt,
                             StagePlan* plan, int32_t* plan_n, int64_t* prefix, cudaStream_t st) {
  partition_kernel<<<1, 1024, 0, st>>>(hdrK, n_streams, n_seg, c, G, part, cta_cnt, prefix);
  plan_kernel<<<G, 32, 0, st>>>(hdrK, c, stage_bytes, part, plan, plan_n);
  return cudaGetLastError();
}

cudaError_t launch_qrot(const DecodeParams& p, cudaStream_t st, const LayerParams* lp, int n) {
  const bool pdl = ((p.pdl >> MKV_KERNEL_QROT) & 1) != 0;
  if (lp)
    return launch_kernel(qrot_kernel_layers, dim3(p.B * p.H, 1, n), dim3(QR_THREADS),
                         (size_t)D * D * 4, st, pdl, 0, *lp);
  return launch_kernel(qrot_kernel, dim3(p.B * p.H), dim3(QR_THREADS), (size_t)D * D * 4, st, pdl,
                       0, p);
}

cudaError_t launch_score(const DecodeParams& p, cudaStream_t st, const LayerParams* lp, int n) {
  const size_t smem = sc_slot(p.stage_bytes) * p.n_stages;
  const bool pdl = ((p.pdl >> MKV_KERNEL_SCORE) & 1) != 0;
  switch (p.c >> 3) {
#define MKV_SCORE_CASE(N)                                                                       \
  case N:                                                                                       \
    if (lp)                                                                                     \
      return launch_kernel(score_kernel_layers<N>, dim3(p.G, 1, n), dim3(SC_THREADS), smem, st, \
                           pdl, 0, *lp);                                                        \
    return launch_kernel(score_kernel<N>, dim3(p.G), dim3(SC_THREADS), smem, st, pdl, 0, p);
    MKV_SCORE_CASE(1) MKV_SCORE_CASE(2) MKV_SCORE_CASE(3) MKV_SCORE_CASE(4) MKV_SCORE_CASE(5)
    MKV_SCORE_CASE(6) MKV_SCORE_CASE(7) MKV_SCORE_CASE(8) MKV_SCORE_CASE(9) MKV_SCORE_CASE(10)
    MKV_SCORE_CASE(11) MKV_SCORE_CASE(12) MKV_SCORE_CASE(13) MKV_SCORE_CASE(14)
    MKV_SCORE_CASE(15) MKV_SCORE_CASE(16)
#undef MKV_SCORE_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mkv
