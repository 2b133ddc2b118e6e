// Decode step, last part: attention over the selected tokens, read in place
// from the packed cache, and the output rotation back to the original basis.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction, "Observation & Method 2":
// attention computed on the packed dense format without unpacking.
#include "decode_common.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// attn: persistent split-K attention.  The selected tokens of all streams,
// flattened in (stream, position) order, are cut into equal slices of
// attn_per positions, one slice per CTA.  A CTA walks its slice in chunks of
// up to 64 tokens that never cross a stream boundary (chunk = the 64-position
// blocks of a stream, clipped to the slice).  Per chunk:
//   issue   (stages - 1 chunks ahead) every lane of the token's 8-lane group
//           reads the token id and its K and V segment headers, and copies
//           its pieces of the two packed rows (16-byte value chunks, 8-byte
//           channel lists) into the chunk's stage slot with cp.async;
//   A       8 lanes per token: partial logits q~_i . k^_t over the lane's
//           stored values (q~ indexed by the stored channel), summed over the
//           group by a fixed butterfly; V values scattered into a zeroed fp16
//           tile V[token][channel];
//   B       per head (one warp each): online softmax over the CTA's tokens of
//           the stream so far (running max m, sum l, factor alpha for the
//           earlier output); weights split into fp16 hi + 2^11 * lo parts;
//   C       per warp (8 output channels): o~ <- alpha o~ + P V on tensor cores
//           (mma.sync, fp32 accumulation, one accumulator per part), then the
//           warp clears its columns of the V tile.
// At the end of its part of a stream the CTA writes one partial (m, l, o~ in
// the rotated V basis); the merge kernel combines the partials of a stream.
// Every sum has a fixed order, so the output is bit-for-bit repeatable.
// grid: ceil(B H k / attn_per), block 512, dynamic smem at_smem_bytes()
// ---------------------------------------------------------------------------
constexpr int AT_THREADS = 512;
constexpr int AT_CHUNK = 64;        // tokens per chunk: 8 lanes each
constexpr int AT_VLD = 136;         // halves per V tile row (272 B: ldmatrix without conflicts)
constexpr int AT_PLD = 72;          // halves per P row (144 B)

constexpr int32_t NO_IDX = (int32_t)0x80000000;
// channel-list field of a PVB row: this flag plus the distance / 8 to the
// row's 16-byte bitmask (SM distances are negative, PV ones below 2^28)
constexpr uint32_t PVB_FLAG = 0x10000000u;

__device__ __forceinline__ bool is_pvb(uint32_t y) { return (int32_t)y > 0 && (y & PVB_FLAG); }
// byte distance from a row's values to its channel list (SM, PV, PVB rows)
__device__ __forceinline__ int64_t list_dist(uint32_t y) {
  return 8 * (int64_t)(is_pvb(y) ? (int32_t)(y & ~PVB_FLAG) : (int32_t)y);
}

// Row of token t in stream s: pool offset of its stored values / 16, and the
// byte distance / 8 from the values to the row's channel list (the segment
// mask for SM, the row's own indices for PV; NO_IDX for dense rows).  Tokens
// before T0 sit in the prefill segments, tokens from T0 to T_packed in the
// committed ones, later tokens in the tail (dense rows at tail16).
__device__ __forceinline__ uint2 row_meta(const DecodeParams& p, const mkv_segment_header* hdr,
                                          int s, int64_t t, uint32_t tail16) {
  const int S = p.S, c = p.c;
  if (t >= p.T_packed)
    return make_uint2(tail16 + (uint32_t)(((int64_t)s * S + (t - p.T_packed)) * 16), (uint32_t)NO_IDX);
  // t < T <= 2^31 - 1: 32-bit division
  uint32_t sg, r;
  if (t < p.T0) {
    sg = (uint32_t)t / (uint32_t)S;
    r = (uint32_t)t - sg * (uint32_t)S;
  } else {
    const uint32_t u = (uint32_t)(t - p.T0), q = u / (uint32_t)S;
    sg = (uint32_t)p.nseg0 + q;
    r = u - q * (uint32_t)S;
  }
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
  if (hd.strategy == MKV_STRATEGY_PVB) {
    const uint32_t dv = c2 * r;
    return make_uint2(hd.off16 + dv / 16u, PVB_FLAG | ((c2 * (hd.rows - r) + 16u * r) / 8u));
  }
  return make_uint2(hd.off16 + 16u * r, (uint32_t)NO_IDX);
}

// One past the last pool byte that the row (values and channel list) spans.
__device__ __forceinline__ uint64_t row_end(const uint2& m, int c) {
  const uint64_t v0 = (uint64_t)m.x * 16u;
  if ((int32_t)m.y == NO_IDX) return v0 + 256u;
  const uint64_t vend = v0 + 2u * (uint32_t)c;
  const uint64_t iend = (uint64_t)((int64_t)v0 + list_dist(m.y)) + (is_pvb(m.y) ? 16u : (uint32_t)c);
  return vend > iend ? vend : iend;
}

// Slot of channel ch in the staged q~ table.  The lanes of a token read
// channels that lie about 8 values apart in a sorted channel list, so their
// high bits differ; placing channel ch at slot 16 (ch mod 8) + ch / 8 puts the
// 16-byte entries (g <= 4) of such channels in different bank groups.
__device__ __forceinline__ int q_slot(int ch) { return ((ch & 7) << 4) | (ch >> 3); }

__device__ __forceinline__ int chan_of(const uint2& x, int e) {
  return (int)(((e < 4 ? x.x : x.y) >> (8 * (e & 3))) & 0x7fu);
}

// Shared-memory carve-up of the attention kernel (byte offsets).
struct AtLayout {
  uint32_t stages, vt, ph, pl, qs, lg, meta, total;
};

// Row addresses resolved per pass (positions of the CTA's slice).
constexpr int AT_META = 1024;

__host__ __device__ inline AtLayout at_layout(int g, int slot, int nst) {
  const int gp = (g + 3) & ~3;
  AtLayout L;
  L.stages = 0;
  L.vt = L.stages + (uint32_t)nst * AT_CHUNK * slot;
  L.ph = L.vt + AT_CHUNK * AT_VLD * 2;
  L.pl = L.ph + MAX_G * AT_PLD * 2;
  L.qs = L.pl + MAX_G * AT_PLD * 2;
  L.lg = L.qs + D * gp * 4;
  L.meta = L.lg + AT_CHUNK * gp * 4;
  L.total = L.meta + AT_META * 16;
  return L;
}

size_t at_smem_bytes(int g, int slot, int nst) { return at_layout(g, slot, nst).total; }

// Chunks of a pass: the 64-position blocks of each stream's selection,
// clipped to the pass [lo, hi) of a slice that ends at slice_hi, walked in
// order without divisions (one per pass, in at_begin).
struct AtChunk {
  int s;        // stream
  int j0;       // first position within the stream's selection
  int n;        // tokens
  bool last;    // the slice's last chunk of this stream
};

// Position coordinates relative to the pass start (pass length <= AT_META).
struct AtIter {
  int rel;         // s * kk - pass start
  int s;
  int b;           // block within the stream
};

__device__ __forceinline__ AtIter at_begin(int kk, int64_t lo) {
  AtIter it;
  it.s = (int)(lo / kk);
  it.rel = (int)((int64_t)it.s * kk - lo);
  it.b = -it.rel / AT_CHUNK;
  return it;
}

__device__ __forceinline__ void at_advance(AtIter& it, int kk) {
  if (AT_CHUNK * (it.b + 1) >= kk) {
    ++it.s;
    it.rel += kk;
    it.b = 0;
  } else {
    ++it.b;
  }
}

// n_pass: positions in the pass; slice_end: the slice's end relative to the
// pass start (clamped to the int range)
__device__ __forceinline__ bool at_get(const AtIter& it, int kk, int n_pass, int slice_end,
                                       AtChunk& c) {
  const int start = it.rel + AT_CHUNK * it.b;
  const int bend = AT_CHUNK * it.b + AT_CHUNK;
  const bool stream_end = bend >= kk;
  const int end = it.rel + (stream_end ? kk : bend);
  const int a = start > 0 ? start : 0;
  const int e = end < n_pass ? end : n_pass;
  if (a >= e) return false;
  c.s = it.s;
  c.j0 = a - it.rel;
  c.n = e - a;
  c.last = (e == slice_end) || (e == end && stream_end);
  return true;
}

// Resolves the rows of positions [lo, hi) (at most AT_META) into meta[]:
// token id -> K and V segment headers -> (value offset, channel-list
// distance) of each row.  Four positions per thread are loaded together.
__device__ __forceinline__ void at_meta_pass(const DecodeParams& p, int64_t lo, int64_t hi,
                                             uint4* meta) {
  const int n = (int)(hi - lo);
  // stream of position lo + x: s0 + (r0 + x) / kk, with r0 + x < kk + AT_META
  const int s0 = (int)(lo / p.kk);
  const uint32_t r0 = (uint32_t)(lo - (int64_t)s0 * p.kk);
  for (int x0 = threadIdx.x; x0 < n; x0 += 4 * AT_THREADS) {
    int64_t t[4];
    int sidx[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * AT_THREADS;
      sidx[u] = 0;
      t[u] = 0;
      if (x < n) {
        sidx[u] = s0 + (int)((r0 + (uint32_t)x) / (uint32_t)p.kk);
        t[u] = p.sel[lo + x];
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int x = x0 + u * AT_THREADS;
      if (x < n) {
        const int64_t tt = clamp_t((int32_t)t[u], p.T);
        uint2 km = row_meta(p, p.hdrK + (size_t)sidx[u] * p.n_seg, sidx[u], tt, p.tail_k16);
        uint2 vm = row_meta(p, p.hdrV + (size_t)sidx[u] * p.n_seg, sidx[u], tt, p.tail_v16);
        if (row_end(km, p.c) > p.pool_check || row_end(vm, p.c) > p.pool_check) {
          // outside the checked pool extent: report it and read a stand-in
          // row of c values with its channel list at pool offset 0 (inside
          // every pool, and the size of a non-dense slot)
          atomicOr(p.err, DEV_ERR_CHECK);
          km = vm = make_uint2(0u, 0u);
        }
        meta[x] = make_uint4(km.x, km.y, vm.x, vm.y);
      }
    }
  }
}

// Issues the copies of chunk ch into stage `st` (rel_s: the chunk stream's
// start relative to the pass): token tid / 8, lane tid % 8; rows from the
// pass's meta[].
__device__ __forceinline__ void at_issue(const DecodeParams& p, int rel_s, const AtChunk& ch,
                                         int st, uint8_t* smem, const AtLayout& L) {
  const int i = threadIdx.x >> 3, cl = threadIdx.x & 7;
  if (i >= ch.n) return;
  const int c = p.c;
  const uint4 m = reinterpret_cast<const uint4*>(smem + L.meta)[ch.j0 + i + rel_s];
  const uint32_t slot = smem_u32(smem + L.stages) + (uint32_t)((st * AT_CHUNK + i) * p.at_slot);
  const bool kd = (int32_t)m.y == NO_IDX, vd = (int32_t)m.w == NO_IDX;
  const int kn = kd ? D : c, vn = vd ? D : c;
  const uint8_t* kv = p.pool + (uint64_t)m.x * 16u;
  const uint8_t* vv = p.pool + (uint64_t)m.z * 16u;
  const uint32_t vs = slot + p.at_kv + p.at_ki;
  const bool kb = is_pvb(m.y), vb = is_pvb(m.w);
#pragma unroll
  for (int ck = cl; ck < 16; ck += 8) {
    if (8 * ck < kn) {
      cpa16(slot + 16 * ck, kv + 16 * ck);
      if (!kd && !kb) cpa8(slot + p.at_kv + 8 * ck, kv + list_dist(m.y) + 8 * ck);
    }
    if (8 * ck < vn) {
      cpa16(vs + 16 * ck, vv + 16 * ck);
      if (!vd && !vb) cpa8(vs + p.at_vv + 8 * ck, vv + list_dist(m.w) + 8 * ck);
    }
  }
  // PVB rows: the 16-byte bitmask in place of the channel list
  if (cl == 0 && kb) cpa16(slot + p.at_kv, kv + list_dist(m.y));
  if (cl == 0 && vb) cpa16(vs + p.at_vv, vv + list_dist(m.w));
}

template <int NST>
__device__ __forceinline__ void attn_kernel_body(const DecodeParams& p) {
  extern __shared__ __align__(128) uint8_t at_smem[];
  __shared__ float s_m[MAX_G], s_l[MAX_G], s_alpha[MAX_G];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok = tid >> 3, cl = tid & 7;
  const int g = p.g, gp = (g + 3) & ~3, c = p.c;
  const AtLayout L = at_layout(g, p.at_slot, NST);
  __half* Vt = reinterpret_cast<__half*>(at_smem + L.vt);
  __half* Ph = reinterpret_cast<__half*>(at_smem + L.ph);
  __half* Pl = reinterpret_cast<__half*>(at_smem + L.pl);
  float* qs = reinterpret_cast<float*>(at_smem + L.qs);
  float* lg = reinterpret_cast<float*>(at_smem + L.lg);
  uint4* meta = reinterpret_cast<uint4*>(at_smem + L.meta);
  const int64_t N = (int64_t)p.B * p.H * p.kk;
  const int64_t lo = (int64_t)blockIdx.x * p.attn_per;
  const int64_t hi = lo + p.attn_per < N ? lo + p.attn_per : N;

  // prologue (shared memory only): zero the V tile and both P parts
  {
    uint4* z = reinterpret_cast<uint4*>(at_smem + L.vt);
    const int nz = (int)((L.qs - L.vt) / 16);
    for (int x = tid; x < nz; x += AT_THREADS) z[x] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < MAX_G) {
      s_m[tid] = -INFINITY;
      s_l[tid] = 0.f;
    }
  }
  griddep_wait();     // the selection comes from the kernel before this one
  if (p.pdl_trigger) griddep_launch();
  if (lo >= N) return;
  const float scale = 0.08838834764831845f;     // 1 / sqrt(128)
  const int mm = lane >> 3, r8 = lane & 7;
  const int n0 = warp * 8;                       // this warp's output channels in phase C
  float acc_h[4] = {0.f, 0.f, 0.f, 0.f}, acc_l[4] = {0.f, 0.f, 0.f, 0.f};
  int cur_s = -1;
  // passes of at most AT_META positions: resolve their rows, then stream them
  for (int64_t pa = lo; pa < hi; pa += AT_META) {
    const int64_t pb = pa + AT_META < hi ? pa + AT_META : hi;
    if (pa != lo) cpa_wait<0>();
    __syncthreads();                     // the previous pass no longer reads meta[]
    at_meta_pass(p, pa, pb, meta);
    __syncthreads();
    const int n_pass = (int)(pb - pa);
    const int slice_end = (int)(hi - pa < 0x7fffffff ? hi - pa : 0x7fffffff);
    AtIter cit = at_begin(p.kk, pa);     // the chunk being computed
    AtIter iit = cit;                     // the chunk being issued
#pragma unroll
    for (int n = 0; n < NST - 1; ++n) {
      AtChunk ich;
      if (at_get(iit, p.kk, n_pass, slice_end, ich)) at_issue(p, iit.rel, ich, n, at_smem, L);
      at_advance(iit, p.kk);
      cpa_commit();
    }
    for (int n = 0;; ++n) {
      AtChunk ch;
      if (!at_get(cit, p.kk, n_pass, slice_end, ch)) break;
      const int x0 = cit.rel + ch.j0;        // the chunk's first meta[] index
      at_advance(cit, p.kk);
      {
        AtChunk ich;
        if (at_get(iit, p.kk, n_pass, slice_end, ich))
          at_issue(p, iit.rel, ich, (n + NST - 1) % NST, at_smem, L);
        at_advance(iit, p.kk);
      }
      cpa_commit();
      cpa_wait<NST - 1>();
      __syncthreads();
      const int st = n % NST;
        if (ch.s != cur_s) {
        cur_s = ch.s;
        const int b = ch.s / p.H, h = ch.s % p.H;
        const float* qt = p.qt + ((size_t)b * p.Hq + (size_t)h * g) * D;
        for (int x = tid; x < D * gp; x += AT_THREADS) {
          const int chn = x / gp, hh = x % gp;
          qs[q_slot(chn) * gp + hh] = hh < g ? qt[hh * D + chn] : 0.f;
        }
        __syncthreads();
      }
      // ---- A: logits and the V tile --------------------------------------------
      {
        const bool valid = tok < ch.n;
        const uint4 mt = valid ? meta[x0 + tok] : make_uint4(0u, 0u, 0u, 0u);
        const uint8_t* slot = at_smem + L.stages + (size_t)(st * AT_CHUNK + tok) * p.at_slot;
        const bool kd = (int32_t)mt.y == NO_IDX, vd = (int32_t)mt.w == NO_IDX;
        const bool kb = valid && is_pvb(mt.y), vb = valid && is_pvb(mt.w);
        const int kn = valid && !kb ? (kd ? D : c) : 0, vn = valid && !vb ? (vd ? D : c) : 0;
        const uint8_t* vs = slot + p.at_kv + p.at_ki;
        // PVB rows: lane cl owns channels [16 cl, 16 cl + 16) of the bitmask;
        // its values follow those of the group's lower lanes (prefix count,
        // taken by every lane of a warp that holds a PVB row, so that the
        // shuffles stay warp-uniform)
        uint32_t kbits = 0u, vbits = 0u;
        int kpre = 0, vpre = 0;
        if (__any_sync(0xffffffffu, kb || vb)) {
          if (kb) kbits = (*reinterpret_cast<const uint32_t*>(slot + p.at_kv + 4 * (cl >> 1)) >>
                           (16 * (cl & 1))) & 0xffffu;
          if (vb) vbits = (*reinterpret_cast<const uint32_t*>(vs + p.at_vv + 4 * (cl >> 1)) >>
                           (16 * (cl & 1))) & 0xffffu;
          kpre = __popc(kbits);
          vpre = __popc(vbits);
          int ki = kpre, vi = vpre;
#pragma unroll
          for (int off = 1; off < 8; off <<= 1) {
            const int ky = __shfl_up_sync(0xffffffffu, ki, off, 8);
            const int vy = __shfl_up_sync(0xffffffffu, vi, off, 8);
            if (cl >= off) {
              ki += ky;
              vi += vy;
            }
          }
          kpre = ki - kpre;
          vpre = vi - vpre;
        }
        for (int h4 = 0; h4 < gp; h4 += 4) {
          float part[4] = {0.f, 0.f, 0.f, 0.f};
          {
            uint32_t b = kbits;
            int i = kpre;
            while (b) {
              const int chn = 16 * cl + __ffs(b) - 1;
              b &= b - 1u;
              const float v = __half2float(*reinterpret_cast<const __half*>(slot + 2 * i));
              ++i;
              const float4 q4 = *reinterpret_cast<const float4*>(qs + q_slot(chn) * gp + h4);
              part[0] = fmaf(q4.x, v, part[0]);
              part[1] = fmaf(q4.y, v, part[1]);
              part[2] = fmaf(q4.z, v, part[2]);
              part[3] = fmaf(q4.w, v, part[3]);
            }
          }
  #pragma unroll
          for (int ck = cl; ck < 16; ck += 8) {
            if (8 * ck < kn) {
              const uint4 kr = *reinterpret_cast<const uint4*>(slot + 16 * ck);
              const uint2 kx = kd ? make_uint2(0u, 0u)
                                  : *reinterpret_cast<const uint2*>(slot + p.at_kv + 8 * ck);
              float v[8];
              h8_to_f(kr, v);
  #pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int chn = kd ? 8 * ck + e : chan_of(kx, e);
                const float4 q4 = *reinterpret_cast<const float4*>(qs + q_slot(chn) * gp + h4);
                part[0] = fmaf(q4.x, v[e], part[0]);
                part[1] = fmaf(q4.y, v[e], part[1]);
                part[2] = fmaf(q4.z, v[e], part[2]);
                part[3] = fmaf(q4.w, v[e], part[3]);
              }
            }
          }
  #pragma unroll
          for (int k = 0; k < 4; ++k) {
            float x = part[k];
            x += __shfl_xor_sync(0xffffffffu, x, 1);
            x += __shfl_xor_sync(0xffffffffu, x, 2);
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            part[k] = x;
          }
          if (valid && cl == 0)
            *reinterpret_cast<float4*>(lg + tok * gp + h4) =
                make_float4(part[0] * scale, part[1] * scale, part[2] * scale, part[3] * scale);
        }
        {
          uint32_t b = vbits;
          int i = vpre;
          __half* vrow = Vt + tok * AT_VLD;
          while (b) {
            const int chn = 16 * cl + __ffs(b) - 1;
            b &= b - 1u;
            vrow[chn] = *reinterpret_cast<const __half*>(vs + 2 * i);
            ++i;
          }
        }
  #pragma unroll
        for (int ck = cl; ck < 16; ck += 8) {
          if (8 * ck < vn) {
            const uint4 vr = *reinterpret_cast<const uint4*>(vs + 16 * ck);
            const uint2 vx = vd ? make_uint2(0u, 0u)
                                : *reinterpret_cast<const uint2*>(vs + p.at_vv + 8 * ck);
            const __half* hv = reinterpret_cast<const __half*>(&vr);
            __half* vrow = Vt + tok * AT_VLD;
  #pragma unroll
            for (int e = 0; e < 8; ++e) vrow[vd ? 8 * ck + e : chan_of(vx, e)] = hv[e];
          }
        }
      }
      __syncthreads();
      // ---- B: online softmax, one warp per head ----------------------------------
      if (warp < g) {
        const int hh = warp;
        float mloc = -INFINITY;
        for (int i = lane; i < ch.n; i += 32) mloc = fmaxf(mloc, lg[i * gp + hh]);
  #pragma unroll
        for (int off = 16; off > 0; off >>= 1)
          mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
        const float m_old = s_m[hh];
        const float m_new = fmaxf(m_old, mloc);
        const float alpha = expf(m_old - m_new);
        float lsum = 0.f;
        for (int i = lane; i < AT_CHUNK; i += 32) {
          const float e = i < ch.n ? expf(lg[i * gp + hh] - m_new) : 0.f;
          const __half hi = __float2half_rn(e);
          Ph[hh * AT_PLD + i] = hi;
          Pl[hh * AT_PLD + i] = __float2half_rn((e - __half2float(hi)) * 2048.f);
          lsum += e;
        }
  #pragma unroll
        for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
        if (lane == 0) {
          s_alpha[hh] = alpha;
          s_m[hh] = m_new;
          s_l[hh] = fmaf(s_l[hh], alpha, lsum);
        }
      }
      __syncthreads();
      // ---- C: o~ <- alpha o~ + P V, warp w owns channels [8w, 8w + 8) -------------
      {
        const int r0 = lane >> 2;
        const float a0 = r0 < g ? s_alpha[r0] : 1.f;
        const float a1 = r0 + 8 < g ? s_alpha[r0 + 8] : 1.f;
        acc_h[0] *= a0;
        acc_h[1] *= a0;
        acc_h[2] *= a1;
        acc_h[3] *= a1;
        acc_l[0] *= a0;
        acc_l[1] *= a0;
        acc_l[2] *= a1;
        acc_l[3] *= a1;
        const uint32_t ph = smem_u32(Ph), pl = smem_u32(Pl), vt = smem_u32(Vt);
        const int ksteps = (ch.n + 15) >> 4;
        for (int ks = 0; ks < ksteps; ++ks) {
          const int k0 = ks * 16;
          uint32_t ah[4], al[4], bb[2];
          const uint32_t aoff = (uint32_t)(((r8 + (mm & 1) * 8) * AT_PLD + k0 + (mm >> 1) * 8) * 2);
          ldsm_x4(ph + aoff, ah);
          ldsm_x4(pl + aoff, al);
          ldsm_x2_t(vt + (uint32_t)(((k0 + (lane & 15)) * AT_VLD + n0) * 2), bb);
          mma16816(acc_h, ah, bb[0], bb[1]);
          mma16816(acc_l, al, bb[0], bb[1]);
        }
        // clear this warp's columns of the V tile for the next chunk
        *reinterpret_cast<uint4*>(Vt + lane * AT_VLD + n0) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(Vt + (lane + 32) * AT_VLD + n0) = make_uint4(0u, 0u, 0u, 0u);
        if (ch.last) {
          // the slice's part of this stream is done: write its partial
          const int first = (int)(((int64_t)ch.s * p.kk) / p.attn_per);
          const size_t pbase = ((size_t)ch.s * p.attn_mp + (blockIdx.x - first)) * g;
          const int col = n0 + 2 * (lane & 3);
          if (r0 < g)
            *reinterpret_cast<float2*>(p.part_o + (pbase + r0) * D + col) =
                make_float2(fmaf(acc_l[0], 1.f / 2048.f, acc_h[0]),
                            fmaf(acc_l[1], 1.f / 2048.f, acc_h[1]));
          if (r0 + 8 < g)
            *reinterpret_cast<float2*>(p.part_o + (pbase + r0 + 8) * D + col) =
                make_float2(fmaf(acc_l[2], 1.f / 2048.f, acc_h[2]),
                            fmaf(acc_l[3], 1.f / 2048.f, acc_h[3]));
  #pragma unroll
          for (int e = 0; e < 4; ++e) acc_h[e] = acc_l[e] = 0.f;
          if (warp < g && lane == 0) {
            p.part_ml[(pbase + warp) * 2] = s_m[warp];
            p.part_ml[(pbase + warp) * 2 + 1] = s_l[warp];
            s_m[warp] = -INFINITY;
            s_l[warp] = 0.f;
          }
        }
      }
    }
  }
  cpa_wait<0>();
}

// one layer (parameters by value), and several layers in one launch (layer = blockIdx.z)
template <int NST>
__global__ void __launch_bounds__(AT_THREADS, 2) attn_kernel(DecodeParams p) { attn_kernel_body<NST>(p); }
template <int NST>
__global__ void __launch_bounds__(AT_THREADS, 2) attn_kernel_layers(const __grid_constant__ LayerParams lp) {
  attn_kernel_body<NST>(lp.p[blockIdx.z]);
}

// Slices that cover stream s's selection: the first one and how many.
__device__ __forceinline__ int at_first_part(const DecodeParams& p, int s) {
  return (int)(((int64_t)s * p.kk) / p.attn_per);
}
__device__ __forceinline__ int at_num_parts(const DecodeParams& p, int s) {
  return (int)((((int64_t)s + 1) * p.kk - 1) / p.attn_per) - at_first_part(p, s) + 1;
}

// ---------------------------------------------------------------------------
// merge: log-sum-exp merge of a stream's partials, then o = o~ R_V^T.  CTA
// (s, q) writes output rows [32q, 32q + 32) of every head of stream s; the
// weights and the merged o~ are recomputed by each of the four CTAs (from
// L2), and the 32 rows of R_V are staged transposed in shared memory.
// grid: (BH, 4), block 128, dynamic smem: partial weights
// ---------------------------------------------------------------------------
constexpr int MG_THREADS = 128;
constexpr int MG_ROWS = 32;
constexpr int MG_LD = MG_ROWS + 1;

__device__ __forceinline__ void merge_kernel_body(const DecodeParams& p) {
  extern __shared__ __align__(16) float wsm[];     // [parts][g] weights
  __shared__ float Rt[D * MG_LD];                  // Rt[j][rr] = R_V[32q + rr][j]
  __shared__ __align__(16) float ot[MAX_G][D];
  __shared__ float Linv[MAX_G];
  const int s = blockIdx.x, r0 = blockIdx.y * MG_ROWS;
  const int b = s / p.H, h = s % p.H;
  const int g = p.g;
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
  if (p.pdl_trigger) griddep_launch();
  const int nc = at_num_parts(p, s);
  const size_t base = (size_t)s * p.attn_mp * g;
  // weights exp(m_c - M) and 1 / L per head: warp per head, lanes over parts
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + base;
  for (int hh = warp; hh < g; hh += MG_THREADS / 32) {
    float M = -INFINITY;
    for (int c = lane; c < nc; c += 32) M = fmaxf(M, __ldcg(ml + c * g + hh).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    for (int c = lane; c < nc; c += 32) {
      const float2 v = __ldcg(ml + c * g + hh);
      const float w = expf(v.x - M);
      wsm[c * g + hh] = w;
      L = fmaf(v.y, w, L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) Linv[hh] = 1.f / L;
  }
  __syncthreads();
  const float* po = p.part_o + base * D;
  for (int x = tid; x < g * D; x += MG_THREADS) {
    const int hh = x / D;
    float o = 0.f;
    for (int c = 0; c < nc; ++c) o = fmaf(__ldcg(po + (size_t)c * g * D + x), wsm[c * g + hh], o);
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

// one layer (parameters by value), and several layers in one launch (layer = blockIdx.z)
__global__ void __launch_bounds__(MG_THREADS) merge_kernel(DecodeParams p) { merge_kernel_body(p); }
__global__ void __launch_bounds__(MG_THREADS) merge_kernel_layers(const __grid_constant__ LayerParams lp) {
  merge_kernel_body(lp.p[blockIdx.z]);
}

cudaError_t attn_shape(int g, int slot, int* stages, int* ctas_per_sm) {
  // four stages when two CTAs still fit an SM, else fewer
  int nst = 2;
  for (int n = 4; n > 2; --n)
    if (at_smem_bytes(g, slot, n) <= 113 * 1024) {
      nst = n;
      break;
    }
  const size_t smem = at_smem_bytes(g, slot, nst);
  if (smem > at_smem_bytes(MAX_G, 768, 2)) return cudaErrorInvalidValue;
  int occ = 0;
  cudaError_t e;
  if (nst == 4) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<4>, AT_THREADS, smem);
  else if (nst == 3) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<3>, AT_THREADS, smem);
  else e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_kernel<2>, AT_THREADS, smem);
  if (e != cudaSuccess) return e;
  *stages = nst;
  *ctas_per_sm = occ > 0 ? occ : 1;
  return cudaSuccess;
}

cudaError_t prepare_attn_kernels() {
  // the largest carve-up attn_shape can choose: two stages of dense rows
  // (256 + 128 bytes of K and of V per token) and 16 heads
  const int mx = (int)at_smem_bytes(MAX_G, 768, 2);
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<2>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<3>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel<4>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel_layers<2>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel_layers<3>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_kernel_layers<4>, a, mx);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(merge_kernel_layers, a, 48 * 1024 + 4 * 1024);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(merge_kernel, a, 48 * 1024 + 4 * 1024);
}

cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st, const LayerParams* lp, int n) {
  const size_t smem = at_smem_bytes(p.g, p.at_slot, p.at_stages);
  const dim3 grid(p.attn_ctas, 1, n), block(AT_THREADS);
  const bool pdl = ((p.pdl >> MKV_KERNEL_ATTN) & 1) != 0;
  if (lp) {
    if (p.at_stages >= 4) return launch_kernel(attn_kernel_layers<4>, grid, block, smem, st, pdl, 0, *lp);
    if (p.at_stages == 3) return launch_kernel(attn_kernel_layers<3>, grid, block, smem, st, pdl, 0, *lp);
    return launch_kernel(attn_kernel_layers<2>, grid, block, smem, st, pdl, 0, *lp);
  }
  if (p.at_stages >= 4) return launch_kernel(attn_kernel<4>, grid, block, smem, st, pdl, 0, p);
  if (p.at_stages == 3) return launch_kernel(attn_kernel<3>, grid, block, smem, st, pdl, 0, p);
  return launch_kernel(attn_kernel<2>, grid, block, smem, st, pdl, 0, p);
}

cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st, const LayerParams* lp, int n) {
  const dim3 grid(p.B * p.H, D / MG_ROWS, n);
  const size_t smem = sizeof(float) * (size_t)p.attn_mp * p.g;
  const bool pdl = ((p.pdl >> MKV_KERNEL_MERGE) & 1) != 0;
  if (lp) return launch_kernel(merge_kernel_layers, grid, dim3(MG_THREADS), smem, st, pdl, 0, *lp);
  return launch_kernel(merge_kernel, grid, dim3(MG_THREADS), smem, st, pdl, 0, p);
}

}  // namespace mkv
