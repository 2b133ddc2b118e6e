// Decode-time appends and the commit of full segments.
//
// MosaicKV (arXiv 2607.00760), §1 Introduction, "Observation & Method 2":
// newly generated KV are kept in a GPU-side buffer and used by later decode
// steps; once a segment's worth has accumulated it is compressed and swapped
// into the compressed cache without blocking decode.  Here the buffer (the
// tail) holds each new token twice: rotated into the stream's existing basis
// as an fp16 dense row inside the pool (read by the score and attention
// kernels like any dense row), and as given (fp16) for the commit, which
// compresses the S buffered tokens with the compression kernels and the
// stream's basis, exactly as the prefill would compress them.
#include "mkv_internal.cuh"

namespace mkv {

// ---------------------------------------------------------------------------
// append: x~ = x R for n new tokens of one (stream, K|V); R staged in shared
// memory, thread j computes channel j (fixed summation order).
// grid: (BH, 2), block 128, dynamic smem 64 KB
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) append_kernel(AppendParams a) {
  extern __shared__ __align__(16) float Rs[];   // [128][128]
  __shared__ float xs[D];
  const int s = blockIdx.x, x = blockIdx.y, j = threadIdx.x;
  const float4* R4 = reinterpret_cast<const float4*>(a.R + ((size_t)x * a.BH + s) * D * D);
  for (int e = j; e < D * D / 4; e += blockDim.x) reinterpret_cast<float4*>(Rs)[e] = R4[e];
  const __half* src = (x == 0 ? a.k : a.v) + (size_t)s * a.n_total * D;
  __half* rot = reinterpret_cast<__half*>(a.pool + (x == 0 ? a.tail_k : a.tail_v)) +
                (size_t)s * a.S * D;
  __half* orig = a.tail_x + ((size_t)x * a.BH + s) * a.S * D;
  for (int t = 0; t < a.n; ++t) {
    __syncthreads();                               // R staged / xs free for the next token
    const __half h = src[(size_t)(a.first + t) * D + j];
    xs[j] = __half2float(h);
    orig[(size_t)(a.tail_len + t) * D + j] = h;
    __syncthreads();
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc = fmaf(xs[i], Rs[i * D + j], acc);
    rot[(size_t)(a.tail_len + t) * D + j] = __float2half_rn(acc);
  }
}

cudaError_t launch_append(const AppendParams& a, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(append_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       D * D * 4);
  if (e != cudaSuccess) return e;
  append_kernel<<<dim3(a.BH, 2), 128, D * D * 4, st>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// commit scan: headers of the one new segment of every stream (K streams,
// then V streams), placed one after another from *packed_end; *packed_end
// then moves past them.  One CTA.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) commit_scan_kernel(CompressParams p) {
  __shared__ unsigned long long ws[32];
  const int64_t n = (int64_t)2 * p.BH * p.n_seg;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per = (n + 1023) / 1024;
  const int64_t lo = imin64(n, tid * per), hi = imin64(n, lo + per);
  const unsigned long long base = *p.packed_end;
  unsigned long long mine = 0;
  for (int64_t e = lo; e < hi; ++e) mine += p.seg[e].size;
  unsigned long long inc = mine;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  unsigned long long off = base + inc - mine;
  for (int w = 0; w < warp; ++w) off += ws[w];
  for (int64_t e = lo; e < hi; ++e) {
    const SegInfo si = p.seg[e];
    mkv_segment_header h;
    h.off16 = (uint32_t)(off >> 4);
    h.strategy = si.strategy;
    h.reserved = 0;
    h.rows = si.rows;
    p.hdr[e] = h;
    off += si.size;
  }
  __syncthreads();
  if (tid == 1023) *p.packed_end = off;
}

cudaError_t launch_commit_scan(const CompressParams& p, cudaStream_t st) {
  commit_scan_kernel<<<1, 1024, 0, st>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// grow headers: out[x_s][j] = old[x_s][j] for j < n_old, seg_new[x_s] at
// j = n_old, for the 2 BH streams x_s.
// ---------------------------------------------------------------------------
__global__ void grow_headers_kernel(const mkv_segment_header* old, int n_old,
                                    const mkv_segment_header* seg_new, int n_streams2,
                                    mkv_segment_header* out) {
  const int64_t n = (int64_t)n_streams2 * (n_old + 1);
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t xs = e / (n_old + 1);
    const int j = (int)(e - xs * (n_old + 1));
    out[e] = j < n_old ? old[xs * n_old + j] : seg_new[xs];
  }
}

cudaError_t launch_grow_headers(const mkv_segment_header* old, int n_old,
                                const mkv_segment_header* seg_new, int n_streams2,
                                mkv_segment_header* out, cudaStream_t st) {
  const int64_t n = (int64_t)n_streams2 * (n_old + 1);
  const int blocks = (int)imin64((n + 255) / 256, 4096);
  grow_headers_kernel<<<blocks, 256, 0, st>>>(old, n_old, seg_new, n_streams2, out);
  return cudaGetLastError();
}

}  // namespace mkv
