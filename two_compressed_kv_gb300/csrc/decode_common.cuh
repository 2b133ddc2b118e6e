// Device helpers shared by the decode-step kernels (score, select, attention):
// order-preserving float keys, fp16 unpacking and the radix bin search.
#pragma once

#include "mkv_internal.cuh"
#include "ptx.cuh"

namespace mkv {

// Launches a decode kernel with cudaLaunchKernelEx: a thread-block cluster of
// cluster_x CTAs when cluster_x > 0, and programmatic stream serialization
// (the kernel may start before the previous kernel of the stream ends; see
// griddep_wait) when pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, bool pdl, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

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

}  // namespace mkv
