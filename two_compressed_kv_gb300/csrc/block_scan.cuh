// Block-wide prefix sums shared by the layout kernels (segment offsets at
// compression, the score kernel's byte partition).
#pragma once

#include <stdint.h>

namespace mkv {

// Block-wide (1024 threads) exclusive scan of one 64-bit value per thread;
// every thread also gets the block total.  Fixed order (integer sums).
__device__ __forceinline__ unsigned long long block_excl_scan64(unsigned long long v,
                                                                unsigned long long* ws,
                                                                unsigned long long& total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned long long inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long o = __shfl_up_sync(0xffffffffu, inc, off);
    if (lane >= off) inc += o;
  }
  __syncthreads();                   // ws of an earlier call has been read
  if (lane == 31) ws[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const unsigned long long w = ws[lane];
    unsigned long long x = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long o = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += o;
    }
    ws[32 + lane] = x - w;           // exclusive prefix of the warp sums
    if (lane == 31) ws[64] = x;
  }
  __syncthreads();
  total = ws[64];
  return ws[32 + warp] + inc - v;
}

}  // namespace mkv
