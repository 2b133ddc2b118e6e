// Internal declarations shared by the library's CUDA translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mkv.h"

namespace mkv {

constexpr int D = 128;                 // head dim
constexpr int MAX_G = 16;              // query heads per KV head
constexpr int HIST1 = 2048;            // radix digit bins: bits 31..21
constexpr int HIST2 = 2048;            //                    bits 20..10
constexpr int HIST3 = 1024;            //                    bits  9..0
constexpr int HIST_WORDS = HIST1 + HIST2 + HIST3;
constexpr int TOPK_CHUNK = 4096;       // tokens per CTA in the selection passes
constexpr int TILE_T = 64;             // tokens per rotation tile

__host__ __device__ inline int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline uint32_t pad16(uint32_t n) { return (n + 15u) & ~15u; }

__host__ __device__ inline uint32_t segment_bytes(int strategy, int rows, int c) {
  switch (strategy) {
    case MKV_STRATEGY_SM: return pad16((uint32_t)c) + 2u * (uint32_t)c * (uint32_t)rows;
    case MKV_STRATEGY_PV: return 2u * (uint32_t)c * (uint32_t)rows + pad16((uint32_t)c * (uint32_t)rows);
    default: return 256u * (uint32_t)rows;
  }
}

// Per-segment result of the statistics pass (one per segment of every stream).
struct SegInfo {
  uint32_t size;       // packed bytes
  uint8_t strategy;
  uint8_t pad;
  uint16_t rows;
  uint32_t mask[4];    // segment-shared channels as a 128-bit set
  float f_sm;
  float f_pv;
};
static_assert(sizeof(SegInfo) == 32, "SegInfo layout");

// ---------------------------------------------------------------------------
// Compression (prefill)
// ---------------------------------------------------------------------------
struct CompressParams {
  const __half* X[2];        // K, V: [B][H][T][128]
  int BH;                    // streams per X
  int64_t T;
  int S;                     // segment size
  int c;
  float tau;
  int n_seg;                 // segments per stream
  // Gram pass
  int gram_chunks;           // CTAs per stream in the Gram pass
  int64_t gram_chunk_tokens; // tokens per Gram CTA (multiple of 64)
  float* gram_part;          // [2][BH][gram_chunks][128][128]
  // basis
  float* R;                  // [2][BH][128][128]
  float* lam;                // [2][BH][128]
  // statistics / pack passes
  int segs_per_cta;          // segments per CTA
  int ctas_per_stream;
  SegInfo* seg;              // [2][BH][n_seg]
  mkv_segment_header* hdr;   // [2][BH][n_seg]
  unsigned long long* total; // device: total packed bytes
  uint8_t* pool;
};

cudaError_t launch_gram(const CompressParams& p, cudaStream_t st);
cudaError_t launch_eig(const CompressParams& p, cudaStream_t st);
cudaError_t launch_analyze(const CompressParams& p, cudaStream_t st);
cudaError_t launch_scan(const CompressParams& p, cudaStream_t st);
cudaError_t launch_pack(const CompressParams& p, cudaStream_t st);

// ---------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------
struct DecodeParams {
  int B, H, Hq, g;
  int64_t T;
  int S, c, n_seg;
  int kk;                          // min(top_k, T)
  const __half* q;                 // [B][Hq][128]
  const float* RK;                 // [BH][128][128]
  const float* RV;                 // [BH][128][128]
  const uint8_t* pool;
  const mkv_segment_header* hdrK;  // [BH][n_seg]
  const mkv_segment_header* hdrV;  // [BH][n_seg]
  float* qt;                       // [B][Hq][128]
  float* qbar;                     // [BH][128]
  float* scores;                   // [BH][T]
  uint32_t* hist;                  // [BH][HIST_WORDS]
  int2* cnt;                       // [BH][topk_chunks]
  int2* res;                       // [BH]: (threshold key, how many equal keys to take)
  int topk_chunks;                 // ceil(T / TOPK_CHUNK)
  int32_t* sel;                    // [BH][kk] (internal)
  int32_t* sel_user;               // optional copy for the caller
  int score_segs_per_cta;
  int score_ctas_per_stream;
  int attn_chunk;                  // selected tokens per attention CTA
  int attn_chunks;                 // ceil(kk / attn_chunk)
  float* part_o;                   // [BH][attn_chunks][g][128]
  float* part_ml;                  // [BH][attn_chunks][g][2]
  float* out;                      // [B][Hq][128]
};

cudaError_t launch_qrot(const DecodeParams& p, cudaStream_t st);
cudaError_t launch_score(const DecodeParams& p, cudaStream_t st);
// the four selection launches; returns after enqueueing all of them
cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st);
cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st);

}  // namespace mkv
