// Internal declarations shared by the library's CUDA translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mkv.h"

namespace mkv {

constexpr int D = 128;                 // head dim
constexpr int MAX_G = 16;              // query heads per KV head
constexpr int GRAM_TILE = 128;         // tokens per tensor-core tile of the prefill kernels
constexpr int HIST1 = 4096;            // level-1 radix digit of the score key: bits 31..20
constexpr int HISTA = 1024;            // candidates, bits 19..10
constexpr int HISTB = 1024;            // candidates, bits  9..0
constexpr int ATTN_MAX_CHUNK = 128;    // largest explicit attention slice (mkv_config.attn_chunk)

__host__ __device__ inline int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ inline uint32_t pad16(uint32_t n) { return (n + 15u) & ~15u; }

__host__ __device__ inline uint32_t segment_bytes(int strategy, int rows, int c) {
  switch (strategy) {
    case MKV_STRATEGY_SM: return pad16((uint32_t)c) + 2u * (uint32_t)c * (uint32_t)rows;
    case MKV_STRATEGY_PV: return 2u * (uint32_t)c * (uint32_t)rows + pad16((uint32_t)c * (uint32_t)rows);
    case MKV_STRATEGY_PVB: return (2u * (uint32_t)c + 16u) * (uint32_t)rows;
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
  int64_t gram_chunk_tokens; // tokens per Gram CTA (multiple of GRAM_TILE)
  float* gram_part;          // [2][BH][gram_chunks][128][128]
  // basis
  float* R;                  // [2][BH][128][128]
  float* lam;                // [2][BH][128]
  // statistics / pack passes
  int segs_per_cta;          // segments per CTA
  int ctas_per_stream;
  SegInfo* seg;              // [2][BH][n_seg]
  uint32_t* tokmask;         // [2][BH][T][4]: per-token channel masks (statistics -> packing)
  float* colE;               // [2][BH][n_seg][128]: column energies per segment
  float* segK;               // [2][BH][n_seg]: kept energy of per-token top-c per segment
  mkv_segment_header* hdr;   // [2][BH][n_seg]
  unsigned long long* total; // device: [0] total packed bytes, [1..2] dense segments of K, V
  uint8_t* pool;
  uint64_t pool_check;       // pack writes must end within this many pool bytes
  int* err;                  // device status word
  uint64_t* packed_end;      // commit: device running end of the packed bytes (scan base)
  int bitmask_pv;            // PVB is a candidate strategy
};

// Decode-time append: rotates n new tokens per stream into the stream's K and
// V bases and stores them, fp16, as rows [tail_len, tail_len + n) of the tail
// (dense rotated rows in the pool, original tokens in tail_x).
struct AppendParams {
  const __half* k;           // [B][H][n_total][128]: this call's new tokens
  const __half* v;
  int64_t n_total;           // tokens per stream in k and v
  int64_t first;             // first of them to store
  int n;                     // tokens stored by this launch
  int tail_len;              // rows already in the tail
  int BH, S;
  const float* R;            // [2][BH][128][128] live bases
  uint8_t* pool;
  uint64_t tail_k, tail_v;   // byte offsets of the rotated tail regions
  __half* tail_x;            // [2][BH][S][128] original tokens
};
cudaError_t launch_append(const AppendParams& a, cudaStream_t st);
// headers of one committed segment per stream: offsets from *packed_end on
// (which then moves past them)
cudaError_t launch_commit_scan(const CompressParams& p, cudaStream_t st);
// out[2][BH][n_old + 1] = old[2][BH][n_old] with seg_new[2][BH] appended per stream
cudaError_t launch_grow_headers(const mkv_segment_header* old, int n_old,
                                const mkv_segment_header* seg_new, int n_streams2,
                                mkv_segment_header* out, cudaStream_t st);

cudaError_t launch_gram(const CompressParams& p, cudaStream_t st);
cudaError_t launch_eig(const CompressParams& p, cudaStream_t st);
cudaError_t launch_analyze(const CompressParams& p, cudaStream_t st);
cudaError_t launch_scan(const CompressParams& p, cudaStream_t st);
cudaError_t launch_pack(const CompressParams& p, cudaStream_t st);

// ---------------------------------------------------------------------------
// Decode
// ---------------------------------------------------------------------------
// Per-stream state of the top-k selection within one decode step.
struct TopkState {
  uint32_t b1;      // level-1 bin holding the k-th largest key
  uint32_t k1;      // keys still needed from that bin
  uint32_t thr;     // the k-th largest key
  int32_t t_cut;    // keys equal to thr are taken up to this token index
};

// One shared-memory stage of the score kernel, planned at compression: the
// whole segments [seg0, seg0 + nseg) of the flattened K segments, copied as
// the 128-byte lines [line0, line0 + nlines) of the pool plus nhdr2 16-byte
// pairs of their headers (from header index seg0 rounded down to even).
struct StagePlan {
  uint32_t seg0;
  uint16_t nseg;
  uint16_t nhdr2;
  uint32_t line0;
  uint32_t nlines;
};

struct DecodeParams {
  int B, H, Hq, g;
  int64_t T;
  int64_t Tp;                      // row stride of scores / candidates: T rounded up to 16
  int S, c, n_seg;                 // n_seg: segments per stream, prefill ones then committed ones
  int kk;                          // min(top_k, T)
  // decode-time appends: tokens [0, T0) are the prefill (segments 0 .. nseg0 - 1
  // at multiples of S, the last possibly ragged); committed segments of S
  // tokens follow from T0; tokens [T_packed, T) wait in the tail, stored as
  // dense rotated rows at pool offset tail_k16 (K) / tail_v16 (V), in 16-byte
  // units, S rows per stream
  int64_t T0, T_packed;
  int nseg0;
  uint32_t tail_k16, tail_v16;
  const __half* q;                 // [B][Hq][128]
  const float* RK;                 // [BH][128][128]
  const float* RV;                 // [BH][128][128]
  const uint8_t* pool;
  uint64_t pool_check;             // pool reads must end within this many bytes
  const mkv_segment_header* hdrK;  // [BH][n_seg] (all K streams, contiguous)
  const mkv_segment_header* hdrV;  // [BH][n_seg]
  float* qt;                       // [B][Hq][128]
  float* qbar;                     // [BH][128]
  float* scores;                   // [BH][Tp]
  uint32_t* hist;                  // [BH][HIST1]
  // score-kernel partition, fixed at compression: CTA i covers the flattened
  // K segments [part[i], part[i+1]) (balanced by bytes); cta_cnt[s] = CTAs
  // that touch stream s
  const int32_t* part;
  const int32_t* cta_cnt;
  // CTA i's stages are plan[part[i] .. part[i] + plan_n[i])
  const StagePlan* plan;
  const int32_t* plan_n;
  int G;
  int stage_bytes;                 // bytes per shared-memory stage of the score kernel
  int n_stages;
  uint32_t* tick1;                 // [BH] tickets: score CTAs done with a stream
  uint2* cand;                     // [BH][Tp] (key, token) of threshold-bin candidates
  TopkState* state;                // [BH]
  int sel_R;                       // CTAs (one cluster) per stream in the selection
  int32_t* sel;                    // [BH][kk] (internal)
  int32_t* sel_user;               // optional copy for the caller
  // attention: the B H kk selected positions, flattened, in slices of
  // attn_per positions (one CTA each); attn_mp partial slots per stream
  int64_t attn_per;
  int attn_ctas;
  int attn_mp;
  // per-token shared-memory slot of the attention kernel: K values, K channel
  // list, V values, V channel list (bytes, multiples of 16), and stages
  int at_kv, at_ki, at_vv, at_vi, at_slot, at_stages;
  float* part_o;                   // [BH][attn_mp][g][128]
  float* part_ml;                  // [BH][attn_mp][g][2]
  float* out;                      // [B][Hq][128]
  int* err;                        // device status word (0 = ok)
  int pdl;                         // bit k: launch decode kernel k (MKV_KERNEL_* order)
                                   // with programmatic dependent launch
  int pdl_trigger;                 // kernels let their dependents start early
};

// First token of segment sg of a stream (prefill segments at multiples of S,
// committed segments of S tokens after the prefill's T0 tokens).
__host__ __device__ inline int64_t seg_start(int sg, int S, int nseg0, int64_t T0) {
  return sg < nseg0 ? (int64_t)sg * S : T0 + (int64_t)(sg - nseg0) * S;
}

// bits of the device status word (0 = ok), set with atomicOr
constexpr int DEV_ERR_TIMEOUT = 1;   // a bounded wait gave up
constexpr int DEV_ERR_CHECK = 2;     // an access fell outside the checked pool extent

// test hook: one CTA runs the library's bounded mbarrier wait on a barrier no
// thread arrives on, with the given limit
cudaError_t launch_wait_test(int* err, uint64_t limit_ns, cudaStream_t st);

// one-time per device: function attributes (not stream-ordered, so not in decode)
cudaError_t prepare_decode_kernels();
cudaError_t prepare_score_kernels();
cudaError_t prepare_select_kernels();
cudaError_t prepare_attn_kernels();
// score-kernel shared-memory plan: stage size and number of stages
void score_stage_plan(int S, int c, int* stage_bytes, int* n_stages);
// partition of the K segments over G score CTAs and their stage plans (run
// once per compression); plan holds n_streams * n_seg entries
cudaError_t launch_partition(const mkv_segment_header* hdrK, int n_streams, int n_seg, int c,
                             int G, int stage_bytes, int32_t* part, int32_t* cta_cnt,
                             StagePlan* plan, int32_t* plan_n, int64_t* prefix, cudaStream_t st);
// Decode parameters of several layers decoded by one launch of each decode
// kernel (layer l = blockIdx.z), passed by value as a __grid_constant__
// kernel parameter.  All layers share every launch-shape field of p[0].
constexpr int MAX_FUSED_LAYERS = MKV_MAX_FUSED_LAYERS;
struct LayerParams {
  DecodeParams p[MAX_FUSED_LAYERS];
};
static_assert(sizeof(LayerParams) <= 32000, "layer parameters must fit the kernel parameter space");

// Decode launches: one layer with p, or layers lp->p[0 .. n) (p == lp->p[0])
// in one launch when lp is given.
cudaError_t launch_qrot(const DecodeParams& p, cudaStream_t st, const LayerParams* lp = nullptr,
                        int n = 1);
cudaError_t launch_score(const DecodeParams& p, cudaStream_t st, const LayerParams* lp = nullptr,
                         int n = 1);
// the selection launch (one cluster of sel_R CTAs per stream)
cudaError_t launch_topk(const DecodeParams& p, cudaStream_t st, const LayerParams* lp = nullptr,
                        int n = 1);
// CTAs per stream for the selection: up to 8 while the grid fits G SMs twice
int select_cluster_size(int n_streams, int64_t T, int G);
cudaError_t launch_attn(const DecodeParams& p, cudaStream_t st, const LayerParams* lp = nullptr,
                        int n = 1);
// attention kernel shape for a slot size: stages and resident CTAs per SM
cudaError_t attn_shape(int g, int slot, int* stages, int* ctas_per_sm);
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t st, const LayerParams* lp = nullptr,
                         int n = 1);

}  // namespace mkv
