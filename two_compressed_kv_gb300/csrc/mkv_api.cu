// Host side of the C ABI in include/mkv.h: ctx lifetime, argument checks,
// device buffers, launch order, kernel timing and introspection.
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "mkv_internal.cuh"
#include "ptx.cuh"

using namespace mkv;

namespace {

constexpr int kSMs = 152;          // GB300
constexpr int64_t kMergeMaxWeights = 12288;   // 48 KB of fp32 (slice, head) weights
constexpr int64_t kMinSlice = 32;              // smallest automatic attention slice
thread_local std::string g_last_error = "no error";

mkv_status cuda_fail(cudaError_t e, const char* what) {
  char buf[256];
  snprintf(buf, sizeof(buf), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
  g_last_error = buf;
  return e == cudaErrorMemoryAllocation ? MKV_ERR_OOM : MKV_ERR_CUDA;
}

#define CK(call)                                         \
  do {                                                   \
    cudaError_t e_ = (call);                             \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
  } while (0)

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct KernelTimer {
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
  std::vector<cudaEvent_t> spare;
  double total_ms = 0.0;
  int64_t launches = 0;
};

}  // namespace

struct mkv_ctx {
  mkv_config cfg;
  int B = 0, H = 0, Hq = 0, g = 0, BH = 0;
  int64_t max_seg = 0;
  int kk_max = 0;
  int gram_chunks_max = 0;
  int64_t attn_per_fixed = 0;      // mkv_config.attn_chunk (0 = spread over the SMs)
  int attn_mp = 0;                 // partial slots per stream
  int at_stages = 2, at_ctas_per_sm = 1;
  int at_kv = 0, at_ki = 0, at_vv = 0, at_vi = 0;
  int64_t Tp_max = 0;              // padded row stride of scores / candidates
  int G = 0;                       // score-kernel CTAs (one per SM)
  int stage_bytes = 0, n_stages = 0;

  // current cache
  int64_t T = 0;
  int n_seg = 0;
  bool ready = false;
  int live = 0;                    // which of the double-buffered copies is live
  float* R[2] = {nullptr, nullptr};
  float* lam[2] = {nullptr, nullptr};
  mkv_segment_header* hdr[2] = {nullptr, nullptr};
  int32_t* part[2] = {nullptr, nullptr};      // score-kernel partition of the K segments
  int32_t* cta_cnt[2] = {nullptr, nullptr};   // score CTAs per stream
  StagePlan* plan[2] = {nullptr, nullptr};    // score-kernel stages
  int32_t* plan_n[2] = {nullptr, nullptr};    // stages per score CTA
  uint8_t* pool = nullptr;
  uint64_t pool_cap = 0;
  uint64_t pool_need = 0;          // bytes of the live cache's pool (packed size + tail pad)
  uint64_t check_override = 0;     // test hook: a smaller checked pool extent (0 = none)
  // decode kernels launched with programmatic dependent launch (bit k =
  // MKV_KERNEL_* id): the rotation, score and attention kernels gain about
  // 1.5 us each at the 128K batch-8 shape; the clustered selection kernel
  // and the merge lose time with it, so they are launched plainly
  uint32_t pdl_mask = (1u << MKV_KERNEL_QROT) | (1u << MKV_KERNEL_SCORE);

  // compression scratch
  SegInfo* seg = nullptr;
  uint32_t* tokmask = nullptr;     // [2][BH][max_ctx][4] per-token channel masks
  float* colE = nullptr;           // [2][BH][max_seg][128] column energies per segment
  float* segK = nullptr;           // [2][BH][max_seg] kept energy per segment
  float* gram_part = nullptr;
  unsigned long long* total_dev = nullptr;
  unsigned long long* total_host = nullptr;

  // decode scratch
  float* qt = nullptr;
  float* qbar = nullptr;
  float* scores = nullptr;
  uint32_t* hist = nullptr;
  uint32_t* tick = nullptr;        // [BH]: score CTAs done with a stream
  uint2* cand = nullptr;
  TopkState* state = nullptr;
  int32_t* sel = nullptr;
  int* err = nullptr;
  float* part_o = nullptr;
  float* part_ml = nullptr;

  // decode-time appends (tokens after the prefill)
  int64_t T0 = 0;                  // prefill tokens
  int nseg0 = 0;                   // prefill segments per stream
  int n_commit = 0;                // committed segments per stream
  int tail_len = 0;                // tokens waiting in the tail
  uint64_t tail_bytes = 0;         // rotated tail rows in the pool (K then V), 0: no appends
  uint64_t tail_off = 0;           // their byte offset in the pool
  uint64_t packed_bound = 0;       // upper bound of the packed bytes' end (host)
  uint64_t* packed_end = nullptr;  // the packed bytes' end (device, moved by commits)
  __half* tail_x = nullptr;        // [2][BH][S][128] tail tokens as given
  mkv_segment_header* hdr_commit = nullptr;   // [2][BH] headers of one commit
  int64_t* kprefix = nullptr;      // [BH * max_seg + 1] cumulative K segment sizes
  int at_stages_dense = 2, at_ctas_dense = 1; // attention shape with room for dense rows

  int64_t decode_calls = 0;
  int64_t launches = 0;
  KernelTimer timers[MKV_KERNEL_COUNT];
};

namespace {

bool timing_on(const mkv_ctx* c, int id) {
  return (c->cfg.flags & MKV_FLAG_KERNEL_TIMING) != 0u ||
         (id == MKV_KERNEL_SCORE && (c->cfg.flags & MKV_FLAG_SCORE_TIMING) != 0u);
}

mkv_status resolve_timer(KernelTimer& t, size_t keep) {
  while (t.pending.size() > keep) {
    auto ev = t.pending.front();
    t.pending.erase(t.pending.begin());
    CK(cudaEventSynchronize(ev.second));
    float ms = 0.f;
    CK(cudaEventElapsedTime(&ms, ev.first, ev.second));
    t.total_ms += ms;
    t.spare.push_back(ev.first);
    t.spare.push_back(ev.second);
  }
  return MKV_OK;
}

mkv_status timer_event(KernelTimer& t, cudaEvent_t* ev) {
  if (!t.spare.empty()) {
    *ev = t.spare.back();
    t.spare.pop_back();
    return MKV_OK;
  }
  CK(cudaEventCreate(ev));
  return MKV_OK;
}

// Records `ev` on `st`.  Inside a stream capture the record must be an
// external event-record node so that every replay of the graph records it.
cudaError_t record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  if (cs == cudaStreamCaptureStatusActive) return cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  return cudaEventRecord(ev, st);
}

// Runs `launch` on `st`, bracketed by events when timing is on.
template <typename F>
mkv_status timed(mkv_ctx* c, int id, cudaStream_t st, int n_kernels, F launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (timing_on(c, id)) {
    if (c->timers[id].pending.size() >= 4096) {
      mkv_status s = resolve_timer(c->timers[id], 2048);
      if (s != MKV_OK) return s;
    }
    mkv_status s = timer_event(c->timers[id], &a);
    if (s != MKV_OK) return s;
    s = timer_event(c->timers[id], &b);
    if (s != MKV_OK) return s;
    CK(record(a, st));
  }
  CK(launch());
  c->launches += n_kernels;
  if (timing_on(c, id)) {
    CK(record(b, st));
    c->timers[id].pending.emplace_back(a, b);
    c->timers[id].launches += 1;
  }
  return MKV_OK;
}

template <typename T>
mkv_status dalloc(T** p, size_t n) {
  *p = nullptr;
  if (n == 0) n = 1;
  CK(cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T)));
  return MKV_OK;
}

void release(mkv_ctx* c) {
  if (!c) return;
  cudaSetDevice(c->cfg.device);
  for (int i = 0; i < 2; ++i) {
    cudaFree(c->R[i]);
    cudaFree(c->lam[i]);
    cudaFree(c->hdr[i]);
    cudaFree(c->part[i]);
    cudaFree(c->cta_cnt[i]);
    cudaFree(c->plan[i]);
    cudaFree(c->plan_n[i]);
  }
  cudaFree(c->pool);
  cudaFree(c->seg);
  cudaFree(c->tokmask);
  cudaFree(c->colE);
  cudaFree(c->segK);
  cudaFree(c->gram_part);
  cudaFree(c->total_dev);
  if (c->total_host) cudaFreeHost(c->total_host);
  cudaFree(c->qt);
  cudaFree(c->qbar);
  cudaFree(c->scores);
  cudaFree(c->hist);
  cudaFree(c->tick);
  cudaFree(c->cand);
  cudaFree(c->state);
  cudaFree(c->sel);
  cudaFree(c->err);
  cudaFree(c->part_o);
  cudaFree(c->part_ml);
  cudaFree(c->packed_end);
  cudaFree(c->tail_x);
  cudaFree(c->hdr_commit);
  cudaFree(c->kprefix);
  for (auto& t : c->timers) {
    for (auto& e : t.pending) {
      cudaEventDestroy(e.first);
      cudaEventDestroy(e.second);
    }
    for (auto& e : t.spare) cudaEventDestroy(e);
  }
  delete c;
}

// Packed bytes of one commit if every new segment were dense.
uint64_t commit_worst(const mkv_ctx* c) {
  return 2ull * c->BH * segment_bytes(MKV_STRATEGY_DENSE, c->cfg.segment, c->cfg.c);
}

int gram_chunks_for(int BH, int64_t T) {
  const int64_t target = 4 * kSMs;
  int64_t ch = ceil_div(target, 2 * (int64_t)BH);
  ch = std::min<int64_t>(ch, std::max<int64_t>(1, ceil_div(T, 256)));
  return (int)std::max<int64_t>(1, ch);
}

}  // namespace

// Scratch of mkv_basis_static: the partial Gram matrices of every (stream,
// chunk), each 128 x 128 fp32.  A file-scope static device array, so that the
// call allocates nothing; its address is looked up at every call.
static __device__ __align__(256) unsigned char g_basis_scratch[MKV_BASIS_STATIC_MAX_BYTES];

namespace {

constexpr int64_t kGramPartBytes = (int64_t)D * D * sizeof(float);
constexpr int64_t kBasisStaticParts = MKV_BASIS_STATIC_MAX_BYTES / kGramPartBytes;

// The buffer's address in the current device's context.  Looked up on every
// call (cheap once the module is loaded): a cached address would go stale
// after a device reset or a new primary context.
mkv_status basis_scratch_here(float** out) {
  void* a = nullptr;
  CK(cudaGetSymbolAddress(&a, g_basis_scratch));
  *out = static_cast<float*>(a);
  return MKV_OK;
}

}  // namespace

extern "C" {

const char* mkv_status_string(mkv_status s) {
  switch (s) {
    case MKV_OK: return "MKV_OK";
    case MKV_ERR_INVALID_ARG: return "MKV_ERR_INVALID_ARG";
    case MKV_ERR_STATE: return "MKV_ERR_STATE";
    case MKV_ERR_OOM: return "MKV_ERR_OOM";
    case MKV_ERR_CUDA: return "MKV_ERR_CUDA";
    case MKV_ERR_DEVICE_CHECK: return "MKV_ERR_DEVICE_CHECK";
    case MKV_ERR_TIMEOUT: return "MKV_ERR_TIMEOUT";
  }
  return "MKV_ERR_UNKNOWN";
}

const char* mkv_last_error_string(void) { return g_last_error.c_str(); }

uint64_t mkv_segment_bytes(int strategy, int rows, int c) {
  if (rows < 1 || rows > 65535 || c < 1 || c > MKV_HEAD_DIM) return 0;
  if (strategy < MKV_STRATEGY_SM || strategy > MKV_STRATEGY_PVB) return 0;
  return segment_bytes(strategy, rows, c);
}

mkv_status mkv_validate_config(const mkv_config* cfg) {
  if (!cfg) return MKV_ERR_INVALID_ARG;
  const mkv_config& c = *cfg;
  if (c.batch < 1 || c.n_kv_heads < 1 || c.n_q_heads < 1) return MKV_ERR_INVALID_ARG;
  if (c.n_q_heads % c.n_kv_heads != 0) return MKV_ERR_INVALID_ARG;
  if (c.n_q_heads / c.n_kv_heads > MAX_G) return MKV_ERR_INVALID_ARG;
  if (c.head_dim != MKV_HEAD_DIM) return MKV_ERR_INVALID_ARG;
  if (c.max_ctx < 1 || c.max_ctx > (int64_t)INT32_MAX) return MKV_ERR_INVALID_ARG;
  if (c.segment < 16 || c.segment > 256 || c.segment % 16 != 0) return MKV_ERR_INVALID_ARG;
  if (c.c < 8 || c.c > MKV_HEAD_DIM || c.c % 8 != 0) return MKV_ERR_INVALID_ARG;
  if (!(c.tau > 0.f && c.tau <= 1.f)) return MKV_ERR_INVALID_ARG;
  if (c.top_k < 1) return MKV_ERR_INVALID_ARG;
  if (c.attn_chunk != 0 && (c.attn_chunk < 8 || c.attn_chunk > ATTN_MAX_CHUNK || c.attn_chunk % 8 != 0))
    return MKV_ERR_INVALID_ARG;
  if (c.flags & ~MKV_FLAGS_ALL) return MKV_ERR_INVALID_ARG;
  if (c.device < 0) return MKV_ERR_INVALID_ARG;
  const int64_t streams = (int64_t)c.batch * c.n_kv_heads;
  if (streams > (1 << 20)) return MKV_ERR_INVALID_ARG;
  return MKV_OK;
}

mkv_status mkv_create(const mkv_config* cfg, mkv_ctx** out) {
  if (!out) return MKV_ERR_INVALID_ARG;
  *out = nullptr;
  mkv_status st = mkv_validate_config(cfg);
  if (st != MKV_OK) return st;
  int ndev = 0;
  CK(cudaGetDeviceCount(&ndev));
  if (cfg->device >= ndev) return MKV_ERR_INVALID_ARG;
  CK(cudaSetDevice(cfg->device));
  CK(prepare_decode_kernels());
  mkv_ctx* c = new (std::nothrow) mkv_ctx();
  if (!c) return MKV_ERR_OOM;
  c->cfg = *cfg;
  c->B = cfg->batch;
  c->H = cfg->n_kv_heads;
  c->Hq = cfg->n_q_heads;
  c->g = c->Hq / c->H;
  c->BH = c->B * c->H;
  // a ragged prefill plus committed segments can need one segment more
  c->max_seg = ceil_div(cfg->max_ctx, cfg->segment) + 1;
  c->kk_max = (int)std::min<int64_t>(cfg->top_k, cfg->max_ctx);
  c->gram_chunks_max = gram_chunks_for(c->BH, cfg->max_ctx);
  c->Tp_max = ceil_div(cfg->max_ctx, 16) * 16;
  {
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, cfg->device);
    if (e != cudaSuccess) {
      delete c;
      return cuda_fail(e, "cudaDeviceGetAttribute");
    }
    c->G = sms;
  }
  // Split-K slices of the attention: an explicit size, or the selected
  // positions spread over at most two CTAs per SM with at least
  // kMinSlice positions each.  A stream's selection then meets at most
  // ceil(kk / slice) + 1 slices; the merge keeps one weight per (slice,
  // head) of a stream in shared memory.
  c->attn_per_fixed = cfg->attn_chunk;
  if (c->attn_per_fixed) {
    while (ceil_div(c->kk_max, c->attn_per_fixed) + 1 > kMergeMaxWeights / c->g &&
           c->attn_per_fixed < ATTN_MAX_CHUNK)
      c->attn_per_fixed = std::min<int64_t>(ATTN_MAX_CHUNK, 2 * c->attn_per_fixed);
    c->attn_mp = (int)ceil_div(c->kk_max, c->attn_per_fixed) + 1;
  } else {
    c->attn_mp = (int)std::min<int64_t>(ceil_div(2 * (int64_t)c->G, c->BH),
                                        ceil_div(c->kk_max, kMinSlice)) + 2;
  }
  if ((int64_t)c->attn_mp * c->g > kMergeMaxWeights) {
    delete c;
    g_last_error = "top_k too large for the split-K merge";
    return MKV_ERR_INVALID_ARG;
  }
  score_stage_plan(cfg->segment, cfg->c, &c->stage_bytes, &c->n_stages);
  const size_t BH = c->BH;
  mkv_status s = MKV_OK;
#define AL(ptr, n)                         \
  if (s == MKV_OK) s = dalloc(&(ptr), (n)); \
  if (s != MKV_OK) {                       \
    release(c);                            \
    return s;                              \
  }
  for (int i = 0; i < 2; ++i) {
    AL(c->R[i], 2 * BH * D * D);
    AL(c->lam[i], 2 * BH * D);
    AL(c->hdr[i], 2 * BH * (size_t)c->max_seg);
    AL(c->part[i], (size_t)c->G + 1);
    AL(c->cta_cnt[i], BH);
    AL(c->plan[i], BH * (size_t)c->max_seg);
    AL(c->plan_n[i], (size_t)c->G);
  }
  AL(c->seg, 2 * BH * (size_t)c->max_seg);
  AL(c->tokmask, 2 * BH * (size_t)cfg->max_ctx * 4);
  AL(c->colE, 2 * BH * (size_t)c->max_seg * D);
  AL(c->segK, 2 * BH * (size_t)c->max_seg);
  AL(c->gram_part, 2 * BH * (size_t)c->gram_chunks_max * D * D);
  AL(c->total_dev, 3);
  AL(c->qt, (size_t)c->B * c->Hq * D);
  AL(c->qbar, BH * D);
  AL(c->scores, BH * (size_t)c->Tp_max);
  AL(c->hist, BH * HIST1);
  AL(c->tick, BH);
  AL(c->cand, BH * (size_t)c->Tp_max);
  AL(c->state, BH);
  AL(c->sel, BH * (size_t)c->kk_max);
  AL(c->err, 1);
  AL(c->packed_end, 1);
  AL(c->tail_x, 2 * BH * (size_t)cfg->segment * D);
  AL(c->hdr_commit, 2 * BH);
  AL(c->kprefix, BH * (size_t)c->max_seg + 1);
  AL(c->part_o, BH * (size_t)c->attn_mp * c->g * D);
  AL(c->part_ml, BH * (size_t)c->attn_mp * c->g * 2);
#undef AL
  cudaError_t e = cudaMallocHost(reinterpret_cast<void**>(&c->total_host),
                                 3 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = cudaMemset(c->tick, 0, BH * sizeof(uint32_t));
  if (e == cudaSuccess) e = cudaMemset(c->err, 0, sizeof(int));
  if (e == cudaSuccess) e = cudaMemset(c->sel, 0, BH * (size_t)c->kk_max * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    release(c);
    return cuda_fail(e, "ctx initialisation");
  }
  *out = c;
  return MKV_OK;
}

void mkv_free(mkv_ctx* ctx) {
  if (!ctx) return;
  cudaSetDevice(ctx->cfg.device);
  cudaDeviceSynchronize();
  release(ctx);
}

mkv_status mkv_compress(mkv_ctx* c, const void* k, const void* v, int64_t ctx_len,
                        mkv_stream_t stream) {
  if (!c || !k || !v) return MKV_ERR_INVALID_ARG;
  if (ctx_len < 1 || ctx_len > c->cfg.max_ctx) return MKV_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) return MKV_ERR_INVALID_ARG;
  CK(cudaSetDevice(c->cfg.device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int stage = 1 - c->live;
  CompressParams p;
  memset(&p, 0, sizeof(p));
  p.X[0] = static_cast<const __half*>(k);
  p.X[1] = static_cast<const __half*>(v);
  p.BH = c->BH;
  p.T = ctx_len;
  p.S = c->cfg.segment;
  p.c = c->cfg.c;
  p.tau = c->cfg.tau;
  p.n_seg = (int)ceil_div(ctx_len, p.S);
  p.gram_chunks = std::min(c->gram_chunks_max, gram_chunks_for(c->BH, ctx_len));
  p.gram_chunk_tokens = ceil_div(ceil_div(ctx_len, p.gram_chunks), GRAM_TILE) * GRAM_TILE;
  p.gram_chunks = (int)ceil_div(ctx_len, p.gram_chunk_tokens);
  p.gram_part = c->gram_part;
  p.R = c->R[stage];
  p.lam = c->lam[stage];
  // analyze/pack: about 4 CTAs of 1 per SM per wave, whole segments each
  const int64_t total_segs = 2 * (int64_t)c->BH * p.n_seg;
  const int64_t want_ctas = 4 * kSMs;
  p.segs_per_cta = (int)std::max<int64_t>(1, ceil_div(total_segs, want_ctas));
  p.ctas_per_stream = (int)ceil_div(p.n_seg, p.segs_per_cta);
  p.seg = c->seg;
  p.tokmask = c->tokmask;
  p.colE = c->colE;
  p.segK = c->segK;
  p.bitmask_pv = (c->cfg.flags & MKV_FLAG_BITMASK_PV) != 0u;
  p.hdr = c->hdr[stage];
  p.total = c->total_dev;
  p.pool = nullptr;

  mkv_status s;
  if ((s = timed(c, MKV_KERNEL_GRAM, st, 1, [&] { return launch_gram(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_EIG, st, 1, [&] { return launch_eig(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_ANALYZE, st, 1, [&] { return launch_analyze(p, st); })) != MKV_OK)
    return s;
  if ((s = timed(c, MKV_KERNEL_LAYOUT, st, 3, [&] {
         cudaError_t e = launch_scan(p, st);
         if (e == cudaSuccess)
           e = launch_partition(p.hdr, c->BH, p.n_seg, p.c, c->G, c->stage_bytes, c->part[stage],
                                c->cta_cnt[stage], c->plan[stage], c->plan_n[stage], c->kprefix,
                                st);
         return e;
       })) != MKV_OK)
    return s;
  CK(cudaMemcpyAsync(c->total_host, c->total_dev, 3 * sizeof(unsigned long long),
                     cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  const uint64_t total = c->total_host[0];
  const bool dense_k = c->total_host[1] != 0, dense_v = c->total_host[2] != 0;
  if ((total >> 4) > 0xffffffffull) {
    g_last_error = "packed cache exceeds 64 GiB per ctx";
    return MKV_ERR_INVALID_ARG;
  }
  if (c->cfg.max_pool_bytes && total > c->cfg.max_pool_bytes) {
    g_last_error = "packed cache exceeds max_pool_bytes";
    return MKV_ERR_OOM;
  }
  // the score kernel copies whole 128-byte lines: 256 bytes of padding after
  // the packed bytes.  When tokens can still be appended, room for two
  // commits (every segment dense) and the rotated tail follow.
  const bool appendable = ctx_len < c->cfg.max_ctx;
  const uint64_t tail_bytes = appendable ? 2ull * c->BH * p.S * D * 2 : 0;
  const uint64_t reserve = appendable ? 2 * commit_worst(c) : 0;
  const uint64_t tail_off = (total + 256 + reserve + 255) & ~255ull;
  const uint64_t need = appendable ? tail_off + tail_bytes : total + 256;
  if (need > c->pool_cap) {
    uint8_t* np = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&np), need);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cuda_fail(e, "cudaMalloc(pool)");
    }
    CK(cudaFree(c->pool));   // synchronises: no decode still reads the old pool
    c->pool = np;
    c->pool_cap = need;
  }
  p.pool = c->pool;
  p.pool_check = c->check_override ? std::min(c->check_override, need) : need;
  p.err = c->err;
  c->ready = false;   // the live headers may no longer match the pool
  if ((s = timed(c, MKV_KERNEL_PACK, st, 1, [&] { return launch_pack(p, st); })) != MKV_OK) return s;
  CK(cudaMemcpyAsync(c->packed_end, c->total_dev, sizeof(uint64_t), cudaMemcpyDeviceToDevice,
                     st));
  c->live = stage;
  c->pool_need = need;
  c->T0 = ctx_len;
  c->nseg0 = p.n_seg;
  c->n_commit = 0;
  c->tail_len = 0;
  c->tail_bytes = tail_bytes;
  c->tail_off = tail_off;
  c->packed_bound = total;
  // the attention kernel's per-token slot: room for a dense row only when
  // the cache has dense segments
  c->at_kv = dense_k ? 256 : 2 * p.c;
  c->at_vv = dense_v ? 256 : 2 * p.c;
  c->at_ki = c->at_vi = (int)pad16((uint32_t)p.c);
  CK(attn_shape(c->g, c->at_kv + c->at_ki + c->at_vv + c->at_vi, &c->at_stages,
                &c->at_ctas_per_sm));
  CK(attn_shape(c->g, 256 + c->at_ki + 256 + c->at_vi, &c->at_stages_dense, &c->at_ctas_dense));
  c->T = ctx_len;
  c->n_seg = p.n_seg;
  c->ready = true;
  return MKV_OK;
}

}  // extern "C"

namespace {

// Attention launch shape: per-token slots holding value rows of at_kv (K)
// and at_vv (V) bytes, `stages` ring stages, `ctas_per_sm` resident CTAs.
void set_attn_shape(const mkv_ctx* c, DecodeParams& p, int at_kv, int at_vv, int stages,
                    int ctas_per_sm) {
  const int64_t N = (int64_t)c->BH * p.kk;
  const int64_t P = (int64_t)c->G * ctas_per_sm;
  p.attn_per = c->attn_per_fixed
                   ? c->attn_per_fixed
                   : std::max({ceil_div(N, P), kMinSlice, ceil_div(p.kk, c->attn_mp - 1)});
  p.attn_ctas = (int)ceil_div(N, p.attn_per);
  p.attn_mp = c->attn_mp;
  p.at_kv = at_kv;
  p.at_ki = c->at_ki;
  p.at_vv = at_vv;
  p.at_vi = c->at_vi;
  p.at_slot = p.at_kv + p.at_ki + p.at_vv + p.at_vi;
  p.at_stages = stages;
}

// Decode parameters of one ctx (compressed) for q, out and sel.
void fill_decode(mkv_ctx* c, const void* q, float* out, int32_t* sel, DecodeParams& p) {
  memset(&p, 0, sizeof(p));
  p.B = c->B;
  p.H = c->H;
  p.Hq = c->Hq;
  p.g = c->g;
  p.T = c->T;
  p.Tp = ceil_div(c->T, 16) * 16;
  p.S = c->cfg.segment;
  p.c = c->cfg.c;
  p.n_seg = c->n_seg;
  p.kk = (int)std::min<int64_t>(c->cfg.top_k, c->T);
  p.T0 = c->T0;
  p.nseg0 = c->nseg0;
  p.T_packed = c->T0 + (int64_t)c->n_commit * p.S;
  p.tail_k16 = (uint32_t)(c->tail_off >> 4);
  p.tail_v16 = (uint32_t)((c->tail_off + c->tail_bytes / 2) >> 4);
  p.q = static_cast<const __half*>(q);
  p.RK = c->R[c->live];
  p.RV = c->R[c->live] + (size_t)c->BH * D * D;
  p.pool = c->pool;
  p.pool_check = c->check_override ? std::min(c->check_override, c->pool_need) : c->pool_need;
  p.hdrK = c->hdr[c->live];
  p.hdrV = c->hdr[c->live] + (size_t)c->BH * c->n_seg;
  p.qt = c->qt;
  p.qbar = c->qbar;
  p.scores = c->scores;
  p.hist = c->hist;
  p.part = c->part[c->live];
  p.cta_cnt = c->cta_cnt[c->live];
  p.plan = c->plan[c->live];
  p.plan_n = c->plan_n[c->live];
  p.G = c->G;
  p.stage_bytes = c->stage_bytes;
  p.n_stages = c->n_stages;
  p.tick1 = c->tick;
  p.cand = c->cand;
  p.state = c->state;
  p.sel_R = select_cluster_size(c->BH, c->T, c->G);
  p.sel = c->sel;
  p.sel_user = sel;
  p.err = c->err;
  {
    // appended tokens are dense rows (the tail) or may sit in dense segments
    const bool appended = c->T > c->T0;
    set_attn_shape(c, p, appended ? 256 : c->at_kv, appended ? 256 : c->at_vv,
                   appended ? c->at_stages_dense : c->at_stages,
                   appended ? c->at_ctas_dense : c->at_ctas_per_sm);
  }
  p.part_o = c->part_o;
  p.part_ml = c->part_ml;
  p.out = out;
  // kernel timing records events between kernels: launch those plainly
  const bool pdl_on =
      (c->cfg.flags & (MKV_FLAG_KERNEL_TIMING | MKV_FLAG_SCORE_TIMING | MKV_FLAG_NO_PDL)) == 0u;
  p.pdl = pdl_on ? (c->pdl_mask & 0x1f) : 0;
  p.pdl_trigger = (c->pdl_mask & 0x100) ? 0 : 1;
}

}  // namespace

extern "C" {

mkv_status mkv_decode(mkv_ctx* c, const void* q, float* out, int32_t* sel, mkv_stream_t stream) {
  if (!c || !q || !out) return MKV_ERR_INVALID_ARG;
  if (!c->ready) return MKV_ERR_STATE;
  CK(cudaSetDevice(c->cfg.device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DecodeParams p;
  fill_decode(c, q, out, sel, p);
  mkv_status s;
  if ((s = timed(c, MKV_KERNEL_QROT, st, 1, [&] { return launch_qrot(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_SCORE, st, 1, [&] { return launch_score(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_TOPK, st, 1, [&] { return launch_topk(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_ATTN, st, 1, [&] { return launch_attn(p, st); })) != MKV_OK) return s;
  if ((s = timed(c, MKV_KERNEL_MERGE, st, 1, [&] { return launch_merge(p, st); })) != MKV_OK) return s;
  c->decode_calls += 1;
  return MKV_OK;
}

mkv_status mkv_decode_layers(mkv_ctx* const* ctxs, int n, const void* const* q, float* const* out,
                             int32_t* const* sel, mkv_stream_t stream) {
  if (!ctxs || !q || !out || n < 1 || n > MKV_MAX_FUSED_LAYERS) return MKV_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!ctxs[i] || !q[i] || !out[i]) return MKV_ERR_INVALID_ARG;
    for (int j = 0; j < i; ++j)
      if (ctxs[j] == ctxs[i]) {
        g_last_error = "mkv_decode_layers: a ctx appears twice";
        return MKV_ERR_INVALID_ARG;
      }
  }
  for (int i = 0; i < n; ++i)
    if (!ctxs[i]->ready) return MKV_ERR_STATE;
  mkv_ctx* c0 = ctxs[0];
  for (int i = 1; i < n; ++i) {
    const mkv_ctx* c = ctxs[i];
    if (c->cfg.device != c0->cfg.device || c->T != c0->T || c->T0 != c0->T0 ||
        c->n_commit != c0->n_commit || c->n_seg != c0->n_seg || c->cfg.c != c0->cfg.c ||
        c->cfg.segment != c0->cfg.segment || c->attn_per_fixed != c0->attn_per_fixed) {
      g_last_error = "mkv_decode_layers: the ctxs differ in device, shape or state";
      return MKV_ERR_INVALID_ARG;
    }
  }
  CK(cudaSetDevice(c0->cfg.device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  LayerParams lp;
  for (int i = 0; i < n; ++i) fill_decode(ctxs[i], q[i], out[i], sel ? sel[i] : nullptr, lp.p[i]);
  // every launch-shape field must agree with layer 0 (the launch uses p[0])
  const DecodeParams& a = lp.p[0];
  for (int i = 1; i < n; ++i) {
    const DecodeParams& b = lp.p[i];
    if (b.B != a.B || b.H != a.H || b.Hq != a.Hq || b.g != a.g || b.T != a.T || b.Tp != a.Tp ||
        b.S != a.S || b.c != a.c || b.n_seg != a.n_seg || b.kk != a.kk || b.T0 != a.T0 ||
        b.T_packed != a.T_packed || b.nseg0 != a.nseg0 || b.G != a.G ||
        b.stage_bytes != a.stage_bytes || b.n_stages != a.n_stages || b.sel_R != a.sel_R ||
        b.attn_mp != a.attn_mp || b.at_ki != a.at_ki || b.at_vi != a.at_vi) {
      g_last_error = "mkv_decode_layers: the ctxs differ in shape";
      return MKV_ERR_INVALID_ARG;
    }
  }
  // one attention shape for all layers: the widest per-token slot of any
  int kv = 0, vv = 0;
  for (int i = 0; i < n; ++i) {
    kv = std::max(kv, lp.p[i].at_kv);
    vv = std::max(vv, lp.p[i].at_vv);
  }
  int stages = a.at_stages, ctas = 1;
  CK(attn_shape(a.g, kv + a.at_ki + vv + a.at_vi, &stages, &ctas));
  for (int i = 0; i < n; ++i) {
    set_attn_shape(ctxs[i], lp.p[i], kv, vv, stages, ctas);
    lp.p[i].pdl = lp.p[0].pdl;
    lp.p[i].pdl_trigger = lp.p[0].pdl_trigger;
  }
  const DecodeParams& p = lp.p[0];
  CK(launch_qrot(p, st, &lp, n));
  CK(launch_score(p, st, &lp, n));
  CK(launch_topk(p, st, &lp, n));
  CK(launch_attn(p, st, &lp, n));
  CK(launch_merge(p, st, &lp, n));
  c0->launches += 5;
  for (int i = 0; i < n; ++i) ctxs[i]->decode_calls += 1;
  return MKV_OK;
}

}  // extern "C"

namespace {

// Moves the packed bytes and the tail to a larger pool when the next commit
// might not fit before the tail.  Synchronises the stream (decode kernels
// may still read the old pool).
mkv_status grow_pool(mkv_ctx* c, cudaStream_t st) {
  uint64_t end = 0;
  CK(cudaMemcpyAsync(&end, c->packed_end, sizeof(uint64_t), cudaMemcpyDeviceToHost, st));
  CK(cudaStreamSynchronize(st));
  c->packed_bound = end;
  const uint64_t worst = commit_worst(c);
  if (end + 256 + worst <= c->tail_off) return MKV_OK;
  const uint64_t tail_off = (end + 256 + 4 * worst + 255) & ~255ull;
  const uint64_t need = tail_off + c->tail_bytes;
  if (c->cfg.max_pool_bytes && need > c->cfg.max_pool_bytes) {
    g_last_error = "appended segments exceed max_pool_bytes";
    return MKV_ERR_OOM;
  }
  uint8_t* np = nullptr;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&np), need);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "cudaMalloc(pool)");
  }
  CK(cudaMemcpyAsync(np, c->pool, end, cudaMemcpyDeviceToDevice, st));
  CK(cudaMemcpyAsync(np + tail_off, c->pool + c->tail_off, c->tail_bytes, cudaMemcpyDeviceToDevice,
                     st));
  CK(cudaStreamSynchronize(st));
  CK(cudaFree(c->pool));
  c->pool = np;
  c->pool_cap = need;
  c->pool_need = need;
  c->tail_off = tail_off;
  return MKV_OK;
}

// Compresses the full tail (S tokens per stream) into one new segment per
// stream with the streams' bases, places the segments after the packed
// bytes, and switches to headers and score plans that include them.
mkv_status commit_tail(mkv_ctx* c, cudaStream_t st) {
  if (c->packed_bound + 256 + commit_worst(c) > c->tail_off) {
    mkv_status s = grow_pool(c, st);
    if (s != MKV_OK) return s;
  }
  const int stage = 1 - c->live;
  CompressParams p;
  memset(&p, 0, sizeof(p));
  p.X[0] = c->tail_x;
  p.X[1] = c->tail_x + (size_t)c->BH * c->cfg.segment * D;
  p.BH = c->BH;
  p.T = c->cfg.segment;
  p.S = c->cfg.segment;
  p.c = c->cfg.c;
  p.tau = c->cfg.tau;
  p.n_seg = 1;
  p.R = c->R[c->live];
  p.segs_per_cta = 1;
  p.ctas_per_stream = 1;
  p.seg = c->seg;
  p.tokmask = c->tokmask;
  p.colE = c->colE;
  p.segK = c->segK;
  p.hdr = c->hdr_commit;
  p.pool = c->pool;
  p.pool_check = c->check_override ? std::min(c->check_override, c->tail_off) : c->tail_off;
  p.err = c->err;
  p.packed_end = c->packed_end;
  p.bitmask_pv = (c->cfg.flags & MKV_FLAG_BITMASK_PV) != 0u;
  CK(launch_analyze(p, st));
  CK(launch_commit_scan(p, st));
  CK(launch_pack(p, st));
  CK(launch_grow_headers(c->hdr[c->live], c->n_seg, c->hdr_commit, 2 * c->BH, c->hdr[stage], st));
  CK(cudaMemcpyAsync(c->R[stage], c->R[c->live], 2 * (size_t)c->BH * D * D * sizeof(float),
                     cudaMemcpyDeviceToDevice, st));
  CK(cudaMemcpyAsync(c->lam[stage], c->lam[c->live], 2 * (size_t)c->BH * D * sizeof(float),
                     cudaMemcpyDeviceToDevice, st));
  CK(launch_partition(c->hdr[stage], c->BH, c->n_seg + 1, c->cfg.c, c->G, c->stage_bytes,
                      c->part[stage], c->cta_cnt[stage], c->plan[stage], c->plan_n[stage],
                      c->kprefix, st));
  c->launches += 7;
  c->live = stage;
  c->n_seg += 1;
  c->n_commit += 1;
  c->tail_len = 0;
  c->packed_bound += commit_worst(c);
  return MKV_OK;
}

}  // namespace

extern "C" {

mkv_status mkv_append(mkv_ctx* c, const void* k, const void* v, int32_t n, mkv_stream_t stream) {
  if (!c || !k || !v || n < 1) return MKV_ERR_INVALID_ARG;
  if (!c->ready) return MKV_ERR_STATE;
  if (c->T + n > c->cfg.max_ctx || c->tail_bytes == 0) {
    g_last_error = "mkv_append: the context would exceed max_ctx";
    return MKV_ERR_INVALID_ARG;
  }
  CK(cudaSetDevice(c->cfg.device));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int S = c->cfg.segment;
  int64_t first = 0;
  while (first < n) {
    const int take = (int)std::min<int64_t>(n - first, S - c->tail_len);
    AppendParams a;
    a.k = static_cast<const __half*>(k);
    a.v = static_cast<const __half*>(v);
    a.n_total = n;
    a.first = first;
    a.n = take;
    a.tail_len = c->tail_len;
    a.BH = c->BH;
    a.S = S;
    a.R = c->R[c->live];
    a.pool = c->pool;
    a.tail_k = c->tail_off;
    a.tail_v = c->tail_off + c->tail_bytes / 2;
    a.tail_x = c->tail_x;
    CK(launch_append(a, st));
    c->launches += 1;
    c->tail_len += take;
    c->T += take;
    first += take;
    if (c->tail_len == S) {
      mkv_status s = commit_tail(c, st);
      if (s != MKV_OK) return s;
    }
  }
  return MKV_OK;
}

mkv_status mkv_stats(const mkv_ctx* c, mkv_stats_t* out) {
  if (!c || !out) return MKV_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  out->pool_capacity = c->pool_cap;
  out->decode_calls = c->decode_calls;
  out->kernel_launches = c->launches;
  if (!c->ready) return MKV_OK;
  CK(cudaSetDevice(c->cfg.device));
  const size_t n = 2 * (size_t)c->BH * c->n_seg;
  std::vector<mkv_segment_header> h(n);
  CK(cudaMemcpy(h.data(), c->hdr[c->live], n * sizeof(mkv_segment_header), cudaMemcpyDeviceToHost));
  out->ctx_len = c->T;
  out->n_segments = c->n_seg;
  for (size_t i = 0; i < n; ++i) {
    const int x = (int)(i / ((size_t)c->BH * c->n_seg));
    const int st = h[i].strategy;
    if (st >= 0 && st < 4) out->strategy_count[x][st] += 1;
    out->payload_bytes[x] += segment_bytes(st, h[i].rows, c->cfg.c);
  }
  out->header_bytes = n * sizeof(mkv_segment_header);
  out->uncompressed_bytes = 2ull * c->BH * (uint64_t)c->T * D * 2ull;
  return MKV_OK;
}

mkv_status mkv_export(const mkv_ctx* c, int b, int h, int which, float* basis, float* eigvals,
                      mkv_segment_header* headers, void* payload, uint64_t* payload_bytes) {
  if (!c || !payload_bytes) return MKV_ERR_INVALID_ARG;
  if (b < 0 || b >= c->B || h < 0 || h >= c->H || which < 0 || which > 1) return MKV_ERR_INVALID_ARG;
  if (!c->ready) return MKV_ERR_STATE;
  CK(cudaSetDevice(c->cfg.device));
  CK(cudaDeviceSynchronize());
  const size_t sx = (size_t)which * c->BH + (size_t)b * c->H + h;
  if (basis)
    CK(cudaMemcpy(basis, c->R[c->live] + sx * D * D, D * D * sizeof(float), cudaMemcpyDeviceToHost));
  if (eigvals)
    CK(cudaMemcpy(eigvals, c->lam[c->live] + sx * D, D * sizeof(float), cudaMemcpyDeviceToHost));
  std::vector<mkv_segment_header> hd(c->n_seg);
  CK(cudaMemcpy(hd.data(), c->hdr[c->live] + sx * c->n_seg, c->n_seg * sizeof(mkv_segment_header),
                cudaMemcpyDeviceToHost));
  // the prefill segments are contiguous; each committed segment is exported
  // after them, in order
  const uint64_t first = (uint64_t)hd[0].off16 * 16u;
  const mkv_segment_header& last0 = hd[c->nseg0 - 1];
  const uint64_t end0 = (uint64_t)last0.off16 * 16u + segment_bytes(last0.strategy, last0.rows, c->cfg.c);
  uint64_t bytes = end0 - first;
  for (int i = c->nseg0; i < c->n_seg; ++i) bytes += segment_bytes(hd[i].strategy, hd[i].rows, c->cfg.c);
  if (payload) {
    if (*payload_bytes < bytes) {
      *payload_bytes = bytes;
      return MKV_ERR_INVALID_ARG;
    }
    uint8_t* out = static_cast<uint8_t*>(payload);
    CK(cudaMemcpy(out, c->pool + first, end0 - first, cudaMemcpyDeviceToHost));
    uint64_t at = end0 - first;
    for (int i = c->nseg0; i < c->n_seg; ++i) {
      const uint64_t sz = segment_bytes(hd[i].strategy, hd[i].rows, c->cfg.c);
      CK(cudaMemcpy(out + at, c->pool + (uint64_t)hd[i].off16 * 16u, sz, cudaMemcpyDeviceToHost));
      at += sz;
    }
  }
  *payload_bytes = bytes;
  if (headers) {
    uint64_t at = end0 - first;
    for (int i = 0; i < c->n_seg; ++i) {
      headers[i] = hd[i];
      if (i < c->nseg0) {
        headers[i].off16 = hd[i].off16 - (uint32_t)(first >> 4);
      } else {
        headers[i].off16 = (uint32_t)(at >> 4);
        at += segment_bytes(hd[i].strategy, hd[i].rows, c->cfg.c);
      }
    }
  }
  return MKV_OK;
}

mkv_status mkv_check_device(mkv_ctx* c) {
  if (!c) return MKV_ERR_INVALID_ARG;
  CK(cudaSetDevice(c->cfg.device));
  CK(cudaDeviceSynchronize());
  int v = 0;
  CK(cudaMemcpy(&v, c->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (v == 0) return MKV_OK;
  CK(cudaMemset(c->err, 0, sizeof(int)));
  if (v & DEV_ERR_CHECK) {
    g_last_error = (v & DEV_ERR_TIMEOUT)
                       ? "a pool access fell outside the checked extent; a bounded wait gave up"
                       : "a pool access fell outside the checked extent";
    return MKV_ERR_DEVICE_CHECK;
  }
  g_last_error = "a bounded device-side wait gave up";
  return MKV_ERR_TIMEOUT;
}

mkv_status mkv_set_flags(mkv_ctx* c, uint32_t flags) {
  if (!c || (flags & ~MKV_FLAGS_ALL)) return MKV_ERR_INVALID_ARG;
  c->cfg.flags = flags;
  return MKV_OK;
}

mkv_status mkv_debug_wait_test(mkv_ctx* c, uint64_t limit_ns, mkv_stream_t stream) {
  if (!c || limit_ns < 1000u || limit_ns > WAIT_LIMIT_NS) return MKV_ERR_INVALID_ARG;
  CK(cudaSetDevice(c->cfg.device));
  CK(launch_wait_test(c->err, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
  c->launches += 1;
  return MKV_OK;
}

mkv_status mkv_debug_set_pdl(mkv_ctx* c, uint32_t mask) {
  if (!c || (mask & ~0x11fu)) return MKV_ERR_INVALID_ARG;
  c->pdl_mask = mask;
  return MKV_OK;
}

mkv_status mkv_debug_set_check_extent(mkv_ctx* c, uint64_t bytes) {
  if (!c) return MKV_ERR_INVALID_ARG;
  c->check_override = bytes;
  return MKV_OK;
}

mkv_status mkv_kernel_time(mkv_ctx* c, int kernel_id, double* total_ms, int64_t* launches,
                           int reset) {
  if (!c || kernel_id < 0 || kernel_id >= MKV_KERNEL_COUNT) return MKV_ERR_INVALID_ARG;
  CK(cudaSetDevice(c->cfg.device));
  KernelTimer& t = c->timers[kernel_id];
  mkv_status s = resolve_timer(t, 0);
  if (s != MKV_OK) return s;
  if (total_ms) *total_ms = t.total_ms;
  if (launches) *launches = t.launches;
  if (reset) {
    t.total_ms = 0.0;
    t.launches = 0;
  }
  return MKV_OK;
}

mkv_status mkv_basis_static(const void* k, const void* v, int batch, int n_kv_heads,
                            int64_t ctx_len, float* basis, float* eigvals,
                            mkv_stream_t stream) {
  if (!k || !v || !basis || !eigvals) {
    g_last_error = "mkv_basis_static: NULL buffer";
    return MKV_ERR_INVALID_ARG;
  }
  if (batch < 1 || n_kv_heads < 1 || ctx_len < 1) {
    g_last_error = "mkv_basis_static: batch, n_kv_heads and ctx_len must be >= 1";
    return MKV_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15u) {
    g_last_error = "mkv_basis_static: k and v must be 16-byte aligned";
    return MKV_ERR_INVALID_ARG;
  }
  const int64_t streams = 2 * (int64_t)batch * n_kv_heads;
  if (streams > kBasisStaticParts) {
    char buf[256];
    snprintf(buf, sizeof(buf),
             "mkv_basis_static: 2*batch*n_kv_heads = %lld streams need at least %lld bytes of "
             "scratch; the static buffer holds %lld bytes (at most %lld streams)",
             (long long)streams, (long long)(streams * kGramPartBytes),
             (long long)MKV_BASIS_STATIC_MAX_BYTES, (long long)kBasisStaticParts);
    g_last_error = buf;
    return MKV_ERR_INVALID_ARG;
  }
  float* scratch = nullptr;
  mkv_status s = basis_scratch_here(&scratch);
  if (s != MKV_OK) return s;
  CompressParams p;
  memset(&p, 0, sizeof(p));
  p.X[0] = static_cast<const __half*>(k);
  p.X[1] = static_cast<const __half*>(v);
  p.BH = (int)(streams / 2);
  p.T = ctx_len;
  // mkv_compress's chunk count, reduced only when the partials would not fit
  p.gram_chunks = (int)std::min<int64_t>(gram_chunks_for(p.BH, ctx_len),
                                         kBasisStaticParts / streams);
  p.gram_chunk_tokens = ceil_div(ceil_div(ctx_len, p.gram_chunks), GRAM_TILE) * GRAM_TILE;
  p.gram_chunks = (int)ceil_div(ctx_len, p.gram_chunk_tokens);
  p.gram_part = scratch;
  p.R = basis;
  p.lam = eigvals;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CK(launch_gram(p, st));
  CK(launch_eig(p, st));
  return MKV_OK;
}

}  // extern "C"
