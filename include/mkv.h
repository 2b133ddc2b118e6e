/*
 * mkv.h -- C ABI of the GB300 library for decode attention over a KV cache
 * compressed along both the sequence and the channel dimension.
 *
 * Method: "MosaicKV: Serving Long-Context LLM with Dynamic Two-D KV Cache
 * Compression" (arXiv 2607.00760), §1 Introduction:
 *   - "Observation & Method 1" (dynamic two-D compression): KV vectors are
 *     rotated into an SVD basis, important elements are picked per vector, and
 *     every fixed-size segment of the cache gets its own compression strategy.
 *   - "Observation & Method 2" (compressed KV cache management): the sparse KV
 *     matrix is packed into a dense format in GPU memory and attention runs on
 *     it, without unpacking, on CUDA cores.
 *   - prior-work paragraph: query-aware token selection (as in Quest) and a
 *     shared channel mask (as in ThinK).
 * The paper gives no interface; these calls follow its problem statement:
 * compress a prefill cache per KV head, then attend over it at every decode
 * step.
 *
 * Conventions for every call:
 *   - Pointers named "device" must point to memory of the ctx's CUDA device.
 *     Host pointers are plain host memory.  No call takes ownership of a
 *     caller pointer; inputs are read and outputs written in stream order on
 *     the given stream (they must stay valid until that work has run).
 *   - Every call returns an mkv_status.  On MKV_ERR_INVALID_ARG and
 *     MKV_ERR_OOM the ctx is left exactly as it was.  MKV_ERR_CUDA means a
 *     CUDA runtime call failed (the CUDA error is printed by
 *     mkv_last_error_string()).
 *   - A ctx is not thread-safe: calls on one ctx must not overlap.
 *   - No call allocates or frees memory other than what the ctx owns.
 *
 * Stream numbering: stream (b, h) of X in {K, V} is the T x 128 matrix
 * X[b][h][0:T][0:128].  Query head i belongs to KV head i / g, g = Hq / H.
 */
#ifndef MKV_H_
#define MKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* mkv_stream_t;

typedef enum {
  MKV_OK = 0,
  MKV_ERR_INVALID_ARG = 1,  /* bad pointer, size or config value */
  MKV_ERR_STATE = 2,        /* e.g. mkv_decode before any mkv_compress */
  MKV_ERR_OOM = 3,          /* device allocation failed or max_pool_bytes exceeded */
  MKV_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  MKV_ERR_DEVICE_CHECK = 5, /* a kernel's bounds check fired (see mkv_check_device) */
  MKV_ERR_TIMEOUT = 6       /* a bounded device-side wait gave up */
} mkv_status;

/* Per-segment strategies (§1 Observation & Method 1: "dynamic compression
 * strategy"; the set is this library's reading). */
enum {
  MKV_STRATEGY_SM = 0,    /* segment-shared mask of c channels */
  MKV_STRATEGY_PV = 1,    /* per-vector top-c channels (values + uint8 indices) */
  MKV_STRATEGY_DENSE = 2, /* all 128 channels */
  MKV_STRATEGY_PVB = 3    /* per-vector top-c channels (values + a 16-byte channel
                             bitmask per row); only with MKV_FLAG_BITMASK_PV */
};

#define MKV_HEAD_DIM 128
/* Record CUDA events around every decode kernel; read with mkv_kernel_time. */
#define MKV_FLAG_KERNEL_TIMING 1u
/* Record CUDA events around the score kernel only (fewer event records in a
 * captured step); read with mkv_kernel_time(ctx, MKV_KERNEL_SCORE, ...). */
#define MKV_FLAG_SCORE_TIMING 2u
/* Launch the decode kernels one after another without programmatic dependent
 * launch.  By default (and whenever no timing flag is set) the rotation,
 * score and attention kernels may start while the kernel before them is
 * finishing: their prologues (staging of ctx data, barrier set-up, the first
 * copies of packed keys) overlap that kernel's tail.  Timing flags imply this
 * flag, since an event between two kernels separates them. */
#define MKV_FLAG_NO_PDL 4u
/* Adds MKV_STRATEGY_PVB to the strategies mkv_compress (and the commits of
 * mkv_append) may choose: the per-vector channels of PV, encoded as a 16-byte
 * bitmask per row instead of c index bytes (cheaper whenever c > 16; on an
 * equal cost PV is kept).  A variant the paper leaves open ("a suitable
 * compression strategy" per segment). */
#define MKV_FLAG_BITMASK_PV 8u
#define MKV_FLAGS_ALL \
  (MKV_FLAG_KERNEL_TIMING | MKV_FLAG_SCORE_TIMING | MKV_FLAG_NO_PDL | MKV_FLAG_BITMASK_PV)

typedef struct {
  int32_t batch;          /* B >= 1 */
  int32_t n_kv_heads;     /* H >= 1 */
  int32_t n_q_heads;      /* Hq, a multiple of H; Hq / H <= 16 */
  int32_t head_dim;       /* must be 128 */
  int64_t max_ctx;        /* largest T that mkv_compress will accept, >= 1 */
  int32_t segment;        /* S: tokens per segment, 16..256, multiple of 16 */
  int32_t c;              /* kept channels per vector: 8..128, multiple of 8 */
  float tau;              /* retained-energy threshold, 0 < tau <= 1 */
  int32_t top_k;          /* tokens attended per KV head per step, >= 1 */
  int32_t attn_chunk;     /* split-K of the attention: selected tokens per slice.
                             0 = auto: the B * H * min(top_k, T) selected
                             positions are spread evenly over the resident
                             attention CTAs (at least 32 per slice); else
                             8..128 and a multiple of 8 (doubled while the
                             merge below would overflow).  A stream then has
                             at most ceil(min(top_k, max_ctx) / slice) + 1
                             slices; with g = Hq / H, slices * g must not
                             exceed 12288 (mkv_create: MKV_ERR_INVALID_ARG) */
  uint64_t max_pool_bytes;/* cap on the packed cache of one ctx; 0 = no cap */
  uint32_t flags;         /* MKV_FLAG_* */
  int32_t device;         /* CUDA device ordinal */
} mkv_config;

typedef struct mkv_ctx mkv_ctx;  /* one ctx = one attention layer */

/* Packed segment header, 8 bytes, one per segment of every stream.
 * off16: payload byte offset / 16 from the start of the ctx's packed pool
 * (in mkv_export: from the start of the exported stream payload). */
typedef struct {
  uint32_t off16;
  uint8_t strategy;
  uint8_t reserved;  /* 0 */
  uint16_t rows;     /* tokens in the segment: S, or T mod S for the last one */
} mkv_segment_header;

typedef struct {
  int64_t ctx_len;                 /* T of the current cache (0 if none) */
  int64_t n_segments;              /* per stream */
  int64_t strategy_count[2][4];    /* [K, V][SM, PV, DENSE, PVB] over all streams */
  uint64_t payload_bytes[2];       /* packed bytes of all K, all V streams */
  uint64_t header_bytes;           /* bytes of all segment headers */
  uint64_t uncompressed_bytes;     /* 2 * B * H * T * 128 * 2 */
  uint64_t pool_capacity;          /* bytes currently allocated for the pool */
  int64_t decode_calls;
  int64_t kernel_launches;         /* kernels launched by this ctx since creation */
} mkv_stats_t;

/* Kernel ids for mkv_kernel_time: the decode kernels, then (with
 * MKV_FLAG_KERNEL_TIMING) the compression steps. */
enum {
  MKV_KERNEL_QROT = 0,
  MKV_KERNEL_SCORE = 1,
  MKV_KERNEL_TOPK = 2,   /* the exact top-k selection */
  MKV_KERNEL_ATTN = 3,
  MKV_KERNEL_MERGE = 4,
  MKV_KERNEL_GRAM = 5,   /* G = X^T X partial sums */
  MKV_KERNEL_EIG = 6,    /* basis and eigenvalues */
  MKV_KERNEL_ANALYZE = 7,/* rotation, per-token channels, segment strategies */
  MKV_KERNEL_LAYOUT = 8, /* offsets, headers, score-kernel partition and plan */
  MKV_KERNEL_PACK = 9,   /* packed payload */
  MKV_KERNEL_COUNT = 10
};

/* Checks a config without touching any GPU.  MKV_OK or MKV_ERR_INVALID_ARG. */
mkv_status mkv_validate_config(const mkv_config* cfg);

/* Packed bytes of one segment with `rows` tokens (host-only, no GPU):
 *   SM:    pad16(c) + rows * 2c      (uint8 mask, then fp16 values per row)
 *   PV:    rows * 2c + pad16(rows*c) (fp16 values per row, then uint8 indices)
 *   DENSE: rows * 256
 *   PVB:   rows * 2c + rows * 16     (fp16 values per row, then a bitmask per
 *                                     row: bit j % 32 of little-endian word
 *                                     j / 32 for channel j)
 * Returns 0 for an invalid argument. */
uint64_t mkv_segment_bytes(int strategy, int rows, int c);

/* Creates a ctx for one layer: validates cfg, then allocates the fixed device
 * buffers (bases, headers, decode scratch).  The packed pool is allocated by
 * mkv_compress.  *out receives the ctx (NULL on failure). */
mkv_status mkv_create(const mkv_config* cfg, mkv_ctx** out);

/* Prefill compression (§1 Observation & Method 1).  For each stream of K and
 * of V: the SVD basis R (eigenvectors of X^T X, eigenvalues descending, each
 * column's largest-magnitude entry positive), x~ = x R, per-token top-c
 * channels by |x~| (ties to the lower channel), per-segment strategy = the
 * cheapest of {SM, PV, DENSE} whose retained energy fraction is >= tau
 * (DENSE always allowed; cost ties resolve SM, PV, DENSE), then packing
 * (values fp16 round-to-nearest-even, channels ascending).
 *   k, v: device fp16 [B][H][ctx_len][128], contiguous.
 *   ctx_len: 1 <= ctx_len <= max_ctx.
 * Replaces any previous cache.  The call blocks once, on `stream`, to read the
 * packed size back before allocating the pool; the final packing kernel is
 * still in flight on `stream` when it returns, so k and v must stay valid
 * until that stream's work has run, and decode must run on the same stream
 * (or after synchronising with it). */
mkv_status mkv_compress(mkv_ctx* ctx, const void* k, const void* v, int64_t ctx_len,
                        mkv_stream_t stream);

/* One decode step over the compressed cache (§1: query-aware token selection
 * and attention on the packed cache without unpacking).  Per KV head:
 * q~_i = q_i R_K; s_t = sum over the group of q~_i . k^_t; the min(top_k, T)
 * tokens with the highest s_t (ties to the lower token index); softmax of
 * q~_i . k^_t / sqrt(128) over them; o_i = (sum_t p_it v^_t) R_V^T.
 *   q:   device fp16 [B][Hq][128].
 *   out: device fp32 [B][Hq][128].
 *   sel: device int32 [B][H][min(top_k, T)] or NULL; receives the selected
 *        token ids in ascending order.
 * Fully asynchronous on `stream`; no host synchronisation, no allocation. */
mkv_status mkv_decode(mkv_ctx* ctx, const void* q, float* out, int32_t* sel,
                      mkv_stream_t stream);

/* Largest n of mkv_decode_layers. */
#define MKV_MAX_FUSED_LAYERS 64

/* mkv_decode of n ctxs (e.g. the attention layers of a model, or the layers
 * of several requests of one shape) with one launch of each decode kernel
 * over all of them, so that the GPU stays full between layers (an interface
 * addition with no counterpart in the paper).  The result for ctx i is
 * exactly (bit for bit) that of mkv_decode(ctxs[i], q[i], out[i], sel[i]).
 *   ctxs: host array of n distinct ctxs, all created with the same batch,
 *         heads, segment, c, top_k and device, and in the same state (same
 *         context length, the same number of appended tokens).
 *   q, out: host arrays of n device pointers, laid out as in mkv_decode.
 *   sel: NULL, or a host array of n device pointers (each may be NULL).
 *   1 <= n <= MKV_MAX_FUSED_LAYERS.
 * Asynchronous on `stream`; no host synchronisation, no allocation.  The
 * per-kernel timing flags do not apply (nothing is timed).
 * MKV_ERR_INVALID_ARG for NULL arrays or pointers, n out of range, a ctx
 * repeated, or ctxs whose shape or state differ (nothing is launched then);
 * MKV_ERR_STATE if a ctx has no compressed cache. */
mkv_status mkv_decode_layers(mkv_ctx* const* ctxs, int n, const void* const* q,
                             float* const* out, int32_t* const* sel, mkv_stream_t stream);

/* Replaces the ctx's MKV_FLAG_* bits (e.g. to time the kernels of a few
 * decode steps).  Host only; applies to later calls.  MKV_ERR_INVALID_ARG for
 * unknown bits. */
mkv_status mkv_set_flags(mkv_ctx* ctx, uint32_t flags);

/* Decode-time appends (§1 "Observation & Method 2": newly generated KV are
 * kept in a GPU-side buffer and used by the following decode steps; once a
 * segment's worth has accumulated it is compressed and switched into the
 * compressed cache without blocking decode).
 * Adds n tokens to every stream; they become tokens T .. T + n - 1 of later
 * decodes (T = prefill tokens + tokens appended so far).  Each token is
 * rotated into its stream's existing K / V basis and kept as an fp16 row with
 * every channel (a dense row) in a buffer of up to `segment` tokens per
 * stream.  Whenever the buffer is full its tokens are compressed as one
 * segment -- the stream's basis, the per-token top-c, the strategy rule and
 * the packing of mkv_compress -- and appended after the cache's segments
 * (a ragged last prefill segment stays as it is; committed segments start at
 * the prefill's end and hold `segment` tokens each).
 *   k, v: device fp16 [B][H][n][128], contiguous; read by the call's work on
 *         `stream`, so they must stay valid until it has run.
 *   n >= 1; the context after the call must not exceed max_ctx (room for
 *   appends exists only when mkv_compress was given fewer than max_ctx
 *   tokens).
 * Asynchronous on `stream`, no host synchronisation, except when a commit
 * might not fit the pool's spare room: the pool then grows once (one
 * synchronisation of `stream`, one allocation, a copy of the packed bytes).
 * Later decodes must run on the same stream or after it.  A new
 * mkv_compress drops all appended tokens.
 * MKV_ERR_STATE before any mkv_compress; MKV_ERR_INVALID_ARG for NULL
 * pointers, n < 1 or max_ctx exceeded (nothing is appended then). */
mkv_status mkv_append(mkv_ctx* ctx, const void* k, const void* v, int32_t n,
                      mkv_stream_t stream);

/* Frees everything the ctx owns.  NULL is allowed.  Synchronises the device. */
void mkv_free(mkv_ctx* ctx);

/* Static string for a status code. */
const char* mkv_status_string(mkv_status s);

/* Text of the last CUDA error seen by this library in the calling thread. */
const char* mkv_last_error_string(void);

/* Counters of the current cache (synchronous; copies headers to the host). */
mkv_status mkv_stats(const mkv_ctx* ctx, mkv_stats_t* out);

/* Copies one compressed stream to host buffers (synchronous).  Its segments
 * are the prefill's followed by those committed by mkv_append (n_segments
 * from mkv_stats); tokens still in the append buffer are not exported.
 *   which: 0 = K, 1 = V.
 *   basis:   host float[128*128] or NULL; R row-major, R[r*128 + j] = entry r of
 *            basis vector j.
 *   eigvals: host float[128] or NULL; descending.
 *   headers: host mkv_segment_header[n_segments] or NULL; off16 relative to
 *            the start of this stream's payload.
 *   payload: host buffer of *payload_bytes bytes or NULL.
 *   payload_bytes: in/out.  On entry the capacity of `payload` (ignored when
 *            payload is NULL); on return the stream's payload size.  A payload
 *            buffer smaller than the stream returns MKV_ERR_INVALID_ARG. */
mkv_status mkv_export(const mkv_ctx* ctx, int b, int h, int which, float* basis,
                      float* eigvals, mkv_segment_header* headers, void* payload,
                      uint64_t* payload_bytes);

/* Waits for all work on the ctx's device, then reports the ctx's device
 * status word since the last check (the word is then cleared):
 *   MKV_ERR_DEVICE_CHECK  a kernel found a packed-cache access that would end
 *                         past the checked pool extent (the live cache's
 *                         pool, or the smaller extent set with
 *                         mkv_debug_set_check_extent); it skipped that access
 *                         (decode reads a stand-in row, the score pass stops,
 *                         packing skips the row), so that call's outputs are
 *                         undefined;
 *   MKV_ERR_TIMEOUT       a kernel gave up a bounded device-side wait (about
 *                         two seconds of device time), abandoned the rest of
 *                         its work (outputs undefined) and returned;
 *   MKV_OK                neither.
 * Kernels never spin without a bound and never trap: the ctx stays usable. */
mkv_status mkv_check_device(mkv_ctx* ctx);

/* Test hooks for the failure detection above (interface additions with no
 * counterpart in the paper).  Neither can fault or hang the GPU.
 *
 * mkv_debug_wait_test: launches, on `stream`, one CTA that runs the library's
 * bounded mbarrier wait on a barrier no thread ever arrives on, with a limit
 * of limit_ns of device time (1000 <= limit_ns <= 2e9, else
 * MKV_ERR_INVALID_ARG).  When the limit runs out the kernel records a timeout
 * in the ctx's status word and returns; mkv_check_device then returns
 * MKV_ERR_TIMEOUT.  No other ctx state is touched.
 *
 * mkv_debug_set_check_extent: makes the kernels of later mkv_compress and
 * mkv_decode calls check packed-cache accesses against `bytes` instead of the
 * live pool's size when `bytes` is smaller (0 restores the pool's size).
 * Accesses are never allowed past the real pool: with a small `bytes`,
 * in-bounds accesses are reported as MKV_ERR_DEVICE_CHECK, which is how the
 * checks are tested without any out-of-bounds access. */
mkv_status mkv_debug_wait_test(mkv_ctx* ctx, uint64_t limit_ns, mkv_stream_t stream);

/* Measurement hook (no counterpart in the paper): which decode kernels are
 * launched with programmatic dependent launch when no flag disables it.  Bit
 * k (k = MKV_KERNEL_* id) enables it for kernel k; bit 8 keeps the kernels
 * from signalling early (the next kernel then starts when they end).
 * Default 0x03 (the rotation and score kernels).  Results do not
 * depend on it.  MKV_ERR_INVALID_ARG for other bits. */
mkv_status mkv_debug_set_pdl(mkv_ctx* ctx, uint32_t mask);
mkv_status mkv_debug_set_check_extent(mkv_ctx* ctx, uint64_t bytes);

/* With MKV_FLAG_KERNEL_TIMING: total device time (ms) and launch count of one
 * decode kernel id since creation or the last reset (synchronous).  reset != 0
 * clears the counters after reading them. */
mkv_status mkv_kernel_time(mkv_ctx* ctx, int kernel_id, double* total_ms,
                           int64_t* launches, int reset);

/* Size of the library's static device buffer used by mkv_basis_static. */
#define MKV_BASIS_STATIC_MAX_BYTES (16u << 20)

/* The basis step of mkv_compress alone, without a ctx and without allocating
 * any memory.  The paper has no counterpart of this call: it is an interface
 * addition of this library.
 *
 * Who it is for: callers that must not allocate device memory at the point of
 * the call, or that hold no ctx (mkv_create allocates a whole layer's buffers)
 * -- e.g. code whose device memory is all reserved by its framework's caching
 * allocator, where a cudaMalloc could fail or stall the device, and that wants
 * the per-stream bases of a prefill chunk (to inspect, calibrate or reuse).
 * The call itself performs no cudaMalloc, cudaFree or other allocating
 * routine: its scratch (the per-chunk partial Gram matrices, 64 KiB each) is a
 * file-scope static device array of MKV_BASIS_STATIC_MAX_BYTES (16 MiB) inside
 * the library.
 *
 * Result: the same as the bases and eigenvalues mkv_compress computes for the
 * same k, v (see mkv_compress and mkv_export for the definition and layout).
 * When 2 * batch * n_kv_heads * chunks * 64 KiB fits the buffer with the
 * number of Gram chunks mkv_compress would use, the summation order is the
 * same and so are the bits; otherwise fewer chunks are used and the results
 * agree to fp32 rounding.
 *   k, v:    device fp16 [batch][n_kv_heads][ctx_len][128], contiguous,
 *            16-byte aligned; only read.
 *   basis:   device float [2][batch * n_kv_heads][128][128] (K streams, then
 *            V streams); R[r*128 + j] = entry r of basis vector j.  Written.
 *   eigvals: device float [2][batch * n_kv_heads][128], descending.  Written.
 *   All four buffers belong to the caller; nothing is kept after the call.
 * Limits: 2 * batch * n_kv_heads <= 256 (one 64 KiB partial per stream must
 * fit the buffer); larger requests return MKV_ERR_INVALID_ARG before any CUDA
 * call, with the reason in mkv_last_error_string.  So do NULL pointers,
 * unaligned k or v, batch, n_kv_heads or ctx_len < 1.
 * Device: the calling thread's current CUDA device; k, v, basis, eigvals and
 * `stream` must all belong to it.  Every call looks the buffer's address up in
 * the current context (cudaGetSymbolAddress), so a device reset or a new
 * primary context is picked up.  The first call on each device may load the
 * library's device code there and reserve the buffer; make that first call
 * before any stream capture begins.  Each call then launches two kernels on
 * `stream` (asynchronous, no host synchronisation).
 * Nothing in the buffer needs to start at zero: every partial Gram matrix is
 * written in full before it is read.
 * The buffer is shared by every call on a device: calls that may overlap in
 * time (different streams, different host threads) race on it and give
 * undefined results.  Issue them on one stream, or order them with events. */
mkv_status mkv_basis_static(const void* k, const void* v, int batch, int n_kv_heads,
                            int64_t ctx_len, float* basis, float* eigvals,
                            mkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MKV_H_ */
