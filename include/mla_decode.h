/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) absorbed-form MLA split-KV decode.
 *
 * What the library computes (sources by page and section):
 *   - TileGym "mla_decoding_split_kv.py", _mla_decoding_split_kv.forward and the
 *     mla_decoding_split_kv entry point: per batch row and head, the absorbed query
 *     [q_nope (512) | q_pe (64)] is scored against each cached token [latent (512) |
 *     k_pe (64)]; softmax with an explicit sm_scale; V is the same token's latent part
 *     (the wrapper passes KV as both K and V).  The KV sequence is cut into splits, each
 *     split emits a partial output plus an fp32 log-sum-exp, and splitk_reduce combines
 *     them.
 *   - tokenspeed "tokenspeed_mla.py", CuteDSLMLABackend.forward_decode and the decode
 *     workspace notes at the top of that file: a paged cache [num_pages, page_size, 576]
 *     addressed through block_tables and seq_lens (seq_lens already count this step's
 *     q_len new tokens); page_size 32 or 64; the workspace holds
 *     B*H*q_len*splits*(512+1) fp32 values and needs no zero-initialisation.
 *   - metrale "kv_cache_mla.rs", mla_paged_decode_nvfp4 / mla_paged_decode_fp8: 576
 *     values per token; an NVFP4 page is the packed E2M1 data section followed by one
 *     E4M3 scale per 16 values; FP8 pages hold one E4M3 byte per value and a scalar scale.
 *     mla_paged_decode_fp8 also takes a sliding_window and nullable per-head fp32 sinks
 *     (mla_decode_ex below; the page names the arguments without defining them, so the
 *     reading used here is stated at mla_decode_ex).
 *
 * Conventions shared by every entry point:
 *   - All buffers belong to the caller.  The library never allocates or frees memory
 *     and never synchronises the host, except mla_decode_read_status (documented).
 *   - Device pointers must be 16-byte aligned; kv_cache must be 128-byte aligned.
 *   - Every argument is validated on the host before anything is enqueued; on any
 *     error nothing is launched and an mla_status_t error is returned.
 *   - Problems only visible on the device (a block-table entry outside [0, num_pages),
 *     seq_len above max_pages*page_size, seq_len below q_len, a bounded wait that ran
 *     out) set bits of a status word in the workspace instead of trapping; the affected
 *     tokens are skipped.  mla_decode_read_status returns the word.
 *   - All work is enqueued on `stream`; the call is safe to capture in a CUDA graph.
 *   - Thread safety: the library's mutable global state is a per-device cache of the
 *     SM count and of the kernel attributes, and (mla_decode_no_alloc only) a per-device
 *     cache of its scratch buffer's address, each filled once under a lock, plus that
 *     scratch buffer itself: one per device, shared by every mla_decode_no_alloc call, so
 *     those calls must be ordered by the caller (see mla_decode_no_alloc); and the
 *     small-call limit (an atomic value, see mla_decode_set_small_call_limit).  Every
 *     other entry point touches only the caller's buffers.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *mla_stream_t; /* == cudaStream_t; NULL = legacy default stream */

/* Storage formats of the cache (one 576-value token = 512 latent + 64 rope). */
typedef enum {
  MLA_KV_BF16 = 0,      /* [num_pages, page_size, 576] bf16 */
  MLA_KV_FP8_E4M3 = 1,  /* [num_pages, page_size, 576] E4M3 codes; value = e4m3 * kv_scale */
  MLA_KV_NVFP4 = 2      /* per page: page_size*288 bytes of E2M1 pairs (element 2j in the low
                           nibble of byte j, token-major), then page_size*36 E4M3 scales
                           (token-major, scale g covers elements 16g..16g+15);
                           page stride = page_size*324 bytes */
} mla_kv_dtype_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,          /* null / misaligned pointer, bad size or scale */
  MLA_ERR_UNSUPPORTED = 2,          /* valid but not built: H, page_size, q_len, B*q_len */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace_bytes below mla_decode_workspace_size */
  MLA_ERR_CUDA = 4,                 /* a CUDA runtime call failed (launch, query, copy) */
  MLA_ERR_DEVICE_STATUS = 5         /* mla_decode_read_status found device-side problems */
} mla_status_t;

/* Bits of the device status word (mla_decode_read_status). */
#define MLA_STATUS_PAGE_OUT_OF_RANGE 0x1u /* a block-table entry outside [0, num_pages) */
#define MLA_STATUS_SEQ_TOO_LONG 0x2u      /* seq_len > max_pages*page_size (clamped) */
#define MLA_STATUS_SEQ_LT_QLEN 0x4u       /* seq_len < q_len (early queries see nothing) */
#define MLA_STATUS_NEG_SEQ_LEN 0x8u       /* seq_len < 0 (treated as 0) */
#define MLA_STATUS_WAIT_TIMEOUT 0x10u     /* a bounded in-kernel wait gave up */
#define MLA_STATUS_Q_RANGE 0x20u          /* a non-finite q value (FP8/NVFP4 caches; the row is not finite) */
#define MLA_STATUS_SLOT_OUT_OF_RANGE 0x40u /* mla_kv_append: a location past the cache (skipped) */

/* Limits of this build. */
#define MLA_LATENT_DIM 512
#define MLA_ROPE_DIM 64
#define MLA_CACHE_DIM 576
#define MLA_MAX_HEADS 128   /* H must be a multiple of 16 in [16, 128] */
#define MLA_MAX_Q_LEN 8
#define MLA_MAX_UNITS 1024  /* B * q_len */

/* ABI version of this header (bumped on any incompatible change). */
int mla_decode_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *mla_status_string(mla_status_t status);

/*
 * Bytes of workspace mla_decode needs on the CURRENT device for this shape:
 * a 32 KB header (status word and the per-(b,i) split plan), then the split partials,
 * B*H*q_len*splits*(512+1)*4 bytes in the tokenspeed formula, with `splits` bounded by
 * the schedule: for num_splits == 0 at most 2 partials per scheduling worker overall
 * (workers = SM count / 2), for num_splits > 0 at most num_splits per (b, i).
 * Returns MLA_ERR_INVALID_ARG for non-positive sizes or a null `bytes`.
 */
mla_status_t mla_decode_workspace_size(int B, int q_len, int H, int num_splits, size_t *bytes);

/*
 * One decode step: out[b,i,h,:] = sum_t softmax_t(sm_scale*kv_scale_k * q[b,i,h].k_t) v_t,
 * lse[b,i,h] = natural log of sum_t exp(sm_scale * q[b,i,h].k_t) (scale included), over
 * the positions t < seq_lens[b] - q_len + i + 1 of request b (causal verify when q_len>1).
 *
 *   q_nope      [B, q_len, H, 512] bf16, contiguous (the absorbed latent query)
 *   q_pe        [B, q_len, H, 64]  bf16, contiguous (rope already applied)
 *   kv_cache    paged cache in kv_dtype's layout above, num_pages pages
 *   block_table [B, max_pages] int32: physical page of logical page j of request b;
 *               only entries below cdiv(seq_lens[b], page_size) are read
 *   seq_lens    [B] int32 on the device, including this step's q_len tokens
 *   sm_scale    softmax scale (finite); kv_scale: FP8 per-tensor scale (finite, > 0),
 *               ignored for the other formats.  The FP8 scale multiplies every stored
 *               value, so it applies to both the scores and the output.
 *   num_splits  0: the library picks the split of every request from the SM count and
 *               all seq_lens (read on the device): the tiles of all (b, i), each preceded
 *               by a fixed per-item cost, are cut into equal contiguous ranges, one per
 *               pair of SMs; > 0: every request is cut into at
 *               most num_splits ranges of roundup(cdiv(len, num_splits), 64) tokens.
 *   workspace   device scratch of workspace_bytes >= mla_decode_workspace_size(...);
 *               its contents need no initialisation and are overwritten.
 *   out         [B, q_len, H, 512] bf16;  lse: [B, q_len, H] fp32 (may be NULL)
 *   stream      the CUDA stream everything is enqueued on.
 *
 * Enqueues two kernels: the decode, and the split-K reduce (which waits for the decode by
 * programmatic dependent launch and also writes the status word).  The decode is the
 * tensor-core kernel, or, for a small bf16 call (see mla_decode_set_small_call_limit), a
 * CUDA-core kernel with the same results contract; with num_splits == 0 that kernel keeps
 * each (b, i) in one range.  No memset, no host synchronisation.  Host-detected errors
 * return before anything is enqueued.
 */
mla_status_t mla_decode(const void *q_nope, const void *q_pe, const void *kv_cache,
                        const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                        int B, int q_len, int H, int num_pages, int page_size, float sm_scale,
                        int kv_dtype, float kv_scale, int num_splits, void *workspace,
                        size_t workspace_bytes, void *out, float *lse, mla_stream_t stream);

/*
 * mla_decode with a sliding window and per-head attention sinks (metrale "kv_cache_mla.rs",
 * mla_paged_decode_fp8, arguments sliding_window and sinks).  Every format is accepted.
 *
 *   window  0: no window.  W > 0: query i of request b attends only the last W of its
 *           visible positions, t in [max(0, V - W), V) with V = seq_lens[b] - q_len + i + 1.
 *   sinks   NULL: none.  Otherwise a device array [H] fp32: one extra logit per head, in
 *           the units of the scaled scores (sm_scale and kv_scale already applied), that
 *           joins the softmax normaliser but has no value row:
 *             lse = log( sum_t exp(x_t) + exp(sinks[h]) ),  out = sum_t exp(x_t - lse) v_t.
 *           -inf means "no sink" for that head; a (b, i) with nothing visible gets out 0
 *           and lse = sinks[h].  Values are read on the device and not validated.
 *
 * num_splits > 0 cuts the window's tiles (64-token tiles from the one holding its first
 * position) into at most num_splits ranges of cdiv(tiles, num_splits) tiles.  Errors and
 * everything else as mla_decode; a negative window or a misaligned sinks pointer is
 * MLA_ERR_INVALID_ARG.
 */
mla_status_t mla_decode_ex(const void *q_nope, const void *q_pe, const void *kv_cache,
                           const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                           int B, int q_len, int H, int num_pages, int page_size, float sm_scale,
                           int kv_dtype, float kv_scale, int num_splits, int window,
                           const float *sinks, void *workspace, size_t workspace_bytes, void *out,
                           float *lse, mla_stream_t stream);

/*
 * Small calls.  A bf16 call whose key ranges span at most `limit` cache positions each
 * (max_pages*page_size; with num_splits > 0, roundup(cdiv(max_pages*page_size,
 * num_splits), 64)), and whose (b, i, range, head) CTAs fit in one wave (at most the SM
 * count), runs its decode on the CUDA cores: the tensor-core kernel's pipeline set-up
 * (~9 us before its first P.V) is longer than such a call's whole work.  Results: as the tensor-core
 * kernel's, to rounding (fp32 throughout, P not rounded to bf16); the forced-split
 * partials and the plan in the workspace follow the same layout.  Sets the limit (0:
 * never) for the calls enqueued after it returns, from any thread; returns the previous
 * limit.  Default: MLA_SMALL_CALL_DEFAULT positions.
 */
#define MLA_SMALL_CALL_DEFAULT 256u
size_t mla_decode_set_small_call_limit(size_t limit);

/*
 * The split-K combine on its own (TileGym splitk_reduce): for every (b, i) whose KV range
 * the last mla_decode on this workspace cut into several splits,
 *   lse = M + log sum_s exp(lse_s - M),  M = max_s lse_s,
 *   out = bf16( sum_s exp(lse_s - lse) * o_s );
 * all splits empty -> out 0, lse -inf.  (b, i) with nothing visible also get 0 / -inf;
 * unsplit (b, i) were written by the decode kernel and are left alone.  With `sinks`
 * (device [H] fp32 or NULL, as in mla_decode_ex) the sink joins the combined normaliser,
 * and (b, i) with nothing visible get lse = sinks[h]; pass the decode's own sinks.
 * mla_decode already enqueues this; it is exported for tests and for callers that run
 * the decode kernel and the combine on different schedules.  Same shapes as mla_decode.
 */
mla_status_t mla_splitk_reduce(const void *workspace, size_t workspace_bytes, int B, int q_len,
                               int H, const float *sinks, void *out, float *lse, mla_stream_t stream);

/*
 * Copies the device status word of the last mla_decode on `workspace` to *device_status,
 * waiting for `stream` to finish (this call synchronises the host with the stream).
 * Returns MLA_ERR_DEVICE_STATUS when any bit is set, MLA_OK otherwise.
 */
mla_status_t mla_decode_read_status(const void *workspace, uint32_t *device_status,
                                    mla_stream_t stream);

/*
 * Number of scheduling workers the decode uses on the current device (host-side query,
 * for tests and sizing): one worker per pair of SMs that can be co-resident.
 */
mla_status_t mla_decode_num_workers(int *workers);

/*
 * Host copy of the device schedule, for tests: for the given seq_lens (HOST array), fills
 * per (b, i) unit: its first position in the schedule (num_splits == 0: the first of its
 * 4 + tiles balancing slots, 4 standing for the fixed cost of a work item; num_splits > 0:
 * its first item), tile count, number of parts and first partial slot
 * (-1 when the unit is written directly); returns the number of partial slots used.
 * Arrays have B*q_len entries.  `window` as in mla_decode_ex (tile counts then start at
 * the window's first tile).  `workers` <= 0 means the current device's worker count.
 */
mla_status_t mla_decode_plan_host(const int32_t *seq_lens, int B, int q_len, int max_pages,
                                  int page_size, int num_splits, int window, int workers,
                                  int32_t *unit_tile_begin, int32_t *unit_tiles,
                                  int32_t *unit_parts, int32_t *unit_slot, int32_t *slots_used);

/*
 * KV-cache append with quantise-on-write: stores this step's new tokens into the paged
 * cache before a decode reads them (tokenspeed "tokenspeed_mla.py", forward_decode, which
 * writes k[..., :512] and k[..., 512:] at out_cache_loc; metrale "kv_cache_mla.rs",
 * mla_cache_assemble and the page layouts of the paged decode launchers).
 *
 *   latent      [T] rows of 512 bf16, row t at latent + t*latent_stride (elements)
 *   rope        [T] rows of 64 bf16, row t at rope + t*rope_stride (elements); both pointers
 *               16-byte aligned and both strides multiples of 8 (e.g. the two halves of
 *               one [T, 576] tensor: rope = latent + 512, strides 576)
 *   slots       [T] int64 device array: flat cache location page*page_size + row of token
 *               t; negative = padding (skipped); >= num_pages*page_size is skipped and
 *               sets MLA_STATUS_SLOT_OUT_OF_RANGE in *device_status.  Locations must be
 *               distinct (two tokens for one location race).
 *   kv_cache    the paged cache in kv_dtype's layout (mla_kv_dtype_t), num_pages pages,
 *               page_size 32 or 64, 128-byte aligned
 *   kv_dtype    bf16: values stored unchanged.  FP8: code = E4M3(x / kv_scale) (finite
 *               kv_scale > 0).  NVFP4: per 16 values s = E4M3(amax / 6) and codes =
 *               E2M1(x / value(s)), zero codes when value(s) is 0.  Quotients are fp32;
 *               rounding is to nearest, ties to even, saturating (+-448 / +-6); a result
 *               that rounds to zero keeps the sign of its input.  Inputs must be finite.
 *   device_status  device uint32 that out-of-range locations OR a bit into (may be NULL;
 *               never cleared by this call)
 *
 * Enqueues one kernel on `stream`; T == 0 enqueues nothing.  Host-detected errors (null or
 * misaligned pointers, bad strides, sizes, format or scale) return before anything is
 * enqueued.
 */
mla_status_t mla_kv_append(const void *latent, int64_t latent_stride, const void *rope,
                           int64_t rope_stride, const int64_t *slots, int T, void *kv_cache,
                           int num_pages, int page_size, int kv_dtype, float kv_scale,
                           uint32_t *device_status, mla_stream_t stream);

/*
 * Per-head batched projection, one launch over all heads (metrale "kv_cache_mla.rs",
 * mla_batched_gemv: output[head, n] = sum_k weight[head, n, k] * input[head, k], BF16),
 * batched over T tokens:
 *
 *   out[t, h, n] = bf16( sum_k weight[h, n, k] * x[t, h, k] ),  fp32 accumulation.
 *
 * In absorbed MLA it is both steps around the decode: Q absorption (x = q_nope [T, H, 128],
 * weight = W_UK^T per head [H, 512, 128], out = the decode's q_nope input [T, H, 512]) and
 * V up-projection (x = the decode's out [T, H, 512], weight = W_UV [H, 128, 512]).
 *
 *   x       bf16, element (t, h, k) at x + t*x_token_stride + h*x_head_stride + k
 *   weight  bf16 [H, N, K] contiguous
 *   out     bf16, element (t, h, n) at out + t*out_token_stride + h*out_head_stride + n
 *   Device pointers 16-byte aligned; x strides multiples of 8 with x_head_stride >= K and
 *   x_token_stride >= H*x_head_stride; K a multiple of 8; T >= 0, H, N, K >= 1.
 *   device_status: optional device uint32 that a bounded wait that gave up ORs
 *   MLA_STATUS_WAIT_TIMEOUT into (never cleared by this call).
 *
 * Enqueues one kernel on `stream` (T == 0: nothing).  Host-detected errors return before
 * anything is enqueued.
 */
mla_status_t mla_batched_gemv(const void *x, int64_t x_token_stride, int64_t x_head_stride,
                              const void *weight, void *out, int64_t out_token_stride,
                              int64_t out_head_stride, int T, int H, int N, int K,
                              uint32_t *device_status, mla_stream_t stream);

/*
 * mla_decode_no_alloc -- mla_decode for callers that cannot allocate device memory.
 * The source pages have no counterpart to this entry point; it exists for users of this
 * library whose code may not call cudaMalloc: for example a plugin or callback that runs
 * inside another runtime which owns every device allocation, or a process that must
 * keep its device footprint fixed after start-up and so cannot create a workspace.
 *
 * Same arguments and results as mla_decode, minus the workspace: the scratch is a
 * file-scope static device buffer of MLA_NO_ALLOC_SCRATCH_BYTES inside this library.
 * Every GPU on which the library's no-alloc code is loaded holds that buffer until the
 * process exits.  No call allocates or frees memory.
 *   - The first call on each device looks up the buffer's device address with that
 *     device current; make that first call before any stream capture.
 *   - A shape whose workspace (mla_decode_workspace_size) exceeds
 *     MLA_NO_ALLOC_SCRATCH_BYTES returns MLA_ERR_WORKSPACE_TOO_SMALL; nothing is enqueued.
 *   - All calls on a device share the one buffer, which keeps the last call's contents;
 *     each call overwrites everything it reads (the status word included).  Calls
 *     that overlap on the GPU (other streams, other host threads) race on the buffer:
 *     the caller must order them.
 *   - *scratch_used (may be NULL) receives the buffer's device address, e.g. for
 *     mla_decode_read_status after the call.
 */
#define MLA_NO_ALLOC_SCRATCH_BYTES (48u << 20) /* 48 MiB per device */
mla_status_t mla_decode_no_alloc(const void *q_nope, const void *q_pe, const void *kv_cache,
                                 const int32_t *block_table, int max_pages, const int32_t *seq_lens,
                                 int B, int q_len, int H, int num_pages, int page_size,
                                 float sm_scale, int kv_dtype, float kv_scale, int num_splits,
                                 void *out, float *lse, mla_stream_t stream, void **scratch_used);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
