/*
 * mla.h -- C ABI of the GB300 (sm_103a) token-sparse MLA decode library.
 *
 * One operation, in three calls: the tile-scheduler metadata (computed once
 * before a decode loop), the sparse decode step itself, and the merge of
 * split-KV partial results.  Sources for what is computed (page title,
 * section):
 *   "flops/flashmla-decode-fp8-fp4-kv" -- "Arithmetic intensity" (the 528-byte
 *       FP8 and 288-byte FP4 token records, scales inlined in each record) and
 *       "Workarounds" (indices tensor (batch, seq_len_q, topk) of
 *       page_block*64+offset entries; metadata computed once before the decode
 *       loop; split decoding with num_splits);
 *   "deepseek-ai/FlashMLA" -- "How to use it" (metadata first, then one decode
 *       call per generation step; output plus log-sum-exp) and "Key technical
 *       details" (data followed by per-token scales; -1 entries ignored);
 *   "flops/attn-mla-kernel-support-matrix" -- "notes" (decode takes FP8 or
 *       FP4 caches only; bf16 KV is not supported).
 *
 * Conventions for every call:
 *   - Pointers named d_* and every tensor argument are DEVICE pointers; the
 *     problem descriptor and the *_out arguments are HOST pointers.
 *   - All tensors are dense, row-major, contiguous, owned by the caller; the
 *     library allocates nothing and keeps no state between calls except a
 *     per-device cache of the SM count.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns without synchronising the host.
 *   - The return status reports argument validation and launch errors only;
 *     on any status other than MLA_OK nothing was enqueued.  Problems found
 *     in device data are reported through the optional device error word.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* mla_stream_t; /* same type as cudaStream_t */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, inconsistent metadata size */
  MLA_ERR_UNSUPPORTED = 2,   /* a legal problem outside what the kernels implement */
  MLA_ERR_WORKSPACE = 3,     /* workspace smaller than mla_get_metadata reported */
  MLA_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
  MLA_ERR_TIMEOUT = 5        /* reserved for host-side waits; device timeouts use MLA_DEVERR_TIMEOUT */
} mla_status_t;

/* KV cache record formats ("Arithmetic intensity" of the FP8/FP4 KV page). */
enum {
  MLA_KV_NONE = 0,
  MLA_KV_FP8_528 = 1,  /* 512 B e4m3 (dim order) + 16 B e8m0 scales, one per 32 dims */
  MLA_KV_FP4_288 = 2,  /* 256 B e2m1 (even dim in the low nibble) + 32 B e4m3 scales, one per 16 dims */
  MLA_KV_BF16 = 3      /* named only to be rejected: decode does not take a bf16 cache */
};

/* Bits OR-ed into the optional device error word. */
enum {
  MLA_DEVERR_BAD_INDEX = 1,     /* an index was < -1 or >= num_pages*64; that entry was skipped */
  MLA_DEVERR_TIMEOUT = 2,       /* a bounded on-chip wait gave up; outputs are undefined */
  MLA_DEVERR_BAD_METADATA = 4   /* scheduler metadata inconsistent with the problem; work skipped */
};

#define MLA_HEAD_DIM 512
#define MLA_PAGE_SIZE 64
#define MLA_SCHED_INTS 8   /* int32 words per scheduler entry */

/* Problem descriptor (host memory). */
typedef struct {
  int32_t batch;           /* b >= 1 */
  int32_t seq_len_q;       /* s >= 1, query tokens per sequence (e.g. 2 for speculative decode) */
  int32_t h_q;             /* query heads: 16, 32, 64 or 128 */
  int32_t head_dim;        /* must be 512 (the shared latent width) */
  int32_t num_kv_heads;    /* must be 1: one latent vector per token serves every head as K and V */
  int32_t topk;            /* main indices per query token, >= 1 */
  int32_t extra_topk;      /* extra-cache indices per query token; 0 = no extra cache */
  int64_t num_pages;       /* pages in the main pool (bounds check of indices) */
  int64_t extra_num_pages; /* pages in the extra pool */
  int32_t page_size;       /* must be 64 */
  int32_t kv_format;       /* must be MLA_KV_FP8_528 */
  int32_t extra_kv_format; /* MLA_KV_FP4_288 when extra_topk > 0, else MLA_KV_NONE */
  float sm_scale;          /* softmax scale applied to q.k, e.g. 1/sqrt(512) */
} mla_problem_t;

/*
 * Tile-scheduler metadata, computed once before a decode loop
 * ("Workarounds": "Tile-scheduler metadata computed once before the decode
 * loop rather than per step"; "How to use it", step 3).
 *
 * Work is the list of (query token, tile) pairs, a tile being up to 128
 * consecutive index slots of one query token (main slots first, then extra
 * slots).  The list is cut into num_parts contiguous, balanced parts, one per
 * CTA group; a query token whose tiles fall into several parts is decoded as
 * several splits that are merged afterwards ("Split decoding with
 * num_splits").  The partition depends only on the problem shape and the SM
 * count, never on index values, so one result serves every step.
 *
 *   num_sms              SMs to plan for; 0 = query the current device.
 *   d_sched              device int32[num_parts][MLA_SCHED_INTS], written.
 *   d_num_splits         device int32[batch*seq_len_q + 1], written: the
 *                        exclusive prefix of per-query split counts.
 *   num_parts_out        host, required: number of parts.
 *   workspace_bytes_out  host, required: bytes of device workspace that
 *                        mla_sparse_decode needs for split partials.
 * Query mode: with d_sched == NULL and d_num_splits == NULL only the two
 * host outputs are filled and nothing is enqueued.
 */
mla_status_t mla_get_metadata(const mla_problem_t* problem, int32_t num_sms,
                              int32_t* d_sched, int32_t* d_num_splits,
                              int32_t* num_parts_out, size_t* workspace_bytes_out,
                              mla_stream_t stream);

/*
 * One sparse decode step ("How to use it", step 3; "Arithmetic intensity";
 * "Workarounds").  For every query token (b, s) and head h, over the tokens
 * T named by the valid entries of indices[b][s][:] (main cache) and
 * extra_indices[b][s][:] (extra cache), each token t contributing its decoded
 * 512-dim latent k_t as both key and value:
 *     x_t = sm_scale * <q[b,s,h,:], k_t>
 *     lse[b,s,h] = ln sum_{t in T} exp(x_t)
 *     out[b,s,h,:] = sum_{t in T} exp(x_t - lse) * k_t      (rounded to bf16)
 * one softmax over main and extra tokens together.  With no valid token the
 * output is +0 and lse is -inf.
 *
 *   q              bf16 [batch][seq_len_q][h_q][512], 16-byte aligned.
 *   kv             uint8 [num_pages][64][528] FP8 records, 16-byte aligned.
 *   indices        int32 [batch][seq_len_q][topk]; entry = page*64 + offset,
 *                  -1 = skip.  Entries < -1 or >= num_pages*64 are skipped
 *                  and flagged (MLA_DEVERR_BAD_INDEX).
 *   extra_kv       uint8 [extra_num_pages][64][288] FP4 records, or NULL.
 *   extra_indices  int32 [batch][seq_len_q][extra_topk], or NULL.
 *   d_sched, d_num_splits, num_parts   from mla_get_metadata for this problem
 *                  (same shape fields and SM count).
 *   workspace      device scratch of at least workspace_bytes (the value
 *                  mla_get_metadata reported); contents need no initialisation.
 *   out            bf16 [batch][seq_len_q][h_q][512].
 *   lse            float [batch][seq_len_q][h_q], natural logarithm.
 *   d_error        device int32 or NULL; error bits are OR-ed into it (the
 *                  caller clears it).
 * Rejections: a main cache that is not MLA_KV_FP8_528 (an FP4 cache is valid
 * only as the extra cache, a bf16 cache not at all), head_dim != 512,
 * page_size != 64, num_kv_heads != 1, unsupported h_q -> MLA_ERR_UNSUPPORTED.
 * Split partials are merged by an internal launch of the combine kernel on
 * the same stream.  Calls that share a workspace must not overlap.
 * out and workspace must be 16-byte aligned (MLA_ERR_INVALID_ARG otherwise).
 * Alignment beyond the minimum: with q 32-byte aligned (any allocator's
 * default), the 128-head kernel loads the query rows in 32-byte pieces; at
 * 16 bytes it uses 16-byte pieces, with identical results.
 */
mla_status_t mla_sparse_decode(const mla_problem_t* problem,
                               const void* q, const void* kv, const int32_t* indices,
                               const void* extra_kv, const int32_t* extra_indices,
                               const int32_t* d_sched, const int32_t* d_num_splits, int32_t num_parts,
                               void* workspace, size_t workspace_bytes,
                               void* out, float* lse, int32_t* d_error,
                               mla_stream_t stream);

/*
 * The decode step with the fused output epilogue ("deepseek-ai/FlashMLA",
 * "What it is": the conjugate RoPE on the output side and the final cast to
 * FP8, outputs ready for a downstream FP8 einsum; "flops/attn-mla-kernel-
 * support-matrix", "notes": qk_rope_head_dim = 64).  Same inputs and LSE as
 * mla_sparse_decode; instead of the bf16 output, each (query token, head)
 * row is
 *   1. the attention output o (fp32, before any rounding),
 *   2. turned on its rotary part -- dims 448..511 as 32 interleaved pairs
 *      (448 + 2j, 449 + 2j) -- by the conjugate rotation: pair j by
 *      -pos * rope_theta^(-2j/64), (a, b) -> (a cos + b sin, b cos - a sin),
 *      pos = positions[b][s],
 *   3. cast to a 528-byte FP8 record in the cache's own format (512 E4M3FN
 *      bytes in dim order, then one e8m0 scale per 32 dims, the writer's
 *      rule: the least power of two 2^e with block amax * 2^-e <= 448, each
 *      value rounded to nearest even).
 *   positions   int32 [batch][seq_len_q] (device): each query token's position.
 *   rope_theta  the rotary base (> 1), e.g. 10000.
 *   out_fp8     uint8 [batch][seq_len_q][h_q][528] (device, 4-byte aligned).
 * The workspace must be at least what mla_get_metadata reports.  With 128
 * heads and no extra cache, the decode kernel writes the records of query
 * tokens that have one split itself and only tokens of several splits pass
 * through the workspace to the merge kernel (the same arithmetic either
 * way); for other shapes every query token's result passes through it on
 * its way to the epilogue in the merge kernel.  Rejections and errors as for
 * mla_sparse_decode; a null positions or out_fp8, or a theta that is not
 * finite and > 1, is MLA_ERR_INVALID_ARG.
 */
mla_status_t mla_sparse_decode_rope_fp8(const mla_problem_t* problem,
                                        const void* q, const void* kv, const int32_t* indices,
                                        const void* extra_kv, const int32_t* extra_indices,
                                        const int32_t* d_sched, const int32_t* d_num_splits, int32_t num_parts,
                                        void* workspace, size_t workspace_bytes,
                                        const int32_t* positions, float rope_theta,
                                        void* out_fp8, float* lse, int32_t* d_error,
                                        mla_stream_t stream);

/*
 * Merge of split-KV partial results ("Workarounds": split decoding with
 * num_splits).  For query token q its splits are
 * num_splits[q] .. num_splits[q+1]-1; split i of head h carries its own
 * normalised output o_partial[i][h][:] and its natural-log lse_partial[i][h]:
 *     L = ln sum_i exp(lse_i);   out = sum_i exp(lse_i - L) * o_i   (bf16)
 * Splits with lse = -inf weigh nothing; if all are -inf the result is +0 and
 * -inf.  A query token with one split is copied.
 *   d_num_splits  int32 [batch*seq_len_q + 1] prefix (device).
 *   o_partial     float [total_splits][h_q][512] (device).
 *   lse_partial   float [total_splits][h_q] (device).
 *   out, lse      as in mla_sparse_decode.
 */
mla_status_t mla_combine(const mla_problem_t* problem, const int32_t* d_num_splits,
                         const float* o_partial, const float* lse_partial,
                         void* out, float* lse, mla_stream_t stream);

/*
 * Dequantize whole cache records to bf16 with the decode kernel's own
 * in-register dequantization ("Arithmetic intensity": e4m3 x e8m0 per 32
 * dims for FP8; e2m1 x e4m3 per 16 dims for FP4).  Every decoded value is
 * exactly representable in bf16, so the result is exact.
 *   kv_format  MLA_KV_FP8_528 or MLA_KV_FP4_288.
 *   records    uint8 [n][528 or 288] (device, 16-byte aligned).
 *   out        bf16 [n][512] (device).
 */
mla_status_t mla_dequantize(int32_t kv_format, const void* records, int64_t n, void* out,
                            mla_stream_t stream);

/*
 * Decode without a caller-provided workspace.  The pages have no counterpart
 * to this entry point; it exists for callers that may not allocate device
 * memory at call time -- a plugin or hook inside another runtime that hands
 * it only input and output buffers, or a serving loop whose device memory is
 * all reserved up front by its own pool and which may not call cudaMalloc on
 * its per-step path.
 *
 * Same arguments and result as mla_sparse_decode minus the workspace: the
 * split partials go to a fixed array of MLA_NOALLOC_SCRATCH_BYTES that every
 * device loading this library holds until the process exits.  Every call
 * looks up that array's address on the current device (a host-side query, so
 * the address stays right after a device reset); the first lookup on a device
 * also loads the library's device code there, so make the first call before
 * any stream capture.  The problem is validated first (MLA_ERR_INVALID_ARG /
 * MLA_ERR_UNSUPPORTED as for mla_sparse_decode); then MLA_ERR_WORKSPACE, with
 * nothing enqueued, when the problem's workspace (the bytes mla_get_metadata
 * reports for it) exceeds MLA_NOALLOC_SCRATCH_BYTES.  All calls share the one
 * array: calls that overlap on the GPU race and must be serialised by the
 * caller (one stream).  Allocates nothing.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (128u * 1024u * 1024u)
mla_status_t mla_sparse_decode_noalloc(const mla_problem_t* problem,
                                       const void* q, const void* kv, const int32_t* indices,
                                       const void* extra_kv, const int32_t* extra_indices,
                                       const int32_t* d_sched, const int32_t* d_num_splits, int32_t num_parts,
                                       void* out, float* lse, int32_t* d_error,
                                       mla_stream_t stream);

/*
 * KV-cache writer: quantize new tokens' latents into records and store each
 * at its slot of the paged pool -- the step that fills the cache the decode
 * reads ("Arithmetic intensity": 528-byte FP8 records, e4m3 data plus one
 * e8m0 scale per 32 values; 288-byte FP4 records, e2m1 data with the even
 * index in the low nibble plus one e4m3 scale per 16 values).  Block scales:
 * FP8 uses 2^e for the least e with amax * 2^-e <= 448 (scale byte 127 + e;
 * 127 for an all-zero block; e clamped to [-127, 127]); FP4 uses amax / 6
 * rounded to E4M3FN (a zero scale stores all-zero data).  Every element rounds
 * to nearest, ties to even, saturating at the format's largest finite value.
 *   kv_format  MLA_KV_FP8_528 or MLA_KV_FP4_288.
 *   latents    bf16 [n][512] (device, 16-byte aligned), finite values.
 *   slots      int32 [n] (device): page * 64 + offset; -1 = skip.  Slots
 *              < -1 or >= num_pages * 64 are skipped and flagged
 *              (MLA_DEVERR_BAD_INDEX).
 *   pool       uint8 [num_pages][64][528 or 288] (device, 16-byte aligned);
 *              only the addressed records are written.  Two tokens with the
 *              same slot race.
 *   d_error    device int32 or NULL, as in mla_sparse_decode.
 */
mla_status_t mla_kv_write(int32_t kv_format, const void* latents, const int32_t* slots, int64_t n, void* pool,
                          int64_t num_pages, int32_t* d_error, mla_stream_t stream);

/* Static description of a status code. */
const char* mla_status_string(mla_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
