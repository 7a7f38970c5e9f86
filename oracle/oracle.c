/*
 * oracle.c -- plain, slow, fp64 CPU definition of token-sparse MLA decode
 * over a quantized paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness oracle that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant with the GPU library, and it does not include or link
 * anything from it.
 *
 * Sources (page title, section):
 *  [FMLA-KV]  "flops/flashmla-decode-fp8-fp4-kv", sections "Arithmetic
 *             intensity" (record formats) and "Workarounds" (indices tensor,
 *             split decoding).
 *  [FMLA-MAT] "flops/attn-mla-kernel-support-matrix", "Arithmetic intensity"
 *             (528/288-byte records).
 *  [FMLA-GH]  "deepseek-ai/FlashMLA", "Key technical details" (data followed
 *             by scales; -1 entries ignored) and "How to use it" (decode
 *             returns the output and the log-sum-exp).
 *
 * Everything is computed in double precision.  Readings of points the pages
 * leave open are stated at the function that takes them.
 *
 * Parity pins: every exported function here is pinned by the CPU test suite
 * (decoders against hand-built bytes and library float8 conversions,
 * encoders by round trips through the decoders, rounding ties, the scale
 * rule and the library float8 conversion,
 * attention against brute-force dense attention from a library routine and
 * closed forms, combine against the unsplit result).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D 512          /* latent width, [FMLA-KV] "head_dim 512" */
#define ORACLE_FP8_REC 528    /* 512 B e4m3 + 16 B e8m0, [FMLA-KV] */
#define ORACLE_FP4_REC 288    /* 256 B e2m1 + 32 B e4m3, [FMLA-KV] */

/* ------------------------------------------------------------------------ */
/* Element decoders (OCP microscaling element formats named by [FMLA-KV]).   */
/* ------------------------------------------------------------------------ */

/* float8_e4m3 read as E4M3FN: 1 sign, 4 exponent (bias 7), 3 mantissa bits,
 * no infinities; S.1111.111 is NaN.  The "fn" reading is the one whose range
 * (max 448) matches an amax/448 scale choice. */
double oracle_e4m3fn(uint8_t b) {
    int s = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);            /* subnormal */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);   /* normal */
    return s ? -v : v;
}

/* float8_e8m0: an unsigned power of two, 2^(b-127); 0xFF is NaN. */
double oracle_e8m0(uint8_t b) {
    if (b == 0xFF) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* e2m1 (4 bits): 1 sign, 2 exponent (bias 1), 1 mantissa bit. */
double oracle_e2m1(uint8_t nib) {
    int s = (nib >> 3) & 1;
    int e = (nib >> 1) & 0x3;
    int m = nib & 0x1;
    double v;
    if (e == 0)
        v = 0.5 * (double)m;                       /* 0 or 0.5 */
    else
        v = ldexp(1.0 + 0.5 * (double)m, e - 1);
    return s ? -v : v;
}

/* ------------------------------------------------------------------------ */
/* Token records.                                                            */
/* ------------------------------------------------------------------------ */

/* 528-byte record, [FMLA-KV] "Arithmetic intensity": 512 e4m3 bytes, one per
 * dim in dim order, followed by 16 e8m0 scales, one per 32 consecutive
 * values, in block order (scale j covers dims 32j..32j+31). */
void oracle_decode_fp8_record(const uint8_t* rec, double* k) {
    for (int j = 0; j < ORACLE_D; ++j)
        k[j] = oracle_e4m3fn(rec[j]) * oracle_e8m0(rec[ORACLE_D + j / 32]);
}

/* 288-byte record, [FMLA-KV] "Arithmetic intensity": 256 bytes holding two
 * e2m1 values each, the even index in the low nibble, followed by 32 e4m3
 * scales, one per 16 values (scale j covers dims 16j..16j+15). */
void oracle_decode_fp4_record(const uint8_t* rec, double* k) {
    for (int j = 0; j < ORACLE_D; ++j) {
        uint8_t byte = rec[j / 2];
        uint8_t nib = (j % 2 == 0) ? (uint8_t)(byte & 0xF) : (uint8_t)(byte >> 4);
        k[j] = oracle_e2m1(nib) * oracle_e4m3fn(rec[256 + j / 16]);
    }
}

void oracle_dequant_fp8(const uint8_t* recs, long long n, double* out) {
    for (long long t = 0; t < n; ++t)
        oracle_decode_fp8_record(recs + t * ORACLE_FP8_REC, out + t * ORACLE_D);
}

void oracle_dequant_fp4(const uint8_t* recs, long long n, double* out) {
    for (long long t = 0; t < n; ++t)
        oracle_decode_fp4_record(recs + t * ORACLE_FP4_REC, out + t * ORACLE_D);
}

/* ------------------------------------------------------------------------ */
/* Record encoders: the quantizer a KV-cache writer applies to a new latent  */
/* before it stores the record.  [FMLA-KV] "Arithmetic intensity" fixes the  */
/* formats and block sizes; how a block scale is chosen is this oracle's     */
/* reading, stated at each function: FP8 takes the smallest power-of-two     */
/* scale that brings the block maximum within 448 (the "amax/448" choice),   */
/* FP4 takes amax/6 rounded to E4M3FN.  Elements round to nearest, ties to   */
/* the even code, saturating at the largest finite value.                    */
/* ------------------------------------------------------------------------ */

/* Nearest E4M3FN byte to a finite x, ties to the even code, saturating at
 * +-448; found by scanning every finite code (the sign is kept, so -0.0 gives
 * 0x80). */
uint8_t oracle_e4m3fn_rne(double x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {            /* 0x7F is NaN */
        double d = fabs(oracle_e4m3fn((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* Nearest e2m1 nibble to a finite x, ties to the even code, saturating at
 * +-6, by the same scan. */
uint8_t oracle_e2m1_rne(double x) {
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double a = fabs(x);
    int best = 0;
    double best_d = INFINITY;
    for (int c = 0; c <= 0x7; ++c) {
        double d = fabs(oracle_e2m1((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | best);
}

/* 528-byte record from 512 finite values.  Per block of 32: e is the least
 * integer with amax * 2^-e <= 448 (0 for an all-zero block), clamped to
 * [-127, 127]; the scale byte is 127 + e; each value is x * 2^-e rounded to
 * E4M3FN. */
void oracle_encode_fp8_record(const double* x, uint8_t* rec) {
    for (int blk = 0; blk < ORACLE_D / 32; ++blk) {
        const double* xb = x + 32 * blk;
        double amax = 0.0;
        for (int j = 0; j < 32; ++j) amax = fmax(amax, fabs(xb[j]));
        int e = 0;
        if (amax > 0.0) {
            int E;
            frexp(amax, &E);                       /* amax = f 2^E, f in [0.5, 1) */
            e = E - 10;                            /* amax 2^-e >= 2^9 > 448 */
            while (ldexp(amax, -e) > 448.0) ++e;
        }
        if (e < -127) e = -127;
        if (e > 127) e = 127;
        rec[ORACLE_D + blk] = (uint8_t)(127 + e);
        for (int j = 0; j < 32; ++j) rec[32 * blk + j] = oracle_e4m3fn_rne(ldexp(xb[j], -e));
    }
}

/* 288-byte record from 512 finite values.  Per block of 16: the scale is
 * amax / 6 rounded to E4M3FN; each value is x / scale rounded to e2m1 (all
 * +0 when the scale rounds to zero); value 2k goes to the low nibble of byte
 * k. */
void oracle_encode_fp4_record(const double* x, uint8_t* rec) {
    uint8_t codes[ORACLE_D];
    for (int blk = 0; blk < ORACLE_D / 16; ++blk) {
        const double* xb = x + 16 * blk;
        double amax = 0.0;
        for (int j = 0; j < 16; ++j) amax = fmax(amax, fabs(xb[j]));
        uint8_t sc = oracle_e4m3fn_rne(amax / 6.0);
        double s = oracle_e4m3fn(sc);
        rec[256 + blk] = sc;
        for (int j = 0; j < 16; ++j) codes[16 * blk + j] = s == 0.0 ? 0 : oracle_e2m1_rne(xb[j] / s);
    }
    for (int k = 0; k < 256; ++k) rec[k] = (uint8_t)(codes[2 * k] | (codes[2 * k + 1] << 4));
}

void oracle_encode_fp8(const double* x, long long n, uint8_t* recs) {
    for (long long t = 0; t < n; ++t) oracle_encode_fp8_record(x + t * ORACLE_D, recs + t * ORACLE_FP8_REC);
}

void oracle_encode_fp4(const double* x, long long n, uint8_t* recs) {
    for (long long t = 0; t < n; ++t) oracle_encode_fp4_record(x + t * ORACLE_D, recs + t * ORACLE_FP4_REC);
}

/* ------------------------------------------------------------------------ */
/* bfloat16                                                                  */
/* ------------------------------------------------------------------------ */

double oracle_bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double once, to nearest with ties to even, onto the bfloat16 grid
 * (8 significant bits, exponent range of binary32, subnormals kept).  This is
 * done directly from the double: going through float first would round
 * twice. */
uint16_t oracle_bf16_rne(double x) {
    if (isnan(x)) return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs(x);
    uint16_t sign = neg ? 0x8000 : 0;
    if (isinf(a)) return (uint16_t)(sign | 0x7F80);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int E = e - 1;                /* a = (1.xxx) * 2^E */
    if (E < -126) E = -126;       /* subnormal range shares the quantum */
    double quantum = ldexp(1.0, E - 7);
    double n = nearbyint(a / quantum);   /* default mode: ties to even */
    double r = n * quantum;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float rf = (float)r;          /* exact: r lies on the bfloat16 grid */
    uint32_t u;
    memcpy(&u, &rf, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

void oracle_bf16_rne_array(const double* x, long long n, uint16_t* out) {
    for (long long i = 0; i < n; ++i) out[i] = oracle_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Sparse attention over the selected tokens of one query token.             */
/* ------------------------------------------------------------------------ */

/* Index semantics, [FMLA-KV] "Workarounds" and [FMLA-GH] "Key technical
 * details": an entry names one token of the paged pool as
 * page_block * 64 + offset, so with pages packed [num_pages][64][record] the
 * record sits at byte entry * record_size from the pool base.  -1 means
 * "ignore".  Any other negative entry, or one at or beyond num_pages * 64, is
 * outside the contract: it is skipped here too and counted. */
static int index_ok(int32_t i, long long pool_tokens) {
    return i >= 0 && (long long)i < pool_tokens;
}

/*
 * Token-sparse MLA decode, fp64.
 *
 * For each query token (b, s) the selected set is the multiset of valid main
 * entries plus the valid extra entries; every selected token contributes its
 * decoded latent k_t both as key and as value (one latent per token shared by
 * all heads).  For each head h:
 *     x_t  = sm_scale * <q[b,s,h,:], k_t>
 *     lse  = log sum_t exp(x_t)                  (natural logarithm)
 *     o[:] = sum_t exp(x_t - lse) * k_t[:]
 * Main and extra tokens share one softmax.  With no selected token the
 * output is +0 and lse is -inf.
 *
 * q:         bf16 bit patterns [b][s][h][512], consumed exactly.
 * kv:        FP8 records [pool_tokens][528].
 * idx:       int32 [b][s][topk].
 * extra_kv:  FP4 records [extra_pool_tokens][288], or NULL with extra_topk 0.
 * extra_idx: int32 [b][s][extra_topk].
 * out_bf16:  [b][s][h][512], the output rounded once to bfloat16 (may be NULL).
 * out_f64:   [b][s][h][512], the unrounded output (may be NULL).
 * lse:       [b][s][h] (may be NULL).
 * Returns the number of index entries outside the contract (skipped).
 */
long long oracle_sparse_mla_decode(
    int batch, int seq_len_q, int h_q, int topk, int extra_topk,
    long long pool_tokens, long long extra_pool_tokens, float sm_scale,
    const uint16_t* q, const uint8_t* kv, const int32_t* idx,
    const uint8_t* extra_kv, const int32_t* extra_idx,
    uint16_t* out_bf16, double* out_f64, double* lse)
{
    long long bad = 0;
    const double scale = (double)sm_scale;   /* the same binary32 value the GPU gets */
    const int nq = batch * seq_len_q;
    for (int qi = 0; qi < nq; ++qi) {
        const int32_t* ids = idx + (long long)qi * topk;
        const int32_t* xids = extra_topk > 0 ? extra_idx + (long long)qi * extra_topk : NULL;

        /* Collect the selected tokens of this query token. */
        int n = 0;
        for (int t = 0; t < topk; ++t) {
            if (ids[t] == -1) continue;
            if (!index_ok(ids[t], pool_tokens)) { ++bad; continue; }
            ++n;
        }
        for (int t = 0; t < extra_topk; ++t) {
            if (xids[t] == -1) continue;
            if (!index_ok(xids[t], extra_pool_tokens)) { ++bad; continue; }
            ++n;
        }

        double* K = n > 0 ? (double*)malloc((size_t)n * ORACLE_D * sizeof(double)) : NULL;
        long long* src = n > 0 ? (long long*)malloc((size_t)n * sizeof(long long)) : NULL;
        int* is_extra = n > 0 ? (int*)malloc((size_t)n * sizeof(int)) : NULL;
        int m = 0;
        for (int t = 0; t < topk; ++t)
            if (ids[t] != -1 && index_ok(ids[t], pool_tokens)) { src[m] = ids[t]; is_extra[m] = 0; ++m; }
        for (int t = 0; t < extra_topk; ++t)
            if (xids[t] != -1 && index_ok(xids[t], extra_pool_tokens)) { src[m] = xids[t]; is_extra[m] = 1; ++m; }

        /* Decode each selected record once; the decoded values are exact, so
         * reusing them for every head changes no result. */
        #pragma omp parallel for schedule(static)
        for (int t = 0; t < n; ++t) {
            if (is_extra[t])
                oracle_decode_fp4_record(extra_kv + src[t] * ORACLE_FP4_REC, K + (long long)t * ORACLE_D);
            else
                oracle_decode_fp8_record(kv + src[t] * ORACLE_FP8_REC, K + (long long)t * ORACLE_D);
        }

        #pragma omp parallel for schedule(dynamic, 1)
        for (int h = 0; h < h_q; ++h) {
            const long long row = (long long)qi * h_q + h;
            const uint16_t* qh = q + row * ORACLE_D;
            double qd[ORACLE_D];
            for (int d = 0; d < ORACLE_D; ++d) qd[d] = oracle_bf16_to_double(qh[d]);
            double o[ORACLE_D];
            double L;
            if (n == 0) {
                for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
                L = -INFINITY;
            } else {
                double* x = (double*)malloc((size_t)n * sizeof(double));
                double M = -INFINITY;
                for (int t = 0; t < n; ++t) {
                    const double* kt = K + (long long)t * ORACLE_D;
                    double acc = 0.0;
                    for (int d = 0; d < ORACLE_D; ++d) acc += qd[d] * kt[d];
                    x[t] = scale * acc;
                    if (x[t] > M) M = x[t];
                }
                double Z = 0.0;
                for (int t = 0; t < n; ++t) Z += exp(x[t] - M);
                L = M + log(Z);
                for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
                for (int t = 0; t < n; ++t) {
                    const double w = exp(x[t] - L);
                    const double* kt = K + (long long)t * ORACLE_D;
                    for (int d = 0; d < ORACLE_D; ++d) o[d] += w * kt[d];
                }
                free(x);
            }
            for (int d = 0; d < ORACLE_D; ++d) {
                if (out_bf16) out_bf16[row * ORACLE_D + d] = oracle_bf16_rne(o[d]);
                if (out_f64) out_f64[row * ORACLE_D + d] = o[d];
            }
            if (lse) lse[row] = L;
        }
        free(K);
        free(src);
        free(is_extra);
    }
    return bad;
}

/*
 * Merge of split results ([FMLA-KV] "Workarounds": split decoding with
 * num_splits).  Each split i of one query head carries its normalised
 * output o_i (softmax over its own tokens) and its lse_i.  Over the union:
 *     L   = log sum_i exp(lse_i)
 *     out = sum_i exp(lse_i - L) * o_i
 * A split with lse_i = -inf carries no tokens and weighs nothing; if every
 * split is empty the result is 0 and -inf.
 *
 * o_part: [n_splits][rows][512], lse_part: [n_splits][rows];
 * out: [rows][512], lse: [rows].
 */
void oracle_combine(int n_splits, long long rows, const double* o_part, const double* lse_part,
                    double* out, double* lse)
{
    for (long long r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int i = 0; i < n_splits; ++i)
            if (lse_part[(long long)i * rows + r] > M) M = lse_part[(long long)i * rows + r];
        double* o = out + r * ORACLE_D;
        for (int d = 0; d < ORACLE_D; ++d) o[d] = 0.0;
        if (M == -INFINITY) { lse[r] = -INFINITY; continue; }
        double Z = 0.0;
        for (int i = 0; i < n_splits; ++i) Z += exp(lse_part[(long long)i * rows + r] - M);
        const double L = M + log(Z);
        for (int i = 0; i < n_splits; ++i) {
            const double li = lse_part[(long long)i * rows + r];
            if (li == -INFINITY) continue;
            const double w = exp(li - L);
            const double* oi = o_part + ((long long)i * rows + r) * ORACLE_D;
            for (int d = 0; d < ORACLE_D; ++d) o[d] += w * oi[d];
        }
        lse[r] = L;
    }
}

/* ------------------------------------------------------------------------ */
/* Output-side epilogue of the fused kernel.                                 */
/* ------------------------------------------------------------------------ */

/* "deepseek-ai/FlashMLA", "What it is": the fused kernel ends with the
 * conjugate RoPE on the output side and the cast to FP8 (outputs ready for a
 * downstream FP8 einsum); "flops/attn-mla-kernel-support-matrix", "notes":
 * qk_rope_head_dim = 64.  Readings (the pages fix none of them): the rotary
 * part is the last 64 of the 512 output dims, taken as 32 interleaved pairs
 * (448 + 2j, 449 + 2j); pair j of a row at position pos turns by
 * phi_j = pos * theta^(-2j/64); a rotation by sign * phi_j maps (a, b) to
 * (a cos - b sin, a sin + b cos) of that angle, and the output side applies
 * the conjugate one (sign = -1).  pos holds one position per row.  Dims
 * below 448 are not touched. */
void oracle_rope_rotate(double* x, long long rows, const int32_t* pos, double theta, int sign) {
    for (long long r = 0; r < rows; ++r) {
        double* v = x + r * ORACLE_D;
        for (int j = 0; j < 32; ++j) {
            const double phi = (double)sign * (double)pos[r] * pow(theta, -2.0 * j / 64.0);
            const double c = cos(phi), s = sin(phi);
            const double a = v[448 + 2 * j], b = v[449 + 2 * j];
            v[448 + 2 * j] = a * c - b * s;
            v[449 + 2 * j] = a * s + b * c;
        }
    }
}

/* The epilogue: each row of o (the attention output, unrounded) turned by
 * the conjugate rotation, then cast to FP8 as a 528-byte record in the
 * cache's own format with the writer's block-scale rule (the FP8 einsum's
 * block scales: one e8m0 scale per 32 values, a reading). */
void oracle_rope_fp8_epilogue(const double* o, long long rows, const int32_t* pos, double theta, uint8_t* recs) {
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < rows; ++r) {
        double x[ORACLE_D];
        memcpy(x, o + r * ORACLE_D, sizeof(x));
        oracle_rope_rotate(x, 1, pos + r, theta, -1);
        oracle_encode_fp8_record(x, recs + r * ORACLE_FP8_REC);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
