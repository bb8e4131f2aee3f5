/*
 * CPU oracle for DeepSeek V4.1 sparse latent attention -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the plain, slow, obviously-correct definition that the CUDA library is checked
 * against.  Only the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no source, header, table or helper with the CUDA path.
 *
 * Everything is written from the definitions on the source pages:
 *   [DOC]  "Module attn" API page (spark_model, deepseek_v41_ref/attn): the precision paragraph,
 *          the ring-cache paragraph, Constants: FP8_BLOCK, Functions: act_quant_inplace,
 *          pow2_ceil, sparse_attn, window_topk_idxs.
 *   [FWD]  "DeepSeek V4.1" attention page (attention/output, prefill): Attention.forward and
 *          Attention.__init__ (softmax_scale = head_dim ** -0.5, attn_sink per local head),
 *          apply_rotary_emb (the inverse rotation of the output's rope dims).
 *   [IDX]  "DeepSeek V4.1" source-layer attention page (indexer view), Indexer.forward: the
 *          selection that turns index scores into the compressed idx (visibility mask, top-k,
 *          position sort, -1 / offset).
 *   [CAND] the same indexer page, select_candidate_blocks: level one of the two-level top-k.
 *   [HC]   "DeepSeek V4.1" attention-write page (decode), hc_split_sinkhorn (and its kernel): a
 *          Hyper-Connections block's mixes split into pre / post weights and a
 *          Sinkhorn-normalised comb matrix.
 *
 * Floating point: dot products, the softmax and the weighted sum are carried in f64; the only
 * rounding to a narrow type is the final bf16 round-to-nearest-even of o.  The act_quant steps
 * are done in f32 exactly where the pages name f32 (amax / 448 and the power-of-two ceiling).
 * Compile with -ffp-contract=off so that no multiply-add is fused behind our back.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* bf16 and f32 bit views                                                                      */
/* ------------------------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) {
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* A bf16 value is the top half of an f32: widening is exact. */
double or_bf16_to_f64(uint16_t h) { return (double)f32_from_bits((uint32_t)h << 16); }

/*
 * Round an f64 to the nearest bf16, ties to even ([DOC] precision paragraph: sparse_attn
 * "returns bf16"; the rounding mode is read as IEEE round-to-nearest-even).
 *
 * bf16 carries 8 significant bits and the f32 exponent range, so a normal number x = m * 2^e
 * with 0.5 <= |m| < 1 is quantised in steps of 2^(e-8); below 2^-126 the subnormal step is
 * 2^-133.  nearbyint() in the default rounding mode resolves ties to the even integer, which is
 * the even last mantissa bit.
 */
uint16_t or_bf16_round(double x) {
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    if (isinf(x)) return signbit(x) ? 0xFF80 : 0x7F80;
    int e;
    (void)frexp(x, &e);
    int q = e - 8;
    if (q < -133) q = -133;
    double r = ldexp(nearbyint(ldexp(x, -q)), q);
    /* r is a bf16 value or overflows it; beyond the largest bf16 it becomes infinity */
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max) return signbit(x) ? 0xFF80 : 0x7F80;
    float f = (float)r; /* exact */
    uint16_t out = (uint16_t)(f32_bits(f) >> 16);
    if (r == 0.0 && signbit(x)) out = 0x8000;
    return out;
}

/* ------------------------------------------------------------------------------------------ */
/* fp8 e4m3 (the "fn" variant: no infinities, S.1111.111 is NaN, largest finite 448)           */
/* ------------------------------------------------------------------------------------------ */

/* Decode from the format definition: exponent bias 7, three mantissa bits. */
double or_e4m3_to_f64(uint8_t c) {
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9); /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(8.0 + m, e - 7 - 3); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/*
 * Encode an f32 to e4m3 with round-to-nearest-even and saturation to +-448 ([DOC]
 * act_quant_inplace: "values to e4m3 (RNE, clamped)").
 *
 * For |x| >= 2^-6 the e4m3 step inside the binade [2^k, 2^(k+1)) is 2^(k-3); below 2^-6 the
 * subnormal step is 2^-9.  Dividing by the step is exact (a power of two), nearbyint() rounds
 * ties to the even integer, which is the even mantissa, and a carry into the next binade lands
 * on its first value, which is representable.  Magnitudes above 448 after rounding clamp to 448.
 */
uint8_t or_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a == 0.0) return sign;
    double step;
    if (a < ldexp(1.0, -6)) {
        step = ldexp(1.0, -9);
    } else {
        int e;
        (void)frexp(a, &e); /* a = f * 2^e, 0.5 <= f < 1, so a is in [2^(e-1), 2^e) */
        step = ldexp(1.0, (e - 1) - 3);
    }
    double r = nearbyint(a / step) * step;
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    /* encode the (now representable) magnitude r */
    if (r < ldexp(1.0, -6)) {
        int m = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(sign | m);
    }
    int e;
    double f = frexp(r, &e); /* r = f * 2^e */
    int exp_field = (e - 1) + 7;
    int m = (int)((f * 2.0 - 1.0) * 8.0);
    return (uint8_t)(sign | (exp_field << 3) | m);
}

/* ------------------------------------------------------------------------------------------ */
/* pow2_ceil and act_quant                                                                     */
/* ------------------------------------------------------------------------------------------ */

/*
 * [DOC] pow2_ceil: 2 ** ceil(log2(v)) for positive normal f32, computed from the IEEE fields:
 * the unbiased exponent, plus one when any mantissa bit is set, becomes the exponent of a
 * mantissa-free result.
 */
float or_pow2_ceil(float v) {
    uint32_t bits = f32_bits(v);
    int32_t e = (int32_t)((bits >> 23) & 0xFF);
    uint32_t m = bits & 0x7FFFFF;
    int32_t exponent = e - 127 + (m != 0 ? 1 : 0);
    return f32_from_bits((uint32_t)(exponent + 127) << 23);
}

/*
 * [DOC] act_quant_inplace, Constants: FP8_BLOCK (= 32): for every block of 32 consecutive
 * elements along the last dimension of each row
 *   amax = max |x_k|, floored at 1e-4
 *   s    = pow2_ceil(amax / 448)                 (f32 division)
 *   y_k  = e4m3_rne_clamped(x_k / s)
 *   x'_k = bf16(y_k * s)                         (exact: e4m3 times a power of two fits bf16)
 * x is [n][d] bf16 bits with d % 32 == 0.  Any of the three outputs may be NULL: x_rt receives
 * the bf16 round trip, codes the e4m3 bytes and scales the e8m0 byte (log2(s) + 127) per block.
 */
int or_act_quant(const uint16_t* x, int64_t n, int64_t d, uint16_t* x_rt, uint8_t* codes,
                 uint8_t* scales) {
    if (d <= 0 || d % 32 != 0 || n < 0) return 1;
    for (int64_t r = 0; r < n; ++r) {
        for (int64_t blk = 0; blk < d / 32; ++blk) {
            const uint16_t* xb = x + r * d + blk * 32;
            float amax = 0.0f;
            for (int k = 0; k < 32; ++k) {
                float v = fabsf((float)or_bf16_to_f64(xb[k]));
                if (v > amax) amax = v;
            }
            const float floor_amax = 1e-4f;
            if (amax < floor_amax) amax = floor_amax;
            float s = or_pow2_ceil(amax / 448.0f);
            int log2s = (int)((f32_bits(s) >> 23) & 0xFF) - 127;
            if (scales) scales[r * (d / 32) + blk] = (uint8_t)(log2s + 127);
            for (int k = 0; k < 32; ++k) {
                float xv = (float)or_bf16_to_f64(xb[k]);
                uint8_t c = or_e4m3_encode(xv / s);
                if (codes) codes[r * d + blk * 32 + k] = c;
                if (x_rt) x_rt[r * d + blk * 32 + k] = or_bf16_round(or_e4m3_to_f64(c) * (double)s);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* window indices and the ring cache                                                            */
/* ------------------------------------------------------------------------------------------ */

/*
 * [DOC] window_topk_idxs and the ring-cache paragraph: a [seqlen][window] table of slot
 * indices, -1 where a slot holds nothing.
 *   prefill (start_pos == 0): query i sees the causal window of the chunk itself,
 *       column j -> position i - window + 1 + j, or -1 before position 0;
 *   decode (seqlen == 1 at position p): the whole ring, oldest first; column j holds position
 *       p - window + 1 + j, which lives in slot (that position) mod window, or -1 when that
 *       position is before 0.
 * Writes ld-strided rows (ld >= window) so the window part can sit in front of other columns.
 * Chunked prefill (start_pos > 0 with seqlen > 1) is not described on the pages: returns 2.
 */
int or_window_idxs(int64_t start_pos, int64_t seqlen, int64_t window, int32_t* idx, int64_t ld) {
    if (window <= 0 || seqlen < 0 || start_pos < 0 || ld < window) return 1;
    if (start_pos > 0 && seqlen != 1) return 2;
    for (int64_t i = 0; i < seqlen; ++i) {
        for (int64_t j = 0; j < window; ++j) {
            int32_t v;
            if (start_pos == 0) {
                int64_t pos = i - window + 1 + j;
                v = pos >= 0 ? (int32_t)pos : -1;
            } else {
                int64_t pos = start_pos - window + 1 + j;
                v = pos >= 0 ? (int32_t)(pos % window) : -1;
            }
            idx[i * ld + j] = v;
        }
    }
    return 0;
}

/* [DOC] ring-cache paragraph: token at position t is stored in slot t mod window; a later token
 * overwrites an earlier one in the same slot.  ring is [window][d], rows [seqlen][d]. */
int or_ring_write(uint16_t* ring, const uint16_t* rows, int64_t start_pos, int64_t seqlen,
                  int64_t window, int64_t d) {
    if (window <= 0 || seqlen < 0 || start_pos < 0 || d <= 0) return 1;
    for (int64_t t = 0; t < seqlen; ++t)
        memcpy(ring + ((start_pos + t) % window) * d, rows + t * d, (size_t)d * sizeof(uint16_t));
    return 0;
}

/* [FWD] apply_rotary_emb (and its use on the attention output, Attention.forward): the last
 * rope_dim elements of a row are read as rope_dim / 2 complex numbers x_{2k} + i x_{2k+1}; each is
 * multiplied by the rotation of the row's position, c_k + i s_k, or by its conjugate c_k - i s_k
 * (inverse), and written back as bf16.  The product is formed in f64 from the bf16 input and the
 * f32 table (the page forms it in f32), then rounded to bf16 (nearest even); the other elements
 * of the row are left as they are.
 *   x    [nrows][d] bf16, in place;  rot [npos][rope_dim / 2][2] f32 (c_k, s_k);  pos [nrows]
 *   x64  optional [nrows][rope_dim] f64: the unrounded rotated values
 * Returns 1 on a bad argument (odd or oversized rope_dim, a position outside the table). */
int or_rope(uint16_t* x, int64_t nrows, int64_t d, int64_t rope_dim, const float* rot,
            int64_t npos, const int64_t* pos, int inverse, double* x64) {
    if (rope_dim <= 0 || rope_dim % 2 || rope_dim > d || nrows < 0) return 1;
    const int64_t half = rope_dim / 2, base = d - rope_dim;
    for (int64_t r = 0; r < nrows; ++r) {
        if (pos[r] < 0 || pos[r] >= npos) return 1;
        for (int64_t k = 0; k < half; ++k) {
            const double a = or_bf16_to_f64(x[r * d + base + 2 * k]);
            const double b = or_bf16_to_f64(x[r * d + base + 2 * k + 1]);
            const double c = (double)rot[(pos[r] * half + k) * 2 + 0];
            const double sn = (inverse ? -1.0 : 1.0) * (double)rot[(pos[r] * half + k) * 2 + 1];
            /* (a + i b)(c + i sn) = (a c - b sn) + i (a sn + b c) */
            const double re = a * c - b * sn, im = a * sn + b * c;
            if (x64) {
                x64[r * rope_dim + 2 * k] = re;
                x64[r * rope_dim + 2 * k + 1] = im;
            }
            x[r * d + base + 2 * k] = or_bf16_round(re);
            x[r * d + base + 2 * k + 1] = or_bf16_round(im);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* sparse_attn                                                                                 */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    const uint16_t* q;    /* [b][s][h][d] bf16 */
    const uint16_t* kv;   /* [b][rows][d] bf16 (fmt 0) */
    const uint8_t* codes; /* [b][rows][d] e4m3 (fmt 1) */
    const uint8_t* scl;   /* [b][rows][d/32] e8m0 (fmt 1) */
    int fmt;
    const float* sink;    /* [h] */
    const int32_t* idx;   /* [b][s][topk] */
    float scale;
    int64_t b, s, h, d, rows, topk;
    const int64_t* tokens; /* flat token ids b*s + s to compute, or NULL for all */
    int64_t ntokens;
    uint16_t* o;   /* [ntokens][h][d] bf16 when tokens != NULL, else [b][s][h][d] */
    double* o64;   /* optional f64 copy, same layout as o */
    int nthreads;
    int64_t next; /* work counter */
    pthread_mutex_t lock;
} attn_job;

/* kv row j of sequence bi, widened to f64 (fp8 rows: e4m3 times 2^(e8m0 - 127)). */
static void load_kv_row(const attn_job* J, int64_t bi, int64_t j, double* out) {
    if (J->fmt == 0) {
        const uint16_t* r = J->kv + (bi * J->rows + j) * J->d;
        for (int64_t k = 0; k < J->d; ++k) out[k] = or_bf16_to_f64(r[k]);
    } else {
        const uint8_t* r = J->codes + (bi * J->rows + j) * J->d;
        const uint8_t* sc = J->scl + (bi * J->rows + j) * (J->d / 32);
        for (int64_t k = 0; k < J->d; ++k)
            out[k] = or_e4m3_to_f64(r[k]) * ldexp(1.0, (int)sc[k / 32] - 127);
    }
}

/*
 * One query token, all heads.  [DOC] sparse_attn: "per query and head, softmax over the gathered
 * rows plus the sink (denominator only), all in f32; output bf16"; [FWD] Attention.forward passes
 * one kv tensor that serves as both keys and values, and -1 marks an empty index slot.
 *   l_j = scale * <q_h, kv_j>                  for every listed j != -1 (repeats kept)
 *   m   = max(sink_h, max_j l_j)
 *   o_h = sum_j exp(l_j - m) kv_j / (exp(sink_h - m) + sum_j exp(l_j - m))
 * A token with no listed row gets o = 0.  Carried in f64 and rounded to bf16 at the end.
 */
static void attend_token(const attn_job* J, int64_t tok, int64_t out_row, double* kvbuf,
                         double* logit) {
    const int64_t bi = tok / J->s;
    const int32_t* ix = J->idx + tok * J->topk;
    int64_t nvalid = 0;
    for (int64_t t = 0; t < J->topk; ++t) {
        if (ix[t] == -1) continue;
        load_kv_row(J, bi, ix[t], kvbuf + nvalid * J->d);
        ++nvalid;
    }
    for (int64_t hh = 0; hh < J->h; ++hh) {
        const uint16_t* qh = J->q + (tok * J->h + hh) * J->d;
        uint16_t* oh = J->o + (out_row * J->h + hh) * J->d;
        double* oh64 = J->o64 ? J->o64 + (out_row * J->h + hh) * J->d : NULL;
        if (nvalid == 0) {
            for (int64_t k = 0; k < J->d; ++k) {
                oh[k] = 0;
                if (oh64) oh64[k] = 0.0;
            }
            continue;
        }
        double sink = (double)J->sink[hh];
        double m = sink;
        for (int64_t t = 0; t < nvalid; ++t) {
            const double* kr = kvbuf + t * J->d;
            double acc = 0.0;
            for (int64_t k = 0; k < J->d; ++k) acc += or_bf16_to_f64(qh[k]) * kr[k];
            logit[t] = (double)J->scale * acc;
            m = fmax(m, logit[t]); /* a sink of -inf drops out here and in exp(sink - m) */
        }
        double den = exp(sink - m);
        for (int64_t t = 0; t < nvalid; ++t) {
            logit[t] = exp(logit[t] - m); /* now the unnormalised weight */
            den += logit[t];
        }
        for (int64_t k = 0; k < J->d; ++k) {
            double acc = 0.0;
            for (int64_t t = 0; t < nvalid; ++t) acc += logit[t] * kvbuf[t * J->d + k];
            double v = acc / den;
            oh[k] = or_bf16_round(v);
            if (oh64) oh64[k] = v;
        }
    }
}

static void* attn_worker(void* arg) {
    attn_job* J = (attn_job*)arg;
    double* kvbuf = (double*)malloc((size_t)(J->topk > 0 ? J->topk : 1) * (size_t)J->d * sizeof(double));
    double* logit = (double*)malloc((size_t)(J->topk > 0 ? J->topk : 1) * sizeof(double));
    if (!kvbuf || !logit) {
        free(kvbuf);
        free(logit);
        return (void*)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= J->ntokens) break;
        int64_t tok = J->tokens ? J->tokens[w] : w;
        attend_token(J, tok, w, kvbuf, logit);
    }
    free(kvbuf);
    free(logit);
    return NULL;
}

/*
 * Returns 0 on success, 1 on a bad argument, 3 when an index is outside [-1, rows) (the pages
 * give no meaning to such an index; the oracle refuses it).
 */
int or_sparse_attn(const uint16_t* q, const uint16_t* kv, const uint8_t* codes, const uint8_t* scl,
                   int fmt, const float* sink, const int32_t* idx, float scale, int64_t b,
                   int64_t s, int64_t h, int64_t d, int64_t rows, int64_t topk,
                   const int64_t* tokens, int64_t ntokens, uint16_t* o, double* o64,
                   int nthreads) {
    if (b < 0 || s < 0 || h <= 0 || d <= 0 || rows < 0 || topk < 0 || !o || !sink || !q || !idx)
        return 1;
    if (fmt == 0 && !kv) return 1;
    if (fmt == 1 && (!codes || !scl || d % 32 != 0)) return 1;
    if (fmt != 0 && fmt != 1) return 1;
    if (!tokens) ntokens = b * s;
    for (int64_t w = 0; w < ntokens; ++w) {
        int64_t tok = tokens ? tokens[w] : w;
        if (tok < 0 || tok >= b * s) return 1;
        for (int64_t t = 0; t < topk; ++t) {
            int32_t j = idx[tok * topk + t];
            if (j < -1 || j >= rows) return 3;
        }
    }
    attn_job J;
    J.q = q; J.kv = kv; J.codes = codes; J.scl = scl; J.fmt = fmt; J.sink = sink; J.idx = idx;
    J.scale = scale; J.b = b; J.s = s; J.h = h; J.d = d; J.rows = rows; J.topk = topk;
    J.tokens = tokens; J.ntokens = ntokens; J.o = o; J.o64 = o64;
    J.nthreads = nthreads < 1 ? 1 : nthreads;
    J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)J.nthreads);
    int rc = 0;
    if (!th) return 1;
    for (int i = 0; i < J.nthreads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
    for (int i = 0; i < J.nthreads; ++i) {
        void* ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = 1;
    }
    free(th);
    pthread_mutex_destroy(&J.lock);
    return rc;
}

/* ------------------------------------------------------------------------------------------ */
/* array forms of the scalar codecs (plain loops, for the exhaustive checks)                   */
/* ------------------------------------------------------------------------------------------ */

void or_bf16_round_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_round(x[i]);
}

void or_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_encode(x[i]);
}

void or_e4m3_decode_array(const uint8_t* c, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_to_f64(c[i]);
}

void or_pow2_ceil_array(const float* x, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_pow2_ceil(x[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* [IDX] the indexer's selection                                                              */
/* ------------------------------------------------------------------------------------------ */

typedef struct {
    double v;
    int64_t pos;
} scored_pos;

/* higher score first; among equal scores the lower position first (the reading taken for the
 * page's topk, which leaves the order of ties open); -0 and +0 compare equal */
static int by_score_then_pos(const void* a, const void* b) {
    const scored_pos* x = (const scored_pos*)a;
    const scored_pos* y = (const scored_pos*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int by_value(const void* a, const void* b) {
    const int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/* [IDX] For every sequence bi and query si, over the n_comp = (start_pos + s) / ratio compressed
 * positions of score [b][s][n_comp]:
 *   visible = (si + 1) / ratio at a prefill (start_pos == 0), where every position t >= visible
 *             has its score replaced by -inf; n_comp at a decode step (no mask)
 *   k       = min(index_topk, n_comp)
 *   pick the k highest scores, sort the picked positions ascending, and write each as
 *   t + offset when t < visible, else -1, to idx [b][s][k].
 * Returns 1 on a bad argument, 2 for a chunked prefill (start_pos > 0 with s > 1), which the
 * page does not describe. */
int or_indexer_topk(const float* score, int64_t b, int64_t s, int64_t n_comp, int64_t start_pos,
                    int64_t ratio, int64_t index_topk, int64_t offset, int32_t* idx) {
    if (b < 0 || s < 0 || start_pos < 0 || ratio < 1 || index_topk < 0) return 1;
    if ((start_pos + s) / ratio != n_comp) return 1;
    if (start_pos > 0 && s > 1) return 2;
    const int64_t k = index_topk < n_comp ? index_topk : n_comp;
    if (b * s == 0 || k == 0) return 0;
    scored_pos* all = (scored_pos*)malloc((size_t)n_comp * sizeof *all);
    int64_t* pick = (int64_t*)malloc((size_t)k * sizeof *pick);
    if (!all || !pick) {
        free(all);
        free(pick);
        return 1;
    }
    for (int64_t bi = 0; bi < b; ++bi) {
        for (int64_t si = 0; si < s; ++si) {
            const float* row = score + (bi * s + si) * n_comp;
            const int64_t visible = start_pos == 0 ? (si + 1) / ratio : n_comp;
            for (int64_t t = 0; t < n_comp; ++t) {
                all[t].v = (start_pos == 0 && t >= visible) ? -INFINITY : (double)row[t];
                all[t].pos = t;
            }
            qsort(all, (size_t)n_comp, sizeof *all, by_score_then_pos);
            for (int64_t j = 0; j < k; ++j) pick[j] = all[j].pos;
            qsort(pick, (size_t)k, sizeof *pick, by_value);
            int32_t* out = idx + (bi * s + si) * k;
            for (int64_t j = 0; j < k; ++j)
                out[j] = pick[j] < visible ? (int32_t)(pick[j] + offset) : -1;
        }
    }
    free(all);
    free(pick);
    return 0;
}

/* [CAND] For every row r of logits [rows][width] whose query sees the first visible[r]
 * positions (positions at or past visible[r] count as -inf, as the page's caller has already
 * masked them):
 *   block j's score = the highest logit among positions j*block_size .. (j+1)*block_size - 1
 *                     (-inf past the row's end, the page's padding)
 *   the block holding position visible[r] - 1 (the newest one the query sees) scores +inf;
 *                     none when visible[r] == 0
 *   the min(topk_blocks, blocks) highest-scoring blocks are picked (ties: lower block first);
 *                     a pick whose score is -inf is dropped
 *   mask[r][t] = 1 when t's block was kept, else 0.
 * Returns 1 on a bad argument. */
int or_candidate_blocks(const float* logits, int64_t rows, int64_t width, const int64_t* visible,
                        int64_t topk_blocks, int64_t block_size, uint8_t* mask) {
    if (rows < 0 || width < 0 || topk_blocks < 0 || block_size < 1) return 1;
    if (rows == 0 || width == 0) return 0;
    const int64_t nb = (width + block_size - 1) / block_size;
    const int64_t k = topk_blocks < nb ? topk_blocks : nb;
    scored_pos* blk = (scored_pos*)malloc((size_t)nb * sizeof *blk);
    uint8_t* kept = (uint8_t*)malloc((size_t)nb);
    if (!blk || !kept) {
        free(blk);
        free(kept);
        return 1;
    }
    for (int64_t r = 0; r < rows; ++r) {
        if (visible[r] < 0 || visible[r] > width) {
            free(blk);
            free(kept);
            return 1;
        }
        const float* row = logits + r * width;
        for (int64_t j = 0; j < nb; ++j) {
            double best = -INFINITY;
            for (int64_t t = j * block_size; t < (j + 1) * block_size && t < width; ++t) {
                const double v = t < visible[r] ? (double)row[t] : -INFINITY;
                if (v > best) best = v;
            }
            blk[j].v = best;
            blk[j].pos = j;
        }
        if (visible[r] > 0) blk[(visible[r] - 1) / block_size].v = INFINITY;
        qsort(blk, (size_t)nb, sizeof *blk, by_score_then_pos);
        memset(kept, 0, (size_t)nb);
        for (int64_t j = 0; j < k; ++j)
            if (blk[j].v > -INFINITY) kept[blk[j].pos] = 1;
        for (int64_t t = 0; t < width; ++t) mask[r * width + t] = kept[t / block_size];
    }
    free(blk);
    free(kept);
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* [HC] hc_split_sinkhorn                                                                     */
/* ------------------------------------------------------------------------------------------ */

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* [HC] For every token i of mixes [n][(2 + hc) * hc], with scale [3] and base [(2 + hc) * hc]
 * (a_j = mixes[i][j] * scale[.] + base[j]):
 *   pre[i][j]  = sigmoid(a_j) + eps,  using scale[0], j < hc
 *   post[i][j] = 2 sigmoid(a_{hc + j}),  scale[1]
 *   comb[i]    = the hc x hc matrix a_{2 hc + j hc + k} (row j, column k),  scale[2];
 *                each row replaced by its softmax, plus eps;
 *                each column divided by (its sum + eps);
 *                then iters - 1 times: each row divided by (its sum + eps), then each column.
 * In f64 from the f32 inputs (the page works in f32).  Returns 1 on a bad argument. */
int or_hc_split_sinkhorn(const float* mixes, int64_t n, int64_t hc, const float* scale,
                         const float* base, int64_t iters, double eps, double* pre, double* post,
                         double* comb) {
    if (n < 0 || hc < 1 || hc > 16 || iters < 1) return 1;
    const int64_t mix = (2 + hc) * hc;
    double c[16][16];
    for (int64_t i = 0; i < n; ++i) {
        const float* m = mixes + i * mix;
        for (int64_t j = 0; j < hc; ++j) {
            pre[i * hc + j] = sigmoid((double)m[j] * scale[0] + base[j]) + eps;
            post[i * hc + j] = 2.0 * sigmoid((double)m[hc + j] * scale[1] + base[hc + j]);
        }
        for (int64_t j = 0; j < hc; ++j)
            for (int64_t k = 0; k < hc; ++k)
                c[j][k] = (double)m[2 * hc + j * hc + k] * scale[2] + base[2 * hc + j * hc + k];
        /* softmax along each row, plus eps */
        for (int64_t j = 0; j < hc; ++j) {
            double mx = c[j][0], sum = 0.0;
            for (int64_t k = 1; k < hc; ++k) mx = c[j][k] > mx ? c[j][k] : mx;
            for (int64_t k = 0; k < hc; ++k) {
                c[j][k] = exp(c[j][k] - mx);
                sum += c[j][k];
            }
            for (int64_t k = 0; k < hc; ++k) c[j][k] = c[j][k] / sum + eps;
        }
        for (int64_t it = 0; it < iters; ++it) {
            if (it > 0) { /* rows (the first round's row step is the softmax) */
                for (int64_t j = 0; j < hc; ++j) {
                    double sum = 0.0;
                    for (int64_t k = 0; k < hc; ++k) sum += c[j][k];
                    for (int64_t k = 0; k < hc; ++k) c[j][k] /= sum + eps;
                }
            }
            for (int64_t k = 0; k < hc; ++k) { /* columns */
                double sum = 0.0;
                for (int64_t j = 0; j < hc; ++j) sum += c[j][k];
                for (int64_t j = 0; j < hc; ++j) c[j][k] /= sum + eps;
            }
        }
        for (int64_t j = 0; j < hc; ++j)
            for (int64_t k = 0; k < hc; ++k) comb[(i * hc + j) * hc + k] = c[j][k];
    }
    return 0;
}
