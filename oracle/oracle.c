/*
 * oracle.c -- plain, slow CPU reference for the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The GPU product path
 * never calls it and shares no code with it (no headers, no tables, no
 * helpers): every codec here is written from its published definition.
 *
 * What the verify step computes (the three calls of one speculative round):
 *   1. append: the window's new K/V rows are written into a paged, quantised
 *      KV cache (FP8 E4M3 with one fp32 scale per (page, kv head), or INT4
 *      with one fp16 scale per group of 32 head dims of a token).
 *      Source: NInfer review (blog.123qwe.co.kr/?p=4624), section
 *      "성능과 평가" (performance records: FP8 E4M3 / INT8 group KV) and the
 *      example config with FP8 KV and max_context 240000 in section
 *      "설치·실행·서빙"; 4-bit KV from the MegaCapybara announcement, item 2.
 *   2. verify attention: every window row (1 + d tokens) attends causally
 *      inside the window, with GQA, over the lane's whole cached context.
 *      Source: Baseten talk summary, section "추측 디코드" (the main model
 *      checks all drafted tokens in one forward pass); NInfer review,
 *      section "아키텍처 ③" (draft counts 1..5 for MTP, 1..15 for DFlash).
 *   3. acceptance: the longest draft prefix that agrees with the target
 *      argmax; the bonus token is the argmax at the first disagreement.
 *      Source: same "추측 디코드" section; commit-after-accept from the
 *      NInfer review, section "아키텍처 ①".
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes with its reason):
 *   R1 FP8 is OCP E4M3 ("fn": no infinities, 0x7F/0xFF are NaN, max 448),
 *      encoded round-to-nearest-even with saturation to +-448.
 *   R2 FP8 scale per (page, kv head), separately for K and V: the scale only
 *      grows while a page fills; an append that starts at page offset 0 resets
 *      it; if it grows, the page's earlier tokens are re-encoded exactly as
 *      encode(fp32(decode(c) * s_old) / s_new).  Dequant = decode(c) * s.
 *   R3 INT4 is symmetric [-7, 7]: s = fp16_rne(min(amax / 7, 65504)),
 *      q = clamp(rint(x / s), -7, 7) with ties to even; dim 2i in the low
 *      nibble and dim 2i+1 in the high nibble, two's complement.
 *   R4 Append happens before attention; window keys are read back from the
 *      cache (quantised).  Window row i of lane b sees keys 0 .. L_b + i.
 *   R5 GQA grouping is contiguous: q head h uses kv head h / (Hq / Hkv).
 *   R6 Argmax ties go to the lowest index; NaN never wins; an all-NaN row
 *      gives 0; -0 and +0 compare equal.  drafts[i] is checked against the
 *      argmax of window position i; accept length a = leading matches; the
 *      commit adds 1 + a to the lane's length.
 *   R7 A lane may carry fewer drafts than the window holds (the draft count is
 *      chosen per workload, NInfer review section "아키텍처 ③"): with d_b
 *      drafts only drafts[b][0 .. d_b) are compared, and the rows after the
 *      first disagreement decide nothing, so the lazy form reports argmaxes
 *      only for rows 0 .. a and -1 after them.
 *   R10 INT8 group-64 KV (the NInfer review, section "성능과 평가", names
 *      "INT8 group-64" only): like R3 with 127 in place of 7 and groups of 64
 *      head dims: s = fp16_rne(min(amax / 127, 65504)), q = clamp(rint(x /
 *      s), -127, 127), halves to even, two's complement bytes.
 *   R11 FP8 E4M3 row KV (the same section names "FP8 E4M3 row-256" only;
 *      read as one scale per row of a token's head, 128 dims here): one fp32
 *      scale per (token, kv head) row, s = amax / 448, codes
 *      e4m3_rne_sat(x / s).
 *      Every token carries its own scale, so nothing is re-encoded.
 *   R9 Draft trees (a reading: the pages describe chains of drafts only):
 *      window slot 0 is the root (the last committed token) and slot i >= 1
 *      has a parent slot parent[i] < i; the window is appended in slot order
 *      as usual.  Row i attends to the context and to the window keys of its
 *      ancestors and itself.  Acceptance walks from the root: at node n it
 *      moves to the first child (in slot order) whose token is the argmax of
 *      row n; a = the nodes accepted, the bonus token = the argmax of the
 *      last node's row.
 *   R8 Lossless stochastic acceptance (DFlash2 keeps the draft model's
 *      conditional distribution q: NInfer review, section "아키텍처 ③"):
 *      p_i = softmax(logits row i) (temperature 1); draft i is accepted when
 *      u_i * q_i(x_i) < p_i(x_i); at the first rejection a, one token is drawn
 *      from max(0, p_a - q_a) normalised (from p_d when every draft is
 *      accepted) by the inverse CDF in index order at u_sample * Z: the
 *      smallest k whose running sum exceeds it, else the last k of positive
 *      weight; a residual of zero mass falls back to p_a.  The uniforms are
 *      inputs.  An out-of-vocabulary draft is a rejection and sets a status bit.
 *
 * Arithmetic: codecs in IEEE fp32 exactly as stated (compiled with
 * -ffp-contract=off, no fast-math); attention in fp64, two-pass softmax.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PAGE 64
#define HEAD_DIM 128
#define MAX_WINDOW 16

enum { ST_BAD_PAGE = 1, ST_OVERFLOW = 2, ST_BAD_DRAFT = 4, ST_BAD_COUNT = 16 };
enum { KV_FP8 = 0, KV_INT4 = 1, KV_INT8 = 2, KV_FP8_ROW = 3 };

/* ------------------------------------------------------------------ */
/* bf16 input values                                                    */
/* ------------------------------------------------------------------ */
static float bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------ */
/* OCP FP8 E4M3 (reading R1)                                            */
/* ------------------------------------------------------------------ */
/* value = (-1)^s * 2^(e-7) * (1 + m/8) for e > 0,
 *         (-1)^s * 2^(-6) * (m/8)      for e = 0,
 * e = 15, m = 7 is NaN. */
double oracle_e4m3_decode(uint8_t code)
{
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid, saturating to +-448. */
uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign;
    double a, q, k, v, f;
    int e;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    /* spacing of the grid at a: 2^-9 below 2^-6, else 2^(floor(log2 a) - 3) */
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
        q = ldexp(1.0, (e - 1) - 3);
    }
    k = nearbyint(a / q); /* a / q is exact; default mode is nearest-even */
    v = k * q;
    if (v > 448.0)
        v = 448.0;
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -6))
        return sign | (uint8_t)(v / ldexp(1.0, -9)); /* subnormal: m = v / 2^-9 */
    f = frexp(v, &e);                                /* v = f * 2^e */
    {
        int biased = (e - 1) + 7;
        int m = (int)((2.0 * f - 1.0) * 8.0);
        return sign | (uint8_t)(biased << 3) | (uint8_t)m;
    }
}

/* ------------------------------------------------------------------ */
/* IEEE binary16, round to nearest even (INT4 group scales, R3)        */
/* ------------------------------------------------------------------ */
double oracle_f16_decode(uint16_t h)
{
    int s = h >> 15;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 31)
        return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp(1.0 + (double)m / 1024.0, e - 15);
    return s ? -v : v;
}

uint16_t oracle_f16_encode(float x)
{
    uint16_t sign;
    double a, q, k, v, f;
    int e;
    if (isnan(x))
        return 0x7E00;
    sign = signbit(x) ? 0x8000 : 0;
    a = fabs((double)x);
    if (a < ldexp(1.0, -14)) {
        q = ldexp(1.0, -24);
    } else {
        frexp(a, &e);
        q = ldexp(1.0, (e - 1) - 10);
    }
    k = nearbyint(a / q);
    v = k * q;
    if (v >= 65536.0)
        return sign | 0x7C00; /* overflow to infinity */
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -14))
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    f = frexp(v, &e);
    {
        int biased = (e - 1) + 15;
        int m = (int)((2.0 * f - 1.0) * 1024.0);
        return sign | (uint16_t)(biased << 10) | (uint16_t)m;
    }
}

/* ------------------------------------------------------------------ */
/* INT4 group codec (R3)                                                */
/* ------------------------------------------------------------------ */
/* Quantise one group of n values symmetrically to [-qmax, qmax]; returns
 * the fp16 scale bits (R3 with qmax 7, R10 with qmax 127). */
static uint16_t int_group(const float* x, int n, int qmax, int8_t* codes)
{
    float amax = 0.0f, t, sf;
    uint16_t s16;
    int i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    t = amax / (float)qmax; /* IEEE fp32 division */
    if (t > 65504.0f)
        t = 65504.0f;
    s16 = oracle_f16_encode(t);
    sf = (float)oracle_f16_decode(s16);
    for (i = 0; i < n; ++i) {
        if (sf == 0.0f) {
            codes[i] = 0;
        } else {
            float r = x[i] / sf; /* IEEE fp32 division */
            double k = nearbyint((double)r);
            if (k > (double)qmax)
                k = (double)qmax;
            if (k < -(double)qmax)
                k = -(double)qmax;
            codes[i] = (int8_t)k;
        }
    }
    return s16;
}

/* Quantise one group of n values; returns the fp16 scale bits and writes
 * codes in [-7, 7]. */
uint16_t oracle_int4_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 7, codes); }

/* INT8 group codec (R10): codes in [-127, 127], fp16 scale. */
uint16_t oracle_int8_group(const float* x, int n, int8_t* codes) { return int_group(x, n, 127, codes); }

/* FP8 row codec (R11): one fp32 scale amax / 448 for the n values of a row;
 * codes e4m3(x / s) (round to nearest even, saturating); a zero scale gives
 * zero codes.  Returns the scale. */
float oracle_fp8_row(const float* x, int n, uint8_t* codes)
{
    float amax = 0.0f, s;
    int i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax)
            amax = a;
    }
    s = amax / 448.0f; /* IEEE fp32 division */
    for (i = 0; i < n; ++i)
        codes[i] = s == 0.0f ? 0x00 : oracle_e4m3_encode(x[i] / s);
    return s;
}

static int int4_nibble_value(uint8_t byte, int high)
{
    int v = high ? (byte >> 4) : (byte & 0xF);
    return v >= 8 ? v - 16 : v;
}

/* ------------------------------------------------------------------ */
/* The cache                                                            */
/* ------------------------------------------------------------------ */
typedef struct {
    int dtype; /* KV_FP8, KV_INT4, KV_INT8 or KV_FP8_ROW */
    int num_pages;
    int num_kv_heads;
    uint8_t* k_codes; /* FP8, INT8, FP8_ROW: [pages][Hkv][64][128]; INT4: [pages][Hkv][64][64] */
    uint8_t* v_codes;
    /* FP8: float [pages][Hkv]; INT4: uint16 (fp16) [pages][Hkv][64][4];
     * INT8: uint16 (fp16) [pages][Hkv][64][2]; FP8_ROW: float [pages][Hkv][64] */
    void* k_scales;
    void* v_scales;
} oracle_cache;

/* Lane check shared by all three cache-touching routines: the lane's token
 * range [lo, hi) must fit in its page-table row and every page holding a
 * token of that range must be a valid page id.  Returns 0 or a status bit. */
static int lane_check(const oracle_cache* c, const int32_t* row, int max_pages, int lo, int hi)
{
    int p;
    if (lo < 0 || hi > max_pages * PAGE || hi < lo)
        return ST_OVERFLOW;
    if (hi == lo)
        return 0;
    for (p = lo / PAGE; p <= (hi - 1) / PAGE; ++p)
        if (row[p] < 0 || row[p] >= c->num_pages)
            return ST_BAD_PAGE;
    return 0;
}

/* Dequantised cache element of logical token t of lane row `row`. */
static double cache_value(const oracle_cache* c, int is_v, const int32_t* row, int h, int t, int d)
{
    int pid = row[t / PAGE], off = t % PAGE;
    size_t ph = (size_t)pid * c->num_kv_heads + h;
    const uint8_t* codes = is_v ? c->v_codes : c->k_codes;
    if (c->dtype == KV_FP8) {
        const float* sc = (const float*)(is_v ? c->v_scales : c->k_scales);
        uint8_t code = codes[(ph * PAGE + off) * HEAD_DIM + d];
        return oracle_e4m3_decode(code) * (double)sc[ph];
    } else if (c->dtype == KV_FP8_ROW) {
        const float* sc = (const float*)(is_v ? c->v_scales : c->k_scales);
        uint8_t code = codes[(ph * PAGE + off) * HEAD_DIM + d];
        return oracle_e4m3_decode(code) * (double)sc[ph * PAGE + off];
    } else if (c->dtype == KV_INT8) {
        const uint16_t* sc = (const uint16_t*)(is_v ? c->v_scales : c->k_scales);
        int8_t q = (int8_t)codes[(ph * PAGE + off) * HEAD_DIM + d];
        return (double)q * oracle_f16_decode(sc[(ph * PAGE + off) * (HEAD_DIM / 64) + d / 64]);
    } else {
        const uint16_t* sc = (const uint16_t*)(is_v ? c->v_scales : c->k_scales);
        uint8_t byte = codes[(ph * PAGE + off) * (HEAD_DIM / 2) + d / 2];
        int q = int4_nibble_value(byte, d & 1);
        double s = oracle_f16_decode(sc[(ph * PAGE + off) * (HEAD_DIM / 32) + d / 32]);
        return (double)q * s;
    }
}

/* ------------------------------------------------------------------ */
/* Append (R2, R3)                                                      */
/* ------------------------------------------------------------------ */
/* new_rows: bf16 bits [B][n_new][Hkv][128] for K then V. */
static void append_fp8_page(const oracle_cache* c, int is_v, int pid, int h, int start, int count,
                            const uint16_t* src, int token_stride)
{
    uint8_t* codes = (is_v ? c->v_codes : c->k_codes) + ((size_t)pid * c->num_kv_heads + h) * PAGE * HEAD_DIM;
    float* scale = (float*)(is_v ? c->v_scales : c->k_scales) + (size_t)pid * c->num_kv_heads + h;
    float amax = 0.0f, s_old = *scale, s_new;
    int t, d;
    for (t = 0; t < count; ++t)
        for (d = 0; d < HEAD_DIM; ++d) {
            float a = fabsf(bf16_value(src[(size_t)t * token_stride + d]));
            if (a > amax)
                amax = a;
        }
    if (start == 0) {
        s_new = amax / 448.0f;
    } else {
        float s_c = amax / 448.0f;
        s_new = s_c > s_old ? s_c : s_old;
        if (s_new > s_old) {
            /* the page's earlier tokens move to the larger scale */
            for (t = 0; t < start; ++t)
                for (d = 0; d < HEAD_DIM; ++d) {
                    uint8_t* p = &codes[t * HEAD_DIM + d];
                    float old_value = (float)oracle_e4m3_decode(*p) * s_old; /* fp32 multiply */
                    *p = oracle_e4m3_encode(old_value / s_new);              /* fp32 divide */
                }
        }
    }
    for (t = 0; t < count; ++t)
        for (d = 0; d < HEAD_DIM; ++d) {
            float x = bf16_value(src[(size_t)t * token_stride + d]);
            codes[(start + t) * HEAD_DIM + d] = (s_new == 0.0f) ? 0x00 : oracle_e4m3_encode(x / s_new);
        }
    *scale = s_new;
}

static void append_int4_token(const oracle_cache* c, int is_v, int pid, int h, int off, const uint16_t* src)
{
    size_t ph = (size_t)pid * c->num_kv_heads + h;
    uint8_t* codes = (is_v ? c->v_codes : c->k_codes) + (ph * PAGE + off) * (HEAD_DIM / 2);
    uint16_t* scales = (uint16_t*)(is_v ? c->v_scales : c->k_scales) + (ph * PAGE + off) * (HEAD_DIM / 32);
    int g, i;
    for (g = 0; g < HEAD_DIM / 32; ++g) {
        float x[32];
        int8_t q[32];
        for (i = 0; i < 32; ++i)
            x[i] = bf16_value(src[g * 32 + i]);
        scales[g] = oracle_int4_group(x, 32, q);
        for (i = 0; i < 32; i += 2)
            codes[(g * 32 + i) / 2] = (uint8_t)((q[i] & 0xF) | ((q[i + 1] & 0xF) << 4));
    }
}

/* INT8 group-64 and FP8 row formats: every token carries its own scales. */
static void append_token_rowscaled(const oracle_cache* c, int is_v, int pid, int h, int off, const uint16_t* src)
{
    size_t ph = (size_t)pid * c->num_kv_heads + h;
    uint8_t* codes = (is_v ? c->v_codes : c->k_codes) + (ph * PAGE + off) * HEAD_DIM;
    float x[HEAD_DIM];
    int i, g;
    for (i = 0; i < HEAD_DIM; ++i)
        x[i] = bf16_value(src[i]);
    if (c->dtype == KV_FP8_ROW) {
        float* scales = (float*)(is_v ? c->v_scales : c->k_scales);
        scales[ph * PAGE + off] = oracle_fp8_row(x, HEAD_DIM, codes);
    } else {
        uint16_t* scales = (uint16_t*)(is_v ? c->v_scales : c->k_scales) + (ph * PAGE + off) * (HEAD_DIM / 64);
        for (g = 0; g < HEAD_DIM / 64; ++g) {
            int8_t q[64];
            scales[g] = oracle_int8_group(x + 64 * g, 64, q);
            for (i = 0; i < 64; ++i)
                codes[64 * g + i] = (uint8_t)q[i];
        }
    }
}

/* Writes tokens [L_b, L_b + n_new) of every lane.  Lanes whose range does
 * not fit or touches an invalid page id are skipped and flagged. */
int oracle_append(int dtype, int num_pages, int num_kv_heads, uint8_t* k_codes, uint8_t* v_codes,
                  void* k_scales, void* v_scales, const uint16_t* k_new, const uint16_t* v_new, int num_lanes,
                  int n_new, const int32_t* page_table, int max_pages, const int32_t* seq_lens, int32_t* status)
{
    oracle_cache c = {dtype, num_pages, num_kv_heads, k_codes, v_codes, k_scales, v_scales};
    int b, h, kv;
    int token_stride = num_kv_heads * HEAD_DIM;
    for (b = 0; b < num_lanes; ++b) {
        const int32_t* row = page_table + (size_t)b * max_pages;
        int L = seq_lens[b];
        int err = lane_check(&c, row, max_pages, L, L + n_new);
        if (err) {
            if (status)
                *status |= err;
            continue;
        }
        for (kv = 0; kv < 2; ++kv) {
            const uint16_t* lane_src = (kv ? v_new : k_new) + (size_t)b * n_new * token_stride;
            for (h = 0; h < num_kv_heads; ++h) {
                if (dtype == KV_FP8) {
                    int t0 = L;
                    while (t0 < L + n_new) {
                        int lp = t0 / PAGE;
                        int t1 = (lp + 1) * PAGE < L + n_new ? (lp + 1) * PAGE : L + n_new;
                        append_fp8_page(&c, kv, row[lp], h, t0 - lp * PAGE, t1 - t0,
                                        lane_src + (size_t)(t0 - L) * token_stride + h * HEAD_DIM, token_stride);
                        t0 = t1;
                    }
                } else {
                    int t;
                    for (t = L; t < L + n_new; ++t) {
                        const uint16_t* src = lane_src + (size_t)(t - L) * token_stride + h * HEAD_DIM;
                        if (dtype == KV_INT4)
                            append_int4_token(&c, kv, row[t / PAGE], h, t % PAGE, src);
                        else
                            append_token_rowscaled(&c, kv, row[t / PAGE], h, t % PAGE, src);
                    }
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Verify attention (R4, R5): fp64, two-pass softmax                    */
/* ------------------------------------------------------------------ */
typedef struct {
    oracle_cache c;
    const uint16_t* q;
    int num_q_heads, num_lanes, window, max_pages;
    const int32_t* page_table;
    const int32_t* seq_lens;
    double sm_scale;
    double* out;
    const int32_t* rows; /* optional list of (b, i, h) triples */
    int nrows;
    const int32_t* parent; /* optional [B][W] draft tree (R9); NULL: causal window */
    int next; /* work counter */
    pthread_mutex_t lock;
    int32_t status;
} verify_job;

/* One output row: lane b, window position i, q head h. */
static int verify_row(verify_job* J, int b, int i, int h, double* o)
{
    const oracle_cache* c = &J->c;
    int G = J->num_q_heads / c->num_kv_heads;
    int hk = h / G;
    const int32_t* row = J->page_table + (size_t)b * J->max_pages;
    int L = J->seq_lens[b];
    int err = lane_check(c, row, J->max_pages, L, L + J->window);
    int n, j, d, seen[MAX_WINDOW];
    const uint16_t* qrow;
    double q[HEAD_DIM], *logit, mx, z;
    if (err) {
        for (d = 0; d < HEAD_DIM; ++d)
            o[d] = 0.0;
        return err;
    }
    n = L + i + 1; /* keys 0 .. L + i */
    /* keys 0 .. L + i are the causal window; with a draft tree (window <= 16)
     * window key L + j is seen only when slot j is i or one of its ancestors */
    if (J->parent != NULL) {
        for (j = 0; j < MAX_WINDOW; ++j)
            seen[j] = 0;
        for (j = i;; j = J->parent[(size_t)b * J->window + j]) {
            seen[j] = 1;
            if (j == 0)
                break;
        }
    }
    qrow = J->q + (((size_t)b * J->window + i) * J->num_q_heads + h) * HEAD_DIM;
    for (d = 0; d < HEAD_DIM; ++d)
        q[d] = (double)bf16_value(qrow[d]);
    logit = (double*)malloc(sizeof(double) * (size_t)n);
    mx = -INFINITY;
    for (j = 0; j < n; ++j) {
        double s = 0.0;
        if (J->parent != NULL && j >= L && !seen[j - L])
            continue;
        for (d = 0; d < HEAD_DIM; ++d)
            s += q[d] * cache_value(c, 0, row, hk, j, d);
        logit[j] = J->sm_scale * s;
        if (logit[j] > mx)
            mx = logit[j];
    }
    for (d = 0; d < HEAD_DIM; ++d)
        o[d] = 0.0;
    z = 0.0;
    for (j = 0; j < n; ++j) {
        double p;
        if (J->parent != NULL && j >= L && !seen[j - L])
            continue;
        p = exp(logit[j] - mx);
        z += p;
        for (d = 0; d < HEAD_DIM; ++d)
            o[d] += p * cache_value(c, 1, row, hk, j, d);
    }
    for (d = 0; d < HEAD_DIM; ++d)
        o[d] /= z;
    free(logit);
    return 0;
}

static void* verify_worker(void* arg)
{
    verify_job* J = (verify_job*)arg;
    int total = J->rows ? J->nrows : J->num_lanes * J->window * J->num_q_heads;
    for (;;) {
        int k, b, i, h, err;
        double* o;
        pthread_mutex_lock(&J->lock);
        k = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (k >= total)
            break;
        if (J->rows) {
            b = J->rows[3 * k];
            i = J->rows[3 * k + 1];
            h = J->rows[3 * k + 2];
            o = J->out + (size_t)k * HEAD_DIM;
        } else {
            b = k / (J->window * J->num_q_heads);
            i = (k / J->num_q_heads) % J->window;
            h = k % J->num_q_heads;
            o = J->out + (size_t)k * HEAD_DIM;
        }
        err = verify_row(J, b, i, h, o);
        if (err) {
            pthread_mutex_lock(&J->lock);
            J->status |= err;
            pthread_mutex_unlock(&J->lock);
        }
    }
    return NULL;
}

/* out: fp64 [B][W][Hq][128] when rows == NULL, else [nrows][128] for the
 * listed (b, i, h) triples.  threads > 1 only spreads independent rows over
 * worker threads; the arithmetic of each row is the same. */
int oracle_verify_attn(int dtype, int num_pages, int num_kv_heads, const uint8_t* k_codes, const uint8_t* v_codes,
                       const void* k_scales, const void* v_scales, const uint16_t* q, int num_q_heads, int num_lanes,
                       int window, const int32_t* page_table, int max_pages, const int32_t* seq_lens, float sm_scale,
                       double* out, const int32_t* rows, int nrows, int threads, int32_t* status)
{
    verify_job J;
    int t;
    pthread_t tid[256];
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    memset(&J, 0, sizeof J);
    J.c.dtype = dtype;
    J.c.num_pages = num_pages;
    J.c.num_kv_heads = num_kv_heads;
    J.c.k_codes = (uint8_t*)k_codes;
    J.c.v_codes = (uint8_t*)v_codes;
    J.c.k_scales = (void*)k_scales;
    J.c.v_scales = (void*)v_scales;
    J.q = q;
    J.num_q_heads = num_q_heads;
    J.num_lanes = num_lanes;
    J.window = window;
    J.max_pages = max_pages;
    J.page_table = page_table;
    J.seq_lens = seq_lens;
    J.sm_scale = (double)sm_scale;
    J.out = out;
    J.rows = rows;
    J.nrows = nrows;
    pthread_mutex_init(&J.lock, NULL);
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (threads == 1) {
        verify_worker(&J);
    } else {
        for (t = 0; t < threads; ++t)
            pthread_create(&tid[t], NULL, verify_worker, &J);
        for (t = 0; t < threads; ++t)
            pthread_join(tid[t], NULL);
    }
    pthread_mutex_destroy(&J.lock);
    if (status)
        *status |= J.status;
    return 0;
}

/* Draft-tree attention (R9): as oracle_verify_attn, but window row i sees
 * the window keys of its ancestors and itself only.  parent [B][W] with
 * 0 <= parent[b][i] < i for i >= 1 (entry 0 unused); window <= 16. */
int oracle_tree_attn(int dtype, int num_pages, int num_kv_heads, const uint8_t* k_codes, const uint8_t* v_codes,
                     const void* k_scales, const void* v_scales, const uint16_t* q, int num_q_heads, int num_lanes,
                     int window, const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                     const int32_t* parent, float sm_scale, double* out, int threads, int32_t* status)
{
    verify_job J;
    int t, b, i;
    pthread_t tid[256];
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || window > MAX_WINDOW || parent == NULL)
        return -1;
    for (b = 0; b < num_lanes; ++b)
        for (i = 1; i < window; ++i)
            if (parent[(size_t)b * window + i] < 0 || parent[(size_t)b * window + i] >= i)
                return -1;
    memset(&J, 0, sizeof J);
    J.c.dtype = dtype;
    J.c.num_pages = num_pages;
    J.c.num_kv_heads = num_kv_heads;
    J.c.k_codes = (uint8_t*)k_codes;
    J.c.v_codes = (uint8_t*)v_codes;
    J.c.k_scales = (void*)k_scales;
    J.c.v_scales = (void*)v_scales;
    J.q = q;
    J.num_q_heads = num_q_heads;
    J.num_lanes = num_lanes;
    J.window = window;
    J.max_pages = max_pages;
    J.page_table = page_table;
    J.seq_lens = seq_lens;
    J.sm_scale = (double)sm_scale;
    J.out = out;
    J.parent = parent;
    pthread_mutex_init(&J.lock, NULL);
    if (threads < 1)
        threads = 1;
    if (threads > 256)
        threads = 256;
    if (threads == 1) {
        verify_worker(&J);
    } else {
        for (t = 0; t < threads; ++t)
            pthread_create(&tid[t], NULL, verify_worker, &J);
        for (t = 0; t < threads; ++t)
            pthread_join(tid[t], NULL);
    }
    pthread_mutex_destroy(&J.lock);
    if (status)
        *status |= J.status;
    return 0;
}

/* Plain decode of one query row against the first n_keys cached tokens of
 * a lane, written independently of oracle_verify_attn (single pass with a
 * running maximum) so that "window of 1 == plain decode" is a real check. */
int oracle_decode_row(int dtype, int num_pages, int num_kv_heads, const uint8_t* k_codes, const uint8_t* v_codes,
                      const void* k_scales, const void* v_scales, const uint16_t* q_row, int kv_head,
                      const int32_t* page_row, int n_keys, float sm_scale, double* out)
{
    oracle_cache c = {dtype, num_pages, num_kv_heads, (uint8_t*)k_codes, (uint8_t*)v_codes, (void*)k_scales,
                      (void*)v_scales};
    double run_max = -INFINITY, run_sum = 0.0, acc[HEAD_DIM];
    int j, d;
    for (d = 0; d < HEAD_DIM; ++d)
        acc[d] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        double dot = 0.0, logit, shrink, w;
        for (d = 0; d < HEAD_DIM; ++d)
            dot += (double)bf16_value(q_row[d]) * cache_value(&c, 0, page_row, kv_head, j, d);
        logit = (double)sm_scale * dot;
        if (logit > run_max) {
            shrink = exp(run_max - logit);
            for (d = 0; d < HEAD_DIM; ++d)
                acc[d] *= shrink;
            run_sum *= shrink;
            run_max = logit;
        }
        w = exp(logit - run_max);
        run_sum += w;
        for (d = 0; d < HEAD_DIM; ++d)
            acc[d] += w * cache_value(&c, 1, page_row, kv_head, j, d);
    }
    for (d = 0; d < HEAD_DIM; ++d)
        out[d] = acc[d] / run_sum;
    return 0;
}

/* ------------------------------------------------------------------ */
/* Acceptance (R6)                                                      */
/* ------------------------------------------------------------------ */
int oracle_argmax(const float* x, int n)
{
    int best = -1, i;
    for (i = 0; i < n; ++i) {
        if (isnan(x[i]))
            continue;
        if (best < 0 || x[i] > x[best])
            best = i;
    }
    return best < 0 ? 0 : best;
}

/* logits fp32 [B][W][V]; drafts [B][W-1]; out_tokens [B][W];
 * accept_len [B]; seq_lens_inout may be NULL (no commit). */
int oracle_spec_accept(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                       int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status)
{
    int b, i, d = window - 1;
    for (b = 0; b < num_lanes; ++b) {
        int a = 0;
        for (i = 0; i < window; ++i)
            out_tokens[b * window + i] = oracle_argmax(logits + ((size_t)b * window + i) * vocab, vocab);
        for (i = 0; i < d; ++i)
            if ((drafts[b * d + i] < 0 || drafts[b * d + i] >= vocab) && status)
                *status |= ST_BAD_DRAFT;
        while (a < d && drafts[b * d + a] == out_tokens[b * window + a])
            ++a;
        accept_len[b] = a;
        if (seq_lens_inout)
            seq_lens_inout[b] += 1 + a;
    }
    return 0;
}

/* Lazy acceptance with per-lane draft counts (R6, R7).
 * num_drafts [B] may be NULL (every lane has window - 1 drafts).  A lane whose
 * count is outside [0, window - 1] sets ST_BAD_COUNT and gets accept_len 0,
 * out_tokens all -1 and no commit.  Otherwise: every one of the lane's d_b
 * drafts outside [0, vocab) sets ST_BAD_DRAFT (and never matches); rows are
 * taken in order, row i's argmax is reported, and the walk stops at the first
 * i that is d_b or whose draft disagrees; a = that i is the accept length,
 * out_tokens after row a are -1, and the commit adds 1 + a. */
int oracle_spec_accept_lazy(const float* logits, int num_lanes, int window, int vocab, const int32_t* drafts,
                            const int32_t* num_drafts, int32_t* accept_len, int32_t* out_tokens,
                            int32_t* seq_lens_inout, int32_t* status)
{
    int b, i, dmax = window - 1;
    for (b = 0; b < num_lanes; ++b) {
        int d = num_drafts ? num_drafts[b] : dmax, a = 0;
        for (i = 0; i < window; ++i)
            out_tokens[b * window + i] = -1;
        if (d < 0 || d > dmax) {
            accept_len[b] = 0;
            if (status)
                *status |= ST_BAD_COUNT;
            continue;
        }
        for (i = 0; i < d; ++i)
            if ((drafts[b * dmax + i] < 0 || drafts[b * dmax + i] >= vocab) && status)
                *status |= ST_BAD_DRAFT;
        for (;;) {
            int t = oracle_argmax(logits + ((size_t)b * window + a) * vocab, vocab);
            out_tokens[b * window + a] = t;
            if (a == d || drafts[b * dmax + a] != t)
                break;
            ++a;
        }
        accept_len[b] = a;
        if (seq_lens_inout)
            seq_lens_inout[b] += 1 + a;
    }
    return 0;
}

/* Lossless stochastic acceptance (R8).  logits [B][W][V]; draft_probs
 * [B][W-1][V] (row i: the draft distribution q_i that drafts[b][i] was drawn
 * from); u_accept [B][W-1] and u_sample [B] uniforms in [0, 1).  Outputs as
 * for the lazy form: out_tokens = drafts[0 .. a), the drawn token at a, -1
 * after; accept_len = a; the commit adds 1 + a. */
static void softmax_row(const float* l, int n, double* p)
{
    double m = l[0], s = 0.0;
    int x;
    for (x = 1; x < n; ++x)
        if (l[x] > m)
            m = l[x];
    for (x = 0; x < n; ++x) {
        p[x] = exp((double)l[x] - m);
        s += p[x];
    }
    for (x = 0; x < n; ++x)
        p[x] /= s;
}

int oracle_spec_accept_sampled(const float* logits, const float* draft_probs, int num_lanes, int window, int vocab,
                               const int32_t* drafts, const float* u_accept, const float* u_sample,
                               int32_t* accept_len, int32_t* out_tokens, int32_t* seq_lens_inout, int32_t* status)
{
    int b, i, x, d = window - 1;
    double* p = malloc(sizeof(double) * (size_t)vocab);
    double* w = malloc(sizeof(double) * (size_t)vocab);
    if (!p || !w) {
        free(p);
        free(w);
        return -1;
    }
    for (b = 0; b < num_lanes; ++b) {
        int a = d, k = -1, last = -1;
        double z = 0.0, target, cum = 0.0;
        for (i = 0; i < d; ++i)
            if ((drafts[b * d + i] < 0 || drafts[b * d + i] >= vocab) && status)
                *status |= ST_BAD_DRAFT;
        for (i = 0; i < d; ++i) {
            const int xi = drafts[b * d + i];
            if (xi < 0 || xi >= vocab) {
                a = i;
                break;
            }
            softmax_row(logits + ((size_t)b * window + i) * vocab, vocab, p);
            if (!((double)u_accept[b * d + i] * (double)draft_probs[((size_t)b * d + i) * vocab + xi] < p[xi])) {
                a = i;
                break;
            }
        }
        softmax_row(logits + ((size_t)b * window + a) * vocab, vocab, p);
        for (x = 0; x < vocab; ++x) {
            w[x] = p[x];
            if (a < d) {
                const double r = p[x] - (double)draft_probs[((size_t)b * d + a) * vocab + x];
                w[x] = r > 0.0 ? r : 0.0;
            }
            z += w[x];
        }
        if (!(z > 0.0)) {
            z = 0.0;
            for (x = 0; x < vocab; ++x) {
                w[x] = p[x];
                z += w[x];
            }
        }
        target = (double)u_sample[b] * z;
        for (x = 0; x < vocab; ++x) {
            if (w[x] > 0.0)
                last = x;
            cum += w[x];
            if (k < 0 && cum > target)
                k = x;
        }
        if (k < 0)
            k = last;
        for (i = 0; i < window; ++i)
            out_tokens[b * window + i] = i < a ? drafts[b * d + i] : (i == a ? k : -1);
        accept_len[b] = a;
        if (seq_lens_inout)
            seq_lens_inout[b] += 1 + a;
    }
    free(p);
    free(w);
    return 0;
}

/* Draft-tree acceptance (R9).  tokens [B][W]: the window's tokens (slot 0,
 * the root, is not checked); parent [B][W] as for oracle_tree_attn.
 * path [B][W] (out): the accepted slots, root first, then -1;
 * out_tokens [B][W] (out): the accepted tokens after the root, then the
 * bonus token, then -1; accept_len [B] = the accepted nodes after the root;
 * the commit adds 1 + a.  A lane with an invalid parent sets bit 32 and gets
 * a = 0, path and tokens -1, no commit.  Token ids outside [0, vocab) set the
 * draft bit and never match. */
int oracle_tree_accept(const float* logits, int num_lanes, int window, int vocab, const int32_t* tokens,
                       const int32_t* parent, int32_t* accept_len, int32_t* path, int32_t* out_tokens,
                       int32_t* seq_lens_inout, int32_t* status)
{
    int b, i, c;
    for (b = 0; b < num_lanes; ++b) {
        const int32_t* par = parent + (size_t)b * window;
        const int32_t* tk = tokens + (size_t)b * window;
        int32_t* pa = path + (size_t)b * window;
        int32_t* ot = out_tokens + (size_t)b * window;
        int bad = 0, a = 0, n = 0;
        for (i = 0; i < window; ++i) {
            pa[i] = -1;
            ot[i] = -1;
        }
        for (i = 1; i < window; ++i) {
            if (par[i] < 0 || par[i] >= i)
                bad = 1;
            if ((tk[i] < 0 || tk[i] >= vocab) && status)
                *status |= ST_BAD_DRAFT;
        }
        if (bad) {
            accept_len[b] = 0;
            if (status)
                *status |= 32;
            continue;
        }
        pa[0] = 0;
        for (;;) {
            int t = oracle_argmax(logits + ((size_t)b * window + n) * vocab, vocab), next = -1;
            for (c = n + 1; c < window && next < 0; ++c)
                if (par[c] == n && tk[c] == t)
                    next = c;
            if (next < 0) {
                ot[a] = t;
                break;
            }
            ot[a] = tk[next];
            ++a;
            pa[a] = next;
            n = next;
        }
        accept_len[b] = a;
        if (seq_lens_inout)
            seq_lens_inout[b] += 1 + a;
    }
    return 0;
}
