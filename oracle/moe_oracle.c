/*
 * moe_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct fp64 CPU oracle of the decode-time MoE
 * layer. It exists so the CUDA path can be checked against something written
 * independently of it. Only the test suite, __graft_entry__.smoke() and the
 * CPU-baseline / reference legs of bench.py load this library; the product
 * path never does. It shares no code, header, table or helper with the CUDA
 * library (the format enum and table layout below are written out again here
 * on purpose, from their definitions).
 *
 * What it computes (the layer as the pages state it):
 *   "Daily AI Hotspot 2026-08-21: Shared-Expert Fusion Lands on NVIDIA and AMD
 *   the Same Day", section "Most Worth Your Attention Today": a DeepSeek-V4
 *   family MoE layer runs routed FP4 experts and an FP8 shared expert that
 *   every token passes through; unfused that is four launches (routed MoE,
 *   shared gate/up, shared down, residual add), fused it is one pass with FP32
 *   accumulation that writes the BF16 output once. For row t:
 *
 *       ref[t] = x[t] + S(x[t]) + sum_p topk_w[t,p] * R_{ids[t,p]}(x[t])
 *       F(x)   = Wd * ( silu(Wg x) .* (Wu x) ),   silu(v) = v / (1 + e^-v)
 *
 *   The oracle returns ref unrounded, in fp64. Expert dedup (one stream of an
 *   expert's weights for all rows that picked it) is an exact regrouping of
 *   this sum, so the oracle does not dedup: it loops row by row, expert by
 *   expert.
 *
 * Group table (the dedup bookkeeping):
 *   MarloweAI/sgl-amd-mono-upstream PR #27 "each expert once", sections
 *   "Motivation" and "Modifications" (commit 1) and "Reviewer notes": the
 *   step's groups are the shared expert and every distinct routed expert in
 *   order of first use; the table holds the group count, each group's expert
 *   and each row's slot in each group. Written here as a plain linear scan.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   residual = x; shared expert weight 1, no gate; topk_w used as given;
 *   SwiGLU = silu(gate) * up with no clamp; gate rows first in the fused
 *   [2I, H] gate/up matrix; NVFP4 low nibble = even element, 16-element
 *   blocks along the input dimension, E4M3 block scale, one fp32 tensor scale
 *   per expert per matrix; FP8 = OCP E4M3FN with one fp32 scale per 128x128
 *   block; first use scanned row-major over (t, p); an out-of-range id sets an
 *   error bit and contributes nothing; a repeated id within a row sets an
 *   error bit and both uses are still computed.
 *
 * FP8 intermediate blocks (the opt-in low-precision variant):
 *   MarloweAI/sgl-amd-mono-upstream PR #27 "each expert once", section
 *   "Modifications": the AMD path keeps the SwiGLU intermediate in FP8 "mid
 *   blocks" before down. The page gives no block size or scale; read here as
 *   blocks of 32 consecutive intermediate values of one expert use, each block
 *   with one power-of-two scale 2^k (the smallest with max|mid| <= 448 * 2^k,
 *   k >= -126), each value replaced by its nearest OCP E4M3FN value at that
 *   scale (ties to even).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* weight formats, as the library's ABI numbers them */
enum { ORC_BF16 = 0, ORC_NVFP4 = 1, ORC_FP8_B128 = 2 };
/* error bits, as the library's ABI numbers them */
enum { ORC_BAD_EXPERT = 1u, ORC_DUP_EXPERT = 2u };
/* flag bit selecting the one-row (no dedup) table */
enum { ORC_FLAG_NO_DEDUP = 1u };

typedef struct {
    int fmt;
    const void *w13;        /* [E][2I][H] (NVFP4: [E][2I][H/2] bytes) */
    const void *w13_scale;  /* NVFP4: E4M3 [E][2I][H/16]; FP8: fp32 [E][2I/128][H/128] */
    const float *w13_gscale;/* NVFP4: fp32 [E] */
    const void *w2;         /* [E][H][I] (NVFP4: [E][H][I/2] bytes) */
    const void *w2_scale;   /* NVFP4: E4M3 [E][H][I/16]; FP8: fp32 [E][H/128][I/128] */
    const float *w2_gscale; /* NVFP4: fp32 [E] */
} oracle_weights;

/* ---- element decodes ------------------------------------------------ */

/* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is the
 * subnormal 0 / 0.5. Written from the bit fields, not from a value list. */
double oracle_e2m1(int code)
{
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* OCP E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinity,
 * S.1111.111 is NaN, exponent 0 is subnormal (m/8 * 2^-6). */
double oracle_e4m3(int byte)
{
    int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* bfloat16: the top 16 bits of an IEEE binary32. */
double oracle_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* One dequantised element of a row-major [rows][cols] matrix of expert e.
 * mat = 0 for gate/up ([2I][H]), 1 for down ([H][I]). */
static double weight_at(const oracle_weights *w, int mat, int rows, int cols,
                        int e, int r, int c)
{
    size_t ri = (size_t)e * rows + r;
    const void *q = mat ? w->w2 : w->w13;
    const void *sc = mat ? w->w2_scale : w->w13_scale;
    if (w->fmt == ORC_BF16) {
        return oracle_bf16(((const uint16_t *)q)[ri * cols + c]);
    } else if (w->fmt == ORC_NVFP4) {
        uint8_t byte = ((const uint8_t *)q)[ri * (cols / 2) + c / 2];
        int code = (c % 2 == 0) ? (byte & 15) : (byte >> 4);
        double blk = oracle_e4m3(((const uint8_t *)sc)[ri * (cols / 16) + c / 16]);
        double g = (mat ? w->w2_gscale : w->w13_gscale)[e];
        return oracle_e2m1(code) * blk * g;
    } else { /* ORC_FP8_B128 */
        double v = oracle_e4m3(((const uint8_t *)q)[ri * cols + c]);
        size_t srow = (size_t)e * (rows / 128) + r / 128;
        double s = ((const float *)sc)[srow * (cols / 128) + c / 128];
        return v * s;
    }
}

/* Dequantised row r (0 <= r < 2I) of expert e's gate/up matrix, length H. */
void oracle_w13_row(const oracle_weights *w, int H, int I, int e, int r, double *row)
{
    for (int h = 0; h < H; ++h) row[h] = weight_at(w, 0, 2 * I, H, e, r, h);
}

/* Dequantised row h of expert e's down matrix, length I. */
void oracle_w2_row(const oracle_weights *w, int H, int I, int e, int h, double *row)
{
    for (int i = 0; i < I; ++i) row[i] = weight_at(w, 1, H, I, e, h, i);
}

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* The nearest OCP E4M3FN value to v (ties to the even mantissa), saturating
 * at +-448. E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits; normals
 * 2^(e-7) (1 + m/8) for e = 1..15 (e = 15, m = 7 is NaN, so 448 is the
 * largest); subnormals m 2^-9. On a grid of spacing `step` the nearest value
 * with ties to even is nearbyint(a / step) * step (default rounding mode:
 * to nearest, ties to even); the spacing is 2^-9 below 2^-6 and 2^(E-3) in the
 * binade [2^E, 2^(E+1)). */
double oracle_e4m3_rne(double v)
{
    double a = fabs(v), q;
    if (a >= 448.0) {
        q = 448.0;
    } else if (a < ldexp(1.0, -6)) {
        q = nearbyint(a / ldexp(1.0, -9)) * ldexp(1.0, -9);
    } else {
        int x;
        (void)frexp(a, &x); /* a = f 2^x, f in [0.5, 1): binade exponent x - 1 */
        double step = ldexp(1.0, x - 1 - 3);
        q = nearbyint(a / step) * step;
    }
    return v < 0 ? -q : q;
}

/* In place: each block of `block` consecutive values shares the scale 2^k,
 * the smallest power of two with max|mid| <= 448 * 2^k (k >= -126), and each
 * value becomes its nearest E4M3 value at that scale. An all-zero block stays
 * zero. 448 = 1.75 * 2^8, so with max|mid| = f 2^E (f in [1, 2)) the scale is
 * k = E - 8, plus one when f > 1.75. */
void oracle_fp8_mid_blocks(double *mid, int n, int block)
{
    for (int b0 = 0; b0 < n; b0 += block) {
        int b1 = b0 + block < n ? b0 + block : n;
        double amax = 0.0;
        for (int i = b0; i < b1; ++i) amax = fabs(mid[i]) > amax ? fabs(mid[i]) : amax;
        if (amax == 0.0) continue;
        int x;
        double f = frexp(amax, &x) * 2.0; /* amax = f 2^(x-1), f in [1, 2) */
        int k = (x - 1) - 8 + (f > 1.75 ? 1 : 0);
        if (k < -126) k = -126;
        for (int i = b0; i < b1; ++i) mid[i] = ldexp(oracle_e4m3_rne(ldexp(mid[i], -k)), k);
    }
}

/* One SwiGLU expert applied to one fp64 activation row:
 *   mid = silu(Wg x) .* (Wu x)     (Wg = rows 0..I-1, Wu = rows I..2I-1)
 *   y   = Wd mid
 * mid may be NULL. scratch needs max(H, I) doubles. */
static void expert_ffn_q(const oracle_weights *w, int H, int I, int e,
                         const double *x, double *mid, double *y, double *row, int fp8_block)
{
    double *m = mid ? mid : (double *)malloc(sizeof(double) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        double g = 0.0, u = 0.0;
        oracle_w13_row(w, H, I, e, i, row);
        for (int h = 0; h < H; ++h) g += row[h] * x[h];
        oracle_w13_row(w, H, I, e, I + i, row);
        for (int h = 0; h < H; ++h) u += row[h] * x[h];
        m[i] = silu(g) * u;
    }
    if (fp8_block > 0) oracle_fp8_mid_blocks(m, I, fp8_block);
    for (int h = 0; h < H; ++h) {
        double acc = 0.0;
        oracle_w2_row(w, H, I, e, h, row);
        for (int i = 0; i < I; ++i) acc += row[i] * m[i];
        y[h] = acc;
    }
    if (!mid) free(m);
}

static void expert_ffn(const oracle_weights *w, int H, int I, int e,
                       const double *x, double *mid, double *y, double *row)
{
    expert_ffn_q(w, H, I, e, x, mid, y, row, 0);
}

void oracle_expert_ffn(const oracle_weights *w, int H, int I, int e,
                       const double *x, double *mid, double *y)
{
    double *row = (double *)malloc(sizeof(double) * (size_t)(H > I ? H : I));
    expert_ffn(w, H, I, e, x, mid, y, row);
    free(row);
}

/* ---- group table ---------------------------------------------------- */
/*
 * Layout (int32), with C = T*(K+1):
 *   [0] G   number of groups      [1] U   number of columns
 *   group_expert[C]  expert of each group (-1 = the shared expert)
 *   group_ncols[C]   columns (using rows) of each group
 *   group_col0[C]    first column of each group (prefix sum, group order)
 *   col_row[C]       row of each column
 *   row_col[T][K+1]  slot 0 = the row's shared column, slot 1+p = the column
 *                    of pick p (-1 if the pick's id is out of range)
 * Entries past G (or U) are 0.
 *
 * Dedup: group 0 is the shared expert (every row uses it, so it is first in
 * order of first use); then each distinct in-range routed id in the order it
 * is first met scanning (t, p) row-major. Columns inside a group follow that
 * same (t, p) order. One-row (no dedup) form: for each row t, a group for the
 * row's shared use, then one group per in-range pick, each of one column.
 */
int oracle_group_table_size(int T, int K) { return 2 + 5 * T * (K + 1); }

int oracle_group_table(const int32_t *ids, int T, int K, int E, unsigned flags,
                       int32_t *table, uint32_t *err_out)
{
    int C = T * (K + 1);
    int32_t *gexp = table + 2, *gn = gexp + C, *g0 = gn + C, *crow = g0 + C,
            *rcol = crow + C;
    int *use_group = (int *)malloc(sizeof(int) * (size_t)(C > 0 ? C : 1));
    uint32_t err = 0;
    int G = 0, U = 0;
    memset(table, 0, sizeof(int32_t) * (size_t)oracle_group_table_size(T, K));

    for (int t = 0; t < T; ++t)
        for (int p = 0; p < K; ++p) {
            int id = ids[t * K + p];
            if (id < 0 || id >= E) { err |= ORC_BAD_EXPERT; continue; }
            for (int q = 0; q < p; ++q)
                if (ids[t * K + q] == id) err |= ORC_DUP_EXPERT;
        }

    if (flags & ORC_FLAG_NO_DEDUP) {
        for (int t = 0; t < T; ++t) {
            gexp[G] = -1; gn[G] = 1; g0[G] = U; crow[U] = t;
            rcol[t * (K + 1)] = U; ++G; ++U;
            for (int p = 0; p < K; ++p) {
                int id = ids[t * K + p];
                if (id < 0 || id >= E) { rcol[t * (K + 1) + 1 + p] = -1; continue; }
                gexp[G] = id; gn[G] = 1; g0[G] = U; crow[U] = t;
                rcol[t * (K + 1) + 1 + p] = U; ++G; ++U;
            }
        }
    } else if (T > 0) {
        /* groups: shared first, then distinct ids in order of first use */
        gexp[G++] = -1;
        for (int t = 0; t < T; ++t)
            for (int p = 0; p < K; ++p) {
                int id = ids[t * K + p], g, found = -1;
                if (id < 0 || id >= E) continue;
                for (g = 1; g < G; ++g) if (gexp[g] == id) { found = g; break; }
                if (found < 0) gexp[G++] = id;
            }
        /* which group each (t, p) use lands in; count columns */
        gn[0] = T;
        for (int t = 0; t < T; ++t)
            for (int p = 0; p < K; ++p) {
                int id = ids[t * K + p];
                use_group[t * K + p] = -1;
                if (id < 0 || id >= E) continue;
                for (int g = 1; g < G; ++g)
                    if (gexp[g] == id) { use_group[t * K + p] = g; gn[g]++; break; }
            }
        for (int g = 0; g < G; ++g) { g0[g] = U; U += gn[g]; }
        /* columns in (t, p) order inside each group */
        {
            int *fill = (int *)calloc((size_t)G, sizeof(int));
            for (int t = 0; t < T; ++t) {
                int c = g0[0] + fill[0]++;
                crow[c] = t; rcol[t * (K + 1)] = c;
            }
            for (int t = 0; t < T; ++t)
                for (int p = 0; p < K; ++p) {
                    int g = use_group[t * K + p];
                    if (g < 0) { rcol[t * (K + 1) + 1 + p] = -1; continue; }
                    int c = g0[g] + fill[g]++;
                    crow[c] = t; rcol[t * (K + 1) + 1 + p] = c;
                }
            free(fill);
        }
    }
    table[0] = G;
    table[1] = U;
    free(use_group);
    if (err_out) *err_out = err;
    return G;
}

/* ---- the router ------------------------------------------------------ */
/*
 * The routing front end that produces topk_ids / topk_w from the layer input.
 * "Daily AI Hotspot 2026-08-21", section "Most Worth Your Attention Today"
 * (the SGLang #32340 paragraph): the shared-expert fusion had to handle a bf16
 * correction bias and a top-k that is not a power of two (top-6). PR #27
 * "each expert once", "Reviewer notes": every CTA routes all rows itself and
 * the tie order is unchanged. The pages give no scoring formula; the reading
 * taken is the DeepSeek-V3 one, for row t and routed expert e:
 *
 *     logit[t,e] = sum_h x[t,h] * Wr[e,h]                (Wr bf16 [E][H])
 *     s[t,e]     = 1 / (1 + exp(-logit[t,e]))            (sigmoid score)
 *     key[t,e]   = s[t,e] + bias[e]                      (bias bf16 [E], or 0)
 *     ids[t,:]   = the K experts of largest key, in decreasing key order;
 *                  equal keys: the lower expert index first
 *     w[t,p]     = scale * s[t,ids[t,p]] / sum_q s[t,ids[t,q]]   (renorm = 1)
 *                  scale * s[t,ids[t,p]]                          (renorm = 0)
 *
 * Everything in fp64 from the bf16 inputs. keys_out (optional, [T][E]) gets
 * the selection keys so a test can tell a near tie from a wrong pick.
 */
void oracle_route(const uint16_t *x_bf16, const uint16_t *wr_bf16, const uint16_t *bias_bf16,
                  int T, int H, int E, int K, double scale, int renorm,
                  int32_t *ids_out, double *w_out, double *keys_out)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
    double *key = (double *)malloc(sizeof(double) * (size_t)(E > 0 ? E : 1));
    char *taken = (char *)malloc((size_t)(E > 0 ? E : 1));
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += oracle_bf16(x_bf16[(size_t)t * H + h]) * oracle_bf16(wr_bf16[(size_t)e * H + h]);
            s[e] = 1.0 / (1.0 + exp(-acc));
            key[e] = s[e] + (bias_bf16 ? oracle_bf16(bias_bf16[e]) : 0.0);
            taken[e] = 0;
            if (keys_out) keys_out[(size_t)t * E + e] = key[e];
        }
        /* K passes of "largest remaining key, lowest index among equals" */
        double sum = 0.0;
        for (int p = 0; p < K; ++p) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || key[e] > key[best])) best = e;
            taken[best] = 1;
            ids_out[t * K + p] = best;
            sum += s[best];
        }
        for (int p = 0; p < K; ++p) {
            double v = s[ids_out[t * K + p]];
            w_out[t * K + p] = scale * (renorm ? v / sum : v);
        }
    }
    free(s); free(key); free(taken);
}

/* ---- the layer ------------------------------------------------------ */

/* ref[j][:] for the rows listed in rows[0..nrows), straight from the
 * definition: x + shared expert + sum over picks of weight * routed expert.
 * Out-of-range picks contribute nothing. nthreads > 1 splits rows over
 * OpenMP threads (rows are independent; the arithmetic of a row is the same). */
void oracle_moe_layer_rows(const uint16_t *x_bf16, const int32_t *ids,
                           const float *topk_w, const oracle_weights *routed,
                           const oracle_weights *shared, int T, int H, int I,
                           int I_shared, int E, int K, const int32_t *rows,
                           int nrows, double *ref, int nthreads)
{
    (void)T;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#else
    (void)nthreads;
#endif
    for (int j = 0; j < nrows; ++j) {
        int t = rows[j];
        int mx = H > I ? H : I;
        if (I_shared > mx) mx = I_shared;
        double *x = (double *)malloc(sizeof(double) * (size_t)H);
        double *y = (double *)malloc(sizeof(double) * (size_t)H);
        double *row = (double *)malloc(sizeof(double) * (size_t)mx);
        double *out = ref + (size_t)j * H;
        for (int h = 0; h < H; ++h) x[h] = oracle_bf16(x_bf16[(size_t)t * H + h]);
        for (int h = 0; h < H; ++h) out[h] = x[h];
        expert_ffn(shared, H, I_shared, 0, x, NULL, y, row);
        for (int h = 0; h < H; ++h) out[h] += y[h];
        for (int p = 0; p < K; ++p) {
            int id = ids[t * K + p];
            if (id < 0 || id >= E) continue;
            expert_ffn(routed, H, I, id, x, NULL, y, row);
            for (int h = 0; h < H; ++h) out[h] += (double)topk_w[t * K + p] * y[h];
        }
        free(x); free(y); free(row);
    }
}

/* The same result as oracle_moe_layer_rows, with the expert evaluations of
 * the listed rows (each row's shared use and its K picks) spread over OpenMP
 * threads, then each row summed in the same fixed order (x, shared, picks
 * 0..K-1) with the same operations, so the two agree bit for bit. Only the
 * scheduling differs: it lets one row's experts run in parallel. */
static void layer_uses(const uint16_t *x_bf16, const int32_t *ids,
                       const float *topk_w, const oracle_weights *routed,
                       const oracle_weights *shared, int T, int H, int I,
                       int I_shared, int E, int K, const int32_t *rows,
                       int nrows, double *ref, int nthreads, int fp8_block);

void oracle_moe_layer_uses(const uint16_t *x_bf16, const int32_t *ids,
                           const float *topk_w, const oracle_weights *routed,
                           const oracle_weights *shared, int T, int H, int I,
                           int I_shared, int E, int K, const int32_t *rows,
                           int nrows, double *ref, int nthreads)
{
    layer_uses(x_bf16, ids, topk_w, routed, shared, T, H, I, I_shared, E, K, rows, nrows, ref, nthreads, 0);
}

/* The layer with the FP8 intermediate blocks of the opt-in variant: every
 * expert use's SwiGLU intermediate goes through oracle_fp8_mid_blocks with
 * blocks of `block` values before down; the rest as oracle_moe_layer_uses. */
void oracle_moe_layer_fp8mid(const uint16_t *x_bf16, const int32_t *ids,
                             const float *topk_w, const oracle_weights *routed,
                             const oracle_weights *shared, int T, int H, int I,
                             int I_shared, int E, int K, const int32_t *rows,
                             int nrows, double *ref, int nthreads, int block)
{
    layer_uses(x_bf16, ids, topk_w, routed, shared, T, H, I, I_shared, E, K, rows, nrows, ref, nthreads, block);
}

static void layer_uses(const uint16_t *x_bf16, const int32_t *ids,
                       const float *topk_w, const oracle_weights *routed,
                       const oracle_weights *shared, int T, int H, int I,
                       int I_shared, int E, int K, const int32_t *rows,
                       int nrows, double *ref, int nthreads, int fp8_block)
{
    int K1 = K + 1, nuse = nrows * K1;
    double *Y = (double *)malloc(sizeof(double) * (size_t)(nuse > 0 ? nuse : 1) * (size_t)H);
    (void)T;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
#else
    (void)nthreads;
#endif
    for (int u = 0; u < nuse; ++u) {
        int j = u / K1, q = u % K1, t = rows[j];
        int mx = H > I ? H : I;
        if (I_shared > mx) mx = I_shared;
        double *x = (double *)malloc(sizeof(double) * (size_t)H);
        double *row = (double *)malloc(sizeof(double) * (size_t)mx);
        double *y = Y + (size_t)u * H;
        for (int h = 0; h < H; ++h) x[h] = oracle_bf16(x_bf16[(size_t)t * H + h]);
        if (q == 0) {
            expert_ffn_q(shared, H, I_shared, 0, x, NULL, y, row, fp8_block);
        } else {
            int id = ids[t * K + q - 1];
            if (id >= 0 && id < E) expert_ffn_q(routed, H, I, id, x, NULL, y, row, fp8_block);
        }
        free(x); free(row);
    }
    for (int j = 0; j < nrows; ++j) {
        int t = rows[j];
        double *out = ref + (size_t)j * H;
        for (int h = 0; h < H; ++h) out[h] = oracle_bf16(x_bf16[(size_t)t * H + h]);
        for (int h = 0; h < H; ++h) out[h] += Y[((size_t)j * K1) * H + h];
        for (int p = 0; p < K; ++p) {
            int id = ids[t * K + p];
            if (id < 0 || id >= E) continue;
            for (int h = 0; h < H; ++h)
                out[h] += (double)topk_w[t * K + p] * Y[((size_t)j * K1 + 1 + p) * H + h];
        }
    }
    free(Y);
}

/* The same layer as the four unfused launches the pages list, each over all
 * rows, with its result held in its own buffer as if written to HBM:
 *   1. routed MoE       R[t] = sum_p w[t,p] * R_{ids[t,p]}(x[t])
 *   2. shared gate/up   M[t] = silu(Wg_s x[t]) .* (Wu_s x[t])
 *   3. shared down      S[t] = Wd_s M[t]
 *   4. residual add     out[t] = x[t] + S[t] + R[t]
 * Kept separate from oracle_moe_layer_rows so a test can compare the two. */
void oracle_unfused_layer(const uint16_t *x_bf16, const int32_t *ids,
                          const float *topk_w, const oracle_weights *routed,
                          const oracle_weights *shared, int T, int H, int I,
                          int I_shared, int E, int K, double *out)
{
    size_t TH = (size_t)T * H;
    int mx = H > I ? H : I;
    if (I_shared > mx) mx = I_shared;
    double *X = (double *)malloc(sizeof(double) * (TH ? TH : 1));
    double *R = (double *)calloc(TH ? TH : 1, sizeof(double));
    double *M = (double *)malloc(sizeof(double) * (size_t)T * I_shared + 1);
    double *S = (double *)malloc(sizeof(double) * (TH ? TH : 1));
    double *mid = (double *)malloc(sizeof(double) * (size_t)(I > 0 ? I : 1));
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    double *row = (double *)malloc(sizeof(double) * (size_t)mx);
    for (size_t i = 0; i < TH; ++i) X[i] = oracle_bf16(x_bf16[i]);

    /* launch 1: routed MoE */
    for (int t = 0; t < T; ++t)
        for (int p = 0; p < K; ++p) {
            int id = ids[t * K + p];
            if (id < 0 || id >= E) continue;
            expert_ffn(routed, H, I, id, X + (size_t)t * H, mid, y, row);
            for (int h = 0; h < H; ++h) R[(size_t)t * H + h] += (double)topk_w[t * K + p] * y[h];
        }
    /* launch 2: shared gate/up, every row */
    for (int t = 0; t < T; ++t)
        for (int i = 0; i < I_shared; ++i) {
            double g = 0.0, u = 0.0;
            oracle_w13_row(shared, H, I_shared, 0, i, row);
            for (int h = 0; h < H; ++h) g += row[h] * X[(size_t)t * H + h];
            oracle_w13_row(shared, H, I_shared, 0, I_shared + i, row);
            for (int h = 0; h < H; ++h) u += row[h] * X[(size_t)t * H + h];
            M[(size_t)t * I_shared + i] = silu(g) * u;
        }
    /* launch 3: shared down, every row */
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            oracle_w2_row(shared, H, I_shared, 0, h, row);
            for (int i = 0; i < I_shared; ++i) acc += row[i] * M[(size_t)t * I_shared + i];
            S[(size_t)t * H + h] = acc;
        }
    /* launch 4: residual add */
    for (size_t i = 0; i < TH; ++i) out[i] = X[i] + S[i] + R[i];

    free(X); free(R); free(M); free(S); free(mid); free(y); free(row);
}
