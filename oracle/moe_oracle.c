/*
 * moe_oracle.c -- plain CPU oracle for the forward pass of one dropless MoE
 * layer.  TEST INFRASTRUCTURE ONLY: it exists to check the CUDA library, is
 * called only from the tests, the smoke check and the CPU-baseline leg of the
 * benchmark, and shares no code, header or table with the CUDA path.
 *
 * Everything is computed in fp64 from bf16 inputs that are widened exactly.
 * The only rounding that the oracle mirrors from the device path is the bf16
 * rounding of the SwiGLU intermediate h (round to nearest, ties to even),
 * because the method stores h in bf16 between the two expert GEMMs.
 *
 * Sources (pages as titled in the reference material):
 *  - "MoE & MLA operators" (TileLang tutorial), sec. 2.2: router GEMM
 *    logits = x W_g, softmax + top-k, group-limited routing
 *    (n_expert_groups / n_limited_groups).
 *  - same page, sec. 2.3: permute is a data-dependent gather, segments are
 *    padded to a multiple of padding_M = 128, and the block table
 *    block_metadata[total_m_blocks, 3] = [expert, m_start, valid_m];
 *    permute -> per-assignment expert -> scatter-reduce equals direct
 *    per-token evaluation exactly.
 *  - same page, sec. 2.4(c): the expert MLP is up * silu(gate).
 *  - same page, sec. 2.5 and 6.4: combine is a k-way sum back into token
 *    order whose summation order must be fixed.
 *  - "Dropless and grouped GEMM" page, sec. 1: the shared expert reads the
 *    original inputs and is added to the routed output.
 *  - same page, sec. 3: each segment rounds up to a multiple of 128, at most
 *    127 pad rows per expert; sec. 5: segments are laid out in ascending
 *    expert order and a tile reads exactly one expert's weights.
 *  - fp8 expert weights: "MoE & MLA operators", sec. 6.1 (one byte per
 *    weight) and "Dropless and grouped GEMM", sec. 12 (the scale multiplies
 *    the product when one scale covers the whole contraction): e4m3 codes
 *    with one fp32 scale per output channel.
 *  - the backward: "Dropless and grouped GEMM", sec. 4 (only the sort
 *    indices need saving; the permutation is undone by the transposed
 *    gather).
 *
 * Readings where the pages are silent or disagree (each one is listed with
 * its reason in the design notes of the repository):
 *  - padded size of a segment is ceil(c/P)*P, 0 for an empty expert;
 *  - rows inside a segment are in ascending assignment index a = t*k + j;
 *  - top-k ties go to the lower expert index, group ties to the lower group;
 *  - the group score is the maximum logit inside the group;
 *  - the routing weight is a softmax over the k selected logits (the same
 *    value as a softmax over all E followed by renormalisation);
 *  - the gate multiplies the down-projection result before the sum;
 *  - fp8 weights: scale = amax / 448 per output channel, codes by
 *    round-to-nearest-even of the fp32 quotient, saturating at 448.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_DATA 2

/* ---------------------------------------------------------------- bf16 -- */

/* Exact widening of a bf16 bit pattern: bf16 is the top half of an fp32. */
double or_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round an fp64 value directly to the nearest bf16 value, ties to even.
 * bf16 keeps 8 significant bits, exponent range of fp32 (min normal 2^-126,
 * subnormal quantum 2^-133, largest finite (2 - 2^-7) * 2^127).  The value is
 * scaled to an integer grid by an exact power of two, rounded with
 * nearbyint() (round-half-even in the default rounding mode) and scaled
 * back, so no intermediate fp32 rounding happens. */
double or_round_bf16(double v)
{
    if (v != v || v == 0.0 || isinf(v)) return v;
    int e;
    (void)frexp(v, &e);           /* |v| = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                /* quantum exponent for 8 significant bits */
    if (q < -133) q = -133;       /* bf16 subnormal spacing */
    double scaled = ldexp(v, -q); /* exact */
    double r = ldexp(nearbyint(scaled), q);
    const double bf16_max = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (fabs(r) > bf16_max) r = v > 0 ? INFINITY : -INFINITY;
    return r;
}

uint16_t or_double_to_bf16_bits(double v)
{
    float f = (float)or_round_bf16(v); /* exact: the value is a bf16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* --------------------------------------------------------------- router -- */

/* logits[t, e] = sum_i x[t, i] * Wg[i, e] + bias[e]
 * x [T, d] bf16, Wg [d, E] bf16 (the page's orientation), bias [E] fp32 or
 * NULL.  Products of two bf16 values are exact in fp64. */
void or_router_logits(int T, int d, int E, const uint16_t *x, const uint16_t *Wg,
                      const float *bias, double *logits)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *row = logits + (size_t)t * E;
        for (int e = 0; e < E; ++e) row[e] = 0.0;
        for (int i = 0; i < d; ++i) {
            double xi = or_bf16_to_double(x[(size_t)t * d + i]);
            const uint16_t *w = Wg + (size_t)i * E;
            for (int e = 0; e < E; ++e) row[e] += xi * or_bf16_to_double(w[e]);
        }
        if (bias)
            for (int e = 0; e < E; ++e) row[e] += (double)bias[e];
    }
}

/* Top-k routing of one token's logits.
 *  n_groups == 0: plain top-k over all E experts.
 *  n_groups  > 0: the E experts form n_groups contiguous groups; a group's
 *                 score is its maximum logit; only the topk_groups best groups
 *                 stay eligible, then top-k among their experts.
 * Selection is repeated argmax; a strict '>' keeps the lower index on ties.
 * Output idx in descending logit order, gates = softmax over the k chosen
 * logits.  margin = smallest gap that decides the output: between the last
 * chosen and the best rejected group, between the last chosen and the best
 * rejected expert, and between consecutive chosen experts (their order is
 * part of the output); +inf when no decision was needed. */
static void route_one(int E, int k, int n_groups, int topk_groups, const double *l,
                      int32_t *idx, double *gate, double *margin, unsigned char *elig,
                      unsigned char *taken)
{
    double m = INFINITY;
    for (int e = 0; e < E; ++e) elig[e] = 1;
    if (n_groups > 0) {
        int gsz = E / n_groups;
        double gs[1024];
        unsigned char gtaken[1024];
        for (int g = 0; g < n_groups; ++g) {
            double best = -INFINITY;
            for (int e = g * gsz; e < (g + 1) * gsz; ++e)
                if (l[e] > best) best = l[e];
            gs[g] = best;
            gtaken[g] = 0;
        }
        double last = INFINITY;
        for (int r = 0; r < topk_groups; ++r) {
            int bi = -1;
            for (int g = 0; g < n_groups; ++g)
                if (!gtaken[g] && (bi < 0 || gs[g] > gs[bi])) bi = g;
            gtaken[bi] = 1;
            last = gs[bi];
        }
        double best_rej = -INFINITY;
        for (int g = 0; g < n_groups; ++g)
            if (!gtaken[g] && gs[g] > best_rej) best_rej = gs[g];
        if (best_rej > -INFINITY && last - best_rej < m) m = last - best_rej;
        for (int e = 0; e < E; ++e) elig[e] = gtaken[e / gsz];
    }
    for (int e = 0; e < E; ++e) taken[e] = 0;
    for (int r = 0; r < k; ++r) {
        int bi = -1;
        for (int e = 0; e < E; ++e)
            if (elig[e] && !taken[e] && (bi < 0 || l[e] > l[bi])) bi = e;
        taken[bi] = 1;
        idx[r] = bi;
    }
    double best_rej = -INFINITY;
    for (int e = 0; e < E; ++e)
        if (elig[e] && !taken[e] && l[e] > best_rej) best_rej = l[e];
    if (best_rej > -INFINITY && l[idx[k - 1]] - best_rej < m) m = l[idx[k - 1]] - best_rej;
    /* the output order is a decision too: gaps between consecutive choices */
    for (int r = 1; r < k; ++r)
        if (l[idx[r - 1]] - l[idx[r]] < m) m = l[idx[r - 1]] - l[idx[r]];
    /* softmax over the selected logits; idx[0] holds the largest */
    double lmax = l[idx[0]], s = 0.0;
    for (int r = 0; r < k; ++r) s += exp(l[idx[r]] - lmax);
    for (int r = 0; r < k; ++r) gate[r] = exp(l[idx[r]] - lmax) / s;
    *margin = m;
}

int or_route(int T, int E, int k, int n_groups, int topk_groups, const double *logits,
             int32_t *topk_idx, double *topk_w, double *margin)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return OR_ERR_ARG;
    if (n_groups > 0) {
        if (E % n_groups || n_groups > 1024 || topk_groups <= 0 || topk_groups > n_groups ||
            topk_groups * (E / n_groups) < k)
            return OR_ERR_ARG;
    }
    int bad = 0;
#pragma omp parallel
    {
        unsigned char *elig = (unsigned char *)malloc((size_t)E);
        unsigned char *taken = (unsigned char *)malloc((size_t)E);
        if (!elig || !taken) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(static)
            for (int t = 0; t < T; ++t)
                route_one(E, k, n_groups, topk_groups, logits + (size_t)t * E,
                          topk_idx + (size_t)t * k, topk_w + (size_t)t * k, margin + t, elig,
                          taken);
        }
        free(elig);
        free(taken);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* ---------------------------------------------------- offsets / metadata -- */

/* Capacity of the padded-row buffer and of the block table: they depend on
 * the sizes only, never on the routing. */
long long or_rows_capacity(long long A, int E, int P) { return A + (long long)E * (P - 1); }
long long or_blocks_capacity(long long A, int E, int P) { return A / P + E; }

/* From the A = T*k routing decisions (expert ids in assignment order,
 * a = t*k + j) build
 *   counts[E]              rows per expert
 *   padded_offsets[E + 1]  exclusive prefix sum of ceil(c/P)*P
 *   block_metadata[NB, 3]  [expert, m_start (global padded row), valid_m]
 *   num_blocks[1]          sum of ceil(c/P)
 *   perm_row[A]            padded row of each assignment
 *   row_src[R]             assignment of each padded row, -1 for a pad row
 *   row_gate[R]            routing weight of each padded row, 0 for a pad
 * for R = rows_capacity, NB = blocks_capacity.  Inside a segment the rows keep
 * ascending assignment order.  Returns OR_ERR_DATA for an expert id outside
 * [0, E). */
int or_build_offsets(long long A, int E, int P, const int32_t *idx, const double *w,
                     int32_t *counts, int32_t *padded_offsets, int32_t *block_metadata,
                     int32_t *num_blocks, int32_t *perm_row, int32_t *row_src, double *row_gate)
{
    if (A < 0 || E <= 0 || P <= 0) return OR_ERR_ARG;
    long long R = or_rows_capacity(A, E, P);
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long long a = 0; a < A; ++a) {
        if (idx[a] < 0 || idx[a] >= E) return OR_ERR_DATA;
        counts[idx[a]] += 1;
    }
    padded_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        int s = ((counts[e] + P - 1) / P) * P; /* ceil(c/P)*P, 0 when c = 0 */
        padded_offsets[e + 1] = padded_offsets[e] + s;
    }
    for (long long r = 0; r < R; ++r) {
        row_src[r] = -1;
        row_gate[r] = 0.0;
    }
    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    if (!next) return OR_ERR_ARG;
    for (int e = 0; e < E; ++e) next[e] = padded_offsets[e];
    for (long long a = 0; a < A; ++a) { /* ascending a: stable inside a segment */
        int e = idx[a];
        int r = next[e]++;
        perm_row[a] = r;
        row_src[r] = (int32_t)a;
        row_gate[r] = w ? w[a] : 1.0;
    }
    free(next);
    int nb = 0;
    for (int e = 0; e < E; ++e) {
        for (int m = 0; m < counts[e]; m += P) {
            int valid = counts[e] - m < P ? counts[e] - m : P;
            block_metadata[3 * nb + 0] = e;
            block_metadata[3 * nb + 1] = padded_offsets[e] + m;
            block_metadata[3 * nb + 2] = valid;
            ++nb;
        }
    }
    *num_blocks = nb;
    return OR_OK;
}

/* The receiving side of the expert-parallel dispatch ("Dropless and grouped
 * GEMM", sec. 4 step 5 and sec. 14: the exchange lands rows already grouped by
 * expert and padded; the receiver learns how many rows each sender has for
 * each of its experts).  counts[s * E + e] rows of sender s for local expert
 * e.  Expert e's segment holds the senders' rows back to back, in sender
 * order, and is padded like any segment: size ceil(c_e / P) * P with
 * c_e = sum over s of counts[s, e].  piece_row[s * E + e] is where sender
 * s's rows for e begin.  The block table follows the segments exactly as in
 * or_build_offsets (its valid rows form a prefix of each segment). */
int or_blocks_from_counts(int n_src, int E, int P, const int32_t *counts, int32_t *padded_offsets,
                          int32_t *block_metadata, int32_t *num_blocks, int32_t *piece_row)
{
    if (n_src <= 0 || E <= 0 || P <= 0) return OR_ERR_ARG;
    padded_offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        long long c = 0;
        for (int s = 0; s < n_src; ++s) {
            if (counts[(size_t)s * E + e] < 0) return OR_ERR_DATA;
            c += counts[(size_t)s * E + e];
        }
        padded_offsets[e + 1] = padded_offsets[e] + (int32_t)(((c + P - 1) / P) * P);
    }
    int nb = 0;
    for (int e = 0; e < E; ++e) {
        int row = padded_offsets[e];
        for (int s = 0; s < n_src; ++s) {
            piece_row[(size_t)s * E + e] = row;
            row += counts[(size_t)s * E + e];
        }
        int c = row - padded_offsets[e];
        for (int m = 0; m < c; m += P) {
            block_metadata[3 * nb + 0] = e;
            block_metadata[3 * nb + 1] = padded_offsets[e] + m;
            block_metadata[3 * nb + 2] = c - m < P ? c - m : P;
            ++nb;
        }
    }
    *num_blocks = nb;
    return OR_OK;
}

/* ------------------------------------------------------------- permute -- */

/* x_perm[r] = x[row_src[r] / k] for every valid padded row r; pad rows are
 * left as they are (the method never reads them). */
void or_permute(long long R, int d, int k, const uint16_t *x, const int32_t *row_src,
                uint16_t *x_perm)
{
#pragma omp parallel for schedule(static)
    for (long long r = 0; r < R; ++r) {
        if (row_src[r] < 0) continue;
        long long t = row_src[r] / k;
        memcpy(x_perm + (size_t)r * d, x + (size_t)t * d, sizeof(uint16_t) * (size_t)d);
    }
}

/* ------------------------------------------------------------- experts -- */

/* One SwiGLU expert applied to one row x[d]:
 *   g = x W1, u = x W3            (W1, W3 [d, de], the page's orientation)
 *   h = bf16( silu(g) * u ),  silu(g) = g / (1 + exp(-g))
 *   y = gate * (h W2)             (W2 [de, d])
 * Sums run over the contraction index in ascending order.  h is returned
 * (as the fp64 value of the bf16) when h_out is not NULL. */
static void expert_row(int d, int de, const uint16_t *x, const uint16_t *W1, const uint16_t *W3,
                       const uint16_t *W2, double gate, double *acc_g, double *acc_u, double *h_out,
                       double *y)
{
    for (int j = 0; j < de; ++j) acc_g[j] = acc_u[j] = 0.0;
    for (int i = 0; i < d; ++i) {
        double xi = or_bf16_to_double(x[i]);
        const uint16_t *w1 = W1 + (size_t)i * de;
        const uint16_t *w3 = W3 + (size_t)i * de;
        for (int j = 0; j < de; ++j) {
            acc_g[j] += xi * or_bf16_to_double(w1[j]);
            acc_u[j] += xi * or_bf16_to_double(w3[j]);
        }
    }
    for (int j = 0; j < de; ++j) {
        double g = acc_g[j];
        double silu = g / (1.0 + exp(-g));
        acc_g[j] = or_round_bf16(silu * acc_u[j]); /* acc_g now holds h */
        if (h_out) h_out[j] = acc_g[j];
    }
    for (int n = 0; n < d; ++n) y[n] = 0.0;
    for (int j = 0; j < de; ++j) {
        double hj = acc_g[j];
        const uint16_t *w2 = W2 + (size_t)j * d;
        for (int n = 0; n < d; ++n) y[n] += hj * or_bf16_to_double(w2[n]);
    }
    for (int n = 0; n < d; ++n) y[n] *= gate;
}

/* Grouped expert stage over a whole padded layout: for each block
 * [e, m_start, valid_m] of the table and each valid row r of it, h[r] and y[r]
 * of expert e applied to x_perm[r] with gate row_gate[r].  Pad rows are not
 * touched.  h may be NULL. */
int or_grouped_experts(int d, int de, int E, int num_blocks, const int32_t *block_metadata,
                       const uint16_t *x_perm, const uint16_t *W1, const uint16_t *W3,
                       const uint16_t *W2, const double *row_gate, double *h, double *y)
{
    for (int b = 0; b < num_blocks; ++b)
        if (block_metadata[3 * b] < 0 || block_metadata[3 * b] >= E) return OR_ERR_DATA;
    int bad = 0;
#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)de);
        double *au = (double *)malloc(sizeof(double) * (size_t)de);
        double *hy = (double *)malloc(sizeof(double) * (size_t)de);
        if (!ag || !au || !hy) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int b = 0; b < num_blocks; ++b) {
                int e = block_metadata[3 * b], m0 = block_metadata[3 * b + 1];
                int vm = block_metadata[3 * b + 2];
                const uint16_t *w1 = W1 + (size_t)e * d * de;
                const uint16_t *w3 = W3 + (size_t)e * d * de;
                const uint16_t *w2 = W2 + (size_t)e * de * d;
                for (int i = 0; i < vm; ++i) {
                    size_t r = (size_t)m0 + (size_t)i;
                    expert_row(d, de, x_perm + r * d, w1, w3, w2, row_gate[r], ag, au, hy,
                               y + r * d);
                    if (h) memcpy(h + r * de, hy, sizeof(double) * (size_t)de);
                }
            }
        }
        free(ag);
        free(au);
        free(hy);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* The same expert arithmetic on a compact list of n rows: row i is
 * xrows[i] sent to expert experts[i] with weight gates[i].  Used to sample
 * single rows of a large layout.  h may be NULL. */
int or_expert_rows(int n, int d, int de, int E, const uint16_t *xrows, const int32_t *experts,
                   const double *gates, const uint16_t *W1, const uint16_t *W3,
                   const uint16_t *W2, double *h, double *y)
{
    for (int i = 0; i < n; ++i)
        if (experts[i] < 0 || experts[i] >= E) return OR_ERR_DATA;
    int bad = 0;
#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)de);
        double *au = (double *)malloc(sizeof(double) * (size_t)de);
        double *hy = (double *)malloc(sizeof(double) * (size_t)de);
        if (!ag || !au || !hy) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int i = 0; i < n; ++i) {
                int e = experts[i];
                expert_row(d, de, xrows + (size_t)i * d, W1 + (size_t)e * d * de,
                           W3 + (size_t)e * d * de, W2 + (size_t)e * de * d, gates[i], ag, au, hy,
                           y + (size_t)i * d);
                if (h) memcpy(h + (size_t)i * de, hy, sizeof(double) * (size_t)de);
            }
        }
        free(ag);
        free(au);
        free(hy);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* Dense shared expert (gate 1) on n token rows xrows[n, d]: it reads the
 * original token rows, with no permute and no group sizes.  hs may be NULL. */
int or_shared_expert(int n, int d, int ds, const uint16_t *xrows, const uint16_t *Ws1,
                     const uint16_t *Ws3, const uint16_t *Ws2, double *hs, double *ys)
{
    int bad = 0;
#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)ds);
        double *au = (double *)malloc(sizeof(double) * (size_t)ds);
        double *hy = (double *)malloc(sizeof(double) * (size_t)ds);
        if (!ag || !au || !hy) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int t = 0; t < n; ++t) {
                expert_row(d, ds, xrows + (size_t)t * d, Ws1, Ws3, Ws2, 1.0, ag, au, hy,
                           ys + (size_t)t * d);
                if (hs) memcpy(hs + (size_t)t * ds, hy, sizeof(double) * (size_t)ds);
            }
        }
        free(ag);
        free(au);
        free(hy);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* ------------------------------------------------ fp8 (e4m3) expert weights -- */
/*
 * Weight-only fp8: a routed expert matrix is kept as 8-bit e4m3 codes with one
 * fp32 scale per output channel, and the weight it stands for is exactly
 * e4m3(q) * s.  "MoE & MLA operators", sec. 6.1 counts expert weights at one
 * byte per element (fp8 weights, b = 1); "Dropless and grouped GEMM", sec. 12
 * says the scale may be applied after the matmul when one scale covers the
 * whole contraction, which is the case for a per-output-channel scale.
 *
 * e4m3 (the OCP 8-bit float, E4M3 variant without infinities): a sign bit,
 * 4 exponent bits with bias 7 and 3 mantissa bits.  Exponent field 0 holds
 * the subnormals m * 2^-9; exponent 15 with mantissa 7 is NaN; the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 */
double or_e4m3_to_double(uint8_t code)
{
    int e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return (code & 0x80) ? -v : v;
}

/* The e4m3 code nearest to v, ties to the even code; magnitudes of 448 and
 * more give 448 (the saturating conversion); NaN gives 0x7F.  The value is
 * put on the grid of 4 significant bits (quantum 2^-9 at the bottom) with
 * nearbyint, i.e. round-half-even in the default rounding mode, and encoded. */
uint8_t or_double_to_e4m3(double v)
{
    if (v != v) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    int q = e - 4;      /* quantum of 4 significant bits */
    if (q < -9) q = -9;
    double r = ldexp(nearbyint(ldexp(a, -q)), q); /* <= 448 since a < 448 */
    if (r == 0.0) return sign;
    if (r <= ldexp(1.0, -6)) /* subnormal (2^-6 itself encodes as field 1, m 0) */
        return sign | (uint8_t)(int)ldexp(r, 9);
    int re;
    double f = frexp(r, &re); /* r = (2f) * 2^(re - 1), 2f in [1, 2) */
    int m = (int)((2.0 * f - 1.0) * 8.0);
    return sign | (uint8_t)((re - 1 + 7) << 3) | (uint8_t)m;
}

/* Per-output-channel quantization of one matrix stored [K][N] (row i is input
 * i, column n is output channel n), from bf16 bit patterns:
 *   amax[n] = max_i |W[i][n]|                   (exact: bf16 fits fp32)
 *   s[n]    = fp32(amax[n] / 448), 1 when amax[n] = 0
 *   q[i][n] = code nearest to fp32(W[i][n] / s[n])
 * Both divisions are single-precision IEEE divisions: the integer codes are
 * decided in fp32. */
void or_quantize_e4m3_columns(int K, int N, const uint16_t *W, uint8_t *q, float *s)
{
    for (int n = 0; n < N; ++n) {
        float amax = 0.0f;
        for (int i = 0; i < K; ++i) {
            float w = (float)or_bf16_to_double(W[(size_t)i * N + n]);
            if (fabsf(w) > amax) amax = fabsf(w);
        }
        float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
        s[n] = sc;
        for (int i = 0; i < K; ++i) {
            float w = (float)or_bf16_to_double(W[(size_t)i * N + n]);
            float ratio = w / sc;
            q[(size_t)i * N + n] = or_double_to_e4m3((double)ratio);
        }
    }
}

/* The same quantization for `batch` matrices of [K][N] stored back to back. */
void or_quantize_e4m3_batch(int batch, int K, int N, const uint16_t *W, uint8_t *q, float *s)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < batch; ++b)
        or_quantize_e4m3_columns(K, N, W + (size_t)b * K * N, q + (size_t)b * K * N,
                                 s + (size_t)b * N);
}

/* expert_row with e4m3 weights: Q1/Q3 [d][de] with scales S1/S3 [de], Q2
 * [de][d] with scales S2 [d]; every weight is e4m3(q) * s formed in fp64, so
 * the arithmetic is that of expert_row on the dequantized matrices. */
static void expert_row_w8(int d, int de, const uint16_t *x, const uint8_t *Q1, const float *S1,
                          const uint8_t *Q3, const float *S3, const uint8_t *Q2, const float *S2,
                          double gate, const double *dec, double *acc_g, double *acc_u,
                          double *h_out, double *y)
{
    for (int j = 0; j < de; ++j) acc_g[j] = acc_u[j] = 0.0;
    for (int i = 0; i < d; ++i) {
        double xi = or_bf16_to_double(x[i]);
        const uint8_t *q1 = Q1 + (size_t)i * de;
        const uint8_t *q3 = Q3 + (size_t)i * de;
        for (int j = 0; j < de; ++j) {
            acc_g[j] += xi * (dec[q1[j]] * (double)S1[j]);
            acc_u[j] += xi * (dec[q3[j]] * (double)S3[j]);
        }
    }
    for (int j = 0; j < de; ++j) {
        double g = acc_g[j];
        double silu = g / (1.0 + exp(-g));
        acc_g[j] = or_round_bf16(silu * acc_u[j]);
        if (h_out) h_out[j] = acc_g[j];
    }
    for (int n = 0; n < d; ++n) y[n] = 0.0;
    for (int j = 0; j < de; ++j) {
        double hj = acc_g[j];
        const uint8_t *q2 = Q2 + (size_t)j * d;
        for (int n = 0; n < d; ++n) y[n] += hj * (dec[q2[n]] * (double)S2[n]);
    }
    for (int n = 0; n < d; ++n) y[n] *= gate;
}

/* or_expert_rows with e4m3 expert weights: Q1/Q3 [E][d][de], S1/S3 [E][de],
 * Q2 [E][de][d], S2 [E][d]. */
int or_expert_rows_w8(int n, int d, int de, int E, const uint16_t *xrows, const int32_t *experts,
                      const double *gates, const uint8_t *Q1, const float *S1, const uint8_t *Q3,
                      const float *S3, const uint8_t *Q2, const float *S2, double *h, double *y)
{
    for (int i = 0; i < n; ++i)
        if (experts[i] < 0 || experts[i] >= E) return OR_ERR_DATA;
    double dec[256];
    for (int c = 0; c < 256; ++c) dec[c] = or_e4m3_to_double((uint8_t)c);
    int bad = 0;
#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)de);
        double *au = (double *)malloc(sizeof(double) * (size_t)de);
        double *hy = (double *)malloc(sizeof(double) * (size_t)de);
        if (!ag || !au || !hy) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int i = 0; i < n; ++i) {
                size_t e = (size_t)experts[i];
                expert_row_w8(d, de, xrows + (size_t)i * d, Q1 + e * d * de, S1 + e * de,
                              Q3 + e * d * de, S3 + e * de, Q2 + e * de * d, S2 + e * d, gates[i],
                              dec, ag, au, hy, y + (size_t)i * d);
                if (h) memcpy(h + (size_t)i * de, hy, sizeof(double) * (size_t)de);
            }
        }
        free(ag);
        free(au);
        free(hy);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* Element-wise e4m3 decode / encode of arrays (test helpers). */
void or_e4m3_to_double_array(long long n, const uint8_t *in, double *out)
{
    for (long long i = 0; i < n; ++i) out[i] = or_e4m3_to_double(in[i]);
}

void or_double_to_e4m3_array(long long n, const double *in, uint8_t *out)
{
    for (long long i = 0; i < n; ++i) out[i] = or_double_to_e4m3(in[i]);
}

/* ------------------------------------------------------------- combine -- */

/* out[t] = sum_{j = 0 .. k-1} y[perm_row[t*k + j]]  (+ ys[t])
 * in that order: the k routed rows first, ascending j, then the shared row.
 * y is the padded layout [R, d]; pad rows are never addressed. */
void or_combine(int T, int d, int k, const double *y, const int32_t *perm_row, const double *ys,
                double *out)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *o = out + (size_t)t * d;
        for (int n = 0; n < d; ++n) o[n] = 0.0;
        for (int j = 0; j < k; ++j) {
            const double *yr = y + (size_t)perm_row[(size_t)t * k + j] * d;
            for (int n = 0; n < d; ++n) o[n] += yr[n];
        }
        if (ys)
            for (int n = 0; n < d; ++n) o[n] += ys[(size_t)t * d + n];
    }
}

/* ------------------------------------------------------ direct evaluation -- */

/* The same layer without any re-layout, for the n tokens listed in tok[]:
 * the k chosen experts are applied to the token's own row and summed with
 * their routing weights in ascending j, then the shared row ys_rows[i] (if
 * given) is added.  Sec. 2.3 of the TileLang page states that permute ->
 * experts -> scatter-reduce equals this exactly. */
int or_direct_layer(int n, const int32_t *tok, int d, int de, int E, int k, const uint16_t *x,
                    const uint16_t *W1, const uint16_t *W3, const uint16_t *W2,
                    const int32_t *topk_idx, const double *topk_w, const double *ys_rows,
                    double *out)
{
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[(size_t)tok[i] * k + j];
            if (e < 0 || e >= E) return OR_ERR_DATA;
        }
    int bad = 0;
#pragma omp parallel
    {
        double *ag = (double *)malloc(sizeof(double) * (size_t)de);
        double *au = (double *)malloc(sizeof(double) * (size_t)de);
        double *yy = (double *)malloc(sizeof(double) * (size_t)d);
        if (!ag || !au || !yy) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int i = 0; i < n; ++i) {
                size_t t = (size_t)tok[i];
                double *o = out + (size_t)i * d;
                for (int c = 0; c < d; ++c) o[c] = 0.0;
                for (int j = 0; j < k; ++j) {
                    int e = topk_idx[t * k + j];
                    expert_row(d, de, x + t * d, W1 + (size_t)e * d * de, W3 + (size_t)e * d * de,
                               W2 + (size_t)e * de * d, topk_w[t * k + j], ag, au, NULL, yy);
                    for (int c = 0; c < d; ++c) o[c] += yy[c];
                }
                if (ys_rows)
                    for (int c = 0; c < d; ++c) o[c] += ys_rows[(size_t)i * d + c];
            }
        }
        free(ag);
        free(au);
        free(yy);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/* ------------------------------------------------------------- backward -- */
/*
 * Gradient of the layer forward above for an upstream gradient dout [T, d]:
 *   out[t] = sum_j p[t,j] * (h_a W2[e]) + ys[t],  a = t*k + j, e = idx[a],
 *   h_a = bf16(silu(x_t W1[e]) * (x_t W3[e])),  p = routing weights.
 * Readings: the expert choice (top-k) is a constant of the step; the bf16
 * rounding of h is passed straight through (its derivative is taken as 1, and
 * the rounded value is the one multiplied by W2 and by the gradient); with a
 * router the weights are a softmax over the k chosen logits, so
 *   dlogit[t, idx[t,j]] = p_j * (dp_j - sum_i p_i dp_i),  other experts 0,
 * and the logit bias receives the sum over tokens.  ("Dropless and grouped
 * GEMM", sec. 4 notes that the backward only needs the sort indices saved
 * from the forward: the permutation is undone by the transposed gather.)
 * Outputs (fp64, every array overwritten): dx [T, d]; dgates [T, k];
 * dW1, dW3 [E, d, de]; dW2 [E, de, d]; with Wg: dlogits [T, E], dWg [d, E],
 * dbias [E]; with a shared expert (ds > 0): dWs1, dWs3 [d, ds], dWs2 [ds, d]. */
static double or_sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* One SwiGLU expert's backward for one row: given x [d] (bf16), the expert's
 * W1/W3 [d][de], W2 [de][d], the row's weight p and the upstream dout [d]:
 * hr [de] (bf16-rounded h), dz = p * dout [d], dp = <dout, h W2>, dg, du [de],
 * and dxa [d] = dg W1^T + du W3^T. */
static void expert_row_bwd(int d, int de, const uint16_t *x, const uint16_t *W1,
                           const uint16_t *W3, const uint16_t *W2, double p, const double *dout,
                           double *g, double *u, double *hr, double *dz, double *dp, double *dg,
                           double *du, double *dxa)
{
    for (int j = 0; j < de; ++j) g[j] = u[j] = 0.0;
    for (int i = 0; i < d; ++i) {
        double xi = or_bf16_to_double(x[i]);
        for (int j = 0; j < de; ++j) {
            g[j] += xi * or_bf16_to_double(W1[(size_t)i * de + j]);
            u[j] += xi * or_bf16_to_double(W3[(size_t)i * de + j]);
        }
    }
    for (int j = 0; j < de; ++j) hr[j] = or_round_bf16(g[j] * or_sigmoid(g[j]) * u[j]);
    double s = 0.0;
    for (int n = 0; n < d; ++n) {
        double z = 0.0;
        for (int j = 0; j < de; ++j) z += hr[j] * or_bf16_to_double(W2[(size_t)j * d + n]);
        s += dout[n] * z;
        dz[n] = p * dout[n];
    }
    *dp = s;
    for (int j = 0; j < de; ++j) {
        double dh = 0.0;
        for (int n = 0; n < d; ++n) dh += dz[n] * or_bf16_to_double(W2[(size_t)j * d + n]);
        double sg = or_sigmoid(g[j]);
        dg[j] = dh * u[j] * sg * (1.0 + g[j] * (1.0 - sg));
        du[j] = dh * g[j] * sg;
    }
    for (int i = 0; i < d; ++i) {
        double acc = 0.0;
        for (int j = 0; j < de; ++j)
            acc += dg[j] * or_bf16_to_double(W1[(size_t)i * de + j]) +
                   du[j] * or_bf16_to_double(W3[(size_t)i * de + j]);
        dxa[i] = acc;
    }
}

int or_layer_backward(int T, int d, int de, int E, int k, int ds, const uint16_t *x,
                      const uint16_t *Wg, const int32_t *idx, const double *gates,
                      const uint16_t *W1, const uint16_t *W3, const uint16_t *W2,
                      const uint16_t *Ws1, const uint16_t *Ws3, const uint16_t *Ws2,
                      const double *dout, double *dx, double *dgates, double *dlogits, double *dWg,
                      double *dbias, double *dW1, double *dW3, double *dW2, double *dWs1,
                      double *dWs3, double *dWs2)
{
    const long long A = (long long)T * k;
    for (long long a = 0; a < A; ++a)
        if (idx[a] < 0 || idx[a] >= E) return OR_ERR_DATA;
    double *hr = (double *)malloc(sizeof(double) * (size_t)A * de);
    double *dz = (double *)malloc(sizeof(double) * (size_t)A * d);
    double *dg = (double *)malloc(sizeof(double) * (size_t)A * de);
    double *du = (double *)malloc(sizeof(double) * (size_t)A * de);
    double *dxa = (double *)malloc(sizeof(double) * (size_t)A * d);
    if (!hr || !dz || !dg || !du || !dxa) {
        free(hr); free(dz); free(dg); free(du); free(dxa);
        return OR_ERR_ARG;
    }
    int bad = 0;
    /* per assignment */
#pragma omp parallel
    {
        double *g = (double *)malloc(sizeof(double) * (size_t)de);
        double *u = (double *)malloc(sizeof(double) * (size_t)de);
        if (!g || !u) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long long a = 0; a < A; ++a) {
                size_t e = (size_t)idx[a], t = (size_t)(a / k);
                expert_row_bwd(d, de, x + t * d, W1 + e * d * de, W3 + e * d * de, W2 + e * de * d,
                               gates[a], dout + t * d, g, u, hr + a * de, dz + a * d, dgates + a,
                               dg + a * de, du + a * de, dxa + a * d);
            }
        }
        free(g);
        free(u);
    }
    if (bad) {
        free(hr); free(dz); free(dg); free(du); free(dxa);
        return OR_ERR_ARG;
    }
    /* expert weight gradients: sums over the expert's rows, ascending a */
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
        double *w1 = dW1 + (size_t)e * d * de, *w3 = dW3 + (size_t)e * d * de;
        double *w2 = dW2 + (size_t)e * de * d;
        memset(w1, 0, sizeof(double) * (size_t)d * de);
        memset(w3, 0, sizeof(double) * (size_t)d * de);
        memset(w2, 0, sizeof(double) * (size_t)de * d);
        for (long long a = 0; a < A; ++a) {
            if (idx[a] != e) continue;
            const uint16_t *xt = x + (size_t)(a / k) * d;
            for (int j = 0; j < de; ++j)
                for (int n = 0; n < d; ++n) w2[(size_t)j * d + n] += hr[a * de + j] * dz[a * d + n];
            for (int i = 0; i < d; ++i) {
                double xi = or_bf16_to_double(xt[i]);
                for (int j = 0; j < de; ++j) {
                    w1[(size_t)i * de + j] += xi * dg[a * de + j];
                    w3[(size_t)i * de + j] += xi * du[a * de + j];
                }
            }
        }
    }
    /* dx: the routed rows of each token (ascending j) */
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        double *o = dx + (size_t)t * d;
        for (int i = 0; i < d; ++i) o[i] = 0.0;
        for (int j = 0; j < k; ++j)
            for (int i = 0; i < d; ++i) o[i] += dxa[((size_t)t * k + j) * d + i];
    }
    /* router */
    if (Wg) {
        for (size_t q = 0; q < (size_t)T * E; ++q) dlogits[q] = 0.0;
        for (int t = 0; t < T; ++t) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += gates[(size_t)t * k + j] * dgates[(size_t)t * k + j];
            for (int j = 0; j < k; ++j) {
                size_t a = (size_t)t * k + j;
                dlogits[(size_t)t * E + idx[a]] += gates[a] * (dgates[a] - s);
            }
        }
        for (int e = 0; e < E; ++e) {
            double s = 0.0;
            for (int t = 0; t < T; ++t) s += dlogits[(size_t)t * E + e];
            dbias[e] = s;
        }
#pragma omp parallel for schedule(static)
        for (int i = 0; i < d; ++i)
            for (int e = 0; e < E; ++e) {
                double s = 0.0;
                for (int t = 0; t < T; ++t)
                    s += or_bf16_to_double(x[(size_t)t * d + i]) * dlogits[(size_t)t * E + e];
                dWg[(size_t)i * E + e] = s;
            }
#pragma omp parallel for schedule(static)
        for (int t = 0; t < T; ++t)
            for (int i = 0; i < d; ++i) {
                double s = 0.0;
                for (int e = 0; e < E; ++e)
                    s += dlogits[(size_t)t * E + e] * or_bf16_to_double(Wg[(size_t)i * E + e]);
                dx[(size_t)t * d + i] += s;
            }
    }
    /* shared expert: the same row backward with weight 1 for every token */
    if (ds > 0) {
        double *shr = (double *)malloc(sizeof(double) * (size_t)T * ds);
        double *sdg = (double *)malloc(sizeof(double) * (size_t)T * ds);
        double *sdu = (double *)malloc(sizeof(double) * (size_t)T * ds);
        double *sdx = (double *)malloc(sizeof(double) * (size_t)T * d);
        double *sdz = (double *)malloc(sizeof(double) * (size_t)T * d);
        if (!shr || !sdg || !sdu || !sdx || !sdz) {
            bad = 1;
        } else {
#pragma omp parallel
            {
                double *g = (double *)malloc(sizeof(double) * (size_t)ds);
                double *u = (double *)malloc(sizeof(double) * (size_t)ds);
                double dp;
                if (g && u) {
#pragma omp for schedule(dynamic, 1)
                    for (int t = 0; t < T; ++t)
                        expert_row_bwd(d, ds, x + (size_t)t * d, Ws1, Ws3, Ws2, 1.0,
                                       dout + (size_t)t * d, g, u, shr + (size_t)t * ds,
                                       sdz + (size_t)t * d, &dp, sdg + (size_t)t * ds,
                                       sdu + (size_t)t * ds, sdx + (size_t)t * d);
                } else {
#pragma omp atomic write
                    bad = 1;
                }
                free(g);
                free(u);
            }
            if (!bad) {
#pragma omp parallel for schedule(static)
                for (int j = 0; j < ds; ++j)
                    for (int n = 0; n < d; ++n) {
                        double s = 0.0;
                        for (int t = 0; t < T; ++t) s += shr[(size_t)t * ds + j] * sdz[(size_t)t * d + n];
                        dWs2[(size_t)j * d + n] = s;
                    }
#pragma omp parallel for schedule(static)
                for (int i = 0; i < d; ++i)
                    for (int j = 0; j < ds; ++j) {
                        double s1 = 0.0, s3 = 0.0;
                        for (int t = 0; t < T; ++t) {
                            double xi = or_bf16_to_double(x[(size_t)t * d + i]);
                            s1 += xi * sdg[(size_t)t * ds + j];
                            s3 += xi * sdu[(size_t)t * ds + j];
                        }
                        dWs1[(size_t)i * ds + j] = s1;
                        dWs3[(size_t)i * ds + j] = s3;
                    }
                for (size_t q = 0; q < (size_t)T * d; ++q) dx[q] += sdx[q];
            }
        }
        free(shr); free(sdg); free(sdu); free(sdx); free(sdz);
    }
    free(hr); free(dz); free(dg); free(du); free(dxa);
    return bad ? OR_ERR_ARG : OR_OK;
}

/* Selected columns of one SwiGLU expert's weight gradients over a set of
 * rows ("Dropless and grouped GEMM", sec. 4: the backward of the expert GEMMs
 * over the rows routed to the expert; the layer backward above, restricted
 * to columns).  Row r brings its token row x_r (bf16 [d]), its upstream
 * gradient dout_r (fp64 [d]) and its routing weight p_r.  For each column j
 * of J (0 <= j < de):
 *   g = x_r . W1[:, j], u = x_r . W3[:, j], h = bf16(silu(g) u),
 *   dh = p_r dout_r . W2[j, :],
 *   dW2[j][n]  = sum_r h p_r dout_r[n]
 *   dW1[i][jj] = sum_r x_r[i] dh u silu'(g),  dW3[i][jj] = sum_r x_r[i] dh silu(g)
 * Outputs (fp64, overwritten): dW1c, dW3c [d][nj], dW2r [nj][d]. */
int or_weight_grad_columns(int n, int d, int de, const uint16_t *x, const double *dout,
                           const double *p, const uint16_t *W1, const uint16_t *W3,
                           const uint16_t *W2, int nj, const int32_t *J, double *dW1c,
                           double *dW3c, double *dW2r)
{
    if (n < 0 || d <= 0 || de <= 0 || nj <= 0) return OR_ERR_ARG;
    for (int jj = 0; jj < nj; ++jj)
        if (J[jj] < 0 || J[jj] >= de) return OR_ERR_ARG;
    for (size_t q = 0; q < (size_t)d * nj; ++q) dW1c[q] = dW3c[q] = 0.0;
    for (size_t q = 0; q < (size_t)nj * d; ++q) dW2r[q] = 0.0;
    for (int r = 0; r < n; ++r) {
        const uint16_t *xr = x + (size_t)r * d;
        const double *dr = dout + (size_t)r * d;
        for (int jj = 0; jj < nj; ++jj) {
            const int j = J[jj];
            double g = 0.0, u = 0.0, dh = 0.0;
            for (int i = 0; i < d; ++i) {
                const double xi = or_bf16_to_double(xr[i]);
                g += xi * or_bf16_to_double(W1[(size_t)i * de + j]);
                u += xi * or_bf16_to_double(W3[(size_t)i * de + j]);
            }
            for (int i = 0; i < d; ++i) dh += p[r] * dr[i] * or_bf16_to_double(W2[(size_t)j * d + i]);
            const double sg = or_sigmoid(g);
            const double h = or_round_bf16(g * sg * u);
            const double dg = dh * u * sg * (1.0 + g * (1.0 - sg));
            const double du = dh * g * sg;
            for (int i = 0; i < d; ++i) {
                const double xi = or_bf16_to_double(xr[i]);
                dW1c[(size_t)i * nj + jj] += xi * dg;
                dW3c[(size_t)i * nj + jj] += xi * du;
                dW2r[(size_t)jj * d + i] += h * p[r] * dr[i];
            }
        }
    }
    return OR_OK;
}

/* Element-wise bf16 rounding of an fp64 array (test helper). */
void or_round_bf16_array(long long n, const double *in, double *out)
{
    for (long long i = 0; i < n; ++i) out[i] = or_round_bf16(in[i]);
}

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
