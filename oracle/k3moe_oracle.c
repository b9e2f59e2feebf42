/*
 * k3moe_oracle.c -- the CPU oracle of the routed-expert layer.
 *
 * TEST INFRASTRUCTURE.  This file is the plain, slow, obviously correct
 * restatement of what the layer computes, used to check the GPU library.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or helper with the GPU path.
 *
 * Source of every rule below: the "kimi-k3-in-c" README (Kimi K3 inference in
 * portable C99; upstar.dev mirror), Part II "How it works":
 *   - section 4 "Reduction one: the experts already ship at half a byte":
 *     the MXFP4 format (E2M1 table, E8M0 scale 2^(b-127) per 32 weights, byte
 *     255 read as zero, low nibble = even element) and the MXFP4 mat-vec
 *     (per-group partial sum, scaled, never dequantised to memory);
 *   - section 5 "Kernels with a floating point contract": double accumulation;
 *     bf16 widened to f32 by a 16-bit shift;
 *   - section 9 "Picking 16 experts of 896": the router (sigmoid score in
 *     float, bias added for selection only, top-k by repeated maximum with a
 *     strict comparison so the lower index wins a tie, weights from the
 *     unbiased score, renormalised when the sum is positive, times the routed
 *     scale), the Stable LatentMoE expert loop (gate = w1, up = w3,
 *     down = w2, weighted accumulation; shared experts added unweighted), and
 *     the SiTU-GLU activation (the sigmoid reads the uncapped gate).
 *
 * The layer built here is the latent-space part of that loop: its input x is
 * already the expert latent (width d), the router scores x directly, and the
 * d -> f -> d shared experts read the same x.  k3o_forward_full adds what sits
 * around it in the write-up's k3_moe (same section): the full-width router
 * input, the down and up projections, the RMSNorm of the aggregate and the
 * full-width shared experts.
 *
 * Precision: the router follows the write-up's float steps exactly, because
 * float rounding decides which experts win; everything else is computed in
 * double and rounded to float once, at the output.
 *
 * Parity pins (each checked by the CPU test-suite, against facts other than
 * this file): E2M1/E8M0 decode against the printed table and the closed form
 * for all 16 x 256 (code, byte) pairs; nibble order by a positional fixture;
 * the MXFP4 mat-vec against a dense fp64 mat-vec of the decoded matrix; top-k
 * against a full lexicographic sort; an adversarial bias fixture; the routing
 * invariants; SiTU's closed-form bound and its small-input limit; the whole
 * layer against an independent dense fp64 brute force on tiny layers; the
 * special cases k = E and E = k = 1; and the shared-expert output's
 * independence from routing.  The full-width block: against an independent
 * dense fp64 brute force on tiny blocks, its reduction to the latent layer
 * (identity projections, no norm), and the norm's scale invariance.  No
 * function here is "parity unpinned".
 *
 * Build: cc -O2 -std=c99 -fPIC -shared -fopenmp -ffp-contract=off -lm
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
static int in_parallel(void) { return omp_in_parallel(); }
#else
static int in_parallel(void) { return 0; }
#endif

/* ------------------------------------------------------------------ config */

typedef struct {
    int32_t d;            /* latent width: input and output of every expert */
    int32_t f;            /* expert FFN width */
    int32_t n_experts;    /* routed experts E */
    int32_t top_k;        /* experts chosen per token k */
    int32_t n_shared;     /* dense shared experts S (may be 0) */
    int32_t group;        /* MXFP4 block size (32) */
    float situ_b1;        /* SiTU gate cap beta1 (4.0) */
    float situ_b2;        /* SiTU linear cap beta2 (25.0) */
    int32_t renorm;       /* 1: renormalise the chosen scores to sum 1 */
    float routed_scale;   /* multiplier on the routing weights (1.0) */
} k3o_cfg;

/* One routed expert in checkpoint layout.  w1, w3: [f][d]; w2: [d][f].
 * packed [rows][cols/2], scale [rows][cols/group]. */
typedef struct {
    const uint8_t *w1_packed, *w1_scale;
    const uint8_t *w3_packed, *w3_scale;
    const uint8_t *w2_packed, *w2_scale;
} k3o_expert;

enum { K3O_OK = 0, K3O_EINVAL = 1, K3O_EMISSING = 2, K3O_ENOMEM = 3 };

int k3o_check_cfg(const k3o_cfg *c)
{
    if (!c || c->d <= 0 || c->f <= 0 || c->n_experts <= 0 || c->top_k <= 0 ||
        c->n_shared < 0 || c->group <= 0 || c->top_k > c->n_experts ||
        c->d % c->group || c->f % c->group || c->group % 2 ||
        !(c->situ_b1 > 0.0f) || !(c->situ_b2 > 0.0f) ||
        (c->renorm != 0 && c->renorm != 1) || !isfinite(c->routed_scale))
        return K3O_EINVAL;
    return K3O_OK;
}

/* ------------------------------------------------------------ formats (s4) */

/* E2M1: sign, two exponent bits, one mantissa bit; the sixteen values in
 * code order as the write-up prints them. */
static const double E2M1[16] = {
    0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
    -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double k3o_e2m1(int code) { return E2M1[code & 15]; }

/* E8M0: 2^(b-127); byte 255 (NaN in the MX specification) reads as zero. */
double k3o_e8m0(int byte)
{
    return (byte == 255) ? 0.0 : ldexp(1.0, (byte & 255) - 127);
}

/* bf16 -> float: the top 16 bits of a float, so a 16-bit shift is exact. */
float k3o_bf16(uint16_t b)
{
    union { uint32_t u; float f; } v;
    v.u = (uint32_t)b << 16;
    return v.f;
}

/* Weight (row, col) of an MXFP4 matrix, decoded exactly to double. */
double k3o_mxfp4_weight(const uint8_t *packed, const uint8_t *scales, int cols,
                        int group, int row, int col)
{
    const uint8_t byte = packed[(size_t)row * (size_t)(cols / 2) + (size_t)(col / 2)];
    const int code = (col & 1) ? (byte >> 4) : (byte & 15);  /* low nibble = even */
    const double s = k3o_e8m0(scales[(size_t)row * (size_t)(cols / group) + (size_t)(col / group)]);
    return E2M1[code] * s;
}

/* y[rows] = W x with W MXFP4 [rows][in]: for each group of `group` inputs a
 * partial dot product in double, times the group's scale; a zero scale skips
 * the group.  Nothing is dequantised to memory.  (write-up s4) */
void k3o_mxfp4_matvec(double *y, const double *x, const uint8_t *packed,
                      const uint8_t *scales, int in, int rows, int group)
{
    const int ngroup = in / group;
    const size_t rowbytes = (size_t)in / 2;
#pragma omp parallel for schedule(static) if (rows >= 256 && !in_parallel())
    for (int o = 0; o < rows; o++) {
        const uint8_t *pb = packed + (size_t)o * rowbytes;
        const uint8_t *sb = scales + (size_t)o * (size_t)ngroup;
        double acc = 0.0;
        for (int g = 0; g < ngroup; g++) {
            const double s = k3o_e8m0(sb[g]);
            if (s == 0.0)
                continue;
            double part = 0.0;
            for (int k = 0; k < group; k += 2) {
                const uint8_t b = pb[(g * group + k) / 2];
                part += x[g * group + k] * E2M1[b & 15];       /* even <- low nibble */
                part += x[g * group + k + 1] * E2M1[b >> 4];   /* odd  <- high nibble */
            }
            acc += part * s;
        }
        y[o] = acc;
    }
}

/* y[rows] = W x with W bf16 [rows][in], double accumulation.  (write-up s5) */
void k3o_bf16_matvec(double *y, const double *x, const uint16_t *W, int in, int rows)
{
#pragma omp parallel for schedule(static) if (rows >= 256 && !in_parallel())
    for (int o = 0; o < rows; o++) {
        const uint16_t *row = W + (size_t)o * (size_t)in;
        double acc = 0.0;
        for (int i = 0; i < in; i++)
            acc += (double)k3o_bf16(row[i]) * x[i];
        y[o] = acc;
    }
}

/* ------------------------------------------------------------- SiTU (s9) */

/* SiTU-GLU on one (gate, up) pair: b1*tanh(g/b1) * sigmoid(g) * b2*tanh(u/b2).
 * The sigmoid reads the uncapped gate g.  |result| < b1*b2. */
double k3o_situ(double g, double u, double b1, double b2)
{
    const double a = b1 * tanh(g / b1) * (1.0 / (1.0 + exp(-g)));
    return a * (b2 * tanh(u / b2));
}

/* ------------------------------------------------------------ router (s9) */

/* Selection for one token.  sc[e] = 1/(1+expf(-logit)) in float (unbiased),
 * ch[e] = sc[e] + bias[e] (selection).  Top-k by repeated maximum of ch with a
 * strict '>' (ties keep the lower index).  Weights are sc of the chosen
 * experts, renormalised by their float sum when renorm and the sum is > 0,
 * then multiplied by routed_scale.  *gap = ch(k-th chosen) - ch(best unchosen),
 * or +inf when every expert is chosen. */
static void route_one(const k3o_cfg *c, const float *sc, const float *ch,
                      int32_t *idx, float *w, float *gap, char *taken)
{
    const int E = c->n_experts, k = c->top_k;
    memset(taken, 0, (size_t)E);
    for (int j = 0; j < k; j++) {
        int best = -1;
        for (int e = 0; e < E; e++)
            if (!taken[e] && (best < 0 || ch[e] > ch[best]))
                best = e;
        taken[best] = 1;
        idx[j] = best;
        w[j] = sc[best];
    }
    if (c->renorm) {
        float s = 0.0f;
        for (int j = 0; j < k; j++)
            s += w[j];
        if (s > 0.0f)
            for (int j = 0; j < k; j++)
                w[j] /= s;
    }
    for (int j = 0; j < k; j++)
        w[j] *= c->routed_scale;
    if (gap) {
        int best = -1;
        for (int e = 0; e < E; e++)
            if (!taken[e] && (best < 0 || ch[e] > ch[best]))
                best = e;
        *gap = (best < 0) ? INFINITY : ch[idx[k - 1]] - ch[best];
    }
}

/* Router for T tokens.  x [T][d] bf16, Wr [E][d] bf16, bias [E] or NULL.
 * Outputs idx [T][k], w [T][k]; optional sc_out/ch_out [T][E] and gap [T]. */
int k3o_route(const k3o_cfg *c, int T, const uint16_t *x, const uint16_t *Wr,
              const float *bias, int32_t *idx, float *w, float *sc_out,
              float *ch_out, float *gap)
{
    if (k3o_check_cfg(c) || T < 0 || (T > 0 && (!x || !Wr || !idx || !w)))
        return K3O_EINVAL;
    const int d = c->d, E = c->n_experts, k = c->top_k;
    int err = K3O_OK;
#pragma omp parallel
    {
        float *sc = malloc(sizeof(float) * (size_t)E);
        float *ch = malloc(sizeof(float) * (size_t)E);
        char *taken = malloc((size_t)E);
        double *xd = malloc(sizeof(double) * (size_t)d);
        if (!sc || !ch || !taken || !xd) {
#pragma omp atomic write
            err = K3O_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int t = 0; t < T; t++) {
                for (int i = 0; i < d; i++)
                    xd[i] = (double)k3o_bf16(x[(size_t)t * d + i]);
                for (int e = 0; e < E; e++) {
                    const uint16_t *row = Wr + (size_t)e * d;
                    double acc = 0.0;
                    for (int i = 0; i < d; i++)
                        acc += xd[i] * (double)k3o_bf16(row[i]);
                    const float logit = (float)acc;
                    sc[e] = 1.0f / (1.0f + expf(-logit));
                    ch[e] = sc[e] + (bias ? bias[e] : 0.0f);
                }
                route_one(c, sc, ch, idx + (size_t)t * k, w + (size_t)t * k,
                          gap ? gap + t : NULL, taken);
                if (sc_out)
                    memcpy(sc_out + (size_t)t * E, sc, sizeof(float) * (size_t)E);
                if (ch_out)
                    memcpy(ch_out + (size_t)t * E, ch, sizeof(float) * (size_t)E);
            }
        }
        free(sc);
        free(ch);
        free(taken);
        free(xd);
    }
    return err;
}

/* Top-k and weights from given float scores (no logits): the selection step
 * alone, for fixtures that fix sc and ch directly. */
int k3o_select(const k3o_cfg *c, int T, const float *sc, const float *ch,
               int32_t *idx, float *w, float *gap)
{
    if (k3o_check_cfg(c) || T < 0)
        return K3O_EINVAL;
    char *taken = malloc((size_t)c->n_experts);
    if (!taken)
        return K3O_ENOMEM;
    for (int t = 0; t < T; t++)
        route_one(c, sc + (size_t)t * c->n_experts, ch + (size_t)t * c->n_experts,
                  idx + (size_t)t * c->top_k, w + (size_t)t * c->top_k,
                  gap ? gap + t : NULL, taken);
    free(taken);
    return K3O_OK;
}

/* ------------------------------------------------------ token -> expert map */

/* Counting sort of the T*k slots by expert, stable in the flat slot id t*k+j:
 * offsets [E+1] is the exclusive prefix sum of the per-expert counts
 * (offsets[E] = T*k); perm[p] is the slot id at position p. */
int k3o_perm(int T, int E, int k, const int32_t *idx, int32_t *offsets, int32_t *perm)
{
    if (T < 0 || E <= 0 || k <= 0)
        return K3O_EINVAL;
    const size_t n = (size_t)T * (size_t)k;
    for (int e = 0; e <= E; e++)
        offsets[e] = 0;
    for (size_t s = 0; s < n; s++) {
        if (idx[s] < 0 || idx[s] >= E)
            return K3O_EINVAL;
        offsets[idx[s] + 1]++;
    }
    for (int e = 0; e < E; e++)
        offsets[e + 1] += offsets[e];
    int32_t *fill = malloc(sizeof(int32_t) * (size_t)E);
    if (!fill)
        return K3O_ENOMEM;
    memcpy(fill, offsets, sizeof(int32_t) * (size_t)E);
    for (size_t s = 0; s < n; s++)
        perm[fill[idx[s]]++] = (int32_t)s;
    free(fill);
    return K3O_OK;
}

/* --------------------------------------------------------- expert layer (s9) */

/* y [d] = W2 . situ(W1 x, W3 x) for one routed MXFP4 expert on x [d];
 * g, u, h are scratch of f doubles. */
static void expert_ffn(const k3o_cfg *c, const k3o_expert *q, const double *x,
                       double *g, double *u, double *h, double *y)
{
    const int d = c->d, f = c->f, G = c->group;
    k3o_mxfp4_matvec(g, x, q->w1_packed, q->w1_scale, d, f, G);
    k3o_mxfp4_matvec(u, x, q->w3_packed, q->w3_scale, d, f, G);
    for (int i = 0; i < f; i++)
        h[i] = k3o_situ(g[i], u[i], c->situ_b1, c->situ_b2);
    k3o_mxfp4_matvec(y, h, q->w2_packed, q->w2_scale, f, d, G);
}

/* Every selected expert of routing idx [T][k] must be present (non-NULL). */
static int check_routing(const k3o_cfg *c, int T, const int32_t *idx, const k3o_expert *experts)
{
    for (size_t s = 0; s < (size_t)T * (size_t)c->top_k; s++) {
        const int e = idx[s];
        if (e < 0 || e >= c->n_experts)
            return K3O_EINVAL;
        const k3o_expert *q = experts + e;
        if (!q->w1_packed || !q->w1_scale || !q->w3_packed || !q->w3_scale ||
            !q->w2_packed || !q->w2_scale)
            return K3O_EMISSING;
    }
    return K3O_OK;
}

/* out[t] = sum_j w[t][j] * FFN_{idx[t][j]}(x_t) + sum_s SharedFFN_s(x_t), where
 * FFN(x) = W2 . situ(W1 x, W3 x) on MXFP4 weights and the shared experts are
 * the same form on bf16 weights, added with weight one.  Everything in double;
 * out rounded to float once.  Optional out_shared [T][d] receives the shared
 * part alone.  A selected expert with NULL tensors is an error (the write-up
 * counts a dropped expert and refuses to call the run valid). */
int k3o_forward(const k3o_cfg *c, int T, const uint16_t *x, const int32_t *idx,
                const float *w, const k3o_expert *experts, const uint16_t *sh_w1,
                const uint16_t *sh_w3, const uint16_t *sh_w2, float *out,
                float *out_shared)
{
    if (k3o_check_cfg(c) || T < 0 || (T > 0 && (!x || !out)) ||
        (c->n_shared > 0 && T > 0 && (!sh_w1 || !sh_w3 || !sh_w2)))
        return K3O_EINVAL;
    const int d = c->d, f = c->f, k = c->top_k;
    int err = check_routing(c, T, idx, experts);
    if (err)
        return err;
#pragma omp parallel if (T > 1)
    {
        double *xd = malloc(sizeof(double) * (size_t)d);
        double *g = malloc(sizeof(double) * (size_t)f);
        double *u = malloc(sizeof(double) * (size_t)f);
        double *h = malloc(sizeof(double) * (size_t)f);
        double *y = malloc(sizeof(double) * (size_t)d);
        double *acc = malloc(sizeof(double) * (size_t)d);
        double *accs = malloc(sizeof(double) * (size_t)d);
        if (!xd || !g || !u || !h || !y || !acc || !accs) {
#pragma omp atomic write
            err = K3O_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int t = 0; t < T; t++) {
                for (int i = 0; i < d; i++)
                    xd[i] = (double)k3o_bf16(x[(size_t)t * d + i]);
                for (int i = 0; i < d; i++)
                    acc[i] = accs[i] = 0.0;
                /* routed experts, weighted */
                for (int j = 0; j < k; j++) {
                    const k3o_expert *q = experts + idx[(size_t)t * k + j];
                    const double wt = (double)w[(size_t)t * k + j];
                    expert_ffn(c, q, xd, g, u, h, y);
                    for (int i = 0; i < d; i++)
                        acc[i] += wt * y[i];
                }
                /* shared experts, unweighted, on the same input */
                for (int s = 0; s < c->n_shared; s++) {
                    k3o_bf16_matvec(g, xd, sh_w1 + (size_t)s * f * d, d, f);
                    k3o_bf16_matvec(u, xd, sh_w3 + (size_t)s * f * d, d, f);
                    for (int i = 0; i < f; i++)
                        h[i] = k3o_situ(g[i], u[i], c->situ_b1, c->situ_b2);
                    k3o_bf16_matvec(y, h, sh_w2 + (size_t)s * d * f, f, d);
                    for (int i = 0; i < d; i++)
                        accs[i] += y[i];
                }
                for (int i = 0; i < d; i++)
                    out[(size_t)t * d + i] = (float)(acc[i] + accs[i]);
                if (out_shared)
                    for (int i = 0; i < d; i++)
                        out_shared[(size_t)t * d + i] = (float)accs[i];
            }
        }
        free(xd); free(g); free(u); free(h); free(y); free(acc); free(accs);
    }
    return err;
}

/* ------------------------------------------- full-width block (s9, k3_moe) */

/* The whole Stable LatentMoE block for T full-width tokens h [T][H] and given
 * routing (the router reads the full-width token: k3o_route on a config whose
 * d is H), in the order of the write-up's six steps:
 *   z = Wd h                          Wd [d][H] bf16, into the expert latent
 *   a = sum_j w_j FFN_{idx_j}(z)      the routed experts, as in k3o_forward
 *   a_i = a_i gain_i / sqrt(sum_i a_i^2 / d + eps)   when latent_norm: the norm
 *                                     of the AGGREGATE, never of one expert
 *   out = Wu a                        Wu [H][d] bf16, back to full width
 *   out += Sh2 situ(Sh1 h, Sh3 h)     the shared experts on the ORIGINAL h,
 *                                     fused to one FFN of width SI = S f:
 *                                     Sh1, Sh3 [SI][H], Sh2 [H][SI] bf16;
 *                                     added unweighted
 * c describes the expert latent (d, f, E, k) and S = c->n_shared.  Everything
 * in double, out [T][H] rounded to float once. */
int k3o_forward_full(const k3o_cfg *c, int H, int latent_norm, double eps, int T,
                     const uint16_t *h, const int32_t *idx, const float *w,
                     const uint16_t *Wd, const k3o_expert *experts, const float *gain,
                     const uint16_t *Wu, const uint16_t *sh1, const uint16_t *sh3,
                     const uint16_t *sh2, float *out)
{
    if (k3o_check_cfg(c) || H <= 0 || T < 0 || !(eps > 0.0) ||
        (latent_norm != 0 && latent_norm != 1) ||
        (T > 0 && (!h || !idx || !w || !Wd || !Wu || !out || (latent_norm && !gain))) ||
        (c->n_shared > 0 && T > 0 && (!sh1 || !sh3 || !sh2)))
        return K3O_EINVAL;
    const int d = c->d, f = c->f, k = c->top_k, SI = c->n_shared * c->f;
    int err = check_routing(c, T, idx, experts);
    if (err)
        return err;
    const int wide = f > SI ? f : SI;
    const int dh = d > H ? d : H;
#pragma omp parallel if (T > 1)
    {
        double *hd = malloc(sizeof(double) * (size_t)H);
        double *z = malloc(sizeof(double) * (size_t)d);
        double *a = malloc(sizeof(double) * (size_t)d);
        double *o = malloc(sizeof(double) * (size_t)H);
        double *y = malloc(sizeof(double) * (size_t)dh);
        double *g = malloc(sizeof(double) * (size_t)wide);
        double *u = malloc(sizeof(double) * (size_t)wide);
        double *act = malloc(sizeof(double) * (size_t)wide);
        if (!hd || !z || !a || !o || !y || !g || !u || !act) {
#pragma omp atomic write
            err = K3O_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int t = 0; t < T; t++) {
                for (int i = 0; i < H; i++)
                    hd[i] = (double)k3o_bf16(h[(size_t)t * H + i]);
                /* 2. down into the expert latent */
                k3o_bf16_matvec(z, hd, Wd, H, d);
                /* 3. the chosen experts, accumulated in the latent */
                for (int i = 0; i < d; i++)
                    a[i] = 0.0;
                for (int j = 0; j < k; j++) {
                    const k3o_expert *q = experts + idx[(size_t)t * k + j];
                    const double wt = (double)w[(size_t)t * k + j];
                    expert_ffn(c, q, z, g, u, act, y);
                    for (int i = 0; i < d; i++)
                        a[i] += wt * y[i];
                }
                /* 4. RMSNorm of the aggregate */
                if (latent_norm) {
                    double ss = 0.0;
                    for (int i = 0; i < d; i++)
                        ss += a[i] * a[i];
                    const double r = 1.0 / sqrt(ss / d + eps);
                    for (int i = 0; i < d; i++)
                        a[i] = a[i] * r * (double)gain[i];
                }
                /* 5. back up to full width */
                k3o_bf16_matvec(o, a, Wu, d, H);
                /* 6. shared experts on the original h, unweighted */
                if (SI > 0) {
                    k3o_bf16_matvec(g, hd, sh1, H, SI);
                    k3o_bf16_matvec(u, hd, sh3, H, SI);
                    for (int i = 0; i < SI; i++)
                        act[i] = k3o_situ(g[i], u[i], c->situ_b1, c->situ_b2);
                    k3o_bf16_matvec(y, act, sh2, SI, H);
                    for (int i = 0; i < H; i++)
                        o[i] += y[i];
                }
                for (int i = 0; i < H; i++)
                    out[(size_t)t * H + i] = (float)o[i];
            }
        }
        free(hd); free(z); free(a); free(o); free(y); free(g); free(u); free(act);
    }
    return err;
}

/* Route then forward: the whole layer for T tokens. */
int k3o_moe(const k3o_cfg *c, int T, const uint16_t *x, const uint16_t *Wr,
            const float *bias, const k3o_expert *experts, const uint16_t *sh_w1,
            const uint16_t *sh_w3, const uint16_t *sh_w2, int32_t *idx, float *w,
            float *out)
{
    int rc = k3o_route(c, T, x, Wr, bias, idx, w, NULL, NULL, NULL);
    if (rc)
        return rc;
    return k3o_forward(c, T, x, idx, w, experts, sh_w1, sh_w3, sh_w2, out, NULL);
}

int k3o_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
