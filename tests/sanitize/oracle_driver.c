/*
 * oracle_driver.c -- drives the CPU oracle and the seeded input generator through every
 * entry point, their edge cases and their error paths, for a build under
 * AddressSanitizer and UndefinedBehaviorSanitizer (tests/test_sanitizers.py).  Test
 * infrastructure: it links oracle/k3moe_oracle.c and k3moe_inputs/k3moe_gen.c and checks
 * return codes and that outputs are finite; the sanitizers check every memory access
 * and every operation with undefined behaviour on the way.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t d, f, n_experts, top_k, n_shared, group;
    float situ_b1, situ_b2;
    int32_t renorm;
    float routed_scale;
} k3o_cfg;
typedef struct {
    const uint8_t *w1_packed, *w1_scale, *w3_packed, *w3_scale, *w2_packed, *w2_scale;
} k3o_expert;

int k3o_check_cfg(const k3o_cfg *c);
double k3o_e2m1(int code);
double k3o_e8m0(int byte);
float k3o_bf16(uint16_t b);
double k3o_mxfp4_weight(const uint8_t *packed, const uint8_t *scales, int cols, int group, int row, int col);
void k3o_mxfp4_matvec(double *y, const double *x, const uint8_t *packed, const uint8_t *scales, int in,
                      int rows, int group);
void k3o_bf16_matvec(double *y, const double *x, const uint16_t *W, int in, int rows);
double k3o_situ(double g, double u, double b1, double b2);
int k3o_route(const k3o_cfg *c, int T, const uint16_t *x, const uint16_t *Wr, const float *bias, int32_t *idx,
              float *w, float *sc_out, float *ch_out, float *gap);
int k3o_select(const k3o_cfg *c, int T, const float *sc, const float *ch, int32_t *idx, float *w, float *gap);
int k3o_perm(int T, int E, int k, const int32_t *idx, int32_t *offsets, int32_t *perm);
int k3o_forward(const k3o_cfg *c, int T, const uint16_t *x, const int32_t *idx, const float *w,
                const k3o_expert *experts, const uint16_t *sh_w1, const uint16_t *sh_w3, const uint16_t *sh_w2,
                float *out, float *out_shared);
int k3o_forward_full(const k3o_cfg *c, int H, int latent_norm, double eps, int T, const uint16_t *h,
                     const int32_t *idx, const float *w, const uint16_t *Wd, const k3o_expert *experts,
                     const float *gain, const uint16_t *Wu, const uint16_t *sh1, const uint16_t *sh3,
                     const uint16_t *sh2, float *out);
int k3o_moe(const k3o_cfg *c, int T, const uint16_t *x, const uint16_t *Wr, const float *bias,
            const k3o_expert *experts, const uint16_t *sh_w1, const uint16_t *sh_w3, const uint16_t *sh_w2,
            int32_t *idx, float *w, float *out);
int k3o_num_threads(void);

void k3g_bf16_normal(uint16_t *out, size_t n, uint64_t seed, uint64_t stream, uint64_t offset, double sigma);
void k3g_uniform_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream, uint64_t offset, int lo, int hi);
void k3g_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream, uint64_t offset);
void k3g_permutation(int32_t *perm, int32_t n, uint64_t seed, uint64_t stream);
void k3g_zipf_bias(float *bias, int32_t n, uint64_t seed, uint64_t stream, double s, double scale);
double k3g_normal(uint64_t seed, uint64_t stream, uint64_t i);
double k3g_log(double u);

static int failures = 0;
#define EXPECT(cond, what)                                              \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "FAILED: %s (line %d)\n", what, __LINE__);  \
            failures++;                                                 \
        }                                                               \
    } while (0)

static void *xalloc(size_t n)
{
    void *p = calloc(n ? n : 1, 1);
    if (!p) {
        fprintf(stderr, "out of memory\n");
        exit(2);
    }
    return p;
}

static int all_finite(const float *v, size_t n)
{
    for (size_t i = 0; i < n; i++)
        if (!isfinite(v[i]))
            return 0;
    return 1;
}

/* Experts with random nibbles and scales in [lo, hi], a few scale bytes 255. */
static k3o_expert *make_experts(const k3o_cfg *c, uint64_t seed)
{
    const int E = c->n_experts, d = c->d, f = c->f, g = c->group;
    k3o_expert *ex = xalloc(sizeof(k3o_expert) * (size_t)E);
    for (int e = 0; e < E; e++) {
        uint8_t *w1 = xalloc((size_t)f * d / 2), *s1 = xalloc((size_t)f * d / g);
        uint8_t *w3 = xalloc((size_t)f * d / 2), *s3 = xalloc((size_t)f * d / g);
        uint8_t *w2 = xalloc((size_t)d * f / 2), *s2 = xalloc((size_t)d * f / g);
        k3g_bytes(w1, (size_t)f * d / 2, seed, 100 + 6 * e, 0);
        k3g_bytes(w3, (size_t)f * d / 2, seed, 101 + 6 * e, 0);
        k3g_bytes(w2, (size_t)d * f / 2, seed, 102 + 6 * e, 0);
        k3g_uniform_bytes(s1, (size_t)f * d / g, seed, 103 + 6 * e, 0, 118, 126);
        k3g_uniform_bytes(s3, (size_t)f * d / g, seed, 104 + 6 * e, 0, 118, 126);
        k3g_uniform_bytes(s2, (size_t)d * f / g, seed, 105 + 6 * e, 0, 118, 126);
        s1[e % (f * d / g)] = 255;
        s2[0] = 0;
        ex[e] = (k3o_expert){w1, s1, w3, s3, w2, s2};
    }
    return ex;
}

static void free_experts(k3o_expert *ex, int E)
{
    for (int e = 0; e < E; e++) {
        free((void *)ex[e].w1_packed); free((void *)ex[e].w1_scale);
        free((void *)ex[e].w3_packed); free((void *)ex[e].w3_scale);
        free((void *)ex[e].w2_packed); free((void *)ex[e].w2_scale);
    }
    free(ex);
}

/* One whole configuration: route, select, perm, forward, moe, forward_full. */
static void run_case(const k3o_cfg *c, int T, int H, uint64_t seed)
{
    const int d = c->d, f = c->f, E = c->n_experts, k = c->top_k, S = c->n_shared, SI = S * f;
    uint16_t *x = xalloc(sizeof(uint16_t) * (size_t)T * d), *Wr = xalloc(sizeof(uint16_t) * (size_t)E * d);
    uint16_t *sh1 = xalloc(sizeof(uint16_t) * (size_t)SI * d), *sh3 = xalloc(sizeof(uint16_t) * (size_t)SI * d);
    uint16_t *sh2 = xalloc(sizeof(uint16_t) * (size_t)d * SI);
    float *bias = xalloc(sizeof(float) * (size_t)E);
    k3g_bf16_normal(x, (size_t)T * d, seed, 1, 0, 1.0);
    k3g_bf16_normal(Wr, (size_t)E * d, seed, 2, 0, 0.02);
    k3g_bf16_normal(sh1, (size_t)SI * d, seed, 3, 0, 0.05);
    k3g_bf16_normal(sh3, (size_t)SI * d, seed, 4, 0, 0.05);
    k3g_bf16_normal(sh2, (size_t)d * SI, seed, 5, 0, 0.05);
    k3g_zipf_bias(bias, E, seed, 6, 1.1, 0.01);
    k3o_expert *ex = make_experts(c, seed);

    int32_t *idx = xalloc(sizeof(int32_t) * (size_t)T * k), *idx2 = xalloc(sizeof(int32_t) * (size_t)T * k);
    float *w = xalloc(sizeof(float) * (size_t)T * k), *w2 = xalloc(sizeof(float) * (size_t)T * k);
    float *sc = xalloc(sizeof(float) * (size_t)T * E), *ch = xalloc(sizeof(float) * (size_t)T * E);
    float *gap = xalloc(sizeof(float) * (size_t)T);
    EXPECT(k3o_route(c, T, x, Wr, bias, idx, w, sc, ch, gap) == 0, "route");
    EXPECT(k3o_select(c, T, sc, ch, idx2, w2, NULL) == 0, "select");
    EXPECT(T == 0 || memcmp(idx, idx2, sizeof(int32_t) * (size_t)T * k) == 0, "select repeats route");
    EXPECT(k3o_route(c, T, x, Wr, NULL, idx2, w2, NULL, NULL, NULL) == 0, "route without bias");

    int32_t *offsets = xalloc(sizeof(int32_t) * (size_t)(E + 1)), *perm = xalloc(sizeof(int32_t) * (size_t)T * k);
    EXPECT(k3o_perm(T, E, k, idx, offsets, perm) == 0, "perm");
    EXPECT(offsets[E] == T * k, "offsets total");

    float *out = xalloc(sizeof(float) * (size_t)T * d), *outs = xalloc(sizeof(float) * (size_t)T * d);
    float *out2 = xalloc(sizeof(float) * (size_t)T * d);
    EXPECT(k3o_forward(c, T, x, idx, w, ex, sh1, sh3, sh2, out, outs) == 0, "forward");
    EXPECT(all_finite(out, (size_t)T * d) && all_finite(outs, (size_t)T * d), "forward finite");
    EXPECT(k3o_moe(c, T, x, Wr, bias, ex, sh1, sh3, sh2, idx2, w2, out2) == 0, "moe");
    EXPECT(T == 0 || memcmp(out, out2, sizeof(float) * (size_t)T * d) == 0, "moe repeats route + forward");

    /* the full-width block around the layer */
    uint16_t *h = xalloc(sizeof(uint16_t) * (size_t)T * H), *Wd = xalloc(sizeof(uint16_t) * (size_t)d * H);
    uint16_t *Wu = xalloc(sizeof(uint16_t) * (size_t)H * d);
    uint16_t *f1 = xalloc(sizeof(uint16_t) * (size_t)SI * H), *f3 = xalloc(sizeof(uint16_t) * (size_t)SI * H);
    uint16_t *f2 = xalloc(sizeof(uint16_t) * (size_t)H * SI);
    float *gain = xalloc(sizeof(float) * (size_t)d), *fo = xalloc(sizeof(float) * (size_t)T * H);
    for (int i = 0; i < d; i++)
        gain[i] = 1.0f + 0.01f * (float)(i % 7);
    k3g_bf16_normal(h, (size_t)T * H, seed, 7, 0, 1.0);
    k3g_bf16_normal(Wd, (size_t)d * H, seed, 8, 0, 0.05);
    k3g_bf16_normal(Wu, (size_t)H * d, seed, 9, 0, 0.05);
    k3g_bf16_normal(f1, (size_t)SI * H, seed, 10, 0, 0.05);
    k3g_bf16_normal(f3, (size_t)SI * H, seed, 11, 0, 0.05);
    k3g_bf16_normal(f2, (size_t)H * SI, seed, 12, 0, 0.05);
    for (int ln = 0; ln < 2; ln++) {
        EXPECT(k3o_forward_full(c, H, ln, 1e-5, T, h, idx, w, Wd, ex, gain, Wu, f1, f3, f2, fo) == 0,
               "forward_full");
        EXPECT(all_finite(fo, (size_t)T * H), "forward_full finite");
    }
    /* error paths: a routed index out of range, a bad norm flag, a bad epsilon */
    if (T > 0) {
        const int32_t keep = idx[0];
        idx[0] = E;
        EXPECT(k3o_forward(c, T, x, idx, w, ex, sh1, sh3, sh2, out, NULL) != 0, "forward rejects idx >= E");
        idx[0] = -1;
        EXPECT(k3o_forward_full(c, H, 1, 1e-5, T, h, idx, w, Wd, ex, gain, Wu, f1, f3, f2, fo) != 0,
               "forward_full rejects idx < 0");
        idx[0] = keep;
        EXPECT(k3o_forward_full(c, H, 2, 1e-5, T, h, idx, w, Wd, ex, gain, Wu, f1, f3, f2, fo) != 0,
               "forward_full rejects a bad norm flag");
        EXPECT(k3o_forward_full(c, H, 1, 0.0, T, h, idx, w, Wd, ex, gain, Wu, f1, f3, f2, fo) != 0,
               "forward_full rejects eps = 0");
    }

    free(h); free(Wd); free(Wu); free(f1); free(f3); free(f2); free(gain); free(fo);
    free(out); free(outs); free(out2); free(offsets); free(perm);
    free(idx); free(idx2); free(w); free(w2); free(sc); free(ch); free(gap);
    free(x); free(Wr); free(sh1); free(sh3); free(sh2); free(bias);
    free_experts(ex, E);
}

int main(void)
{
    /* scalar pieces over their whole input ranges */
    for (int code = 0; code < 16; code++)
        EXPECT(isfinite(k3o_e2m1(code)), "e2m1");
    for (int b = 0; b < 256; b++)
        EXPECT(k3o_e8m0(b) >= 0.0, "e8m0");
    for (uint32_t b = 0; b < 65536; b += 97)
        (void)k3o_bf16((uint16_t)b);
    EXPECT(isfinite(k3o_situ(1e30, -1e30, 4.0, 25.0)) && isfinite(k3o_situ(-800.0, 3.0, 4.0, 25.0)), "situ");
    for (int i = 0; i < 1000; i++)
        EXPECT(isfinite(k3g_normal(7, 3, (uint64_t)i)), "normal");
    EXPECT(fabs(k3g_log(1.0)) < 1e-15 && isfinite(k3g_log(1e-300)), "log");
    {
        int32_t p[37];
        k3g_permutation(p, 37, 5, 1);
        int seen[37] = {0};
        for (int i = 0; i < 37; i++)
            if (p[i] >= 0 && p[i] < 37)
                seen[p[i]]++;
        for (int i = 0; i < 37; i++)
            EXPECT(seen[i] == 1, "permutation");
    }
    /* mat-vecs on a ragged row count */
    {
        const int in = 96, rows = 13, g = 32;
        uint8_t *pk = xalloc((size_t)rows * in / 2), *sc = xalloc((size_t)rows * in / g);
        uint16_t *W = xalloc(sizeof(uint16_t) * (size_t)rows * in);
        double *xv = xalloc(sizeof(double) * in), *y = xalloc(sizeof(double) * rows);
        k3g_bytes(pk, (size_t)rows * in / 2, 1, 1, 0);
        k3g_uniform_bytes(sc, (size_t)rows * in / g, 1, 2, 0, 100, 140);
        k3g_bf16_normal(W, (size_t)rows * in, 1, 3, 0, 1.0);
        for (int i = 0; i < in; i++)
            xv[i] = 0.5 - (double)(i % 5);
        k3o_mxfp4_matvec(y, xv, pk, sc, in, rows, g);
        k3o_bf16_matvec(y, xv, W, in, rows);
        EXPECT(isfinite(k3o_mxfp4_weight(pk, sc, in, g, rows - 1, in - 1)), "mxfp4 weight");
        free(pk); free(sc); free(W); free(xv); free(y);
    }
    /* configurations: a general one, several shared experts, k = E, E = k = 1, no shared
     * expert, no renormalisation, and T = 0 */
    const k3o_cfg base = {64, 64, 8, 2, 1, 32, 4.0f, 25.0f, 1, 1.0f};
    run_case(&base, 5, 96, 11);
    k3o_cfg c = base;
    c.n_shared = 3;
    run_case(&c, 3, 64, 12);
    c = base;
    c.top_k = c.n_experts;
    run_case(&c, 4, 32, 13);
    c = base;
    c.n_experts = 1;
    c.top_k = 1;
    run_case(&c, 2, 64, 14);
    c = base;
    c.n_shared = 0;
    c.renorm = 0;
    c.routed_scale = 2.5f;
    run_case(&c, 3, 64, 15);
    run_case(&base, 0, 64, 16);
    /* invalid configurations are refused */
    k3o_cfg bad = base;
    bad.top_k = 9;
    EXPECT(k3o_check_cfg(&bad) != 0, "top_k > E");
    bad = base;
    bad.group = 0;
    EXPECT(k3o_check_cfg(&bad) != 0, "group 0");
    bad = base;
    bad.d = 48;
    EXPECT(k3o_check_cfg(&bad) != 0, "d not a multiple of the group");
    EXPECT(k3o_check_cfg(NULL) != 0, "null config");
    EXPECT(k3o_perm(-1, 8, 2, NULL, NULL, NULL) != 0, "perm T < 0");
    EXPECT(k3o_num_threads() >= 1, "threads");
    if (failures) {
        fprintf(stderr, "%d failures\n", failures);
        return 1;
    }
    printf("oracle driver: all checks passed\n");
    return 0;
}
