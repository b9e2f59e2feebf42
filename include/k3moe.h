/*
 * k3moe.h -- C ABI of the routed-expert layer of a Kimi-K3-style latent MoE,
 * GPU library (libk3moe.so) for GB300 / sm_103a.
 *
 * What the layer computes (kimi-k3-in-c README, Part II, section 9 "Picking 16
 * experts of 896", with the MXFP4 format of section 4): for each token x (the
 * expert latent, width d, bf16)
 *   1. score every routed expert e: sc[e] = sigmoid(x . Wr[e]) in float;
 *      ch[e] = sc[e] + bias[e] steers selection only;
 *   2. take the top_k experts by ch, ties to the lower index; their weights
 *      are the unbiased sc, renormalised to sum 1 when renorm and the sum is
 *      positive, then multiplied by routed_scale;
 *   3. run each chosen expert's gated FFN straight from packed MXFP4 weights:
 *      y = W2 . SiTU(W1 x, W3 x), SiTU(g, u) = b1 tanh(g/b1) sigmoid(g) *
 *      b2 tanh(u/b2) (the sigmoid reads the uncapped gate);
 *   4. add the n_shared dense bf16 experts (same form) with weight one;
 *   5. out = sum_j weight_j * y_j + sum_s y_s, float.
 *
 * Conventions for every call:
 *   - Every array pointer is DEVICE memory owned by the caller.  The library
 *     allocates and frees nothing on these calls; scratch comes from the
 *     caller's workspace (see k3moe_workspace_bytes).
 *   - bf16 arrays are passed as uint16_t bit patterns; all arrays are dense,
 *     row-major, with the shapes stated at each argument.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  A host-side validation error returns before any
 *     launch, so nothing is half-written.
 *   - Device-side anomalies (an expert index outside [0, E), offsets or a
 *     permutation that do not describe the routing, an MXFP4 scale byte of
 *     255) are never skipped silently: they set bits of the device status
 *     word in the workspace, read with k3moe_device_status.  The kernels
 *     bounds-check every index they derive from such inputs before using it.
 *   - The library waits on nothing it cannot bound: no kernel spins.
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *k3moe_stream;

/* Layer configuration.  Every field is required; k3moe_validate_config
 * rejects an unset (zero) or out-of-range field instead of defaulting it
 * (kimi-k3-in-c README, Part II, section 2 "The config reader that refuses to
 * guess").  The K3 values are d=3584, f=3072, n_experts=896, top_k=16,
 * n_shared=2, group=32, situ_b1=4.0, situ_b2=25.0, renorm=1,
 * routed_scale=1.0 (same section's K3Cfg struct). */
typedef struct k3moe_config {
    int32_t d;            /* expert latent width; multiple of 128, <= 8192 */
    int32_t f;            /* expert FFN width; multiple of 128, <= 8192 */
    int32_t n_experts;    /* routed experts E, 1..1024 */
    int32_t top_k;        /* experts per token k, 1..16 and <= E */
    int32_t n_shared;     /* dense shared experts S, 0..8 */
    int32_t group;        /* MXFP4 block size; must be 32 */
    float situ_b1;        /* SiTU gate cap, finite and > 0 */
    float situ_b2;        /* SiTU linear cap, finite and > 0 */
    int32_t renorm;       /* 0 or 1 */
    float routed_scale;   /* finite */
} k3moe_config;

typedef enum k3moe_status {
    K3MOE_OK = 0,
    K3MOE_EINVAL = 1,      /* a config field or argument is invalid */
    K3MOE_ESHAPE = 2,      /* T or a size outside what the call supports */
    K3MOE_EALIGN = 3,      /* a pointer lacks the alignment the call needs */
    K3MOE_EWORKSPACE = 4,  /* workspace NULL, misaligned or too small */
    K3MOE_ECUDA = 5,       /* a CUDA runtime call failed (launch or copy) */
    K3MOE_EDEVICE = 6,     /* the device status word reports an error */
    K3MOE_ETIMEOUT = 7     /* a bounded device-side wait gave up */
} k3moe_status;

/* Bits of the device status word. */
#define K3MOE_DEV_BAD_INDEX   0x1  /* routing index outside [0, E) */
#define K3MOE_DEV_BAD_OFFSETS 0x2  /* offsets/perm inconsistent with idx */
#define K3MOE_DEV_NAN_SCALE   0x4  /* warning: an E8M0 scale byte of 255 (read as 0) */
#define K3MOE_DEV_TIMEOUT     0x8  /* a bounded wait gave up */
/* Debug builds only (the library compiled with -DK3MOE_DEBUG, libk3moe_debug.so): an
 * index was outside its buffer where a kernel was about to use it; the access was
 * skipped or clamped.  Release builds keep the same guards but do not record them. */
#define K3MOE_DEV_BOUNDS      0x10
#define K3MOE_DEV_ERROR_MASK  (K3MOE_DEV_BAD_INDEX | K3MOE_DEV_BAD_OFFSETS | K3MOE_DEV_TIMEOUT | \
                               K3MOE_DEV_BOUNDS)

/* Human-readable name of a status code (static string). */
const char *k3moe_strerror(k3moe_status s);

/* K3MOE_OK when every field of *cfg is in range, else K3MOE_EINVAL or
 * K3MOE_ESHAPE.  Pure host function. */
k3moe_status k3moe_validate_config(const k3moe_config *cfg);

/* Bytes of the packed routed-expert table for cfg->n_experts experts: per expert
 * 3 * f * d * 17/32 bytes of codes and scales (half a byte per weight plus one
 * scale byte per 32: 17,547,264 bytes at the K3 shape, kimi-k3-in-c README,
 * Part II, "The problem: a model that does not fit") in the tiles the mat-vecs and
 * the f16 GEMM read, a 1024-byte summary of the largest scale of every 128-row
 * block and a flag for scale bytes 0 and 255 in the expert, and the same codes and
 * scales a second time (another 3 * f * d * 17/32 bytes) in the layouts the
 * block-scaled prefill GEMM's tensor-map loads take: the codes row-major as the
 * checkpoint has them, the scales in 512-byte blocks of 128 rows x 4 groups.  At
 * the K3 shape 896 experts take 31.4 GB.  0 for an invalid config. */
size_t k3moe_packed_bytes(const k3moe_config *cfg);

/* Workspace bytes that k3moe_route and k3moe_forward need for any
 * 0 <= T <= T_max.  The workspace is one caller-owned device buffer,
 * 256-byte aligned, shared by both calls; its first 256 bytes hold the
 * device status word, and the block after them the counters the kernels
 * return to zero at the end of every call.  Zero-fill it once before first
 * use; the calls keep everything else consistent, so one workspace serves
 * calls of any T <= T_max in any order (calls on one stream). */
k3moe_status k3moe_workspace_bytes(const k3moe_config *cfg, int32_t T_max, size_t *bytes);

/* Relayout experts [expert_lo, expert_lo + n_in) from the checkpoint's MXFP4
 * layout into the library's packed table (a relayout of codes and scales,
 * not a quantiser: kimi-k3-in-c README, Part II, section 4).  Inputs, per
 * tensor with a leading expert axis of n_in:
 *   w1_packed, w3_packed [n_in][f][d/2]  (low nibble = even column)
 *   w1_scale,  w3_scale  [n_in][f][d/32] (E8M0 bytes)
 *   w2_packed            [n_in][d][f/2]
 *   w2_scale             [n_in][d][f/32]
 * The *_packed pointers must be 16-byte aligned.  `table` (table_bytes >=
 * k3moe_packed_bytes) must be 256-byte aligned.  Each expert is written twice:
 * into the tiles the streamed mat-vecs and the f16 GEMM read, and into the
 * block-scaled section (row-major codes, scales in 512-byte blocks) the default
 * prefill GEMMs read; both are complete once the call's work has run.  Scale
 * bytes of 255 raise K3MOE_DEV_NAN_SCALE in `ws` when ws is not NULL (ws as for
 * k3moe_route). */
k3moe_status k3moe_pack_mxfp4(const k3moe_config *cfg, int32_t expert_lo, int32_t n_in,
                              const uint8_t *w1_packed, const uint8_t *w1_scale,
                              const uint8_t *w3_packed, const uint8_t *w3_scale,
                              const uint8_t *w2_packed, const uint8_t *w2_scale,
                              void *table, size_t table_bytes, void *ws,
                              k3moe_stream stream);

/* Inverse of k3moe_pack_mxfp4: writes experts [expert_lo, expert_lo + n_out)
 * of `table` back in checkpoint layout (same shapes and alignment rules). */
k3moe_status k3moe_unpack_mxfp4(const k3moe_config *cfg, int32_t expert_lo, int32_t n_out,
                                const void *table, size_t table_bytes,
                                uint8_t *w1_packed, uint8_t *w1_scale,
                                uint8_t *w3_packed, uint8_t *w3_scale,
                                uint8_t *w2_packed, uint8_t *w2_scale,
                                k3moe_stream stream);

/* Router (kimi-k3-in-c README, Part II, section 9, the k3_router listing):
 * logit = x . Wr^T, the exact sum of the bf16 products rounded once to float
 * (what the listing's double accumulation gives), sc = 1/(1+expf(-logit)) and
 * ch = sc + bias in float, top_k by ch with ties to the lower index, weights
 * from sc (renormalised when renorm and their float sum is > 0, summed in
 * rank order, then times routed_scale).  For many tokens the logits are first
 * approximated on the tensor cores and only the experts that can still be
 * chosen are scored exactly; the result is the same selection.  Then the
 * token -> expert map:
 *   x        [T][d] bf16         w_router [E][d] bf16     bias [E] f32 or NULL
 *   idx      [T][k] int32  out: chosen experts, ch descending, ties index ascending
 *   weight   [T][k] f32    out: routing weights in the same order
 *   offsets  [E+1] int32   out: exclusive prefix sum of per-expert slot counts
 *   perm     [T*k] int32   out: flat slot ids t*k+j grouped by expert, ascending
 *                               within each expert (a stable counting sort)
 * T may be 0 (offsets all zero).  ws per k3moe_workspace_bytes(T_max >= T). */
k3moe_status k3moe_route(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                         const uint16_t *w_router, const float *bias,
                         int32_t *idx, float *weight, int32_t *offsets, int32_t *perm,
                         void *ws, size_t ws_bytes, k3moe_stream stream);

/* The router's exact scores for every (token, expert), as k3moe_route's
 * selection uses them (kimi-k3-in-c README, Part II, section 9, the k3_router
 * listing):
 *   scores [T][E] f32  out: sc = 1/(1+expf(-logit)), logit = x . Wr^T rounded once
 *   choice [T][E] f32  out: ch = sc + bias (sc when bias is NULL)
 * k3moe_route's idx and weight are exactly the top-k of `choice` and the
 * renormalised `scores` of the chosen experts, for any T.  Every pair is
 * scored exactly here (no tensor-core shortcut), so at large T this call
 * costs far more than k3moe_route.  x, w_router 16-byte aligned; scores, choice, bias 4-byte
 * aligned.  T may be 0 (nothing written).  ws per k3moe_workspace_bytes(T_max
 * >= T); only its status word is used. */
k3moe_status k3moe_router_scores(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                                 const uint16_t *w_router, const float *bias, float *scores,
                                 float *choice, void *ws, size_t ws_bytes, k3moe_stream stream);

/* Expert part of the layer for given routing (as k3moe_route writes it, or
 * any routing with the same conventions), kimi-k3-in-c README, Part II,
 * section 9, the k3_moe listing's expert loop and shared-expert step:
 *   out[t] = sum_j weight[t][j] * W2_e . SiTU(W1_e x_t, W3_e x_t),  e = idx[t][j]
 *          + sum_s Sh2_s . SiTU(Sh1_s x_t, Sh3_s x_t)
 *   x            [T][d] bf16
 *   idx, weight  [T][k] int32 / f32;  offsets [E+1], perm [T*k] int32
 *   expert_table packed routed experts (k3moe_pack_mxfp4), table_bytes of it
 *   sh_w1, sh_w3 [S][f][d] bf16;  sh_w2 [S][d][f] bf16 (NULL when S == 0);
 *                16-byte aligned
 *   out          [T][d] f32, written (not accumulated)
 * Precision: every accumulation is fp32 and the MXFP4 weights enter exactly
 * (decoded, or as codes with their scales on the block-scaled MMAs).  On the
 * streamed mat-vecs (small T) x enters as f16 times a per-token power of two
 * (exact for every bf16 element within 2^31 of the token's largest), a routed
 * expert's SiTU output is rounded to f16 before its down projection, and a shared
 * expert's is kept as a bf16 hi + lo pair.  On the tensor-core path (large T) the
 * routed experts take x and their SiTU output as the two e4m3 planes of
 * k3moe_set_prefill_gemm's variant 2 (or f16, as above, with variant 1), and the
 * shared experts' SiTU output is rounded to bf16.
 * ws per k3moe_workspace_bytes(T_max >= T). */
k3moe_status k3moe_forward(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                           const int32_t *idx, const float *weight,
                           const int32_t *offsets, const int32_t *perm,
                           const void *expert_table, size_t table_bytes,
                           const uint16_t *sh_w1, const uint16_t *sh_w3, const uint16_t *sh_w2,
                           float *out, void *ws, size_t ws_bytes, k3moe_stream stream);

/* k3moe_forward without a caller workspace, for callers that cannot allocate
 * device memory: code running inside another framework's execution callback
 * (a plugin's enqueue, a serving hook) that receives only inputs and outputs,
 * and real-time or embedded callers with a fixed memory plan that forbids
 * cudaMalloc on the serving path (it can synchronise the device and can fail
 * under memory pressure).  The pages have no counterpart: their engine owns
 * all its buffers.
 *   Arguments, results and errors as k3moe_forward, minus ws/ws_bytes, plus
 *   status_out: optional device int32 that receives this call's device
 *   status word (K3MOE_DEV_* bits; 0 for T == 0); NULL to skip.
 * Scratch comes from a 32 MiB array inside the library (a file-scope
 * __device__ object): every GPU that loads the library holds it until the
 * process exits.  Calls whose k3moe_workspace_bytes(cfg, T) exceeds 32 MiB
 * return K3MOE_EWORKSPACE without launching (at the K3 shape, T <= 67 fits).
 * The first call on each device looks up the array's device address with
 * that device current; make it before any stream capture.  The address is
 * kept with the device's context and looked up again if that context is
 * replaced (a device reset).  All calls share the array and it keeps the
 * last call's contents (each call clears its status block first); calls
 * that overlap on the GPU race on it, so order them on one stream.
 * Allocates nothing: no cudaMalloc or cudaFree. */
k3moe_status k3moe_forward_noalloc(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                                   const int32_t *idx, const float *weight,
                                   const int32_t *offsets, const int32_t *perm,
                                   const void *expert_table, size_t table_bytes,
                                   const uint16_t *sh_w1, const uint16_t *sh_w3,
                                   const uint16_t *sh_w2, float *out, int32_t *status_out,
                                   k3moe_stream stream);

/* ---- The full-width block around the layer: the six steps of the k3_moe
 * listing (kimi-k3-in-c README, Part II, section 9 "Picking 16 experts of 896"),
 * for T full-width tokens h of width H:
 *   1. route on h (not on the latent): the rules of k3moe_route with a router
 *      [E][H] (cfg's d replaced by H);
 *   2. z = Wd . h, into the expert latent (width cfg->d);
 *   3. a = sum_j weight_j * W2_e . SiTU(W1_e z, W3_e z), the routed experts
 *      of k3moe_forward on z, WITHOUT its shared experts;
 *   4. when latent_norm: a_i = a_i * gain_i / sqrt(sum_i a_i^2 / d + rms_eps),
 *      the RMSNorm of the weighted sum (never of one expert);
 *   5. out = Wu . a, back to width H;
 *   6. out += Sh2 . SiTU(Sh1 h, Sh3 h): the cfg->n_shared shared experts on
 *      the ORIGINAL h, fused into one FFN of width SI = n_shared * f, added
 *      with weight one.
 * The K3 block has H = 7168, latent_norm = 1, rms_eps = 1e-5 (the K3Cfg
 * struct of section 2). */
typedef struct k3moe_full_dims {
    int32_t hidden;       /* H; multiple of 128, <= 8192 */
    int32_t latent_norm;  /* 1: RMSNorm the aggregate (step 4); 0: skip it */
    float rms_eps;        /* > 0 and finite */
} k3moe_full_dims;

/* Workspace bytes k3moe_full_forward needs for any 0 <= T <= T_max (the
 * layer's regions plus the block's z, a and shared intermediates, and the
 * projections' split-K partial sums: up to 1024 rows of the widest
 * projection, and as many again for the shared experts' projections, which
 * run beside the others). */
k3moe_status k3moe_full_workspace_bytes(const k3moe_config *cfg, const k3moe_full_dims *fd,
                                        int32_t T_max, size_t *bytes);

/* The full-width block, steps 1-6 above, asynchronous on `stream`:
 *   h          [T][H] bf16
 *   w_router   [E][H] bf16;  bias [E] f32 or NULL (selection only)
 *   w_down     [d][H] bf16 (Wd);  w_up [H][d] bf16 (Wu)
 *   expert_table, table_bytes: as k3moe_forward (packed at width d)
 *   norm_gain  [d] f32 (NULL allowed when latent_norm == 0)
 *   sh_w1, sh_w3 [SI][H] bf16;  sh_w2 [H][SI] bf16 (NULL when n_shared == 0)
 *   idx, weight, offsets, perm: out, the routing, as k3moe_route writes it
 *   out        [T][H] f32, written
 * Matrices and h 16-byte aligned; expert_table 256-byte aligned.  The dense
 * projections (Wd, Wu, the fused Sh1/Sh3 with SiTU, Sh2) run on the library's
 * tensor-core kernel with bf16 operands and fp32 accumulation, so z, the
 * normed a and the shared SiTU output are rounded to bf16 as their inputs.
 * Step 6 needs only h: it runs beside steps 1-4 on a stream the library keeps
 * per device, forked from `stream` where the call begins and joined back into
 * it before step 5, which adds Wu a to the shared experts' out (the same sum,
 * one rounding).  The side stream is created by the first call on a device
 * that is not made during a stream capture (until then step 6 runs on
 * `stream` after step 5); calls enqueue under one lock.  A call captured into
 * a graph takes the side stream into the capture until that capture ends, so
 * calls on one device that overlap a capture come from the capturing thread.
 * T may be 0 (offsets zeroed, nothing else written).  ws per
 * k3moe_full_workspace_bytes(T_max >= T); its status word as k3moe_route's. */
k3moe_status k3moe_full_forward(const k3moe_config *cfg, const k3moe_full_dims *fd, int32_t T,
                                const uint16_t *h, const uint16_t *w_router, const float *bias,
                                const uint16_t *w_down, const void *expert_table,
                                size_t table_bytes, const float *norm_gain,
                                const uint16_t *w_up, const uint16_t *sh_w1,
                                const uint16_t *sh_w3, const uint16_t *sh_w2, int32_t *idx,
                                float *weight, int32_t *offsets, int32_t *perm, float *out,
                                void *ws, size_t ws_bytes, k3moe_stream stream);

/* Synchronises `stream`, returns the device status word of `ws` in *code,
 * and clears it: the report of the README's rule that corruption is counted,
 * never silent (kimi-k3-in-c README, Part II, section 9, the k3_moe listing's
 * count of dropped experts).  Returns K3MOE_ETIMEOUT when the timeout bit is
 * set, else K3MOE_EDEVICE when another error bit is set, K3MOE_OK otherwise
 * (the NAN_SCALE warning alone is OK). */
k3moe_status k3moe_device_status(void *ws, k3moe_stream stream, int32_t *code);

/* Exercises the failure report of a bounded wait (kimi-k3-in-c README, Part II,
 * section 9: a fault is counted, never silent).  Every device-side wait of the
 * library is bounded; when one runs out, its kernel sets K3MOE_DEV_TIMEOUT in
 * the status word, drops its remaining work and returns, and the context stays
 * usable.  This call runs both of the library's wait routines (the streamed
 * mat-vecs' and the tensor-core kernels') on an mbarrier that nothing ever
 * arrives on, each giving up after `limit_cycles` SM clock cycles (1 .. 4e9),
 * so the timeout bit is set in `ws`'s status word; k3moe_device_status then
 * returns K3MOE_ETIMEOUT.  For tests of the failure path; asynchronous on
 * `stream`.  ws: a workspace as for k3moe_route (only its status word is used). */
k3moe_status k3moe_check_wait_timeout(void *ws, int64_t limit_cycles, k3moe_stream stream);

/* Exercises the index checks of a debug build (kimi-k3-in-c README, Part II,
 * section 9: a fault is counted, never silent).  Launches one thread that checks
 * `index` against [0, limit) the way the library's kernels check an index before
 * they use it; nothing is read or written through the index.  In a debug build
 * (k3moe_build_flags() & K3MOE_BUILD_DEBUG) an index outside the range sets
 * K3MOE_DEV_BOUNDS in `ws`'s status word, and k3moe_device_status then returns
 * K3MOE_EDEVICE; a release build records nothing.  Asynchronous on `stream`.
 * ws: a workspace as for k3moe_route (only its status word is used); K3MOE_ESHAPE
 * when limit < 1. */
k3moe_status k3moe_check_bounds(void *ws, int32_t index, int32_t limit, k3moe_stream stream);

/* How the library was built: K3MOE_BUILD_DEBUG when compiled with -DK3MOE_DEBUG
 * (the device-side index checks record K3MOE_DEV_BOUNDS). */
#define K3MOE_BUILD_DEBUG 0x1
int32_t k3moe_build_flags(void);

/* Which kernels run the routed experts' projections on the prefill path (the
 * tensor-core path k3moe_forward takes for T >= 32 and T*top_k >= 8*E).  Both compute
 * g = W1 x, u = W3 x and y = W2 h straight from the packed MXFP4 table (kimi-k3-in-c
 * README, Part II, section 4 "Reduction one: the experts already ship at half a
 * byte": an E2M1 code times the E8M0 scale of its 32-element group):
 *   1  f16 MMAs on weights dequantised into shared memory (code x 2^(scale - block
 *      maximum), exact in f16), the tokens as f16 x 2^-u;
 *   2  block-scaled MMAs (tcgen05 kind::mxf8f6f4): the E2M1 codes and their E8M0
 *      scales go to the tensor core as they are (from the table's row-major section,
 *      k3moe_packed_bytes), and the tensor core applies the scales per 32 elements;
 *      the tokens, and h for the down projection, as two e4m3 planes with their own
 *      E8M0 scales per 32 elements, hi = rn(v / 2^sa) and lo = rn((v / 2^sa - hi) /
 *      2^sl), so each 32-wide K step is two MMAs into the same fp32 accumulator.  The
 *      two planes hold a bf16 token exactly while its element lies within 2^12 of its
 *      32-block's largest magnitude (smaller ones: absolute error below 2^-21 of that
 *      magnitude); h (fp32) keeps about 8 significant bits, as bf16 would.  A scale
 *      byte of 255, which the format reads as zero, becomes 2^-127 (a contribution
 *      below 2^-120 of the group's codes);
 *   0  the library's default, which is 2.
 * The shared experts (bf16) run on the f16 kernels either way.
 * Process-wide; takes effect at the next k3moe_forward call (a captured graph keeps
 * the kernels it recorded).  K3MOE_EINVAL for another value.  The workspace
 * (k3moe_workspace_bytes) covers both. */
k3moe_status k3moe_set_prefill_gemm(int32_t variant);
int32_t k3moe_get_prefill_gemm(void);

/* Number of GPU kernels this library has launched in this process (all
 * calls, all devices); for launch accounting in benchmarks. */
int64_t k3moe_launch_count(void);

/* Per-kernel timing: when enabled, every launch is bracketed by CUDA events
 * on its stream.  k3moe_timing_read fills up to `cap` entries with kernel
 * names, launch counts and summed milliseconds (it synchronises the events)
 * and returns the number of kernel kinds; k3moe_timing_reset clears them.
 * Timing is off by default and costs nothing then. */
void k3moe_timing_enable(int32_t on);
int32_t k3moe_timing_read(const char **names, int64_t *launches, double *ms, int32_t cap);
void k3moe_timing_reset(void);

#ifdef __cplusplus
}
#endif

#endif /* K3MOE_H */
