// k3moe_internal.cuh -- shared definitions of the GPU library (not public).
//
// Packed routed-expert table (the layout k3moe_pack_mxfp4 writes):
//   expert e starts at e * expert_bytes; inside it
//   - gate/up block: for row block rb in [0, f/128), for K tile kt in [0, d/128):
//       [W1 tile (rb, kt)][W3 tile (rb, kt)]
//   - down block:    for row block rb in [0, d/128), for K tile kt in [0, f/128):
//       [W2 tile (rb, kt)]
//   A tile is 128 rows x 128 columns of one matrix, 8704 bytes:
//   - bytes [0, 8192): the E2M1 codes, in 32 blocks of 256 bytes, block (s, c) at
//     (s * 4 + c) * 256 for the 16-row strip s (rows 16s..16s+15) and the 32-column
//     group c.  Inside a block, lane L = 4g + t (g < 8, t < 4) owns 8 bytes at 8L:
//     bytes t, t+4, t+8, t+12 of row 16s+g's 16-byte group, then the same four bytes
//     of row 16s+g+8 (checkpoint byte order: low nibble = even column).  These are
//     exactly the A-operand pairs that lane holds in a 16x16 tensor-core fragment, for
//     the group's two 16-column steps, so one 8-byte load per lane feeds them.
//   - bytes [8192, 8704): E8M0 scale of (row r, group c) at 8192 + r * 4 + c.
//   Tiles are contiguous, so one bulk copy moves a tile, and a gate/up K step
//   (both matrices) is one 17408-byte copy.  Bytes per expert = 3*f*d*17/32.
// After the E expert payloads comes a trailer of kTrailerBytes per expert: for each
// matrix (W1, W3, W2) and each 128-row block, the largest E8M0 byte of the block other
// than 255, as a uint32 (the tensor-core path scales the block's weights by it); and in
// the trailer's last word a flag, nonzero when any scale byte of the expert is 0 (the
// subnormal 2^-127) or 255 (read as zero), the two bytes the fast conversion of the
// decode path does not give exactly.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#ifdef __CUDACC__
#include <cuda_fp16.h>
#endif

#include "../../include/k3moe.h"

namespace k3moe {

constexpr int kTileRows = 128;
constexpr int kTileK = 128;
constexpr int kGroup = 32;
constexpr int kTileNibbleBytes = kTileRows * kTileK / 2;            // 8192
constexpr int kTileScaleBytes = kTileRows * kTileK / kGroup;        // 512
constexpr int kTileBytes = kTileNibbleBytes + kTileScaleBytes;      // 8704
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kMaxShared = 8;
constexpr int kMaxWidth = 8192;
constexpr int kChunkTokens = 64;      // tokens per top-k block; its slots form one chunk
constexpr int kTrailerBytes = 1024;   // per-expert row-block scale summary (<= 3*64 uint32)

__host__ __device__ inline size_t gateup_block_bytes(int d, int f)
{
    return (size_t)(f / kTileRows) * (size_t)(d / kTileK) * 2 * kTileBytes;
}
__host__ __device__ inline size_t down_block_bytes(int d, int f)
{
    return (size_t)(d / kTileRows) * (size_t)(f / kTileK) * kTileBytes;
}
__host__ __device__ inline size_t expert_bytes(int d, int f)
{
    return gateup_block_bytes(d, f) + down_block_bytes(d, f);
}
// After the trailers, the block-scaled section: the codes again in the checkpoint's own
// row-major order, for tensor-map loads, and the scales in the tensor core's scale-block
// order (the prefill block-scaled GEMM reads only this section):
//   W1 [E*f][d/2], W3 [E*f][d/2], W2 [E*d][f/2] packed bytes (low nibble = even column);
//   gate/up scale blocks [E][f/128][d/128][2: W1, W3][512], down [E][d/128][f/128][512]:
//   a block covers rows 128 rb.. of one matrix and K columns 128 kc..; row r's 4 bytes
//   (its 4 groups of 32) at 16 (r % 32) + 4 (r / 32); byte 255 (read as zero) stored as 0.
__host__ __device__ inline size_t mx_w1_offset(int E, int d, int f)
{
    return (size_t)E * (expert_bytes(d, f) + kTrailerBytes);
}
__host__ __device__ inline size_t mx_w3_offset(int E, int d, int f)
{
    return mx_w1_offset(E, d, f) + (size_t)E * f * d / 2;
}
__host__ __device__ inline size_t mx_w2_offset(int E, int d, int f)
{
    return mx_w3_offset(E, d, f) + (size_t)E * f * d / 2;
}
__host__ __device__ inline size_t mx_sfgu_offset(int E, int d, int f)
{
    return mx_w2_offset(E, d, f) + (size_t)E * d * f / 2;
}
__host__ __device__ inline size_t mx_sfdn_offset(int E, int d, int f)
{
    return mx_sfgu_offset(E, d, f) + (size_t)E * (f / kTileRows) * (d / kTileK) * 1024;
}
// Whole table: E payloads, E trailers, the block-scaled section.
__host__ __device__ inline size_t packed_table_bytes(int E, int d, int f)
{
    return mx_sfdn_offset(E, d, f) + (size_t)E * (d / kTileRows) * (f / kTileK) * 512;
}
// Trailer word of (expert e, matrix m in {0: W1, 1: W3, 2: W2}, row block rb).
__host__ __device__ inline size_t trailer_offset(int E, int d, int f, int e, int m, int rb)
{
    const int nrb_f = f / kTileRows;
    const int idx = (m < 2) ? m * nrb_f + rb : 2 * nrb_f + rb;
    return (size_t)E * expert_bytes(d, f) + (size_t)e * kTrailerBytes + (size_t)idx * 4;
}

// Trailer word of expert e that flags scale bytes 0 and 255 anywhere in the expert.
__host__ __device__ inline size_t special_flag_offset(int E, int d, int f, int e)
{
    return (size_t)E * expert_bytes(d, f) + (size_t)e * kTrailerBytes + kTrailerBytes - 4;
}
static_assert(3 * (kMaxWidth / kTileRows) * 4 <= kTrailerBytes - 4,
              "the block maxima and the flag word share the trailer");

// Device status word and abort flag live in the first 256 bytes of the workspace.
// Words: 0 status (K3MOE_DEV_* bits); 1 abort (nonzero: the routing failed validation,
// later kernels skip work); 2, 3 the work counters of the two mat-vec kernels; 4 the
// top-k kernel's last-block counter; 5 the gate/up mat-vec's exit counter; 6 the flag the
// gate/up mat-vec raises once the routing is visible to it; 7 the down mat-vec's exit
// counter; 8 the flag the last gate/up block raises when all of h is published.  Counters
// and flags are back at zero after every call.
struct StatusBlock {
    int32_t status;
    int32_t abort;
    int32_t pad[62];
};


// Forward path: the tensor-core GEMMs once an expert sees on average at least 8 tokens
// (T*k >= 8*E) and T >= 32; the streamed mat-vecs otherwise.
inline bool use_gemm_path(const k3moe_config &c, int T)
{
    return T >= 32 && (long long)T * c.top_k >= 8LL * c.n_experts;
}

// Workspace regions (byte offsets), sized for one call's T.
// Counters that kernels keep at zero between calls live in one block at a fixed offset
// (right after the status block) in every layout, whatever T and the path: buffers of a
// call with another T must never overlap them.  Sized for the largest configuration.
constexpr size_t kCtrShared = (size_t)kMaxShared * (kMaxWidth / kTileRows);  // shared gate/up K-part arrivals
constexpr size_t kCtrReady = (size_t)kMaxExperts + kMaxShared;                // h rows ready, per unit
// dense split-K arrivals: 128-row blocks of the widest projection (N <= S f) x 4 token
// tiles (K is split only while T <= 512) x 4 quadrants; a second set for the projections
// the full-width block runs on its side stream
constexpr size_t kCtrDense = (size_t)kMaxShared * (kMaxWidth / 128) * 4 * 4;
constexpr size_t kCtrOffset = 256;
constexpr size_t kCtrBytes = ((kCtrShared + kCtrReady + 2 * kCtrDense) * 4 + 255) & ~(size_t)255;

struct WsLayout {
    size_t status;
    size_t shctr;                // fixed counter block: shared gate/up arrival counters [S][f/128] int32
    size_t ready;                // fixed counter block: h-ready counters per unit [E + S] int32
    size_t dctr;                 // fixed counter block: dense split-K arrival counters
    size_t dctr2;                // fixed counter block: the same for the full block's side stream
    size_t sc, ch;               // router scores [T][E] f32 (tensor-core router: sc holds its logits)
    size_t wnorm;                // router row norms |Wr[e]| [E] f32 (tensor-core router)
    size_t chunk_counts;         // [n_chunks][E] int32
    size_t chunk_base;           // [n_chunks][E] int32
    size_t local_rank;           // [T*k] int32
    size_t active;               // [E + 1] int32: active expert ids, then the count
    size_t inv;                  // [T*k] int32: slot -> position in perm
    size_t tok_scale;            // [2][T] f32: activation multiplier 2^-u, output factor 2^u
    size_t hp;                   // decode: SiTU output as hi and lo planes [2][rows][f] 16-bit
    size_t xs;                   // decode: activations x * 2^-u per token [T][d] f16
    size_t ys;                   // decode: y rows [rows_y][d] f32 (a shared expert's K parts: one row each)
    size_t gush;                 // decode: shared gate/up partials [parts][S][T][2][f] f32
    size_t xg;                   // prefill: routed activations in perm order [T*k][d] f16
    size_t units;                // prefill: unit list [E+S][4], item prefixes, unit count
    size_t sfa;                  // prefill, block-scaled GEMMs: token tiles' e8m0 scales [tiles][d/128][2][512]
    size_t sfa_dn;               //   and h's, the down projection's tokens [tiles][f/128][2][512]
    size_t total;
    bool gemm;                   // which forward path this T takes
    int n_chunks;
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// K parts of a shared-expert gate/up work item on the decode path.  A bf16 shared item
// carries four times the bytes of a packed routed one; with a single token (16 routed
// experts) it would set the kernel's length, so its K range is split into up to 4 parts
// (the parts' sums are added in order).  From two tokens on the routed items outnumber
// the blocks enough to absorb whole shared items, and the split costs more than it
// balances (measured at T = 2..16).  ktiles: 128-column tiles of K.  The down
// projection is not split: measured at T = 1, its split items cost more than the
// balance gains (gemv_down 43.8 us whole, 43.9 in two parts, 47.4 in four).
constexpr int kMaxSharedParts = 4;
__host__ __device__ inline int shared_kparts(int ktiles, int T)
{
    if (T > 1) return 1;
    return ktiles % 4 == 0 ? 4 : (ktiles % 2 == 0 ? 2 : 1);
}

// Token tiles of 128 rows over the prefill units (shared experts' first, as the GEMMs
// number them): each unit needs ceil(rows / 128), so at most S ceil(T / 128) for the
// shared units plus T k / 128 + (one partial tile per active expert) for the routed ones.
inline size_t gemm_token_tiles(const k3moe_config &c, int T)
{
    const size_t slots = (size_t)T * c.top_k;
    return (size_t)c.n_shared * (((size_t)T + 127) / 128) + (slots + 127) / 128 +
           std::min(slots, (size_t)c.n_experts);
}

// Which kernel the prefill gate/up projection of the routed experts uses (a process-wide
// choice, k3moe_set_prefill_gemm): 1 the f16 GEMM on dequantised weights, 2 the
// block-scaled GEMM on the packed MXFP4 weights, 0 the default (prefill_gemm_choice).
int prefill_gemm_setting();
bool prefill_gemm_block_scaled(const k3moe_config &c, int T);

inline WsLayout ws_layout(const k3moe_config &c, int T)
{
    WsLayout L{};
    const size_t E = (size_t)c.n_experts, k = (size_t)c.top_k, S = (size_t)c.n_shared;
    const size_t slots = (size_t)T * k;
    L.n_chunks = (T + kChunkTokens - 1) / kChunkTokens;
    L.gemm = use_gemm_path(c, T);
    size_t o = 0;
    L.status = o; o += 256;
    L.shctr = kCtrOffset;
    L.ready = L.shctr + kCtrShared * 4;
    L.dctr = L.ready + kCtrReady * 4;
    L.dctr2 = L.dctr + kCtrDense * 4;
    o = kCtrOffset + kCtrBytes;
    L.sc = o; o = align256(o + (size_t)T * E * 4);
    L.ch = o; o = align256(o + (size_t)T * E * 4);
    L.wnorm = o; o = align256(o + E * 4);
    L.chunk_counts = o; o = align256(o + (size_t)L.n_chunks * E * 4);
    L.chunk_base = o; o = align256(o + (size_t)L.n_chunks * E * 4);
    L.local_rank = o; o = align256(o + slots * 4);
    L.active = o; o = align256(o + (E + 1) * 4);
    L.inv = o; o = align256(o + slots * 4);
    L.tok_scale = o; o = align256(o + (size_t)T * 2 * 4);
    const size_t rows = slots + S * (size_t)T;
    L.hp = o; o = align256(o + rows * (size_t)c.f * 2 * (L.gemm ? 1 : 2));
    L.xs = o; o = align256(o + (L.gemm ? 0 : (size_t)T * c.d * 2));
    const size_t pgu = (size_t)shared_kparts(c.d / kTileK, T), pdn = 1;
    L.ys = o; o = align256(o + (L.gemm ? 0 : (slots + S * pdn * (size_t)T) * (size_t)c.d * 4));
    L.gush = o; o = align256(o + (L.gemm || pgu == 1 ? 0 : pgu * S * (size_t)T * 2 * c.f * 4));
    L.xg = o; o = align256(o + (L.gemm ? slots * (size_t)c.d * 2 : 0));
    L.units = o; o = align256(o + (L.gemm ? (4 * (E + S) + 2 * (E + S + 1) + 1) * 4 : 0));
    L.sfa = o; o = align256(o + (L.gemm ? gemm_token_tiles(c, T) * (size_t)(c.d / 128) * 1024 : 0));
    L.sfa_dn = o; o = align256(o + (L.gemm ? gemm_token_tiles(c, T) * (size_t)(c.f / 128) * 1024 : 0));
    L.total = o;
    return L;
}

// Dense projections (k3moe_dense.cu): y[t][n] = epilogue(sum_k x[t][k] W[n][k]).
enum DenseEpi { kDenseBf16 = 0, kDenseF32 = 1, kDenseAddF32 = 2, kDenseSitu = 3 };
constexpr int kDenseTargetItems = 456;   // work items that fill the GPU (3 per SM of 152)
constexpr int kDensePartRows = 1024;     // at most this many partial rows (K parts x tokens)
constexpr int kDenseMaxParts = 16;
constexpr int kDenseRowsMaxT = 4;        // up to this many tokens: the row-streaming kernel
struct DensePlan {
    int bn, n_tt, n_rb, P, nkp, kb, mats, stage_bytes, nstg;
};
DensePlan dense_plan(int T, int N, int K, int epi);
bool dense_applies(int N, int K);
// part: kDensePartRows x N x mats floats when the plan splits K; ctr: n_rb * n_tt * 4 int32
// counters at zero (left at zero).
cudaError_t launch_dense(int epi, int T, int N, int K, const uint16_t *x, const uint16_t *w,
                         const uint16_t *w3, void *y, float b1, float b2, float *part, int32_t *ctr,
                         int32_t *status, cudaStream_t s, const char *name);

// Full-width block (k3moe_full_forward).  Its router call reads the full-width token (a
// config whose d is the hidden width H), its expert call runs the layer on the latent
// with no shared experts (they run on the full width here).  The two calls run one after
// the other and share the layer's regions; the block's own buffers follow them.
struct FullLayout {
    k3moe_config cr, cl;         // router config (d = H), latent config (n_shared = 0)
    WsLayout route, latent;
    size_t z;                    // [T][d] bf16: the token projected into the latent
    size_t acc;                  // [T][d] f32: the experts' weighted sum
    size_t y;                    // [T][d] bf16: the normed sum, the up projection's input
    size_t act;                  // [T][S*f] bf16: the shared experts' SiTU
    size_t part;                 // dense projections' K-part partial sums
    size_t ctr;                  // their arrival counters: the fixed counter block's
    size_t part2, ctr2;          // the same for the shared experts' projections (side stream)
    size_t total;
};

inline FullLayout full_layout(const k3moe_config &c, int hidden, int T)
{
    FullLayout F{};
    F.cr = c;
    F.cr.d = hidden;
    F.cl = c;
    F.cl.n_shared = 0;
    F.route = ws_layout(F.cr, T);
    F.latent = ws_layout(F.cl, T);
    const size_t td = (size_t)T * c.d, ts = (size_t)T * c.n_shared * c.f;
    const size_t SI = (size_t)c.n_shared * c.f;
    // widest partial row over the four projections: Wd (d), Wu and Sh2 (H), Sh1 + Sh3 (2 SI)
    const size_t wmax = std::max(std::max((size_t)c.d, (size_t)hidden), 2 * SI);
    size_t o = align256(F.route.total > F.latent.total ? F.route.total : F.latent.total);
    F.z = o; o = align256(o + td * 2);
    F.acc = o; o = align256(o + td * 4);
    F.y = o; o = align256(o + td * 2);
    F.act = o; o = align256(o + ts * 2);
    F.part = o; o = align256(o + (T > 0 ? (size_t)kDensePartRows * wmax * 4 : 0));
    // the shared experts' projections run beside the others (side stream): partials of
    // their own, Sh1 + Sh3 (2 SI) or Sh2 (H) wide
    const size_t wsh = SI > 0 ? std::max((size_t)hidden, 2 * SI) : 0;
    F.part2 = o; o = align256(o + (T > 0 ? (size_t)kDensePartRows * wsh * 4 : 0));
    F.ctr = F.route.dctr;        // at the same fixed offset in the route and latent layouts
    F.ctr2 = F.route.dctr2;
    F.total = o;
    return F;
}

// ----------------------------------------------------------------------------------- programmatic dependent launch
// Every kernel of the route and forward chains starts with pdl_wait(): it waits until the
// previous kernel in the stream has completed and its writes are visible, before touching
// memory, so the kernel may be launched early (launch_pdl) and its launch latency overlaps
// the previous kernel.  pdl_trigger() then lets the next kernel launch the same way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ----------------------------------------------------------------------------------- launch bookkeeping
// Every launch goes through these so launches can be counted and, on request, timed.
void timing_begin(const char *name, cudaStream_t s);
void timing_end(const char *name, cudaStream_t s);
void count_launch();

// Host launchers implemented in the kernel files.
cudaError_t launch_pack(const k3moe_config &c, int expert_lo, int n, const uint8_t *w1p,
                        const uint8_t *w1s, const uint8_t *w3p, const uint8_t *w3s,
                        const uint8_t *w2p, const uint8_t *w2s, uint8_t *table,
                        int32_t *status, cudaStream_t s);
cudaError_t launch_unpack(const k3moe_config &c, int expert_lo, int n, const uint8_t *table,
                          uint8_t *w1p, uint8_t *w1s, uint8_t *w3p, uint8_t *w3s,
                          uint8_t *w2p, uint8_t *w2s, cudaStream_t s);
cudaError_t launch_route(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                         const float *bias, int32_t *idx, float *weight, int32_t *offsets,
                         int32_t *perm, uint8_t *ws, const WsLayout &L, cudaStream_t s);
// Exact router scores sc, ch [T][E] f32 for every expert (the per-token kernel, any T).
cudaError_t launch_router_scores(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                                 const float *bias, float *sc, float *ch, int32_t *status, cudaStream_t s);
// Approximate router logits on the tensor cores (many tokens): logit [T][E] f32, within a
// small multiple of 2^-22 |x_t| |Wr[e]| of the exact logit; the top-k re-scores exactly
// every expert the approximation cannot rule out.
constexpr int kRouterTcMinTokens = 32;
bool router_tc_applies(const k3moe_config &c, int T);
cudaError_t launch_router_logits_tc(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                                    float *logit, int32_t *status, cudaStream_t s);
cudaError_t launch_forward_gemm(const k3moe_config &c, int T, const uint16_t *x, const int32_t *idx,
                                const float *weight, const int32_t *offsets, const int32_t *perm,
                                const uint8_t *table, const uint16_t *sh_w1, const uint16_t *sh_w3,
                                const uint16_t *sh_w2, float *out, uint8_t *ws, const WsLayout &L,
                                cudaStream_t s);
// The full-width block (k3moe_full_forward), all six steps on stream s.
cudaError_t launch_full(const k3moe_config &c, int hidden, int latent_norm, float rms_eps, int T,
                        const uint16_t *h, const uint16_t *wr, const float *bias, const uint16_t *wd,
                        const uint8_t *table, const float *gain, const uint16_t *wu,
                        const uint16_t *sh1, const uint16_t *sh3, const uint16_t *sh2, int32_t *idx,
                        float *weight, int32_t *offsets, int32_t *perm, float *out, uint8_t *ws,
                        const FullLayout &F, cudaStream_t s);
// One bounded wait of each kind (the mat-vec kernels', the tensor-core kernels') on an
// mbarrier nothing arrives on, giving up after `limit` cycles: sets K3MOE_DEV_TIMEOUT.
cudaError_t launch_wait_check_gemv(int32_t *status, long long limit, cudaStream_t s);
cudaError_t launch_wait_check_tc(int32_t *status, long long limit, cudaStream_t s);
// Largest T any call accepts.
constexpr int32_t kMaxT = 1 << 20;
// Either path, as the layout chose it.
inline cudaError_t launch_forward(const k3moe_config &c, int T, const uint16_t *x, const int32_t *idx,
                                  const float *weight, const int32_t *offsets, const int32_t *perm,
                                  const uint8_t *table, const uint16_t *sh_w1, const uint16_t *sh_w3,
                                  const uint16_t *sh_w2, float *out, uint8_t *ws, const WsLayout &L,
                                  cudaStream_t s, bool x_is_input = true);
// x_is_input: x is complete when the call is made (not written by the kernel launched just
// before with programmatic dependent launch), so the mat-vec path may read it before its
// wait for the routing.
cudaError_t launch_forward_gemv(const k3moe_config &c, int T, const uint16_t *x,
                                const int32_t *idx, const float *weight, const int32_t *offsets,
                                const int32_t *perm, const uint8_t *table, const uint16_t *sh_w1,
                                const uint16_t *sh_w3, const uint16_t *sh_w2, float *out,
                                uint8_t *ws, const WsLayout &L, cudaStream_t s, bool x_is_input = true);

inline cudaError_t launch_forward(const k3moe_config &c, int T, const uint16_t *x, const int32_t *idx,
                                  const float *weight, const int32_t *offsets, const int32_t *perm,
                                  const uint8_t *table, const uint16_t *sh_w1, const uint16_t *sh_w3,
                                  const uint16_t *sh_w2, float *out, uint8_t *ws, const WsLayout &L,
                                  cudaStream_t s, bool x_is_input)
{
    return L.gemm ? launch_forward_gemm(c, T, x, idx, weight, offsets, perm, table, sh_w1, sh_w3, sh_w2,
                                        out, ws, L, s)
                  : launch_forward_gemv(c, T, x, idx, weight, offsets, perm, table, sh_w1, sh_w3, sh_w2,
                                        out, ws, L, s, x_is_input);
}

// ----------------------------------------------------------------------------------- device helpers
#ifdef __CUDACC__

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// E8M0 byte -> 2^(b-127) as float; byte 0 is the subnormal 2^-127; 255 -> 0.
__device__ __forceinline__ float e8m0_to_f32(uint32_t b)
{
    b &= 255u;
    if (b == 255u) return 0.0f;
    if (b == 0u) return __uint_as_float(0x00400000u);
    return __uint_as_float(b << 23);
}

// Two E2M1 codes (one packed byte: low nibble = even element) -> two exact floats.
// The conversion instruction decodes the pair to f16x2; E2M1 values are exact in f16.
__device__ __forceinline__ float2 e2m1x2_to_f32x2(uint32_t byte_in_low_bits)
{
    uint32_t h;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(h) : "r"(byte_in_low_bits));
    __half2 hh = *reinterpret_cast<__half2 *>(&h);
    return __half22float2(hh);
}

__device__ __forceinline__ void set_status(int32_t *status, int32_t bits)
{
    atomicOr(status, bits);
}

// Index checks at the point of use.
//   dguard(status, ok): a guard every build keeps (the caller skips or clamps the
//     access when ok is false); debug builds also record K3MOE_DEV_BOUNDS.
//   dcheck(status, ok): a check only debug builds make (the caller skips the access
//     when it fails); release builds compile it to true.
__device__ __forceinline__ bool dguard(int32_t *status, bool ok)
{
#ifdef K3MOE_DEBUG
    if (!ok) set_status(status, K3MOE_DEV_BOUNDS);
#else
    (void)status;
#endif
    return ok;
}
__device__ __forceinline__ bool dcheck(int32_t *status, bool ok)
{
#ifdef K3MOE_DEBUG
    if (!ok) set_status(status, K3MOE_DEV_BOUNDS);
    return ok;
#else
    (void)status;
    (void)ok;
    return true;
#endif
}
// A clamp of an index into [lo, hi] that debug builds record when it changes the value.
__device__ __forceinline__ int dclamp(int32_t *status, int v, int lo, int hi)
{
    const int c = min(max(v, lo), hi);
    dguard(status, c == v);
    return c;
}

#endif

}  // namespace k3moe
