// k3moe_route.cu -- router and token -> expert map (kimi-k3-in-c README,
// Part II, section 9 "Picking 16 experts of 896").
//
// Kernels, in launch order:
//   router_scores   logits = x . Wr^T (fp32 accumulation of exact bf16 products),
//                   sc = 1/(1+expf(-logit)), ch = sc + bias, both float, to the workspace;
//   router_topk     one warp per token: top_k by ch via repeated warp arg-max (strict
//                   comparison, ties to the lower index), weights from sc renormalised in
//                   rank order; then, per block of 64 tokens (one "chunk" of slots), the
//                   per-expert slot counts and each slot's stable rank inside the chunk
//                   (warp match + ballot prefix).  A single-chunk launch finishes the
//                   map in place: scan, offsets, perm;
//   perm_scan       (several chunks) per-expert exclusive scan over chunks, then over
//                   experts -> offsets and every chunk's base;
//   perm_scatter    (several chunks) perm[base + rank] = slot.
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kScoreWarps = 4;      // experts per router_scores block (one per warp)
constexpr int kScoreTok = 8;        // tokens per register tile in router_scores

// -------------------------------------------------------------------------------- scores
// One warp per expert row of Wr; lanes stride along d in 16-byte chunks (8 bf16), so each
// warp-wide load is 512 contiguous bytes.  Tokens go in register tiles of kScoreTok.
__global__ void __launch_bounds__(kScoreWarps * 32) router_scores_kernel(
    int T, int d, int E, const uint16_t *__restrict__ x, const uint16_t *__restrict__ wr,
    const float *__restrict__ bias, float *__restrict__ sc_out, float *__restrict__ ch_out)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kScoreWarps + warp;
    if (e >= E) return;
    const uint4 *wrow = reinterpret_cast<const uint4 *>(wr + (size_t)e * d);
    const int nchunk = d / 8;
    const float b = bias ? bias[e] : 0.0f;
    for (int t0 = 0; t0 < T; t0 += kScoreTok) {
        float acc[kScoreTok];
#pragma unroll
        for (int i = 0; i < kScoreTok; i++) acc[i] = 0.0f;
        const int nt = min(kScoreTok, T - t0);
        for (int c = lane; c < nchunk; c += 32) {
            const uint4 w = __ldg(wrow + c);
            float wf[8];
            const uint32_t wu[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int q = 0; q < 4; q++) {
                wf[2 * q] = __uint_as_float(wu[q] << 16);
                wf[2 * q + 1] = __uint_as_float(wu[q] & 0xFFFF0000u);
            }
#pragma unroll
            for (int i = 0; i < kScoreTok; i++) {
                if (i < nt) {
                    const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(
                                               x + (size_t)(t0 + i) * d) + c);
                    const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
                    float a = acc[i];
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        a = fmaf(__uint_as_float(xu[q] << 16), wf[2 * q], a);
                        a = fmaf(__uint_as_float(xu[q] & 0xFFFF0000u), wf[2 * q + 1], a);
                    }
                    acc[i] = a;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kScoreTok; i++) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[i] = v;
        }
        if (lane < nt) {
            float logit = acc[0];
#pragma unroll
            for (int i = 1; i < kScoreTok; i++)
                if (lane == i) logit = acc[i];
            const float s = 1.0f / (1.0f + expf(-logit));
            sc_out[(size_t)(t0 + lane) * E + e] = s;
            ch_out[(size_t)(t0 + lane) * E + e] = s + b;
        }
    }
}

// -------------------------------------------------------------------------------- top-k
// (value, index) order: larger value first; equal values -> lower index first.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

struct TopkArgs {
    int T, E, k, renorm;
    float routed_scale;
    const float *sc, *ch;
    int32_t *idx;
    float *weight;
    int32_t *offsets, *perm;
    int32_t *chunk_counts, *local_rank;
    int32_t *status;
};

// blockDim = 1024 (32 warps); block b owns tokens [64b, 64b+64): its slots are chunk b.
__global__ void __launch_bounds__(1024) router_topk_kernel(TopkArgs a)
{
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t slot_e[kChunkTokens * kMaxTopK];
    __shared__ int32_t scan_tmp[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t_begin = blockIdx.x * kChunkTokens;
    const int t_end = min(a.T, t_begin + kChunkTokens);
    const int E = a.E, k = a.k;

    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;

    // ---- selection: warp per token
    for (int t = t_begin + warp; t < t_end; t += 32) {
        const float *chr = a.ch + (size_t)t * E;
        float v[kMaxExperts / 32];
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; i++) {
            const int e = lane + 32 * i;
            // -0.0 and +0.0 compare equal in the repeated maximum; canonicalise to +0.0.
            v[i] = (e < E) ? (chr[e] + 0.0f) : -INFINITY;
        }
        uint32_t taken = 0;
        int my_idx = -1;
        for (int j = 0; j < k; j++) {
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < kMaxExperts / 32; i++) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (bi == 0x7fffffff || beats(v[i], e, bv, bi))) {
                    bv = v[i];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (oi != 0x7fffffff && (bi == 0x7fffffff || beats(ov, oi, bv, bi))) {
                    bv = ov;
                    bi = oi;
                }
            }
            // bi is now the winner on every lane; its owner marks it taken.
            if (bi >= 0 && bi < E && (bi & 31) == lane) taken |= 1u << (bi >> 5);
            if (lane == j) my_idx = bi;
        }
        // weights: unbiased sc of the chosen experts, renormalised in rank order
        float w = 0.0f;
        if (lane < k) {
            if (my_idx < 0 || my_idx >= E) {      // cannot happen with k <= E; stay in bounds
                set_status(a.status, K3MOE_DEV_BAD_INDEX);
                my_idx = 0;
            }
            w = a.sc[(size_t)t * E + my_idx];
        }
        float s = 0.0f;
        for (int j = 0; j < k; j++) s += __shfl_sync(0xffffffffu, w, j);
        if (lane < k) {
            if (a.renorm && s > 0.0f) w = w / s;
            w = w * a.routed_scale;
            a.idx[(size_t)t * k + lane] = my_idx;
            a.weight[(size_t)t * k + lane] = w;
            slot_e[(t - t_begin) * k + lane] = my_idx;
        }
    }
    __syncthreads();

    // ---- chunk-local counts and stable ranks (slot order = t*k + j), warp by warp
    const int nslots = (t_end - t_begin) * k;
    int my_rank = 0, my_e = -1;
    for (int w = 0; w < 32; w++) {
        if (warp == w) {
            const int s = w * 32 + lane;
            const bool valid = s < nslots;
            const int e = valid ? slot_e[s] : -1 - lane;   // invalid lanes never match
            const uint32_t m = __match_any_sync(0xffffffffu, e);
            if (valid) {
                const uint32_t lower = m & ((1u << lane) - 1u);
                my_rank = cnt[e] + __popc(lower);
                my_e = e;
            }
            __syncwarp();
            if (valid && (__ffs(m) - 1) == lane) cnt[e] += __popc(m);   // group leader
        }
        __syncthreads();
    }

    if (gridDim.x == 1) {
        // single chunk: offsets = exclusive scan of cnt, then scatter
        int run = 0;
        for (int base = 0; base < E; base += blockDim.x) {
            const int e = base + threadIdx.x;
            const int v = (e < E) ? cnt[e] : 0;
            // block-wide exclusive scan of v
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (lane == 31) scan_tmp[warp] = incl;
            __syncthreads();
            if (warp == 0) {
                int wv = scan_tmp[lane];
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int n = __shfl_up_sync(0xffffffffu, wv, o);
                    if (lane >= o) wv += n;
                }
                scan_tmp[lane] = wv;          // inclusive over warps
            }
            __syncthreads();
            const int excl = run + incl - v + (warp > 0 ? scan_tmp[warp - 1] : 0);
            if (e < E) {
                a.offsets[e] = excl;
                cnt[e] = excl;                // becomes the segment base
            }
            run += scan_tmp[31];
            __syncthreads();
        }
        if (threadIdx.x == 0) a.offsets[E] = a.T * k;
        __syncthreads();
        if (my_e >= 0) a.perm[cnt[my_e] + my_rank] = t_begin * k + threadIdx.x;
    } else {
        if (my_e >= 0) a.local_rank[(size_t)t_begin * k + threadIdx.x] = my_rank;
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            a.chunk_counts[(size_t)blockIdx.x * E + e] = cnt[e];
    }
}

// -------------------------------------------------------------------------------- multi-chunk map
// One thread per expert runs over the chunks (exclusive scan down a column), then a
// block-wide scan over experts turns totals into offsets, which are added back.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int n_chunks, int E, int total_slots,
                                                         const int32_t *__restrict__ chunk_counts,
                                                         int32_t *__restrict__ chunk_base,
                                                         int32_t *__restrict__ offsets)
{
    __shared__ int32_t scan_tmp[32];
    const int e = threadIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < n_chunks; c++) {
            const int v = chunk_counts[(size_t)c * E + e];
            chunk_base[(size_t)c * E + e] = run;
            run += v;
        }
    }
    const int v = (e < E) ? run : 0;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scan_tmp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int wv = scan_tmp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, wv, o);
            if (lane >= o) wv += n;
        }
        scan_tmp[lane] = wv;
    }
    __syncthreads();
    const int excl = incl - v + (warp > 0 ? scan_tmp[warp - 1] : 0);
    if (e < E) {
        offsets[e] = excl;
        for (int c = 0; c < n_chunks; c++) chunk_base[(size_t)c * E + e] += excl;
    }
    if (threadIdx.x == 0) offsets[E] = total_slots;
}

__global__ void __launch_bounds__(256) perm_scatter_kernel(int total_slots, int k, int E,
                                                           const int32_t *__restrict__ idx,
                                                           const int32_t *__restrict__ chunk_base,
                                                           const int32_t *__restrict__ local_rank,
                                                           int32_t *__restrict__ perm)
{
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= total_slots) return;
    const int e = idx[s];
    if (e < 0 || e >= E) return;
    const int chunk = s / (kChunkTokens * k);
    const int p = chunk_base[(size_t)chunk * E + e] + local_rank[s];
    if (p >= 0 && p < total_slots) perm[p] = s;
}

}  // namespace

cudaError_t launch_route(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                         const float *bias, int32_t *idx, float *weight, int32_t *offsets,
                         int32_t *perm, uint8_t *ws, const WsLayout &L, cudaStream_t s)
{
    const int E = c.n_experts, k = c.top_k;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    if (T == 0) {
        timing_begin("route_zero", s);
        cudaError_t err = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), s);
        timing_end("route_zero", s);
        return err;
    }
    float *sc = reinterpret_cast<float *>(ws + L.sc);
    float *ch = reinterpret_cast<float *>(ws + L.ch);
    timing_begin("router_scores", s);
    router_scores_kernel<<<(E + kScoreWarps - 1) / kScoreWarps, kScoreWarps * 32, 0, s>>>(
        T, c.d, E, x, wr, bias, sc, ch);
    count_launch();
    timing_end("router_scores", s);

    TopkArgs a{T, E, k, c.renorm, c.routed_scale, sc, ch, idx, weight, offsets, perm,
               reinterpret_cast<int32_t *>(ws + L.chunk_counts),
               reinterpret_cast<int32_t *>(ws + L.local_rank), status};
    timing_begin("router_topk", s);
    router_topk_kernel<<<L.n_chunks, 1024, 0, s>>>(a);
    count_launch();
    timing_end("router_topk", s);
    if (L.n_chunks > 1) {
        int32_t *base = reinterpret_cast<int32_t *>(ws + L.chunk_base);
        timing_begin("perm_scan", s);
        perm_scan_kernel<<<1, 1024, 0, s>>>(L.n_chunks, E, T * k, a.chunk_counts, base, offsets);
        count_launch();
        timing_end("perm_scan", s);
        timing_begin("perm_scatter", s);
        perm_scatter_kernel<<<(T * k + 255) / 256, 256, 0, s>>>(T * k, k, E, idx, base,
                                                                 a.local_rank, perm);
        count_launch();
        timing_end("perm_scatter", s);
    }
    return cudaGetLastError();
}

}  // namespace k3moe
