// k3moe_route.cu -- router and token -> expert map (kimi-k3-in-c README, Part II,
// section 9 "Picking 16 experts of 896").
//
// Kernels, in launch order:
//   router_scores  logits = x . Wr^T (fp32 accumulation of exact bf16 products),
//                  sc = 1/(1+expf(-logit)), ch = sc + bias, both float, to the workspace.
//                  A block owns 4 experts (one per warp, its Wr row held in registers)
//                  and walks the tokens 8 at a time through shared memory;
//   router_topk    one block per token: warp-level bitonic sorts and merges of the E keys
//                  (ch, then the lower index first) pick the top k in rank order; the
//                  weights are the chosen sc renormalised by their float sum in rank
//                  order, times routed_scale.  With at most 64 tokens the last block to
//                  finish (the only one, for one token) also builds the map;
//   perm_count     (more tokens) per chunk of 64 tokens: per-expert slot counts and each
//                  slot's stable rank inside the chunk (warp match + popc, warp by warp);
//   perm_scan      per-expert exclusive scan over chunks, then over experts -> offsets;
//   perm_scatter   perm[base + rank] = slot.
// The map is a stable counting sort: offsets = exclusive prefix sum of the per-expert
// counts, and inside an expert's segment the flat slot ids t*k+j ascend.
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kScoreWarps = 4;       // experts per block (one per warp)
constexpr int kScoreTok = 8;         // tokens staged per round
constexpr int kScoreChunks = 16;     // 16-byte Wr chunks per lane held at once (4096 columns)

// -------------------------------------------------------------------------------- scores
__global__ void __launch_bounds__(kScoreWarps * 32) router_scores_kernel(
    int T, int d, int E, const uint16_t *__restrict__ x, const uint16_t *__restrict__ wr,
    const float *__restrict__ bias, float *__restrict__ sc_out, float *__restrict__ ch_out)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint8_t xs_raw[];        // kScoreTok x d bf16
    uint4 *xs = reinterpret_cast<uint4 *>(xs_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kScoreWarps + warp;
    const int nchunk = d / 8;                                  // 16-byte chunks per row
    const uint4 *wrow = reinterpret_cast<const uint4 *>(wr + (size_t)min(e, E - 1) * d);
    const float b = (bias && e < E) ? bias[e] : 0.0f;
    // the first 4096 columns of the row stay in registers across the token rounds (the
    // whole row for d <= 4096); their loads are in flight with the first x tile's
    uint4 w0[kScoreChunks];
#pragma unroll
    for (int j = 0; j < kScoreChunks; j++) {
        const int c = lane + 32 * j;
        w0[j] = c < nchunk ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
    }
    for (int t0 = 0; t0 < T; t0 += kScoreTok) {
        const int nt = min(kScoreTok, T - t0);
        __syncthreads();
        for (int q = threadIdx.x; q < nt * nchunk; q += blockDim.x) {
            const int i = q / nchunk, c = q % nchunk;
            xs[i * nchunk + c] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + i) * d) + c);
        }
        __syncthreads();
        float acc[kScoreTok];
#pragma unroll
        for (int i = 0; i < kScoreTok; i++) acc[i] = 0.0f;
        for (int c0 = 0; c0 < nchunk; c0 += 32 * kScoreChunks) {
            uint4 w[kScoreChunks];
#pragma unroll
            for (int j = 0; j < kScoreChunks; j++) {
                const int c = c0 + lane + 32 * j;
                w[j] = c0 == 0 ? w0[j] : (c < nchunk ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0));
            }
#pragma unroll
            for (int i = 0; i < kScoreTok; i++) {
                if (i >= nt) break;
                float a = acc[i];
#pragma unroll
                for (int j = 0; j < kScoreChunks; j++) {
                    const int c = c0 + lane + 32 * j;
                    if (c < nchunk) {
                        const uint4 xv = xs[i * nchunk + c];
                        const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
                        const uint32_t wu[4] = {w[j].x, w[j].y, w[j].z, w[j].w};
#pragma unroll
                        for (int q = 0; q < 4; q++) {
                            a = fmaf(__uint_as_float(xu[q] << 16), __uint_as_float(wu[q] << 16), a);
                            a = fmaf(__uint_as_float(xu[q] & 0xFFFF0000u), __uint_as_float(wu[q] & 0xFFFF0000u), a);
                        }
                    }
                }
                acc[i] = a;
            }
        }
#pragma unroll
        for (int i = 0; i < kScoreTok; i++) {
            float v = acc[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[i] = v;
        }
        if (e < E && lane < nt) {
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

// -------------------------------------------------------------------------------- token -> expert map
struct MapArgs {
    int T, E, k;
    const int32_t *idx;
    int32_t *offsets, *perm;
    int32_t *chunk_counts, *local_rank;
    int32_t *status;
};

// One chunk of 64 tokens (k*64 <= 1024 slots) with 1024 threads: per-expert counts and
// stable ranks; when `single`, also the scan to offsets and the scatter to perm.
__device__ void map_chunk(const MapArgs &a, int chunk, bool single, int32_t *cnt, int32_t *slot_e,
                          int32_t *scan_tmp)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = a.E, k = a.k;
    const int t_begin = chunk * kChunkTokens, t_end = min(a.T, t_begin + kChunkTokens);
    const int nslots = (t_end - t_begin) * k;
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    if (threadIdx.x < nslots) {
        int e = a.idx[(size_t)t_begin * k + threadIdx.x];
        if (e < 0 || e >= E) {
            set_status(a.status, K3MOE_DEV_BAD_INDEX);
            e = 0;
        }
        slot_e[threadIdx.x] = e;
    }
    __syncthreads();
    int my_rank = 0, my_e = -1;
    for (int w = 0; w < 32; w++) {
        if (w * 32 >= nslots) break;
        if (warp == w) {
            const int s = w * 32 + lane;
            const bool valid = s < nslots;
            const int e = valid ? slot_e[s] : -1 - lane;   // invalid lanes never match
            const uint32_t m = __match_any_sync(0xffffffffu, e);
            if (valid) {
                my_rank = cnt[e] + __popc(m & ((1u << lane) - 1u));
                my_e = e;
            }
            __syncwarp();
            if (valid && (__ffs(m) - 1) == lane) cnt[e] += __popc(m);   // group leader
        }
        __syncthreads();
    }
    if (single) {
        int run = 0;
        for (int base = 0; base < E; base += blockDim.x) {
            const int e = base + threadIdx.x;
            const int v = (e < E) ? cnt[e] : 0;
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
            a.chunk_counts[(size_t)chunk * E + e] = cnt[e];
    }
}

// -------------------------------------------------------------------------------- top-k
// Orderable image of a float: larger float -> larger unsigned (after -0.0 -> +0.0).
__device__ __forceinline__ uint32_t orderable(float v)
{
    const uint32_t u = __float_as_uint(v + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkArgs {
    int T, E, k, renorm;
    float routed_scale;
    const float *sc, *ch;
    int32_t *idx;
    float *weight;
    int32_t *done;          // last-block counter (kept at zero between calls)
    MapArgs map;
};

// Keys of one warp, one per lane, sorted descending across the lanes (bitonic network
// on shuffles).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t key, int lane)
{
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
        const bool desc = (lane & size) == 0;
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const uint64_t other = __shfl_xor_sync(0xffffffffu, key, stride);
            const bool keep_max = desc == ((lane & stride) == 0);
            key = keep_max ? (key > other ? key : other) : (key < other ? key : other);
        }
    }
    return key;
}
// Lanes 0-15 hold a descending list, lanes 16-31 another one in ascending order: together
// a bitonic sequence, merged descending, so lanes 0-15 end with the 16 largest keys.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t key, int lane)
{
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, key, stride);
        const bool keep_max = (lane & stride) == 0;
        key = keep_max ? (key > other ? key : other) : (key < other ? key : other);
    }
    return key;
}

// blockDim = 1024; block t owns token t.  Key = (orderable(ch) << 32) | ~index, so a
// descending order sorts by ch and, among equal ch, by ascending index -- the order the
// repeated maximum with a strict comparison produces.  Every key is distinct, so the k
// largest keys are the selection.  Warp w sorts keys 32w..32w+31 and keeps its 16
// largest; pairs of lists are then merged warp by warp (16 of 32 kept) until one remains.
__global__ void __launch_bounds__(1024) router_topk_kernel(TopkArgs a)
{
    pdl_wait();
    pdl_trigger();
    __shared__ uint64_t lists[2][32][kMaxTopK];
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t slot_e[kChunkTokens * kMaxTopK];
    __shared__ int32_t scan_tmp[32];
    __shared__ int last;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    const int t = blockIdx.x, E = a.E, k = a.k;
    const int nl0 = (E + 31) >> 5;                 // lists after the first level
    uint64_t key = 0;
    if (warp < nl0) {
        if (i < E) key = ((uint64_t)orderable(a.ch[(size_t)t * E + i]) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)i);
        key = warp_sort_desc(key, lane);
        if (lane < kMaxTopK) lists[0][warp][lane] = key;
    }
    int nl = nl0, cur = 0;
    while (nl > 1) {
        __syncthreads();
        const int half = (nl + 1) >> 1;
        if (warp < half) {
            const int la = 2 * warp, lb = 2 * warp + 1;
            uint64_t v;
            if (lane < 16) v = lists[cur][la][lane];
            else v = lb < nl ? lists[cur][lb][31 - lane] : 0;
            v = warp_merge_desc(v, lane);
            if (lane < kMaxTopK) lists[cur ^ 1][warp][lane] = v;
        }
        cur ^= 1;
        nl = half;
    }
    __syncthreads();
    if (warp == 0) key = lane < kMaxTopK ? lists[cur][0][lane] : 0;
    // lane r < k of warp 0 now holds the rank-r key
    if (i < 32) {
        int e = -1;
        float w = 0.0f;
        if (i < k) {
            e = (int)(0xFFFFFFFFu - (uint32_t)key);
            if (e < 0 || e >= E) {                 // cannot happen with k <= E; stay in bounds
                set_status(a.map.status, K3MOE_DEV_BAD_INDEX);
                e = 0;
            }
            w = a.sc[(size_t)t * E + e];
        }
        float s = 0.0f;
        for (int j = 0; j < k; j++) s += __shfl_sync(0xffffffffu, w, j);
        if (i < k) {
            if (a.renorm && s > 0.0f) w = w / s;
            w = w * a.routed_scale;
            a.idx[(size_t)t * k + i] = e;
            a.weight[(size_t)t * k + i] = w;
            slot_e[i] = e;
        }
    }
    if (a.done == nullptr) return;                 // the map is built by perm_count
    if (gridDim.x == 1) {                          // one token: its block builds the map
        __syncthreads();
        if (a.T == 1) {
            // its k experts are distinct, one slot each: offsets[e] counts the chosen
            // experts below e, and a slot's position in perm is the rank of its expert
            for (int ee = i; ee <= E; ee += blockDim.x) {
                int below = 0;
                for (int j = 0; j < k; j++) below += slot_e[j] < ee ? 1 : 0;
                a.map.offsets[ee] = below;
            }
            if (i < k) {
                int rank = 0;
                for (int j = 0; j < k; j++) rank += slot_e[j] < slot_e[i] ? 1 : 0;
                a.map.perm[rank] = i;
            }
            return;
        }
        map_chunk(a.map, 0, true, cnt, slot_e, scan_tmp);
        return;
    }
    // the last block to finish builds the map of all (at most 64) tokens
    __threadfence();
    __syncthreads();
    if (i == 0) last = (atomicAdd(a.done, 1) == (int)gridDim.x - 1);
    __syncthreads();
    if (!last) return;
    __threadfence();
    map_chunk(a.map, 0, true, cnt, slot_e, scan_tmp);
    if (i == 0) *a.done = 0;
}

__global__ void __launch_bounds__(1024) perm_count_kernel(MapArgs a)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t slot_e[kChunkTokens * kMaxTopK];
    __shared__ int32_t scan_tmp[32];
    map_chunk(a, blockIdx.x, gridDim.x == 1, cnt, slot_e, scan_tmp);
}

// One thread per expert runs over the chunks (exclusive scan down a column), then a
// block-wide scan over experts turns totals into offsets, which are added back.
__global__ void __launch_bounds__(1024) perm_scan_kernel(int n_chunks, int E, int total_slots,
                                                         const int32_t *__restrict__ chunk_counts,
                                                         int32_t *__restrict__ chunk_base,
                                                         int32_t *__restrict__ offsets)
{
    pdl_wait();
    pdl_trigger();
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
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= total_slots) return;
    const int e = idx[s];
    if (e < 0 || e >= E) return;
    const int chunk = s / (kChunkTokens * k);
    const int p = chunk_base[(size_t)chunk * E + e] + local_rank[s];
    if (p >= 0 && p < total_slots) perm[p] = s;
}

}  // namespace

cudaError_t launch_router_scores(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                                 const float *bias, float *sc, float *ch, int32_t *status, cudaStream_t s)
{
    const int E = c.n_experts;
    if (router_tc_applies(c, T)) {
        timing_begin("router_scores_tc", s);
        cudaError_t err = launch_router_scores_tc(c, T, x, wr, bias, sc, ch, status, s);
        timing_end("router_scores_tc", s);
        if (err != cudaSuccess) return err;
    } else {
        static size_t smem_set = 0;
        const size_t smem = (size_t)kScoreTok * c.d * 2;
        if (smem > smem_set) {
            cudaFuncSetAttribute(router_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            smem_set = smem;
        }
        timing_begin("router_scores", s);
        cudaError_t err = launch_pdl(router_scores_kernel, dim3((E + kScoreWarps - 1) / kScoreWarps),
                                     dim3(kScoreWarps * 32), smem, s, T, c.d, E, x, wr, bias, sc, ch);
        count_launch();
        timing_end("router_scores", s);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

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
    cudaError_t err = launch_router_scores(c, T, x, wr, bias, sc, ch, status, s);
    if (err != cudaSuccess) return err;
    MapArgs m{T, E, k, idx, offsets, perm, reinterpret_cast<int32_t *>(ws + L.chunk_counts),
              reinterpret_cast<int32_t *>(ws + L.local_rank), status};
    // status block word 4 is the last-block counter of router_topk
    TopkArgs a{T, E, k, c.renorm, c.routed_scale, sc, ch, idx, weight,
               L.n_chunks == 1 ? status + 4 : nullptr, m};
    timing_begin("router_topk", s);
    err = launch_pdl(router_topk_kernel, dim3(T), dim3(1024), 0, s, a);
    count_launch();
    timing_end("router_topk", s);
    if (err != cudaSuccess) return err;
    if (L.n_chunks > 1) {
        int32_t *base = reinterpret_cast<int32_t *>(ws + L.chunk_base);
        timing_begin("perm_count", s);
        err = launch_pdl(perm_count_kernel, dim3(L.n_chunks), dim3(1024), 0, s, m);
        count_launch();
        timing_end("perm_count", s);
        if (err != cudaSuccess) return err;
        timing_begin("perm_scan", s);
        err = launch_pdl(perm_scan_kernel, dim3(1), dim3(1024), 0, s, L.n_chunks, E, T * k,
                         (const int32_t *)m.chunk_counts, base, offsets);
        count_launch();
        timing_end("perm_scan", s);
        if (err != cudaSuccess) return err;
        timing_begin("perm_scatter", s);
        err = launch_pdl(perm_scatter_kernel, dim3((T * k + 255) / 256), dim3(256), 0, s, T * k, k, E,
                         (const int32_t *)idx, (const int32_t *)base, (const int32_t *)m.local_rank, perm);
        count_launch();
        timing_end("perm_scatter", s);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

}  // namespace k3moe
