// k3moe_route.cu -- router and token -> expert map (kimi-k3-in-c README, Part II,
// section 9 "Picking 16 experts of 896").
//
// The router listing accumulates each logit in double and rounds it to float once, then
// takes sc = 1/(1+expf(-logit)) and ch = sc + bias in float.  Those float values decide
// which experts win, so the kernels here reproduce them: a logit is computed exactly
// (up to the final rounding) and the sigmoid from a double exponential rounded to float.
//
// Kernels, in launch order:
//   router_scores  (few tokens) exact logits, sc and ch for every (token, expert), to the
//                  workspace.  A block owns 4 experts (one per warp, its Wr row held in
//                  registers) and walks its tokens 8 at a time through shared memory;
//   router_wnorm   (many tokens) |Wr[e]| for every expert, for the bound below;
//   router_logits_tc (many tokens, k3moe_route_tc.cu) approximate logits on the tensor
//                  cores;
//   router_topk    one block per token: warp-level bitonic sorts and merges of 64-bit keys
//                  (ch, then the lower index first) pick the top k in rank order.  With
//                  approximate logits it first brackets every expert's exact ch between
//                  a lower and an upper bound, keeps the experts whose upper bound reaches
//                  the k-th largest lower bound (the only ones that can be chosen),
//                  re-scores those exactly and selects among them.  The weights are the
//                  chosen sc renormalised by their float sum in rank order, times
//                  routed_scale.  With at most 64 tokens the last block to finish (the
//                  only one, for one token) also builds the map;
//   perm_count     (more tokens) per chunk of 64 tokens: per-expert slot counts and each
//                  slot's stable rank inside the chunk (warp match + popc, warp by warp);
//   perm_scan      per-expert exclusive scan over chunks, then over experts -> offsets;
//   perm_scatter   perm[base + rank] = slot.
// The map is a stable counting sort: offsets = exclusive prefix sum of the per-expert
// counts, and inside an expert's segment the flat slot ids t*k+j ascend.
#include "k3moe_exp.cuh"
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kScoreWarps = 4;       // experts per block (one per warp)
constexpr int kScoreTok = 8;         // tokens staged per round
constexpr int kScoreTokBlock = 8;    // tokens per block (grid.y walks the rest)
constexpr int kScoreChunks = 16;     // 16-byte Wr chunks per lane held at once (4096 columns)

// Bound on the tensor-core logits' error, relative to |x_t| |Wr[e]|.  Their fp32
// accumulation was measured within 2^-22 of that scale (3.7e-6 on unit-scale scores,
// 1.3e-5 on tokens scaled by 8, over 14.7M scores); the bound keeps a factor of 1024
// above it.  It only widens the set of experts re-scored exactly, never the result.
constexpr float kTcLogitRel = 0x1p-12f;

// -------------------------------------------------------------------------------- exact logits
// A logit is a sum of d products of two bf16 values, each exact in fp32.  It is carried
// as an unevaluated pair (s, c): s the fp32 running sum, c the running sum of the exact
// rounding errors of s's additions (Knuth's two-sum), and rounded once, to s + c.  A lane
// keeps four such pairs (its 16-byte chunks take them in turn, for four independent
// dependency chains); the pairs, then the lanes, are merged by the same rule.  The result is the float nearest the exact sum
// unless that sum lies within about 2^-40 (relative) of a rounding boundary -- what the
// listing's double accumulation rounded to float gives.  Every kernel that computes a
// logit exactly goes through these functions with the same chunk-to-lane assignment
// (chunk lane + 32 m, pair m & 3, m ascending), so their results are bitwise equal.
struct Acc2 {
    float s, c;
};

__device__ __forceinline__ void acc_add(Acc2 &a, float p)
{
    const float t = __fadd_rn(a.s, p);
    const float z = __fsub_rn(t, a.s);
    const float e = __fadd_rn(__fsub_rn(a.s, __fsub_rn(t, z)), __fsub_rn(p, z));
    a.s = t;
    a.c = __fadd_rn(a.c, e);
}

// Merging is symmetric in its arguments (the two-sum error of s_a + s_b is unique), so
// both lanes of a butterfly step hold the same pair afterwards.
__device__ __forceinline__ Acc2 acc_merge(Acc2 a, const Acc2 b)
{
    a.c = __fadd_rn(a.c, b.c);
    acc_add(a, b.s);
    return a;
}

// One 16-byte chunk: 8 products in element order (low half of each word first).
__device__ __forceinline__ void acc_chunk(Acc2 &a, const uint4 xv, const uint4 wv)
{
    const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t wu[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
        acc_add(a, __fmul_rn(__uint_as_float(xu[q] << 16), __uint_as_float(wu[q] << 16)));
        acc_add(a, __fmul_rn(__uint_as_float(xu[q] & 0xFFFF0000u), __uint_as_float(wu[q] & 0xFFFF0000u)));
    }
}

// The four pairs of every lane -> the rounded logit, on every lane.
__device__ __forceinline__ float acc_finish(const Acc2 a0, const Acc2 a1, const Acc2 a2, const Acc2 a3)
{
    Acc2 a = acc_merge(acc_merge(a0, a1), acc_merge(a2, a3));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        Acc2 b;
        b.s = __shfl_xor_sync(0xffffffffu, a.s, o);
        b.c = __shfl_xor_sync(0xffffffffu, a.c, o);
        a = acc_merge(a, b);
    }
    return __fadd_rn(a.s, a.c);
}

// sc = 1/(1+expf(-logit)) and ch = sc + bias, each step rounded to float as the listing
// writes them, with the correctly rounded float exponential (exp_rn: wrong only within
// ~2^-40 of a rounding tie).
__device__ __forceinline__ void exact_scores(float logit, float bias, float &sc, float &ch)
{
    const float ef = exp_rn(-logit);
    sc = __fdiv_rn(1.0f, __fadd_rn(1.0f, ef));
    ch = __fadd_rn(sc, bias);
}

// Exact logit of one (token, expert) pair by one warp: the token row in shared memory, the
// router row in global memory, nchunk 16-byte chunks each.
__device__ __forceinline__ float exact_logit_warp(const uint4 *xs, const uint4 *__restrict__ wrow, int nchunk,
                                                  int lane)
{
    Acc2 a[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
    // eight router chunks in flight per lane, then added in order (pair m & 3)
    for (int m0 = 0; lane + 32 * m0 < nchunk; m0 += 8) {
        uint4 w[8];
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int c = lane + 32 * (m0 + j);
            w[j] = c < nchunk ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int c = lane + 32 * (m0 + j);
            if (c < nchunk) acc_chunk(a[j & 3], xs[c], w[j]);
        }
    }
    return acc_finish(a[0], a[1], a[2], a[3]);
}

// -------------------------------------------------------------------------------- exact scores
// grid (ceil(E / 4), ceil(T / 8)); block y owns tokens [8 y, 8 y + 8).
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
    const int tb0 = blockIdx.y * kScoreTokBlock, tb1 = min(T, tb0 + kScoreTokBlock);
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
    for (int t0 = tb0; t0 < tb1; t0 += kScoreTok) {
        const int nt = min(kScoreTok, tb1 - t0);
        __syncthreads();
        for (int q = threadIdx.x; q < nt * nchunk; q += blockDim.x) {
            const int i = q / nchunk, c = q % nchunk;
            xs[i * nchunk + c] = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + i) * d) + c);
        }
        __syncthreads();
        // one token at a time (a loop, not unrolled: the unrolled body of all tokens would
        // not fit the instruction cache); its two chains over the lane's chunks, the row
        // chunks held in registers across the tokens
        float logit = 0.0f;
#pragma unroll 1
        for (int i = 0; i < nt; i++) {
            Acc2 a[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
            for (int c0 = 0; c0 < nchunk; c0 += 32 * kScoreChunks) {
                uint4 w[kScoreChunks];
#pragma unroll
                for (int j = 0; j < kScoreChunks; j++) {
                    const int c = c0 + lane + 32 * j;
                    w[j] = c0 == 0 ? w0[j] : (c < nchunk ? __ldg(wrow + c) : make_uint4(0, 0, 0, 0));
                }
#pragma unroll
                for (int j = 0; j < kScoreChunks; j++) {
                    const int c = c0 + lane + 32 * j;   // this lane's chunk number c0 / 32 + j = j mod 4
                    if (c < nchunk) acc_chunk(a[j & 3], xs[i * nchunk + c], w[j]);
                }
            }
            const float v = acc_finish(a[0], a[1], a[2], a[3]);
            if (lane == i) logit = v;
        }
        if (e < E && lane < nt) {
            float s, ch;
            exact_scores(logit, b, s, ch);
            sc_out[(size_t)(t0 + lane) * E + e] = s;
            ch_out[(size_t)(t0 + lane) * E + e] = ch;
        }
    }
}

// |Wr[e]| (times 1.001, above the fp32 rounding of the sum of squares), one warp per row.
__global__ void __launch_bounds__(256) router_wnorm_kernel(int d, int E, const uint16_t *__restrict__ wr,
                                                           float *__restrict__ wnorm)
{
    pdl_wait();
    pdl_trigger();
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (e >= E) return;
    const uint4 *row = reinterpret_cast<const uint4 *>(wr + (size_t)e * d);
    float ss = 0.0f;
    for (int c = lane; c < d / 8; c += 32) {
        const uint4 v = __ldg(row + c);
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const float lo = __uint_as_float(u[q] << 16), hi = __uint_as_float(u[q] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) wnorm[e] = sqrtf(ss) * 1.001f;
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
        if (my_e >= 0) {
            const int p = cnt[my_e] + my_rank;
            if (dcheck(a.status, p >= 0 && p < a.T * k)) a.perm[p] = t_begin * k + threadIdx.x;
        }
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

__device__ __forceinline__ uint64_t choice_key(float ch, int e)
{
    return ((uint64_t)orderable(ch) << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)e);
}

struct TopkArgs {
    int T, E, k, renorm;
    float routed_scale;
    const float *sc, *ch;   // exact scores [T][E] (per-token kernel), or:
    const float *logit;     // approximate logits [T][E] (tensor cores), re-scored here
    const float *bias;      // [E] or NULL (re-scoring only)
    const float *wnorm;     // |Wr[e]| [E] (re-scoring only)
    const uint16_t *x, *wr; // token rows and router rows (re-scoring only)
    int d;
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

// The 16 largest of the keys that threads 0..n-1 offer (n <= 1024; a missing key counts
// as 0, below every real key).  Warp w sorts keys 32w..32w+31 and keeps its 16 largest;
// pairs of lists are then merged warp by warp (16 of 32 kept) until one remains.  Returns
// the rank-r key in lane r < 16 of warp 0 (0 elsewhere).  Called by the whole block.
__device__ uint64_t block_top16(uint64_t key, int n, uint64_t (*lists)[32][kMaxTopK])
{
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    const int nl0 = max(1, (n + 31) >> 5);         // lists after the first level
    __syncthreads();                               // the lists may be in use from a previous call
    if (warp < nl0) {
        key = warp_sort_desc(i < n ? key : 0, lane);
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
    return (warp == 0 && lane < kMaxTopK) ? lists[cur][0][lane] : 0;
}

// Float sigmoid for the bounds of the re-scoring step (any accuracy within a few ulp).
__device__ __forceinline__ float sigmoid_bound(float v) { return 1.0f / (1.0f + expf(-v)); }

// blockDim = 1024; block t owns token t; the scores are the exact ones of the per-token
// kernel.  Key = (orderable(ch) << 32) | ~index, so a descending order sorts by ch and,
// among equal ch, by ascending index -- the order the repeated maximum with a strict
// comparison produces.  Every key is distinct, so the k largest keys are the selection.
__global__ void __launch_bounds__(1024) router_topk_kernel(TopkArgs a)
{
    pdl_trigger();      // the next kernel may launch now: it waits for this one
    pdl_wait();
    __shared__ uint64_t lists[2][32][kMaxTopK];
    __shared__ int32_t cnt[kMaxExperts];
    __shared__ int32_t slot_e[kChunkTokens * kMaxTopK];
    __shared__ int32_t scan_tmp[32];
    __shared__ int last;
    const int i = threadIdx.x;
    const int t = blockIdx.x, E = a.E, k = a.k;
    const uint64_t key = i < E ? choice_key(a.ch[(size_t)t * E + i], i) : 0;
    const uint64_t top = block_top16(key, E, lists);
    // lane r < k of warp 0 now holds the rank-r key
    if (i < 32) {
        int e = -1;
        float w = 0.0f;
        if (i < k) {
            e = (int)(0xFFFFFFFFu - (uint32_t)top);
            if (e < 0 || e >= E) {                 // no valid key (non-finite scores); stay in bounds
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

// ---------------------------------------------------------------- top-k from tensor-core logits
constexpr int kSelThreads = 128;    // one token per block of 4 warps

// Warp w merges a list of keys (lanes 0-15 of `run`, descending) with the 32 keys of a
// chunk (one per lane): the chunk is sorted, its 16 largest reversed into lanes 16-31,
// and the bitonic merge leaves the 16 largest of both in lanes 0-15.
__device__ __forceinline__ uint64_t merge_chunk(uint64_t run, uint64_t key, int lane)
{
    key = warp_sort_desc(key, lane);
    const uint64_t rev = __shfl_sync(0xffffffffu, key, 31 - lane);   // lane 16+j gets rank 15-j
    const uint64_t v = lane < 16 ? run : rev;
    return warp_merge_desc(v, lane);
}

// The 16 largest of n keys in `keys` (shared memory; n <= 1024), by the 4 warps of the
// block: each warp merges its chunks of 32 into a list, then warp 0 merges the 4 lists.
// Returns the rank-r key in lane r < 16 of warp 0.  Called by the whole block.
__device__ uint64_t sel_top16(const uint64_t *keys, int n, uint64_t (*lists)[kMaxTopK])
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t run = 0;
    for (int c0 = 32 * warp; c0 < n; c0 += 32 * (kSelThreads / 32)) {
        const int i = c0 + lane;
        run = merge_chunk(run, i < n ? keys[i] : 0, lane);
    }
    if (lane < kMaxTopK) lists[warp][lane] = run;
    __syncthreads();
    uint64_t top = 0;
    if (warp == 0) {
        top = lane < kMaxTopK ? lists[0][lane] : 0;
        for (int w = 1; w < kSelThreads / 32; w++) {
            const uint64_t other = lane < kMaxTopK ? lists[w][lane] : 0;    // descending in 0-15
            const uint64_t rev = __shfl_sync(0xffffffffu, other, 31 - lane);
            top = warp_merge_desc(lane < 16 ? top : rev, lane);
        }
    }
    __syncthreads();
    return top;
}

// blockDim = 128; block t owns token t.  The tensor-core logits la bound every expert's
// exact choice score (|la - logit| <= L = 2^-12 |x_t| |Wr[e]|): lo/hi = sigmoid(la -/+ L)
// + bias -/+ slack.  The k-th largest exact ch is at least the k-th largest lo, so only the
// experts whose hi reaches it can be chosen (and none below it can tie with the k-th);
// those are re-scored exactly and the selection is the top k of their exact keys.
__global__ void __launch_bounds__(kSelThreads) router_select_kernel(TopkArgs a)
{
    pdl_trigger();      // the next kernel may launch now: it waits for this one
    pdl_wait();
    extern __shared__ __align__(16) uint8_t sel_dyn[];   // the token row (d bf16)
    __shared__ uint64_t keys[kMaxExperts];
    __shared__ uint32_t hio[kMaxExperts];
    __shared__ int32_t cand[kMaxExperts];
    __shared__ float scx[kMaxExperts];
    __shared__ uint64_t lists[kSelThreads / 32][kMaxTopK];
    __shared__ float red[kSelThreads / 32];
    __shared__ uint32_t thr_o;
    __shared__ int n_cand;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5;
    const int t = blockIdx.x, E = a.E, k = a.k;
    const int nchunk = a.d / 8;
    uint4 *xs = reinterpret_cast<uint4 *>(sel_dyn);
    const uint4 *xg = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.d);
    float ss = 0.0f;
    for (int q = i; q < nchunk; q += kSelThreads) {
        const uint4 v = __ldg(xg + q);
        xs[q] = v;
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int r = 0; r < 4; r++) {
            const float lo = __uint_as_float(u[r] << 16), hi = __uint_as_float(u[r] & 0xFFFF0000u);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) red[warp] = ss;
    if (i == 0) n_cand = 0;
    __syncthreads();
    float xn2 = 0.0f;
#pragma unroll
    for (int w = 0; w < kSelThreads / 32; w++) xn2 += red[w];
    const float xn = sqrtf(xn2) * 1.001f;
    for (int e = i; e < E; e += kSelThreads) {
        const float la = a.logit[(size_t)t * E + e];
        const float L = kTcLogitRel * xn * a.wnorm[e];
        const float b = a.bias ? a.bias[e] : 0.0f;
        const float slack = 1e-6f + fabsf(b) * 0x1p-20f;
        const float lo = sigmoid_bound(la - L) + b - slack;
        const float hi = sigmoid_bound(la + L) + b + slack;
        keys[e] = choice_key(lo, e);
        hio[e] = hi == hi ? orderable(hi) : 0u;          // NaN never passes
    }
    __syncthreads();
    const uint64_t lk = sel_top16(keys, E, lists);
    if (warp == 0 && lane == k - 1) thr_o = (uint32_t)(lk >> 32);
    __syncthreads();
    // candidates (their order does not matter: the selection sorts their keys)
    for (int e = i; e < E; e += kSelThreads)
        if (hio[e] >= thr_o) {
            const int c = atomicAdd(&n_cand, 1);
            if (dcheck(a.map.status, c < E)) cand[c] = e;
        }
    __syncthreads();
    const int C = min(n_cand, E);
    // exact scores of the candidates, one warp per candidate
    const uint4 *wr = reinterpret_cast<const uint4 *>(a.wr);
    for (int c = warp; c < C; c += kSelThreads / 32) {
        const int e = cand[c];
        const float logit = exact_logit_warp(xs, wr + (size_t)e * nchunk, nchunk, lane);
        if (lane == 0) {
            float sv, cv;
            exact_scores(logit, a.bias ? a.bias[e] : 0.0f, sv, cv);
            scx[e] = sv;
            keys[c] = choice_key(cv, e);
        }
    }
    __syncthreads();
    const uint64_t top = sel_top16(keys, C, lists);
    if (warp == 0) {
        int e = -1;
        float w = 0.0f;
        if (lane < k) {
            e = (int)(0xFFFFFFFFu - (uint32_t)top);
            if (e < 0 || e >= E) {                 // no valid key (non-finite scores); stay in bounds
                set_status(a.map.status, K3MOE_DEV_BAD_INDEX);
                e = 0;
            }
            w = scx[e];
        }
        float s = 0.0f;
        for (int j = 0; j < k; j++) s += __shfl_sync(0xffffffffu, w, j);
        if (lane < k) {
            if (a.renorm && s > 0.0f) w = w / s;
            w = w * a.routed_scale;
            a.idx[(size_t)t * k + lane] = e;
            a.weight[(size_t)t * k + lane] = w;
        }
    }
}

__global__ void __launch_bounds__(1024) perm_count_kernel(MapArgs a)
{
    pdl_trigger();      // the next kernel may launch now: it waits for this one
    pdl_wait();
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
    pdl_trigger();      // the next kernel may launch now: it waits for this one
    pdl_wait();
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
                                                           int32_t *__restrict__ perm, int32_t *status)
{
    pdl_trigger();      // the next kernel may launch now: it waits for this one
    pdl_wait();
    const int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= total_slots) return;
    const int e = idx[s];
    if (!dguard(status, e >= 0 && e < E)) return;
    const int chunk = s / (kChunkTokens * k);
    const int p = chunk_base[(size_t)chunk * E + e] + local_rank[s];
    if (dguard(status, p >= 0 && p < total_slots)) perm[p] = s;
}

}  // namespace

cudaError_t launch_router_scores(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                                 const float *bias, float *sc, float *ch, int32_t *status, cudaStream_t s)
{
    (void)status;
    const int E = c.n_experts;
    static size_t smem_set = 0;
    const size_t smem = (size_t)kScoreTok * c.d * 2;
    if (smem > smem_set) {
        cudaFuncSetAttribute(router_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        smem_set = smem;
    }
    timing_begin("router_scores", s);
    cudaError_t err = launch_pdl(router_scores_kernel,
                                 dim3((E + kScoreWarps - 1) / kScoreWarps, (T + kScoreTokBlock - 1) / kScoreTokBlock),
                                 dim3(kScoreWarps * 32), smem, s, T, c.d, E, x, wr, bias, sc, ch);
    count_launch();
    timing_end("router_scores", s);
    if (err != cudaSuccess) return err;
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
    float *wnorm = reinterpret_cast<float *>(ws + L.wnorm);
    const bool tc = router_tc_applies(c, T);
    cudaError_t err;
    if (tc) {
        // approximate logits into the sc region, re-scored by the top-k
        timing_begin("router_wnorm", s);
        err = launch_pdl(router_wnorm_kernel, dim3((E + 7) / 8), dim3(256), 0, s, c.d, E, wr, wnorm);
        count_launch();
        timing_end("router_wnorm", s);
        if (err != cudaSuccess) return err;
        timing_begin("router_logits_tc", s);
        err = launch_router_logits_tc(c, T, x, wr, sc, status, s);
        timing_end("router_logits_tc", s);
    } else {
        err = launch_router_scores(c, T, x, wr, bias, sc, ch, status, s);
    }
    if (err != cudaSuccess) return err;
    MapArgs m{T, E, k, idx, offsets, perm, reinterpret_cast<int32_t *>(ws + L.chunk_counts),
              reinterpret_cast<int32_t *>(ws + L.local_rank), status};
    // status block word 4 is the last-block counter of router_topk
    // the per-token kernel's exact scores: the 1024-thread top-k, which for at most 64
    // tokens also builds the map; the tensor-core logits: the 128-thread select kernel
    // (re-scoring its candidates), the map by the perm kernels
    TopkArgs a{T, E, k, c.renorm, c.routed_scale, sc, ch, tc ? sc : nullptr, bias, wnorm, x, wr, c.d,
               idx, weight, (!tc && L.n_chunks == 1) ? status + 4 : nullptr, m};
    timing_begin("router_topk", s);
    if (tc) {
        static size_t sel_smem = 0;
        const size_t smem = (size_t)c.d * 2;
        if (smem > sel_smem) {
            cudaFuncSetAttribute(router_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            sel_smem = smem;
        }
        err = launch_pdl(router_select_kernel, dim3(T), dim3(kSelThreads), smem, s, a);
    } else {
        err = launch_pdl(router_topk_kernel, dim3(T), dim3(1024), 0, s, a);
    }
    count_launch();
    timing_end("router_topk", s);
    if (err != cudaSuccess) return err;
    if (tc && L.n_chunks == 1) {          // one chunk: perm_count builds the whole map
        timing_begin("perm_count", s);
        err = launch_pdl(perm_count_kernel, dim3(1), dim3(1024), 0, s, m);
        count_launch();
        timing_end("perm_count", s);
        if (err != cudaSuccess) return err;
    }
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
                         (const int32_t *)idx, (const int32_t *)base, (const int32_t *)m.local_rank, perm,
                         status);
        count_launch();
        timing_end("perm_scatter", s);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

}  // namespace k3moe
