// k3moe_gemv.cu -- the expert part of the layer as grouped, streamed mat-vecs:
// the decode path (few tokens per expert).  kimi-k3-in-c README, Part II,
// section 4 (MXFP4 mat-vec: per-32 partial sums times the E8M0 scale, nothing
// dequantised to memory) and section 9 (the k3_moe expert loop: gate = w1,
// up = w3, SiTU-GLU, down = w2, weighted sum; shared experts unweighted).
//
// Kernels, in launch order:
//   fwd_prep     validates offsets/perm against idx, lists the active experts and
//                inverts perm (slot -> position); sets the abort flag on bad input;
//   gemv_gateup  h = SiTU(W1 x, W3 x) for every (active expert, token) and every
//                (shared expert, token), fp32, rows of h in perm order;
//   gemv_down    y = W2 h, fp32, same row order;
//   fwd_combine  out[t] = sum_j w[t][j] y[pos(t,j)] + sum_s y_shared[s][t], in j order.
//
// Streaming: a persistent grid; each block owns a contiguous range of work items
// (64 weight rows of one expert), so consecutive items share the expert and its
// staged activations.  Weight tiles move global -> shared with bulk async copies
// (cp.async.bulk for the packed MXFP4 tiles, tensor-map TMA loads for the bf16
// shared experts) through a 4-stage mbarrier ring; each thread owns one weight
// row and a K slice, so the activations it needs are the same for the whole
// warp (shared-memory broadcast) and the packed bytes it reads are consecutive
// across the warp.  MXFP4 pairs decode with the hardware e2m1x2 conversion.
#include <cuda.h>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kThreads = 256;
constexpr int kItemRows = 64;
constexpr int kStages = 4;
constexpr int kStageBytes = 16384;
constexpr int kNT = 4;                    // tokens per pass
constexpr uint32_t kWaitLimit = 1u << 26; // bounded mbarrier polls

enum Mode { kGateUp = 0, kDown = 1 };

// -------------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}
// Returns false when the bounded wait gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t a = smem_addr(bar);
    for (uint32_t i = 0; i < kWaitLimit; i++) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_2d_g2s(void *dst, const CUtensorMap *map, int c0, int c1,
                                           uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float situ(float g, float u, float b1, float b2)
{
    const float a = b1 * tanhf(g / b1) * (1.0f / (1.0f + expf(-g)));
    return a * (b2 * tanhf(u / b2));
}

// -------------------------------------------------------------------------------- prep
struct PrepArgs {
    int T, E, k;
    const int32_t *idx, *offsets, *perm;
    int32_t *active;     // [E + 1]
    int32_t *inv;        // [T * k]
    int32_t *status;
    int32_t *abort;
};

__global__ void __launch_bounds__(1024) fwd_prep_kernel(PrepArgs a)
{
    __shared__ int32_t bad;
    __shared__ int32_t scan_tmp[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, slots = a.T * a.k;
    if (tid == 0) bad = 0;
    __syncthreads();
    // offsets: monotone, start 0, end T*k
    for (int e = tid; e < E; e += blockDim.x) {
        const int lo = a.offsets[e], hi = a.offsets[e + 1];
        if (lo < 0 || hi < lo || hi > slots) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    }
    if (tid == 0 && (a.offsets[0] != 0 || a.offsets[E] != slots)) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    for (int s = tid; s < slots; s += blockDim.x) {
        const int e = a.idx[s];
        if (e < 0 || e >= E) atomicOr(&bad, K3MOE_DEV_BAD_INDEX);
        a.inv[s] = -1;
    }
    __syncthreads();
    const bool offsets_ok = !(bad & K3MOE_DEV_BAD_OFFSETS);
    // active experts in ascending order (block scan over flags)
    int run = 0;
    for (int base = 0; base < E; base += blockDim.x) {
        const int e = base + tid;
        const int flag = (offsets_ok && e < E && a.offsets[e + 1] > a.offsets[e]) ? 1 : 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) scan_tmp[warp] = __popc(bal);
        __syncthreads();
        int before = run;
        for (int w = 0; w < warp; w++) before += scan_tmp[w];
        if (flag) a.active[before + __popc(bal & ((1u << lane) - 1u))] = e;
        int tot = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += scan_tmp[w];
        run += tot;
        __syncthreads();
    }
    if (tid == 0) a.active[E] = offsets_ok ? run : 0;
    // perm: a permutation of the slots, each in the segment of its expert
    if (offsets_ok) {
        for (int p = tid; p < slots; p += blockDim.x) {
            const int s = a.perm[p];
            if (s < 0 || s >= slots) {
                atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
                continue;
            }
            int lo = 0, hi = E;   // find e with offsets[e] <= p < offsets[e+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (a.offsets[mid] <= p) lo = mid; else hi = mid;
            }
            if (a.idx[s] != lo) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
            if (atomicExch(&a.inv[s], p) != -1) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (bad) atomicOr(a.status, bad);
        *a.abort = bad ? 1 : 0;
    }
}

// -------------------------------------------------------------------------------- streamed mat-vec
struct GemvArgs {
    int T, d, f, k, S, E;
    float b1, b2;
    const uint16_t *x;
    const int32_t *offsets, *perm, *active;
    const uint8_t *table;
    size_t expert_bytes, gateup_bytes;
    float *h, *ys;
    const int32_t *abort;
    int32_t *status;
};

struct Unit {         // one expert (routed or shared) with its tokens
    int shared;       // 0: routed expert e; 1: shared expert s
    int id;           // e or s
    int tok0, ntok;   // routed: positions [tok0, tok0+ntok) of perm; shared: tokens [0, T)
};

__device__ __forceinline__ Unit unit_of(const GemvArgs &a, int n_active, int u)
{
    Unit r;
    if (u < n_active) {
        r.shared = 0;
        r.id = a.active[u];
        r.id = min(max(r.id, 0), a.E - 1);
        r.tok0 = a.offsets[r.id];
        r.ntok = a.offsets[r.id + 1] - r.tok0;
    } else {
        r.shared = 1;
        r.id = u - n_active;
        r.tok0 = 0;
        r.ntok = a.T;
    }
    return r;
}

// The flat sequence of stages one block streams: items -> token groups -> K tiles.
struct Cursor {
    int item, grp, kt;
};

template <int MODE>
struct Geo {
    __host__ __device__ static constexpr int rows_of(int d, int f) { return MODE == kGateUp ? f : d; }
    __host__ __device__ static constexpr int k_of(int d, int f) { return MODE == kGateUp ? d : f; }
};

// Issue the copies of one stage (thread 0 only).
template <int MODE>
__device__ void issue_stage(const GemvArgs &a, const CUtensorMap *m1, const CUtensorMap *m3,
                            const CUtensorMap *m2, const Unit &un, int item_row, int kt,
                            uint8_t *buf, uint64_t *bar)
{
    const int rb = item_row / kTileRows, half = (item_row % kTileRows) / kItemRows;
    if (!un.shared) {
        const uint8_t *ex = a.table + (size_t)un.id * a.expert_bytes;
        if (MODE == kGateUp) {
            const int ktn = a.d / kTileK;
            const uint8_t *pair = ex + ((size_t)rb * ktn + kt) * 2 * kTileBytes;
            mbar_expect_tx(bar, 2 * (4 * 1024 + 256));
            for (int m = 0; m < 2; m++) {
                const uint8_t *tile = pair + (size_t)m * kTileBytes;
                uint8_t *dst = buf + m * 4352;
                for (int c = 0; c < 4; c++)
                    bulk_g2s(dst + c * 1024, tile + c * 2048 + half * 1024, 1024, bar);
                bulk_g2s(dst + 4096, tile + kTileNibbleBytes + half * 256, 256, bar);
            }
        } else {
            const int ktn = a.f / kTileK;
            const uint8_t *tile = ex + a.gateup_bytes + ((size_t)rb * ktn + kt) * kTileBytes;
            mbar_expect_tx(bar, 4 * 1024 + 256);
            for (int c = 0; c < 4; c++)
                bulk_g2s(buf + c * 1024, tile + c * 2048 + half * 1024, 1024, bar);
            bulk_g2s(buf + 4096, tile + kTileNibbleBytes + half * 256, 256, bar);
        }
    } else {
        // bf16 shared experts: boxes of 64 K x 64 rows (8 KB), 128-byte swizzle
        const int k0 = kt * 64;
        if (MODE == kGateUp) {
            const int row = un.id * a.f + item_row;
            mbar_expect_tx(bar, 2 * 8192);
            tma_2d_g2s(buf, m1, k0, row, bar);
            tma_2d_g2s(buf + 8192, m3, k0, row, bar);
        } else {
            const int row = un.id * a.d + item_row;
            mbar_expect_tx(bar, 8192);
            tma_2d_g2s(buf, m2, k0, row, bar);
        }
    }
}

template <int MODE>
__device__ __forceinline__ int n_ktiles(const GemvArgs &a, int shared)
{
    const int K = Geo<MODE>::k_of(a.d, a.f);
    return shared ? K / 64 : K / kTileK;
}

// Stage NT activation rows (f32) for token group `grp` of unit `un` into xs.
template <int MODE>
__device__ void stage_x(const GemvArgs &a, const Unit &un, int grp, float *xs, int &nvalid)
{
    const int K = Geo<MODE>::k_of(a.d, a.f);
    const int first = grp * kNT;
    nvalid = min(kNT, un.ntok - first);
    for (int i = 0; i < kNT; i++) {
        float *dst = xs + (size_t)i * K;
        if (i >= nvalid) {
            for (int q = threadIdx.x; q < K; q += kThreads) dst[q] = 0.0f;
            continue;
        }
        if (MODE == kGateUp) {
            int t;
            if (un.shared) t = first + i;
            else {
                const int slot = a.perm[un.tok0 + first + i];
                t = min(max(slot, 0), a.T * a.k - 1) / a.k;
            }
            const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (size_t)t * K);
            for (int q = threadIdx.x; q < K / 8; q += kThreads) {
                const uint4 v = src[q];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float4 lo, hi;
                lo.x = __uint_as_float(w[0] << 16); lo.y = __uint_as_float(w[0] & 0xFFFF0000u);
                lo.z = __uint_as_float(w[1] << 16); lo.w = __uint_as_float(w[1] & 0xFFFF0000u);
                hi.x = __uint_as_float(w[2] << 16); hi.y = __uint_as_float(w[2] & 0xFFFF0000u);
                hi.z = __uint_as_float(w[3] << 16); hi.w = __uint_as_float(w[3] & 0xFFFF0000u);
                reinterpret_cast<float4 *>(dst)[2 * q] = lo;
                reinterpret_cast<float4 *>(dst)[2 * q + 1] = hi;
            }
        } else {
            const size_t hrow = un.shared ? (size_t)a.T * a.k + (size_t)un.id * a.T + first + i
                                          : (size_t)(un.tok0 + first + i);
            const float4 *src = reinterpret_cast<const float4 *>(a.h + hrow * K);
            for (int q = threadIdx.x; q < K / 4; q += kThreads)
                reinterpret_cast<float4 *>(dst)[q] = src[q];
        }
    }
}

// One 32-column MXFP4 group of one row against NV activation rows (row stride K):
// the group's partial sums, then times the group's power-of-two scale.
template <int NV>
__device__ __forceinline__ void mxfp4_group(const uint4 nib, float scale, const float *xk, int K,
                                            float acc[kNT])
{
    float part[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) part[i] = 0.0f;
    const uint32_t w[4] = {nib.x, nib.y, nib.z, nib.w};
#pragma unroll
    for (int q = 0; q < 4; q++) {
#pragma unroll
        for (int b = 0; b < 4; b += 2) {
            const float2 w01 = e2m1x2_to_f32x2(w[q] >> (8 * b));
            const float2 w23 = e2m1x2_to_f32x2(w[q] >> (8 * b + 8));
            const int col = q * 8 + b * 2;
#pragma unroll
            for (int i = 0; i < NV; i++) {
                const float4 xv = *reinterpret_cast<const float4 *>(xk + (size_t)i * K + col);
                part[i] = fmaf(w01.x, xv.x, part[i]);
                part[i] = fmaf(w01.y, xv.y, part[i]);
                part[i] = fmaf(w23.x, xv.z, part[i]);
                part[i] = fmaf(w23.y, xv.w, part[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NV; i++) acc[i] = fmaf(part[i], scale, acc[i]);
}

// 8 bf16 weights (one 16-byte chunk) against NV activation rows.
template <int NV>
__device__ __forceinline__ void bf16_chunk(const uint4 wv, const float *xk, int K, float acc[kNT])
{
    const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int q = 0; q < 4; q += 2) {
        const float w0 = __uint_as_float(w[q] << 16), w1 = __uint_as_float(w[q] & 0xFFFF0000u);
        const float w2 = __uint_as_float(w[q + 1] << 16), w3 = __uint_as_float(w[q + 1] & 0xFFFF0000u);
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const float4 xv = *reinterpret_cast<const float4 *>(xk + (size_t)i * K + 2 * q);
            acc[i] = fmaf(w0, xv.x, acc[i]);
            acc[i] = fmaf(w1, xv.y, acc[i]);
            acc[i] = fmaf(w2, xv.z, acc[i]);
            acc[i] = fmaf(w3, xv.w, acc[i]);
        }
    }
}

// The per-thread work on one staged weight tile.
template <int MODE, int NV>
__device__ __forceinline__ void consume_tile(const uint8_t *buf, int shared, int kt, int K,
                                             const float *xs, float acc[kNT])
{
    const int tid = threadIdx.x, r = tid & (kItemRows - 1);
    if (!shared) {
        if (MODE == kGateUp) {
            // thread: row r of matrix tid>>7, groups 2*kh, 2*kh+1 of the 128-column tile
            const int mat = tid >> 7, kh = (tid >> 6) & 1;
            const uint8_t *mb = buf + mat * 4352;
            const uint32_t sc4 = *reinterpret_cast<const uint32_t *>(mb + 4096 + r * 4);
#pragma unroll
            for (int cc = 0; cc < 2; cc++) {
                const int c = 2 * kh + cc;
                const float scale = e8m0_to_f32(sc4 >> (8 * c));
                if (scale != 0.0f) {
                    const uint4 nib = *reinterpret_cast<const uint4 *>(mb + c * 1024 + r * 16);
                    mxfp4_group<NV>(nib, scale, xs + kt * kTileK + c * 32, K, acc);
                }
            }
        } else {
            const int c = tid >> 6;
            const uint32_t sc4 = *reinterpret_cast<const uint32_t *>(buf + 4096 + r * 4);
            const float scale = e8m0_to_f32(sc4 >> (8 * c));
            if (scale != 0.0f) {
                const uint4 nib = *reinterpret_cast<const uint4 *>(buf + c * 1024 + r * 16);
                mxfp4_group<NV>(nib, scale, xs + kt * kTileK + c * 32, K, acc);
            }
        }
    } else {
        // 128-byte swizzled rows of 64 bf16: chunk q of row r sits at r*128 + ((q ^ (r&7))*16)
        if (MODE == kGateUp) {
            const int mat = tid >> 7, kh = (tid >> 6) & 1;
            const uint8_t *mb = buf + mat * 8192;
#pragma unroll
            for (int cc = 0; cc < 4; cc++) {
                const int q = kh * 4 + cc;
                const uint4 wv = *reinterpret_cast<const uint4 *>(mb + r * 128 + ((q ^ (r & 7)) << 4));
                bf16_chunk<NV>(wv, xs + kt * 64 + q * 8, K, acc);
            }
        } else {
            const int kq = tid >> 6;
#pragma unroll
            for (int cc = 0; cc < 2; cc++) {
                const int q = kq * 2 + cc;
                const uint4 wv = *reinterpret_cast<const uint4 *>(buf + r * 128 + ((q ^ (r & 7)) << 4));
                bf16_chunk<NV>(wv, xs + kt * 64 + q * 8, K, acc);
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvArgs a,
                                                        const __grid_constant__ CUtensorMap m1,
                                                        const __grid_constant__ CUtensorMap m3,
                                                        const __grid_constant__ CUtensorMap m2)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *bufs = smem;                                          // kStages * kStageBytes
    float *xs = reinterpret_cast<float *>(smem + kStages * kStageBytes);
    const int K = Geo<MODE>::k_of(a.d, a.f);
    float *red = xs + (size_t)kNT * K;                              // reduction scratch
    __shared__ uint64_t full[kStages];
    __shared__ int bail;

    if (*a.abort) return;
    const int rows = Geo<MODE>::rows_of(a.d, a.f);
    const int n_ri = rows / kItemRows;
    const int n_active = min(max(a.active[a.E], 0), a.E);
    const int n_items = (n_active + a.S) * n_ri;
    const int i_begin = (int)((long long)n_items * blockIdx.x / gridDim.x);
    const int i_end = (int)((long long)n_items * (blockIdx.x + 1) / gridDim.x);
    if (i_begin >= i_end) return;

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    __syncthreads();

    // producer cursor (thread 0)
    Cursor pc{i_begin, 0, 0};
    int produced = 0;
    auto groups_of = [&](const Unit &un) { return max(1, (un.ntok + kNT - 1) / kNT); };
    auto advance = [&](Cursor &c) {
        const Unit un = unit_of(a, n_active, c.item / n_ri);
        if (++c.kt == n_ktiles<MODE>(a, un.shared)) {
            c.kt = 0;
            if (++c.grp == groups_of(un)) {
                c.grp = 0;
                ++c.item;
            }
        }
    };
    auto produce = [&]() {
        if (pc.item >= i_end) return;
        const Unit un = unit_of(a, n_active, pc.item / n_ri);
        const int slot = produced % kStages;
        fence_proxy_async();
        issue_stage<MODE>(a, &m1, &m3, &m2, un, (pc.item % n_ri) * kItemRows, pc.kt,
                          bufs + slot * kStageBytes, &full[slot]);
        ++produced;
        advance(pc);
    };
    if (tid == 0)
        for (int s = 0; s < kStages; s++) produce();

    const int r = tid & (kItemRows - 1);
    int consumed = 0;
    int staged_unit = -1, staged_grp = -1, nvalid = 0;
    for (int item = i_begin; item < i_end; item++) {
        const int u = item / n_ri;
        const Unit un = unit_of(a, n_active, u);
        const int item_row = (item % n_ri) * kItemRows;
        const int ngrp = groups_of(un);
        for (int grp = 0; grp < ngrp; grp++) {
            if (staged_unit != u || staged_grp != grp) {
                __syncthreads();
                stage_x<MODE>(a, un, grp, xs, nvalid);
                staged_unit = u;
                staged_grp = grp;
                __syncthreads();
            }
            float acc[kNT];
#pragma unroll
            for (int i = 0; i < kNT; i++) acc[i] = 0.0f;
            const int nkt = n_ktiles<MODE>(a, un.shared);
            for (int kt = 0; kt < nkt; kt++) {
                const int slot = consumed % kStages;
                const uint32_t parity = (uint32_t)(consumed / kStages) & 1u;
                if (!mbar_wait(&full[slot], parity)) {
                    set_status(a.status, K3MOE_DEV_TIMEOUT);
                    bail = 1;
                }
                const uint8_t *buf = bufs + slot * kStageBytes;
                switch (nvalid) {
                case 1: consume_tile<MODE, 1>(buf, un.shared, kt, K, xs, acc); break;
                case 2: consume_tile<MODE, 2>(buf, un.shared, kt, K, xs, acc); break;
                case 3: consume_tile<MODE, 3>(buf, un.shared, kt, K, xs, acc); break;
                default: consume_tile<MODE, 4>(buf, un.shared, kt, K, xs, acc); break;
                }
                ++consumed;
                __syncthreads();                 // everyone is done with this slot
                if (tid == 0 && !bail) produce();
                if (bail) break;
            }
            if (bail) break;
            // reduce the K slices of each row and write the item's outputs
#pragma unroll
            for (int i = 0; i < kNT; i++) red[(size_t)i * kThreads + tid] = acc[i];
            __syncthreads();
            if (tid < kItemRows) {
                for (int i = 0; i < nvalid; i++) {
                    const float *ri = red + (size_t)i * kThreads;
                    const size_t orow = un.shared
                                            ? (size_t)a.T * a.k + (size_t)un.id * a.T + grp * kNT + i
                                            : (size_t)(un.tok0 + grp * kNT + i);
                    if (MODE == kGateUp) {
                        const float g = ri[tid] + ri[tid + 64];
                        const float uu = ri[tid + 128] + ri[tid + 192];
                        a.h[orow * a.f + item_row + tid] = situ(g, uu, a.b1, a.b2);
                    } else {
                        const float y = (ri[tid] + ri[tid + 64]) + (ri[tid + 128] + ri[tid + 192]);
                        a.ys[orow * a.d + item_row + tid] = y;
                    }
                }
            }
            // red is rewritten only after the next item's K loop, which has barriers
        }
        if (bail) break;
    }
    if (bail && tid == 0) {
        // let copies still in flight land before the block's shared memory is released
        for (int n = consumed; n < produced; n++) mbar_wait(&full[n % kStages], (uint32_t)(n / kStages) & 1u);
    }
}

// -------------------------------------------------------------------------------- combine
struct CombineArgs {
    int T, d, k, S;
    const float *weight;
    const int32_t *inv;
    const float *ys;
    float *out;
    const int32_t *abort;
};

__global__ void __launch_bounds__(256) fwd_combine_kernel(CombineArgs a)
{
    const int d4 = a.d / 4;
    const size_t n = (size_t)a.T * d4;
    const bool ab = *a.abort != 0;
    const int slots = a.T * a.k;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n;
         q += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(q / d4), c4 = (int)(q % d4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!ab) {
            for (int j = 0; j < a.k; j++) {
                const int p = a.inv[(size_t)t * a.k + j];
                if (p < 0 || p >= slots) continue;
                const float w = a.weight[(size_t)t * a.k + j];
                const float4 y = reinterpret_cast<const float4 *>(a.ys + (size_t)p * a.d)[c4];
                acc.x = fmaf(w, y.x, acc.x);
                acc.y = fmaf(w, y.y, acc.y);
                acc.z = fmaf(w, y.z, acc.z);
                acc.w = fmaf(w, y.w, acc.w);
            }
            for (int s = 0; s < a.S; s++) {
                const size_t row = (size_t)slots + (size_t)s * a.T + t;
                const float4 y = reinterpret_cast<const float4 *>(a.ys + row * a.d)[c4];
                acc.x += y.x;
                acc.y += y.y;
                acc.z += y.z;
                acc.w += y.w;
            }
        }
        reinterpret_cast<float4 *>(a.out + (size_t)t * a.d)[c4] = acc;
    }
}

// -------------------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// bf16 matrix [rows][cols] row-major; boxes of 64 cols x 64 rows, 128-byte swizzle.
bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64, kItemRows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count()
{
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

// Persistent grid: every SM filled to the occupancy the kernel's resources allow.
template <typename Kern>
int grid_blocks(Kern kernel, size_t smem)
{
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, smem) != cudaSuccess || occ < 1)
        occ = 1;
    return sm_count() * occ;
}

}  // namespace

cudaError_t launch_forward_gemv(const k3moe_config &c, int T, const uint16_t *x,
                                const int32_t *idx, const float *weight, const int32_t *offsets,
                                const int32_t *perm, const uint8_t *table, const uint16_t *sh_w1,
                                const uint16_t *sh_w3, const uint16_t *sh_w2, float *out,
                                uint8_t *ws, const WsLayout &L, cudaStream_t s)
{
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    int32_t *abort = status + 1;
    int32_t *active = reinterpret_cast<int32_t *>(ws + L.active);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    float *h = reinterpret_cast<float *>(ws + L.h);
    float *ys = reinterpret_cast<float *>(ws + L.ys);

    PrepArgs pa{T, c.n_experts, c.top_k, idx, offsets, perm, active, inv, status, abort};
    timing_begin("fwd_prep", s);
    fwd_prep_kernel<<<1, 1024, 0, s>>>(pa);
    count_launch();
    timing_end("fwd_prep", s);

    CUtensorMap m1{}, m3{}, m2{};
    if (c.n_shared > 0) {
        if (!make_bf16_map(&m1, sh_w1, (uint64_t)c.n_shared * c.f, c.d) ||
            !make_bf16_map(&m3, sh_w3, (uint64_t)c.n_shared * c.f, c.d) ||
            !make_bf16_map(&m2, sh_w2, (uint64_t)c.n_shared * c.d, c.f))
            return cudaErrorInvalidValue;
    }
    GemvArgs ga{T, c.d, c.f, c.top_k, c.n_shared, c.n_experts, c.situ_b1, c.situ_b2, x, offsets,
                perm, active, table, expert_bytes(c.d, c.f), gateup_block_bytes(c.d, c.f), h, ys,
                abort, status};
    {
        const size_t smem = 1024 + kStages * kStageBytes + (size_t)kNT * c.d * 4 + (size_t)kNT * kThreads * 4;
        cudaFuncSetAttribute(gemv_kernel<kGateUp>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const int blocks = grid_blocks(gemv_kernel<kGateUp>, smem);
        timing_begin("gemv_gateup", s);
        gemv_kernel<kGateUp><<<blocks, kThreads, smem, s>>>(ga, m1, m3, m2);
        count_launch();
        timing_end("gemv_gateup", s);
    }
    {
        const size_t smem = 1024 + kStages * kStageBytes + (size_t)kNT * c.f * 4 + (size_t)kNT * kThreads * 4;
        cudaFuncSetAttribute(gemv_kernel<kDown>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        const int blocks = grid_blocks(gemv_kernel<kDown>, smem);
        timing_begin("gemv_down", s);
        gemv_kernel<kDown><<<blocks, kThreads, smem, s>>>(ga, m1, m3, m2);
        count_launch();
        timing_end("gemv_down", s);
    }
    CombineArgs ca{T, c.d, c.top_k, c.n_shared, weight, inv, ys, out, abort};
    {
        const size_t n = (size_t)T * c.d / 4;
        int grid = (int)((n + 255) / 256);
        if (grid > sm_count() * 8) grid = sm_count() * 8;
        if (grid < 1) grid = 1;
        timing_begin("fwd_combine", s);
        fwd_combine_kernel<<<grid, 256, 0, s>>>(ca);
        count_launch();
        timing_end("fwd_combine", s);
    }
    return cudaGetLastError();
}

}  // namespace k3moe
