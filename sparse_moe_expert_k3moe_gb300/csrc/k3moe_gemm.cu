// k3moe_gemm.cu -- the expert part of the layer as grouped tensor-core GEMMs: the
// prefill path (many tokens per expert).  Same mathematics as the decode path
// (kimi-k3-in-c README, Part II, section 4 for the MXFP4 format, section 9 for the
// expert loop and SiTU-GLU); here the weights are the 128-row M side of tcgen05 MMAs
// ("swap AB"), an expert's tokens the N side, so an expert with few tokens still fills
// the 128-row tile.
//
// Kernels, in launch order:
//   gemm_units   validates offsets, lists the units (shared experts first, heaviest,
//                then the active routed experts) and the prefix of their work items;
//   gemm_scales  per-token activation scale 2^-u (max |x_t| in [2^14, 2^15));
//   gemm_gather  routed-expert activations in perm order, f16, times 2^-u_t; validates
//                perm against idx;
//   gemm<GU>     g = W1 x, u = W3 x; h = SiTU(g, u) written as f16 (routed) / bf16
//                (shared) rows;
//   gemm<DN>     y = W2 h; out[t] += w_slot * y (routed) or += y (shared) with fp32
//                atomics onto out (zeroed first).
//
// One work item = 128 weight rows of one unit x up to 128 (gate/up) or 256 (down) of its
// tokens x the whole K.  Warp roles in a block (one block per SM):
//   warp 0       producer: TMA 2-D loads of the B tiles (64 columns x 16 rows per copy)
//                and, for bf16 shared experts, of the A tiles;
//   warp 1       MMA: one thread issues tcgen05.mma (kind::f16, M=128, N=tile, K=16)
//                into fp32 accumulators in tensor memory, two buffers of 256 columns
//                (gate/up: g at +0, u at +128), so one item's MMAs overlap the previous
//                item's epilogue;
//   warps 2-9    dequant: packed MXFP4 tiles from shared memory to f16 A tiles
//                (128-byte swizzle, K-major) -- the E2M1 pair decoded by the hardware
//                conversion, times 2^(b - bmax + 13) where bmax is the largest scale of
//                the 128-row block (the packed table's trailer), so every value is exact
//                in f16 while the block's scales span at most 36 binades; the epilogue
//                multiplies by 2^(bmax - 140);
//   warps 10-13  epilogue: tcgen05.ld the accumulators (warp w reads lanes 32(w%4)..),
//                apply the scales, SiTU or the weighted combine, store;
//   warp 14      packed-weight producer: one bulk copy per 128-column packed tile (pair),
//                kStgP tiles ahead of the dequant warps.
// Rings: packed tiles (kStgP), f16 A stages (kStgA) and B stages (kStgB); the MMA thread
// releases an A and a B stage with one tcgen05.commit each.
// Every wait is bounded by a clock limit; a timeout sets the status word and the
// roles drop out.
#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "k3moe_internal.cuh"
#include "k3moe_tc.cuh"

namespace k3moe {
namespace {

constexpr int kBM = 128, kBK = 64;
constexpr int kStgP = 3, kStgA = 2, kStgB = 3;               // packed, A and B rings
constexpr int kNumDq = 8;
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpDq0 = 2, kWarpEpi0 = 2 + kNumDq, kNumEpi = 4;
constexpr int kWarpPack = kWarpEpi0 + kNumEpi;                 // 14
constexpr int kGemmThreads = (kWarpPack + 1) * 32;             // 480
constexpr int kTmemCols = 512;

enum { kGU = 0, kDN = 1 };

template <int MODE>
struct GG {
    static constexpr int kMats = MODE == kGU ? 2 : 1;
    // tokens per tile: gate/up keeps two accumulators (g, u) per buffer, so 128 tokens
    // fit twice in the 512 TMEM columns; down keeps one
    static constexpr int kBNMax = MODE == kGU ? 128 : 256;
    static constexpr int kPBytes = kMats * kTileBytes;         // packed tile (pair) of 128 columns
    static constexpr int kABytes = kMats * kBM * kBK * 2;      // f16/bf16 A tiles of a stage
    static constexpr int kBBytes = kBNMax * kBK * 2;           // B tile of a stage
    static constexpr int kSmem = kStgP * kPBytes + kStgA * kABytes + kStgB * kBBytes + 2048;
};

__device__ __forceinline__ uint32_t e2m1x2_f16x2(uint32_t byte)
{
    uint32_t h;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(h) : "r"(byte));
    return h;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<__half2 *>(&a), *reinterpret_cast<__half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ float situ(float g, float u, float b1, float b2)
{
    const float a = b1 * tanhf(g / b1) * (1.0f / (1.0f + expf(-g)));
    return a * (b2 * tanhf(u / b2));
}
// f16 of 2^e for e in [-24, 15] (subnormals below -14), 0 outside.
__device__ __forceinline__ uint32_t f16_pow2(int e)
{
    if (e > 15 || e < -24) return 0u;
    if (e >= -14) return (uint32_t)(e + 15) << 10;
    return 1u << (e + 24);
}

// ---------------------------------------------------------------------------------- units
struct UnitsArgs {
    int T, E, k, S, rb_gu, rb_dn;
    const int32_t *offsets;
    int32_t *units;          // [E + S][4]: shared flag, id, tok0, ntok
    int32_t *prefix_gu;      // [E + S + 1]
    int32_t *prefix_dn;      // [E + S + 1]
    int32_t *n_units;
    int32_t *status, *abort;
};

__global__ void __launch_bounds__(1024) gemm_units_kernel(UnitsArgs a)
{
    __shared__ int32_t bad, scan_tmp[32], base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, slots = a.T * a.k;
    if (tid == 0) { bad = 0; base = a.S; }
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        const int lo = a.offsets[e], hi = a.offsets[e + 1];
        if (lo < 0 || hi < lo || hi > slots) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    }
    if (tid == 0 && (a.offsets[0] != 0 || a.offsets[E] != slots)) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    __syncthreads();
    const bool ok = bad == 0;
    if (tid < a.S) {
        int32_t *u = a.units + 4 * tid;
        u[0] = 1; u[1] = tid; u[2] = 0; u[3] = a.T;
    }
    // active routed experts after the shared units, ascending (block scan of flags)
    for (int b0 = 0; b0 < E; b0 += blockDim.x) {
        const int e = b0 + tid;
        const int flag = (ok && e < E && a.offsets[e + 1] > a.offsets[e]) ? 1 : 0;
        const uint32_t bal = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) scan_tmp[warp] = __popc(bal);
        __syncthreads();
        int before = base;
        for (int w = 0; w < warp; w++) before += scan_tmp[w];
        if (flag) {
            int32_t *u = a.units + 4 * (before + __popc(bal & ((1u << lane) - 1u)));
            u[0] = 0; u[1] = e; u[2] = a.offsets[e]; u[3] = a.offsets[e + 1] - a.offsets[e];
        }
        __syncthreads();
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < (int)(blockDim.x >> 5); w++) tot += scan_tmp[w];
            base += tot;
        }
        __syncthreads();
    }
    // item prefix (one thread: at most E + S units)
    if (tid == 0) {
        const int n = base;
        *a.n_units = n;
        int pg = 0, pd = 0;
        for (int u = 0; u < n; u++) {
            a.prefix_gu[u] = pg;
            a.prefix_dn[u] = pd;
            const int ntok = a.units[4 * u + 3];
            pg += (ntok + GG<kGU>::kBNMax - 1) / GG<kGU>::kBNMax * a.rb_gu;
            pd += (ntok + GG<kDN>::kBNMax - 1) / GG<kDN>::kBNMax * a.rb_dn;
        }
        a.prefix_gu[n] = pg;
        a.prefix_dn[n] = pd;
        if (bad) atomicOr(a.status, bad);
        *a.abort = bad ? 1 : 0;
    }
}

// per-token activation scale 2^-u with max|x_t| * 2^-u in [2^14, 2^15), u in [-113, 113]
__global__ void __launch_bounds__(256) gemm_scales_kernel(int T, int d, const uint16_t *x, float *tok_scale)
{
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= T) return;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)warp * d);
    uint32_t m = 0;
    for (int q = lane; q < d / 8; q += 32) {
        const uint4 v = row[q];
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; h++) m = max(m, max(w4[h] & 0x7FFFu, (w4[h] >> 16) & 0x7FFFu));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
        int u = 0;
        const int eb = (int)(m >> 7);
        if (m != 0 && eb < 255) u = min(max(eb - 127 - 14, -113), 113);
        tok_scale[warp] = __uint_as_float((uint32_t)(127 - u) << 23);
        tok_scale[T + warp] = __uint_as_float((uint32_t)(127 + u) << 23);
    }
}

// xg[p] = f16(x[token(p)] * 2^-u) for every routed position p; validates perm.
struct GatherArgs {
    int T, d, k, E;
    const uint16_t *x;
    const int32_t *idx, *offsets, *perm;
    const float *tok_scale;
    uint16_t *xg;
    int32_t *status, *abort;
};
__global__ void __launch_bounds__(256) gemm_gather_kernel(GatherArgs a)
{
    const int slots = a.T * a.k, d8 = a.d / 8;
    const bool ok_off = *a.abort == 0;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < (size_t)slots * d8;
         q += (size_t)gridDim.x * blockDim.x) {
        const int p = (int)(q / d8), c = (int)(q % d8);
        int s = a.perm[p];
        if (c == 0) {
            bool bad = s < 0 || s >= slots;
            if (!bad && ok_off) {
                int lo = 0, hi = a.E;
                while (hi - lo > 1) {
                    const int mid = (lo + hi) >> 1;
                    if (a.offsets[mid] <= p) lo = mid; else hi = mid;
                }
                if (a.idx[s] != lo) bad = true;
            }
            if (bad) {
                set_status(a.status, K3MOE_DEV_BAD_OFFSETS);
                atomicOr(a.abort, 1);
            }
        }
        s = min(max(s, 0), slots - 1);
        const int t = s / a.k;
        const float m = a.tok_scale[t];
        const uint4 v = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.d)[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const __half2 h2 = __floats2half2_rn(__uint_as_float(w[h] << 16) * m,
                                                 __uint_as_float(w[h] & 0xFFFF0000u) * m);
            o[h] = *reinterpret_cast<const uint32_t *>(&h2);
        }
        reinterpret_cast<uint4 *>(a.xg + (size_t)p * a.d)[c] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ---------------------------------------------------------------------------------- GEMM
struct GemmArgs {
    int T, d, f, k, S, E;
    float b1, b2;
    const int32_t *units, *prefix, *n_units;
    const int32_t *perm;
    const float *weight, *tok_scale;
    const uint8_t *table;
    size_t expert_bytes, gateup_bytes;
    uint16_t *hp;                   // h rows (routed f16, shared bf16)
    float *out;
    const int32_t *abort;
    int32_t *status;
};

struct GItem {
    int shared, id, tok0, ntok;     // unit
    int rb, n0, ncols, bn;          // row block, first column, valid columns, MMA N
};

template <int MODE>
__device__ __forceinline__ int rows_of(const GemmArgs &a) { return MODE == kGU ? a.f : a.d; }
template <int MODE>
__device__ __forceinline__ int k_of(const GemmArgs &a) { return MODE == kGU ? a.d : a.f; }

template <int MODE>
__device__ __forceinline__ GItem gitem(const GemmArgs &a, int n_units, int i)
{
    int lo = 0, hi = n_units;                      // unit u with prefix[u] <= i < prefix[u+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.prefix[mid] <= i) lo = mid; else hi = mid;
    }
    const int32_t *u = a.units + 4 * lo;
    GItem it;
    it.shared = u[0];
    it.id = u[1];
    it.tok0 = u[2];
    it.ntok = u[3];
    constexpr int BN = GG<MODE>::kBNMax;
    const int ntiles = max(1, (it.ntok + BN - 1) / BN);
    const int j = i - a.prefix[lo];
    const int nt = j % ntiles;                     // token tile fastest: the block's weights stay hot in L2
    it.rb = j / ntiles;
    it.n0 = nt * BN;
    it.ncols = min(BN, it.ntok - it.n0);
    it.bn = (it.ncols + 15) & ~15;
    return it;
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs a,
                                                                const __grid_constant__ CUtensorMap mb_routed,
                                                                const __grid_constant__ CUtensorMap mb_shared,
                                                                const __grid_constant__ CUtensorMap ma1,
                                                                const __grid_constant__ CUtensorMap ma3)
{
    extern __shared__ __align__(1024) uint8_t gsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int kMats = GG<MODE>::kMats;
    constexpr int kPBytes = GG<MODE>::kPBytes, kABytes = GG<MODE>::kABytes, kBBytes = GG<MODE>::kBBytes;
    uint8_t *smA = sm;                                   // kStgA x kABytes (1024-aligned)
    uint8_t *smB = smA + kStgA * kABytes;                // kStgB x kBBytes
    uint8_t *smP = smB + kStgB * kBBytes;                // kStgP x kPBytes
    __shared__ uint64_t full_p[kStgP], empty_p[kStgP], full_a[kStgA], empty_a[kStgA], full_b[kStgB],
        empty_b[kStgB], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int bail;

    if (*a.abort) return;
    const int n_units = *a.n_units;
    const int n_items = a.prefix[n_units];
    if ((int)blockIdx.x >= n_items) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = k_of<MODE>(a), nks = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStgP; s++) { mb_init(&full_p[s], 1); mb_init(&empty_p[s], kNumDq); }
        for (int s = 0; s < kStgA; s++) { mb_init(&full_a[s], kNumDq); mb_init(&empty_a[s], 1); }
        for (int s = 0; s < kStgB; s++) { mb_init(&full_b[s], 1); mb_init(&empty_b[s], 1); }
        for (int b = 0; b < 2; b++) { mb_init(&acc_full[b], 1); mb_init(&acc_empty[b], kNumEpi); }
        mb_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    auto timeout = [&]() {
        set_status(a.status, K3MOE_DEV_TIMEOUT);
        bail = 1;
    };
    // a stage counter st of a ring of depth D: slot st % D, fill number st / D
    auto wait_free = [&](uint64_t *bars, int D, uint32_t st) -> bool {
        return st < (uint32_t)D || mb_wait(&bars[st % D], ((st / D) - 1) & 1u);
    };
    // after a timeout: wait (bounded) for the copies of the last D fills of a ring
    auto drain_fills = [&](uint64_t *bars, int D, uint32_t n) {
        for (uint32_t f = n > (uint32_t)D ? n - D : 0; f < n; f++) mb_wait(&bars[f % D], (f / D) & 1u);
    };

    if (warp == kWarpPack) {
        // ------------------------------------------------------------ packed-weight producer
        if (lane == 0) {
            uint32_t cp = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x) {
                const GItem it = gitem<MODE>(a, n_units, i);
                if (it.shared) continue;
                const uint8_t *ex = a.table + (size_t)it.id * a.expert_bytes;
                for (int kt = 0; kt < K / kTileK; kt++, cp++) {
                    if (!wait_free(empty_p, kStgP, cp)) { timeout(); break; }
                    const int sp = cp % kStgP;
                    const uint8_t *src = MODE == kGU ? ex + ((size_t)it.rb * (a.d / kTileK) + kt) * 2 * kTileBytes
                                                     : ex + a.gateup_bytes + ((size_t)it.rb * (a.f / kTileK) + kt) * kTileBytes;
                    mb_expect_tx(&full_p[sp], (uint32_t)kPBytes);
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                            saddr(smP + sp * kPBytes)),
                        "l"(src), "r"((uint32_t)kPBytes), "r"(saddr(&full_p[sp]))
                        : "memory");
                }
            }
            if (bail) drain_fills(full_p, kStgP, cp);
        }
    } else if (warp == kWarpProd) {
        // ------------------------------------------------------------ B (and bf16 A) producer
        if (lane == 0) {
            uint32_t sa = 0, sb = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x) {
                const GItem it = gitem<MODE>(a, n_units, i);
                int brow0;
                const CUtensorMap *mb = &mb_routed;
                if (MODE == kGU) {
                    if (it.shared) { mb = &mb_shared; brow0 = it.n0; }
                    else brow0 = it.tok0 + it.n0;
                } else {
                    brow0 = it.shared ? a.T * a.k + it.id * a.T + it.n0 : it.tok0 + it.n0;
                }
                for (int ks = 0; ks < nks; ks++, sa++, sb++) {
                    if (!wait_free(empty_b, kStgB, sb) || (it.shared && !wait_free(empty_a, kStgA, sa))) {
                        timeout();
                        break;
                    }
                    uint8_t *B = smB + (sb % kStgB) * kBBytes;
                    uint64_t *fb = &full_b[sb % kStgB];
                    // the bf16 A tiles of a shared expert land on the B barrier too
                    mb_expect_tx(fb, (uint32_t)it.bn * kBK * 2 + (it.shared ? (uint32_t)kABytes : 0u));
                    for (int j = 0; j < it.bn / 16; j++) tma2d(B + j * 16 * 128, mb, ks * kBK, brow0 + 16 * j, fb);
                    if (it.shared) {
                        uint8_t *A = smA + (sa % kStgA) * kABytes;
                        const int arow = it.id * rows_of<MODE>(a) + it.rb * kBM;
                        tma2d(A, &ma1, ks * kBK, arow, fb);
                        if (MODE == kGU) tma2d(A + kBM * kBK * 2, &ma3, ks * kBK, arow, fb);
                    }
                }
            }
            if (bail) drain_fills(full_b, kStgB, sb);
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            uint32_t sa = 0, sb = 0, n = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
                const GItem it = gitem<MODE>(a, n_units, i);
                const uint32_t id = idesc(it.shared ? 1 : 0, it.bn);
                const int buf = n & 1;
                if (n >= 2 && !mb_wait(&acc_empty[buf], ((n >> 1) - 1) & 1u)) { timeout(); break; }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)buf * 256u;
                for (int ks = 0; ks < nks; ks++, sa++, sb++) {
                    if (!mb_wait(&full_a[sa % kStgA], (sa / kStgA) & 1u) ||
                        !mb_wait(&full_b[sb % kStgB], (sb / kStgB) & 1u)) { timeout(); break; }
                    tc_fence_after();
                    const uint32_t A = saddr(smA + (sa % kStgA) * kABytes), B = saddr(smB + (sb % kStgB) * kBBytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; kk++) {
                        const uint64_t bd = sdesc(B + kk * 32);
                        const uint32_t accum = (ks | kk) != 0;
                        umma(d0, sdesc(A + kk * 32), bd, id, accum);
                        if (MODE == kGU) umma(d0 + 128, sdesc(A + kBM * kBK * 2 + kk * 32), bd, id, accum);
                    }
                    umma_commit(&empty_a[sa % kStgA]);
                    umma_commit(&empty_b[sb % kStgB]);
                }
                if (bail) break;
                umma_commit(&acc_full[buf]);
            }
            umma_commit(&drain);                       // every issued MMA done before the dealloc
            mb_wait(&drain, 0);
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------------ dequant (packed smem -> f16 A)
        const int t = threadIdx.x - kWarpDq0 * 32;             // 0..255
        const int m = (MODE == kGU) ? (t >> 7) : 0;
        const bool active = (MODE == kGU) || t < 128;
        const int r7 = t & 127, strip = r7 >> 4, gsel = (r7 >> 3) & 1, g = r7 & 7;
        uint32_t sa = 0, cp = 0;
        for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x) {
            const GItem it = gitem<MODE>(a, n_units, i);
            int bmax = 0;
            if (!it.shared && active) {
                const int mm = MODE == kGU ? m : 2;
                bmax = (int)*reinterpret_cast<const uint32_t *>(
                    a.table + trailer_offset(a.E, a.d, a.f, it.id, mm, it.rb));
            }
            for (int ks = 0; ks < nks; ks++, sa++) {
                if (!it.shared && (ks & 1) == 0 && !mb_wait(&full_p[cp % kStgP], (cp / kStgP) & 1u)) { timeout(); break; }
                if (!wait_free(empty_a, kStgA, sa)) { timeout(); break; }
                if (!it.shared && active) {
                    const int c = 2 * (ks & 1) + gsel;
                    const uint8_t *tile = smP + (cp % kStgP) * kPBytes + m * kTileBytes;
                    const uint4 *src = reinterpret_cast<const uint4 *>(tile + (strip * 4 + c) * 256 + 32 * g);
                    const uint4 p0 = src[0], p1 = src[1];
                    const uint32_t w[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                    uint8_t *A = smA + (sa % kStgA) * kABytes + m * (kBM * kBK * 2);
#pragma unroll
                    for (int hr = 0; hr < 2; hr++) {            // rows g and g+8 of the strip
                        const int r = strip * 16 + g + 8 * hr;
                        const uint32_t b = tile[kTileNibbleBytes + r * 4 + c];
                        const uint32_t s1 = b == 255u ? 0u : f16_pow2((int)b - bmax + 13);
                        const uint32_t s2 = s1 | (s1 << 16);
#pragma unroll
                        for (int j = 0; j < 4; j++) {           // 8 columns per 16-byte store
                            uint32_t v[4];
#pragma unroll
                            for (int tt = 0; tt < 4; tt++)
                                v[tt] = hmul2(e2m1x2_f16x2(w[2 * tt + hr] >> (8 * j)), s2);
                            const int chunk = 4 * gsel + j;
                            *reinterpret_cast<uint4 *>(A + r * 128 + ((chunk ^ (r & 7)) << 4)) =
                                make_uint4(v[0], v[1], v[2], v[3]);
                        }
                    }
                    fence_async_smem();
                }
                __syncwarp();
                if (lane == 0) {
                    mb_arrive(&full_a[sa % kStgA]);
                    if (!it.shared && (ks & 1)) mb_arrive(&empty_p[cp % kStgP]);
                }
                if (!it.shared && (ks & 1)) cp++;
            }
        }
    } else if (warp < kWarpPack) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                                 // TMEM lane quadrant
        const int row = 32 * q + lane;
        uint32_t n = 0;
        for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
            const GItem it = gitem<MODE>(a, n_units, i);
            const int buf = n & 1;
            float f1 = 1.0f, f3 = 1.0f;
            if (!it.shared) {
                const int mm1 = MODE == kGU ? 0 : 2;
                f1 = ldexpf(1.0f, (int)*reinterpret_cast<const uint32_t *>(
                                      a.table + trailer_offset(a.E, a.d, a.f, it.id, mm1, it.rb)) - 140);
                if (MODE == kGU)
                    f3 = ldexpf(1.0f, (int)*reinterpret_cast<const uint32_t *>(
                                          a.table + trailer_offset(a.E, a.d, a.f, it.id, 1, it.rb)) - 140);
            }
            if (!mb_wait(&acc_full[buf], (n >> 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            const int grow = it.rb * kBM + row;
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 256u;
            for (int c0 = 0; c0 < it.bn; c0 += 16) {
                float vg[16], vu[16];
                tmem_ld16(lane_addr + c0, vg);
                if (MODE == kGU) tmem_ld16(lane_addr + 128 + c0, vu);
#pragma unroll
                for (int jj = 0; jj < 16; jj++) {
                    const int col = c0 + jj;
                    if (col >= it.ncols) break;
                    if (MODE == kGU) {
                        size_t hrow;
                        float fo = 1.0f;
                        if (it.shared) {
                            hrow = (size_t)a.T * a.k + (size_t)it.id * a.T + it.n0 + col;
                        } else {
                            const int p = it.tok0 + it.n0 + col;
                            hrow = (size_t)p;
                            const int slot = min(max(a.perm[p], 0), a.T * a.k - 1);
                            fo = a.tok_scale[a.T + slot / a.k];
                        }
                        const float h = situ(vg[jj] * f1 * fo, vu[jj] * f3 * fo, a.b1, a.b2);
                        uint16_t hv;
                        if (it.shared) {
                            const __nv_bfloat16 hb = __float2bfloat16_rn(h);
                            hv = *reinterpret_cast<const uint16_t *>(&hb);
                        } else {
                            const __half hh = __float2half_rn(h);
                            hv = *reinterpret_cast<const uint16_t *>(&hh);
                        }
                        a.hp[hrow * a.f + grow] = hv;
                    } else {
                        int t;
                        float wt = 1.0f;
                        if (it.shared) {
                            t = it.n0 + col;
                        } else {
                            const int p = it.tok0 + it.n0 + col;
                            const int slot = min(max(a.perm[p], 0), a.T * a.k - 1);
                            t = slot / a.k;
                            wt = a.weight[slot];
                        }
                        atomicAdd(a.out + (size_t)t * a.d + grow, wt * (vg[jj] * f1));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&acc_empty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

// ---------------------------------------------------------------------------------- host
template <int MODE>
cudaError_t launch_gemm(const GemmArgs &ga, const CUtensorMap &mbr, const CUtensorMap &mbs,
                        const CUtensorMap &ma1, const CUtensorMap &ma3, int max_items, cudaStream_t s,
                        const char *name)
{
    static bool set = false;
    if (!set) {
        cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, GG<MODE>::kSmem);
        set = true;
    }
    const int grid = max(1, min(num_sms(), max_items));
    timing_begin(name, s);
    gemm_kernel<MODE><<<grid, kGemmThreads, GG<MODE>::kSmem, s>>>(ga, mbr, mbs, ma1, ma3);
    count_launch();
    timing_end(name, s);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_forward_gemm(const k3moe_config &c, int T, const uint16_t *x, const int32_t *idx,
                                const float *weight, const int32_t *offsets, const int32_t *perm,
                                const uint8_t *table, const uint16_t *sh_w1, const uint16_t *sh_w3,
                                const uint16_t *sh_w2, float *out, uint8_t *ws, const WsLayout &L,
                                cudaStream_t s)
{
    const int E = c.n_experts, k = c.top_k, S = c.n_shared;
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    int32_t *abort = status + 1;
    int32_t *units = reinterpret_cast<int32_t *>(ws + L.units);
    int32_t *prefix_gu = units + 4 * (E + S);
    int32_t *prefix_dn = prefix_gu + (E + S + 1);
    int32_t *n_units = prefix_dn + (E + S + 1);
    float *tok_scale = reinterpret_cast<float *>(ws + L.tok_scale);
    uint16_t *xg = reinterpret_cast<uint16_t *>(ws + L.xg);
    uint16_t *hp = reinterpret_cast<uint16_t *>(ws + L.hp);
    const size_t rows_all = (size_t)T * k + (size_t)S * T;

    cudaError_t err = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)T * c.d, s);
    if (err != cudaSuccess) return err;
    UnitsArgs ua{T, E, k, S, c.f / kBM, c.d / kBM, offsets, units, prefix_gu, prefix_dn, n_units, status, abort};
    timing_begin("gemm_units", s);
    gemm_units_kernel<<<1, 1024, 0, s>>>(ua);
    count_launch();
    timing_end("gemm_units", s);
    timing_begin("gemm_scales", s);
    gemm_scales_kernel<<<(T * 32 + 255) / 256, 256, 0, s>>>(T, c.d, x, tok_scale);
    count_launch();
    timing_end("gemm_scales", s);
    GatherArgs gta{T, c.d, k, E, x, idx, offsets, perm, tok_scale, xg, status, abort};
    {
        const size_t work = (size_t)T * k * (c.d / 8);
        int grid = (int)std::min<size_t>((work + 255) / 256, (size_t)num_sms() * 16);
        timing_begin("gemm_gather", s);
        gemm_gather_kernel<<<std::max(grid, 1), 256, 0, s>>>(gta);
        count_launch();
        timing_end("gemm_gather", s);
    }

    CUtensorMap mb_routed{}, mb_shared{}, ma1{}, ma3{}, mb_h{}, ma2{};
    bool ok = map16(&mb_routed, xg, (uint64_t)T * k, c.d, 16) && map16(&mb_h, hp, rows_all, c.f, 16);
    if (S > 0)
        ok = ok && map16(&mb_shared, x, (uint64_t)T, c.d, 16) &&
             map16(&ma1, sh_w1, (uint64_t)S * c.f, c.d, kBM) && map16(&ma3, sh_w3, (uint64_t)S * c.f, c.d, kBM) &&
             map16(&ma2, sh_w2, (uint64_t)S * c.d, c.f, kBM);
    if (!ok) return cudaErrorInvalidValue;

    GemmArgs ga{T, c.d, c.f, k, S, E, c.situ_b1, c.situ_b2, units, prefix_gu, n_units, perm, weight,
                tok_scale, table, expert_bytes(c.d, c.f), gateup_block_bytes(c.d, c.f), hp, out, abort, status};
    // an upper bound on the items: every slot its own expert
    const int max_tiles = (int)std::min<long long>((long long)T * k + (long long)(E + S), (long long)1 << 30);
    err = launch_gemm<kGU>(ga, mb_routed, mb_shared, ma1, ma3, max_tiles * (c.f / kBM), s, "gemm_gateup");
    if (err != cudaSuccess) return err;
    GemmArgs gd = ga;
    gd.prefix = prefix_dn;
    err = launch_gemm<kDN>(gd, mb_h, mb_h, ma2, ma2, max_tiles * (c.d / kBM), s, "gemm_down");
    return err;
}

}  // namespace k3moe
