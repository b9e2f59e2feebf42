// k3moe_gemm.cu -- the expert part of the layer as grouped tensor-core GEMMs: the
// prefill path (many tokens per expert).  Same mathematics as the decode path
// (kimi-k3-in-c README, Part II, section 4 for the MXFP4 format, section 9 for the
// expert loop and SiTU-GLU).  An expert's tokens are the 128-row M side of the tcgen05
// MMAs and its dequantised weight rows the 256-wide N side: an MMA instruction costs
// about the same whatever its N, so only N = 256 runs at the tensor rate.
//
// Two variants, chosen per call by k3moe_set_prefill_gemm.  The block-scaled one (the
// default) is at the end of this file (gemm_gather_mx, gemm_mx_kernel); it runs the
// shared experts on the f16 kernels below, restricted to their items.  The f16 variant,
// in launch order:
//   gemm_units   validates offsets, lists the units (shared experts first, heaviest,
//                then the active routed experts) and the prefix of their work items;
//   gemm_scales  per-token activation scale 2^-u (max |x_t| in [2^14, 2^15));
//   gemm_gather  zeroes out; routed-expert activations in perm order, f16, times
//                2^-u_t; validates perm against idx;
//   gemm<GU>     g = W1 x, u = W3 x; h = SiTU(g, u) written as f16 (routed) / bf16
//                (shared) rows;
//   gemm<DN>     y = W2 h; out[t] += w_slot * y (routed) or += y (shared) with fp32
//                atomics onto out (zeroed by gemm_gather).
// Every kernel starts with pdl_wait(), so each is launched with programmatic dependent
// launch and its launch overlaps the previous kernel.
//
// One work item = 128 tokens of one unit (the MMA M side) x 256 weight rows (N: gate/up
// the 128-row blocks of W1 and W3 for one block of f, down two 128-row blocks of W2)
// x the whole K.  Warp roles in a block (one block per SM):
//   warp 0       producer: TMA 2-D loads of the token tiles (64 columns x 128 rows) and,
//                for bf16 shared experts, of the weight tiles; also the L2 prefetch of the
//                packed weight tiles, kL2Ahead tiles ahead;
//   warp 1       MMA: one thread issues tcgen05.mma (kind::f16, M=128, N=256, K=16) into
//                fp32 accumulators in tensor memory, two buffers of 256 columns, so one
//                item's MMAs overlap the previous item's epilogue;
//   warps 2-17   dequant: packed MXFP4 tiles, loaded from global memory into registers
//                two tiles ahead, to f16 weight tiles in shared memory (128-byte
//                swizzle, K-major) -- the E2M1 pair decoded by the hardware
//                conversion, times 2^(b - bmax + 13) where bmax is the largest scale of
//                the 128-row block (the packed table's trailer), so every value is exact
//                in f16 while the block's scales span at most 36 binades; the epilogue
//                multiplies by 2^(bmax - 140);
//   warps 18-21  epilogue, one token per thread (warp w reads TMEM lanes 32(w%4)..):
//                gate/up SiTU to h rows, down the weighted combine as float4 atomics.
// Ring: kStg stages of one token tile and one weight tile, each stage with one full barrier (TMA bytes + an arrive per dequant warp) and one
// empty barrier (the MMA thread's tcgen05.commit).
// Every wait is bounded by a clock limit; a timeout sets the status word and the
// roles drop out.
#include <cuda.h>
#include <cuda_bf16.h>

#include <climits>
#include <mutex>

#include "k3moe_internal.cuh"
#include "k3moe_tc.cuh"

namespace k3moe {
namespace {

constexpr int kBM = 128, kBK = 64;          // token rows per tile (MMA M), K per stage
constexpr int kWRows = 256;                 // weight rows per item (MMA N): W1|W3, or two W2 blocks
constexpr int kStg = 4;                     // stage ring (token + weight tiles)
constexpr int kL2Ahead = 6;                 // packed tiles prefetched into L2 ahead of the token producer
constexpr int kNumDq = 16;
constexpr int kWarpProd = 0, kWarpMma = 1, kWarpDq0 = 2, kWarpEpi0 = 2 + kNumDq, kNumEpi = 4;
constexpr int kGemmThreads = (kWarpEpi0 + kNumEpi) * 32;       // 704
constexpr int kTmemCols = 512;
constexpr int kABytes = kBM * kBK * 2;                          // token tile of a stage
constexpr int kWBytes = kWRows * kBK * 2;                       // weight tile of a stage
constexpr int kGemmSmem = kStg * (kABytes + kWBytes) + 2048;
static_assert(kGemmSmem + 8 * 1024 <= 232448, "shared memory per block (dynamic + static)");

enum { kGU = 0, kDN = 1 };

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
// tanh(x) = 1 - 2 / (e^(2x) + 1) with the fast exponential; |x| clamped to 15, where
// tanh is 1 to float precision.  Absolute error a few ulp of 1.
__device__ __forceinline__ float tanh_fast(float x)
{
    x = fminf(fmaxf(x, -15.0f), 15.0f);
    return 1.0f - __fdividef(2.0f, __expf(2.0f * x) + 1.0f);
}
// SiTU of the GEMM epilogue: b1 tanh(g/b1) sigmoid(g) b2 tanh(u/b2) with the fast
// exponential.  Its error (a few 1e-7 relative to the gate and linear caps) is far
// below the f16 / bf16 rounding of h that follows.
__device__ __forceinline__ float situ(float g, float u, float b1, float b2)
{
    const float sg = __fdividef(1.0f, 1.0f + __expf(-fminf(fmaxf(g, -80.0f), 80.0f)));
    return b1 * tanh_fast(__fdividef(g, b1)) * sg * (b2 * tanh_fast(__fdividef(u, b2)));
}
// SiTU of the block-scaled GEMM's epilogue, whose h is split into two e4m3 terms (about
// 8 significant bits, 2^-9 relative): the two caps by the hardware tanh approximation
// (tanh.approx.f32, relative error about 2^-11), the sigmoid by the fast exponential and
// reciprocal; ib1 = 1/b1, ib2 = 1/b2.
__device__ __forceinline__ float tanh_approx(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float situ_mx(float g, float u, float b1, float b2, float ib1, float ib2)
{
    const float sg = __fdividef(1.0f, 1.0f + __expf(-g));
    return b1 * tanh_approx(g * ib1) * sg * (b2 * tanh_approx(u * ib2));
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

// One block: validates offsets, lists the units (shared experts first, then the active
// routed experts ascending) and their item prefixes.  A unit's items start after every
// earlier unit's token tiles times the row blocks per tile, so the prefixes come from a
// block scan of the tile counts, done in the same pass as the scan of the active flags.
__global__ void __launch_bounds__(1024) gemm_units_kernel(UnitsArgs a)
{
    pdl_wait();
    pdl_trigger();
    __shared__ int32_t bad, scan_n[32], scan_t[32], base, tbase;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = (int)(blockDim.x >> 5);
    const int E = a.E, slots = a.T * a.k;
    const int ntS = (a.T + kBM - 1) / kBM;             // token tiles of a shared unit
    if (tid == 0) { bad = 0; base = a.S; tbase = a.S * ntS; }
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
        a.prefix_gu[tid] = tid * ntS * a.rb_gu;
        a.prefix_dn[tid] = tid * ntS * a.rb_dn;
    }
    // active routed experts after the shared units, ascending (block scans of the flags
    // and of the token tiles)
    for (int b0 = 0; b0 < E; b0 += blockDim.x) {
        const int e = b0 + tid;
        const int lo = ok && e < E ? a.offsets[e] : 0;
        const int cnt = ok && e < E ? a.offsets[e + 1] - lo : 0;
        const int flag = cnt > 0 ? 1 : 0;
        const int nt = (cnt + kBM - 1) / kBM;
        const uint32_t bal = __ballot_sync(0xffffffffu, flag);
        int incl = nt;                                  // inclusive warp scan of the tiles
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) { scan_n[warp] = __popc(bal); scan_t[warp] = incl; }
        __syncthreads();
        int before = base, tiles = tbase;
        for (int w = 0; w < warp; w++) { before += scan_n[w]; tiles += scan_t[w]; }
        if (flag) {
            const int ui = before + __popc(bal & ((1u << lane) - 1u));
            int32_t *u = a.units + 4 * ui;
            u[0] = 0; u[1] = e; u[2] = lo; u[3] = cnt;
            const int t0 = tiles + incl - nt;           // tiles of every earlier unit
            a.prefix_gu[ui] = t0 * a.rb_gu;
            a.prefix_dn[ui] = t0 * a.rb_dn;
        }
        __syncthreads();
        if (tid == 0) {
            int tot = 0, ttot = 0;
            for (int w = 0; w < nwarps; w++) { tot += scan_n[w]; ttot += scan_t[w]; }
            base += tot;
            tbase += ttot;
        }
        __syncthreads();
    }
    if (tid == 0) {
        const int n = base;
        *a.n_units = n;
        a.prefix_gu[n] = tbase * a.rb_gu;
        a.prefix_dn[n] = tbase * a.rb_dn;
        if (bad) atomicOr(a.status, bad);
        *a.abort = bad ? 1 : 0;
    }
}

// per-token activation scale 2^-u with max|x_t| * 2^-u in [2^14, 2^15), u in [-113, 113]
__global__ void __launch_bounds__(256) gemm_scales_kernel(int T, int d, const uint16_t *x, float *tok_scale)
{
    pdl_wait();
    pdl_trigger();
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
    float *out;                     // zeroed here: the down GEMM adds into it
    int32_t *status, *abort;
};
__global__ void __launch_bounds__(256) gemm_gather_kernel(GatherArgs a)
{
    pdl_wait();
    pdl_trigger();
    const int slots = a.T * a.k, d8 = a.d / 8;
    const bool ok_off = *a.abort == 0;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < (size_t)a.T * (a.d / 4);
         q += (size_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(a.out)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
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
        s = dclamp(a.status, s, 0, slots - 1);
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
    int item_hi;                    // the kernel takes items [0, min(item_hi, all items))
    const uint8_t *sfa;             // block-scaled GEMMs: gate/up's token tiles' scale blocks
    uint8_t *sfa_dn;                //   down's (h) token tiles' scale blocks
    uint8_t *hq;                    //   routed h as two e4m3 planes [2][T*k][f] (in hp's routed rows)
};

struct GItem {
    int shared, id, tok0, ntok;     // unit
    int rb;                         // gate/up: 128-row block of f; down: pair of 128-row blocks of d
    int n0, ncols;                  // first token of the tile within the unit, tokens in the tile
    int nw;                         // weight rows (MMA N): 256, or 128 for a last odd block of d
};

template <int MODE>
__device__ __forceinline__ int k_of(const GemmArgs &a) { return MODE == kGU ? a.d : a.f; }

template <int MODE>
__device__ __forceinline__ GItem gitem(const GemmArgs &a, const int32_t *prefix, int n_units, int i)
{
    int lo = 0, hi = n_units;                      // unit u with prefix[u] <= i < prefix[u+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= i) lo = mid; else hi = mid;
    }
    const int4 u = *reinterpret_cast<const int4 *>(a.units + 4 * lo);
    GItem it;
    it.shared = u.x;
    // the unit list comes from gemm_units (validated offsets); debug builds record a unit
    // outside the table or the slots, every build keeps the expert index in range
    it.id = dclamp(a.status, u.y, 0, (u.x ? a.S : a.E) - 1);
    dcheck(a.status, u.z >= 0 && u.w >= 0 && (size_t)u.z + u.w <= (u.x ? (size_t)a.T : (size_t)a.T * a.k));
    it.tok0 = u.z;
    it.ntok = u.w;
    const int ntiles = max(1, (it.ntok + kBM - 1) / kBM);
    const int j = i - prefix[lo];
    const int nt = j % ntiles;                     // token tile fastest: the weight block stays hot in L2
    it.rb = j / ntiles;
    it.n0 = nt * kBM;
    it.ncols = min(kBM, it.ntok - it.n0);
    it.nw = (MODE == kGU || 2 * it.rb + 1 < a.d / kTileRows) ? kWRows : kWRows / 2;
    return it;
}

template <int MODE>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs a,
                                                                const __grid_constant__ CUtensorMap mtok_routed,
                                                                const __grid_constant__ CUtensorMap mtok_shared,
                                                                const __grid_constant__ CUtensorMap mw1,
                                                                const __grid_constant__ CUtensorMap mw3)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t gsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *smA = sm;                                   // kStg x kABytes: token tiles
    uint8_t *smW = smA + kStg * kABytes;                 // kStg x kWBytes: weight tiles
    // full[s]: the token tile (TMA bytes, one arrive by the producer) and the weight tile
    // (one arrive per dequant warp); empty[s]: one tcgen05.commit per stage
    __shared__ uint64_t full[kStg], empty[kStg], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int bail;
    __shared__ int32_t s_prefix[kMaxExperts + kMaxShared + 1];   // item prefix of the units

    if (*a.abort) return;
    const int n_units = *a.n_units;
    const int n_items = min(a.prefix[n_units], a.item_hi);
    if ((int)blockIdx.x >= n_items) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = k_of<MODE>(a), nks = K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStg; s++) { mb_init(&full[s], 1 + kNumDq); mb_init(&empty[s], 1); }
        for (int b = 0; b < 2; b++) { mb_init(&acc_full[b], 1); mb_init(&acc_empty[b], kNumEpi); }
        mb_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    for (int u = threadIdx.x; u <= n_units; u += blockDim.x) s_prefix[u] = a.prefix[u];
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
    auto wait_free_warp = [&](uint64_t *bars, int D, uint32_t st) -> bool {
        return st < (uint32_t)D || mb_wait_warp(&bars[st % D], ((st / D) - 1) & 1u);
    };
    // after a timeout: wait (bounded) for the copies of the last D fills of a ring
    auto drain_fills = [&](uint64_t *bars, int D, uint32_t n) {
        for (uint32_t f = n > (uint32_t)D ? n - D : 0; f < n; f++) mb_wait(&bars[f % D], (f / D) & 1u);
    };
    // the shared stop flag as lane 0 of the warp reads it (keeps loop exits warp-uniform)
    auto stop = [&]() -> bool { return __shfl_sync(0xffffffffu, bail, 0) != 0; };

    const int nkt = K / kTileK;
    // a position in this block's sequence of packed tiles: item i, K tile kt
    struct Cur {
        int i, kt;
        GItem it;
    };
    auto cur_item = [&](Cur &c, int i) {
        c.i = i;
        c.kt = 0;
        if (i < n_items) c.it = gitem<MODE>(a, s_prefix, n_units, i);
    };
    auto cur_next = [&](Cur &c) {
        if (++c.kt == nkt) cur_item(c, c.i + gridDim.x);
    };
    // the packed tile of weight block mb at a position (routed items only)
    auto tile_at = [&](const Cur &c, int mb) -> const uint8_t * {
        const uint8_t *ex = a.table + (size_t)c.it.id * a.expert_bytes;
        if (MODE == kGU) return ex + ((size_t)c.it.rb * nkt + c.kt) * 2 * kTileBytes + (size_t)mb * kTileBytes;
        return ex + a.gateup_bytes + ((size_t)(2 * c.it.rb + mb) * nkt + c.kt) * kTileBytes;
    };
    auto block_on = [&](const Cur &c, int mb) { return c.i < n_items && !c.it.shared && mb * kTileRows < c.it.nw; };
    auto prefetch_l2 = [&](const Cur &c) {
        if (!block_on(c, 0)) return;
        if (MODE == kGU) {
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(tile_at(c, 0)), "r"(2 * kTileBytes) : "memory");
        } else {
            for (int mb = 0; mb < 2; mb++)
                if (block_on(c, mb))
                    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(tile_at(c, mb)), "r"(kTileBytes) : "memory");
        }
    };
    if (warp == kWarpProd) {
        // ------------------------------------------------------------ token tiles (and bf16 weights)
        uint32_t st = 0;
        bool failed = false;
        // lane 0 also prefetches the packed tiles into L2, kL2Ahead tiles before the
        // stage it issues (the dequant warps load them into registers two tiles ahead)
        Cur pf;
        if (lane == 0) {
            cur_item(pf, blockIdx.x);
            for (int j = 0; j < kL2Ahead; j++) { prefetch_l2(pf); cur_next(pf); }
        }
        for (int i = blockIdx.x; i < n_items && !failed && !stop(); i += gridDim.x) {
            const GItem it = gitem<MODE>(a, s_prefix, n_units, i);
            const CUtensorMap *mt = it.shared ? &mtok_shared : &mtok_routed;
            int row0;
            if (MODE == kGU) row0 = it.shared ? it.n0 : it.tok0 + it.n0;
            else row0 = it.shared ? a.T * a.k + it.id * a.T + it.n0 : it.tok0 + it.n0;
            const int nb = it.nw / kTileRows;
            for (int ks = 0; ks < nks; ks++, st++) {
                if (!wait_free_warp(empty, kStg, st)) {
                    timeout();
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    if ((ks & 1) == 0) { prefetch_l2(pf); cur_next(pf); }
                    uint64_t *fa = &full[st % kStg];
                    // the bf16 weight tiles of a shared expert come by TMA too
                    mb_expect_tx(fa, (uint32_t)kABytes + (it.shared ? (uint32_t)(nb * kTileRows * kBK * 2) : 0u));
                    tma2d(smA + (st % kStg) * kABytes, mt, ks * kBK, row0, fa);
                    if (it.shared) {
                        uint8_t *W = smW + (st % kStg) * kWBytes;
                        if (MODE == kGU) {
                            const int wrow = it.id * a.f + it.rb * kTileRows;
                            tma2d(W, &mw1, ks * kBK, wrow, fa);
                            tma2d(W + kTileRows * kBK * 2, &mw3, ks * kBK, wrow, fa);
                        } else {
                            for (int b = 0; b < nb; b++)
                                tma2d(W + b * kTileRows * kBK * 2, &mw1, ks * kBK,
                                      it.id * a.d + (2 * it.rb + b) * kTileRows, fa);
                        }
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0 && bail) drain_fills(full, kStg, st);
        __syncwarp();
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issue: D[token][weight row]
        uint32_t st = 0, n = 0;
        bool failed = false;
        for (int i = blockIdx.x; i < n_items && !failed && !stop(); i += gridDim.x, n++) {
            const GItem it = gitem<MODE>(a, s_prefix, n_units, i);
            const uint32_t id = idesc(it.shared ? 1 : 0, it.nw);
            const int buf = n & 1;
            if (n >= 2 && !mb_wait_warp(&acc_empty[buf], ((n >> 1) - 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            const uint32_t d0 = tmem + (uint32_t)buf * 256u;
            // the two stages of a packed tile at a time (their weight halves are written
            // together): both waits first, so the second stage's MMAs queue right behind
            // the first's
            for (int ks = 0; ks < nks; ks += 2, st += 2) {
                if (!mb_wait_warp(&full[st % kStg], (st / kStg) & 1u) ||
                    !mb_wait_warp(&full[(st + 1) % kStg], ((st + 1) / kStg) & 1u)) {
                    timeout();
                    failed = true;
                    break;
                }
                if (lane == 0) {
#pragma unroll
                    for (int s2 = 0; s2 < 2; s2++) {
                        const uint32_t ss = st + s2;
                        // descriptors of the stage's first K slice; each further slice of
                        // 16 is 32 bytes on, i.e. 2 in the descriptor's start-address field
                        const uint64_t dA = sdesc(saddr(smA + (ss % kStg) * kABytes));
                        const uint64_t dW = sdesc(saddr(smW + (ss % kStg) * kWBytes));
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; kk++)
                            umma(d0, dA + 2 * kk, dW + 2 * kk, id, ((ks + s2) | kk) != 0);
                        umma_commit(&empty[ss % kStg]);
                    }
                }
                __syncwarp();
            }
            if (failed) break;
            if (lane == 0) umma_commit(&acc_full[buf]);
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(&drain);                       // every issued MMA done before the dealloc
            mb_wait(&drain, 0);
        }
        __syncwarp();
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------------ dequant (packed -> f16 weights)
        // Thread t: weight block m (gate/up: W1 / W3; down: first / second W2 block), strip
        // of 16 rows, 32-column group gsel of the stage, rows g and g + 8 of the strip, half
        // h of their 32 columns.  Its bytes of a packed 128 x 128 tile come straight from
        // global memory (no shared-memory copy): two 16-byte pieces (the tile's even and
        // odd stage; a warp reads 512 contiguous bytes) and the scale words of its two
        // rows, loaded two tiles ahead.  Per stage 2 x 4 eight-byte stores.
        const int t = threadIdx.x - kWarpDq0 * 32;             // 0..511
        const int m = t >> 8;
        const int u = t & 255, strip = u >> 5, gsel = (u >> 4) & 1, g = (u >> 1) & 7, h = u & 1;
        const int offA = (strip * 4 + gsel) * 256 + 32 * g + 16 * h, offB = offA + 2 * 256;
        const int offS = kTileNibbleBytes + (strip * 16 + g) * 4;
        auto bmax_at = [&](const Cur &c) -> int {
            const size_t o = MODE == kGU ? trailer_offset(a.E, a.d, a.f, c.it.id, m, c.it.rb)
                                         : trailer_offset(a.E, a.d, a.f, c.it.id, 2, 2 * c.it.rb + m);
            return (int)__ldg(reinterpret_cast<const uint32_t *>(a.table + o));
        };
        // this thread's bytes of one packed tile, and the tile's block scale maximum
        struct TileRegs {
            uint4 qa, qb;
            uint32_t s0, s1;
            int bmax;
        };
        auto load_tile = [&](const Cur &c, TileRegs &r, int bmax_prev) {
            r.bmax = bmax_prev;
            if (!block_on(c, m)) return;
            const uint8_t *p = tile_at(c, m);
            r.qa = __ldg(reinterpret_cast<const uint4 *>(p + offA));
            r.qb = __ldg(reinterpret_cast<const uint4 *>(p + offB));
            r.s0 = __ldg(reinterpret_cast<const uint32_t *>(p + offS));
            r.s1 = __ldg(reinterpret_cast<const uint32_t *>(p + offS + 32));
            if (c.kt == 0) r.bmax = bmax_at(c);
        };
        uint32_t st = 0;
        bool failed = false;
        // the two stages of the tile at c from registers r
        // both stages of the tile at c from registers r: the two slots are claimed, both
        // stages written, then one proxy fence and both arrivals.  A slot is free once the
        // MMAs that read it have completed, and they complete in issue order, so the
        // later slot's release covers the earlier one: one wait per tile.
        auto dequant_tile = [&](const Cur &c, const TileRegs &r) {
            const bool on = block_on(c, m);
            constexpr int kSpt = kTileK / kBK;                  // stages per tile
            if (!wait_free_warp(empty, kStg, st + kSpt - 1)) { timeout(); failed = true; return; }
            if (on) {
#pragma unroll
                for (int s2 = 0; s2 < kSpt; s2++) {
                    const int cc = 2 * s2 + gsel;
                    const uint4 q = s2 ? r.qb : r.qa;
                    uint8_t *Wt = smW + ((st + s2) % kStg) * kWBytes + m * (kTileRows * kBK * 2);
#pragma unroll
                    for (int hr = 0; hr < 2; hr++) {            // rows g and g+8 of the strip
                        const int row = strip * 16 + g + 8 * hr;
                        const uint32_t b = ((hr ? r.s1 : r.s0) >> (8 * cc)) & 0xFFu;
                        const uint32_t s1 = b == 255u ? 0u : f16_pow2((int)b - r.bmax + 13);
                        const uint32_t sc2 = s1 | (s1 << 16);
                        const uint32_t wa = hr ? q.y : q.x, wb = hr ? q.w : q.z;
#pragma unroll
                        for (int j = 0; j < 4; j++) {           // columns 8j + 4h .. +3 of the group
                            const uint32_t v0 = hmul2(e2m1x2_f16x2(wa >> (8 * j)), sc2);
                            const uint32_t v1 = hmul2(e2m1x2_f16x2(wb >> (8 * j)), sc2);
                            const int chunk = 4 * gsel + j;
                            *reinterpret_cast<uint2 *>(Wt + row * 128 + ((chunk ^ (row & 7)) << 4) + 8 * h) =
                                make_uint2(v0, v1);
                        }
                    }
                }
                fence_async_smem();
            }
            __syncwarp();
            if (lane == 0)
#pragma unroll
                for (int s2 = 0; s2 < kSpt; s2++) mb_arrive(&full[(st + s2) % kStg]);
            st += kSpt;
        };
        // tiles in sequence: position p from register set p % 2, loaded two tiles ahead
        Cur c0, c1, tail;
        cur_item(c0, blockIdx.x);
        c1 = c0;
        cur_next(c1);
        tail = c1;
        TileRegs r0{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), 0, 0, 0}, r1 = r0;
        load_tile(c0, r0, 0);
        load_tile(c1, r1, r0.bmax);
        while (c0.i < n_items && !stop()) {
            dequant_tile(c0, r0);
            if (failed) break;
            c0 = tail;
            cur_next(c0);                                   // position p + 2
            load_tile(c0, r0, r1.bmax);
            if (c1.i >= n_items || stop()) break;
            dequant_tile(c1, r1);
            if (failed) break;
            c1 = c0;
            cur_next(c1);                                   // position p + 3
            load_tile(c1, r1, r0.bmax);
            tail = c1;
        }
    } else {
        // ------------------------------------------------------------ epilogue: one token per thread
        const int q = warp & 3;                                 // TMEM lane quadrant
        const int tr = 32 * q + lane;                           // token row of the tile
        uint32_t n = 0;
        for (int i = blockIdx.x; i < n_items && !stop(); i += gridDim.x, n++) {
            const GItem it = gitem<MODE>(a, s_prefix, n_units, i);
            const int buf = n & 1;
            const bool valid = tr < it.ncols;
            int row = 0;                                        // gate/up: h row; down: output token
            float fo = 1.0f;                                    // gate/up: token factor; down: routing weight
            if (valid) {
                if (it.shared) {
                    row = MODE == kGU ? a.T * a.k + it.id * a.T + it.n0 + tr : it.n0 + tr;
                } else {
                    const int p = it.tok0 + it.n0 + tr;
                    const int slot = dclamp(a.status, a.perm[p], 0, a.T * a.k - 1);
                    if (MODE == kGU) {
                        row = p;
                        fo = a.tok_scale[a.T + slot / a.k];
                    } else {
                        row = slot / a.k;
                        fo = a.weight[slot];
                    }
                }
            }
            float f1 = 1.0f, f3 = 1.0f;                         // block factors 2^(bmax - 140)
            if (!it.shared) {
                const size_t o1 = MODE == kGU ? trailer_offset(a.E, a.d, a.f, it.id, 0, it.rb)
                                              : trailer_offset(a.E, a.d, a.f, it.id, 2, 2 * it.rb);
                f1 = ldexpf(1.0f, (int)*reinterpret_cast<const uint32_t *>(a.table + o1) - 140);
                if (it.nw == kWRows) {
                    const size_t o3 = MODE == kGU ? trailer_offset(a.E, a.d, a.f, it.id, 1, it.rb)
                                                  : trailer_offset(a.E, a.d, a.f, it.id, 2, 2 * it.rb + 1);
                    f3 = ldexpf(1.0f, (int)*reinterpret_cast<const uint32_t *>(a.table + o3) - 140);
                }
            }
            if (!mb_wait_warp(&acc_full[buf], (n >> 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 256u;
            if (MODE == kGU) {
                const float fg = f1 * fo, fu = f3 * fo;
                uint16_t *hrow = a.hp + (size_t)row * a.f + it.rb * kTileRows;
                for (int c0 = 0; c0 < kTileRows; c0 += 16) {
                    float vg[16], vu[16];
                    tmem_ld16(lane_addr + c0, vg);
                    tmem_ld16(lane_addr + kTileRows + c0, vu);
                    uint32_t pk[8];
#pragma unroll
                    for (int jj = 0; jj < 16; jj += 2) {
                        const float h0 = situ(vg[jj] * fg, vu[jj] * fu, a.b1, a.b2);
                        const float h1 = situ(vg[jj + 1] * fg, vu[jj + 1] * fu, a.b1, a.b2);
                        if (it.shared) {
                            const __nv_bfloat162 hb = __floats2bfloat162_rn(h0, h1);
                            pk[jj / 2] = *reinterpret_cast<const uint32_t *>(&hb);
                        } else {
                            const __half2 hh = __floats2half2_rn(h0, h1);
                            pk[jj / 2] = *reinterpret_cast<const uint32_t *>(&hh);
                        }
                    }
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(hrow + c0);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            } else {
                float *orow = a.out + (size_t)row * a.d + 2 * it.rb * kTileRows;
                for (int c0 = 0; c0 < it.nw; c0 += 16) {
                    float v[16];
                    tmem_ld16(lane_addr + c0, v);
                    const float fw = fo * (c0 < kTileRows ? f1 : f3);
                    if (valid) {
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            atomicAdd(reinterpret_cast<float4 *>(orow + c0 + jj),
                                      make_float4(v[jj] * fw, v[jj + 1] * fw, v[jj + 2] * fw, v[jj + 3] * fw));
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

// ---------------------------------------------------------------------------------- block-scaled GEMMs
// The routed experts' gate/up and down projections on kind::mxf8f6f4 MMAs: the weights
// stay in their E2M1 codes and the tensor core applies their E8M0 scales; nothing is
// dequantised.  The tokens (gemm_gather_mx) and h (the gate/up epilogue) enter as two
// e4m3 planes with their own per-32 scales: a 32-wide K step is two MMAs, hi and lo, into
// the same fp32 accumulator.  For a bf16 token the two planes hold it exactly while its
// element lies within 2^12 of its 32-block's largest; a smaller element keeps an absolute
// error below 2^-21 of that largest.  h (fp32) keeps about 8 significant bits.

// Two floats -> two e4m3 bytes (round to nearest even, saturating), x0 in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float x0, float x1)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
    return r;
}
// Two e4m3 bytes (low byte first) -> two exact floats.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t b2)
{
    uint32_t h;
    asm("{\n\t.reg .b16 b;\n\tcvt.u16.u32 b, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, b;\n\t}" : "=r"(h) : "r"(b2));
    return __half22float2(*reinterpret_cast<__half2 *>(&h));
}
// The smallest s with v / 2^s <= 448 (the largest e4m3) for finite v > 0: with
// v = m 2^e, m in [1, 2), s = e - 8, or e - 7 when m > 1.75.  Subnormal v gives a value
// below -127, which the callers clamp.
__device__ __forceinline__ int pow2_over448(float v)
{
    const uint32_t u = __float_as_uint(v);
    const int b = (int)((u >> 23) & 255u);
    return (b == 0 ? -127 : b - 127) - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
}

struct GatherMxArgs {
    int T, d, k, E, S, rb;          // rb: items per token tile (128-row blocks of f)
    const uint16_t *x;
    const int32_t *idx, *offsets, *perm;
    const int32_t *units, *prefix, *n_units;
    uint8_t *hi, *lo;               // [T*k][d] e4m3 planes, perm order
    uint8_t *sfa;                   // [tiles][d/128][2][512] e8m0 scale blocks of the token tiles
    size_t tiles;                   // tiles the scale region holds
    float *out;                     // zeroed here: the down GEMM adds into it
    int32_t *status, *abort;
};

// One warp per routed position p (perm order).  For each 32-element block of the token's
// row (four lanes, eight elements each): 2^sa the smallest power of two that brings the
// block's largest |x| to 448 or below, hi = rn(x / 2^sa); the residual r = x / 2^sa - hi
// is exact in fp32; 2^sl likewise for max |r|, lo = rn(r / 2^sl).
// Scale bytes sa + 127 and sa + sl + 127 go to the token tile's scale blocks (row m of the
// tile at 16 (m % 32) + 4 (m / 32) + the block's index within its 128 columns).
__global__ void __launch_bounds__(256) gemm_gather_mx_kernel(GatherMxArgs a)
{
    pdl_wait();
    pdl_trigger();
    const int slots = a.T * a.k, nkc = a.d / 128;
    const bool ok_off = *a.abort == 0;
    const int n_units = *a.n_units;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < (size_t)a.T * (a.d / 4);
         q += (size_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(a.out)[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int lane = threadIdx.x & 31;
    const int n_warps = (int)((gridDim.x * blockDim.x) >> 5);
    for (int p = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5); p < slots; p += n_warps) {
        int s = a.perm[p];
        if (lane == 0) {
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
        s = dclamp(a.status, s, 0, slots - 1);
        const int t = s / a.k;
        // the routed unit holding p (units after the shared ones ascend in their first row)
        int tile = -1, m = 0;
        if (ok_off && n_units > a.S) {
            int lo = a.S, hi = n_units;
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (a.units[4 * mid + 2] <= p) lo = mid; else hi = mid;
            }
            const int l = p - a.units[4 * lo + 2];
            if (l >= 0 && l < a.units[4 * lo + 3]) {
                tile = a.prefix[lo] / a.rb + l / kBM;
                m = l % kBM;
            }
            if (!dguard(a.status, tile >= 0 && (size_t)tile < a.tiles)) tile = -1;
        }
        const uint4 *xr = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.d);
        uint2 *hr = reinterpret_cast<uint2 *>(a.hi + (size_t)p * a.d);
        uint2 *lr = reinterpret_cast<uint2 *>(a.lo + (size_t)p * a.d);
        for (int c0 = 0; c0 < a.d / 8; c0 += 32) {
            const int c = c0 + lane;                       // 8-element chunk; block c / 4
            const bool on = c < a.d / 8;                   // whole blocks are on or off (d % 128 == 0)
            float v[8];
            float mx = 0.0f;
            {
                const uint4 w = on ? xr[c] : make_uint4(0, 0, 0, 0);
                const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int h = 0; h < 4; h++) {
                    v[2 * h] = __uint_as_float(w4[h] << 16);
                    v[2 * h + 1] = __uint_as_float(w4[h] & 0xFFFF0000u);
                }
#pragma unroll
                for (int j = 0; j < 8; j++) mx = fmaxf(mx, fabsf(v[j]));
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const int sa = mx > 0.0f ? max(pow2_over448(mx), -127) : 0;
            const float inv_a = __uint_as_float((uint32_t)(127 - sa) << 23);    // 2^-sa, sa in [-127, 120]
            uint32_t hw[4];
            float rmx = 0.0f;
#pragma unroll
            for (int h = 0; h < 4; h++) {
                const float a0 = v[2 * h] * inv_a, a1 = v[2 * h + 1] * inv_a;
                hw[h] = e4m3x2_rn(a0, a1);
                const float2 hf = e4m3x2_to_f32x2(hw[h]);
                v[2 * h] = a0 - hf.x;                      // exact residuals
                v[2 * h + 1] = a1 - hf.y;
                rmx = fmaxf(rmx, fmaxf(fabsf(v[2 * h]), fabsf(v[2 * h + 1])));
            }
            rmx = fmaxf(rmx, __shfl_xor_sync(0xffffffffu, rmx, 1));
            rmx = fmaxf(rmx, __shfl_xor_sync(0xffffffffu, rmx, 2));
            // lo's scale 2^(sa + sl) must stay an e8m0 value, sa + sl in [-127, 127]; |r| <= 16
            // (half the e4m3 step at 448), so sl <= -4 and 2^-sl is a normal float
            const int sl = rmx > 0.0f ? min(max(pow2_over448(rmx), max(-127, -127 - sa)), 127 - sa) : 0;
            const float inv_l = __uint_as_float((uint32_t)(127 - sl) << 23);
            uint32_t lw[4];
#pragma unroll
            for (int h = 0; h < 4; h++) lw[h] = e4m3x2_rn(v[2 * h] * inv_l, v[2 * h + 1] * inv_l);
            if (on) {
                hr[c] = make_uint2(hw[0] | (hw[1] << 16), hw[2] | (hw[3] << 16));
                lr[c] = make_uint2(lw[0] | (lw[1] << 16), lw[2] | (lw[3] << 16));
                if ((lane & 3) == 0 && tile >= 0) {
                    const int b = c >> 2, kc = b >> 2, kb = b & 3;
                    uint8_t *sf = a.sfa + ((size_t)tile * nkc + kc) * 1024 + 16 * (m & 31) + 4 * (m >> 5) + kb;
                    sf[0] = (uint8_t)(sa + 127);
                    sf[512] = (uint8_t)(sa + sl + 127);
                }
            }
        }
    }
}

constexpr int kMxStg = 3;                              // stage ring
constexpr int kMxBK = 128;                             // K per stage
constexpr int kMxA = kBM * kMxBK;                      // one e4m3 token plane tile: 16 KB
constexpr int kMxW = kWRows * kMxBK;                   // e2m1 weight tile (16 elements per 16 bytes): 32 KB
constexpr int kMxSF = 4 * 512;                         // scale blocks: token hi, token lo, W1 rows, W3 rows
constexpr int kMxStage = 2 * kMxA + kMxW + kMxSF;      // 67584 (a multiple of 1024)
constexpr int kMxNumEpi = 16;
constexpr int kMxWarpProd = 0, kMxWarpMma = 1, kMxWarpEpi0 = 2;
constexpr int kMxThreads = (kMxWarpEpi0 + kMxNumEpi) * 32;     // 576
constexpr uint32_t kMxWBox = kTileRows * kMxBK / 2;   // packed bytes of one 128 x 128 weight box (the TMA's count)
constexpr int kMxSmem = kMxStg * kMxStage + 1024;
constexpr uint32_t kMxSfCol = 256;                     // scale columns: 16 per stage slot after the accumulator
static_assert(kMxStage % 1024 == 0, "stage slots keep the 1024-byte alignment of the swizzled tiles");
static_assert(kMxSmem + 8 * 1024 <= 232448, "shared memory per block (dynamic + static)");
static_assert(kMxSfCol + 16 * kMxStg <= 512, "tensor-memory columns");

struct MxItem {
    int id, tok0, ntok, rb, n0, ncols, tile, nw;
};
// Item i of the routed items: unit, weight block (gate/up: a 128-row block of f, W1 and W3;
// down: a pair of 128-row blocks of d, or the last single block), token tile.  Tile numbers
// count the 128-row token tiles of all units in unit order (the same for both projections).
template <int MODE>
__device__ __forceinline__ MxItem mx_item(const GemmArgs &a, const int32_t *prefix, int n_units, int rbn, int i)
{
    int lo = 0, hi = n_units;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= i) lo = mid; else hi = mid;
    }
    const int4 u = *reinterpret_cast<const int4 *>(a.units + 4 * lo);
    MxItem it;
    it.id = dclamp(a.status, u.y, 0, a.E - 1);
    dcheck(a.status, u.x == 0 && u.z >= 0 && u.w >= 0 && (size_t)u.z + u.w <= (size_t)a.T * a.k);
    it.tok0 = u.z;
    it.ntok = u.w;
    const int ntiles = max(1, (it.ntok + kBM - 1) / kBM);
    const int j = i - prefix[lo];
    const int nt = j % ntiles;
    it.rb = j / ntiles;
    it.n0 = nt * kBM;
    it.ncols = min(kBM, it.ntok - it.n0);
    it.tile = prefix[lo] / rbn + nt;
    it.nw = (MODE == kGU || 2 * it.rb + 1 < a.d / kTileRows) ? kWRows : kWRows / 2;
    return it;
}

// 32 values of one row -> the two e4m3 planes' 32 bytes each and the two scale exponents:
// the split gemm_gather_mx makes, for a block one thread holds.
__device__ __forceinline__ void split32(float (&v)[32], uint4 (&hq)[2], uint4 (&lq)[2], int &sa, int &sl)
{
    float mx = 0.0f;
#pragma unroll
    for (int j = 0; j < 32; j++) mx = fmaxf(mx, fabsf(v[j]));
    sa = mx > 0.0f ? max(pow2_over448(mx), -127) : 0;
    const float ia = __uint_as_float((uint32_t)(127 - sa) << 23);
    uint32_t hw[8], lw[8];
    float rmx = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; j++) {
        const float a0 = v[2 * j] * ia, a1 = v[2 * j + 1] * ia;
        const uint32_t h2 = e4m3x2_rn(a0, a1);
        const float2 hf = e4m3x2_to_f32x2(h2);
        v[2 * j] = a0 - hf.x;
        v[2 * j + 1] = a1 - hf.y;
        rmx = fmaxf(rmx, fmaxf(fabsf(v[2 * j]), fabsf(v[2 * j + 1])));
        if (j & 1) hw[j >> 1] |= h2 << 16; else hw[j >> 1] = h2;
    }
    sl = rmx > 0.0f ? min(max(pow2_over448(rmx), max(-127, -127 - sa)), 127 - sa) : 0;
    const float il = __uint_as_float((uint32_t)(127 - sl) << 23);
#pragma unroll
    for (int j = 0; j < 16; j++) {
        const uint32_t l2 = e4m3x2_rn(v[2 * j] * il, v[2 * j + 1] * il);
        if (j & 1) lw[j >> 1] |= l2 << 16; else lw[j >> 1] = l2;
    }
    hq[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    hq[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    lq[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    lq[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
}

// Roles (one block per SM):
//   warp 0       producer, everything by TMA or bulk copy into the stage ring: the two
//                token planes' tiles (128 columns x 128 rows; gate/up: the gathered
//                tokens, down: h), the tile's two token scale blocks, the item's two weight
//                boxes (128 columns x 128 rows each: W1 and W3 of a block of f, or two W2
//                blocks of d) from the table's row-major codes with the packed-FP4
//                tensor-map type (each 16 codes land as 8 bytes at the start of a 16-byte
//                chunk: the MMA's e2m1 layout), and their scale blocks; the L2 prefetch of
//                the weight boxes kL2Ahead stages ahead;
//   warp 1       MMA: tcgen05.cp of the four scale blocks into tensor memory, then per
//                32-wide K step the hi and the lo MMA (M=128 tokens, N=256 weight rows,
//                or 128 for a last odd block of d); one accumulator of 256 columns;
//   warps 2-17   epilogue, four warps per lane quadrant, 64 accumulator columns each
//                (gate/up: 32 of g and the matching 32 of u); the accumulator is read into
//                registers and released before the arithmetic.  Gate/up: h = SiTU(g, u),
//                split into the down projection's two e4m3 planes and scale blocks; down:
//                out[t] += w * y, float4 atomics.
template <int MODE>
__global__ void __launch_bounds__(kMxThreads, 1) gemm_mx_kernel(const __grid_constant__ GemmArgs a, int item_lo,
                                                                const __grid_constant__ CUtensorMap mhi,
                                                                const __grid_constant__ CUtensorMap mlo,
                                                                const __grid_constant__ CUtensorMap mw0,
                                                                const __grid_constant__ CUtensorMap mw1)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t gsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[kMxStg], empty[kMxStg], acc_full, acc_empty, drain;
    __shared__ uint32_t tmem_base;
    __shared__ int bail;
    __shared__ int32_t s_prefix[kMaxExperts + kMaxShared + 1];

    if (*a.abort) return;
    const int n_units = *a.n_units;
    const int n_items = a.prefix[n_units];
    if (item_lo + (int)blockIdx.x >= n_items) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int K = MODE == kGU ? a.d : a.f;
    const int nkc = K / kMxBK;
    const int rbn = MODE == kGU ? a.f / kTileRows : (a.d / kTileRows + 1) / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kMxStg; s++) { mb_init(&full[s], 1); mb_init(&empty[s], 1); }
        mb_init(&acc_full, 1);
        mb_init(&acc_empty, kMxNumEpi);
        mb_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    for (int u = threadIdx.x; u <= n_units; u += blockDim.x) s_prefix[u] = a.prefix[u];
    if (warp == kMxWarpMma) {
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
    auto stop = [&]() -> bool { return __shfl_sync(0xffffffffu, bail, 0) != 0; };
    const int i0 = item_lo + (int)blockIdx.x;
    // weight box mm of an item: its first row in the row-major codes (the tensor map mw0
    // or mw1), and the scale block of (item, mm, K stage)
    auto wrow = [&](const MxItem &it, int mm) -> int {
        return MODE == kGU ? it.id * a.f + it.rb * kTileRows : it.id * a.d + (2 * it.rb + mm) * kTileRows;
    };
    auto wsf = [&](const MxItem &it, int mm, int kc) -> const uint8_t * {
        if (MODE == kGU)
            return a.table + mx_sfgu_offset(a.E, a.d, a.f) + ((((size_t)it.id * rbn + it.rb) * nkc + kc) * 2 + mm) * 512;
        return a.table + mx_sfdn_offset(a.E, a.d, a.f) +
               (((size_t)it.id * (a.d / kTileRows) + 2 * it.rb + mm) * nkc + kc) * 512;
    };
    const uint8_t *sfa_in = MODE == kGU ? a.sfa : a.sfa_dn;

    if (warp == kMxWarpProd) {
        // ------------------------------------------------------------ everything by TMA
        uint32_t st = 0;
        bool failed = false;
        int pf_i = i0, pf_kc = 0;
        MxItem pf{};
        auto pf_step = [&]() {
            if (pf_i >= n_items) return;
            if (pf_kc == 0) pf = mx_item<MODE>(a, s_prefix, n_units, rbn, pf_i);
            asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(&mw0),
                         "r"(pf_kc * kMxBK), "r"(wrow(pf, 0)) : "memory");
            if (pf.nw > kTileRows)
                asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(&mw1),
                             "r"(pf_kc * kMxBK), "r"(wrow(pf, 1)) : "memory");
            if (++pf_kc == nkc) { pf_kc = 0; pf_i += gridDim.x; }
        };
        if (lane == 0)
            for (int j = 0; j < kL2Ahead; j++) pf_step();
        for (int i = i0; i < n_items && !failed && !stop(); i += gridDim.x) {
            const MxItem it = mx_item<MODE>(a, s_prefix, n_units, rbn, i);
            const int row0 = it.tok0 + it.n0;
            const bool two = it.nw > kTileRows;
            for (int kc = 0; kc < nkc; kc++, st++) {
                if (st >= (uint32_t)kMxStg && !mb_wait_warp(&empty[st % kMxStg], ((st / kMxStg) - 1) & 1u)) {
                    timeout();
                    failed = true;
                    break;
                }
                if (lane == 0) {
                    pf_step();
                    uint8_t *sb = sm + (st % kMxStg) * kMxStage;
                    uint64_t *fb = &full[st % kMxStg];
                    mb_expect_tx(fb, 2u * kMxA + 1024u + (two ? 2u : 1u) * (kMxWBox + 512u));
                    tma2d(sb, &mhi, kc * kMxBK, row0, fb);
                    tma2d(sb + kMxA, &mlo, kc * kMxBK, row0, fb);
                    bulk_g2s(sb + 2 * kMxA + kMxW, sfa_in + ((size_t)it.tile * nkc + kc) * 1024, 1024u, fb);
                    tma2d(sb + 2 * kMxA, &mw0, kc * kMxBK, wrow(it, 0), fb);
                    bulk_g2s(sb + 2 * kMxA + kMxW + 1024, wsf(it, 0, kc), 512u, fb);
                    if (two) {
                        tma2d(sb + 2 * kMxA + kMxW / 2, &mw1, kc * kMxBK, wrow(it, 1), fb);
                        bulk_g2s(sb + 2 * kMxA + kMxW + 1536, wsf(it, 1, kc), 512u, fb);
                    }
                }
                __syncwarp();
            }
        }
        if (lane == 0 && bail)
            for (uint32_t f = st > (uint32_t)kMxStg ? st - kMxStg : 0; f < st; f++)
                mb_wait(&full[f % kMxStg], (f / kMxStg) & 1u);
        __syncwarp();
    } else if (warp == kMxWarpMma) {
        // ------------------------------------------------------------ scales to tensor memory, MMAs
        uint32_t st = 0, n = 0;
        bool failed = false;
        for (int i = i0; i < n_items && !failed && !stop(); i += gridDim.x, n++) {
            const int nw = MODE == kGU ? kWRows : mx_item<MODE>(a, s_prefix, n_units, rbn, i).nw;
            if (n >= 1 && !mb_wait_warp(&acc_empty, (n - 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            for (int kc = 0; kc < nkc; kc++, st++) {
                if (!mb_wait_warp(&full[st % kMxStg], (st / kMxStg) & 1u)) {
                    timeout();
                    failed = true;
                    break;
                }
                tc_fence_after();
                if (lane == 0) {
                    uint8_t *sb = sm + (st % kMxStg) * kMxStage;
                    uint8_t *sf = sb + 2 * kMxA + kMxW;
                    const uint32_t sft = tmem + kMxSfCol + 16u * (st % kMxStg);
                    tc_cp_sf(sft, sdesc_sf(saddr(sf)));                // token hi
                    tc_cp_sf(sft + 4, sdesc_sf(saddr(sf + 512)));      // token lo
                    tc_cp_sf(sft + 8, sdesc_sf(saddr(sf + 1024)));     // weight rows N 0..127
                    if (nw > kTileRows) tc_cp_sf(sft + 12, sdesc_sf(saddr(sf + 1536)));   // N 128..255
                    const uint64_t dh = sdesc(saddr(sb)), dl = sdesc(saddr(sb + kMxA)),
                                   dw = sdesc(saddr(sb + 2 * kMxA));
#pragma unroll
                    for (int kb = 0; kb < kMxBK / 32; kb++) {
                        const uint32_t id = idesc_mx(nw, kb, kb);
                        umma_mx(tmem, dh + 2 * kb, dw + 2 * kb, id, sft, sft + 8, (kc | kb) != 0);
                        umma_mx(tmem, dl + 2 * kb, dw + 2 * kb, id, sft + 4, sft + 8, 1u);
                    }
                    umma_commit(&empty[st % kMxStg]);
                }
                __syncwarp();
            }
            if (failed) break;
            if (lane == 0) umma_commit(&acc_full);
            __syncwarp();
        }
        if (lane == 0) {
            umma_commit(&drain);
            mb_wait(&drain, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                                 // TMEM lane quadrant
        const int part = (warp - kMxWarpEpi0) >> 2;             // 0..3
        const int tr = 32 * q + lane;
        const int nkc_dn = a.f / kMxBK;
        uint32_t n = 0;
        for (int i = i0; i < n_items && !stop(); i += gridDim.x, n++) {
            const MxItem it = mx_item<MODE>(a, s_prefix, n_units, rbn, i);
            const bool valid = tr < it.ncols;
            const int p = it.tok0 + it.n0 + tr;                  // position (perm order) of the row
            if (!mb_wait_warp(&acc_full, n & 1u)) { timeout(); break; }
            tc_fence_after();
            const uint32_t lrow = tmem + ((uint32_t)(32 * q) << 16);
            // gate/up: g columns 32 part.., u columns 128 + 32 part..; down: columns 64 part..
            const uint32_t c0 = MODE == kGU ? 32u * part : 64u * part;
            const uint32_t c1 = MODE == kGU ? kTileRows + 32u * part : 64u * part + 32u;
            const bool on = MODE == kGU || (int)c0 < it.nw;
            uint32_t r0[16], r1[16], r2[16], r3[16];
            if (on) {
                tmem_ld16_nowait(lrow + c0, r0);
                tmem_ld16_nowait(lrow + c0 + 16, r1);
                tmem_ld16_nowait(lrow + c1, r2);
                tmem_ld16_nowait(lrow + c1 + 16, r3);
                tmem_wait_ld();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&acc_empty);
            if (!on || !valid) continue;
            if (MODE == kGU) {
                const float ib1 = 1.0f / a.b1, ib2 = 1.0f / a.b2;
                float hv[32];
#pragma unroll
                for (int jj = 0; jj < 16; jj++) {
                    hv[jj] = situ_mx(__uint_as_float(r0[jj]), __uint_as_float(r2[jj]), a.b1, a.b2, ib1, ib2);
                    hv[16 + jj] = situ_mx(__uint_as_float(r1[jj]), __uint_as_float(r3[jj]), a.b1, a.b2, ib1, ib2);
                }
                uint4 hq[2], lq[2];
                int sa, sl;
                split32(hv, hq, lq, sa, sl);
                const size_t at = (size_t)p * a.f + it.rb * kTileRows + 32 * part;
                uint4 *dh = reinterpret_cast<uint4 *>(a.hq + at);
                uint4 *dl = reinterpret_cast<uint4 *>(a.hq + (size_t)a.T * a.k * a.f + at);
                dh[0] = hq[0]; dh[1] = hq[1];
                dl[0] = lq[0]; dl[1] = lq[1];
                uint8_t *sf = a.sfa_dn + ((size_t)it.tile * nkc_dn + it.rb) * 1024 + 16 * (tr & 31) + 4 * (tr >> 5) + part;
                sf[0] = (uint8_t)(sa + 127);
                sf[512] = (uint8_t)(sa + sl + 127);
            } else {
                const int slot = dclamp(a.status, a.perm[p], 0, a.T * a.k - 1);
                const float fw = a.weight[slot];
                float *orow = a.out + (size_t)(slot / a.k) * a.d + 2 * it.rb * kTileRows + 64 * part;
#pragma unroll
                for (int jj = 0; jj < 16; jj += 4) {
                    atomicAdd(reinterpret_cast<float4 *>(orow + jj),
                              make_float4(__uint_as_float(r0[jj]) * fw, __uint_as_float(r0[jj + 1]) * fw,
                                          __uint_as_float(r0[jj + 2]) * fw, __uint_as_float(r0[jj + 3]) * fw));
                    atomicAdd(reinterpret_cast<float4 *>(orow + 16 + jj),
                              make_float4(__uint_as_float(r1[jj]) * fw, __uint_as_float(r1[jj + 1]) * fw,
                                          __uint_as_float(r1[jj + 2]) * fw, __uint_as_float(r1[jj + 3]) * fw));
                    atomicAdd(reinterpret_cast<float4 *>(orow + 32 + jj),
                              make_float4(__uint_as_float(r2[jj]) * fw, __uint_as_float(r2[jj + 1]) * fw,
                                          __uint_as_float(r2[jj + 2]) * fw, __uint_as_float(r2[jj + 3]) * fw));
                    atomicAdd(reinterpret_cast<float4 *>(orow + 48 + jj),
                              make_float4(__uint_as_float(r3[jj]) * fw, __uint_as_float(r3[jj + 1]) * fw,
                                          __uint_as_float(r3[jj + 2]) * fw, __uint_as_float(r3[jj + 3]) * fw));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMxWarpMma) {
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
        cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        set = true;
    }
    const int grid = max(1, min(num_sms(), max_items));
    timing_begin(name, s);
    const cudaError_t err = launch_pdl(gemm_kernel<MODE>, dim3(grid), dim3(kGemmThreads), kGemmSmem, s, ga, mbr,
                                       mbs, ma1, ma3);
    count_launch();
    timing_end(name, s);
    return err;
}

template <int MODE>
cudaError_t launch_gemm_mx(const GemmArgs &ga, int item_lo, const CUtensorMap &mhi, const CUtensorMap &mlo,
                           const CUtensorMap &mw0, const CUtensorMap &mw1, int max_items, cudaStream_t s,
                           const char *name)
{
    static bool set = false;
    if (!set) {
        cudaFuncSetAttribute(gemm_mx_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxSmem);
        set = true;
    }
    const int grid = max(1, min(num_sms(), max_items));
    timing_begin(name, s);
    const cudaError_t err =
        launch_pdl(gemm_mx_kernel<MODE>, dim3(grid), dim3(kMxThreads), kMxSmem, s, ga, item_lo, mhi, mlo, mw0, mw1);
    count_launch();
    timing_end(name, s);
    return err;
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

    cudaError_t err = cudaSuccess;
    // items per token tile: gate/up one per 128-row block of f, down one per pair of 128-row blocks of d
    UnitsArgs ua{T, E, k, S, c.f / kTileRows, (c.d / kTileRows + 1) / 2, offsets, units, prefix_gu,
                 prefix_dn, n_units, status, abort};
    timing_begin("gemm_units", s);
    err = launch_pdl(gemm_units_kernel, dim3(1), dim3(1024), 0, s, ua);
    count_launch();
    timing_end("gemm_units", s);
    if (err != cudaSuccess) return err;
    // the routed gate/up projection on the block-scaled MMAs: the tokens as two e4m3
    // planes in xg's bytes, their scale blocks per token tile
    const bool mx = prefill_gemm_block_scaled(c, T);
    uint8_t *xhi = reinterpret_cast<uint8_t *>(xg), *xlo = xhi + (size_t)T * k * c.d;
    if (!mx) {
        timing_begin("gemm_scales", s);
        err = launch_pdl(gemm_scales_kernel, dim3((T * 32 + 255) / 256), dim3(256), 0, s, T, c.d, x, tok_scale);
        count_launch();
        timing_end("gemm_scales", s);
        if (err != cudaSuccess) return err;
        GatherArgs gta{T, c.d, k, E, x, idx, offsets, perm, tok_scale, xg, out, status, abort};
        const size_t work = (size_t)T * k * (c.d / 8);
        int grid = (int)std::min<size_t>((work + 255) / 256, (size_t)num_sms() * 16);
        timing_begin("gemm_gather", s);
        err = launch_pdl(gemm_gather_kernel, dim3(std::max(grid, 1)), dim3(256), 0, s, gta);
        count_launch();
        timing_end("gemm_gather", s);
        if (err != cudaSuccess) return err;
    } else {
        GatherMxArgs gmx{T, c.d, k, E, S, c.f / kTileRows, x, idx, offsets, perm, units, prefix_gu, n_units,
                         xhi, xlo, ws + L.sfa, gemm_token_tiles(c, T), out, status, abort};
        const size_t warps = (size_t)T * k;
        int grid = (int)std::min<size_t>((warps * 32 + 255) / 256, (size_t)num_sms() * 16);
        timing_begin("gemm_gather_mx", s);
        err = launch_pdl(gemm_gather_mx_kernel, dim3(std::max(grid, 1)), dim3(256), 0, s, gmx);
        count_launch();
        timing_end("gemm_gather_mx", s);
        if (err != cudaSuccess) return err;
    }

    CUtensorMap mb_routed{}, mb_shared{}, ma1{}, ma3{}, mb_h{}, ma2{}, mhi{}, mlo{};
    bool ok = map16(&mb_h, hp, rows_all, c.f, kBM);
    if (mx) ok = ok && map8(&mhi, xhi, (uint64_t)T * k, c.d, kBM) && map8(&mlo, xlo, (uint64_t)T * k, c.d, kBM);
    else ok = ok && map16(&mb_routed, xg, (uint64_t)T * k, c.d, kBM);
    if (S > 0)
        ok = ok && map16(&mb_shared, x, (uint64_t)T, c.d, kBM) &&
             map16(&ma1, sh_w1, (uint64_t)S * c.f, c.d, kBM) && map16(&ma3, sh_w3, (uint64_t)S * c.f, c.d, kBM) &&
             map16(&ma2, sh_w2, (uint64_t)S * c.d, c.f, kBM);
    if (!ok) return cudaErrorInvalidValue;

    GemmArgs ga{T, c.d, c.f, k, S, E, c.situ_b1, c.situ_b2, units, prefix_gu, n_units, perm, weight,
                tok_scale, table, expert_bytes(c.d, c.f), gateup_block_bytes(c.d, c.f), hp, out, abort, status,
                INT_MAX, ws + L.sfa, ws + L.sfa_dn, reinterpret_cast<uint8_t *>(hp)};
    // an upper bound on the items: every slot its own expert
    const int max_tiles = (int)std::min<long long>((long long)T * k + (long long)(E + S), (long long)1 << 30);
    if (!mx) {
        err = launch_gemm<kGU>(ga, mb_routed, mb_shared, ma1, ma3, max_tiles * (c.f / kTileRows), s, "gemm_gateup");
        if (err != cudaSuccess) return err;
    } else {
        // the shared experts' items (the first S ceil(T/128) rb of the gate/up items) on the
        // f16 kernel, then the routed ones on the block-scaled kernel
        const int shared_items = S * ((T + kBM - 1) / kBM) * (c.f / kTileRows);
        if (S > 0) {
            GemmArgs gs = ga;
            gs.item_hi = shared_items;
            err = launch_gemm<kGU>(gs, mb_shared, mb_shared, ma1, ma3, shared_items, s, "gemm_gateup");
            if (err != cudaSuccess) return err;
        }
        CUtensorMap mw1{}, mw3{};
        if (!map4(&mw1, table + mx_w1_offset(E, c.d, c.f), (uint64_t)E * c.f, c.d) ||
            !map4(&mw3, table + mx_w3_offset(E, c.d, c.f), (uint64_t)E * c.f, c.d))
            return cudaErrorInvalidValue;
        err = launch_gemm_mx<kGU>(ga, shared_items, mhi, mlo, mw1, mw3, max_tiles * (c.f / kTileRows), s,
                                  "gemm_gateup_mx");
        if (err != cudaSuccess) return err;
    }
    GemmArgs gd = ga;
    gd.prefix = prefix_dn;
    const int rb_dn = (c.d / kTileRows + 1) / 2;
    if (!mx) return launch_gemm<kDN>(gd, mb_h, mb_h, ma2, ma2, max_tiles * rb_dn, s, "gemm_down");
    // block-scaled: the shared experts' down items on the f16 kernel, the routed ones (h as
    // the two e4m3 planes the gate/up epilogue wrote in hp's routed rows) on the block-scaled one
    const int shared_dn = S * ((T + kBM - 1) / kBM) * rb_dn;
    if (S > 0) {
        GemmArgs gs = gd;
        gs.item_hi = shared_dn;
        err = launch_gemm<kDN>(gs, mb_h, mb_h, ma2, ma2, shared_dn, s, "gemm_down");
        if (err != cudaSuccess) return err;
    }
    CUtensorMap mhh{}, mhl{}, mw2{};
    uint8_t *hq = reinterpret_cast<uint8_t *>(hp);
    if (!map8(&mhh, hq, (uint64_t)T * k, c.f, kBM) || !map8(&mhl, hq + (size_t)T * k * c.f, (uint64_t)T * k, c.f, kBM) ||
        !map4(&mw2, table + mx_w2_offset(E, c.d, c.f), (uint64_t)E * c.d, c.f))
        return cudaErrorInvalidValue;
    return launch_gemm_mx<kDN>(gd, shared_dn, mhh, mhl, mw2, mw2, max_tiles * rb_dn, s, "gemm_down_mx");
}

}  // namespace k3moe
