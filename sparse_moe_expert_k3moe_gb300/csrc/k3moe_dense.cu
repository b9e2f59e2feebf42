// k3moe_dense.cu -- the dense projections of the full-width block (kimi-k3-in-c README,
// Part II, section 9 "Picking 16 experts of 896", the k3_moe listing: step 2 z = Wd h,
// step 5 out = Wu a, step 6 the fused shared experts Sh1, Sh3 and Sh2):
//   y[t][n] = epilogue(sum_k x[t][k] W[n][k]),  x [T][K] and W [N][K] bf16 (rows = outputs),
// fp32 accumulation on the tensor cores (tcgen05, operands staged by TMA).
//
// Swap AB: M = 128 weight rows (a row block), N = a tile of up to 256 tokens (a multiple
// of 16; 128 for the gated form, which keeps two accumulators), K in 64-column stages.  A
// work item is (row block, token tile, K part).  Few tokens leave few items (28 row blocks
// of Wd at T = 1), so K is cut into P parts until the items fill the GPU: each part
// stores its fp32 partial sums, and for each 32-row quadrant of the row block the last
// part to finish adds the P partials in order p = 0..P-1 and applies the epilogue -- a
// fixed order, so results do not vary from run to run.  With one part the epilogue
// reads the accumulators directly.
//
// Epilogues: bf16 store (z), f32 store (out), f32 add (out += Sh2 act: every element
// belongs to one item, so a plain read-modify-write), and the gated form: two matrices W1
// and W3 with one accumulator each, y = bf16(SiTU(g, u)) with g = W1 x, u = W3 x.
//
// Warp roles, one persistent block per SM: warp 0 TMA producer, warp 1 MMA issue, warps
// 2-5 epilogue (one weight row per thread, 32x32b tensor-memory loads).  Every wait is
// bounded; a timeout sets the status word, the roles drop out, copies in flight land and
// the tensor memory is freed before the block leaves.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "k3moe_internal.cuh"
#include "k3moe_tc.cuh"

namespace k3moe {
namespace {

constexpr int kDnBM = 128, kDnBK = 64;
constexpr int kDnABytes = kDnBM * kDnBK * 2;                  // one weight tile: 16 KB
constexpr int kDnSmemBudget = 200 * 1024;                      // the stage ring
constexpr int kDnMaxStg = 8;
constexpr int kDnWarpProd = 0, kDnWarpMma = 1, kDnWarpEpi0 = 2, kDnNumEpi = 4;
constexpr int kDnThreads = (kDnWarpEpi0 + kDnNumEpi) * 32;     // 192
constexpr int kDnTmemCols = 512;

struct DenseArgs {
    int T, N, K, epi;
    int bn, P, n_rb, n_tt, nkp, kb, nstg, stage_bytes;
    float b1, b2;
    void *y;
    float *part;                   // [P][mats][T][N] partial sums (P > 1)
    int32_t *ctr;                  // [n_rb][n_tt][4] arrival counters (P > 1), back at zero after
    int32_t *status;
};

__device__ __forceinline__ float situ_f(float g, float u, float b1, float b2)
{
    const float a = b1 * tanhf(g / b1) * (1.0f / (1.0f + expf(-g)));
    return a * (b2 * tanhf(u / b2));
}

// Output element (t, n) from its sum (and the up sum for the gated form).
__device__ __forceinline__ void dense_store(const DenseArgs &a, int t, int n, float v, float u)
{
    const size_t o = (size_t)t * a.N + n;
    if (a.epi == kDenseBf16 || a.epi == kDenseSitu) {
        const float r = a.epi == kDenseSitu ? situ_f(v, u, a.b1, a.b2) : v;
        const __nv_bfloat16 b = __float2bfloat16_rn(r);
        reinterpret_cast<uint16_t *>(a.y)[o] = *reinterpret_cast<const uint16_t *>(&b);
    } else if (a.epi == kDenseF32) {
        reinterpret_cast<float *>(a.y)[o] = v;
    } else {
        reinterpret_cast<float *>(a.y)[o] += v;
    }
}

__global__ void __launch_bounds__(kDnThreads, 1) dense_tc_kernel(const DenseArgs a,
                                                                 const __grid_constant__ CUtensorMap mw,
                                                                 const __grid_constant__ CUtensorMap mw3,
                                                                 const __grid_constant__ CUtensorMap mx)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t dsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t full[kDnMaxStg], empty[kDnMaxStg], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int bail;

    const bool gated = a.epi == kDenseSitu;
    const int mats = gated ? 2 : 1;
    const int n_items = a.n_rb * a.n_tt * a.P, nstg = a.nstg;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < nstg; s++) { mb_init(&full[s], 1); mb_init(&empty[s], 1); }
        for (int b = 0; b < 2; b++) { mb_init(&acc_full[b], 1); mb_init(&acc_empty[b], kDnNumEpi); }
        mb_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    if (warp == kDnWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base)),
                     "r"(kDnTmemCols));
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
    // item i -> K part, token tile, row block: the token tiles of one row block are
    // consecutive, so the blocks working at once share a few row blocks' weights (read
    // from DRAM once, then from L2) and the tokens (which fit L2) are re-read from L2
    auto part_of = [&](int i) { return i % a.P; };
    auto tt_of = [&](int i) { return (i / a.P) % a.n_tt; };
    auto rb_of = [&](int i) { return i / (a.P * a.n_tt); };

    if (warp == kDnWarpProd) {
        if (lane == 0) {
            uint32_t st = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x) {
                const int p = part_of(i), rb = rb_of(i), t0 = tt_of(i) * a.bn;
                for (int ks = p * a.nkp; ks < (p + 1) * a.nkp; ks++, st++) {
                    const int s = st % nstg;
                    if (st >= (uint32_t)nstg && !mb_wait(&empty[s], ((st / nstg) - 1) & 1u)) {
                        timeout();
                        break;
                    }
                    // a stage is kb boxes of 64 columns: weight box (m, b) at (m kb + b) 16 KB,
                    // token box b after the weights at b bn 128 bytes
                    // one copy per box: the token box is a.bn rows (rows past T read as zero)
                    uint8_t *stage = sm + (size_t)s * a.stage_bytes;
                    mb_expect_tx(&full[s], (uint32_t)(a.kb * (mats * kDnABytes + a.bn * kDnBK * 2)));
                    uint8_t *bs = stage + mats * a.kb * kDnABytes;
                    for (int b = 0; b < a.kb; b++) {
                        const int k0 = (ks * a.kb + b) * kDnBK;
                        tma2d(stage + b * kDnABytes, &mw, k0, rb * kDnBM, &full[s]);
                        if (gated) tma2d(stage + (a.kb + b) * kDnABytes, &mw3, k0, rb * kDnBM, &full[s]);
                        tma2d(bs + (size_t)b * a.bn * 128, &mx, k0, t0, &full[s]);
                    }
                }
            }
            if (bail)   // wait (bounded) for the copies already issued
                for (uint32_t f = st > (uint32_t)nstg ? st - nstg : 0; f < st; f++)
                    mb_wait(&full[f % nstg], (f / nstg) & 1u);
        }
    } else if (warp == kDnWarpMma) {
        if (lane == 0) {
            uint32_t st = 0, n = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
                const int p = part_of(i), t0 = tt_of(i) * a.bn;
                const int bn = (min(a.bn, a.T - t0) + 15) & ~15;
                const uint32_t id = idesc(1, bn);
                const int buf = n & 1;
                if (n >= 2 && !mb_wait(&acc_empty[buf], ((n >> 1) - 1) & 1u)) { timeout(); break; }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)buf * 256u;        // gated: g at d0, u at d0 + 128
                for (int ks = p * a.nkp; ks < (p + 1) * a.nkp; ks++, st++) {
                    const int s = st % nstg;
                    if (!mb_wait(&full[s], (st / nstg) & 1u)) { timeout(); break; }
                    tc_fence_after();
                    const uint8_t *stage = sm + (size_t)s * a.stage_bytes;
                    const uint32_t A = saddr(stage), B0 = saddr(stage + mats * a.kb * kDnABytes);
                    const bool first = ks == p * a.nkp;
                    for (int b = 0; b < a.kb; b++) {
                        const uint32_t Ab = A + b * kDnABytes, Bb = B0 + b * a.bn * 128;
#pragma unroll
                        for (int kk = 0; kk < kDnBK / 16; kk++) {
                            const uint32_t acc = (!first || b || kk) ? 1u : 0u;
                            umma(d0, sdesc(Ab + kk * 32), sdesc(Bb + kk * 32), id, acc);
                            if (gated) umma(d0 + 128u, sdesc(Ab + a.kb * kDnABytes + kk * 32), sdesc(Bb + kk * 32), id, acc);
                        }
                    }
                    umma_commit(&empty[s]);
                }
                if (bail) break;
                umma_commit(&acc_full[buf]);
            }
            umma_commit(&drain);                       // every issued MMA done before the dealloc
            mb_wait(&drain, 0);
        }
    } else {
        // ---------------- epilogue: weight row 32q + lane of the row block per thread
        const int q = warp & 3;                         // tensor-memory lane quadrant of this warp
        const int row = 32 * q + lane;
        uint32_t n = 0;
        for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
            const int p = part_of(i), rb = rb_of(i), tt = tt_of(i), t0 = tt * a.bn;
            const int ncols = min(a.bn, a.T - t0);
            const int bn = (ncols + 15) & ~15;
            const int nr = rb * kDnBM + row;             // output column n of this thread
            const int buf = n & 1;
            if (!mb_wait_warp(&acc_full[buf], (n >> 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 256u;
            for (int c0 = 0; c0 < bn; c0 += 16) {
                float v[16], u[16];
                tmem_ld16(lane_addr + c0, v);
                if (gated) tmem_ld16(lane_addr + 128u + c0, u);
                if (a.P == 1 && a.epi == kDenseAddF32) {
                    // every old value is loaded before any is stored (loads in flight together)
                    float *yb = reinterpret_cast<float *>(a.y) + (size_t)(t0 + c0) * a.N + nr;
                    float old[16];
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) old[jj] = c0 + jj < ncols ? yb[(size_t)jj * a.N] : 0.0f;
#pragma unroll
                    for (int jj = 0; jj < 16; jj++)
                        if (c0 + jj < ncols) yb[(size_t)jj * a.N] = old[jj] + v[jj];
                    continue;
                }
#pragma unroll
                for (int jj = 0; jj < 16; jj++) {
                    const int t = t0 + c0 + jj;
                    if (c0 + jj >= ncols) break;
                    if (a.P == 1) {
                        dense_store(a, t, nr, v[jj], gated ? u[jj] : 0.0f);
                    } else {
                        float *pp = a.part + (((size_t)p * mats) * a.T + t) * a.N + nr;
                        pp[0] = v[jj];
                        if (gated) pp[(size_t)a.T * a.N] = u[jj];
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mb_arrive(&acc_empty[buf]);
            if (a.P > 1) {
                // the last of the P parts of this quadrant adds the partials in order
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    int32_t *c = a.ctr + ((size_t)rb * a.n_tt + tt) * 4 + q;
                    last = atomicAdd(c, 1) == a.P - 1;
                    if (last) *c = 0;
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    __threadfence();
                    for (int c = 0; c < ncols; c++) {
                        const int t = t0 + c;
                        // every part's value is loaded before any is added (loads in flight together)
                        float pv[kDenseMaxParts], pu[kDenseMaxParts];
#pragma unroll
                        for (int pp = 0; pp < kDenseMaxParts; pp++) {
                            pv[pp] = pu[pp] = 0.0f;
                            if (pp < a.P) {
                                const float *src = a.part + (((size_t)pp * mats) * a.T + t) * a.N + nr;
                                pv[pp] = __ldcg(src);
                                if (gated) pu[pp] = __ldcg(src + (size_t)a.T * a.N);
                            }
                        }
                        float sv = 0.0f, su = 0.0f;
#pragma unroll
                        for (int pp = 0; pp < kDenseMaxParts; pp++)
                            if (pp < a.P) {
                                sv += pv[pp];
                                su += pu[pp];
                            }
                        dense_store(a, t, nr, sv, su);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kDnWarpMma) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kDnTmemCols));
    }
}

// ---------------------------------------------------------------- few tokens: row streaming
// With at most kDenseRowsMaxT tokens the projection is a mat-vec bound by the weight
// stream.  One warp per output row at a time: the row (and for the gated form the same
// row of W3) read with 16-byte loads, eight in flight per lane -- whole contiguous rows,
// which the DRAM serves better than the tensor-core kernel's 128-row boxes -- against the
// tokens held in shared memory; fp32 products summed per lane in chunk order, then over
// the warp by a fixed butterfly, so results repeat bit for bit.
constexpr int kRowsThreads = 256;

template <int NT>
__global__ void __launch_bounds__(kRowsThreads) dense_rows_kernel(const DenseArgs a, const uint16_t *__restrict__ x,
                                                                 const uint16_t *__restrict__ w,
                                                                 const uint16_t *__restrict__ w3)
{
    pdl_wait();
    pdl_trigger();
    extern __shared__ __align__(16) uint4 xsm[];         // NT x K bf16
    const int nchunk = a.K / 8;
    const bool gated = a.epi == kDenseSitu;
    for (int q = threadIdx.x; q < NT * nchunk; q += kRowsThreads) {
        const int t = q / nchunk, c = q % nchunk;
        xsm[q] = t < a.T ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * a.K) + c) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = gridDim.x * (kRowsThreads / 32);
    for (int n = blockIdx.x * (kRowsThreads / 32) + warp; n < a.N; n += nw) {
        const uint4 *wr = reinterpret_cast<const uint4 *>(w + (size_t)n * a.K);
        const uint4 *wr3 = reinterpret_cast<const uint4 *>((gated ? w3 : w) + (size_t)n * a.K);
        float acc[NT], accu[NT];
#pragma unroll
        for (int t = 0; t < NT; t++) acc[t] = accu[t] = 0.0f;
        for (int c0 = lane; c0 < nchunk; c0 += 32 * 8) {
            uint4 wv[8], uv[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int c = c0 + 32 * j;
                wv[j] = c < nchunk ? __ldg(wr + c) : make_uint4(0, 0, 0, 0);
                uv[j] = gated && c < nchunk ? __ldg(wr3 + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const int c = c0 + 32 * j;
                if (c >= nchunk) break;
                const uint32_t wu[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
                const uint32_t uu[4] = {uv[j].x, uv[j].y, uv[j].z, uv[j].w};
#pragma unroll
                for (int t = 0; t < NT; t++) {
                    const uint4 xv = xsm[t * nchunk + c];
                    const uint32_t xu[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int r = 0; r < 4; r++) {
                        const float x0 = __uint_as_float(xu[r] << 16), x1 = __uint_as_float(xu[r] & 0xFFFF0000u);
                        acc[t] = fmaf(x0, __uint_as_float(wu[r] << 16), acc[t]);
                        acc[t] = fmaf(x1, __uint_as_float(wu[r] & 0xFFFF0000u), acc[t]);
                        if (gated) {
                            accu[t] = fmaf(x0, __uint_as_float(uu[r] << 16), accu[t]);
                            accu[t] = fmaf(x1, __uint_as_float(uu[r] & 0xFFFF0000u), accu[t]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < NT; t++) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
                accu[t] += __shfl_xor_sync(0xffffffffu, accu[t], o);
            }
            if (lane == 0 && t < a.T) dense_store(a, t, n, acc[t], accu[t]);
        }
    }
}

}  // namespace

DensePlan dense_plan(int T, int N, int K, int epi)
{
    DensePlan pl{};
    const bool gated = epi == kDenseSitu;
    const int bn_max = gated ? 128 : 256;
    pl.bn = T >= bn_max ? bn_max : std::max(16, (T + 15) & ~15);
    pl.n_tt = (T + pl.bn - 1) / pl.bn;
    pl.n_rb = N / kDnBM;
    pl.mats = gated ? 2 : 1;
    // stages of two 64-column boxes when one box would make a small stage (one weight
    // matrix, few tokens): half the barrier round trips per byte
    pl.kb = (!gated && pl.bn <= 64 && (K / kDnBK) % 2 == 0) ? 2 : 1;
    const int nks = K / (kDnBK * pl.kb);
    pl.P = 1;
    // few items: cut K until they fill the GPU (kDenseTargetItems), at least 4 stages a
    // part, at most kDenseMaxParts parts and kDensePartRows partial rows (P * T)
    while ((long long)pl.n_rb * pl.n_tt * pl.P * 2 <= kDenseTargetItems && nks % (2 * pl.P) == 0 &&
           nks / (2 * pl.P) >= 4 && 2 * pl.P <= kDenseMaxParts && (long long)2 * pl.P * T <= kDensePartRows)
        pl.P *= 2;
    pl.nkp = nks / pl.P;
    pl.stage_bytes = pl.kb * (pl.mats * kDnABytes + pl.bn * kDnBK * 2);
    pl.nstg = std::min(kDnMaxStg, kDnSmemBudget / pl.stage_bytes);
    return pl;
}

bool dense_applies(int N, int K) { return N % kDnBM == 0 && K % kDnBK == 0; }

cudaError_t launch_dense(int epi, int T, int N, int K, const uint16_t *x, const uint16_t *w,
                         const uint16_t *w3, void *y, float b1, float b2, float *part, int32_t *ctr,
                         int32_t *status, cudaStream_t s, const char *name)
{
    if (T <= 0) return cudaSuccess;
    if (!dense_applies(N, K)) return cudaErrorInvalidValue;
    if (T <= kDenseRowsMaxT) {
        DenseArgs a{T, N, K, epi, 0, 1, 0, 0, 0, 1, 0, 0, b1, b2, y, part, ctr, status};
        const int nt = T <= 1 ? 1 : (T <= 2 ? 2 : 4);
        const size_t smem = (size_t)nt * K * 2;
        static size_t smem_set[3] = {0, 0, 0};
        auto kern = nt == 1 ? dense_rows_kernel<1> : (nt == 2 ? dense_rows_kernel<2> : dense_rows_kernel<4>);
        const int ki = nt == 1 ? 0 : (nt == 2 ? 1 : 2);
        if (smem > smem_set[ki]) {
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            smem_set[ki] = smem;
        }
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRowsThreads, smem) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        const int grid = std::max(1, std::min(num_sms() * per_sm, (N + kRowsThreads / 32 - 1) / (kRowsThreads / 32)));
        timing_begin(name, s);
        const cudaError_t err = launch_pdl(kern, dim3(grid), dim3(kRowsThreads), smem, s, a, x, w, w3);
        count_launch();
        timing_end(name, s);
        return err;
    }
    const DensePlan pl = dense_plan(T, N, K, epi);
    CUtensorMap mw{}, mw3{}, mx{};
    if (!map16(&mw, w, (uint64_t)N, (uint64_t)K, kDnBM) ||
        !map16(&mw3, epi == kDenseSitu ? w3 : w, (uint64_t)N, (uint64_t)K, kDnBM) ||
        !map16(&mx, x, (uint64_t)T, (uint64_t)K, (uint32_t)pl.bn))
        return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)pl.nstg * pl.stage_bytes;
    static size_t smem_set = 0;
    if (smem > smem_set) {
        cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        smem_set = smem;
    }
    DenseArgs a{T, N, K, epi, pl.bn, pl.P, pl.n_rb, pl.n_tt, pl.nkp, pl.kb, pl.nstg, pl.stage_bytes, b1, b2,
                y, part, ctr, status};
    const int n_items = pl.n_rb * pl.n_tt * pl.P;
    const int grid = std::max(1, std::min(num_sms(), n_items));
    timing_begin(name, s);
    const cudaError_t err = launch_pdl(dense_tc_kernel, dim3(grid), dim3(kDnThreads), smem, s, a, mw, mw3, mx);
    count_launch();
    timing_end(name, s);
    return err;
}

}  // namespace k3moe
