// k3moe_route_tc.cu -- approximate router logits on the tensor cores, for many tokens
// (kimi-k3-in-c README, Part II, section 9 "Picking 16 experts of 896": the router
// logits are the dot products of the token with each expert's bf16 router row).
//
// logits[t][e] = x[t] . Wr[e] is a plain bf16 GEMM with fp32 accumulation.  The tensor
// cores' accumulation is coarser than fp32 addition (measured within 2^-22 |x_t| |Wr[e]|),
// so these logits only bracket the exact ones: the top-k kernel re-scores exactly every
// expert they cannot rule out.  Swap AB again: M = 128 router rows (experts), N = up to 256
// tokens, K = d.  One work item = one (128-expert block, 256-token tile); items are
// walked token tile by token tile so the blocks reading one x tile run together.
// Warp roles: warp 0 TMA producer (A box 64 x 128 rows, B boxes 64 x 16), warp 1
// tcgen05.mma issue (bf16, fp32 accumulators, two 256-column buffers), warps 2-5
// epilogue: the logits, stored [T][E].  Every wait is bounded; a timeout sets the status
// word and the roles drop out.
#include <cuda.h>

#include <algorithm>

#include "k3moe_internal.cuh"
#include "k3moe_tc.cuh"

namespace k3moe {
namespace {

constexpr int kRtBM = 128, kRtBK = 64, kRtBN = 256, kRtStg = 4;
constexpr int kRtABytes = kRtBM * kRtBK * 2, kRtBBytes = kRtBN * kRtBK * 2;
constexpr int kRtSmem = kRtStg * (kRtABytes + kRtBBytes) + 1024;
constexpr int kRtWarpProd = 0, kRtWarpMma = 1, kRtWarpEpi0 = 2, kRtNumEpi = 4;
constexpr int kRtThreads = (kRtWarpEpi0 + kRtNumEpi) * 32;   // 192
constexpr int kRtTmemCols = 512;

struct RtArgs {
    int T, d, E;
    int bnx;                // rows of the token box: min(256, T rounded up to 16)
    float *logit;
    int32_t *status;
};

__global__ void __launch_bounds__(kRtThreads, 1) router_logits_tc_kernel(const RtArgs a,
                                                                         const __grid_constant__ CUtensorMap mwr,
                                                                         const __grid_constant__ CUtensorMap mx)
{
    // the logits need nothing from the kernel before (the row-norm kernel, launched first,
    // which waited for the previous call): start at once, and wait for it only before
    // leaving, so that the top-k's wait on this grid covers both
    pdl_trigger();
    extern __shared__ __align__(1024) uint8_t rsm_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(rsm_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *smA = sm, *smB = sm + kRtStg * kRtABytes;
    __shared__ uint64_t full[kRtStg], empty[kRtStg], acc_full[2], acc_empty[2], drain;
    __shared__ uint32_t tmem_base;
    __shared__ int bail;

    const int n_eb = (a.E + kRtBM - 1) / kRtBM, n_tt = (a.T + kRtBN - 1) / kRtBN;
    const int n_items = n_eb * n_tt, nks = a.d / kRtBK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRtStg; s++) { mb_init(&full[s], 1); mb_init(&empty[s], 1); }
        for (int b = 0; b < 2; b++) { mb_init(&acc_full[b], 1); mb_init(&acc_empty[b], kRtNumEpi); }
        mb_init(&drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
    }
    if (warp == kRtWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tmem_base)),
                     "r"(kRtTmemCols));
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

    if (warp == kRtWarpProd) {
        if (lane == 0) {
            uint32_t st = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x) {
                const int eb = i % n_eb, t0 = (i / n_eb) * kRtBN;
                for (int ks = 0; ks < nks; ks++, st++) {
                    const int s = st % kRtStg;
                    if (st >= (uint32_t)kRtStg && !mb_wait(&empty[s], ((st / kRtStg) - 1) & 1u)) {
                        timeout();
                        break;
                    }
                    // one copy of the token box (a.bnx rows; rows past T read as zero)
                    mb_expect_tx(&full[s], (uint32_t)(kRtABytes + a.bnx * kRtBK * 2));
                    tma2d(smA + s * kRtABytes, &mwr, ks * kRtBK, eb * kRtBM, &full[s]);
                    tma2d(smB + s * kRtBBytes, &mx, ks * kRtBK, t0, &full[s]);
                }
            }
            if (bail)   // wait (bounded) for the copies already issued
                for (uint32_t f = st > (uint32_t)kRtStg ? st - kRtStg : 0; f < st; f++)
                    mb_wait(&full[f % kRtStg], (f / kRtStg) & 1u);
        }
    } else if (warp == kRtWarpMma) {
        if (lane == 0) {
            uint32_t st = 0, n = 0;
            for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
                const int t0 = (i / n_eb) * kRtBN;
                const int bn = (min(kRtBN, a.T - t0) + 15) & ~15;
                const uint32_t id = idesc(1, bn);
                const int buf = n & 1;
                if (n >= 2 && !mb_wait(&acc_empty[buf], ((n >> 1) - 1) & 1u)) { timeout(); break; }
                tc_fence_after();
                const uint32_t d0 = tmem + (uint32_t)buf * 256u;
                for (int ks = 0; ks < nks; ks++, st++) {
                    const int s = st % kRtStg;
                    if (!mb_wait(&full[s], (st / kRtStg) & 1u)) { timeout(); break; }
                    tc_fence_after();
                    const uint32_t A = saddr(smA + s * kRtABytes), B = saddr(smB + s * kRtBBytes);
#pragma unroll
                    for (int kk = 0; kk < kRtBK / 16; kk++)
                        umma(d0, sdesc(A + kk * 32), sdesc(B + kk * 32), id, (ks | kk) != 0);
                    umma_commit(&empty[s]);
                }
                if (bail) break;
                umma_commit(&acc_full[buf]);
            }
            umma_commit(&drain);                       // every issued MMA done before the dealloc
            mb_wait(&drain, 0);
        }
    } else {
        const int q = warp & 3;                         // TMEM lane quadrant of this warp
        const int row = 32 * q + lane;
        uint32_t n = 0;
        for (int i = blockIdx.x; i < n_items && !bail; i += gridDim.x, n++) {
            const int eb = i % n_eb, t0 = (i / n_eb) * kRtBN;
            const int ncols = min(kRtBN, a.T - t0);
            const int bn = (ncols + 15) & ~15;
            const int e = eb * kRtBM + row;
            const int buf = n & 1;
            if (!mb_wait(&acc_full[buf], (n >> 1) & 1u)) { timeout(); break; }
            tc_fence_after();
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)buf * 256u;
            for (int c0 = 0; c0 < bn; c0 += 16) {
                float v[16];
                tmem_ld16(lane_addr + c0, v);
                if (e < a.E) {
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) {
                        if (c0 + jj >= ncols) break;
                        a.logit[(size_t)(t0 + c0 + jj) * a.E + e] = v[jj];
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
    if (warp == kRtWarpMma) {
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kRtTmemCols));
    }
    if (threadIdx.x == 0) pdl_wait();
}

// The tensor-core kernels' bounded wait (mb_wait) on an mbarrier nothing arrives on,
// with the given limit: it gives up, and the kernel sets the status word's timeout bit
// as those kernels do.  For tests of that path.
__global__ void __launch_bounds__(32) wait_check_tc_kernel(int32_t *status, long long limit)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mb_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mb_wait(&bar, 0, limit)) set_status(status, K3MOE_DEV_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_wait_check_tc(int32_t *status, long long limit, cudaStream_t s)
{
    wait_check_tc_kernel<<<1, 32, 0, s>>>(status, limit);
    count_launch();
    return cudaGetLastError();
}

// the A box is 128 router rows: at least that many experts
bool router_tc_applies(const k3moe_config &c, int T)
{
    return T >= kRouterTcMinTokens && c.n_experts >= kRtBM && c.d % kRtBK == 0;
}

cudaError_t launch_router_logits_tc(const k3moe_config &c, int T, const uint16_t *x, const uint16_t *wr,
                                    float *logit, int32_t *status, cudaStream_t s)
{
    static bool set = false;
    if (!set) {
        cudaFuncSetAttribute(router_logits_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRtSmem);
        set = true;
    }
    CUtensorMap mwr{}, mx{};
    if (!map16(&mwr, wr, (uint64_t)c.n_experts, (uint64_t)c.d, kRtBM) ||
        !map16(&mx, x, (uint64_t)T, (uint64_t)c.d, (uint32_t)std::min(kRtBN, (T + 15) & ~15)))
        return cudaErrorInvalidValue;
    const int n_items = ((c.n_experts + kRtBM - 1) / kRtBM) * ((T + kRtBN - 1) / kRtBN);
    const int grid = std::max(1, std::min(num_sms(), n_items));
    RtArgs a{T, c.d, c.n_experts, std::min(kRtBN, (T + 15) & ~15), logit, status};
    const cudaError_t err = launch_pdl(router_logits_tc_kernel, dim3(grid), dim3(kRtThreads), kRtSmem, s, a, mwr, mx);
    count_launch();
    return err;
}

}  // namespace k3moe
