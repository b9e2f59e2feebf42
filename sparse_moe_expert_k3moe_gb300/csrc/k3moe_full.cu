// k3moe_full.cu -- the full-width Stable LatentMoE block around the routed-expert
// layer, in the order of the six steps of the k3_moe listing (kimi-k3-in-c README,
// Part II, section 9 "Picking 16 experts of 896"):
//   1. route on the full-width token h (width H): the layer's router kernels, fed a
//      config whose width is H;
//   2. z = Wd h: into the expert latent;
//   3. a = sum_j w_j FFN_j(z): the layer's expert kernels on z, without shared experts;
//   4. a = a * gain / sqrt(mean(a^2) + eps): the RMSNorm of the AGGREGATE (never of one
//      expert), when the block asks for it;
//   5. out = Wu a: back to full width;
//   6. out += Sh2 SiTU(Sh1 h, Sh3 h): the shared experts on the ORIGINAL token, fused to
//      one FFN of width S*f, added with weight one.
// Steps 2, 5 and 6's projections run on the dense tensor-core kernel (k3moe_dense.cu):
// bf16 operands, fp32 accumulation; z, the normed aggregate and the shared SiTU output
// are rounded to bf16 as they become the next projection's operand.  The norm is a
// kernel here.
// Step 6 reads only h, so it runs beside steps 1-4 on a side stream: forked from the
// caller's stream where the call begins, it stores Sh2 SiTU(...) into out, and step 5,
// after the join, adds Wu a to it (one rounding of the same two terms either way).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

// ---------------------------------------------------------------------------------- kernels
constexpr int kNormThreads = 256;

// One block per token: y = bf16(a * gain / sqrt(sum(a^2) / d + eps)) when norm, else
// bf16(a).  The sum of squares is taken in a fixed order (per thread, then per warp by
// shuffles, then over the warps), so the result does not vary from run to run.
__global__ void __launch_bounds__(kNormThreads) latent_norm_kernel(int d, int norm, float eps,
                                                                  const float *__restrict__ a,
                                                                  const float *__restrict__ gain,
                                                                  uint16_t *__restrict__ y)
{
    pdl_wait();
    pdl_trigger();
    __shared__ float part[kNormThreads / 32];
    const float *ar = a + (size_t)blockIdx.x * d;
    uint16_t *yr = y + (size_t)blockIdx.x * d;
    float r = 1.0f;
    if (norm) {
        float ss = 0.0f;
        for (int i = threadIdx.x; i < d; i += kNormThreads) ss = fmaf(ar[i], ar[i], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; w++) tot += part[w];
        r = 1.0f / sqrtf(tot / (float)d + eps);
    }
    for (int i = threadIdx.x; i < d; i += kNormThreads) {
        float v = ar[i] * r;
        if (norm) v *= gain[i];
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        yr[i] = *reinterpret_cast<const uint16_t *>(&b);
    }
}

// One side stream per device with its fork and join events, created on first use outside
// a stream capture (a call made while its stream is capturing, before the device has one,
// runs step 6 on the caller's stream instead).  Calls enqueue under one lock, so two host
// threads never interleave their fork and join.
constexpr int kMaxSideDevices = 64;
struct Side {
    bool tried;
    cudaStream_t s;
    cudaEvent_t fork, join;
};
Side g_side[kMaxSideDevices];
std::mutex g_side_mu;

Side *side_stream(cudaStream_t caller)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
    Side &sd = g_side[dev];
    if (sd.s) return &sd;
    if (sd.tried) return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    sd.tried = true;
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return nullptr;
    if (cudaEventCreateWithFlags(&f, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) != cudaSuccess) {
        if (f) cudaEventDestroy(f);
        cudaStreamDestroy(st);
        return nullptr;
    }
    sd.fork = f;
    sd.join = j;
    sd.s = st;
    return &sd;
}

}  // namespace

cudaError_t launch_full(const k3moe_config &c, int hidden, int latent_norm, float rms_eps, int T,
                        const uint16_t *h, const uint16_t *wr, const float *bias, const uint16_t *wd,
                        const uint8_t *table, const float *gain, const uint16_t *wu,
                        const uint16_t *sh1, const uint16_t *sh3, const uint16_t *sh2, int32_t *idx,
                        float *weight, int32_t *offsets, int32_t *perm, float *out, uint8_t *ws,
                        const FullLayout &F, cudaStream_t s)
{
    const int d = c.d, H = hidden, SI = c.n_shared * c.f;
    uint16_t *z = reinterpret_cast<uint16_t *>(ws + F.z);
    float *acc = reinterpret_cast<float *>(ws + F.acc);
    uint16_t *y = reinterpret_cast<uint16_t *>(ws + F.y);
    float *part = reinterpret_cast<float *>(ws + F.part);
    int32_t *ctr = reinterpret_cast<int32_t *>(ws + F.ctr);
    int32_t *status = reinterpret_cast<int32_t *>(ws + F.route.status);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + F.act);
    std::lock_guard<std::mutex> lk(g_side_mu);
    Side *sd = SI > 0 ? side_stream(s) : nullptr;
    cudaError_t es = cudaSuccess;
    if (sd) {
        // 6. the shared experts on the original token, from where the caller's stream is,
        // into out (stored; step 5 adds to it): their own partials and counters
        float *part2 = reinterpret_cast<float *>(ws + F.part2);
        int32_t *ctr2 = reinterpret_cast<int32_t *>(ws + F.ctr2);
        es = cudaEventRecord(sd->fork, s);
        if (es != cudaSuccess) return es;
        es = cudaStreamWaitEvent(sd->s, sd->fork, 0);
        if (es != cudaSuccess) return es;
        es = launch_dense(kDenseSitu, T, SI, H, h, sh1, sh3, act, c.situ_b1, c.situ_b2, part2, ctr2, status, sd->s,
                          "full_shared_gateup");
        if (es == cudaSuccess)
            es = launch_dense(kDenseF32, T, H, SI, act, sh2, nullptr, out, 0.0f, 0.0f, part2, ctr2, status, sd->s,
                              "full_shared_down");
        // joined back in every case, so a capture of the caller's stream stays whole
        const cudaError_t ej = cudaEventRecord(sd->join, sd->s);
        if (es == cudaSuccess) es = ej;
    }
    auto join = [&](cudaError_t e) -> cudaError_t {
        if (sd) {
            const cudaError_t ew = cudaStreamWaitEvent(s, sd->join, 0);
            if (e == cudaSuccess) e = es != cudaSuccess ? es : ew;
        }
        return e;
    };
    // 1. route on the full-width token
    cudaError_t e = launch_route(F.cr, T, h, wr, bias, idx, weight, offsets, perm, ws, F.route, s);
    if (e != cudaSuccess) return join(e);
    // 2. into the expert latent
    e = launch_dense(kDenseBf16, T, d, H, h, wd, nullptr, z, 0.0f, 0.0f, part, ctr, status, s, "full_down_proj");
    if (e != cudaSuccess) return join(e);
    // 3. the chosen experts, summed with their weights
    e = launch_forward(F.cl, T, z, idx, weight, offsets, perm, table, nullptr, nullptr, nullptr, acc, ws,
                       F.latent, s, /*x_is_input=*/false);    // z is written just before
    if (e != cudaSuccess) return join(e);
    // 4. RMSNorm of the aggregate
    timing_begin("latent_norm", s);
    e = launch_pdl(latent_norm_kernel, dim3(T), dim3(kNormThreads), 0, s, d, latent_norm, rms_eps,
                   (const float *)acc, gain, y);
    count_launch();
    timing_end("latent_norm", s);
    if (e != cudaSuccess) return join(e);
    // 5. back to full width: added to the shared experts' out after the join
    e = join(cudaSuccess);
    if (e != cudaSuccess) return e;
    e = launch_dense(sd ? kDenseAddF32 : kDenseF32, T, H, d, y, wu, nullptr, out, 0.0f, 0.0f, part, ctr, status, s,
                     "full_up_proj");
    if (e != cudaSuccess || SI == 0 || sd) return e != cudaSuccess ? e : cudaGetLastError();
    // 6. without a side stream: the shared experts after step 5, added with weight one
    e = launch_dense(kDenseSitu, T, SI, H, h, sh1, sh3, act, c.situ_b1, c.situ_b2, part, ctr, status, s,
                     "full_shared_gateup");
    if (e != cudaSuccess) return e;
    e = launch_dense(kDenseAddF32, T, H, SI, act, sh2, nullptr, out, 0.0f, 0.0f, part, ctr, status, s,
                     "full_shared_down");
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace k3moe
