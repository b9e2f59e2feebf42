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
// Steps 2, 5 and 6's three projections are plain dense bf16 GEMMs (fp32 accumulation)
// and run on cuBLASLt, which is loaded at first use so that the rest of the library
// does not depend on it.  The norm and the SiTU are kernels here; each rounds its
// output to bf16, the GEMMs' operand type.
#include <cublasLt.h>
#include <dlfcn.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>

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

// act = bf16(SiTU(gate, up)) elementwise over n values (n a multiple of 4):
// b1 tanh(g/b1) sigmoid(g) * b2 tanh(u/b2), the sigmoid on the uncapped gate.
__global__ void __launch_bounds__(256) shared_situ_kernel(size_t n, float b1, float b2,
                                                         const float *__restrict__ gate,
                                                         const float *__restrict__ up,
                                                         uint16_t *__restrict__ act)
{
    pdl_wait();
    pdl_trigger();
    for (size_t q = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q < n / 4;
         q += (size_t)gridDim.x * blockDim.x) {
        const float4 g = reinterpret_cast<const float4 *>(gate)[q];
        const float4 u = reinterpret_cast<const float4 *>(up)[q];
        const float gv[4] = {g.x, g.y, g.z, g.w}, uv[4] = {u.x, u.y, u.z, u.w};
        uint16_t o[4];
#pragma unroll
        for (int j = 0; j < 4; j++) {
            const float s = b1 * tanhf(gv[j] / b1) * (1.0f / (1.0f + expf(-gv[j])));
            const __nv_bfloat16 b = __float2bfloat16_rn(s * (b2 * tanhf(uv[j] / b2)));
            o[j] = *reinterpret_cast<const uint16_t *>(&b);
        }
        reinterpret_cast<uint2 *>(act)[q] =
            make_uint2((uint32_t)o[0] | ((uint32_t)o[1] << 16), (uint32_t)o[2] | ((uint32_t)o[3] << 16));
    }
}

// ---------------------------------------------------------------------------------- cuBLASLt
// The entry points this file uses, looked up in the shared library at first use.
struct Lt {
    bool ok = false;
    cublasLtHandle_t handle = nullptr;
    decltype(&cublasLtCreate) create = nullptr;
    decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
    decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
    decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
    decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
    decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
    decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
    decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
    decltype(&cublasLtMatmul) matmul = nullptr;
};

template <typename F>
bool sym(void *so, const char *name, F &fn)
{
    fn = reinterpret_cast<F>(dlsym(so, name));
    return fn != nullptr;
}

Lt &lt()
{
    static Lt L;
    static std::once_flag once;
    std::call_once(once, [] {
        // the soname first (a copy already loaded in the process, or the loader's
        // search path), then the toolkit's own directory
        const char *names[] = {"libcublasLt.so.13", "libcublasLt.so", "/usr/local/cuda/lib64/libcublasLt.so.13"};
        void *so = nullptr;
        for (const char *n : names)
            if ((so = dlopen(n, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
        if (!so) return;
        const bool all = sym(so, "cublasLtCreate", L.create) &&
                         sym(so, "cublasLtMatmulDescCreate", L.desc_create) &&
                         sym(so, "cublasLtMatmulDescSetAttribute", L.desc_set) &&
                         sym(so, "cublasLtMatrixLayoutCreate", L.layout_create) &&
                         sym(so, "cublasLtMatmulPreferenceCreate", L.pref_create) &&
                         sym(so, "cublasLtMatmulPreferenceSetAttribute", L.pref_set) &&
                         sym(so, "cublasLtMatmulPreferenceDestroy", L.pref_destroy) &&
                         sym(so, "cublasLtMatmulAlgoGetHeuristic", L.heuristic) &&
                         sym(so, "cublasLtMatmul", L.matmul);
        L.ok = all && L.create(&L.handle) == CUBLAS_STATUS_SUCCESS;
    });
    return L;
}

// One GEMM shape's descriptors and chosen algorithm, made once and kept (one plan per
// distinct token count T, a few hundred bytes each).
struct Plan {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, d = nullptr;
    cublasLtMatmulAlgo_t algo{};
    bool made = false, ok = false;
};

// D [n][m] (row-major) = B [n][k] . A^T (+ D when accumulate): each of the n token rows
// of B times the weight matrix A [m][k] (row-major, out x in), fp32 accumulation; D is
// bf16 or f32.  In cuBLASLt's column-major terms D (m x n) = op_T(A: k x m) . B (k x n).
cudaError_t lt_gemm(int m, int n, int k, const uint16_t *A, const uint16_t *B, void *D, bool d_f32,
                    bool accumulate, void *ws, size_t ws_bytes, cudaStream_t s, const char *name)
{
    Lt &L = lt();
    if (!L.ok) return cudaErrorSharedObjectInitFailed;
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, bool, bool>, Plan> plans;
    Plan *p;
    {
        std::lock_guard<std::mutex> lk(mu);
        p = &plans[std::make_tuple(m, n, k, d_f32, accumulate)];
        if (!p->made) {
            p->made = true;
            const cudaDataType_t dt = d_f32 ? CUDA_R_32F : CUDA_R_16BF;
            const cublasOperation_t opT = CUBLAS_OP_T, opN = CUBLAS_OP_N;
            bool ok = L.desc_create(&p->op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS &&
                      L.desc_set(p->op, CUBLASLT_MATMUL_DESC_TRANSA, &opT, sizeof(opT)) == CUBLAS_STATUS_SUCCESS &&
                      L.desc_set(p->op, CUBLASLT_MATMUL_DESC_TRANSB, &opN, sizeof(opN)) == CUBLAS_STATUS_SUCCESS &&
                      L.layout_create(&p->a, CUDA_R_16BF, k, m, k) == CUBLAS_STATUS_SUCCESS &&
                      L.layout_create(&p->b, CUDA_R_16BF, k, n, k) == CUBLAS_STATUS_SUCCESS &&
                      L.layout_create(&p->d, dt, m, n, m) == CUBLAS_STATUS_SUCCESS;
            cublasLtMatmulPreference_t pref = nullptr;
            ok = ok && L.pref_create(&pref) == CUBLAS_STATUS_SUCCESS;
            const uint64_t wsb = ws_bytes;
            ok = ok && L.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)) ==
                           CUBLAS_STATUS_SUCCESS;
            cublasLtMatmulHeuristicResult_t res{};
            int nres = 0;
            ok = ok && L.heuristic(L.handle, p->op, p->a, p->b, p->d, p->d, pref, 1, &res, &nres) ==
                           CUBLAS_STATUS_SUCCESS && nres > 0;
            if (pref) L.pref_destroy(pref);
            p->algo = res.algo;
            p->ok = ok;
        }
    }
    if (!p->ok) return cudaErrorNotSupported;
    const float alpha = 1.0f, beta = accumulate ? 1.0f : 0.0f;
    timing_begin(name, s);
    const cublasStatus_t st = L.matmul(L.handle, p->op, &alpha, A, p->a, B, p->b, &beta, D, p->d, D, p->d,
                                       &p->algo, ws, ws_bytes, s);
    timing_end(name, s);
    return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorLaunchFailure;
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
    void *ltws = ws + F.lt;
    // 1. route on the full-width token
    cudaError_t e = launch_route(F.cr, T, h, wr, bias, idx, weight, offsets, perm, ws, F.route, s);
    if (e != cudaSuccess) return e;
    // 2. into the expert latent
    e = lt_gemm(d, T, H, wd, h, z, false, false, ltws, kLtWorkspace, s, "full_down_gemm");
    if (e != cudaSuccess) return e;
    // 3. the chosen experts, summed with their weights
    e = launch_forward(F.cl, T, z, idx, weight, offsets, perm, table, nullptr, nullptr, nullptr, acc, ws,
                       F.latent, s, /*x_is_input=*/false);    // z is written just before
    if (e != cudaSuccess) return e;
    // 4. RMSNorm of the aggregate
    timing_begin("latent_norm", s);
    e = launch_pdl(latent_norm_kernel, dim3(T), dim3(kNormThreads), 0, s, d, latent_norm, rms_eps,
                   (const float *)acc, gain, y);
    count_launch();
    timing_end("latent_norm", s);
    if (e != cudaSuccess) return e;
    // 5. back to full width
    e = lt_gemm(H, T, d, wu, y, out, true, false, ltws, kLtWorkspace, s, "full_up_gemm");
    if (e != cudaSuccess) return e;
    if (SI == 0) return cudaGetLastError();
    // 6. the shared experts on the original token, added with weight one
    float *gate = reinterpret_cast<float *>(ws + F.gate), *up = reinterpret_cast<float *>(ws + F.up);
    uint16_t *act = reinterpret_cast<uint16_t *>(ws + F.act);
    e = lt_gemm(SI, T, H, sh1, h, gate, true, false, ltws, kLtWorkspace, s, "full_shared_gate_gemm");
    if (e != cudaSuccess) return e;
    e = lt_gemm(SI, T, H, sh3, h, up, true, false, ltws, kLtWorkspace, s, "full_shared_up_gemm");
    if (e != cudaSuccess) return e;
    const size_t n = (size_t)T * SI;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 1;
    const int grid = (int)std::max<size_t>(1, std::min<size_t>((n / 4 + 255) / 256, (size_t)sms * 8));
    timing_begin("shared_situ", s);
    e = launch_pdl(shared_situ_kernel, dim3(grid), dim3(256), 0, s, n, c.situ_b1, c.situ_b2,
                   (const float *)gate, (const float *)up, act);
    count_launch();
    timing_end("shared_situ", s);
    if (e != cudaSuccess) return e;
    e = lt_gemm(H, T, SI, sh2, act, out, true, true, ltws, kLtWorkspace, s, "full_shared_down_gemm");
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace k3moe
