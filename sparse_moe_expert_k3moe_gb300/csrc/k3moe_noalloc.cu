// k3moe_noalloc.cu -- k3moe_forward_noalloc: the expert forward pass for callers
// that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs inside
// another framework's execution callback (a plugin's enqueue, an inference server's
// per-request hook) where only the inputs and outputs are handed over, and
// real-time or embedded callers with a fixed, pre-planned memory budget that forbids
// cudaMalloc on the serving path (it can implicitly synchronise the device and can
// fail under memory pressure in the middle of a request).  For them this entry point
// takes its scratch from a file-scope device array instead of a caller workspace.
//
// The array is a static __device__ object of kNoAllocScratchBytes: every GPU that
// loads the library holds it until the process exits.  Host code cannot use the
// array's name as a device address (in host code it is a host-side stand-in), so the
// first call on each device, with that device current, looks up its device address
// with cudaGetSymbolAddress and caches it together with the device's current context;
// make that first call before any stream capture.  Should the context be destroyed and
// created again (a device reset), the array gets a new address in the new context: the
// next call sees the changed context and looks the address up again.  All calls share the one array and it keeps the last call's contents: each
// call clears the status block that must start at zero, and calls that overlap on the
// GPU (different streams, no ordering between them) race on the array.
#include <cuda.h>

#include <mutex>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;   // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices] = {};
CUcontext g_noalloc_ctx[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The calling thread's current context (NULL before the runtime has set one up), through
// the driver entry point the runtime exposes.
cudaError_t current_context(CUcontext *ctx)
{
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return cudaErrorNotSupported;
        fn = reinterpret_cast<CtxGetCurrentFn>(p);
    }
    return fn(ctx) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of the scratch array on the current device, looked up once per device
// and context.
cudaError_t noalloc_scratch(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    CUcontext ctx = nullptr;                // NULL until the runtime has set up the device
    e = current_context(&ctx);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || !ctx || g_noalloc_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // sets up the context if needed
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        e = current_context(&ctx);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

bool is_aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace
}  // namespace k3moe

using namespace k3moe;

extern "C" k3moe_status k3moe_forward_noalloc(
    const k3moe_config *cfg, int32_t T, const uint16_t *x, const int32_t *idx, const float *weight,
    const int32_t *offsets, const int32_t *perm, const void *expert_table, size_t table_bytes,
    const uint16_t *sh_w1, const uint16_t *sh_w3, const uint16_t *sh_w2, float *out,
    int32_t *status_out, k3moe_stream stream)
{
    k3moe_status st = k3moe_validate_config(cfg);
    if (st != K3MOE_OK) return st;
    if (T < 0 || T > kMaxT) return K3MOE_ESHAPE;
    if (status_out && !is_aligned(status_out, 4)) return K3MOE_EALIGN;
    if (T == 0) {
        // nothing to compute; the status word still reports this call: clean
        if (status_out && cudaMemsetAsync(status_out, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess)
            return K3MOE_ECUDA;
        return K3MOE_OK;
    }
    if (!x || !idx || !weight || !offsets || !perm || !expert_table || !out) return K3MOE_EINVAL;
    if (cfg->n_shared > 0 && (!sh_w1 || !sh_w3 || !sh_w2)) return K3MOE_EINVAL;
    if (!is_aligned(x, 16) || !is_aligned(out, 16) || !is_aligned(expert_table, 256) ||
        !is_aligned(idx, 4) || !is_aligned(weight, 4) || !is_aligned(offsets, 4) ||
        !is_aligned(perm, 4) || (status_out && !is_aligned(status_out, 4)))
        return K3MOE_EALIGN;
    if (cfg->n_shared > 0 &&
        (!is_aligned(sh_w1, 16) || !is_aligned(sh_w3, 16) || !is_aligned(sh_w2, 16)))
        return K3MOE_EALIGN;
    if (table_bytes < packed_table_bytes(cfg->n_experts, cfg->d, cfg->f)) return K3MOE_ESHAPE;
    const WsLayout L = ws_layout(*cfg, T);
    if (L.total > kNoAllocScratchBytes) return K3MOE_EWORKSPACE;   // T too large for the array

    void *scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return K3MOE_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    if (cudaMemsetAsync(ws + L.status, 0, sizeof(StatusBlock), s) != cudaSuccess) return K3MOE_ECUDA;
    cudaError_t e = launch_forward(*cfg, T, x, idx, weight, offsets, perm,
                                        static_cast<const uint8_t *>(expert_table), sh_w1, sh_w3,
                                        sh_w2, out, ws, L, s);
    if (e != cudaSuccess) return K3MOE_ECUDA;
    if (status_out &&
        cudaMemcpyAsync(status_out, ws + L.status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) !=
            cudaSuccess)
        return K3MOE_ECUDA;
    return K3MOE_OK;
}
