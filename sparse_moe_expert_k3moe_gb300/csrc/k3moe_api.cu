// k3moe_api.cu -- the C ABI entry points: argument validation, workspace
// layout, path choice, launch accounting and timing.  Kernels live in the other
// files; nothing here computes on the host beyond bookkeeping.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "k3moe_internal.cuh"

namespace k3moe {

// ----------------------------------------------------------------------------------- accounting
static std::atomic<int64_t> g_launches{0};
static std::atomic<int> g_timing_on{0};

struct TimingEntry {
    int64_t launches = 0;
    double ms = 0.0;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending;
    cudaEvent_t open = nullptr;
};
static std::mutex g_tmu;
static std::map<std::string, TimingEntry> g_timing;
static std::vector<cudaEvent_t> g_event_pool;

static cudaEvent_t take_event()
{
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int> g_prefill_gemm{0};
int prefill_gemm_setting() { return g_prefill_gemm.load(std::memory_order_relaxed); }
// The default (setting 0) is the block-scaled GEMM: measured faster on the K3 shape at
// T = 4096 (routed gate/up 3.73 against 4.67 ms) and T = 16384.
bool prefill_gemm_block_scaled(const k3moe_config &c, int T)
{
    (void)c;
    (void)T;
    return prefill_gemm_setting() != 1;
}

void timing_begin(const char *name, cudaStream_t s)
{
    if (!g_timing_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_tmu);
    TimingEntry &t = g_timing[name];
    t.open = take_event();
    cudaEventRecord(t.open, s);
}

void timing_end(const char *name, cudaStream_t s)
{
    if (!g_timing_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lk(g_tmu);
    TimingEntry &t = g_timing[name];
    if (!t.open) return;
    cudaEvent_t e = take_event();
    cudaEventRecord(e, s);
    t.pending.emplace_back(t.open, e);
    t.open = nullptr;
    t.launches++;
}

// ----------------------------------------------------------------------------------- validation
static bool finite_pos(float v) { return std::isfinite(v) && v > 0.0f; }

static k3moe_status check_config(const k3moe_config *c)
{
    if (!c) return K3MOE_EINVAL;
    if (c->d <= 0 || c->f <= 0 || c->n_experts <= 0 || c->top_k <= 0 || c->group <= 0 ||
        c->n_shared < 0)
        return K3MOE_EINVAL;
    if (c->group != kGroup) return K3MOE_EINVAL;
    if (!finite_pos(c->situ_b1) || !finite_pos(c->situ_b2)) return K3MOE_EINVAL;
    if (c->renorm != 0 && c->renorm != 1) return K3MOE_EINVAL;
    if (!std::isfinite(c->routed_scale)) return K3MOE_EINVAL;
    if (c->top_k > c->n_experts) return K3MOE_EINVAL;
    if (c->d % kTileK || c->f % kTileK || c->d > kMaxWidth || c->f > kMaxWidth) return K3MOE_ESHAPE;
    if (c->n_experts > kMaxExperts || c->top_k > kMaxTopK || c->n_shared > kMaxShared)
        return K3MOE_ESHAPE;
    return K3MOE_OK;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The largest workspace any 0 <= T <= T_max needs.  Sizes grow with T within each
// forward path, with two exceptions: a single token on the mat-vec path also holds the
// split shared-expert partials, and the first T of the tensor-core path can need less
// than the last T of the mat-vec path.  So the maximum is at T = 1, at the last mat-vec
// T, or at T_max.  total(T) is the layout size of one call with T tokens.
template <typename Total>
static size_t max_total(const k3moe_config &c, int32_t T_max, Total total)
{
    size_t m = total(T_max);
    if (T_max >= 1) m = std::max(m, total(1));
    const int64_t first_gemm = std::max<int64_t>(32, (8LL * c.n_experts + c.top_k - 1) / c.top_k);
    const int64_t last_gemv = std::min<int64_t>(T_max, first_gemm - 1);
    if (last_gemv >= 1) m = std::max(m, total((int32_t)last_gemv));
    return m;
}

// The index check of k3moe_check_bounds: the guard the kernels use, with no access.
__global__ void check_bounds_kernel(int32_t *status, int32_t index, int32_t limit)
{
    (void)dguard(status, index >= 0 && index < limit);
}

}  // namespace k3moe

using namespace k3moe;

extern "C" {

const char *k3moe_strerror(k3moe_status s)
{
    switch (s) {
    case K3MOE_OK: return "ok";
    case K3MOE_EINVAL: return "invalid config field or argument";
    case K3MOE_ESHAPE: return "size outside what the call supports";
    case K3MOE_EALIGN: return "pointer lacks the required alignment";
    case K3MOE_EWORKSPACE: return "workspace missing, misaligned or too small";
    case K3MOE_ECUDA: return "CUDA runtime call failed";
    case K3MOE_EDEVICE: return "device status word reports an error";
    case K3MOE_ETIMEOUT: return "a bounded device-side wait gave up";
    }
    return "unknown status";
}

k3moe_status k3moe_validate_config(const k3moe_config *cfg) { return check_config(cfg); }

size_t k3moe_packed_bytes(const k3moe_config *cfg)
{
    if (check_config(cfg) != K3MOE_OK) return 0;
    return packed_table_bytes(cfg->n_experts, cfg->d, cfg->f);
}

k3moe_status k3moe_workspace_bytes(const k3moe_config *cfg, int32_t T_max, size_t *bytes)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (!bytes) return K3MOE_EINVAL;
    if (T_max < 0 || T_max > kMaxT) return K3MOE_ESHAPE;
    *bytes = max_total(*cfg, T_max, [&](int32_t T) { return ws_layout(*cfg, T).total; });
    return K3MOE_OK;
}

static k3moe_status pack_checks(const k3moe_config *cfg, int32_t lo, int32_t n, const void *p1,
                                const void *s1, const void *p3, const void *s3, const void *p2,
                                const void *s2, const void *table, size_t table_bytes)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (lo < 0 || n < 0 || (int64_t)lo + n > cfg->n_experts) return K3MOE_ESHAPE;
    if (n == 0) return K3MOE_OK;
    if (!p1 || !s1 || !p3 || !s3 || !p2 || !s2 || !table) return K3MOE_EINVAL;
    if (!aligned(p1, 16) || !aligned(p3, 16) || !aligned(p2, 16) || !aligned(table, 256))
        return K3MOE_EALIGN;
    if (table_bytes < packed_table_bytes(cfg->n_experts, cfg->d, cfg->f)) return K3MOE_ESHAPE;
    return K3MOE_OK;
}

k3moe_status k3moe_pack_mxfp4(const k3moe_config *cfg, int32_t expert_lo, int32_t n_in,
                              const uint8_t *w1_packed, const uint8_t *w1_scale,
                              const uint8_t *w3_packed, const uint8_t *w3_scale,
                              const uint8_t *w2_packed, const uint8_t *w2_scale, void *table,
                              size_t table_bytes, void *ws, k3moe_stream stream)
{
    k3moe_status st = pack_checks(cfg, expert_lo, n_in, w1_packed, w1_scale, w3_packed, w3_scale,
                                  w2_packed, w2_scale, table, table_bytes);
    if (st != K3MOE_OK || n_in == 0) return st;
    if (ws && !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    cudaError_t e = launch_pack(*cfg, expert_lo, n_in, w1_packed, w1_scale, w3_packed, w3_scale,
                                w2_packed, w2_scale, static_cast<uint8_t *>(table),
                                ws ? static_cast<int32_t *>(ws) : nullptr, (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

k3moe_status k3moe_unpack_mxfp4(const k3moe_config *cfg, int32_t expert_lo, int32_t n_out,
                                const void *table, size_t table_bytes, uint8_t *w1_packed,
                                uint8_t *w1_scale, uint8_t *w3_packed, uint8_t *w3_scale,
                                uint8_t *w2_packed, uint8_t *w2_scale, k3moe_stream stream)
{
    k3moe_status st = pack_checks(cfg, expert_lo, n_out, w1_packed, w1_scale, w3_packed, w3_scale,
                                  w2_packed, w2_scale, table, table_bytes);
    if (st != K3MOE_OK || n_out == 0) return st;
    cudaError_t e = launch_unpack(*cfg, expert_lo, n_out, static_cast<const uint8_t *>(table),
                                  w1_packed, w1_scale, w3_packed, w3_scale, w2_packed, w2_scale,
                                  (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

k3moe_status k3moe_route(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                         const uint16_t *w_router, const float *bias, int32_t *idx, float *weight,
                         int32_t *offsets, int32_t *perm, void *ws, size_t ws_bytes,
                         k3moe_stream stream)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (T < 0 || T > kMaxT) return K3MOE_ESHAPE;
    if (!offsets) return K3MOE_EINVAL;
    if (T > 0 && (!x || !w_router || !idx || !weight || !perm)) return K3MOE_EINVAL;
    if (T > 0 && (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(idx, 4) ||
                  !aligned(weight, 4) || !aligned(perm, 4) || (bias && !aligned(bias, 4))))
        return K3MOE_EALIGN;
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    const WsLayout L = ws_layout(*cfg, T);
    if (ws_bytes < L.total) return K3MOE_EWORKSPACE;
    cudaError_t e = launch_route(*cfg, T, x, w_router, bias, idx, weight, offsets, perm,
                                 static_cast<uint8_t *>(ws), L, (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

k3moe_status k3moe_router_scores(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                                 const uint16_t *w_router, const float *bias, float *scores,
                                 float *choice, void *ws, size_t ws_bytes, k3moe_stream stream)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (T < 0 || T > kMaxT) return K3MOE_ESHAPE;
    if (T == 0) return K3MOE_OK;
    if (!x || !w_router || !scores || !choice) return K3MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(w_router, 16) || !aligned(scores, 4) || !aligned(choice, 4) ||
        (bias && !aligned(bias, 4)))
        return K3MOE_EALIGN;
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    const WsLayout L = ws_layout(*cfg, T);
    if (ws_bytes < L.total) return K3MOE_EWORKSPACE;
    cudaError_t e = launch_router_scores(*cfg, T, x, w_router, bias, scores, choice,
                                         reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + L.status),
                                         (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

k3moe_status k3moe_forward(const k3moe_config *cfg, int32_t T, const uint16_t *x,
                           const int32_t *idx, const float *weight, const int32_t *offsets,
                           const int32_t *perm, const void *expert_table, size_t table_bytes,
                           const uint16_t *sh_w1, const uint16_t *sh_w3, const uint16_t *sh_w2,
                           float *out, void *ws, size_t ws_bytes, k3moe_stream stream)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (T < 0 || T > kMaxT) return K3MOE_ESHAPE;
    if (T == 0) return K3MOE_OK;
    if (!x || !idx || !weight || !offsets || !perm || !expert_table || !out) return K3MOE_EINVAL;
    if (cfg->n_shared > 0 && (!sh_w1 || !sh_w3 || !sh_w2)) return K3MOE_EINVAL;
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(expert_table, 256) || !aligned(idx, 4) ||
        !aligned(weight, 4) || !aligned(offsets, 4) || !aligned(perm, 4))
        return K3MOE_EALIGN;
    if (cfg->n_shared > 0 && (!aligned(sh_w1, 16) || !aligned(sh_w3, 16) || !aligned(sh_w2, 16)))
        return K3MOE_EALIGN;
    if (table_bytes < packed_table_bytes(cfg->n_experts, cfg->d, cfg->f)) return K3MOE_ESHAPE;
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    const WsLayout L = ws_layout(*cfg, T);
    if (ws_bytes < L.total) return K3MOE_EWORKSPACE;
    cudaError_t e = launch_forward(*cfg, T, x, idx, weight, offsets, perm,
                                        static_cast<const uint8_t *>(expert_table), sh_w1, sh_w3,
                                        sh_w2, out, static_cast<uint8_t *>(ws), L, (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

static k3moe_status check_full(const k3moe_config *cfg, const k3moe_full_dims *fd)
{
    k3moe_status st = check_config(cfg);
    if (st != K3MOE_OK) return st;
    if (!fd || fd->hidden <= 0 || (fd->latent_norm != 0 && fd->latent_norm != 1) ||
        !finite_pos(fd->rms_eps))
        return K3MOE_EINVAL;
    if (fd->hidden % kTileK || fd->hidden > kMaxWidth) return K3MOE_ESHAPE;
    return K3MOE_OK;
}

k3moe_status k3moe_full_workspace_bytes(const k3moe_config *cfg, const k3moe_full_dims *fd,
                                        int32_t T_max, size_t *bytes)
{
    k3moe_status st = check_full(cfg, fd);
    if (st != K3MOE_OK) return st;
    if (!bytes) return K3MOE_EINVAL;
    if (T_max < 0 || T_max > kMaxT) return K3MOE_ESHAPE;
    *bytes = max_total(*cfg, T_max, [&](int32_t T) { return full_layout(*cfg, fd->hidden, T).total; });
    return K3MOE_OK;
}

k3moe_status k3moe_full_forward(const k3moe_config *cfg, const k3moe_full_dims *fd, int32_t T,
                                const uint16_t *h, const uint16_t *w_router, const float *bias,
                                const uint16_t *w_down, const void *expert_table,
                                size_t table_bytes, const float *norm_gain,
                                const uint16_t *w_up, const uint16_t *sh_w1,
                                const uint16_t *sh_w3, const uint16_t *sh_w2, int32_t *idx,
                                float *weight, int32_t *offsets, int32_t *perm, float *out,
                                void *ws, size_t ws_bytes, k3moe_stream stream)
{
    k3moe_status st = check_full(cfg, fd);
    if (st != K3MOE_OK) return st;
    if (T < 0 || T > kMaxT) return K3MOE_ESHAPE;
    if (!offsets) return K3MOE_EINVAL;
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    const FullLayout F = full_layout(*cfg, fd->hidden, T);
    if (ws_bytes < F.total) return K3MOE_EWORKSPACE;
    if (T == 0) {
        // no tokens: the routing is empty, exactly as k3moe_route leaves it
        cudaError_t e = launch_route(F.cr, 0, h, w_router, bias, idx, weight, offsets, perm,
                                     static_cast<uint8_t *>(ws), F.route, (cudaStream_t)stream);
        return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
    }
    if (!h || !w_router || !w_down || !expert_table || !w_up || !idx || !weight || !perm || !out ||
        (fd->latent_norm && !norm_gain))
        return K3MOE_EINVAL;
    if (cfg->n_shared > 0 && (!sh_w1 || !sh_w3 || !sh_w2)) return K3MOE_EINVAL;
    if (!aligned(h, 16) || !aligned(w_router, 16) || !aligned(w_down, 16) || !aligned(w_up, 16) ||
        !aligned(out, 16) || !aligned(expert_table, 256) || !aligned(idx, 4) || !aligned(weight, 4) ||
        !aligned(offsets, 4) || !aligned(perm, 4) || (bias && !aligned(bias, 4)) ||
        (norm_gain && !aligned(norm_gain, 4)))
        return K3MOE_EALIGN;
    if (cfg->n_shared > 0 && (!aligned(sh_w1, 16) || !aligned(sh_w3, 16) || !aligned(sh_w2, 16)))
        return K3MOE_EALIGN;
    if (table_bytes < packed_table_bytes(cfg->n_experts, cfg->d, cfg->f)) return K3MOE_ESHAPE;
    cudaError_t e = launch_full(*cfg, fd->hidden, fd->latent_norm, fd->rms_eps, T, h, w_router, bias,
                                w_down, static_cast<const uint8_t *>(expert_table), norm_gain, w_up,
                                sh_w1, sh_w3, sh_w2, idx, weight, offsets, perm, out,
                                static_cast<uint8_t *>(ws), F, (cudaStream_t)stream);
    return e == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

k3moe_status k3moe_device_status(void *ws, k3moe_stream stream, int32_t *code)
{
    if (!ws || !aligned(ws, 256) || !code) return K3MOE_EINVAL;
    int32_t v = 0;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return K3MOE_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_ECUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), s) != cudaSuccess) return K3MOE_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return K3MOE_ECUDA;
    *code = v;
    if (v & K3MOE_DEV_TIMEOUT) return K3MOE_ETIMEOUT;
    return (v & K3MOE_DEV_ERROR_MASK) ? K3MOE_EDEVICE : K3MOE_OK;
}

k3moe_status k3moe_check_wait_timeout(void *ws, int64_t limit_cycles, k3moe_stream stream)
{
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    if (limit_cycles < 1 || limit_cycles > 4000000000ll) return K3MOE_ESHAPE;
    int32_t *status = static_cast<int32_t *>(ws);
    cudaStream_t s = (cudaStream_t)stream;
    if (launch_wait_check_gemv(status, limit_cycles, s) != cudaSuccess) return K3MOE_ECUDA;
    if (launch_wait_check_tc(status, limit_cycles, s) != cudaSuccess) return K3MOE_ECUDA;
    return K3MOE_OK;
}

k3moe_status k3moe_check_bounds(void *ws, int32_t index, int32_t limit, k3moe_stream stream)
{
    if (!ws || !aligned(ws, 256)) return K3MOE_EWORKSPACE;
    if (limit < 1) return K3MOE_ESHAPE;
    cudaStream_t s = (cudaStream_t)stream;
    check_bounds_kernel<<<1, 1, 0, s>>>(static_cast<int32_t *>(ws), index, limit);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? K3MOE_OK : K3MOE_ECUDA;
}

int32_t k3moe_build_flags(void)
{
#ifdef K3MOE_DEBUG
    return K3MOE_BUILD_DEBUG;
#else
    return 0;
#endif
}

int64_t k3moe_launch_count(void) { return g_launches.load(); }

k3moe_status k3moe_set_prefill_gemm(int32_t variant)
{
    if (variant < 0 || variant > 2) return K3MOE_EINVAL;
    g_prefill_gemm.store(variant, std::memory_order_relaxed);
    return K3MOE_OK;
}

int32_t k3moe_get_prefill_gemm(void) { return prefill_gemm_setting(); }

void k3moe_timing_enable(int32_t on) { g_timing_on.store(on ? 1 : 0); }

int32_t k3moe_timing_read(const char **names, int64_t *launches, double *ms, int32_t cap)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    int32_t n = 0;
    for (auto &kv : g_timing) {
        TimingEntry &t = kv.second;
        for (auto &pr : t.pending) {
            float v = 0.0f;
            cudaEventSynchronize(pr.second);
            if (cudaEventElapsedTime(&v, pr.first, pr.second) == cudaSuccess) t.ms += v;
            g_event_pool.push_back(pr.first);
            g_event_pool.push_back(pr.second);
        }
        t.pending.clear();
        if (n < cap) {
            if (names) names[n] = kv.first.c_str();
            if (launches) launches[n] = t.launches;
            if (ms) ms[n] = t.ms;
        }
        n++;
    }
    return n;
}

void k3moe_timing_reset(void)
{
    std::lock_guard<std::mutex> lk(g_tmu);
    for (auto &kv : g_timing) {
        for (auto &pr : kv.second.pending) {
            cudaEventSynchronize(pr.second);
            g_event_pool.push_back(pr.first);
            g_event_pool.push_back(pr.second);
        }
        kv.second.pending.clear();
        kv.second.launches = 0;
        kv.second.ms = 0.0;
    }
}

}  // extern "C"
