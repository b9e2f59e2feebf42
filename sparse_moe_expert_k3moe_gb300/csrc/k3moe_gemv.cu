// k3moe_gemv.cu -- the expert part of the layer as grouped, streamed mat-vecs: the
// decode path (few tokens per expert).  kimi-k3-in-c README, Part II, section 4 (MXFP4
// mat-vec: per-32 partial sums times the E8M0 scale, nothing dequantised to memory)
// and section 9 (the k3_moe expert loop: gate = w1, up = w3, SiTU-GLU, down = w2,
// weighted sum; shared experts unweighted).
//
// Kernels, in launch order:
//   fwd_prep     validates offsets/perm against idx, lists the active experts, inverts
//                perm (slot -> position), picks each token's activation scale 2^-u and
//                writes x * 2^-u as f16; sets the abort flag on bad input;
//   gemv_gateup  for every (active expert, token) and (shared expert, token): g = W1 x,
//                u = W3 x, h = SiTU(g, u), stored as f16 (routed) or a bf16 hi + lo
//                pair (shared);
//   gemv_down    y = W2 h, fp32, one row per (slot or shared expert, token); for up to
//                three tokens it does not wait for the whole gate/up grid: each item waits for
//                its unit's h rows, which the gate/up warps publish (per-unit counters,
//                release / acquire), so down items stream while gate/up's last items run;
//   fwd_combine  out[t] = sum_j w[t][j] y[pos(t,j)] + sum_s y_shared[s][t], terms added
//                in a fixed order.
//
// Arithmetic: a streamed mat-vec is bound by HBM bandwidth, so the inner loop must stay
// cheap.  The tensor-core warp MMA (m16n8k16) serves as the multiply-add engine: each
// 16x16 MXFP4 sub-tile is decoded with the hardware e2m1x2 -> f16x2 conversion (exact;
// the table layout hands every lane its fragment bytes in one 8-byte load), multiplied
// against the activations in f16 and accumulated in fp32, one 32-column group at a time;
// the group's E8M0 scale multiplies the fp32 group result (converted by the hardware
// ue8m0 conversion, or exactly for the rare expert whose table flags a scale byte 0 or
// 255).  Activations enter f16 with a
// per-token power-of-two scale that puts the token's largest magnitude in [2^14, 2^15):
// every bf16 element within 2^31 of that maximum converts exactly.  The SiTU output
// enters the routed down projection as f16 (as on the tensor-core path).  The bf16
// shared experts use bf16 MMAs on tensor-map (TMA) tiles, with h as a bf16 hi + lo pair.
//
// Streaming: a persistent grid, two blocks per SM; work items (128 weight rows of one
// unit over the whole K) are handed out longest first through an atomic counter.  In
// each block one producer warp moves everything by bulk async copies and never waits for
// data: the weight stages (a packed W1+W3 tile pair for gate/up, two consecutive packed
// W2 tiles for down, or a bf16 tile through a tensor map) through a 4-stage mbarrier
// ring, and the B operand (the tokens' activations or h rows, one copy per token row) in
// chunks through two alternating slots.  Eight consumer warps each own rows 16w..16w+15
// of the item and never synchronise the block.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

constexpr int kThreads = 256;
constexpr int kItemRows = 128;
constexpr int kStages = 4;                         // weight-stage ring depth
constexpr int kNBMax = 2;                          // n-blocks of 8 tokens per pass
constexpr int kPassTok = 8 * kNBMax;
constexpr int kSharedK = 64;                       // K per stage for bf16 tiles (one matrix)
constexpr int kBSlots = 2;                         // staged B operands (double buffer)
constexpr long long kWaitCycles = 4000000000ll;      // bounded waits: ~2 s at 2 GHz

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
// Returns false when the bounded wait gave up (a clock limit, checked every 32 polls).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit = kWaitCycles)
{
    const uint32_t a = smem_addr(bar);
    {   // fast path: the phase is often complete already
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
    }
    const long long t0 = clock64();
    for (uint32_t i = 0;; i++) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(a), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 31u) == 31u && clock64() - t0 > limit) return false;
    }
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
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
// Orders this thread's earlier generic-proxy accesses (an acquire of data other SMs
// wrote) before its later bulk copies, which read global memory through the async proxy.
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }
__device__ __forceinline__ int ld_acquire(const int32_t *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed(const int32_t *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_acq_rel() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
// Waits (bounded, with short sleeps) until *p >= want; false when the limit ran out.
__device__ __forceinline__ bool wait_at_least(const int32_t *p, int want, long long limit = kWaitCycles)
{
    if (ld_acquire(p) >= want) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(200);
        if (ld_acquire(p) >= want) return true;
        if (clock64() - t0 > limit) return false;
    }
}
// Publishes what this warp stored: every lane's release fence, then lane 0 adds n to *p.
__device__ __forceinline__ void publish_add(int32_t *p, int n, int lane)
{
    fence_acq_rel();
    __syncwarp();
    if (lane == 0) atomicAdd(p, n);
}

// Four packed bytes -> four f16x2 (each byte: low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t &h0, uint32_t &h1,
                                                uint32_t &h2, uint32_t &h3)
{
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(w));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1, const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1, const float (&c)[4])
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
          "f"(c[2]), "f"(c[3]));
}
// Shared-memory operand reads at 32-bit shared addresses (the stage buffers' addresses are
// taken once per stage; the per-fragment offsets are immediates).
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t a)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ uint32_t lds32(uint32_t a)
{
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a)
{
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}

__device__ __forceinline__ float situ(float g, float u, float b1, float b2)
{
    const float a = b1 * tanhf(g / b1) * (1.0f / (1.0f + expf(-g)));
    return a * (b2 * tanhf(u / b2));
}

// The four E8M0 scales of one row (one byte per group) as floats: the hardware
// ue8m0x2 -> bf16x2 conversion gives 2^(b-127) exactly for bytes 1..254; bf16 -> f32 is
// a shift.  Bytes 0 (a subnormal) and 255 (read as zero) need the exact path, which
// EXACT selects for experts whose table flags such a byte.
template <bool EXACT>
__device__ __forceinline__ void row_scales(uint32_t s4, float (&f)[4])
{
    const bool special = EXACT && (__vcmpeq4(s4, 0u) | __vcmpeq4(s4, 0xFFFFFFFFu)) != 0u;
    if (!special) {
        uint32_t lo, hi;
        asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
            "cvt.rn.bf16x2.ue8m0x2 %0, a;\n\tcvt.rn.bf16x2.ue8m0x2 %1, b;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(s4));
        f[0] = __uint_as_float(lo << 16);
        f[1] = __uint_as_float(lo & 0xFFFF0000u);
        f[2] = __uint_as_float(hi << 16);
        f[3] = __uint_as_float(hi & 0xFFFF0000u);
    } else {
#pragma unroll
        for (int c = 0; c < 4; c++) f[c] = e8m0_to_f32(s4 >> (8 * c));
    }
}

// -------------------------------------------------------------------------------- prep
struct PrepArgs {
    int T, E, k, d;
    const uint16_t *x;
    const int32_t *idx, *offsets, *perm;
    int32_t *active;     // [E + 1]
    int32_t *inv;        // [T * k]
    float *tok_scale;    // [2][T]
    uint16_t *xs;        // [T][d] f16: x * 2^-u per token (the routed experts' B operand)
    int32_t *status;
    int32_t *abort;
    int early;           // 1: x is complete at launch (its conversion need not wait)
};

// Block 0 validates the routing (offsets, idx and perm, through a copy of offsets in
// shared memory) and builds the active list and the inverse permutation; block b >= 1
// converts tokens [32(b-1), 32b): warp per token, its scale 2^-u (max|x_t| in [2^14, 2^15),
// u in [-113, 113]) and the f16 row x * 2^-u.  The kernel lets the gate/up kernel launch
// at once (its shared items need nothing from here); the token conversion reads only x,
// so when x is complete at launch it runs before the wait for the routing.
__global__ void __launch_bounds__(1024) fwd_prep_kernel(PrepArgs a)
{
    pdl_trigger();
    if (blockIdx.x == 0 || !a.early) pdl_wait();
    __shared__ int32_t bad;
    __shared__ int32_t scan_tmp[32];
    __shared__ int32_t off[kMaxExperts + 1];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = a.E, slots = a.T * a.k;
    if (blockIdx.x > 0) {
        const int t = (blockIdx.x - 1) * 32 + warp;
        if (t >= a.T) {
            if (lane == 0) pdl_wait();      // the grid completes after the routing did
            return;
        }
        const uint4 *row = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.d);
        const int n16 = a.d / 8;
        uint32_t m = 0;
        for (int q0 = lane; q0 < n16; q0 += 32 * 8) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; j++) {          // eight independent loads in flight
                const int q = q0 + 32 * j;
                v[j] = q < n16 ? row[q] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int h = 0; h < 4; h++) m = max(m, max(w4[h] & 0x7FFFu, (w4[h] >> 16) & 0x7FFFu));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        int u = 0;
        const int eb = (int)(m >> 7);                      // biased exponent of max|x_t|
        if (m != 0 && eb < 255) u = min(max(eb - 127 - 14, -113), 113);
        const float xin = __uint_as_float((uint32_t)(127 - u) << 23);
        if (lane == 0) {
            a.tok_scale[t] = xin;
            a.tok_scale[a.T + t] = __uint_as_float((uint32_t)(127 + u) << 23);
        }
        uint4 *dst = reinterpret_cast<uint4 *>(a.xs + (size_t)t * a.d);
        for (int q = lane; q < n16; q += 32) {
            const uint4 v = row[q];
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[4];
#pragma unroll
            for (int h = 0; h < 4; h++) {
                const __half2 h2 = __floats2half2_rn(__uint_as_float(w4[h] << 16) * xin,
                                                     __uint_as_float(w4[h] & 0xFFFF0000u) * xin);
                o[h] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            dst[q] = make_uint4(o[0], o[1], o[2], o[3]);
        }
        if (lane == 0) pdl_wait();          // the grid completes after the routing did
        return;
    }
    // with up to kPrepSlots slots, idx and perm are read into shared memory together with
    // offsets (one round of loads) and the inverse permutation is built there
    constexpr int kPrepSlots = 2048;
    __shared__ int32_t sidx[kPrepSlots], sperm[kPrepSlots], sinv[kPrepSlots];
    const bool small = slots <= kPrepSlots;
    if (tid == 0) bad = 0;
    for (int e = tid; e <= E; e += blockDim.x) off[e] = a.offsets[e];
    if (small) {
        for (int s = tid; s < slots; s += blockDim.x) {
            sidx[s] = a.idx[s];
            sperm[s] = a.perm[s];
            sinv[s] = -1;
        }
    } else {
        for (int s = tid; s < slots; s += blockDim.x) a.inv[s] = -1;
    }
    __syncthreads();
    const int32_t *pidx = small ? sidx : a.idx, *pperm = small ? sperm : a.perm;
    int32_t *pinv = small ? sinv : a.inv;
    // offsets: monotone, start 0, end T*k; idx in range
    for (int e = tid; e < E; e += blockDim.x) {
        const int lo = off[e], hi = off[e + 1];
        if (lo < 0 || hi < lo || hi > slots) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    }
    if (tid == 0 && (off[0] != 0 || off[E] != slots)) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
    for (int s = tid; s < slots; s += blockDim.x) {
        const int e = pidx[s];
        if (e < 0 || e >= E) atomicOr(&bad, K3MOE_DEV_BAD_INDEX);
    }
    __syncthreads();
    const bool offsets_ok = !(bad & K3MOE_DEV_BAD_OFFSETS);
    // active experts in ascending order (block scan over flags)
    int run = 0;
    for (int base = 0; base < E; base += blockDim.x) {
        const int e = base + tid;
        const int flag = (offsets_ok && e < E && off[e + 1] > off[e]) ? 1 : 0;
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
            const int s = pperm[p];
            if (s < 0 || s >= slots) {
                atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
                continue;
            }
            int lo = 0, hi = E;   // find e with off[e] <= p < off[e+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (off[mid] <= p) lo = mid; else hi = mid;
            }
            if (pidx[s] != lo) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
            if (atomicExch(&pinv[s], p) != -1) atomicOr(&bad, K3MOE_DEV_BAD_OFFSETS);
        }
    }
    __syncthreads();
    if (small)
        for (int s = tid; s < slots; s += blockDim.x) a.inv[s] = sinv[s];
    if (tid == 0) {
        if (bad) atomicOr(a.status, bad);
        *a.abort = bad ? 1 : 0;
        a.abort[2] = 0;                      // the down kernel's work counter (it starts after this)
    }
}

// -------------------------------------------------------------------------------- streamed mat-vec
struct GemvArgs {
    int T, d, f, k, S, E;
    int brows;                      // token rows of a staged B chunk: min(16, T)
    float b1, b2;
    const uint16_t *x, *xs;
    const int32_t *offsets, *perm, *active;
    const float *tok_scale;
    const uint8_t *table;
    size_t expert_bytes, gateup_bytes;
    float *ys;                      // y rows: slots, then per shared expert its K parts x T
    float *gush;                    // shared gate/up partials [parts][S][T][2][f]
    int32_t *shctr;                 // shared gate/up arrival counters [S][f/128]
    uint16_t *hp;                   // SiTU output planes: hi at [0], lo at [rows * f]
    const int32_t *abort;
    int32_t *status;
    int32_t *work;                  // [2] work counters: gate/up (reset by its last block), down (zeroed by fwd_prep)
    int32_t *exits;                 // gate/up blocks that have finished (reset by the last)
    int early;                      // 1: x is complete at launch (the gate/up shared items start at once)
    int32_t *ready;                 // [E + S] h rows published per unit (gate/up warps add, down reads)
    int32_t *route_seen;            // raised by gate/up once the routing is visible to it
    int32_t *dn_exits;              // down blocks that have finished (the last resets ready, route_seen)
    int32_t *gu_done;               // raised by the last gate/up block to finish (all h published)
};

// gate/up, after a wait for the routing: tells the down kernel that the routing (and
// what the forward's prep wrote) is visible; release, so an acquire of the flag carries it.
__device__ __forceinline__ void raise_route_seen(const GemvArgs &a)
{
    __threadfence();
    atomicExch(a.route_seen, 1);
}

struct Unit {         // one expert (routed or shared) with its tokens
    int shared;       // 0: routed expert e; 1: shared expert s
    int id;           // e or s
    int tok0, ntok;   // routed: positions [tok0, tok0+ntok) of perm; shared: tokens [0, T)
};

// u >= 0: the u-th active routed expert; u < 0: shared expert -1 - u.
__device__ __forceinline__ Unit unit_of(const GemvArgs &a, int u)
{
    Unit r;
    if (u >= 0) {
        r.shared = 0;
        r.id = dclamp(a.status, a.active[u], 0, a.E - 1);
        r.tok0 = a.offsets[r.id];
        r.ntok = a.offsets[r.id + 1] - r.tok0;
        dcheck(a.status, r.tok0 >= 0 && r.ntok >= 0 && r.tok0 + r.ntok <= a.T * a.k);
    } else {
        r.shared = 1;
        r.id = -1 - u;
        dcheck(a.status, r.id < a.S);
        r.tok0 = 0;
        r.ntok = a.T;
    }
    return r;
}

template <int MODE>
struct Geo {
    // stage bytes: a W1+W3 tile pair (gate/up) or up to two consecutive K tiles (down);
    // bf16 boxes fit in both (multiples of 1024 so every stage buffer meets the
    // swizzled-TMA alignment)
    static constexpr int kStageBytes = 2 * kTileBytes;
    // B operand staged in chunks of at most this many 128-column tiles (two chunk
    // buffers per block; down stages hi and lo halves)
    static constexpr int kChunkTilesMax = MODE == kGateUp ? 4 : 2;
    // bf16 stages carry one matrix: gate/up alternates W1 and W3 slices
    static constexpr int kSharedMats = MODE == kGateUp ? 2 : 1;
    __host__ __device__ static int rows(const GemvArgs &a) { return MODE == kGateUp ? a.f : a.d; }
    __host__ __device__ static int K(const GemvArgs &a) { return MODE == kGateUp ? a.d : a.f; }
    __host__ __device__ static int Psh(const GemvArgs &a)
    {
        return MODE == kGateUp ? shared_kparts(K(a) / kTileK, a.T) : 1;
    }
    // 128-column tiles per staged B chunk (the last chunk of K may be shorter)
    __host__ __device__ static int chunk_tiles(const GemvArgs &a)
    {
        const int kt = K(a) / kTileK;
        return kt < kChunkTilesMax ? kt : kChunkTilesMax;
    }
    // bytes between two token rows of a staged B chunk: 16 bytes of padding keep the
    // ldmatrix row reads of eight tokens on distinct banks
    __host__ __device__ static int b_row_bytes(const GemvArgs &a) { return chunk_tiles(a) * kTileK * 2 + 16; }
};

// A work item: 128 rows of one unit over the whole K, for passes [pass0, pass1).
struct Item {
    int u, rb, pass0, pass1;
    int kp, nkp;                    // K part of a shared item (routed: 0 of 1)
};
__device__ __forceinline__ int shared_passes(const GemvArgs &a) { return max(1, (a.T + kPassTok - 1) / kPassTok); }
// Shared items first: they depend on nothing the routing produces, so the gate/up kernel
// streams them while the router and the forward's prep are still running (it waits for
// them only before its first routed item), and a whole shared item (bf16, four times the
// bytes of a packed one) outlasts a routed one anyway.  A routed item holds all passes of
// its expert; a shared item one token pass (gate/up: one of P K parts).
template <int MODE>
__device__ __forceinline__ int n_shared_items(const GemvArgs &a)
{
    return a.S * shared_passes(a) * Geo<MODE>::Psh(a) * (Geo<MODE>::rows(a) / kItemRows);
}
template <int MODE>
__device__ __forceinline__ Item item_of(const GemvArgs &a, int i)
{
    const int nrb = Geo<MODE>::rows(a) / kItemRows;
    const int nsp = shared_passes(a), P = Geo<MODE>::Psh(a), n_sh = a.S * nsp * P * nrb;
    Item it;
    if (i < n_sh) {
        it.rb = i % nrb;
        int j = i / nrb;
        it.kp = j % P;
        it.nkp = P;
        j /= P;
        it.pass0 = j % nsp;
        it.pass1 = it.pass0 + 1;
        it.u = -1 - j / nsp;
    } else {
        const int j = i - n_sh;
        it.rb = j % nrb;
        it.u = j / nrb;
        it.kp = 0;
        it.nkp = 1;
        it.pass0 = 0;
        it.pass1 = -1;          // all passes of the unit
    }
    return it;
}
// TPS: K tiles per routed stage (gate/up 1: a W1+W3 pair; down 2 when K has an even
// number of tiles, else 1)
template <int MODE, int TPS>
__device__ __forceinline__ int n_stages(const GemvArgs &a, int shared)
{
    const int K = Geo<MODE>::K(a);
    return shared ? Geo<MODE>::kSharedMats * (K / Geo<MODE>::Psh(a) / kSharedK) : K / kTileK / TPS;
}
__device__ __forceinline__ int n_passes(const Unit &un) { return max(1, (un.ntok + kPassTok - 1) / kPassTok); }

// Row of the g/u/h and y buffers for token n of pass `pass` of unit `un`.
__device__ __forceinline__ size_t out_row(const GemvArgs &a, const Unit &un, int pass, int n)
{
    return un.shared ? (size_t)a.T * a.k + (size_t)un.id * a.T + pass * kPassTok + n
                     : (size_t)(un.tok0 + pass * kPassTok + n);
}
__device__ __forceinline__ int token_of(const GemvArgs &a, const Unit &un, int pass, int n)
{
    if (un.shared) return pass * kPassTok + n;
    const int slot = a.perm[un.tok0 + pass * kPassTok + n];
    return dclamp(a.status, slot, 0, a.T * a.k - 1) / a.k;
}

// Copies of one weight stage (thread 0 only).
template <int MODE, int TPS>
__device__ void issue_stage(const GemvArgs &a, const CUtensorMap *m1, const CUtensorMap *m3,
                            const CUtensorMap *m2, const Unit &un, const Item &it, int st,
                            uint8_t *buf, uint64_t *bar)
{
    if (!un.shared) {
        const uint8_t *ex = a.table + (size_t)un.id * a.expert_bytes;
        const int kt = st * TPS;
        if (MODE == kGateUp) {
            const int ktn = a.d / kTileK;
            mbar_expect_tx(bar, 2 * kTileBytes);
            bulk_g2s(buf, ex + ((size_t)it.rb * ktn + kt) * 2 * kTileBytes, 2 * kTileBytes, bar);
        } else {
            const int ktn = a.f / kTileK;           // the stage's TPS tiles are adjacent
            mbar_expect_tx(bar, TPS * kTileBytes);
            bulk_g2s(buf, ex + a.gateup_bytes + ((size_t)it.rb * ktn + kt) * kTileBytes, TPS * kTileBytes, bar);
        }
    } else {
        // one 64-column slice of one matrix; gate/up alternates W1 (even) and W3 (odd)
        const int slice = st / Geo<MODE>::kSharedMats;
        const int k0 = it.kp * (Geo<MODE>::K(a) / it.nkp) + slice * kSharedK;
        const CUtensorMap *m = MODE == kGateUp ? ((st & 1) ? m3 : m1) : m2;
        const int row = un.id * Geo<MODE>::rows(a) + it.rb * kItemRows;
        mbar_expect_tx(bar, kItemRows * kSharedK * 2);
        tma_2d_g2s(buf, m, k0, row, bar);
    }
}

// Per-pass token facts, computed once per pass into shared memory.
struct PassTok {
    int tok[kPassTok];        // token index t
    long long row[kPassTok];  // row of the g/u/h and y buffers
    float xin[kPassTok];      // activation multiplier (routed: 2^-u_t; shared: 1)
    float fo[kPassTok];       // output factor (routed: 2^u_t; shared: 1)
};

// B chunks in shared memory: token n's row of the chunk at n * b_row_bytes, 16-bit
// elements in K order (routed gate/up: f16 x * 2^-u; shared gate/up: bf16 x; down: the
// hi plane of h, and the lo plane in a second region).  The producer warp fills a chunk
// with one bulk copy per token row (lane n copies token n); rows of invalid tokens are
// left as they are: a column of the B operand only reaches the same column of the
// result, and those results are never stored.
template <int MODE>
__device__ __forceinline__ void issue_b_chunk(const GemvArgs &a, const Unit &un, const Item &it, int chunk,
                                              int nvalid, int tok, long long row, uint8_t *bhi, uint8_t *blo,
                                              int32_t *flag, uint64_t *bar, int lane)
{
    const int Kp = Geo<MODE>::K(a) / it.nkp, CT = Geo<MODE>::chunk_tiles(a);   // this item's K range
    const int RS = Geo<MODE>::b_row_bytes(a);
    const int c0 = chunk * CT * kTileK;                         // first column of the chunk
    const int cols = min(CT * kTileK, Kp - c0);
    const uint32_t row_bytes = (uint32_t)cols * 2;
    const int k0 = it.kp * Kp + c0;
    // down: a shared expert's h is a bf16 hi + lo pair; a routed expert's is one f16 plane
    const bool two = MODE == kDown && un.shared;
    // a routed expert's chunk also brings the last 16 trailer bytes, whose last word flags
    // scale bytes 0 and 255 in the expert (flag[3])
    const uint32_t fbytes = un.shared ? 0u : 16u;
    if (lane == 0) mbar_expect_tx(bar, (uint32_t)nvalid * row_bytes * (two ? 2u : 1u) + fbytes);
    __syncwarp();
    if (lane == 31 && fbytes)
        bulk_g2s(flag, a.table + special_flag_offset(a.E, a.d, a.f, un.id) - 12, fbytes, bar);
    if (lane < nvalid) {
        if (MODE == kGateUp) {
            const uint16_t *src = (un.shared ? a.x : a.xs) + (size_t)tok * a.d + k0;
            bulk_g2s(bhi + lane * RS, src, row_bytes, bar);
        } else {
            const size_t plane = ((size_t)a.T * a.k + (size_t)a.S * a.T) * a.f;
            const uint16_t *src = a.hp + (size_t)row * a.f + k0;
            bulk_g2s(bhi + lane * RS, src, row_bytes, bar);
            if (two) bulk_g2s(blo + lane * RS, src + plane, row_bytes, bar);
        }
    }
}

// One weight stage of warp `w` (rows 16w..16w+15 of the item).
// B fragments of k-steps ks, ks+1 for n-block nb from a row-major chunk: ldmatrix x4,
// lanes 8j..8j+7 address matrix j (tokens 8nb..8nb+7; columns 16ks + 8j .. +7).  A chunk
// holds `brows` token rows; the n-block's rows past them read the last row instead
// (their results are never stored), so every address stays inside the chunk.
__device__ __forceinline__ void ldb2(uint32_t (&r)[4], uint32_t b, int RS, int brows, int nb, int ks,
                                     int lane)
{
    const int m = lane >> 3;
    const int row = min(8 * nb + (lane & 7), brows - 1);
    ldmatrix_x4(r, b + (uint32_t)(row * RS + (16 * ks + 8 * m) * 2));
}

template <int MODE, int NB, int TPS, bool EXACT>
__device__ __forceinline__ void consume_stage(uint32_t buf0, int shared, int st, int RS, int brows, uint32_t bhi,
                                              uint32_t blo, int w, int lane, float (&acc1)[kNBMax][4],
                                              float (&acc3)[kNBMax][4])
{
    const int g = lane >> 2;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    if (!shared) {
#pragma unroll
      for (int tt = 0; tt < TPS; tt++) {
        const uint32_t buf = buf0 + tt * kTileBytes;
        const int ks0 = (st * TPS + tt) * 8;                  // 8 k-steps per 128-column tile
        float f1[4], f1b[4], f3[4], f3b[4];
        const uint32_t srow = buf + kTileNibbleBytes + (16 * w + g) * 4;
        row_scales<EXACT>(lds32(srow), f1);
        row_scales<EXACT>(lds32(srow + 32), f1b);
        if (MODE == kGateUp) {
            row_scales<EXACT>(lds32(srow + kTileBytes), f3);
            row_scales<EXACT>(lds32(srow + kTileBytes + 32), f3b);
        }
        const uint32_t wrow = buf + w * 1024 + 8 * lane;      // this lane's fragment bytes
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint2 wa = lds64(wrow + c * 256);
            uint32_t A0[4], A1[4];
            e2m1x8_to_f16x2(wa.x, A0[0], A0[2], A1[0], A1[2]);
            e2m1x8_to_f16x2(wa.y, A0[1], A0[3], A1[1], A1[3]);
            uint32_t C0[4], C1[4];
            if (MODE == kGateUp) {
                const uint2 wc = lds64(wrow + kTileBytes + c * 256);
                e2m1x8_to_f16x2(wc.x, C0[0], C0[2], C1[0], C1[2]);
                e2m1x8_to_f16x2(wc.y, C0[1], C0[3], C1[1], C1[3]);
            }
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                uint32_t bb[4];
                ldb2(bb, bhi, RS, brows, nb, ks0 + 2 * c, lane);
                float t1[4];
                mma_f16(t1, A0, bb[0], bb[1], zero);
                mma_f16(t1, A1, bb[2], bb[3], t1);
                acc1[nb][0] = fmaf(f1[c], t1[0], acc1[nb][0]);
                acc1[nb][1] = fmaf(f1[c], t1[1], acc1[nb][1]);
                acc1[nb][2] = fmaf(f1b[c], t1[2], acc1[nb][2]);
                acc1[nb][3] = fmaf(f1b[c], t1[3], acc1[nb][3]);
                if (MODE == kGateUp) {
                    float t3[4];
                    mma_f16(t3, C0, bb[0], bb[1], zero);
                    mma_f16(t3, C1, bb[2], bb[3], t3);
                    acc3[nb][0] = fmaf(f3[c], t3[0], acc3[nb][0]);
                    acc3[nb][1] = fmaf(f3[c], t3[1], acc3[nb][1]);
                    acc3[nb][2] = fmaf(f3b[c], t3[2], acc3[nb][2]);
                    acc3[nb][3] = fmaf(f3b[c], t3[3], acc3[nb][3]);
                }
            }
        }
      }
    } else if (!EXACT) {                                      // (shared units never take EXACT)
        // bf16 tile: 128 rows x 64 columns, 128-byte swizzle (chunk q of row r at
        // r*128 + ((q ^ (r&7))*16)); gate/up stages alternate W1 (even) and W3 (odd)
        const int mats = Geo<MODE>::kSharedMats;
        const int ks0 = (st / mats) * (kSharedK / 16);
        const bool up = MODE == kGateUp && (st & 1);
        const int r = 16 * w + (lane & 15);
#pragma unroll
        for (int kk = 0; kk < kSharedK / 16; kk += 2) {
            uint32_t A[2][4];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int q = 2 * (kk + h) + (lane >> 4);
                ldmatrix_x4(A[h], buf0 + (uint32_t)(r * 128 + ((q ^ (r & 7)) << 4)));
            }
#pragma unroll
            for (int nb = 0; nb < NB; nb++) {
                uint32_t bb[4];
                ldb2(bb, bhi, RS, brows, nb, ks0 + kk, lane);
                if (MODE == kDown) {
                    uint32_t ll[4];
                    ldb2(ll, blo, RS, brows, nb, ks0 + kk, lane);
                    mma_bf16(acc1[nb], A[0], bb[0], bb[1], acc1[nb]);
                    mma_bf16(acc1[nb], A[0], ll[0], ll[1], acc1[nb]);
                    mma_bf16(acc1[nb], A[1], bb[2], bb[3], acc1[nb]);
                    mma_bf16(acc1[nb], A[1], ll[2], ll[3], acc1[nb]);
                } else if (up) {
                    mma_bf16(acc3[nb], A[0], bb[0], bb[1], acc3[nb]);
                    mma_bf16(acc3[nb], A[1], bb[2], bb[3], acc3[nb]);
                } else {
                    mma_bf16(acc1[nb], A[0], bb[0], bb[1], acc1[nb]);
                    mma_bf16(acc1[nb], A[1], bb[2], bb[3], acc1[nb]);
                }
            }
        }
    }
}

// h of a routed expert as f16 (11 significant bits: the down projection's relative
// error from it is about 1e-4); of a shared expert as a bf16 hi + lo pair, since its
// down projection runs on bf16 MMAs.
__device__ __forceinline__ void store_h(const GemvArgs &a, int shared, size_t at, size_t plane, float hv)
{
    if (shared) {
        const __nv_bfloat16 hb = __float2bfloat16_rn(hv);
        const __nv_bfloat16 lb = __float2bfloat16_rn(hv - __bfloat162float(hb));
        a.hp[at] = *reinterpret_cast<const uint16_t *>(&hb);
        a.hp[plane + at] = *reinterpret_cast<const uint16_t *>(&lb);
    } else {
        const __half hh = __float2half_rn(hv);
        a.hp[at] = *reinterpret_cast<const uint16_t *>(&hh);
    }
}

// Bounded wait by every lane of a warp; the same result on every lane.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity)
{
    const bool ok = mbar_wait(bar, parity);
    return __all_sync(0xffffffffu, ok);
}

// Facts of the unit, item and pass a staged B chunk belongs to (written by the producer).
struct BHdr {
    int item, pass;
    int nvalid;                     // tokens of the pass (<= 16); the single-token schedule sets bit 8 on the item's last pass
    int shared, id, rb, kp, nkp;
};
constexpr int kLastPass = 1 << 8;

template <int MODE, int TPS, bool STREAM>
__global__ void __launch_bounds__(kThreads + 32, 2) gemv_kernel(const __grid_constant__ GemvArgs a,
                                                             const __grid_constant__ CUtensorMap m1,
                                                             const __grid_constant__ CUtensorMap m3,
                                                             const __grid_constant__ CUtensorMap m2)
{
    // gate/up: launched early (programmatic dependent launch) and waits for the routing only
    // before its first routed item.  down, for several tokens: waits for gate/up first.
    // down for up to three tokens (STREAM), where gate/up's last items leave most blocks
    // idle: launched early too, and it waits neither for the gate/up grid nor for all of
    // h: first for the routing to be visible (the flag gate/up raises after its own wait
    // for it), then, item by item, for its unit's h rows, which gate/up publishes unit by
    // unit (a.ready).  That down never lets its dependents launch early, and each block
    // waits for the gate/up grid before it exits, so the kernels after it still start on a
    // completed chain.
    if (MODE == kGateUp) {
        if (!a.early) {
            pdl_wait();
            if (STREAM && threadIdx.x == 0) raise_route_seen(a);
        }
        pdl_trigger();
    } else if (!STREAM) {
        pdl_wait();
        pdl_trigger();
    }
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    constexpr int kStageBytes = Geo<MODE>::kStageBytes;
    constexpr int kHalves = MODE == kDown ? 2 : 1;
    uint8_t *bufs = smem;                                          // kStages * kStageBytes
    const int CT = Geo<MODE>::chunk_tiles(a), RS = Geo<MODE>::b_row_bytes(a);
    const size_t bbytes = (size_t)a.brows * RS;                    // one half of one B slot
    uint8_t *bbase = smem + kStages * kStageBytes;                 // slot b, half h at (kHalves*b + h)
    __shared__ uint64_t full[kStages], empty[kStages], bfull[kBSlots], bempty[kBSlots];
    __shared__ int hdr_item[kStages], hdr_st[kStages], hdr_bu[kStages], hdr_sic[kStages];
    __shared__ int issued[kStages], bissued[kBSlots];
    __shared__ PassTok pts[kBSlots];
    __shared__ BHdr bh[kBSlots];
    __shared__ __align__(16) int32_t bflag[kBSlots][4];
    __shared__ int bail, route_ok, last_dn;

    if (MODE == kDown && !STREAM && *a.abort) return;
    const int n_sh = n_shared_items<MODE>(a);
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int nwarps = kThreads / 32;
    if (tid == 0) {
        for (int s = 0; s < kStages; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nwarps);
            issued[s] = 0;
        }
        for (int b = 0; b < kBSlots; b++) {
            mbar_init(&bfull[b], 1);
            mbar_init(&bempty[b], nwarps);
            bissued[b] = 0;
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        bail = 0;
        if (MODE == kDown && STREAM) {
            route_ok = 1;
            if (!wait_at_least(a.route_seen, 1)) {
                set_status(a.status, K3MOE_DEV_TIMEOUT);
                route_ok = 0;
            }
        }
    }
    __syncthreads();
    auto timeout = [&]() {
        set_status(a.status, K3MOE_DEV_TIMEOUT);
        bail = 1;
    };
    // down: every thread acquires the flag itself before it reads the routing; no items
    // when the routing failed validation or never became visible
    bool down_skip = false;
    if (MODE == kDown && STREAM) {
        if (route_ok) (void)ld_acquire(a.route_seen);
        down_skip = !route_ok || *a.abort != 0;
    }

    if (w == nwarps) {
        // ---------------- producer warp: work items, B chunks and weight stages, all by
        // bulk copies; nothing here waits for data
        int n = 0, bu = 0;
        bool stop = false;
        int n_items = -1;                       // known once the routing is
        bool gu_seen = false;                   // down: gate/up's last block has finished
        for (;;) {
            int i = 0;
            if (lane == 0 && !down_skip) i = atomicAdd(&a.work[MODE], 1);
            i = __shfl_sync(0xffffffffu, i, 0);
            if (!down_skip && i >= n_sh && n_items < 0) {
                // the first routed item: the routing (and the forward's prep) must be complete
                if (MODE == kGateUp) {
                    pdl_wait();
                    if (STREAM && lane == 0) raise_route_seen(a);
                }
                const int n_active = *a.abort ? 0 : dclamp(a.status, a.active[a.E], 0, a.E);
                n_items = n_sh + n_active * (Geo<MODE>::rows(a) / kItemRows);
            }
            const bool done = down_skip || (i >= n_sh && i >= n_items) || __shfl_sync(0xffffffffu, bail, 0) != 0;
            if (done) {
                // end of stream: one stage with no copy
                const int slot = n % kStages;
                if (n >= kStages && !mbar_wait_warp(&empty[slot], (uint32_t)((n / kStages) - 1) & 1u)) timeout();
                else if (lane == 0) {
                    hdr_item[slot] = -1;
                    mbar_arrive(&full[slot]);
                }
                break;
            }
            const Item it = item_of<MODE>(a, i);
            const Unit un = unit_of(a, it.u);
            const int pass1 = it.pass1 < 0 ? n_passes(un) : it.pass1;
            const int nst = n_stages<MODE, TPS>(a, un.shared);
            if (MODE == kDown && STREAM && !gu_seen) {
                // the unit's h rows are complete once every gate/up warp of every row block
                // (and token pass) has published them, and all of h once gate/up's last block
                // has finished; after that flag is seen no item checks again.  Lane 0 reads
                // both (relaxed, one round trip), then acquires; the warp's bulk copies that
                // read h are ordered after it.
                const int want = nwarps * (a.f / kItemRows) * (un.shared ? shared_passes(a) : 1);
                const int32_t *rp = a.ready + (un.shared ? a.E + un.id : un.id);
                int ok = 1, done_all = 0;
                if (lane == 0) {
                    done_all = ld_relaxed(a.gu_done);
                    const int r = ld_relaxed(rp);
                    if (!done_all && r < want) ok = wait_at_least(rp, want) ? 1 : 0;
                    fence_acq_rel();
                }
                __syncwarp();
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    timeout();
                    break;
                }
                gu_seen = __shfl_sync(0xffffffffu, done_all, 0) != 0;
                fence_proxy_async_all();
            }
            for (int pass = it.pass0; pass < pass1 && !stop; pass++) {
                const int nvalid = min(kPassTok, un.ntok - pass * kPassTok);
                // token facts of this pass: lane n holds token n's
                int tok = 0;
                long long row = 0;
                float fo = 1.0f;
                if (lane < nvalid) {
                    tok = token_of(a, un, pass, lane);
                    row = (long long)out_row(a, un, pass, lane);
                    fo = un.shared ? 1.0f : a.tok_scale[a.T + tok];
                }
                // stages per B chunk (of CT tiles)
                const int spc = un.shared ? Geo<MODE>::kSharedMats * (kTileK / kSharedK) * CT : CT / TPS;
                for (int st = 0, sic = 0; st < nst; st++, n++, sic = (sic + 1 == spc) ? 0 : sic + 1) {
                    if (sic == 0) {
                        // the B chunk of this (item, pass) for the next CT tiles of K
                        const int b = bu % kBSlots;
                        if (bu >= kBSlots && !mbar_wait_warp(&bempty[b], (uint32_t)((bu / kBSlots) - 1) & 1u)) {
                            timeout();
                            stop = true;
                            break;
                        }
                        if (lane < nvalid) {
                            pts[b].tok[lane] = tok;
                            pts[b].row[lane] = row;
                            pts[b].fo[lane] = fo;
                        }
                        if (lane == 0)
                            bh[b] = BHdr{i, pass, nvalid | (STREAM && pass == pass1 - 1 ? kLastPass : 0), un.shared,
                                         un.id, it.rb, it.kp, it.nkp};
                        __syncwarp();
                        issue_b_chunk<MODE>(a, un, it, st / spc, nvalid, tok, row, bbase + kHalves * b * bbytes,
                                            bbase + (kHalves * b + kHalves - 1) * bbytes, bflag[b], &bfull[b], lane);
                        if (lane == 0) bissued[b]++;
                        bu++;
                    }
                    const int slot = n % kStages;
                    if (n >= kStages && !mbar_wait_warp(&empty[slot], (uint32_t)((n / kStages) - 1) & 1u)) {
                        timeout();
                        stop = true;
                        break;
                    }
                    if (lane == 0) {
                        hdr_item[slot] = i;
                        hdr_st[slot] = st;
                        hdr_bu[slot] = bu - 1;
                        // stage within its B chunk; bit 16: the chunk's last stage; bit 17: the pass's last
                        hdr_sic[slot] = sic | ((sic + 1 == spc || st == nst - 1) ? 1 << 16 : 0) |
                                        (st == nst - 1 ? 1 << 17 : 0);
                        fence_proxy_async();
                        issue_stage<MODE, TPS>(a, &m1, &m3, &m2, un, it, st, bufs + slot * kStageBytes, &full[slot]);
                        issued[slot]++;
                    }
                    __syncwarp();
                }
            }
            if (stop) break;
        }
    } else {
        // ---------------- consumers: warp w owns rows 16w..16w+15 of every item
        const int g = lane >> 2, t4 = lane & 3;
        float acc1[kNBMax][4], acc3[kNBMax][4];
        int cur_bu = -1, b = 0, var = 0;
        uint32_t bhi = 0, blo = 0;
        const uint32_t sbufs = smem_addr(bufs);
        for (int n = 0;; n++) {
            const int slot = n % kStages;
            if (!mbar_wait_warp(&full[slot], (uint32_t)(n / kStages) & 1u)) {
                timeout();
                break;
            }
            const int item = hdr_item[slot];
            if (item < 0) break;
            const int st = hdr_st[slot], bun = hdr_bu[slot], sicf = hdr_sic[slot];
            const int sic = sicf & 0xFFFF;
            if (bun != cur_bu) {                                // a new B chunk
                b = bun % kBSlots;
                if (!mbar_wait_warp(&bfull[b], (uint32_t)(bun / kBSlots) & 1u)) {
                    timeout();
                    break;
                }
                cur_bu = bun;
                // once per chunk: its B operand addresses and the consume variant of its
                // stages (bit 0: more than 8 tokens, two n-blocks; bit 1: a routed expert
                // whose trailer flags a scale byte 0 or 255, the exact scale path; bit 2:
                // bf16 shared-expert tiles)
                bhi = smem_addr(bbase + kHalves * b * bbytes);
                blo = smem_addr(bbase + (kHalves * b + kHalves - 1) * bbytes);
                const int nv = STREAM ? bh[b].nvalid & 0xFF : bh[b].nvalid;
                var = (nv > 8 ? 1 : 0) | (bh[b].shared ? 4 : (bflag[b][3] != 0 ? 2 : 0));
            }
            const BHdr &h = bh[b];
            const PassTok &pt = pts[b];
            if (st == 0) {
#pragma unroll
                for (int nb = 0; nb < kNBMax; nb++)
#pragma unroll
                    for (int i = 0; i < 4; i++) acc1[nb][i] = acc3[nb][i] = 0.0f;
            }
            const uint32_t buf = sbufs + slot * kStageBytes;
            switch (var) {
            case 3: consume_stage<MODE, 2, TPS, true>(buf, 0, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            case 2: consume_stage<MODE, 1, TPS, true>(buf, 0, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            case 5: consume_stage<MODE, 2, TPS, false>(buf, 1, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            case 4: consume_stage<MODE, 1, TPS, false>(buf, 1, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            case 1: consume_stage<MODE, 2, TPS, false>(buf, 0, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            default: consume_stage<MODE, 1, TPS, false>(buf, 0, sic, RS, a.brows, bhi, blo, w, lane, acc1, acc3); break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            const bool chunk_end = (sicf >> 16) & 1;
            if ((sicf >> 17) & 1) {
                // epilogue: this thread holds rows 16w+g (+8) x tokens 8nb+2t4 (+1)
                const int row0 = h.rb * kItemRows + 16 * w + g;
                const size_t rows_all = (size_t)a.T * a.k + (size_t)a.S * a.T;
                const int nvalid = STREAM ? h.nvalid & 0xFF : h.nvalid;
                const size_t slots = (size_t)a.T * a.k;
                if (MODE == kDown) {
                    // y row: the slot's, or for a shared expert its K part's (the combine
                    // adds the parts in order)
#pragma unroll
                    for (int nb = 0; nb < kNBMax; nb++)
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int nn = nb * 8 + 2 * t4 + (i & 1);
                            if (nn >= nvalid) continue;
                            const int row = row0 + ((i >> 1) << 3);
                            size_t yrow = (size_t)pt.row[nn];
                            if (h.shared) {
                                const size_t t = yrow - slots - (size_t)h.id * a.T;
                                yrow = slots + ((size_t)h.id * h.nkp + h.kp) * a.T + t;
                            }
                            a.ys[yrow * a.d + row] = acc1[nb][i];
                        }
                } else if (h.nkp > 1) {
                    // a K part of a shared expert (one token pass): publish the partial sums;
                    // the last of the parts' 8 x nkp warps of this row block adds the parts
                    // in order and applies SiTU to all 128 rows
#pragma unroll
                    for (int nb = 0; nb < kNBMax; nb++)
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int nn = nb * 8 + 2 * t4 + (i & 1);
                            if (nn >= nvalid) continue;
                            const int row = row0 + ((i >> 1) << 3);
                            float *base = a.gush + ((((size_t)h.kp * a.S + h.id) * a.T + nn) * 2) * a.f;
                            base[row] = acc1[nb][i];
                            base[a.f + row] = acc3[nb][i];
                        }
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0) {
                        int32_t *ctr = a.shctr + (size_t)h.id * (a.f / kItemRows) + h.rb;
                        const int old = atomicAdd(ctr, 1);
                        last = (old == h.nkp * nwarps - 1);
                        if (last) *ctr = 0;
                    }
                    if (__shfl_sync(0xffffffffu, last, 0)) {
                        __threadfence();
                        const size_t plane = rows_all * a.f;
                        // every part of this lane's four rows is loaded before any is added,
                        // so the loads are in flight together
                        for (int nn = 0; nn < nvalid; nn++) {
                            float gv[kItemRows / 32][kMaxSharedParts], uv[kItemRows / 32][kMaxSharedParts];
#pragma unroll
                            for (int q = 0; q < kItemRows / 32; q++)
#pragma unroll
                                for (int p = 0; p < kMaxSharedParts; p++) {
                                    gv[q][p] = uv[q][p] = 0.0f;
                                    if (p < h.nkp) {
                                        const float *base = a.gush + ((((size_t)p * a.S + h.id) * a.T + nn) * 2) * a.f;
                                        const int row = h.rb * kItemRows + 32 * q + lane;
                                        gv[q][p] = __ldcg(base + row);
                                        uv[q][p] = __ldcg(base + a.f + row);
                                    }
                                }
#pragma unroll
                            for (int q = 0; q < kItemRows / 32; q++) {
                                float gs = 0.0f, us = 0.0f;
#pragma unroll
                                for (int p = 0; p < kMaxSharedParts; p++)
                                    if (p < h.nkp) {
                                        gs += gv[q][p];
                                        us += uv[q][p];
                                    }
                                const int row = h.rb * kItemRows + 32 * q + lane;
                                store_h(a, 1, (size_t)pt.row[nn] * a.f + row, plane, situ(gs, us, a.b1, a.b2));
                            }
                        }
                        // this warp wrote the row block's 128 rows: as much as eight warps of
                        // an unsplit item
                        if (STREAM) publish_add(a.ready + a.E + h.id, nwarps, lane);
                    }
                } else {
                    const size_t plane = rows_all * a.f;
#pragma unroll
                    for (int nb = 0; nb < kNBMax; nb++)
#pragma unroll
                        for (int i = 0; i < 4; i++) {
                            const int nn = nb * 8 + 2 * t4 + (i & 1);
                            if (nn >= nvalid) continue;
                            const int row = row0 + ((i >> 1) << 3);
                            const float fo = pt.fo[nn];
                            store_h(a, h.shared, (size_t)pt.row[nn] * a.f + row, plane,
                                    situ(acc1[nb][i] * fo, acc3[nb][i] * fo, a.b1, a.b2));
                        }
                    // after the item's last pass this warp's 16 rows of h are complete
                    if (STREAM && (h.nvalid & kLastPass)) publish_add(a.ready + (h.shared ? a.E + h.id : h.id), 1, lane);
                }
            }
            if (chunk_end) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&bempty[b]);
            }
        }
    }
    __syncthreads();
    if (bail && tid == 0) {
        // a wait gave up: let every copy still in flight land before the block's shared
        // memory is released (each wait bounded)
        for (int s = 0; s < kStages; s++)
            if (issued[s] > 0) mbar_wait(&full[s], (uint32_t)(issued[s] - 1) & 1u);
        for (int s = 0; s < kBSlots; s++)
            if (bissued[s] > 0) mbar_wait(&bfull[s], (uint32_t)(bissued[s] - 1) & 1u);
    }
    if (MODE == kGateUp && tid == 0) {
        // the grid completes only after the routing did (the next kernel's wait covers both)
        pdl_wait();
        if (STREAM) raise_route_seen(a);
        // the last block to leave resets the work counter and the K-part arrival counters
        // for the next call (prep cannot: this kernel may run before it)
        __threadfence();
        if (atomicAdd(a.exits, 1) == (int)gridDim.x - 1) {
            a.work[MODE] = 0;
            for (int q = 0; q < a.S * (a.f / kItemRows); q++) a.shctr[q] = 0;
            __threadfence();
            *a.exits = 0;
            // every block has finished, after its fence: all of h is published
            if (STREAM) atomicExch(a.gu_done, 1);
        }
    }
    if (MODE == kDown && STREAM) {
        if (tid == 0) {
            // the grid completes only after gate/up did: the kernels after it rely on that
            pdl_wait();
            __threadfence();
            last_dn = atomicAdd(a.dn_exits, 1) == (int)gridDim.x - 1;
        }
        __syncthreads();
        if (last_dn) {
            // the last block to leave (every gate/up increment is done, every down block has
            // read its counters): reset the h-ready counters and the routing flag
            for (int u = tid; u < a.E + a.S; u += blockDim.x) a.ready[u] = 0;
            __syncthreads();
            if (tid == 0) {
                *a.route_seen = 0;
                *a.gu_done = 0;
                __threadfence();
                *a.dn_exits = 0;
            }
        }
    }
}

// -------------------------------------------------------------------------------- combine
struct CombineArgs {
    int T, d, k, S;
    int psh;                        // K parts of a shared expert's y (rows in order)
    const float *weight;
    const int32_t *inv;
    const float *ys;
    float *out;
    const int32_t *abort;
    int32_t *status;
};

// One thread per output element; the token's k positions and weights are read first and
// every y row is then loaded (unconditionally: prep has validated the positions, and an
// aborted call writes zeros) before any is summed, so a thread's loads are all in flight
// together.  Sum order: slot j ascending, then the shared experts in order (each its K
// parts in order).
__device__ __forceinline__ float combine_one(const CombineArgs &a, int t, int c)
{
    const int slots = a.T * a.k;
    int pos[kMaxTopK];
    float wt[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; j++) {
        const int jj = j < a.k ? j : 0;
        const int p = a.inv[(size_t)t * a.k + jj];
        pos[j] = dclamp(a.status, p, 0, slots - 1);
        wt[j] = j < a.k ? a.weight[(size_t)t * a.k + jj] : 0.0f;
    }
    float y[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; j++) y[j] = j < a.k ? a.ys[(size_t)pos[j] * a.d + c] : 0.0f;
    float acc = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; j++)
        if (j < a.k) acc = fmaf(wt[j], y[j], acc);
    for (int s = 0; s < a.S; s++) {
        float ysh = 0.0f;
        for (int p = 0; p < a.psh; p++) ysh += a.ys[((size_t)slots + ((size_t)s * a.psh + p) * a.T + t) * a.d + c];
        acc += ysh;
    }
    return acc;
}

__global__ void __launch_bounds__(256) fwd_combine_kernel(CombineArgs a)
{
    pdl_wait();
    pdl_trigger();
    const size_t n = (size_t)a.T * a.d;
    const bool ab = *a.abort != 0;
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < n;
         q += (size_t)gridDim.x * blockDim.x) {
        const int t = (int)(q / a.d), c = (int)(q % a.d);
        a.out[q] = ab ? 0.0f : combine_one(a, t, c);
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

// bf16 matrix [rows][cols] row-major; boxes of 64 cols x 128 rows, 128-byte swizzle.
bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {kSharedK, kItemRows};
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

// Persistent grid: every SM filled to the occupancy the kernel's resources allow
// (shared memory carve-out at its maximum).  Occupancy is computed once per (kernel,
// shared-memory size) and cached.  A kernel's dynamic shared-memory limit is a property
// of the function, so it is only ever raised: a launch that needs less than an earlier
// one still fits.
template <typename Kern>
int grid_blocks(Kern kernel, size_t smem)
{
    struct Entry { const void *k; size_t smem; int blocks; };
    struct Limit { const void *k; size_t smem; };
    static Entry cache[16];
    static Limit limit[8];               // the six mat-vec kernels (mode x ring x schedule)
    static int n_cache = 0, n_limit = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    int li = 0;
    while (li < n_limit && limit[li].k != (const void *)kernel) li++;
    if (li == n_limit) {
        if (n_limit < 8) limit[n_limit++] = Limit{(const void *)kernel, 0};
        else li = -1;                    // not cached: the attributes are set on every call
        cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    }
    if (li < 0 || smem > limit[li].smem) {
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (li >= 0) limit[li].smem = smem;
    }
    for (int i = 0; i < n_cache; i++)
        if (cache[i].k == (const void *)kernel && cache[i].smem == smem) return cache[i].blocks;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads + 32, smem) != cudaSuccess || occ < 1)
        occ = 1;
    const int blocks = sm_count() * occ;
    if (n_cache < 16) cache[n_cache++] = Entry{(const void *)kernel, smem, blocks};
    return blocks;
}

// Tensor maps of the shared-expert weights, cached by (address, shape).
bool cached_bf16_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols)
{
    struct Entry { const void *base; uint64_t rows, cols; CUtensorMap map; };
    static Entry cache[32];
    static int n_cache = 0, next = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cache; i++)
        if (cache[i].base == base && cache[i].rows == rows && cache[i].cols == cols) {
            *m = cache[i].map;
            return true;
        }
    if (!make_bf16_map(m, base, rows, cols)) return false;
    Entry &e = cache[n_cache < 32 ? n_cache++ : (next++ % 32)];
    e.base = base;
    e.rows = rows;
    e.cols = cols;
    e.map = *m;
    return true;
}

// One mbarrier that nothing arrives on, waited on by this file's bounded wait with the
// given limit: the wait gives up and the kernel reports it the way the mat-vec kernels
// do, by the status word's timeout bit.  For tests of that path.
__global__ void __launch_bounds__(32) wait_check_gemv_kernel(int32_t *status, long long limit)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (!mbar_wait(&bar, 0, limit)) atomicOr(status, K3MOE_DEV_TIMEOUT);
    }
}

}  // namespace

cudaError_t launch_wait_check_gemv(int32_t *status, long long limit, cudaStream_t s)
{
    wait_check_gemv_kernel<<<1, 32, 0, s>>>(status, limit);
    count_launch();
    return cudaGetLastError();
}

cudaError_t launch_forward_gemv(const k3moe_config &c, int T, const uint16_t *x,
                                const int32_t *idx, const float *weight, const int32_t *offsets,
                                const int32_t *perm, const uint8_t *table, const uint16_t *sh_w1,
                                const uint16_t *sh_w3, const uint16_t *sh_w2, float *out,
                                uint8_t *ws, const WsLayout &L, cudaStream_t s, bool x_is_input)
{
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    int32_t *abort = status + 1;
    int32_t *active = reinterpret_cast<int32_t *>(ws + L.active);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    float *tok_scale = reinterpret_cast<float *>(ws + L.tok_scale);
    uint16_t *hp = reinterpret_cast<uint16_t *>(ws + L.hp);
    float *ys = reinterpret_cast<float *>(ws + L.ys);

    uint16_t *xs = reinterpret_cast<uint16_t *>(ws + L.xs);
    int32_t *shctr = reinterpret_cast<int32_t *>(ws + L.shctr);
    float *gush = reinterpret_cast<float *>(ws + L.gush);
    PrepArgs pa{T, c.n_experts, c.top_k, c.d, x, idx, offsets, perm, active, inv, tok_scale, xs, status, abort,
                x_is_input ? 1 : 0};
    timing_begin("fwd_prep", s);
    cudaError_t err = launch_pdl(fwd_prep_kernel, dim3(1 + (T + 31) / 32), dim3(1024), 0, s, pa);
    count_launch();
    timing_end("fwd_prep", s);
    if (err != cudaSuccess) return err;

    CUtensorMap m1{}, m3{}, m2{};
    if (c.n_shared > 0) {
        if (!cached_bf16_map(&m1, sh_w1, (uint64_t)c.n_shared * c.f, c.d) ||
            !cached_bf16_map(&m3, sh_w3, (uint64_t)c.n_shared * c.f, c.d) ||
            !cached_bf16_map(&m2, sh_w2, (uint64_t)c.n_shared * c.d, c.f))
            return cudaErrorInvalidValue;
    }
    GemvArgs ga{T, c.d, c.f, c.top_k, c.n_shared, c.n_experts, 0, c.situ_b1, c.situ_b2,
                x, xs, offsets, perm, active, tok_scale, table, expert_bytes(c.d, c.f),
                gateup_block_bytes(c.d, c.f), ys, gush, shctr, hp, abort, status, abort + 1, status + 5,
                x_is_input ? 1 : 0, reinterpret_cast<int32_t *>(ws + L.ready), status + 6, status + 7,
                status + 8};
    // up to three tokens: down starts unit by unit as gate/up publishes h (measured: T = 1
    // -6.5%, 2 -2.8%, 3 -1.5% a step; from T = 4 gate/up's blocks finish together)
    const bool stream = T <= 3;
    // B chunks hold min(16, T) token rows
    ga.brows = T < kPassTok ? T : kPassTok;
    {
        const size_t bsl = (size_t)kBSlots * ga.brows * Geo<kGateUp>::b_row_bytes(ga);
        const size_t smem = 1024 + (size_t)kStages * Geo<kGateUp>::kStageBytes + bsl;
        const auto kern = stream ? gemv_kernel<kGateUp, 1, true> : gemv_kernel<kGateUp, 1, false>;
        const int blocks = grid_blocks(kern, smem);
        timing_begin("gemv_gateup", s);
        err = launch_pdl(kern, dim3(blocks), dim3(kThreads + 32), smem, s, ga, m1, m3, m2);
        count_launch();
        timing_end("gemv_gateup", s);
        if (err != cudaSuccess) return err;
    }
    {
        const size_t bsl = 2 * (size_t)kBSlots * ga.brows * Geo<kDown>::b_row_bytes(ga);
        const size_t smem = 1024 + (size_t)kStages * Geo<kDown>::kStageBytes + bsl;
        // two K tiles per routed stage when K has an even number of tiles
        const bool two = (c.f / kTileK) % 2 == 0;
        const auto kern = two ? (stream ? gemv_kernel<kDown, 2, true> : gemv_kernel<kDown, 2, false>)
                              : (stream ? gemv_kernel<kDown, 1, true> : gemv_kernel<kDown, 1, false>);
        const int blocks = grid_blocks(kern, smem);
        timing_begin("gemv_down", s);
        err = launch_pdl(kern, dim3(blocks), dim3(kThreads + 32), smem, s, ga, m1, m3, m2);
        count_launch();
        timing_end("gemv_down", s);
        if (err != cudaSuccess) return err;
    }
    CombineArgs ca{T, c.d, c.top_k, c.n_shared, 1, weight, inv, ys, out, abort, status};
    {
        const size_t n = (size_t)T * c.d;
        int grid = (int)((n + 255) / 256);
        if (grid > sm_count() * 8) grid = sm_count() * 8;
        if (grid < 1) grid = 1;
        timing_begin("fwd_combine", s);
        err = launch_pdl(fwd_combine_kernel, dim3(grid), dim3(256), 0, s, ca);
        count_launch();
        timing_end("fwd_combine", s);
        if (err != cudaSuccess) return err;
    }
    return cudaGetLastError();
}

}  // namespace k3moe
