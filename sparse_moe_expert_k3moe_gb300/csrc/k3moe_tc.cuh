// k3moe_tc.cuh -- inline-PTX helpers shared by the tensor-core kernels (sm_103a):
// mbarriers with bounded waits, TMA 2-D tile loads, tcgen05 shared-memory and
// instruction descriptors, MMA issue and commit, tensor-memory loads; and the host-side
// tensor-map encoder (a per-process cache keyed by base, shape and box).
#pragma once
#include <cuda.h>

#include <mutex>

#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

// clock cycles a wait spins before it gives up (about two seconds)
constexpr long long kTcWaitCyc = 4000000000ll;

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mb_init(uint64_t *b, uint32_t n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(n));
}
__device__ __forceinline__ void mb_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
__device__ __forceinline__ void mb_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mb_wait(uint64_t *b, uint32_t parity, long long limit = kTcWaitCyc)
{
    const uint32_t a = saddr(b);
    {   // fast path: the phase is usually complete already
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
// The whole warp waits (every lane polls); the result is the same on every lane.  A
// role whose loop runs on all 32 lanes keeps its warp converged, and issues its single
// thread operations under lane 0.
__device__ __forceinline__ bool mb_wait_warp(uint64_t *b, uint32_t parity)
{
    const bool ok = mb_wait(b, parity);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tma2d(void *dst, const CUtensorMap *m, int c0, int c1, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(saddr(dst)),
        "l"(m), "r"(c0), "r"(c1), "r"(saddr(bar))
        : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completing on an mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            saddr(dst)),
        "l"(src), "r"(bytes), "r"(saddr(bar))
        : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);            // start address
    d |= (uint64_t)1u << 16;                            // leading byte offset (unused here)
    d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset
    d |= (uint64_t)1u << 46;                            // descriptor version
    d |= (uint64_t)2u << 61;                            // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: fp32 D, A and B both f16 (fmt 0) or bf16 (fmt 1),
// both K-major, N = n, M = 128.
__device__ __forceinline__ uint32_t idesc(int fmt, int n)
{
    return (1u << 4) | ((uint32_t)fmt << 7) | ((uint32_t)fmt << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(a), "l"(b), "r"(id), "r"(acc));
}
// ---- block-scaled MMA (kind::mxf8f6f4): A e4m3, B e2m1, one ue8m0 scale per 32 K
// elements of every A row and B row, read by the tensor core from tensor memory.
// Operand layouts, as measured on sm_103a: K-major, 128-byte swizzle like the f16 tiles,
// an e4m3 row of 128 elements is 128 bytes; an e2m1 row keeps 16 elements per 16-byte
// chunk, their 8 packed bytes (low nibble = even element) first and 8 bytes that are not
// read.  Scales: a 512-byte shared-memory block per 128 rows and 4 K blocks, row m's 4
// bytes at 16 (m % 32) + 4 (m / 32); tcgen05.cp 32x128b.warpx4 puts them in tensor
// memory as 4 columns (row m in column m / 32 of lane m % 32, every lane quadrant a
// copy); the instruction descriptor's scale ids pick the byte, i.e. the K block.
// Instruction descriptor: fp32 D, A e4m3 (0), B e2m1 (5), both K-major, N = n, M = 128,
// ue8m0 scales, scale ids sfa (A) and sfb (B).
__device__ __forceinline__ uint32_t idesc_mx(int n, int sfa, int sfb)
{
    return ((uint32_t)sfb << 4) | (0u << 7) | (5u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(128 >> 7) << 27) | ((uint32_t)sfa << 29);
}
__device__ __forceinline__ void umma_mx(uint32_t dtmem, uint64_t a, uint64_t b, uint32_t id, uint32_t sfa_tmem,
                                        uint32_t sfb_tmem, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            dtmem),
        "l"(a), "l"(b), "r"(id), "r"(sfa_tmem), "r"(sfb_tmem), "r"(acc));
}
// Shared-memory descriptor of a contiguous 512-byte scale block (no swizzle, 8-row groups
// of 16-byte rows 128 bytes apart) for tcgen05.cp.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     saddr(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}
// The same load without the wait: several loads in flight, then one tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
inline EncodeTiledFn encode_tiled()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}
// 16-bit matrix [rows][cols]: boxes of 64 columns x box_rows rows, 128-byte swizzle.
inline bool map16(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    struct Entry { const void *base; uint64_t rows, cols; uint32_t br; CUtensorMap map; };
    static Entry cache[64];
    static int n_cache = 0, next = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < n_cache; i++)
        if (cache[i].base == base && cache[i].rows == rows && cache[i].cols == cols && cache[i].br == box_rows) {
            *m = cache[i].map;
            return true;
        }
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64u, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    Entry &e = cache[n_cache < 64 ? n_cache++ : (next++ % 64)];
    e.base = base; e.rows = rows; e.cols = cols; e.br = box_rows; e.map = *m;
    return true;
}

// 8-bit matrix [rows][cols]: boxes of 128 columns x box_rows rows, 128-byte swizzle.
inline bool map8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols};
    const cuuint32_t box[2] = {128u, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed 4-bit matrix [rows][cols / 2 bytes] (low nibble = even column): boxes of 128
// columns x 128 rows with the packed-FP4 type, which lands each 16 codes as 8 bytes at the
// start of a 16-byte chunk (the e2m1 operand layout of the block-scaled MMA), 128-byte
// swizzle.  The box's transaction count is its packed size, 8192 bytes (measured).  Needs
// cols % 128 == 0, a 32-byte aligned base and a row stride that is a multiple of 32.
inline bool map4(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols)
{
    EncodeTiledFn fn = encode_tiled();
    if (!fn || cols % 128 != 0 || (cols / 2) % 32 != 0 || reinterpret_cast<uintptr_t>(base) % 32 != 0) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols / 2};
    const cuuint32_t box[2] = {128u, 128u};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int num_sms()
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

}  // namespace
}  // namespace k3moe
