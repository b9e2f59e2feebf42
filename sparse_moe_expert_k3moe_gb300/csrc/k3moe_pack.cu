// k3moe_pack.cu -- relayout of routed experts between the checkpoint's MXFP4
// layout and the library's tiled table (kimi-k3-in-c README, Part II,
// section 4: codes and E8M0 scales are copied, never re-quantised).
#include "k3moe_internal.cuh"

namespace k3moe {
namespace {

struct PackArgs {
    int d, f, E, expert_lo, n;
    const uint8_t *w1p, *w1s, *w3p, *w3s, *w2p, *w2s;   // checkpoint side
    uint8_t *table;                                     // packed side (full table base)
    int32_t *status;
};

// Decompose the 16-byte source group number q (within one expert, in table order) into
// the matrix (0 = W1, 1 = W3, 2 = W2), the source row and the source group, and the
// destination offsets, within the expert, of the group's lane words and scale byte:
// byte b of the group goes to lane 4*(r%8) + b%4, word r%16/8, byte position b/4.
__device__ __forceinline__ void chunk_coords(int d, int f, size_t q, int &mat, int &row,
                                             int &grp, size_t &dst_lane0, size_t &dst_scale)
{
    const size_t chunks_per_tile = (size_t)kTileNibbleBytes / 16;     // 512
    const size_t tile = q / chunks_per_tile;
    const int within = (int)(q % chunks_per_tile);
    const int c = within / kTileRows, r = within % kTileRows;
    const size_t gu_tiles = (size_t)(f / kTileRows) * (size_t)(d / kTileK) * 2;
    int rb, kt;
    if (tile < gu_tiles) {
        const int ktd = d / kTileK;
        rb = (int)(tile / (size_t)(2 * ktd));
        const int rem = (int)(tile % (size_t)(2 * ktd));
        kt = rem / 2;
        mat = rem % 2;
    } else {
        const size_t t2 = tile - gu_tiles;
        const int ktf = f / kTileK;
        rb = (int)(t2 / (size_t)ktf);
        kt = (int)(t2 % (size_t)ktf);
        mat = 2;
    }
    row = rb * kTileRows + r;
    grp = kt * (kTileK / kGroup) + c;
    const int s = r / 16, g = r % 8, hi = (r % 16) / 8;
    dst_lane0 = tile * kTileBytes + (size_t)(s * 4 + c) * 256 + (size_t)(4 * g) * 8 + hi * 4;
    dst_scale = tile * kTileBytes + kTileNibbleBytes + (size_t)r * 4 + c;
}

// The four lane words of a group: word t = bytes t, t+4, t+8, t+12.
__device__ __forceinline__ uint32_t lane_word(const uint4 v, int t)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const int sh = 8 * t;
    return ((w[0] >> sh) & 0xFFu) | (((w[1] >> sh) & 0xFFu) << 8) | (((w[2] >> sh) & 0xFFu) << 16) |
           (((w[3] >> sh) & 0xFFu) << 24);
}

__global__ void __launch_bounds__(256) pack_kernel(PackArgs a)
{
    const size_t per_expert = (size_t)3 * a.f * a.d / 32;             // chunks per expert
    const size_t total = per_expert * (size_t)a.n;
    const size_t eb = expert_bytes(a.d, a.f);
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < total;
         q += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(q / per_expert);
        int mat, row, grp;
        size_t dn, ds;
        chunk_coords(a.d, a.f, q % per_expert, mat, row, grp, dn, ds);
        const int cols = (mat == 2) ? a.f : a.d;
        const int rows = (mat == 2) ? a.d : a.f;
        const uint8_t *sp = mat == 0 ? a.w1p : (mat == 1 ? a.w3p : a.w2p);
        const uint8_t *ss = mat == 0 ? a.w1s : (mat == 1 ? a.w3s : a.w2s);
        const size_t mat_nib = (size_t)rows * cols / 2, mat_sc = (size_t)rows * cols / kGroup;
        const uint4 v = *reinterpret_cast<const uint4 *>(
            sp + (size_t)e * mat_nib + (size_t)row * (cols / 2) + (size_t)grp * 16);
        const uint8_t sb = ss[(size_t)e * mat_sc + (size_t)row * (cols / kGroup) + grp];
        uint8_t *dst = a.table + (size_t)(a.expert_lo + e) * eb;
        for (int t = 0; t < 4; t++)
            *reinterpret_cast<uint32_t *>(dst + dn + (size_t)t * 8) = lane_word(v, t);
        dst[ds] = sb;
        // the block-scaled section: the group in row-major order, its scale in its block
        {
            const int ex = a.expert_lo + e;
            const size_t rmo = (mat == 0 ? mx_w1_offset(a.E, a.d, a.f)
                                         : (mat == 1 ? mx_w3_offset(a.E, a.d, a.f) : mx_w2_offset(a.E, a.d, a.f))) +
                               ((size_t)ex * rows + row) * (cols / 2) + (size_t)grp * 16;
            *reinterpret_cast<uint4 *>(a.table + rmo) = v;
            const int rb = row / kTileRows, r = row % kTileRows, kc = grp / 4, kb = grp % 4;
            const size_t so = mat < 2
                ? mx_sfgu_offset(a.E, a.d, a.f) + ((((size_t)ex * (a.f / kTileRows) + rb) * (a.d / kTileK) + kc) * 2 + mat) * 512
                : mx_sfdn_offset(a.E, a.d, a.f) + (((size_t)ex * (a.d / kTileRows) + rb) * (a.f / kTileK) + kc) * 512;
            a.table[so + 16 * (r % 32) + 4 * (r / 32) + kb] = sb == 255 ? 0 : sb;
        }
        if (sb == 0 || sb == 255)
            atomicOr(reinterpret_cast<unsigned int *>(
                         a.table + special_flag_offset(a.E, a.d, a.f, a.expert_lo + e)), 1u);
        if (sb == 255) {
            if (a.status) set_status(a.status, K3MOE_DEV_NAN_SCALE);
        } else {
            atomicMax(reinterpret_cast<unsigned int *>(
                          a.table + trailer_offset(a.E, a.d, a.f, a.expert_lo + e, mat, row / kTileRows)),
                      (unsigned int)sb);
        }
    }
}

struct UnpackArgs {
    int d, f, expert_lo, n;
    const uint8_t *table;
    uint8_t *w1p, *w1s, *w3p, *w3s, *w2p, *w2s;
};

__global__ void __launch_bounds__(256) unpack_kernel(UnpackArgs a)
{
    const size_t per_expert = (size_t)3 * a.f * a.d / 32;
    const size_t total = per_expert * (size_t)a.n;
    const size_t eb = expert_bytes(a.d, a.f);
    for (size_t q = blockIdx.x * (size_t)blockDim.x + threadIdx.x; q < total;
         q += (size_t)gridDim.x * blockDim.x) {
        const int e = (int)(q / per_expert);
        int mat, row, grp;
        size_t dn, ds;
        chunk_coords(a.d, a.f, q % per_expert, mat, row, grp, dn, ds);
        const int cols = (mat == 2) ? a.f : a.d;
        const int rows = (mat == 2) ? a.d : a.f;
        uint8_t *dp = mat == 0 ? a.w1p : (mat == 1 ? a.w3p : a.w2p);
        uint8_t *dsx = mat == 0 ? a.w1s : (mat == 1 ? a.w3s : a.w2s);
        const size_t mat_nib = (size_t)rows * cols / 2, mat_sc = (size_t)rows * cols / kGroup;
        const uint8_t *src = a.table + (size_t)(a.expert_lo + e) * eb;
        uint32_t w[4] = {0, 0, 0, 0};
        for (int t = 0; t < 4; t++) {
            const uint32_t lw = *reinterpret_cast<const uint32_t *>(src + dn + (size_t)t * 8);
            for (int q = 0; q < 4; q++) w[q] |= ((lw >> (8 * q)) & 0xFFu) << (8 * t);
        }
        *reinterpret_cast<uint4 *>(dp + (size_t)e * mat_nib + (size_t)row * (cols / 2) +
                                   (size_t)grp * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        dsx[(size_t)e * mat_sc + (size_t)row * (cols / kGroup) + grp] = src[ds];
    }
}

int grid_for(size_t work)
{
    size_t blocks = (work + 255) / 256;
    const size_t cap = 152 * 16;
    return (int)(blocks < cap ? (blocks ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_pack(const k3moe_config &c, int expert_lo, int n, const uint8_t *w1p,
                        const uint8_t *w1s, const uint8_t *w3p, const uint8_t *w3s,
                        const uint8_t *w2p, const uint8_t *w2s, uint8_t *table,
                        int32_t *status, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    PackArgs a{c.d, c.f, c.n_experts, expert_lo, n, w1p, w1s, w3p, w3s, w2p, w2s, table, status};
    const size_t work = (size_t)3 * c.f * c.d / 32 * (size_t)n;
    cudaError_t e = cudaMemsetAsync(table + (size_t)c.n_experts * expert_bytes(c.d, c.f) +
                                        (size_t)expert_lo * kTrailerBytes,
                                    0, (size_t)n * kTrailerBytes, s);
    if (e != cudaSuccess) return e;
    timing_begin("pack_mxfp4", s);
    pack_kernel<<<grid_for(work), 256, 0, s>>>(a);
    count_launch();
    timing_end("pack_mxfp4", s);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const k3moe_config &c, int expert_lo, int n, const uint8_t *table,
                          uint8_t *w1p, uint8_t *w1s, uint8_t *w3p, uint8_t *w3s,
                          uint8_t *w2p, uint8_t *w2s, cudaStream_t s)
{
    if (n == 0) return cudaSuccess;
    UnpackArgs a{c.d, c.f, expert_lo, n, table, w1p, w1s, w3p, w3s, w2p, w2s};
    const size_t work = (size_t)3 * c.f * c.d / 32 * (size_t)n;
    timing_begin("unpack_mxfp4", s);
    unpack_kernel<<<grid_for(work), 256, 0, s>>>(a);
    count_launch();
    timing_end("unpack_mxfp4", s);
    return cudaGetLastError();
}

}  // namespace k3moe
