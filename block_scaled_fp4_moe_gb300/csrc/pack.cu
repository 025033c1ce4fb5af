// pack.cu -- one-time repacking of an MXFP4 expert bank into the order the
// expert-FFN kernels stream it (sm_103a).
//
// The repacked bank holds exactly the bytes of the canonical bank (E2M1 codes
// and E8M0 exponents), permuted so that one warp-wide 16-byte load per lane
// delivers the mma.sync A-fragments of a 16-row x 64-element tile and one
// 4-byte load per lane its block exponents.  Layout (see packed_layout()):
//
// followed by two small sections (not a permutation of the canonical bytes)
// that the tensor-memory kernels read: one exponent base per weight row, in
// the unit-row order of each section (gate/up [E+S][2I], down [E+S][H]),
// each at a 256-byte aligned offset (launch_rowexp in tc.cu).
//
//   section gate/up: for expert e, for row block rb < I/8 (MMA rows 0..7 =
//     gate rows 8rb..8rb+7, MMA rows 8..15 = up rows I+8rb..I+8rb+7):
//   section down:    for expert e, for row block rb < H/16 (MMA rows 0..15 =
//     output rows 16rb..16rb+15):
//     for each 64-element step q < K/64 (K = H for gate/up, I for down),
//     544 bytes:
//       codes  512 B: lane l (g = l/4, c = l%4) owns bytes [16l, 16l+16) =
//              word c of block 2q of MMA row g, of row g+8, then word c of
//              block 2q+1 of row g, of row g+8 (a word = 8 codes);
//       scales  32 B: for g < 8, bytes [4g, 4g+4) = exponents of blocks 2q and
//              2q+1 of MMA row g, then of MMA row g+8.
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void pack_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, int n_experts,
                            int rows_per_expert, int K, int n_rb, int row_step, int row_gap,
                            uint8_t *__restrict__ out) {
    const int steps = K / 64;
    const long long n_items = (long long)n_experts * n_rb * steps * 34;   // 32 code lanes + 2 scale chunks
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_items;
         i += (long long)gridDim.x * blockDim.x) {
        const int part = (int)(i % 34);
        const long long step_id = i / 34;                 // (e, rb, q)
        const int q = (int)(step_id % steps);
        const long long unit = step_id / steps;           // e * n_rb + rb
        const int rb = (int)(unit % n_rb);
        const int e = (int)(unit / n_rb);
        uint8_t *dst = out + step_id * 544;
        auto mma_row = [&](int m) -> size_t {
            const int r = rb * row_step + m + (m >= 8 ? row_gap : 0);
            return (size_t)e * rows_per_expert + r;
        };
        if (part < 32) {
            const int g = part >> 2, c = part & 3;
            uint32_t w[4];
            const int blk[4] = {2 * q, 2 * q, 2 * q + 1, 2 * q + 1};
            const int mrow[4] = {g, g + 8, g, g + 8};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint8_t *src = codes + mma_row(mrow[j]) * (size_t)(K / 2) + blk[j] * 16 + c * 4;
                w[j] = *reinterpret_cast<const uint32_t *>(src);
            }
            *reinterpret_cast<uint4 *>(dst + part * 16) = make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            const int half = part - 32;                   // scale bytes of g = 4*half .. 4*half+3
            uint32_t v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int g = 4 * half + j;
                const uint8_t *s0 = scales + mma_row(g) * (size_t)(K / 32) + 2 * q;
                const uint8_t *s1 = scales + mma_row(g + 8) * (size_t)(K / 32) + 2 * q;
                v[j] = (uint32_t)s0[0] | ((uint32_t)s0[1] << 8) | ((uint32_t)s1[0] << 16) | ((uint32_t)s1[1] << 24);
            }
            *reinterpret_cast<uint4 *>(dst + 512 + half * 16) = make_uint4(v[0], v[1], v[2], v[3]);
        }
    }
}

PackedLayout packed_layout(int H, int I, int n_experts_total) {
    PackedLayout p{};
    p.gu_unit_bytes = (size_t)(H / 64) * 544;
    p.dn_unit_bytes = (size_t)(I / 64) * 544;
    p.gu_units_per_expert = I / 8;
    p.dn_units_per_expert = H / 16;
    p.gu_offset = 0;
    p.dn_offset = align_up(p.gu_unit_bytes * p.gu_units_per_expert * n_experts_total, 256);
    p.gu_rowexp = align_up(p.dn_offset + p.dn_unit_bytes * p.dn_units_per_expert * n_experts_total, 256);
    p.dn_rowexp = align_up(p.gu_rowexp + (size_t)n_experts_total * 2 * I, 256);
    p.total = align_up(p.dn_rowexp + (size_t)n_experts_total * H, 256);
    return p;
}

cudaError_t launch_pack(const moe_mxfp4_bank_t &b, uint8_t *out, cudaStream_t stream) {
    const int n = b.num_experts + b.has_shared;
    const PackedLayout L = packed_layout(b.hidden, b.inter, n);
    const int threads = 256, blocks = 4096;
    pack_kernel<<<blocks, threads, 0, stream>>>(b.w13, b.s13, n, 2 * b.inter, b.hidden, b.inter / 8, 8,
                                                b.inter - 8, out + L.gu_offset);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    pack_kernel<<<blocks, threads, 0, stream>>>(b.w2, b.s2, n, b.hidden, b.inter, b.hidden / 16, 16, 0,
                                                out + L.dn_offset);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    return launch_rowexp(b, out, stream);
}

}  // namespace moe
