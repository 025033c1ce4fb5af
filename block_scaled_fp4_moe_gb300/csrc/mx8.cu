// mx8.cu -- the MXFP8 live-activation-quantisation variant of the layer, sm_103a.
//
// GLM-5.2 on B300 (d9249.github.io), kernel section 1: FP8 activation
// quantisation fused in front of the GEMM, and section 2: tcgen05 with the
// accumulators and scale handling in tensor memory (TMEM) instead of
// registers.  Here x (per token, along H) and h (per entry, along I) are
// quantised to MXFP8 -- E4M3 elements, one E8M0 scale per 32, the OCP MX v1.0
// conversion -- and both projections run as block-scaled tensor-core MMAs,
// `tcgen05.mma.kind::mxf8f6f4.block_scale`: A = MXFP4 weights read as E2M1 by
// the tensor core, B = the MXFP8 activations, both block scales applied by the
// hardware, fp32 accumulators in TMEM.  The weights are read from a
// stage-ordered copy of the bank (below); no decode instruction runs.
//
// Launches: routing + grouping and the x quantisation (for T <= 8 the
// routing phases of the single-launch kernel, which quantise x while they
// wait; else route.cu's two launches and mx8_quant_kernel), the gate/up GEMM
// (the g and u sums of each K chunk), mx8_hfin_kernel (h = silu(g) * u in
// fp32, quantised), the down GEMM (per-entry outputs Y), the combine
// (ffn.cu's combine_kernel).
//
// GEMM CTA: 128 weight rows x one pass of <= N entries (MMA M = 128, N = 16,
// or 32 for T > 128), K in stages of 128 (four MMAs of K = 32), warp-specialised: four
// producer warps load every operand of a stage into registers kMxRegStages
// stages ahead, store it into a 3-buffer shared-memory ring, write its scale
// factors into TMEM and arrive on the buffer's "full" mbarrier; a fifth warp
// waits on it, issues the four MMAs and commits them to the buffer's "empty"
// mbarrier, which the producers wait on before refilling the buffer.  The
// shared operands use the
// K-major no-swizzle layout: core matrices of 8 rows x 16 bytes, adjacent in
// K 128 bytes apart, 8-row groups 1,024 bytes apart.  An E2M1 operand of
// kind::mxf8f6f4 occupies a 16-byte slot per 16 elements with the 8 bytes of
// codes in the low half.  Scale factors go into TMEM with tcgen05.st: row r
// of A at lane r % 32 (in every 32-lane quarter), column base + r / 32;
// column n of B at lane n; byte j of a 32-bit cell is the scale of the
// stage's K block j, selected by the MMA's scale-factor id.
//
// The GEMMs read a stage-ordered copy of the bank (moe_pack_bank_mx): per
// (expert, 128-row tile, K stage) one contiguous block of 8,704 bytes: the
// codes in the order of the shared-memory image ([8-row group][16-byte slot]
// [row], 8 bytes each, at half the image's stride) except that within a
// group pieces w and w + 32 sit side by side, then the 128 rows' four scale
// bytes.  A stage is one linear 8.5 KB read (instead of 64 bytes from each
// of 128 rows), streamed through registers kMxRegStages stages ahead; a
// 16-byte chunk then holds two pieces whose slots are 32 apart, so the
// 8-byte shared stores of a warp cover 32 consecutive slots.  Scale-factor
// regions start on 32-column (A) and 16-column (B) boundaries of the CTA's
// 128-column allocation (three CTAs per SM).
#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kMxProducers = 128;              // warps 0..3 load and stage the operands
constexpr int kMxThreads = kMxProducers + 32;  // warp 4 issues the MMAs
constexpr int kMxStageK = 128;                 // K elements per stage
constexpr int kMxStages = 3;                   // shared-memory ring buffers
constexpr int kMxRegStages = 3;                // stages of operands in flight in registers
constexpr int kMxLbo = 128;                    // bytes between core matrices adjacent in K
constexpr int kMxSbo = 8 * 128;                // bytes between 8-row groups (8 K slots of 16 B)
constexpr int kMxABytes = 128 * kMxStageK;     // 128 rows x 8 slots x 16 B
constexpr int kMxTmemCols = 128;               // D: columns 0..N-1; scale factors on aligned columns
constexpr int kMxColSfa = 32;                  // SFA of buffer b: 4 columns at 32 + 32 b
constexpr int kMxColSfb = 48;                  // SFB of buffer b: 1 column at 48 + 32 b
constexpr int kMxCtasPerSm = 3;                // 3 x 128 TMEM columns, 3 x 55 (N = 16) or 61 KB shared memory
constexpr int kMxBlockBytes = 8192 + 512;      // one stage of a 128-row tile in the stage-ordered bank
constexpr unsigned long long kMxWaitLimitNs = 200ull * 1000 * 1000;
// Per MMA width N (entries of one pass: 16, or 32 for the wide passes of
// the multi-launch grouping): the B tile, a ring stage and the shared memory.
template <int NN>
struct MxTile {
    static_assert(NN == 16 || NN == 32, "N");
    static constexpr int kB = NN * kMxStageK;                 // NN rows x 128 E4M3
    static constexpr int kStage = kMxABytes + kB;
    static constexpr size_t kSmem = (size_t)kMxStages * kStage + 2 * kMxStages * 8;   // buffers, full / empty barriers
};

static_assert(kMxColSfb + 32 * (kMxStages - 1) + 1 <= kMxTmemCols && kMxCtasPerSm * kMxTmemCols <= 512 &&
                  32 <= kMxColSfa,
              "TMEM columns: D (up to 32 columns) below the scale factors");

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor: start, leading (K) and stride (8-row)
// byte offsets, the fixed 0b001 at bits 46-48, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)(kMxLbo >> 4) << 16;
    d |= (uint64_t)(kMxSbo >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E2M1 (5),
// B E4M3 (0), both K-major, N >> 3 at bit 17, UE8M0 scales (bit 23),
// M >> 4 at bit 24; scale-factor ids (byte of the TMEM cell) of B at bits
// 4-5 and of A at bits 29-30.
template <int NN>
__host__ __device__ constexpr uint32_t mx_idesc(int sf_id) {
    return ((uint32_t)(sf_id & 3) << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(NN >> 3) << 17) | (1u << 23) |
           ((uint32_t)(128 >> 4) << 24) | ((uint32_t)(sf_id & 3) << 29);
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait until the barrier's phase with this parity has completed; false after
// kMxWaitLimitNs.
__device__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try(bar, parity))
        if (globaltimer_ns() - t0 > kMxWaitLimitNs)
            return false;
    return true;
}

struct MxGemmArgs {
    const uint8_t *blocks;      // section of the stage-ordered bank: [n_tot][tiles][K/128] blocks
    const uint8_t *aq;          // E4M3 activations [act_rows][K]
    const uint8_t *asc;         // E8M0 scales [act_rows][K/32]
    const Pass *passes;         // passes of <= N entries
    int npass_word;             // header word holding the number of passes
    const int32_t *sorted_tok;  // gate/up: entry -> activation row (token); down: null (row = entry)
    float *out;                 // [kc][entries][rows]: per K chunk, the sums of every weight row
                                // (gate/up: g then u, 2I columns; down: Y, H columns)
    uint32_t *hdr;
    int tiles;                  // 128-row tiles per expert: I/64 (gate/up) or H/128 (down)
    int K;                      // H (gate/up) or I (down)
    int half;                   // gate/up: I (up rows start there); down: 0
    int out_ld;                 // 2I (gate/up) or H (down)
    int kc;                     // K chunks (split K): blockIdx.x = tile * kc + chunk
    size_t kstride;             // floats between the chunks' outputs
    int n_tot;                  // experts in the bank
    int act_rows;               // rows of aq: T (gate/up) or entries (down)
    int entries;                // T * (k + S)
};

// ------------------------------------------------------------------ GEMM

template <bool GATEUP, int NN>
__global__ void __launch_bounds__(kMxThreads, kMxCtasPerSm) mx8_gemm_kernel(const __grid_constant__ MxGemmArgs a) {
    using Tile = MxTile<NN>;
    extern __shared__ __align__(1024) uint8_t mx_smem[];
    __shared__ uint32_t s_taddr;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_trigger();
    const int n_pass = (int)*reinterpret_cast<const volatile uint32_t *>(a.hdr + a.npass_word);
    if ((int)blockIdx.y >= n_pass)
        return;
    const Pass ps = a.passes[blockIdx.y];
    const int tile = blockIdx.x / a.kc, chunk = blockIdx.x - tile * a.kc;
    // the pass and its activation rows must lie inside the buffers
    {
        int bad = ps.expert < 0 || ps.expert >= a.n_tot || ps.count < 1 || ps.count > NN || ps.begin < 0 ||
                  ps.begin + ps.count > a.entries;
        if (!bad && tid < ps.count) {
            const int row = GATEUP ? a.sorted_tok[ps.begin + tid] : ps.begin + tid;
            bad = row < 0 || row >= a.act_rows;
        }
        if (__syncthreads_or(bad)) {
            if (tid == 0)
                record_status(a.hdr, MOE_ERR_DEVICE_ASSERT);
            return;
        }
    }
    const int K32 = a.K / 32;
    const int nst = a.K / kMxStageK / a.kc;          // stages of this chunk
    const int s_first = chunk * nst;
    const uint32_t sbase = smem_addr(mx_smem);
    // ---- producers.  Every operand of a stage is loaded into registers
    // kMxRegStages stages ahead: weight codes as 16-byte chunks c = tid +
    // 128 i (i < 4) of the block, holding the pieces q0 = 64 (c / 32) +
    // c % 32 and q0 + 32 of the shared-memory image (each 8-byte store of
    // a warp then covers 32 consecutive slots); the scale words of rows
    // lane + 32 q (q < 4); 16 bytes of activation rows tid / 8 + 16 j
    // (j < N / 16), slot tid % 8; the scale word of activation row
    // lane % N.  Each warp writes the scale factors into its own 32-lane
    // quarter of TMEM.
    const uint8_t *wblk =
        a.blocks + (((size_t)ps.expert * a.tiles + tile) * a.kc * nst + s_first) * kMxBlockBytes;
    auto arow = [&](int n) {
        const int e = ps.begin + min(n, ps.count - 1);
        return GATEUP ? a.sorted_tok[e] : e;
    };
    const int slot = tid & 7, r0 = tid >> 3;
    constexpr int NB = NN / 16;                  // activation chunks per thread
    const uint8_t *asrc[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j)
        asrc[j] = a.aq + (size_t)arow(r0 + 16 * j) * a.K + (size_t)s_first * kMxStageK + slot * 16;
    const uint8_t *sfb_src = a.asc + (size_t)arow(lane % NN) * K32 + s_first * 4;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const uint64_t pol = l2_evict_first_policy();
    uint4 rq[kMxRegStages][4];
    uint32_t rsa[kMxRegStages][4];
    uint4 rb[kMxRegStages][NB];
    uint32_t rsb[kMxRegStages];
    auto load_stage = [&](int s, uint4(&q)[4], uint32_t(&sa)[4], uint4(&bq)[NB], uint32_t &sb) {
        const uint8_t *blk = wblk + (size_t)s * kMxBlockBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q[i] = ld_stream16(blk + 16 * (tid + kMxProducers * i), pol);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            sa[i] = __ldg(reinterpret_cast<const uint32_t *>(blk + 8192 + 4 * (lane + 32 * i)));
#pragma unroll
        for (int j = 0; j < NB; ++j)
            bq[j] = __ldg(reinterpret_cast<const uint4 *>(asrc[j] + (size_t)s * kMxStageK));
        sb = __ldg(reinterpret_cast<const uint32_t *>(sfb_src + s * 4));
    };
    // the first stages' loads go out before the TMEM allocation and barrier
    // set-up, whose latency they hide (they need only the pass)
    if (warp < kMxProducers / 32) {
#pragma unroll
        for (int k = 0; k < kMxRegStages; ++k)
            if (k < nst)
                load_stage(k, rq[k], rsa[k], rb[k], rsb[k]);
    }
    // buffer b: full[b] completes when the 128 producers have staged a stage
    // in it (shared operands, scale factors in TMEM); empty[b] when the MMAs
    // reading it are done (tcgen05.commit)
    uint64_t *full = reinterpret_cast<uint64_t *>(mx_smem + (size_t)kMxStages * Tile::kStage);
    uint64_t *empty = full + kMxStages;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_taddr)),
                     "n"(kMxTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 0) {
        for (int b = 0; b < kMxStages; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(full + b)), "r"(kMxProducers));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(empty + b)));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_taddr;
    bool ok = true;

    if (warp < kMxProducers / 32) {
        for (int s0 = 0; s0 < nst && ok; s0 += kMxRegStages) {
#pragma unroll
            for (int k = 0; k < kMxRegStages; ++k) {
                const int s = s0 + k;
                if (s >= nst)
                    break;
                const int b = s % kMxStages;
                // buffer b and its TMEM columns were read by the MMAs of stage s - kMxStages
                if (s >= kMxStages &&
                    !__all_sync(0xffffffffu, mbar_wait(smem_addr(empty + b), ((s - kMxStages) / kMxStages) & 1))) {
                    ok = false;           // warp-uniform: the tcgen05 stores below are .sync.aligned
                    break;
                }
                uint8_t *st = mx_smem + (size_t)b * Tile::kStage;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = tid + kMxProducers * i;
                    const int q0 = 64 * (c >> 5) + (c & 31);
                    *reinterpret_cast<uint2 *>(st + 16 * q0) = make_uint2(rq[k][i].x, rq[k][i].y);
                    *reinterpret_cast<uint2 *>(st + 16 * (q0 + 32)) = make_uint2(rq[k][i].z, rq[k][i].w);
                }
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int r = r0 + 16 * j;
                    *reinterpret_cast<uint4 *>(st + kMxABytes + (r >> 3) * kMxSbo + slot * kMxLbo + (r & 7) * 16) =
                        rb[k][j];
                }
                const uint32_t colA = (uint32_t)(kMxColSfa + 32 * b), colB = (uint32_t)(kMxColSfb + 32 * b);
                asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 tmem + lane_base + colA),
                             "r"(rsa[k][0]), "r"(rsa[k][1]), "r"(rsa[k][2]), "r"(rsa[k][3])
                             : "memory");
                asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tmem + lane_base + colB),
                             "r"(rsb[k])
                             : "memory");
                if (s + kMxRegStages < nst)
                    load_stage(s + kMxRegStages, rq[k], rsa[k], rb[k], rsb[k]);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(full + b)) : "memory");
            }
        }
        // the last commit covers every MMA of the CTA
        if (ok)
            ok = __all_sync(0xffffffffu,
                            mbar_wait(smem_addr(empty + (nst - 1) % kMxStages), ((nst - 1) / kMxStages) & 1));
    } else if (lane == 0) {
        // ---- the MMA issuer
        int committed = -1;                  // last stage whose MMAs were committed
        for (int s = 0; s < nst; ++s) {
            const int b = s % kMxStages;
            if (!mbar_wait(smem_addr(full + b), (s / kMxStages) & 1)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t colA = (uint32_t)(kMxColSfa + 32 * b), colB = (uint32_t)(kMxColSfb + 32 * b);
            const uint32_t sa = sbase + (uint32_t)(b * Tile::kStage), sb = sa + kMxABytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t ad = smem_desc(sa + j * 2 * kMxLbo), bd = smem_desc(sb + j * 2 * kMxLbo);
                const uint32_t acc = (s > 0 || j > 0) ? 1u : 0u;
                asm volatile(
                    "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                    "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n}\n"
                    ::"r"(tmem), "l"(ad), "l"(bd), "r"(mx_idesc<NN>(j)), "r"(acc), "r"(tmem + colA), "r"(tmem + colB)
                    : "memory");
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_addr(empty + b))
                         : "memory");
            committed = s;
        }
        // a wait gave up: the MMAs already issued may still read shared
        // memory and TMEM; wait (bounded) for the last commit, which tracks
        // all of them, before the CTA frees its TMEM and leaves
        if (!ok && committed >= 0)
            mbar_wait(smem_addr(empty + committed % kMxStages), (committed / kMxStages) & 1);
    }
    ok = !__syncthreads_or(!ok);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (!ok) {
        if (tid == 0)
            record_status(a.hdr, MOE_ERR_DEVICE_TIMEOUT);
    } else if (warp < kMxProducers / 32) {
        uint32_t v[NN];
#pragma unroll
        for (int c0 = 0; c0 < NN; c0 += 16)
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                "[%16];"
                : "=r"(v[c0]), "=r"(v[c0 + 1]), "=r"(v[c0 + 2]), "=r"(v[c0 + 3]), "=r"(v[c0 + 4]), "=r"(v[c0 + 5]),
                  "=r"(v[c0 + 6]), "=r"(v[c0 + 7]), "=r"(v[c0 + 8]), "=r"(v[c0 + 9]), "=r"(v[c0 + 10]),
                  "=r"(v[c0 + 11]), "=r"(v[c0 + 12]), "=r"(v[c0 + 13]), "=r"(v[c0 + 14]), "=r"(v[c0 + 15])
                : "r"(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        // MMA row r = TMEM lane = weight row of the tile: gate/up rows 0..63
        // are gate rows 64 tile.., 64..127 the up rows; output column = that
        // weight row's index
        const int r = tid;
        const int col = GATEUP ? (r < 64 ? tile * 64 + r : a.half + tile * 64 + r - 64) : tile * 128 + r;
        float *dst = a.out + chunk * a.kstride + (size_t)ps.begin * a.out_ld + col;
#pragma unroll
        for (int n = 0; n < NN; ++n)
            if (n < ps.count)
                dst[(size_t)n * a.out_ld] = __uint_as_float(v[n]);
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kMxTmemCols));
}

// ------------------------------------------------------------ quantisation

// x (bf16 [T][H]) to MXFP8, one warp per block of 32.
__global__ void __launch_bounds__(256) mx8_quant_kernel(const uint16_t *__restrict__ x, int rows, int cols,
                                                        uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
    pdl_wait();
    pdl_trigger();
    const long long blk = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (blk >= (long long)rows * (cols / 32))
        return;
    const size_t i = (size_t)blk * 32 + (threadIdx.x & 31);
    mxfp8_quant_block(__uint_as_float((uint32_t)x[i] << 16), codes + i, scales + blk);
}

// h = silu(g) * u from the gate/up GEMM's K-chunk sums (g and u each summed
// over the chunks in chunk order), written in fp32 and as MXFP8; one warp per
// block of 32 of an entry's h.
__global__ void __launch_bounds__(256) mx8_hfin_kernel(const float *__restrict__ gu, int kc, size_t kstride,
                                                       int entries, int I, float *__restrict__ h32,
                                                       uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
    pdl_wait();
    pdl_trigger();
    const long long blk = (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int per = I / 32;
    if (blk >= (long long)entries * per)
        return;
    const int e = (int)(blk / per), j = (int)(blk - (long long)e * per);
    const int i = 32 * j + (threadIdx.x & 31);
    const float *src = gu + (size_t)e * 2 * I + i;
    float g = 0.0f, u = 0.0f;
    for (int c = 0; c < kc; ++c) {
        g += __ldcg(src + c * kstride);
        u += __ldcg(src + c * kstride + I);
    }
    const float h = g / (1.0f + expf(-g)) * u;
    h32[(size_t)e * I + i] = h;
    mxfp8_quant_block(h, codes + (size_t)e * I + i, scales + blk);
}

// Stage-ordered copy of one section of the bank: one thread per 8-byte code
// piece (q < 1024) or 4-byte scale word (q >= 1024) of a block.  Tile rows:
// gate/up (half = I) rows 0..63 are gate rows 64t.., rows 64..127 the up rows
// I + 64t..; down (half = 0) rows 128t...
__global__ void __launch_bounds__(256) mx8_pack_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sc,
                                                       int n_tot, int rows, int K, int tiles, int half,
                                                       uint8_t *__restrict__ out) {
    const int nst = K / kMxStageK, K2 = K / 2, K32 = K / 32;
    const long long items = (long long)n_tot * tiles * nst * 1152;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (long long)gridDim.x * blockDim.x) {
        const long long blk = it / 1152;
        const int q = (int)(it - blk * 1152);
        const int s = (int)(blk % nst);
        const long long et = blk / nst;
        const int t = (int)(et % tiles), e = (int)(et / tiles);
        const int r = q < 1024 ? 8 * (q >> 6) + (q & 7) : q - 1024;
        const int row = half ? (r < 64 ? 64 * t + r : half + 64 * t + r - 64) : 128 * t + r;
        uint8_t *dst = out + blk * kMxBlockBytes;
        if (q < 1024) {
            const int j = (q >> 3) & 7, piece = q & 63;
            const int pos = (q & ~63) + 2 * (piece & 31) + (piece >> 5);   // pieces l and l + 32 side by side
            *reinterpret_cast<uint2 *>(dst + 8 * pos) =
                *reinterpret_cast<const uint2 *>(w + ((size_t)e * rows + row) * K2 + s * 64 + j * 8);
        } else {
            *reinterpret_cast<uint32_t *>(dst + 8192 + 4 * r) =
                *reinterpret_cast<const uint32_t *>(sc + ((size_t)e * rows + row) * K32 + s * 4);
        }
    }
}

}  // namespace

// ------------------------------------------------------------------ host

size_t mx8_packed_size(int H, int I, int n_tot) {
    return (size_t)n_tot * ((size_t)(I / 64) * (H / 128) + (size_t)(H / 128) * (I / 128)) * kMxBlockBytes;
}

static size_t mx8_dn_offset(int H, int I, int n_tot) {
    return (size_t)n_tot * (I / 64) * (H / 128) * kMxBlockBytes;
}

cudaError_t launch_mx8_pack(const moe_mxfp4_bank_t &b, uint8_t *out, cudaStream_t stream) {
    const int H = b.hidden, I = b.inter, n = b.num_experts + b.has_shared;
    mx8_pack_kernel<<<4096, 256, 0, stream>>>(b.w13, b.s13, n, 2 * I, H, I / 64, I, out);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    mx8_pack_kernel<<<4096, 256, 0, stream>>>(b.w2, b.s2, n, H, I, H / 128, 0, out + mx8_dn_offset(H, I, n));
    return cudaGetLastError();
}

bool mx8_shape_supported(int H, int I) { return H > 0 && I > 0 && H % 128 == 0 && I % 128 == 0; }

// The two GEMMs with MMA width NN around the h finalisation, then the combine.
template <int NN>
static cudaError_t launch_gemms(const Mx8Problem &p, void *ws, const WsLayout &L, cudaStream_t stream,
                                cudaEvent_t *ev, const Pass *passes, int npass_word, int max_pass) {
    const moe_mxfp4_bank_t &b = *p.bank;
    const int H = b.hidden, I = b.inter, T = p.T, kps = p.kps;
    const int entries = T * kps;
    const int n_tot = b.num_experts + b.has_shared;
    constexpr size_t smem = MxTile<NN>::kSmem;
    static std::atomic<int> attr_set{0};
    cudaError_t err;
    if (!attr_set.load()) {
        if ((err = cudaFuncSetAttribute(mx8_gemm_kernel<true, NN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(mx8_gemm_kernel<false, NN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess)
            return err;
        attr_set.store(1);
    }
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    uint8_t *hq = ws_at<uint8_t>(ws, L.mx_hq), *hs = ws_at<uint8_t>(ws, L.mx_hs);
    float *h32 = ws_at<float>(ws, L.mx_h32), *yent = ws_at<float>(ws, L.mx_y), *gu = ws_at<float>(ws, L.mx_gu);
    MxGemmArgs g{};
    g.blocks = p.packed_mx;
    g.aq = ws_at<uint8_t>(ws, L.mx_xq);
    g.asc = ws_at<uint8_t>(ws, L.mx_xs);
    g.passes = passes;
    g.npass_word = npass_word;
    g.sorted_tok = ws_at<int32_t>(ws, L.sorted_tok);
    g.out = gu;
    g.hdr = hdr;
    g.tiles = I / 64;
    g.K = H;
    g.half = I;
    g.kc = L.mx_kc_gu;
    g.kstride = (size_t)entries * 2 * I;
    g.out_ld = 2 * I;
    g.n_tot = n_tot;
    g.act_rows = T;
    g.entries = entries;
    if ((err = launch_pdl(mx8_gemm_kernel<true, NN>, dim3(I / 64 * g.kc, max_pass), dim3(kMxThreads), smem, stream,
                          g)) != cudaSuccess)
        return err;
    if (ev && (err = cudaEventRecord(ev[1], stream)) != cudaSuccess)
        return err;
    const int hblocks = entries * (I / 32);
    if ((err = launch_pdl(mx8_hfin_kernel, dim3((hblocks + 7) / 8), dim3(256), 0, stream, (const float *)gu, g.kc,
                          g.kstride, entries, I, h32, hq, hs)) != cudaSuccess)
        return err;
    MxGemmArgs d = g;
    d.blocks = p.packed_mx + mx8_dn_offset(H, I, n_tot);
    d.aq = hq;
    d.asc = hs;
    d.sorted_tok = nullptr;
    d.out = yent;
    d.tiles = H / 128;
    d.K = I;
    d.half = 0;
    d.kc = 1;
    d.kstride = 0;
    d.out_ld = H;
    d.act_rows = entries;
    if ((err = launch_pdl(mx8_gemm_kernel<false, NN>, dim3(H / 128, max_pass), dim3(kMxThreads), smem, stream, d)) !=
        cudaSuccess)
        return err;
    return launch_combine(yent, entries, ws_at<int32_t>(ws, L.inv_pos), p.topk_w, T, kps, H, p.y, hdr, stream);
}

cudaError_t launch_mx8_ffn(const Mx8Problem &p, void *ws, const WsLayout &L, cudaStream_t stream, cudaEvent_t *ev) {
    const moe_mxfp4_bank_t &b = *p.bank;
    const int H = b.hidden, T = p.T, kps = p.kps;
    const int n_tot = b.num_experts + b.has_shared;
    cudaError_t err = cudaSuccess;
    if (!p.x_quantised &&
        (err = launch_pdl(mx8_quant_kernel, dim3((T * (H / 32) + 7) / 8), dim3(256), 0, stream, p.x, T, H,
                          ws_at<uint8_t>(ws, L.mx_xq), ws_at<uint8_t>(ws, L.mx_xs))) != cudaSuccess)
        return err;
    if (ev && (err = cudaEventRecord(ev[0], stream)) != cudaSuccess)
        return err;
    // routing by the single-launch kernel's phases (which also quantised x)
    // exports passes of one expert's <= 8 entries; the multi-launch grouping
    // also writes passes of <= 32, which the wider MMA (N = 32) reads for
    // T > 128, where experts with many tokens re-read their weights half as
    // often (measured: Zipf T = 256 798 -> 764 us; at T = 64 the fewer,
    // heavier CTAs cost more than that: 355 -> 388 us)
    if (p.x_quantised || T <= 128)
        return launch_gemms<16>(p, ws, L, stream, ev, ws_at<Pass>(ws, L.passesw4), kHdrNumPassesW4,
                                max_passes(T, kps, n_tot, kWidePassEntries));
    return launch_gemms<32>(p, ws, L, stream, ev, ws_at<Pass>(ws, L.passesw), kHdrNumPassesW,
                            max_passes(T, kps, n_tot, kWidePassTokens));
}

}  // namespace moe
