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
// hardware, fp32 accumulators in TMEM.  The weight codes reach shared memory
// by tensor copies straight from row-major arrays; no decode instruction runs.
//
// Launches: routing + grouping and the x quantisation (for T <= 8 the
// routing phases of the single-launch kernel, which quantise x while they
// wait; else route.cu's two launches and mx8_quant_kernel), the gate/up GEMM
// (the g and u sums of each K chunk), mx8_hfin_kernel (h = silu(g) * u in
// fp32, quantised), the down GEMM (per-entry outputs Y), the combine
// (ffn.cu's combine_kernel).
//
// GEMM CTA: 128 weight rows x one pass of <= N entries (MMA M = 128, N = 16,
// or 32 for T > 128), K in stages of 128 (four MMAs of K = 32), over a
// 3-buffer shared-memory ring.  Thread 0 issues a stage's weight tile as two
// tensor copies of 64 rows x 128 codes (gate/up: the 64 gate rows, then the
// 64 up rows of the same indices) with the data type that gives every 16
// E2M1 codes a 16-byte slot (8 bytes of codes, the other 8 not written) and
// the 128-byte swizzle; the copies' 8,192 bytes complete the buffer's "full"
// mbarrier together with the four producer warps, which load the other
// operands into registers kMxRegStages stages ahead -- the activation codes
// (stored in the K-major no-swizzle layout: core matrices of 8 rows x 16
// bytes, adjacent in K 128 bytes apart, 8-row groups 1,024 bytes apart), the
// weight rows' and the activation rows' scale words (written into TMEM with
// tcgen05.st: row r of A at lane r % 32 of every 32-lane quarter, column base
// + r / 32; column n of B at lane n; byte j of a 32-bit cell is the scale of
// the stage's K block j, selected by the MMA's scale-factor id).  A fifth
// warp waits on the full barrier, issues the four MMAs (the weight operand
// through a 128-byte-swizzle descriptor: rows of 128 bytes, 8-row atoms 1,024
// bytes apart, a K step of 32 moving the start by 32 bytes) and commits them
// to the buffer's "empty" mbarrier, which the producers wait on before
// refilling the buffer; thread 0 then issues that buffer's next weight tile.
// Scale-factor regions start on 32-column (A) and 16-column (B) boundaries of
// the CTA's 128-column allocation (three CTAs per SM).
//
// The bank (moe_pack_bank_mx) is K-chunk major (below), so that a stage's
// 64-row tensor copy reads 4 KB of consecutive bytes.
#include <cuda.h>
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
constexpr int kMxABytes = 128 * kMxStageK;     // 128 rows x 8 slots x 16 B (the padded E2M1 image)
constexpr int kMxATx = 128 * kMxStageK / 2;    // bytes the tensor copies of a stage write (the codes)
constexpr int kMxTmemCols = 128;               // D: columns 0..N-1; scale factors on aligned columns
constexpr int kMxColSfa = 32;                  // SFA of buffer b: 4 columns at 32 + 32 b
constexpr int kMxColSfb = 48;                  // SFB of buffer b: 1 column at 48 + 32 b
constexpr int kMxCtasPerSm = 3;                // 3 x 128 TMEM columns, 3 x 55 (N = 16) or 61 KB shared memory
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
    const uint8_t *wscale;      // E8M0 scales of the weight rows [n_tot * rows][K/32]
    int rows;                   // weight rows per expert: 2I (gate/up) or H (down)
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

// 128-byte-swizzle K-major shared-memory descriptor (the weight tiles the
// tensor copies write): rows of 128 bytes, 8-row atoms 1,024 bytes apart,
// layout type 2 in bits 61-63; a K step of 32 elements moves the start by
// 32 bytes inside the atom.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

template <bool GATEUP, int NN>
__global__ void __launch_bounds__(kMxThreads, kMxCtasPerSm)
    mx8_gemm_kernel(const __grid_constant__ MxGemmArgs a, const __grid_constant__ CUtensorMap wmap) {
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
    // ---- weights: the tensor copies of a stage bring its 128 rows x 128
    // codes (gate/up: 64 gate rows, then the 64 up rows of the same
    // indices; down: 128 rows) into the stage's 128-byte-swizzled tile,
    // expanded by the copy to a 16-byte slot per 16 codes.
    // ---- producers: every other operand of a stage is loaded into
    // registers kMxRegStages stages ahead: the scale words of weight rows
    // lane + 32 q (q < 4); 16 bytes of activation rows tid / 8 + 16 j
    // (j < N / 16), slot tid % 8; the scale word of activation row
    // lane % N.  Each warp writes the scale factors into its own 32-lane
    // quarter of TMEM.
    auto wrow = [&](int r) {                      // weight row (within the expert) of MMA row r
        return GATEUP ? (r < 64 ? 64 * tile + r : a.half + 64 * tile + r - 64) : 128 * tile + r;
    };
    const int nch = a.K / kMxStageK;
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
    const uint8_t *sfa_src[4];                   // scale words: [expert][chunk][row][4]
#pragma unroll
    for (int i = 0; i < 4; ++i)
        sfa_src[i] = a.wscale + (((size_t)ps.expert * nch + s_first) * a.rows + wrow(lane + 32 * i)) * 4;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t rsa[kMxRegStages][4];
    uint4 rb[kMxRegStages][NB];
    uint32_t rsb[kMxRegStages];
    auto load_stage = [&](int s, uint32_t(&sa)[4], uint4(&bq)[NB], uint32_t &sb) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            sa[i] = __ldg(reinterpret_cast<const uint32_t *>(sfa_src[i] + (size_t)s * a.rows * 4));
#pragma unroll
        for (int j = 0; j < NB; ++j)
            bq[j] = __ldg(reinterpret_cast<const uint4 *>(asrc[j] + (size_t)s * kMxStageK));
        sb = __ldg(reinterpret_cast<const uint32_t *>(sfb_src + s * 4));
    };
    // weight rows of the tile for the tensor copies (row coordinate of each 64-row box)
    const int wr0 = wrow(0), wr1 = wrow(64);
    auto issue_weights = [&](int s, int b, uint32_t fb) {
        const uint32_t dst = sbase + (uint32_t)(b * kMxABytes);
        const int ck = ps.expert * nch + s_first + s;    // the expert's chunk
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(kMxATx) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {0, %2, %3}], "
            "[%4];" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(&wmap)), "r"(wr0), "r"(ck), "r"(fb)
            : "memory");
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {0, %2, %3}], "
            "[%4];" ::"r"(dst + kMxABytes / 2), "l"(reinterpret_cast<uint64_t>(&wmap)), "r"(wr1), "r"(ck), "r"(fb)
            : "memory");
    };
    // the first stages' loads go out before the TMEM allocation and barrier
    // set-up, whose latency they hide (they need only the pass)
    if (warp < kMxProducers / 32) {
#pragma unroll
        for (int k = 0; k < kMxRegStages; ++k)
            if (k < nst)
                load_stage(k, rsa[k], rb[k], rsb[k]);
    }
    // buffer b: full[b] completes when the 128 producers have staged a stage
    // in it (shared operands, scale factors in TMEM); empty[b] when the MMAs
    // reading it are done (tcgen05.commit)
    uint64_t *full = reinterpret_cast<uint64_t *>(mx_smem + (size_t)kMxStages * Tile::kStage);
    uint64_t *empty = full + kMxStages;
    uint8_t *bring = mx_smem + (size_t)kMxStages * kMxABytes;      // activation tiles after the weight tiles
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_taddr)),
                     "n"(kMxTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    // full[b]: the 128 producers' arrivals after their stores, plus the
    // weight copies' arrival with their byte count
    if (tid == 0) {
        for (int b = 0; b < kMxStages; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(full + b)), "r"(kMxProducers + 1));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(empty + b)));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int s = 0; s < kMxStages && s < nst; ++s)
            issue_weights(s, s, smem_addr(full + s));
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
                if (s >= kMxStages) {
                    if (!__all_sync(0xffffffffu,
                                    mbar_wait(smem_addr(empty + b), ((s - kMxStages) / kMxStages) & 1))) {
                        ok = false;       // warp-uniform: the tcgen05 stores below are .sync.aligned
                        break;
                    }
                    if (tid == 0)         // the buffer is free: its next weight tile
                        issue_weights(s, b, smem_addr(full + b));
                }
                uint8_t *st = bring + (size_t)b * Tile::kB;
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    const int r = r0 + 16 * j;
                    *reinterpret_cast<uint4 *>(st + (r >> 3) * kMxSbo + slot * kMxLbo + (r & 7) * 16) = rb[k][j];
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
                    load_stage(s + kMxRegStages, rsa[k], rb[k], rsb[k]);
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
            const uint32_t sa = sbase + (uint32_t)(b * kMxABytes);
            const uint32_t sb = smem_addr(bring) + (uint32_t)(b * Tile::kB);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint64_t ad = smem_desc_sw128(sa + 32 * j), bd = smem_desc(sb + j * 2 * kMxLbo);
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

}  // namespace

// ------------------------------------------------------------------ host

// The MXFP8 variant's bank, K-chunk major: per section (gate/up, then down),
// per expert, per chunk of 128 K elements, every weight row's 64 bytes of
// codes, then (separate sections) every row's 4 scale bytes of the chunk --
// codes [n_tot][K/128][rows][64], scales [n_tot][K/128][rows][4], each
// section at a 256-byte aligned offset.  A stage's 64-row tensor copy is then
// one contiguous 4 KB read and its scale words 512 contiguous bytes.
struct MxLayout {
    size_t w13, w2, s13, s2, total;
};
static MxLayout mx8_layout(int H, int I, int n_tot) {
    MxLayout m{};
    size_t o = 0;
    auto take = [&](size_t bytes) { o = align_up(o, 256); const size_t r = o; o += bytes; return r; };
    m.w13 = take((size_t)n_tot * 2 * I * (H / 2));
    m.w2 = take((size_t)n_tot * H * (I / 2));
    m.s13 = take((size_t)n_tot * 2 * I * (H / 32));
    m.s2 = take((size_t)n_tot * H * (I / 32));
    m.total = align_up(o, 256);
    return m;
}

size_t mx8_packed_size(int H, int I, int n_tot) { return mx8_layout(H, I, n_tot).total; }

// One 16-byte piece (codes) or 4-byte word (scales) per item: row r's bytes of
// chunk c go to [e][c][r].
__global__ void __launch_bounds__(256) mx8_pack_kernel(const uint8_t *__restrict__ w, const uint8_t *__restrict__ sc,
                                                       int n_tot, int rows, int K, uint8_t *__restrict__ wout,
                                                       uint8_t *__restrict__ sout) {
    const int nch = K / kMxStageK, K2 = K / 2, K32 = K / 32;
    const long long code_items = (long long)n_tot * rows * nch * 4;   // 4 pieces of 16 bytes per row and chunk
    const long long items = code_items + (long long)n_tot * rows * nch;
    for (long long it = (long long)blockIdx.x * blockDim.x + threadIdx.x; it < items;
         it += (long long)gridDim.x * blockDim.x) {
        if (it < code_items) {
            const int q = (int)(it & 3);
            const long long rc = it >> 2;                       // (e, c, r) in output order
            const int r = (int)(rc % rows);
            const long long ec = rc / rows;
            const int c = (int)(ec % nch), e = (int)(ec / nch);
            *reinterpret_cast<uint4 *>(wout + rc * 64 + 16 * q) =
                *reinterpret_cast<const uint4 *>(w + ((size_t)e * rows + r) * K2 + (size_t)c * 64 + 16 * q);
        } else {
            const long long rc = it - code_items;
            const int r = (int)(rc % rows);
            const long long ec = rc / rows;
            const int c = (int)(ec % nch), e = (int)(ec / nch);
            *reinterpret_cast<uint32_t *>(sout + rc * 4) =
                *reinterpret_cast<const uint32_t *>(sc + ((size_t)e * rows + r) * K32 + (size_t)c * 4);
        }
    }
}

cudaError_t launch_mx8_pack(const moe_mxfp4_bank_t &b, uint8_t *out, cudaStream_t stream) {
    const int H = b.hidden, I = b.inter, n = b.num_experts + b.has_shared;
    const MxLayout m = mx8_layout(H, I, n);
    mx8_pack_kernel<<<4096, 256, 0, stream>>>(b.w13, b.s13, n, 2 * I, H, out + m.w13, out + m.s13);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    mx8_pack_kernel<<<4096, 256, 0, stream>>>(b.w2, b.s2, n, H, I, out + m.w2, out + m.s2);
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
    // weight codes as 16 x E2M1 per 16-byte slot, 128-byte swizzle, boxes of
    // 128 codes x 64 rows
    const MxLayout ml = mx8_layout(H, I, n_tot);
    CUtensorMap gmap, dmap;
    {
        const uint64_t gdims[3] = {kMxStageK, (uint64_t)2 * I, (uint64_t)n_tot * (H / kMxStageK)};
        const uint64_t gstr[2] = {64, (uint64_t)2 * I * 64};
        const uint64_t ddims[3] = {kMxStageK, (uint64_t)H, (uint64_t)n_tot * (I / kMxStageK)};
        const uint64_t dstr[2] = {64, (uint64_t)H * 64};
        const uint32_t box[3] = {kMxStageK, 64, 1};
        if ((err = encode_tiled(&gmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, p.packed_mx + ml.w13, gdims, gstr,
                                box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess ||
            (err = encode_tiled(&dmap, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, p.packed_mx + ml.w2, ddims, dstr,
                                box, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
            return err;
    }
    MxGemmArgs g{};
    g.wscale = p.packed_mx + ml.s13;
    g.rows = 2 * I;
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
                          g, gmap)) != cudaSuccess)
        return err;
    if (ev && (err = cudaEventRecord(ev[1], stream)) != cudaSuccess)
        return err;
    const int hblocks = entries * (I / 32);
    if ((err = launch_pdl(mx8_hfin_kernel, dim3((hblocks + 7) / 8), dim3(256), 0, stream, (const float *)gu, g.kc,
                          g.kstride, entries, I, h32, hq, hs)) != cudaSuccess)
        return err;
    MxGemmArgs d = g;
    d.wscale = p.packed_mx + ml.s2;
    d.rows = H;
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
    if ((err = launch_pdl(mx8_gemm_kernel<false, NN>, dim3(H / 128, max_pass), dim3(kMxThreads), smem, stream, d,
                          dmap)) != cudaSuccess)
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
