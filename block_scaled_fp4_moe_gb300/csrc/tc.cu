// tc.cu -- the expert FFN for T > 8 on the fifth-generation tensor cores
// (tcgen05, sm_103a): exact MXFP4 weights x f16 activations, fp32
// accumulators in tensor memory.
//
// What it computes is the expert FFN of the layer (a4 gate/up + SiLU*up
// through the h finalisation, a5 down): "Optimizing GLM4-MoE for production"
// (SGLang / novita.ai), section 1 (the routed and shared experts as batched
// per-expert GEMMs over the grouped tokens); the MXFP4 block format is that of
// "GLM-5.2 on B300" (d9249.github.io), the quantisation section (E2M1 codes,
// one E8M0 exponent per 32 along K).  The tensor-memory accumulators follow
// the same page's kernel section 2 (tcgen05, accumulators and scale handling
// in TMEM instead of registers).
//
// Why this shape.  At T > 8 a pass carries 16..32 columns, so an mma.sync
// kernel issues four to eight MMAs and their block-scale FMAs per decoded
// fragment and becomes issue-bound well below the HBM rate.  Here the decode
// (E2M1 -> f16, the block exponent folded in by one f16x2 multiply per pair)
// is the only per-element work: the decoded 16-row units go straight into
// TMEM with tcgen05.st and are the A operand of tcgen05.mma.kind::f16
// (M = 128 weight rows, N = the pass's columns, K = 16); the activations are
// the B operand, brought into shared memory by one TMA tensor copy per
// stage.  The products are exact (f16 x f16), accumulated in fp32 over all
// of K by the tensor core.
//
// Layouts (found on the GPU with in-bounds probe MMAs):
//  * tcgen05.st.16x256b: thread t = 4g + c writes its registers r0, r1 to
//    lane g, columns 2c and 2c + 1, and r2, r3 to lane g + 8, same columns;
//    repetition j of .xN adds 8 j to the columns.
//  * kind::f16, A in TMEM, M = 128: lane m is row m; column j holds the pair
//    of K elements (2j, 2j + 1), the lower one in the low half.
//  * B in shared memory, K-major, no swizzle: core matrices of 8 rows x 16
//    bytes; the descriptor's leading offset is the stride between core
//    matrices adjacent in K, the stride offset the one between 8-row groups.
//
// K order.  A lane's 16-byte word of the repacked bank holds, for rows g and
// g + 8 of a unit, the codes of K positions 8c..8c+7 of two 32-blocks.  Stored
// with 16x256b, the 64 elements of a step land in TMEM in the order kappa =
// 32 r1 + 16 r0 + 4 c + 2 b + h for the element k = 32 r1 + 8 c + 4 r0 + 2 b
// + h of the step: a fixed permutation inside every 64-element step.  The
// products need the same K order on both sides, so the activations are kept
// in it: xsort_kernel writes x (f16, per-token scaled) per sorted entry in
// that order, and hfin_kernel writes h16 in it.  A 3-D tensor map (8
// elements x rows x K/8) then copies a stage of a pass's rows -- 256 K
// elements -- into the core-matrix layout in one instruction.
//
// Exponent range.  A decoded weight is code x 2^(s - b) in f16, where b is an
// exponent base per weight row chosen when the bank is packed (its largest
// block exponent minus 28, at least 0): every block whose exponent lies
// within 27 binades of the row's largest is exact in f16; a block 28 or more
// binades below it contributes zero (its products are below 2^-28 of the
// largest block's).  The epilogue multiplies the row's sums by 2^(b - 112),
// which restores 2^(s - 127); a row holding the NaN exponent 255 gets NaN.
//
// CTA (one per SM, persistent over work items = pass x 128-row tile of 8
// units).  Warp 8 streams the weights: a raw stage is each unit's next eight
// 544-byte steps (one 4,352-byte bulk copy per unit, read once from HBM with
// an evict-first hint) into a ring of four raw stages; warp 9 copies the
// pass's activation rows over the same 512 K elements (one tensor copy) into
// a ring of two tiles.  Warps 0..7 decode one unit each (warp w: unit
// 2 (w % 4) + w / 4 of the tile, TMEM lane quarter w % 4) from shared memory
// into a ring of three TMEM stages of 256 K elements.  Warp 10 issues a TMEM
// stage's 16 MMAs (K = 16) once it and its activation tile are full and
// commits them to the stages' "empty" barriers; after an item's last stage it
// commits to the accumulator's "full" barrier (two accumulators, so an item's
// epilogue overlaps the next item's MMAs).  Warps 12..15 (lane quarters
// 0..3) read the accumulator with tcgen05.ld and write the item's sums.
// Every wait is bounded (200 ms, then MOE_ERR_DEVICE_TIMEOUT) and stops the
// whole CTA.
//
// Items per CTA: the items are equal in cost, so every CTA first takes the
// same number of whole ones; the few left over are cut along K into pieces
// that go to the first CTAs, each writing its raw sums to a tail slot, and
// the CTA whose piece arrives last adds the slots in piece order (see
// TcSchedule).  The weight warp and the decoders start before the wait on
// the preceding grid: the pass lists and the weights are final when this
// grid launches; the activation warp and the epilogue wait first.
//
// Issue costs measured on the GPU (clock64 around back-to-back MMAs of one
// warp): a kind::f16 MMA with A in TMEM issues every ~17 cycles at N <= 32
// when its warp runs alone on its scheduler (A from shared memory: ~42, the
// operand read), ~130 at N = 256 (the tensor core's own rate); with three
// busy warps on the same scheduler it takes ~55-70 cycles.  The MMA warp
// therefore issues from a converged warp (one elected lane), with N a
// compile-time constant so that its operands stay warp-uniform.
#include <cuda.h>
#include <cuda_fp16.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Warp w may access only TMEM lane quarter w % 4 (MMA rows 32 (w % 4) ..).
constexpr int kTcUnits = 8;                               // 16-row units per 128-row tile
constexpr int kTcDecWarps = 8;                            // warp w < 8 decodes unit 2 (w % 4) + w / 4
constexpr int kTcProdWarp = 8;                            // weight stream
constexpr int kTcBProdWarp = 9;                           // activation tiles
constexpr int kTcMmaWarp = 10;
constexpr int kTcEpiWarp0 = 12;                           // warps 12..15: lane quarters 0..3
constexpr int kTcEpiWarps = 4;
constexpr int kTcWarps = 16;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcStageSteps = 4;                          // 64-element steps per TMEM stage
constexpr int kTcStageK = 64 * kTcStageSteps;             // 256
constexpr int kTcAStages = 3;                             // TMEM ring of decoded weights
constexpr int kTcNMax = 32;                               // MMA N (B rows per stage)
constexpr int kTcColsPerStage = kTcStageK / 2;            // 128 columns of f16 pairs
constexpr int kTcDCol = kTcAStages * kTcColsPerStage;     // 384: the two accumulators
constexpr int kTcTmemCols = 512;
constexpr int kTcRawSteps = 8;                            // steps per raw (shared-memory) stage: two TMEM stages
constexpr int kTcRawK = 64 * kTcRawSteps;                 // 512
constexpr int kTcRawStages = 4;                          // ring of weight stages
constexpr int kTcBStages = 2;                             // ring of activation tiles
constexpr int kTcUnitStage = kTcRawSteps * kStepBytes;    // 4,352 bytes of one unit per raw stage
constexpr int kTcRawA = kTcUnits * kTcUnitStage;          // 34,816: the tile's 8 units
constexpr int kTcRawBytes = 35 * 1024;                    // one weight stage, 1 KB aligned
constexpr int kTcBBytes = kTcNMax * kTcRawK * 2;          // one activation tile (32 KB)
constexpr int kTcBOff = kTcRawStages * kTcRawBytes;
static_assert(kTcRawA <= kTcRawBytes && kTcBOff % 1024 == 0, "stage layout");
constexpr size_t kTcSmem = (size_t)kTcBOff + (size_t)kTcBStages * kTcBBytes + 256;
constexpr unsigned long long kTcWaitLimitNs = 200ull * 1000 * 1000;
static_assert(kTcDCol + 2 * kTcNMax <= kTcTmemCols, "TMEM columns");

struct TcArgs {
    const uint8_t *packed;      // section of the repacked bank
    const uint8_t *rowexp;      // exponent bases of the section's rows, [n_tot][upe * 16] in unit-row order
    size_t unit_bytes;          // (K / 64) * 544
    int upe;                    // 16-row units per expert (a multiple of 8)
    int steps;                  // K / 64 (a multiple of 8)
    const Pass *passes;
    int passes_word;            // header word holding their number
    int rows_per_entry;         // B rows per entry: 1 (gate/up: x), 2 (down: h hi, lo)
    int n_entries;              // T * (k + S)
    int n_tot;
    uint32_t *hdr;
    float *part;                // gate/up: [entries][2][I] g, u sums; down: [entries][H] outputs
    int out_len;                // I (gate/up) or H (down)
    const float *bundo;         // down: per-entry factor undoing the h scaling
    float *tail;                // [kTcMaxPieces][128][32] partial sums of the K pieces of the last items
    uint32_t *tickets;          // [kTcMaxPieces] pieces done per split item (zero at kernel start)
};

constexpr int kTcMinSplitSaving = 4;        // raw stages a split must save on the busiest CTA

// Work of one CTA (index b of G): items b, b + G, ... whole while every CTA
// has one, then the r = n_items mod G items that are left, each cut along K
// into P pieces of S raw stages (P = 1: whole, round robin), so that the
// CTAs end together.  Pieces of item q G + k go to CTAs k P .. k P + P - 1;
// each writes its raw sums to the tail slot of its CTA index, and the CTA
// whose piece arrives last adds the P slots in piece order and writes the
// item's outputs -- the same order on every call.
struct TcSchedule {
    long long q;      // whole items per CTA
    int r, P, S;      // items left, pieces per such item, raw stages per piece
    int my_items;     // work items of this CTA
};

__device__ __forceinline__ TcSchedule tc_schedule(long long n_items, int G, int b, int nraw) {
    TcSchedule w;
    w.q = n_items / G;
    w.r = (int)(n_items % G);
    w.P = 1;
    w.S = nraw;
    if (w.r > 0) {
        int p0 = min(nraw, min(G, kTcMaxPieces) / w.r);
        p0 = max(p0, 1);
        w.S = (nraw + p0 - 1) / p0;
        w.P = (nraw + w.S - 1) / w.S;
        // a split costs the last piece's CTA an arrival and the sum (about
        // as long as three raw stages): only worth it for a larger saving
        if (nraw - w.S < kTcMinSplitSaving) {
            w.S = nraw;
            w.P = 1;
        }
    }
    w.my_items = (int)w.q + ((w.P > 1 ? b < w.r * w.P : b < w.r) ? 1 : 0);
    return w;
}

__device__ __forceinline__ bool tc_mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// try_wait that may suspend the thread for up to 0.1 ms (it resumes when the
// phase completes), so that waiting warps take no issue slots from the warps
// sharing their scheduler.
__device__ __forceinline__ bool tc_mbar_sleep(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(100000)
        : "memory");
    return done != 0;
}

// Wait for the phase of the barrier with this parity; false when the CTA's
// abort flag is up or after the time limit (which raises the flag).
__device__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag) {
    if (tc_mbar_try(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    while (!tc_mbar_sleep(bar, parity)) {
        if (*abort_flag)
            return false;
        if (globaltimer_ns() - t0 > kTcWaitLimitNs) {
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tc_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier 1 of the four epilogue warps; with a vote: true when every
// thread's v is true.
__device__ __forceinline__ void tc_epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kTcEpiWarps * 32) : "memory"); }

__device__ __forceinline__ bool tc_epi_and(bool v) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, %2, p;\nselp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kTcEpiWarps * 32)
        : "memory");
    return r != 0;
}

// Arrival counter of a split item: add one with acquire-release semantics at
// GPU scope, return the old count.
__device__ __forceinline__ uint32_t tc_ticket(uint32_t *t) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
    return old;
}

// Shared-memory descriptor, K-major, no swizzle.
__device__ __forceinline__ uint64_t tc_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr & 0x3FFFF) >> 4);
    d |= (uint64_t)(lbo >> 4) << 16;
    d |= (uint64_t)(sbo >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::f16: fp32 D (bits 4-5 = 1), A and B f16
// (format 0), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t tc_idesc_c(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24); }

// The f16x2 with both halves 2^(f - 15) for byte k of a word of f16 exponent
// fields pre-shifted left by 2 (f <= 28): bytes 1 and 3 of the result take
// byte k, bytes 0 and 2 are zero.
template <int K>
__device__ __forceinline__ uint32_t tc_splat(uint32_t f4s) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(f4s), "n"(4 | (K << 4) | (4 << 8) | (K << 12)));
    return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The fp32 factor that restores a row's block exponents: 2^(b - 112), NaN for
// a row holding the NaN exponent (b = 255).
__device__ __forceinline__ float tc_row_factor(uint32_t b) {
    return b == 255u ? __uint_as_float(0x7FC00000u) : __uint_as_float((b + 15u) << 23);
}

// The 16 MMAs (K = 16 each) of one TMEM stage, issued by one elected lane of
// a converged warp: A = TMEM columns acol + 8 k, B = half h of the raw
// stage's activation tile (core-matrix columns 32 h + 2 k, 2 k + 1); the
// item's first stage starts the accumulator.  N is a template parameter so
// that every descriptor is warp-uniform.
template <int N>
__device__ __forceinline__ void tc_issue_stage(uint32_t dcol, uint32_t acol, uint32_t bbase, int h, bool first) {
    constexpr uint32_t lbo = N * 16;
    const uint64_t bd0 = tc_desc(bbase + (uint32_t)h * 32u * lbo, lbo, 128);
    const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll
    for (int k = 0; k < kTcStageK / 16; ++k) {
        const uint32_t acc = k > 0 ? 1u : acc0;
        asm volatile(
            "{\n.reg .pred p, q;\nelect.sync _|p, 0xffffffff;\nsetp.ne.b32 q, %4, 0;\n"
            "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q;\n}\n" ::"r"(dcol),
            "r"(acol + 8 * k), "l"(bd0 + (uint64_t)((2 * k * lbo) >> 4)), "n"(tc_idesc_c(N)), "r"(acc)
            : "memory");
    }
}

template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    ffn_tc_kernel(const __grid_constant__ TcArgs a, const __grid_constant__ CUtensorMap map16,
                  const __grid_constant__ CUtensorMap map32) {
    extern __shared__ __align__(1024) uint8_t tc_smem[];
    __shared__ uint32_t s_taddr;
    __shared__ int s_abort;
    __shared__ int s_bad;
    __shared__ int s_last;
    __shared__ Pass s_pps;                    // the split item's pass and tile, and its rows'
    __shared__ int s_ptile;                   // exponent bases, left by the epilogue for the
    __shared__ uint32_t s_prb[128];           // sum after the final barrier
    // the warp index and every value a warp's control flow depends on are
    // broadcast from lane 0, so that the compiler treats them as warp-uniform
    const int tid = threadIdx.x, lane = tid & 31;
    const int warp = __shfl_sync(0xffffffffu, tid >> 5, 0);
    // The pass lists and the weights are final when this grid starts (the
    // grouping finished before the preceding kernel let it launch), so the
    // weight stream and the decode start at once; the warps that read what
    // the preceding kernel writes (activations, the h scale factors, the
    // arrival counters it clears) wait for it first.
    pdl_trigger();
    const int n_passes =
        __shfl_sync(0xffffffffu, (int)*reinterpret_cast<const volatile uint32_t *>(a.hdr + a.passes_word), 0);
    const int tiles = (a.upe + kTcUnits - 1) / kTcUnits;
    const int nraw = a.steps / kTcRawSteps;           // raw stages per item
    const long long n_items = (long long)n_passes * tiles;
    const TcSchedule sch = tc_schedule(n_items, (int)gridDim.x, (int)blockIdx.x, nraw);
    const int my_items = sch.my_items;
    if (my_items == 0)
        return;
    // work item j of this CTA: the item index, its raw stages [r0, r1) and
    // the tail slot it writes (-1: a whole item, written directly)
    auto item_of = [&](int j) -> long long {
        if (j < sch.q)
            return blockIdx.x + (long long)j * gridDim.x;
        return sch.q * gridDim.x + (sch.P > 1 ? (int)blockIdx.x / sch.P : (int)blockIdx.x);
    };
    auto stage_r0 = [&](int j) { return j < sch.q || sch.P == 1 ? 0 : ((int)blockIdx.x % sch.P) * sch.S; };
    auto stage_r1 = [&](int j) { return j < sch.q || sch.P == 1 ? nraw : min(nraw, stage_r0(j) + sch.S); };
    // every pass of this CTA's items lies inside the buffers, or the CTA does nothing
    if (tid == 0) {
        s_abort = 0;
        s_bad = 0;
        s_last = 0;
    }
    __syncthreads();
    for (int j = tid; j < my_items; j += blockDim.x) {
        const Pass ps = a.passes[item_of(j) / tiles];
        if (ps.expert < 0 || ps.expert >= a.n_tot || ps.count < 1 || ps.count * a.rows_per_entry > kTcNMax ||
            ps.begin < 0 || ps.begin + ps.count > a.n_entries)
            s_bad = 1;
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0)
            record_status(a.hdr, MOE_ERR_DEVICE_ASSERT);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(tc_smem + (size_t)kTcBOff + (size_t)kTcBStages * kTcBBytes);
    uint64_t *r_full = bars, *r_empty = bars + kTcRawStages;
    uint64_t *b_full = bars + 2 * kTcRawStages, *b_empty = b_full + kTcBStages;
    uint64_t *a_full = b_empty + kTcBStages, *a_empty = a_full + kTcAStages;
    uint64_t *d_full = a_empty + kTcAStages, *d_empty = d_full + 2;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_taddr)),
                     "n"(kTcTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (tid == 32) {
        for (int b = 0; b < kTcRawStages; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(r_full + b)));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(r_empty + b)), "r"(kTcDecWarps));
        }
        for (int b = 0; b < kTcBStages; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(b_full + b)));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(b_empty + b)));
        }
        for (int b = 0; b < kTcAStages; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(a_full + b)), "r"(kTcDecWarps));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(a_empty + b)));
        }
        for (int b = 0; b < 2; ++b) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(d_full + b)));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(d_empty + b)), "r"(kTcEpiWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_taddr;
    volatile int *abort_flag = &s_abort;
    auto item_pass = [&](int j) { return a.passes[item_of(j) / tiles]; };
    auto item_tile = [&](int j) { return (int)(item_of(j) % tiles); };
    auto tile_units = [&](int tile) { return min(kTcUnits, a.upe - tile * kTcUnits); };
    const uint32_t raw_base = smem_u32(tc_smem);

    if (warp < kTcDecWarps) {
        // ---- decoders: unit uw of each item's tile from the raw stage in
        // shared memory; rows g and g + 8 of the unit are TMEM lanes 16 uw + g, + 8
        const int uw = 2 * (warp & 3) + (warp >> 2);      // unit of the tile
        const int g = lane >> 2;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3) + 16 * (warp >> 2)) << 16;
        int rs = 0, gs = 0;
        bool ok = true;
        for (int j = 0; j < my_items && ok; ++j) {
            const Pass ps = item_pass(j);
            const int tile = item_tile(j);
            const bool present = uw < tile_units(tile);       // the last tile of an expert may be short
            uint32_t b4 = 0;
            if (present) {
                const uint8_t *re = a.rowexp + ((size_t)ps.expert * a.upe + tile * kTcUnits + uw) * 16;
                const uint32_t b0 = __ldg(re + g), b8 = __ldg(re + g + 8);
                b4 = b0 | (b0 << 8) | (b8 << 16) | (b8 << 24);
            }
            const int r1 = stage_r1(j);
            for (int r = stage_r0(j); r < r1; ++r, ++rs) {
                const int rb = rs % kTcRawStages;
                if (!__all_sync(0xffffffffu, tc_wait(smem_u32(r_full + rb), (rs / kTcRawStages) & 1, abort_flag))) {
                    ok = false;
                    break;
                }
                const uint8_t *src = tc_smem + (size_t)rb * kTcRawBytes + uw * kTcUnitStage;
#pragma unroll
                for (int h = 0; h < 2; ++h, ++gs) {
                    const int ab = gs % kTcAStages;
                    if (gs >= kTcAStages &&
                        !__all_sync(0xffffffffu,
                                    tc_wait(smem_u32(a_empty + ab), ((gs / kTcAStages) + 1) & 1, abort_flag))) {
                        ok = false;
                        break;
                    }
                    const uint32_t col = (uint32_t)(ab * kTcColsPerStage);
#pragma unroll
                    for (int t4 = 0; t4 < 4 && present; ++t4) {
                        const uint8_t *stp = src + (4 * h + t4) * kStepBytes;
                        const uint4 qq = *reinterpret_cast<const uint4 *>(stp + lane * 16);
                        const uint32_t ss = *reinterpret_cast<const uint32_t *>(stp + 512 + g * 4);
                        uint32_t P0[4], Q0[4], P1[4], Q1[4];
                        decode_e2m1x8(qq.x, P0);
                        decode_e2m1x8(qq.y, Q0);
                        decode_e2m1x8(qq.z, P1);
                        decode_e2m1x8(qq.w, Q1);
                        const uint32_t f4s = __vsubus4(ss, b4) << 2;
                        const uint32_t sg0 = tc_splat<0>(f4s), sg1 = tc_splat<1>(f4s);
                        const uint32_t sh0 = tc_splat<2>(f4s), sh1 = tc_splat<3>(f4s);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            P0[i] = hmul2(P0[i], sg0);
                            P1[i] = hmul2(P1[i], sg1);
                            Q0[i] = hmul2(Q0[i], sh0);
                            Q1[i] = hmul2(Q1[i], sh1);
                        }
                        asm volatile(
                            "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
                            "%13,%14,%15,%16};" ::"r"(tmem + lane_off + col + 32 * t4),
                            "r"(P0[0]), "r"(P0[1]), "r"(Q0[0]), "r"(Q0[1]), "r"(P0[2]), "r"(P0[3]), "r"(Q0[2]),
                            "r"(Q0[3]), "r"(P1[0]), "r"(P1[1]), "r"(Q1[0]), "r"(Q1[1]), "r"(P1[2]), "r"(P1[3]),
                            "r"(Q1[2]), "r"(Q1[3])
                            : "memory");
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0)
                        tc_arrive(smem_u32(a_full + ab));
                }
                if (!ok)
                    break;
                __syncwarp();                         // the unit's bytes of this raw stage are read
                if (lane == 0)
                    tc_arrive(smem_u32(r_empty + rb));
            }
        }
    } else if (warp == kTcProdWarp || warp == kTcBProdWarp) {
        // ---- producers.  Warp kTcProdWarp: a weight stage = each unit's next
        // 8 steps (one bulk copy per unit).  Warp kTcBProdWarp: an activation
        // tile = the pass's rows over the same 512 K elements (one tensor
        // copy).  Both rings advance once per raw stage.
        const bool weights = warp == kTcProdWarp;
        if (!weights)
            pdl_wait();
        const int nst = weights ? kTcRawStages : kTcBStages;
        uint64_t *full = weights ? r_full : b_full, *empty = weights ? r_empty : b_empty;
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int rs = 0;
            bool ok = true;
            for (int j = 0; j < my_items && ok; ++j) {
                const Pass ps = item_pass(j);
                const int rows = ps.count * a.rows_per_entry;
                const bool narrow = rows <= 16;
                const CUtensorMap *map = narrow ? &map16 : &map32;
                const int tile = item_tile(j), nu = tile_units(tile);
                const uint32_t bytes = weights ? (uint32_t)(nu * kTcUnitStage) : (narrow ? 16u : 32u) * (uint32_t)kTcRawK * 2u;
                const int row0 = ps.begin * a.rows_per_entry;
                const uint8_t *ubase = a.packed + ((size_t)ps.expert * a.upe + tile * kTcUnits) * a.unit_bytes;
                const int r1 = stage_r1(j);
                for (int r = stage_r0(j); r < r1; ++r, ++rs) {
                    const int rb = rs % nst;
                    if (rs >= nst && !tc_wait(smem_u32(empty + rb), ((rs / nst) + 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(full + rb);
                    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes)
                                 : "memory");
                    if (weights) {
                        const uint32_t dst = raw_base + (uint32_t)(rb * kTcRawBytes);
                        for (int u = 0; u < nu; ++u)
                            asm volatile(
                                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
                                "[%0], [%1], %2, [%3], %4;" ::"r"(dst + u * kTcUnitStage),
                                "l"(ubase + (size_t)u * a.unit_bytes + (size_t)r * kTcUnitStage), "n"(kTcUnitStage),
                                "r"(fb), "l"(pol)
                                : "memory");
                    } else {
                        asm volatile(
                            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
                            "[%1, {%2, %3, %4}], [%5];" ::"r"(raw_base + (uint32_t)(kTcBOff + rb * kTcBBytes)),
                            "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(r * (kTcRawK / 8)), "r"(fb)
                            : "memory");
                    }
                }
            }
            // copies still in flight land before the CTA leaves
            if (!ok)
                for (int k = 1; k <= nst && rs - k >= 0; ++k) {
                    const int c = rs - k;
                    const uint64_t t0 = globaltimer_ns();
                    while (!tc_mbar_try(smem_u32(full + c % nst), (c / nst) & 1) &&
                           globaltimer_ns() - t0 < kTcWaitLimitNs) {
                    }
                }
        }
    } else if (warp == kTcMmaWarp) {
        // ---- MMA issuer: the whole warp runs the loop (its values stay
        // warp-uniform) and one elected lane issues; TMEM stage gs is half
        // gs % 2 of raw stage gs / 2
        int gs = 0, committed = -1;
        bool ok = true;
        for (int j = 0; j < my_items && ok; ++j) {
            const int rows = __shfl_sync(0xffffffffu, item_pass(j).count * a.rows_per_entry, 0);
            const int n = rows <= 16 ? 16 : 32;
            const int db = j & 1;
            if (j >= 2 && !__all_sync(0xffffffffu, tc_wait(smem_u32(d_empty + db), ((j / 2) + 1) & 1, abort_flag))) {
                ok = false;
                break;
            }
            const uint32_t dcol = tmem + (uint32_t)(kTcDCol + kTcNMax * db);
            const int nst2 = 2 * (stage_r1(j) - stage_r0(j));
            for (int st = 0; st < nst2; ++st, ++gs) {
                const int ab = gs % kTcAStages, rs = gs >> 1, rb = rs % kTcBStages, h = gs & 1;
                if (!__all_sync(0xffffffffu, tc_wait(smem_u32(a_full + ab), (gs / kTcAStages) & 1, abort_flag)) ||
                    (h == 0 &&
                     !__all_sync(0xffffffffu, tc_wait(smem_u32(b_full + rb), (rs / kTcBStages) & 1, abort_flag)))) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t acol = tmem + (uint32_t)(ab * kTcColsPerStage);
                const uint32_t bbase = raw_base + (uint32_t)(kTcBOff + rb * kTcBBytes);
                if (n == 16)
                    tc_issue_stage<16>(dcol, acol, bbase, h, st == 0);
                else
                    tc_issue_stage<32>(dcol, acol, bbase, h, st == 0);
                asm volatile(
                    "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\n"
                    "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
                        smem_u32(a_empty + ab))
                    : "memory");
                if (h == 1)
                    asm volatile(
                        "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\n"
                        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
                            smem_u32(b_empty + rb))
                        : "memory");
                committed = gs;
            }
            if (!ok)
                break;
            asm volatile(
                "{\n.reg .pred p;\nelect.sync _|p, 0xffffffff;\n"
                "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
                    smem_u32(d_full + db))
                : "memory");
        }
        // a wait gave up: the MMAs already issued may still read TMEM and
        // shared memory; wait (bounded) for the commit that tracks them all
        if (!ok && committed >= 0 && lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            while (!tc_mbar_try(smem_u32(a_empty + committed % kTcAStages), (committed / kTcAStages) & 1) &&
                   globaltimer_ns() - t0 < kTcWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (warp >= kTcEpiWarp0 && warp < kTcEpiWarp0 + kTcEpiWarps) {
        // ---- epilogue: lane quarter q of the accumulator = MMA rows 32 q ..
        pdl_wait();
        const int qd = warp & 3;
        const int m = 32 * qd + lane;                 // MMA row of this lane
        bool ok = true;
        for (int j = 0; j < my_items && ok; ++j) {
            const Pass ps = item_pass(j);
            const int tile = item_tile(j);
            const int rows = ps.count * a.rows_per_entry;
            const int db = j & 1;
            const bool piece = j >= sch.q && sch.P > 1;
            const bool present = (m >> 4) < tile_units(tile);
            const uint32_t rb = present ? __ldg(a.rowexp + ((size_t)ps.expert * a.upe + tile * kTcUnits) * 16 + m) : 0u;
            const float fac = tc_row_factor(rb);
            if (piece) {
                s_prb[m] = rb;
                if (m == 0) {
                    s_pps = ps;
                    s_ptile = tile;
                }
            }
            const int u = tile * kTcUnits + (m >> 4), r = m & 15;
            const int col = MODE == kFfnGateUp ? (r < 8 ? 8 * u + r : a.out_len + 8 * u + r - 8) : 16 * u + r;
            // the outputs of the 16 columns of sums from column c0 on
            auto emit = [&](int c0, const float *v) {
                if (MODE == kFfnGateUp) {
                    // MMA row m = unit row r of unit u: gate row 8 u + r (r < 8), up row 8 u + r - 8
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int n = c0 + i;
                        if (present && n < ps.count && MOE_DBG_IN_RANGE(ps.begin + n, a.n_entries, a.hdr) &&
                            MOE_DBG_IN_RANGE(col, 2 * a.out_len, a.hdr))
                            a.part[(size_t)(ps.begin + n) * 2 * a.out_len + col] = v[i] * fac;
                    }
                } else {
                    // columns 2 j and 2 j + 1: the hi and lo parts of entry j
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int jj = c0 / 2 + i;
                        if (present && jj < ps.count && MOE_DBG_IN_RANGE(ps.begin + jj, a.n_entries, a.hdr) &&
                            MOE_DBG_IN_RANGE(col, a.out_len, a.hdr)) {
                            const int e = ps.begin + jj;
                            a.part[(size_t)e * a.out_len + col] = (v[2 * i] + v[2 * i + 1]) * fac * a.bundo[e];
                        }
                    }
                }
            };
            ok = __all_sync(0xffffffffu, tc_wait(smem_u32(d_full + db), (j / 2) & 1, abort_flag));
            // the four epilogue warps take every decision together (they meet
            // at a named barrier below)
            ok = tc_epi_and(ok);
            if (!ok)
                break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // the accumulator, 16 columns at a time: a whole item's outputs,
            // or a piece's raw sums into the tail slot of this CTA
            const uint32_t taddr = tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(kTcDCol + kTcNMax * db);
            float4 *slot = reinterpret_cast<float4 *>(a.tail + ((size_t)blockIdx.x * 128 + m) * kTcNMax);
#pragma unroll
            for (int c0 = 0; c0 < kTcNMax; c0 += 16) {
                if (c0 >= rows)
                    break;
                uint32_t w[16];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
                    "[%16];"
                    : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7]),
                      "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]),
                      "=r"(w[15])
                    : "r"(taddr + (uint32_t)c0));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                float v[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = __uint_as_float(w[i]);
                if (piece) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        slot[c0 / 4 + i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                } else {
                    emit(c0, v);
                }
            }
            // the accumulators are read: the MMAs of item j + 2 may overwrite them
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                tc_arrive(smem_u32(d_empty + db));
            if (piece) {
                // count the piece in (the acquire-release add publishes the
                // slot stores ordered before it by the barrier); the CTA of the
                // item's last piece adds the slots after the final barrier below
                tc_epi_sync();
                if (qd == 0 && lane == 0)
                    s_last = tc_ticket(a.tickets + (int)blockIdx.x / sch.P) == (uint32_t)(sch.P - 1);
            }
        }
    }
    pdl_wait();
    __syncthreads();
    if (s_abort && tid == 0)
        record_status(a.hdr, MOE_ERR_DEVICE_TIMEOUT);
    if (s_last && !s_abort) {
        // the split item's outputs: thread t takes row t / 4 of the tile and,
        // per 16 columns, columns 4 (t % 4) .. + 3, adding the P slots in
        // piece order (all slot loads issued at once)
        const Pass piece_ps = s_pps;
        const int piece_tile = s_ptile;
        const int rows = piece_ps.count * a.rows_per_entry;
        const int m = tid >> 2, c4 = 4 * (tid & 3);
        const int k = (int)blockIdx.x / sch.P;
        const int u = piece_tile * kTcUnits + (m >> 4), r = m & 15;
        const float fac = tc_row_factor(s_prb[m]);
        const bool present = (m >> 4) < tile_units(piece_tile);
        constexpr int kBatch = 16;
        for (int c0 = 0; c0 < kTcNMax && c0 < rows && present; c0 += 16) {
            float v[4];
            for (int p0 = 0; p0 < sch.P; p0 += kBatch) {
                float4 t[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
                    if (p0 + i < sch.P)
                        t[i] = __ldcg(reinterpret_cast<const float4 *>(
                            a.tail + ((size_t)(k * sch.P + p0 + i) * 128 + m) * kTcNMax + c0 + c4));
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
                    if (p0 + i < sch.P) {
                        if (p0 + i == 0) {
                            v[0] = t[i].x, v[1] = t[i].y, v[2] = t[i].z, v[3] = t[i].w;
                        } else {
                            v[0] += t[i].x, v[1] += t[i].y, v[2] += t[i].z, v[3] += t[i].w;
                        }
                    }
            }
            if (MODE == kFfnGateUp) {
                const int col = r < 8 ? 8 * u + r : a.out_len + 8 * u + r - 8;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int n = c0 + c4 + c;
                    if (n < piece_ps.count && MOE_DBG_IN_RANGE(piece_ps.begin + n, a.n_entries, a.hdr) &&
                        MOE_DBG_IN_RANGE(col, 2 * a.out_len, a.hdr))
                        a.part[(size_t)(piece_ps.begin + n) * 2 * a.out_len + col] = v[c] * fac;
                }
            } else {
                const int col = 16 * u + r;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int jj = (c0 + c4) / 2 + c;
                    if (jj < piece_ps.count && MOE_DBG_IN_RANGE(piece_ps.begin + jj, a.n_entries, a.hdr) &&
                        MOE_DBG_IN_RANGE(col, a.out_len, a.hdr)) {
                        const int e = piece_ps.begin + jj;
                        a.part[(size_t)e * a.out_len + col] = (v[2 * c] + v[2 * c + 1]) * fac * a.bundo[e];
                    }
                }
            }
        }
    }
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTcTmemCols));
}

// x (the per-token scaled f16 copy) gathered into sorted entry order, each
// 64-element step in the tensor-memory K order: position kappa of a step
// holds element k(kappa), so 16-byte chunk m of the step holds elements
// base_m .. base_m + 3 and base_m + 8 .. base_m + 11 with base_m = 32 (m / 4)
// + 16 (m % 2) + 4 ((m / 2) % 2).
__global__ void __launch_bounds__(256) xsort_kernel(const __half *__restrict__ x16, int H,
                                                   const int32_t *__restrict__ sorted_tok, int T, int entries,
                                                   __half *__restrict__ xs16, uint32_t *__restrict__ tickets,
                                                   uint32_t *__restrict__ hdr) {
    pdl_wait();
    pdl_trigger();
    // the arrival counters of the two tensor-memory kernels that follow
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < 2 * kTcMaxPieces; i += blockDim.x)
            tickets[i] = 0;
    const int e = blockIdx.x;
    if (e >= entries)
        return;
    const int tok = sorted_tok[e];
    if (tok < 0 || tok >= T) {
        if (threadIdx.x == 0)
            record_status(hdr, MOE_ERR_DEVICE_ASSERT);
        return;
    }
    const __half *src = x16 + (size_t)tok * H;
    __half *dst = xs16 + (size_t)e * H;
    for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
        const int step = c >> 3, mm = c & 7;
        const int base = 64 * step + 32 * (mm >> 2) + 16 * (mm & 1) + 4 * ((mm >> 1) & 1);
        const uint2 lo = *reinterpret_cast<const uint2 *>(src + base);
        const uint2 hi = *reinterpret_cast<const uint2 *>(src + base + 8);
        *reinterpret_cast<uint4 *>(dst + 8 * c) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
}

// Exponent base of each weight row (unit-row order of the repacked bank):
// 255 if the row holds the NaN exponent, else max(largest exponent - 28, 0).
__global__ void rowexp_kernel(const uint8_t *__restrict__ scales, int n_experts, int rows_per_expert, int K,
                              int n_units, int row_step, int row_gap, uint8_t *__restrict__ out) {
    const long long n = (long long)n_experts * n_units * 16;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i % 16);
        const long long uid = i / 16;
        const int u = (int)(uid % n_units);
        const int e = (int)(uid / n_units);
        const int r = u * row_step + m + (m >= 8 ? row_gap : 0);
        const uint8_t *s = scales + ((size_t)e * rows_per_expert + r) * (size_t)(K / 32);
        int mx = 0;
        bool nan = false;
        for (int b = 0; b < K / 32; ++b) {
            const int v = s[b];
            nan |= v == 255;
            mx = v > mx ? v : mx;
        }
        out[i] = nan ? (uint8_t)255 : (uint8_t)(mx > 28 ? mx - 28 : 0);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

}  // namespace

cudaError_t encode_tiled(CUtensorMap *m, CUtensorMapDataType type, int rank, const void *base, const uint64_t *dims,
                         const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i < rank - 1)
            st[i] = strides[i];
    }
    const CUresult r = fn(m, type, (cuuint32_t)rank, const_cast<void *>(base), d, st, b, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

// A 3-D view of rows x K f16 (rows in the tensor-memory K order) whose box of
// 8 elements x box_rows rows x 64 chunks is one raw stage of B in the
// core-matrix layout [chunk][row][16 bytes].
cudaError_t encode_b_map(CUtensorMap *m, const __half *base, long long rows, int K, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {8, (cuuint64_t)rows, (cuuint64_t)(K / 8)};
    const cuuint64_t strides[2] = {(cuuint64_t)K * 2, 16};
    const cuuint32_t box[3] = {8, (cuuint32_t)box_rows, (cuuint32_t)(kTcRawK / 8)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<__half *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int MODE>
cudaError_t launch_tc(const TcArgs &a, const CUtensorMap &m16, const CUtensorMap &m32, int num_sms,
                      cudaStream_t stream) {
    static std::atomic<int> attr_set{0};
    cudaError_t err;
    if (!attr_set.load()) {
        if ((err = cudaFuncSetAttribute(ffn_tc_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)kTcSmem)) != cudaSuccess)
            return err;
        attr_set.store(1);
    }
    return launch_pdl(ffn_tc_kernel<MODE>, dim3(num_sms), dim3(kTcThreads), kTcSmem, stream, a, m16, m32);
}

}  // namespace

bool tc_shape_supported(int H, int I) { return H % 512 == 0 && I % 512 == 0; }

cudaError_t launch_rowexp(const moe_mxfp4_bank_t &b, uint8_t *packed, cudaStream_t stream) {
    const int n = b.num_experts + b.has_shared;
    const PackedLayout L = packed_layout(b.hidden, b.inter, n);
    rowexp_kernel<<<1024, 256, 0, stream>>>(b.s13, n, 2 * b.inter, b.hidden, b.inter / 8, 8, b.inter - 8,
                                           packed + L.gu_rowexp);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess)
        return err;
    rowexp_kernel<<<1024, 256, 0, stream>>>(b.s2, n, b.hidden, b.inter, b.hidden / 16, 16, 0, packed + L.dn_rowexp);
    return cudaGetLastError();
}

cudaError_t launch_ffn_tc(const FfnProblem &pr, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                          cudaEvent_t ev_after_gateup) {
    const moe_mxfp4_bank_t &b = *pr.bank;
    const int H = b.hidden, I = b.inter, T = pr.T, kps = pr.kps;
    const int n_tot = b.num_experts + b.has_shared;
    const int entries = T * kps;
    const PackedLayout PL = packed_layout(H, I, n_tot);
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    cudaError_t err;
    __half *xs16 = ws_at<__half>(ws, L.xs16);
    __half *h16 = ws_at<__half>(ws, L.h16);
    uint32_t *tickets = ws_at<uint32_t>(ws, L.tc_tickets);
    float *tail = ws_at<float>(ws, L.tc_tail);
    CUtensorMap gm16, gm32, dm16, dm32;
    if ((err = encode_b_map(&gm16, xs16, entries, H, 16)) != cudaSuccess ||
        (err = encode_b_map(&gm32, xs16, entries, H, 32)) != cudaSuccess ||
        (err = encode_b_map(&dm16, h16, 2LL * entries, I, 16)) != cudaSuccess ||
        (err = encode_b_map(&dm32, h16, 2LL * entries, I, 32)) != cudaSuccess)
        return err;
    err = launch_pdl(xsort_kernel, dim3(entries), dim3(256), 0, stream, (const __half *)ws_at<__half>(ws, L.x16), H,
                     (const int32_t *)ws_at<int32_t>(ws, L.sorted_tok), T, entries, xs16, tickets, hdr);
    if (err != cudaSuccess)
        return err;
    TcArgs g{};
    g.packed = b.packed + PL.gu_offset;
    g.rowexp = b.packed + PL.gu_rowexp;
    g.unit_bytes = PL.gu_unit_bytes;
    g.upe = PL.gu_units_per_expert;
    g.steps = H / 64;
    g.passes = ws_at<Pass>(ws, L.passesw);
    g.passes_word = kHdrNumPassesW;
    g.rows_per_entry = 1;
    g.n_entries = entries;
    g.n_tot = n_tot;
    g.hdr = hdr;
    g.part = ws_at<float>(ws, L.gpart);
    g.out_len = I;
    g.tail = tail;
    g.tickets = tickets;
    if ((err = launch_tc<kFfnGateUp>(g, gm16, gm32, num_sms, stream)) != cudaSuccess)
        return err;
    if ((err = launch_hfin(ws, L, T, entries, I, true, stream)) != cudaSuccess)
        return err;
    if (ev_after_gateup && (err = cudaEventRecord(ev_after_gateup, stream)) != cudaSuccess)
        return err;
    TcArgs d{};
    d.packed = b.packed + PL.dn_offset;
    d.rowexp = b.packed + PL.dn_rowexp;
    d.unit_bytes = PL.dn_unit_bytes;
    d.upe = PL.dn_units_per_expert;
    d.steps = I / 64;
    d.passes = ws_at<Pass>(ws, L.passesw4);
    d.passes_word = kHdrNumPassesW4;
    d.rows_per_entry = 2;
    d.n_entries = entries;
    d.n_tot = n_tot;
    d.hdr = hdr;
    d.part = ws_at<float>(ws, L.ypart);
    d.out_len = H;
    d.bundo = ws_at<float>(ws, L.hundo);
    d.tail = tail;
    d.tickets = tickets + kTcMaxPieces;
    if ((err = launch_tc<kFfnDown>(d, dm16, dm32, num_sms, stream)) != cudaSuccess)
        return err;
    return launch_combine(ws_at<float>(ws, L.ypart), entries, ws_at<int32_t>(ws, L.inv_pos), pr.topk_w, T, kps, H,
                          pr.y, hdr, stream);
}

}  // namespace moe
