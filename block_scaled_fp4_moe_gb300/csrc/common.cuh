// common.cuh -- shared definitions of the sm_103a MoE kernels: workspace
// layout, status word, and thin wrappers over the PTX the kernels use
// (mbarrier, bulk async copies, mma.sync, E2M1 conversion).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "moe_fp4.h"

namespace moe {

// ------------------------------------------------------------------ sizes

constexpr int kRouteRows = 512;       // router rows (of H) per CTA
constexpr int kRouteCols = 32;        // router experts per CTA (one per lane)
constexpr int kRouteThreads = 256;
constexpr int kGroupThreads = 256;
constexpr int kPassTokens = 8;        // MMA N: tokens per gate/up pass
constexpr int kWidePassTokens = 32;   // tiled kernels (large T): four MMA column groups per decoded tile
constexpr int kWidePassEntries = 16;  //   down: 16 entries x (hi, lo)
constexpr int kPassEntries = 4;       // entries per down pass (hi and lo f16 terms fill N = 8)
constexpr int kFfnWarps = 12;         // warps per expert-FFN CTA (one CTA per SM)
constexpr int kFfnBatch = 8;          // steps per batch of loads (two batches in flight)
constexpr int kTargetWarps = 152 * kFfnWarps;
constexpr int kMaxKChunks = 16;       // K-chunks per row block (partial sums per output)
constexpr size_t kAlignedPartialBudget = 64u << 20;   // partial-sum bytes allowed for one-batch K-chunks
constexpr int kWindowBudget = 200 * 1024;   // shared memory for an FFN CTA's activation window
enum FfnMode { kFfnGateUp = 0, kFfnDown = 1 };
constexpr int kMaxExperts = 1025;     // E + S (E <= 1024)
constexpr int kMaxSlots = 32;         // k + S
constexpr int kMaxTokens = 4096;
constexpr int kFusedWarps = 12;       // warps per CTA of the single-launch layer kernel
constexpr int kFusedMaxTokens = 8;    // token counts the single-launch kernel takes
constexpr int kFusedGridTarget = 152; // CTAs the router tiling is cut for (one per SM)
constexpr size_t kFusedSmemBudget = 200 * 1024;

// header words of the workspace
enum HeaderWord : int {
    kHdrStatus = 0,
    kHdrReserved = 1,
    kHdrRouteTicket = 2,
    kHdrNumActive = 3,
    kHdrNumPasses = 4,
    kHdrNumPasses4 = 5,
    kHdrNumPassesW = 6,   // wide passes (<= kWidePassTokens) of the tiled gate/up kernel
    kHdrNumPassesW4 = 7,  // wide passes (<= kWidePassEntries) of the tiled down kernel
    kHdrBarrier = 32,     // grid-wait arrivals of the fused layer kernel (own 128-byte line)
    kHdrAbort = 33,       // set when a fused-kernel wait gave up
    kHdrDone = 34,        // CTAs of the fused layer kernel that have finished
    kHdrStamps = 64,      // 16 x u64 phase timestamps of the fused kernel (words 64..95)
    kHdrRouterTickets = 96,   // fused kernel: router tiles done per group of 32 experts (words 96..127)
    kHdrWords = 128
};

// The header words are followed by per-CTA phase-end times of the fused
// kernel (diagnostics, 4 x u64 per CTA).
constexpr size_t kCtaStampOffset = kHdrWords * sizeof(uint32_t);
constexpr int kFusedMaxCtaStamps = 256;
constexpr size_t kHeaderBytes = kCtaStampOffset + kFusedMaxCtaStamps * 4 * sizeof(unsigned long long);

// Most K pieces the tensor-memory FFN kernels split their last items into.
constexpr int kTcMaxPieces = 256;

// A pass: up to kPassTokens consecutive entries of one expert's group.
struct Pass {
    int32_t expert;
    int32_t begin;   // first entry (sorted position)
    int32_t count;   // 1..kPassTokens
    int32_t pad;
};

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Upper bound on the passes of capacity `cap` over T*kps entries.
inline int max_passes(int T, int kps, int n_tot, int cap = kPassTokens) {
    long entries = (long)T * kps;
    long na = entries < n_tot ? entries : n_tot;
    return (int)((entries + cap - 1) / cap + na + 1);
}

// Split of a row block's K/64 steps into K-chunks, a function of the shapes
// only so that every call agrees on it.  When K is a multiple of 512 and the
// partial sums stay small, K-chunks of exactly kFfnBatch steps: then a unit
// is one batch of loads and the streaming loop needs no per-step bookkeeping.
// Otherwise the smallest divisor of `steps` that gives a full grid
// (kTargetWarps warps) about eight units per warp.
inline int pick_kchunks(int steps, long long units_no_split, size_t partial_bytes_per_chunk) {
    if (steps % kFfnBatch == 0 && steps / kFfnBatch <= kMaxKChunks &&
        partial_bytes_per_chunk * (steps / kFfnBatch) <= kAlignedPartialBudget)
        return steps / kFfnBatch;
    const long long target = 8LL * kTargetWarps;
    int best = 1;
    for (int d = 1; d <= steps && d <= kMaxKChunks; ++d) {
        if (steps % d)
            continue;
        best = d;
        if (units_no_split * d >= target)
            break;
    }
    return best;
}

// Copies of the router partials the single-launch kernel writes when every
// CTA sums them (CTAs read copy blockIdx % kRouterCopies).
constexpr int kRouterCopies = 4;

// Router tiles of the single-launch kernel: groups of 32 experts x chunks of
// `rows` router rows (a multiple of 8), about one tile per CTA; a tile's weight
// lines (rows x 128 B, pulled into L1 ahead of use) stay within 96 KB.
inline void fused_router_tiling(int H, int E, int *groups, int *chunks, int *rows) {
    *groups = (E + 31) / 32;
    int target = kFusedGridTarget / *groups;
    const int max_rows = 768;
    const int min_target = (H + max_rows - 1) / max_rows;
    if (target < min_target)
        target = min_target;
    if (target < 1)
        target = 1;
    int r = (H + target - 1) / target;
    r = (r + 7) / 8 * 8;
    *rows = r;
    *chunks = (H + r - 1) / r;
}

// Offsets (bytes) of the workspace regions for one problem size.
struct WsLayout {
    size_t route_part, topk_ids, topk_w, offsets, sorted_tok, sorted_slot, inv_pos, active, passes, passes4, passesw,
        passesw4, x16, xundo, xs16, tc_tail, tc_tickets,
        gpart, h16, hundo, ypart, counters, xstage, ystage, fz_rpart, fz_h32, fz_yent, mx_xq, mx_xs, mx_gu, mx_h32,
        mx_hq, mx_hs, mx_y, total;
    int n_kc_gu, n_kc_dn;
    int mx_kc_gu;          // MXFP8 variant: K chunks of the gate/up GEMM

    static WsLayout make(int T, int H, int I, int E, int k, int S) {
        WsLayout L{};
        const int kps = k + S, n_tot = E + S;
        const size_t entries = (size_t)T * kps;
        const int nh = (H + kRouteRows - 1) / kRouteRows;
        // largest possible number of (expert, <= 8 tokens) passes, without splits
        const long long active = entries < (size_t)n_tot ? (long long)entries : n_tot;
        L.n_kc_gu = pick_kchunks(H / 64, active * (I / 8), entries * 2 * (size_t)I * sizeof(float));
        L.n_kc_dn = pick_kchunks(I / 64, active * (H / 16), entries * (size_t)H * sizeof(float));
        size_t o = kHeaderBytes;
        auto take = [&](size_t bytes) { o = align_up(o, 256); size_t r = o; o += bytes; return r; };
        L.route_part = take((size_t)nh * T * E * 2 * sizeof(float));
        L.topk_ids = take(entries * sizeof(int32_t));
        L.topk_w = take(entries * sizeof(float));
        L.offsets = take((size_t)(n_tot + 1) * sizeof(int32_t));
        L.sorted_tok = take(entries * sizeof(int32_t));
        L.sorted_slot = take(entries * sizeof(int32_t));
        L.inv_pos = take(entries * sizeof(int32_t));
        L.active = take((size_t)n_tot * sizeof(int32_t));
        L.passes = take((size_t)max_passes(T, kps, n_tot) * sizeof(Pass));
        L.passes4 = take((size_t)max_passes(T, kps, n_tot, kPassEntries) * sizeof(Pass));
        L.passesw = take((size_t)max_passes(T, kps, n_tot, kWidePassTokens) * sizeof(Pass));
        L.passesw4 = take((size_t)max_passes(T, kps, n_tot, kWidePassEntries) * sizeof(Pass));
        L.x16 = take((size_t)T * H * 2);
        L.xundo = take((size_t)T * sizeof(float));
        L.xs16 = T > kFusedMaxTokens ? take(entries * H * 2) : 0;   // x per sorted entry (tensor-memory kernels)
        // tensor-memory kernels: K pieces of the last items (128 rows x 32
        // columns of partial sums each) and their arrival counters
        L.tc_tail = T > kFusedMaxTokens ? take((size_t)kTcMaxPieces * 128 * 32 * sizeof(float)) : 0;
        L.tc_tickets = T > kFusedMaxTokens ? take(2 * (size_t)kTcMaxPieces * sizeof(uint32_t)) : 0;
        L.gpart = take((size_t)L.n_kc_gu * entries * 2 * I * sizeof(float));
        L.h16 = take(entries * 2 * (size_t)I * 2);
        L.hundo = take(entries * sizeof(float));
        L.ypart = take((size_t)L.n_kc_dn * entries * H * sizeof(float));
        L.counters = take(256);
        L.xstage = take((size_t)T * H * sizeof(uint16_t));
        L.ystage = take((size_t)T * H * sizeof(uint16_t));
        if (T <= kFusedMaxTokens) {          // single-launch kernel
            int g, ch, r;
            fused_router_tiling(H, E, &g, &ch, &r);
            L.fz_rpart = take((size_t)kRouterCopies * ch * T * E * sizeof(float2));
            L.fz_h32 = take(entries * (size_t)I * sizeof(float));
            L.fz_yent = take(entries * (size_t)H * sizeof(float));
        }
        // MXFP8 variant: quantised x and h, the gate/up GEMM's K-chunk sums,
        // fp32 h and per-entry outputs.  The gate/up GEMM splits K into 1, 2
        // or 4 chunks (a function of the shapes only): the count whose CTAs
        // (128-row tiles = active experts x I/64, times the chunks) fill the
        // 3 x 152 CTA slots of its waves best; ties go to fewer chunks.
        L.mx_kc_gu = 1;
        if (H % 128 == 0 && I % 64 == 0) {
            const long long tiles = active * (I / 64), slots = 3LL * kFusedGridTarget;
            double best = 0.0;
            for (int kc = 1; kc <= 4; kc *= 2) {
                if ((H / 128) % kc)
                    break;
                const long long ctas = tiles * kc;
                const double fill = (double)ctas / (double)(((ctas + slots - 1) / slots) * slots);
                if (fill > best + 1e-9) {
                    best = fill;
                    L.mx_kc_gu = kc;
                }
            }
        }
        L.mx_xq = take((size_t)T * H);
        L.mx_xs = take((size_t)T * (H / 32));
        L.mx_gu = take((size_t)L.mx_kc_gu * entries * 2 * (size_t)I * sizeof(float));
        L.mx_h32 = take(entries * (size_t)I * sizeof(float));
        L.mx_hq = take(entries * (size_t)I);
        L.mx_hs = take(entries * (size_t)(I / 32));
        L.mx_y = take(entries * (size_t)H * sizeof(float));
        L.total = align_up(o, 256);
        return L;
    }
};

template <typename P>
inline P *ws_at(void *ws, size_t off) { return reinterpret_cast<P *>(static_cast<char *>(ws) + off); }

// --------------------------------------------------------- device helpers

__device__ __forceinline__ void record_status(uint32_t *hdr, uint32_t code) {
    atomicCAS(hdr + kHdrStatus, 0u, code);
}

// Debug build (-DMOE_DEBUG_BOUNDS, libmoe_fp4_debug.so): range checks on the
// accesses whose indices are computed from routing data -- sorted positions,
// window rows, output rows.  A failed check records MOE_ERR_DEVICE_ASSERT in
// the status word and the access is skipped, so no kernel reads or writes
// outside its buffers and none traps.  In the normal build the checks are
// the constant true.
#ifdef MOE_DEBUG_BOUNDS
__device__ __forceinline__ bool dbg_in_range(long long i, long long n, const uint32_t *hdr) {
    if (i >= 0 && i < n)
        return true;
    record_status(const_cast<uint32_t *>(hdr), MOE_ERR_DEVICE_ASSERT);
    return false;
}
#define MOE_DBG_IN_RANGE(i, n, hdr) (::moe::dbg_in_range((long long)(i), (long long)(n), (hdr)))
#else
#define MOE_DBG_IN_RANGE(i, n, hdr) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make initialised barriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// L2 policy for data read exactly once (streamed expert weights).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait until the preceding grid on the stream
// has completed and its writes are visible (a no-op without a prerequisite
// grid), and allow the next grid to be scheduled.
// Order key of a logit held as an unevaluated pair (hi, lo) with |lo| at most
// half an ulp of hi: the two floats mapped to unsigned integers that sort as
// the floats do, hi in the high word, so that keys compare as the pairs'
// values.  logit_from_key inverts the mapping of one word.
__device__ __forceinline__ unsigned long long logit_order_key(float hi, float lo) {
    auto mono = [](float v) -> uint32_t {
        const uint32_t b = __float_as_uint(v);
        return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    };
    return ((unsigned long long)mono(hi) << 32) | mono(lo);
}

__device__ __forceinline__ float logit_from_key(uint32_t m) {
    return __uint_as_float((m & 0x80000000u) ? (m & 0x7FFFFFFFu) : ~m);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + C, fp32 accumulate.  Not
// volatile: independent MMAs may be interleaved by the compiler.
__device__ __forceinline__ void mma_m16n8k16_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                                 uint32_t a3, uint32_t b0, uint32_t b1,
                                                 const float (&c)[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// Four bytes of packed E2M1 pairs -> four f16x2 (element of the low nibble in
// the low half), using the sm_100-family conversion instruction.
__device__ __forceinline__ void decode_e2m1x8(uint32_t w, uint32_t (&out)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
        : "r"(w));
}

// E8M0 exponent byte -> 2^(s-127) as fp32 (s = 0 gives the subnormal 2^-127,
// s = 255 gives NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
    uint32_t bits = s == 0 ? 0x00400000u : (s == 255 ? 0x7FFFFFFFu : (s << 23));
    return __uint_as_float(bits);
}

// 2^e as fp32 for |e| <= 126.
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

// MXFP8 (OCP MX v1.0) of one block of 32 values, one per lane: the shared
// exponent is floor(log2(max |v|)) - 8 (E4M3's largest exponent), kept in
// [-127, 127], -127 for an all-zero block; each element is v / 2^e rounded
// to E4M3, ties to even, saturating at 448.  v / 2^e is exact in fp32, so the
// codes are those of the exact quotient.  Lane 0 writes the scale byte.
__device__ __forceinline__ void mxfp8_quant_block(float v, uint8_t *code, uint8_t *scale) {
    const uint32_t amax = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v)));
    const int ef = (int)(amax >> 23);           // biased exponent of max |v| (0: zero or subnormal)
    int se = ef == 0 ? -127 : ef - 127 - 8;
    se = max(-127, min(127, se));
    const float q = v * exp2i(-se);             // -se <= 127: a normal power of two
    uint16_t pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.0f), "f"(q));
    *code = (uint8_t)(pair & 0xFF);
    if ((threadIdx.x & 31) == 0)
        *scale = (uint8_t)(se + 127);
}


// Exponent shift that maps a maximum magnitude m into [2^14, 2^15), clamped
// so that 2^shift stays a normal fp32.
__device__ __forceinline__ int f16_shift_for_max(float m) {
    if (!(m > 0.0f) || !isfinite(m))
        return 0;
    int e;
    frexpf(m, &e);          // m = f * 2^e, 0.5 <= f < 1
    int s = 15 - e;
    return s < -126 ? -126 : (s > 126 ? 126 : s);
}

// ------------------------------------------------- error-free arithmetic

// p + e = a * b exactly (one FMA).
__device__ __forceinline__ void two_prod(float a, float b, float &p, float &e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

// s + e = a + b exactly (Knuth's branch-free TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    float z = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// (p, s) += (p2, s2) for unevaluated sums p + s.
__device__ __forceinline__ void pair_add(float &p, float &s, float p2, float s2) {
    float q;
    two_sum(p, p2, p, q);
    s = __fadd_rn(s, __fadd_rn(s2, q));
}

// ------------------------------------------------------ weight streaming

constexpr int kStepBytes = 544;          // one 16 x 64 tile of the repacked bank: 512 B codes + 32 B exponents

// 16-byte asynchronous copy global -> shared (L2 only), and its group fences.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint4 ld_stream16(const void *p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ uint32_t ld_stream4(const void *p, uint64_t policy) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(p), "l"(policy));
    return v;
}

// A word of four E8M0 exponents [s0 s1 s2 s3] (s0 in the low byte) ->
// 2^(s-127) of each in fp32, via the sm_100-family conversion of exponent
// pairs to bf16 (exact for 0..254; 0 gives the subnormal 2^-127) and the
// exact widening of bf16 to fp32.
__device__ __forceinline__ void e8m0x4_to_f32(uint32_t s, float &f0, float &f1, float &f2, float &f3) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.rn.bf16x2.ue8m0x2 %0, a;\n\t"
        "cvt.rn.bf16x2.ue8m0x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(s));
    f0 = __uint_as_float(lo << 16);
    f1 = __uint_as_float(lo & 0xFFFF0000u);
    f2 = __uint_as_float(hi << 16);
    f3 = __uint_as_float(hi & 0xFFFF0000u);
}

// Byte k of a word of E8M0 exponents -> 2^(s-127) in fp32 (s = 0: 2^-127).
__device__ __forceinline__ float e8m0_byte(uint32_t w, int k) {
    const uint32_t top = __byte_perm(w, 0u, 0x0444u | ((uint32_t)k << 12));   // s << 24
    return __uint_as_float(max(top >> 1, 0x00400000u));
}

}  // namespace moe

namespace moe {

// x[t] (bf16, length H, H % 8 == 0) -> x16[t] = f16(x * 2^s), where s maps
// the row's largest magnitude into [2^14, 2^15), and xundo[t] = 2^-s.  Run by
// the warps first_warp .. first_warp+nwarps-1 of the CTA, which synchronise
// on named barrier bar_id (nwarps == all warps may use barrier 0).
__device__ inline void convert_x_row(const uint16_t *__restrict__ x, int t, int H, __half *x16, float *xundo,
                                     int first_warp, int nwarps, int bar_id) {
    __shared__ float red[32];
    const int lt = threadIdx.x - first_warp * 32, nt = nwarps * 32;
    const uint16_t *xr = x + (size_t)t * H;
    const int nchunk = H / 8;
    uint4 keep[4];                        // rows of up to 32 * nt elements stay in registers
    float m = 0.0f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = lt + q * nt;
        keep[q] = i < nchunk ? __ldg(reinterpret_cast<const uint4 *>(xr) + i) : make_uint4(0, 0, 0, 0);
    }
    for (int i = lt + 4 * nt; i < nchunk; i += nt) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {keep[q].x, keep[q].y, keep[q].z, keep[q].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[j] << 16)), fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    if ((lt & 31) == 0)
        red[lt >> 5] = m;
    named_barrier_sync(bar_id, nt);
    m = red[0];
    for (int w = 1; w < nwarps; ++w)
        m = fmaxf(m, red[w]);
    const int sh = f16_shift_for_max(m);
    const float sc = exp2i(sh);
    auto convert = [&](uint4 v, int i) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 h2 = __floats2half2_rn(__uint_as_float(w[j] << 16) * sc, __uint_as_float(w[j] & 0xFFFF0000u) * sc);
            o[j] = *reinterpret_cast<uint32_t *>(&h2);
        }
        reinterpret_cast<uint4 *>(x16 + (size_t)t * H)[i] = make_uint4(o[0], o[1], o[2], o[3]);
    };
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int i = lt + q * nt;
        if (i < nchunk)
            convert(keep[q], i);
    }
    for (int i = lt + 4 * nt; i < nchunk; i += nt)
        convert(__ldg(reinterpret_cast<const uint4 *>(xr) + i), i);
    if (lt == 0)
        xundo[t] = exp2i(-sh);
    named_barrier_sync(bar_id, nt);
}

}  // namespace moe
