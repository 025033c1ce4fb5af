// ffn.cu -- expert FFN kernels of the MXFP4 MoE layer (sm_103a).
//
// Decode of a few tokens is bound by streaming each active expert's packed
// weights from HBM once (GLM-5.2 on B300, d9249.github.io, "What it solves":
// batch-1 decode time is set by how fast the active expert weights stream, and
// the first GEMMs reached 26% of peak because too few CTAs issued requests).
// The design here follows from that:
//
//  * Work is split into units of 16 weight rows of one expert (gate/up: 8 gate
//    rows + the 8 matching up rows; down: 16 output rows) for one "pass" (up
//    to 8 tokens routed to that expert).  Units of all active experts are
//    spread evenly over one persistent CTA per SM, so every SM streams at
//    T = 1 as well; no split of K across CTAs is needed for parallelism.
//  * Inside a CTA one producer warp streams each unit's rows with bulk async
//    copies (cp.async.bulk, completion on mbarriers) into a ring of shared
//    memory stages; 8 consumer warps split each stage along K.
//  * Consumers decode E2M1 codes in registers (cvt.rn.f16x2.e2m1x2) into the
//    A operand of mma.sync m16n8k16 (f16 in, fp32 accumulate); the tokens are
//    the N = 8 columns.  Each 32-element block is accumulated separately and
//    then scaled by its E8M0 exponent in fp32, so block scales never enter the
//    f16 operands and are exact.
//  * Activations enter as f16: x (bf16) is scaled per token by a power of two
//    that maps its largest magnitude into [2^14, 2^15), which represents
//    every bf16 value within 2^28 of that maximum exactly; h (fp32) is split
//    into two f16 terms, hi + lo, after the same kind of scaling, and both are
//    multiplied in (the spare MMA work is free at these sizes).  The scale is
//    undone in fp32 after accumulation.
//  * The down kernel writes per-entry partial outputs; the CTA that finishes
//    the last pass of a 16-row block (atomic counter, no spin-waits) sums the
//    entries of every token in slot order and rounds to bf16.
//  * Every mbarrier wait is bounded (2 s by %globaltimer); on timeout the
//    kernel records MOE_ERR_DEVICE_TIMEOUT, stops issuing copies, waits for
//    its copies in flight and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxStages = 16;
constexpr int kSmemLimit = 227 * 1024;

enum FfnMode { kGateUp = 0, kDown = 1 };

struct FfnParams {
    const uint8_t *codes;     // w13 or w2 of the whole bank
    const uint8_t *scales;    // s13 or s2
    int K;                    // reduction length (H for gate/up, I for down)
    int KC;                   // K per pipeline stage
    int n_kc;                 // K / KC
    int scale_block_mode;     // 1: KC == K and scales arrive as two 8-row blocks
    int rows_per_expert;      // 2I or H
    int n_rowblocks;          // I/8 or H/16
    int row_step;             // first row of row block rb is rb * row_step
    int row_gap;              // rows 8..15 of a unit start at base + 8 + row_gap
    int n_stages;
    // shared memory plan (bytes)
    int codes_stride, scales_off, stage_bytes, win_off, win_stride, red_off, bar_off, meta_off, smem_bytes;
    // activations
    int T, window_all;        // gate/up: whole batch held in the window (T <= 8)
    const uint16_t *x;        // [T, H] bf16
    const float *hin;         // [entries, I]
    // routing
    const int32_t *sorted_tok;
    const Pass *passes;
    uint32_t *hdr;
    // outputs
    float *hout;              // [entries, I]
    int I;
    float *ypart;             // [entries, H]
    uint32_t *counters;       // [H / 16]
    const int32_t *inv_pos;   // [T * kps]
    const float *topk_w;      // [T * kps]
    int kps;
    uint16_t *y;              // [T, H]
    int H;
};

// ------------------------------------------------------------ waiting

// Warp-uniform bounded wait for phase `parity` of `bar`.  Returns false when
// the CTA is aborting (another warp timed out) or this wait timed out.
__device__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint32_t *hdr,
                          bool force_timeout) {
    const int lane = threadIdx.x & 31;
    if (force_timeout) {
        if (lane == 0) {
            record_status(hdr, MOE_ERR_DEVICE_TIMEOUT);
            *abort_flag = 1;
        }
        __syncwarp();
        return false;
    }
    bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (!ok)
            ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok))
            return true;
        int stop = 0;
        if (lane == 0) {
            if (*abort_flag) {
                stop = 1;
            } else if ((it & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) {
                record_status(hdr, MOE_ERR_DEVICE_TIMEOUT);
                *abort_flag = 1;
                stop = 1;
            }
        }
        if (__shfl_sync(0xffffffffu, stop, 0))
            return false;
    }
}

// Bounded wait of one thread, used only to drain copies already issued.
__device__ void drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > kWaitLimitNs)
            return;
}

// --------------------------------------------------------- activations

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
    return m;
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// One warp: x row (bf16, H) -> f16 window row scaled by 2^shift; stores the
// factor that undoes the scaling.
__device__ void load_x_row(const uint16_t *__restrict__ xrow, int H, uint8_t *dst, float *undo) {
    const int lane = threadIdx.x & 31;
    float m = 0.0f;
    for (int i = lane * 8; i < H; i += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xrow + i));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
            m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    }
    m = warp_max(m);
    const int sh = f16_shift_for_max(m);
    const float sc = exp2i(sh);
    for (int i = lane * 8; i < H; i += 256) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xrow + i));
        uint4 o;
        o.x = pack_half2(bf16_lo(v.x) * sc, bf16_hi(v.x) * sc);
        o.y = pack_half2(bf16_lo(v.y) * sc, bf16_hi(v.y) * sc);
        o.z = pack_half2(bf16_lo(v.z) * sc, bf16_hi(v.z) * sc);
        o.w = pack_half2(bf16_lo(v.w) * sc, bf16_hi(v.w) * sc);
        *reinterpret_cast<uint4 *>(dst + (size_t)i * 2) = o;
    }
    if (lane == 0)
        *undo = exp2i(-sh);
}

// One warp: h row (fp32, I) -> f16 hi and lo window rows, h * 2^shift = hi + lo.
__device__ void load_h_row(const float *__restrict__ hrow, int I, uint8_t *dst_hi, uint8_t *dst_lo,
                           float *undo) {
    const int lane = threadIdx.x & 31;
    float m = 0.0f;
    for (int i = lane * 8; i < I; i += 256) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(hrow + i));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(hrow + i + 4));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
    }
    m = warp_max(m);
    const int sh = f16_shift_for_max(m);
    const float sc = exp2i(sh);
    for (int i = lane * 8; i < I; i += 256) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(hrow + i));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(hrow + i + 4));
        const float v[8] = {a.x * sc, a.y * sc, a.z * sc, a.w * sc, b.x * sc, b.y * sc, b.z * sc, b.w * sc};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half h0 = __float2half_rn(v[2 * j]), h1 = __float2half_rn(v[2 * j + 1]);
            const float r0 = v[2 * j] - __half2float(h0), r1 = v[2 * j + 1] - __half2float(h1);
            __half2 hh = __halves2half2(h0, h1);
            hi[j] = *reinterpret_cast<uint32_t *>(&hh);
            lo[j] = pack_half2(r0, r1);
        }
        *reinterpret_cast<uint4 *>(dst_hi + (size_t)i * 2) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst_lo + (size_t)i * 2) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (lane == 0)
        *undo = exp2i(-sh);
}

// ---------------------------------------------------------------- kernel

template <int MODE>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_kernel(const __grid_constant__ FfnParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.bar_off);
    uint64_t *empty = full + p.n_stages;
    int *meta = reinterpret_cast<int *>(smem + p.meta_off);
    volatile int *abort_flag = meta;
    volatile int *last_flag = meta + 1;
    float *win_undo = reinterpret_cast<float *>(meta + 8);   // [8]
    float *red = reinterpret_cast<float *>(smem + p.red_off);
    uint8_t *win = smem + p.win_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *hdr = p.hdr;
    const bool force_timeout = (*reinterpret_cast<volatile uint32_t *>(hdr + kHdrDebugFlags)) & kDebugForceTimeout;
    const int n_passes = *reinterpret_cast<volatile int *>(hdr + kHdrNumPasses);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        meta[0] = 0;
        meta[1] = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const long long n_units = (long long)n_passes * p.n_rowblocks;
    const long long u0 = n_units * blockIdx.x / gridDim.x;
    const long long u1 = n_units * (blockIdx.x + 1) / gridDim.x;
    const int nrb = p.n_rowblocks;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        const uint64_t policy = l2_evict_first_policy();
        const uint32_t stage_tx = 16u * (uint32_t)(p.KC / 2) + 16u * (uint32_t)(p.KC / 32);
        int stage = 0;
        uint32_t ph = 0, filled = 0, fill_parity = 0;
        bool aborted = false;
        for (long long u = u0; u < u1 && !aborted; ++u) {
            const int P = (int)(u / nrb), rb = (int)(u % nrb);
            const Pass ps = p.passes[P];
            const size_t ebase = (size_t)ps.expert * p.rows_per_expert;
            const int rbase = rb * p.row_step;
            for (int kc = 0; kc < p.n_kc; ++kc) {
                if (!warp_wait(&empty[stage], ph ^ 1u, abort_flag, hdr, false)) {
                    aborted = true;
                    break;
                }
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[stage], stage_tx);
                __syncwarp();
                uint8_t *sb = smem + (size_t)stage * p.stage_bytes;
                if (lane < 16) {
                    const int row = rbase + lane + (lane >= 8 ? p.row_gap : 0);
                    const uint8_t *src = p.codes + (ebase + row) * (size_t)(p.K / 2) + (size_t)kc * (p.KC / 2);
                    bulk_g2s(sb + lane * p.codes_stride, src, p.KC / 2, &full[stage], policy);
                } else if (!p.scale_block_mode) {
                    const int i = lane - 16;
                    const int row = rbase + i + (i >= 8 ? p.row_gap : 0);
                    const uint8_t *src =
                        p.scales + (ebase + row) * (size_t)(p.K / 32) + (size_t)kc * (p.KC / 32);
                    bulk_g2s(sb + p.scales_off + i * (p.KC / 32), src, p.KC / 32, &full[stage], policy);
                } else if (lane < 18) {
                    const int half = lane - 16;
                    const int row = rbase + half * (8 + p.row_gap);
                    const uint8_t *src = p.scales + (ebase + row) * (size_t)(p.K / 32);
                    bulk_g2s(sb + p.scales_off + half * 8 * (p.K / 32), src, 8 * (p.K / 32), &full[stage],
                             policy);
                }
                filled |= 1u << stage;
                fill_parity = (fill_parity & ~(1u << stage)) | (ph << stage);
                if (++stage == p.n_stages) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
        // Never leave the CTA with bulk copies still writing its shared memory:
        // wait (bounded) for the latest fill of every stage.  On the normal path
        // these phases have already completed.
        if (lane == 0)
            for (int s = 0; s < p.n_stages; ++s)
                if ((filled >> s) & 1u)
                    drain_wait(&full[s], (fill_parity >> s) & 1u);
        __syncwarp();
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1, ctid = threadIdx.x - 32;
    const int g = lane >> 2, c = lane & 3;
    const int nblk = p.KC / 32;
    const int sstride = p.KC / 32;
    constexpr int kBar = 1, kBarThreads = 32 * kConsumerWarps;

    // clear the activation window once (unused MMA columns read zeros)
    {
        const int win_rows = MODE == kGateUp ? 8 : 16;
        uint4 *wz = reinterpret_cast<uint4 *>(win);
        const int n16 = win_rows * p.win_stride / 16;
        for (int i = ctid; i < n16; i += kBarThreads)
            wz[i] = make_uint4(0, 0, 0, 0);
    }
    named_barrier_sync(kBar, kBarThreads);
    const bool whole_batch = MODE == kGateUp && p.window_all;
    if (whole_batch) {
        if (cw < p.T)
            load_x_row(p.x + (size_t)cw * p.H, p.H, win + cw * p.win_stride, &win_undo[cw]);
        named_barrier_sync(kBar, kBarThreads);
    }

    int stage = 0;
    uint32_t ph = 0;
    int loaded = -1, buf = 0;
    bool aborted = false;
    for (long long u = u0; u < u1; ++u) {
        const int P = (int)(u / nrb), rb = (int)(u % nrb);
        const Pass ps = p.passes[P];
        if (!whole_batch && P != loaded) {
            named_barrier_sync(kBar, kBarThreads);
            if (cw < ps.count) {
                if (MODE == kGateUp) {
                    const int t = p.sorted_tok[ps.begin + cw];
                    load_x_row(p.x + (size_t)t * p.H, p.H, win + cw * p.win_stride, &win_undo[cw]);
                } else {
                    load_h_row(p.hin + (size_t)(ps.begin + cw) * p.I, p.I, win + cw * p.win_stride,
                               win + (8 + cw) * p.win_stride, &win_undo[cw]);
                }
            }
            named_barrier_sync(kBar, kBarThreads);
            loaded = P;
        }
        int brow = g;
        if (whole_batch)
            brow = g < ps.count ? p.sorted_tok[ps.begin + g] : 0;
        const uint8_t *bptr = win + brow * p.win_stride + 16 * c;

        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int kc = 0; kc < p.n_kc; ++kc) {
            if (!aborted)
                aborted = !warp_wait(&full[stage], ph, abort_flag, hdr, force_timeout);
            if (!aborted) {
                const uint8_t *sb = smem + (size_t)stage * p.stage_bytes;
                const uint8_t *arow = sb + g * p.codes_stride + 4 * c;
                const uint8_t *srow = sb + p.scales_off + g * sstride;
                const uint8_t *bk = bptr + (size_t)kc * p.KC * 2;
#pragma unroll 2
                for (int kb = cw; kb < nblk; kb += kConsumerWarps) {
                    const uint32_t alo = *reinterpret_cast<const uint32_t *>(arow + kb * 16);
                    const uint32_t ahi = *reinterpret_cast<const uint32_t *>(arow + 8 * p.codes_stride + kb * 16);
                    const float slo = e8m0_to_f32(srow[kb]);
                    const float shi = e8m0_to_f32(srow[8 * sstride + kb]);
                    const uint4 b = *reinterpret_cast<const uint4 *>(bk + kb * 64);
                    uint32_t pa[4], qa[4];
                    decode_e2m1x8(alo, pa);
                    decode_e2m1x8(ahi, qa);
                    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    float d[4];
                    mma_m16n8k16_f16(d, pa[0], qa[0], pa[1], qa[1], b.x, b.y, zero);
                    mma_m16n8k16_f16(d, pa[2], qa[2], pa[3], qa[3], b.z, b.w, d);
                    if (MODE == kDown) {
                        const uint4 bl = *reinterpret_cast<const uint4 *>(bk + 8 * p.win_stride + kb * 64);
                        mma_m16n8k16_f16(d, pa[0], qa[0], pa[1], qa[1], bl.x, bl.y, d);
                        mma_m16n8k16_f16(d, pa[2], qa[2], pa[3], qa[3], bl.z, bl.w, d);
                    }
                    acc[0] = fmaf(d[0], slo, acc[0]);
                    acc[1] = fmaf(d[1], slo, acc[1]);
                    acc[2] = fmaf(d[2], shi, acc[2]);
                    acc[3] = fmaf(d[3], shi, acc[3]);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[stage]);
            }
            if (++stage == p.n_stages) {
                stage = 0;
                ph ^= 1u;
            }
        }

        // ------------------------------------------------ unit epilogue
        float *mine = red + buf * (kConsumerWarps * 128) + cw * 128;
        mine[g * 8 + 2 * c] = acc[0];
        mine[g * 8 + 2 * c + 1] = acc[1];
        mine[(g + 8) * 8 + 2 * c] = acc[2];
        mine[(g + 8) * 8 + 2 * c + 1] = acc[3];
        named_barrier_sync(kBar, kBarThreads);
        const float *rr = red + buf * (kConsumerWarps * 128);
        const bool ok = !*abort_flag;
        if (MODE == kGateUp) {
            if (ctid < 64 && ok) {
                const int jj = ctid >> 3, n = ctid & 7;
                if (n < ps.count) {
                    float G = 0.0f, U = 0.0f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w) {
                        G += rr[w * 128 + jj * 8 + n];
                        U += rr[w * 128 + (jj + 8) * 8 + n];
                    }
                    const float undo = whole_batch ? win_undo[p.sorted_tok[ps.begin + n]] : win_undo[n];
                    G *= undo;
                    U *= undo;
                    const float hv = G / (1.0f + expf(-G)) * U;
                    p.hout[(size_t)(ps.begin + n) * p.I + rb * 8 + jj] = hv;
                }
            }
        } else {
            if (ctid < 128 && ok) {
                const int i = ctid >> 3, n = ctid & 7;
                if (n < ps.count) {
                    float Y = 0.0f;
#pragma unroll
                    for (int w = 0; w < kConsumerWarps; ++w)
                        Y += rr[w * 128 + i * 8 + n];
                    p.ypart[(size_t)(ps.begin + n) * p.H + rb * 16 + i] = Y * win_undo[n];
                }
            }
            __threadfence();
            named_barrier_sync(kBar, kBarThreads);
            if (ctid == 0) {
                int last = 0;
                if (!*abort_flag) {
                    const unsigned old = atomicAdd(&p.counters[rb], 1u);
                    last = old == (unsigned)(n_passes - 1);
                }
                *last_flag = last;
            }
            named_barrier_sync(kBar, kBarThreads);
            if (*last_flag) {
                __threadfence();
                for (int idx = ctid; idx < p.T * 16; idx += kBarThreads) {
                    const int t = idx >> 4, i = idx & 15;
                    float s = 0.0f;
                    for (int sl = 0; sl < p.kps; ++sl) {
                        const int pos = __ldcg(p.inv_pos + t * p.kps + sl);
                        s = fmaf(__ldcg(p.topk_w + t * p.kps + sl),
                                 __ldcg(p.ypart + (size_t)pos * p.H + rb * 16 + i), s);
                    }
                    const __nv_bfloat16 b = __float2bfloat16_rn(s);
                    p.y[(size_t)t * p.H + rb * 16 + i] = *reinterpret_cast<const uint16_t *>(&b);
                }
                if (ctid == 0)
                    p.counters[rb] = 0;
            }
        }
        buf ^= 1;
    }
}

__global__ void selftest_decode_kernel(const uint8_t *codes, uint16_t *out, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * i >= n)
        return;
    uint32_t w = 0;
    for (int j = 0; j < 4 && 4 * i + j < n; ++j)
        w |= (uint32_t)codes[4 * i + j] << (8 * j);
    uint32_t o[4];
    decode_e2m1x8(w, o);
    for (int j = 0; j < 4 && 4 * i + j < n; ++j) {
        out[2 * (4 * i + j)] = (uint16_t)(o[j] & 0xFFFFu);
        out[2 * (4 * i + j) + 1] = (uint16_t)(o[j] >> 16);
    }
}

// ---------------------------------------------------------------- host side

static bool ok_K(int K) { return K > 0 && K % 64 == 0 && (K % 512 == 0 || K <= 2048); }

bool ffn_shape_supported(int H, int I) { return ok_K(H) && ok_K(I); }

static int pick_kc(int K) {
    if (K % 512 == 0) {
        const int cands[] = {2048, 1536, 1024, 512};
        for (int kc : cands)
            if (K % kc == 0)
                return kc;
    }
    return K;
}

// Fills the K / staging / shared-memory fields of p; returns false if no plan fits.
static bool plan_ffn(FfnParams &p, int K, int win_rows) {
    p.K = K;
    p.KC = pick_kc(K);
    p.n_kc = K / p.KC;
    p.scale_block_mode = K % 512 != 0;
    p.codes_stride = p.KC / 2 + 16;
    p.scales_off = 16 * p.codes_stride;
    p.stage_bytes = (int)align_up((size_t)p.scales_off + 16 * (p.KC / 32), 128);
    p.win_stride = 2 * K + 64;
    const int win_bytes = win_rows * p.win_stride;
    const int red_bytes = 2 * kConsumerWarps * 128 * (int)sizeof(float);
    const int fixed = win_bytes + red_bytes + 2 * kMaxStages * 8 + 256 + 128;
    int n = (72 * 1024 + p.stage_bytes - 1) / p.stage_bytes;
    n = n < 4 ? 4 : (n > kMaxStages ? kMaxStages : n);
    while (n > 2 && n * p.stage_bytes + fixed > kSmemLimit)
        --n;
    if (n * p.stage_bytes + fixed > kSmemLimit)
        return false;
    p.n_stages = n;
    p.win_off = n * p.stage_bytes;
    p.red_off = (int)align_up((size_t)p.win_off + win_bytes, 128);
    p.bar_off = (int)align_up((size_t)p.red_off + red_bytes, 16);
    p.meta_off = p.bar_off + 2 * n * 8;
    p.smem_bytes = (int)align_up((size_t)p.meta_off + 256, 128);
    return true;
}

static std::atomic<int> g_smem_set[2][64];

template <int MODE>
static cudaError_t ensure_smem(int bytes) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    std::atomic<int> &cur = g_smem_set[MODE][dev & 63];
    if (cur.load(std::memory_order_relaxed) >= bytes)
        return cudaSuccess;
    err = cudaFuncSetAttribute(ffn_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess) {
        int prev = cur.load();
        while (prev < bytes && !cur.compare_exchange_weak(prev, bytes)) {
        }
    }
    return err;
}

cudaError_t launch_ffn(const FfnProblem &pr, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                       cudaEvent_t ev_after_gateup) {
    const moe_mxfp4_bank_t &b = *pr.bank;
    const int H = b.hidden, I = b.inter, T = pr.T;
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);

    FfnParams g{};
    g.codes = b.w13;
    g.scales = b.s13;
    g.rows_per_expert = 2 * I;
    g.n_rowblocks = I / 8;
    g.row_step = 8;
    g.row_gap = I - 8;
    g.T = T;
    g.window_all = T <= kPassTokens;
    g.x = pr.x;
    g.sorted_tok = ws_at<int32_t>(ws, L.sorted_tok);
    g.passes = ws_at<Pass>(ws, L.passes);
    g.hdr = hdr;
    g.hout = ws_at<float>(ws, L.h);
    g.I = I;
    g.H = H;
    if (!plan_ffn(g, H, 8))
        return cudaErrorInvalidConfiguration;

    FfnParams d{};
    d.codes = b.w2;
    d.scales = b.s2;
    d.rows_per_expert = H;
    d.n_rowblocks = H / 16;
    d.row_step = 16;
    d.row_gap = 0;
    d.T = T;
    d.window_all = 0;
    d.hin = ws_at<float>(ws, L.h);
    d.sorted_tok = g.sorted_tok;
    d.passes = g.passes;
    d.hdr = hdr;
    d.I = I;
    d.H = H;
    d.ypart = ws_at<float>(ws, L.ypart);
    d.counters = ws_at<uint32_t>(ws, L.counters);
    d.inv_pos = ws_at<int32_t>(ws, L.inv_pos);
    d.topk_w = pr.topk_w;
    d.kps = pr.kps;
    d.y = pr.y;
    if (!plan_ffn(d, I, 16))
        return cudaErrorInvalidConfiguration;

    cudaError_t err = ensure_smem<kGateUp>(g.smem_bytes);
    if (err == cudaSuccess)
        err = ensure_smem<kDown>(d.smem_bytes);
    if (err != cudaSuccess)
        return err;
    ffn_kernel<kGateUp><<<num_sms, kFfnThreads, g.smem_bytes, stream>>>(g);
    if ((err = cudaGetLastError()) != cudaSuccess)
        return err;
    if (ev_after_gateup &&
        (err = cudaEventRecordWithFlags(ev_after_gateup, stream, cudaEventRecordExternal)) != cudaSuccess)
        return err;
    ffn_kernel<kDown><<<num_sms, kFfnThreads, d.smem_bytes, stream>>>(d);
    return cudaGetLastError();
}

cudaError_t launch_selftest_decode(const uint8_t *codes, uint16_t *out, int n, cudaStream_t stream) {
    const int threads = 128, items = (n + 3) / 4;
    selftest_decode_kernel<<<(items + threads - 1) / threads, threads, 0, stream>>>(codes, out, n);
    return cudaGetLastError();
}

}  // namespace moe
