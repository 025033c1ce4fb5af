// ffn.cu -- expert FFN kernels of the MXFP4 MoE layer (sm_103a).
//
// Decode of a few tokens is bound by streaming each active expert's packed
// weights from HBM once (GLM-5.2 on B300, d9249.github.io, "What it solves":
// the first batch-1 GEMMs reached 26% of peak because too few CTAs issued too
// few requests).  The kernels here are built around that stream:
//
//  * The bank is repacked once (pack.cu) so that a warp-wide 16-byte load per
//    lane returns exactly the mma.sync A-fragments of a 16-row x 64-element
//    tile; no shared memory staging and no inter-warp synchronisation is
//    needed.  Each warp keeps D such loads in flight (L1 no-allocate, L2
//    evict-first), enough for the SM to pull its share of HBM bandwidth.
//  * Work is cut into units of 16 rows x one K-chunk of one pass (<= 8
//    tokens of one expert) and spread as contiguous ranges over all warps of
//    the grid; K-chunks keep every warp busy even at T = 1.  Each unit writes
//    fp32 partial sums; small kernels sum the partials in a fixed order
//    (deterministic, no atomics).
//  * E2M1 codes are decoded in registers (cvt.rn.f16x2.e2m1x2) into f16 A
//    operands; tokens are the N = 8 columns of mma.sync m16n8k16 with fp32
//    accumulation.  Each 32-element block is accumulated on its own and then
//    scaled by its E8M0 exponent in fp32, so block scales are exact and never
//    enter the f16 operands.
//  * Activations enter as f16: x is scaled per token by a power of two that
//    maps its largest magnitude into [2^14, 2^15) (exact for every bf16 value
//    within 2^28 of the maximum), h is split into hi + lo f16 terms after the
//    same kind of scaling; scales are undone in fp32.
//
// From T = 9 on (and H, I multiples of 512) the gate/up and down projections
// run instead on the tensor-memory kernels of tc.cu; the kernels here cover
// the single-launch kernel's shapes that do not fit it and the other shapes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCacheInts = 20;           // per cached pass: expert, begin, count, pad, boff[8], boff_lo[8]

struct FfnArgs {
    const uint8_t *packed;       // section of the repacked bank
    size_t unit_bytes;           // steps * 544
    int units_per_expert;        // row blocks per expert
    int steps;                   // K / 64
    int n_kc;                    // K-chunks per row block (divides steps)
    const __half *b16;           // gate/up: x16 [T][H]; down: h16 [entries][2][I]
    int b_row;                   // B row length (H or I)
    const Pass *passes;          // gate/up: passes of <= 8 tokens; down: of <= 4 entries
    int passes_word;             // header word holding the number of passes
    const int32_t *sorted_tok;
    const uint32_t *hdr;
    float *part;                 // gate/up: [n_kc][entries][2][I]; down: [n_kc][entries][H]
    int n_entries;
    int out_len;                 // I (gate/up) or H (down)
    const float *bundo;          // down: per-entry factor that undoes the h scaling
    int T;                       // tokens (gate/up window rows)
    int win_offset;              // byte offset of the activation window in shared memory
    int win_row;                 // window row stride in elements (B row length + 32)
};

// Position of one warp in its list of units, one 64-element step at a time.
struct Cursor {
    int it;                      // step within the unit's K-chunk
    int P, rb, kc;
    const int *pc;               // cached pass record
    const uint8_t *ptr;          // address of the current step
    int bk;                      // element offset of this lane's B fragment for the step
};

struct Walker {
    const FfnArgs &a;
    const int *cache;
    int P0, m, upp;

    __device__ Walker(const FfnArgs &args, const int *c, int p0, int m_, int upp_)
        : a(args), cache(c), P0(p0), m(m_), upp(upp_) {}

    __device__ void seek(Cursor &cu, long long u) const {
        cu.it = 0;
        cu.P = (int)(u / upp);
        const int r = (int)(u % upp);
        cu.rb = r / a.n_kc;
        cu.kc = r % a.n_kc;
        locate(cu);
    }
    __device__ void locate(Cursor &cu) const {
        cu.pc = cache + (cu.P - P0) * kCacheInts;
        const int expert = cu.pc[0];
        cu.ptr = a.packed + ((size_t)expert * a.units_per_expert + cu.rb) * a.unit_bytes +
                 (size_t)(cu.kc * m) * kStepBytes;
        const int lane = threadIdx.x & 31;
        cu.bk = cu.pc[4 + (lane >> 2)] + cu.kc * m * 64 + 8 * (lane & 3);
    }
    // One step forward; true when a unit was completed (the cursor then
    // points at the next unit, which may lie past the warp's range).
    __device__ bool advance(Cursor &cu) const {
        cu.ptr += kStepBytes;
        cu.bk += 64;
        if (++cu.it < m)
            return false;
        cu.it = 0;
        if (++cu.kc == a.n_kc) {
            cu.kc = 0;
            if (++cu.rb == a.units_per_expert) {
                cu.rb = 0;
                ++cu.P;
            }
        }
        return true;
    }
};

// A unit is finished: write the partial sums of its real columns.  Kept out
// of line so that the unrolled streaming loop stays small in the I-cache.
template <int MODE>
__device__ __noinline__ void write_partials(const FfnArgs *a, float a0, float a1, float a2, float a3, int begin,
                                            int count, int rb, int kc, int lane) {
    const int g = lane >> 2, c = lane & 3;
    const float acc[4] = {a0, a1, a2, a3};
    if (MODE == kFfnGateUp) {
        const int j0 = rb * 8 + g;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = 2 * c + h;
            if (n < count && MOE_DBG_IN_RANGE(begin + n, a->n_entries, a->hdr) &&
                MOE_DBG_IN_RANGE(j0, a->out_len, a->hdr)) {
                float *dst = a->part + ((size_t)kc * a->n_entries + begin + n) * 2 * a->out_len + j0;
                dst[0] = acc[h];                 // gate row j0
                dst[a->out_len] = acc[2 + h];    // up row j0
            }
        }
    } else {
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)              // add the lo column n+4 to the hi column n
            y[i] = acc[i] + __shfl_xor_sync(0xffffffffu, acc[i], 2);
        if (c < 2) {                             // threads c < 2 own columns 0..3
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = 2 * c + h;
                if (n < count && MOE_DBG_IN_RANGE(begin + n, a->n_entries, a->hdr) &&
                    MOE_DBG_IN_RANGE(rb * 16 + g + 8, a->out_len, a->hdr)) {
                    const int e = begin + n;
                    const float u = a->bundo[e];
                    float *dst = a->part + ((size_t)kc * a->n_entries + e) * a->out_len + rb * 16;
                    dst[g] = y[h] * u;
                    dst[g + 8] = y[2 + h] * u;
                }
            }
        }
    }
}

// WIN: the B operand (x16 rows for gate/up, h16 hi/lo rows for down) of the
// CTA's passes is first copied to a shared-memory window; otherwise it is read
// from global memory.
template <int MODE, int NW, int S, bool WIN, bool ALIGNED>
__global__ void __launch_bounds__(NW * 32, 1) ffn_kernel(const __grid_constant__ FfnArgs a) {
    extern __shared__ __align__(16) int cache[];
    __half *win = reinterpret_cast<__half *>(reinterpret_cast<uint8_t *>(cache) + a.win_offset);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    pdl_wait();
    pdl_trigger();
    const int n_passes = *reinterpret_cast<const volatile int *>(a.hdr + a.passes_word);
    const int m = a.steps / a.n_kc;
    const int upp = a.units_per_expert * a.n_kc;
    const long long n_units = (long long)n_passes * upp;
    const long long W = (long long)gridDim.x * NW;
    const long long gw0 = (long long)blockIdx.x * NW;
    const long long U0 = gw0 * n_units / W, U1 = (gw0 + NW) * n_units / W;
    if (U1 <= U0)
        return;
    const int P0 = (int)(U0 / upp), P1 = (int)((U1 - 1) / upp);

    // Cache the passes this CTA touches: expert, begin, count and the B-row
    // element offsets of the 8 MMA columns.  A cursor is only located on a
    // unit inside its warp's range, so it never reads past these records.
    const int n_cached = P1 - P0 + 1;
    // first entry of the CTA's passes: the window of the down kernel starts
    // there (B offsets are window-relative with WIN, absolute without)
    const int e_lo = MODE == kFfnDown ? a.passes[P0].begin : 0;
    const int e_base = WIN ? e_lo : 0;
    const int brow = WIN ? a.win_row : a.b_row;        // element stride of B rows
    for (int i = threadIdx.x; i < n_cached * 8; i += blockDim.x) {
        const int pi = i >> 3, n = i & 7;
        const Pass ps = a.passes[P0 + pi];
        int *rec = cache + pi * kCacheInts;
        if (n == 0) {
            rec[0] = ps.expert;
            rec[1] = ps.begin;
            rec[2] = ps.count;
            rec[3] = 0;
        }
        if (MODE == kFfnGateUp) {
            const int col = n < ps.count ? n : 0;
            rec[4 + n] = a.sorted_tok[ps.begin + col] * brow;
            rec[12 + n] = 0;
        } else {                         // columns 0..3: hi of entries, 4..7: lo of the same entries
            const int e = ps.begin + ((n & 3) < ps.count ? (n & 3) : 0) - e_base;
            rec[4 + n] = (e * 2 + (n >> 2)) * brow;
            rec[12 + n] = 0;
        }
    }
    __syncthreads();

    const long long gw = gw0 + warp;
    const long long ub = gw * n_units / W, ue = (gw + 1) * n_units / W;
    const long long F = (ue - ub) * m;

    Walker wk(a, cache, P0, m, upp);
    const uint64_t policy = l2_evict_first_policy();
    Cursor pf, cc;
    // Two buffers of S steps.  The loads of one batch are issued together and
    // consumed together after the next batch has been issued: the hardware
    // tracks outstanding loads with a handful of scoreboards per warp, so a
    // finer-grained ring (one step consumed per step issued) serialises.
    uint4 bq[2][S];
    uint32_t bs[2][S];
    auto issue = [&](uint4 (&q)[S], uint32_t (&sc)[S], long long f_first) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            if (f_first + j < F) {
                q[j] = ld_stream16(pf.ptr + lane * 16, policy);
                sc[j] = ld_stream4(pf.ptr + 512 + g * 4, policy);
                if (wk.advance(pf) && f_first + j + 1 < F)
                    wk.locate(pf);
            }
        }
    };
    if (F > 0) {
        wk.seek(pf, ub);
        wk.seek(cc, ub);
        issue(bq[0], bs[0], 0);          // start the weight stream before the window copy
    }
    if (WIN) {
        // copy the B rows of the CTA's passes into the window (16-byte chunks)
        const int row_len = a.b_row;                      // elements per B row in global memory
        const int chunks_per_row = row_len / 8;
        int rows;
        const __half *src;
        if (MODE == kFfnGateUp) {
            rows = a.T;
            src = a.b16;
        } else {
            const int *last = cache + (n_cached - 1) * kCacheInts;
            rows = 2 * (last[1] + last[2] - e_lo);
            src = a.b16 + (size_t)e_lo * 2 * row_len;
        }
        const int total = rows * chunks_per_row;
        for (int i0 = threadIdx.x; i0 < total; i0 += 4 * blockDim.x) {
            uint4 v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i0 + q * blockDim.x;
                if (i < total) {
                    const int r = i / chunks_per_row, k8 = i - r * chunks_per_row;
                    v[q] = __ldg(reinterpret_cast<const uint4 *>(src + (size_t)r * row_len) + k8);
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int i = i0 + q * blockDim.x;
                if (i < total) {
                    const int r = i / chunks_per_row, k8 = i - r * chunks_per_row;
                    *reinterpret_cast<uint4 *>(win + (size_t)r * a.win_row + k8 * 8) = v[q];
                }
            }
        }
        __syncthreads();
    }
    if (F == 0)
        return;
    const __half *bbase = WIN ? win : a.b16;
    auto load_b = [](const __half *p) -> uint4 {
        if (WIN)
            return *reinterpret_cast<const uint4 *>(p);
        return __ldg(reinterpret_cast<const uint4 *>(p));
    };

    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    // one 16 x 64 step: decode, two (or four) MMAs per 32-element block, block scales
    auto step_at = [&](const uint4 q, const uint32_t s, const __half *bp) {
        const uint4 b0 = load_b(bp);
        const uint4 b1 = load_b(bp + 32);
        uint32_t pa[4], qa[4];
        const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float d[4];
        // block 2q: words q.x (row g), q.y (row g+8)
        decode_e2m1x8(q.x, pa);
        decode_e2m1x8(q.y, qa);
        mma_m16n8k16_f16(d, pa[0], qa[0], pa[1], qa[1], b0.x, b0.y, zero);
        mma_m16n8k16_f16(d, pa[2], qa[2], pa[3], qa[3], b0.z, b0.w, d);
        const float sg0 = e8m0_byte(s, 0), sh0 = e8m0_byte(s, 2);
        acc[0] = fmaf(d[0], sg0, acc[0]);
        acc[1] = fmaf(d[1], sg0, acc[1]);
        acc[2] = fmaf(d[2], sh0, acc[2]);
        acc[3] = fmaf(d[3], sh0, acc[3]);
        // block 2q+1: words q.z (row g), q.w (row g+8)
        decode_e2m1x8(q.z, pa);
        decode_e2m1x8(q.w, qa);
        mma_m16n8k16_f16(d, pa[0], qa[0], pa[1], qa[1], b1.x, b1.y, zero);
        mma_m16n8k16_f16(d, pa[2], qa[2], pa[3], qa[3], b1.z, b1.w, d);
        const float sg1 = e8m0_byte(s, 1), sh1 = e8m0_byte(s, 3);
        acc[0] = fmaf(d[0], sg1, acc[0]);
        acc[1] = fmaf(d[1], sg1, acc[1]);
        acc[2] = fmaf(d[2], sh1, acc[2]);
        acc[3] = fmaf(d[3], sh1, acc[3]);
    };
    auto step = [&](const uint4 q, const uint32_t s) {
        const int *pc = cc.pc;
        step_at(q, s, bbase + cc.bk);
        return pc;
    };
    auto consume = [&](const uint4 (&q)[S], const uint32_t (&sc)[S], long long f_first) {
#pragma unroll
        for (int j = 0; j < S; ++j) {
            if (f_first + j < F) {
                const int rb = cc.rb, kc = cc.kc;
                const int *pc = step(q[j], sc[j]);
                if (wk.advance(cc)) {
                    write_partials<MODE>(&a, acc[0], acc[1], acc[2], acc[3], pc[1], pc[2], rb, kc, lane);
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
                    if (f_first + j + 1 < F)
                        wk.locate(cc);
                }
            }
        }
    };

    if (ALIGNED) {
        // every unit is exactly one batch of S steps: straight-line code, the
        // next unit's loads in flight while the current one is computed
        auto consume_unit = [&](const uint4 (&q)[S], const uint32_t (&sc)[S]) {
            const int rb = cc.rb, kc = cc.kc;
            const int *pc = cc.pc;
            const __half *bp = bbase + cc.bk;
#pragma unroll
            for (int j = 0; j < S; ++j) {
                step_at(q[j], sc[j], bp + 64 * j);
            }
            write_partials<MODE>(&a, acc[0], acc[1], acc[2], acc[3], pc[1], pc[2], rb, kc, lane);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        };
        const long long nu = ue - ub;
        for (long long u = 0; u < nu; u += 2) {
            if (u + 1 < nu)
                issue(bq[1], bs[1], (u + 1) * S);
            consume_unit(bq[0], bs[0]);
            for (int j = 0; j < S; ++j)
                wk.advance(cc);
            if (u + 1 >= nu)
                break;
            wk.locate(cc);
            if (u + 2 < nu)
                issue(bq[0], bs[0], (u + 2) * S);
            consume_unit(bq[1], bs[1]);
            for (int j = 0; j < S; ++j)
                wk.advance(cc);
            if (u + 2 < nu)
                wk.locate(cc);
        }
        return;
    }
    for (long long f0 = 0; f0 < F; f0 += 2 * S) {
        issue(bq[1], bs[1], f0 + S);             // no-op past the end
        consume(bq[0], bs[0], f0);
        if (f0 + S >= F)
            break;
        issue(bq[0], bs[0], f0 + 2 * S);
        consume(bq[1], bs[1], f0 + S);
    }
}

// T from which the expert FFN runs on the tensor-memory kernels (tc.cu).
constexpr int kTiledMinTokens = 9;

// --------------------------------------------------------- finalize + combine

// h = silu(G) * U from the K-chunk partials of gate/up (fp32, summed in
// K-chunk order), then h * 2^shift = hi + lo in f16 with the shift chosen per
// entry.  Loads of four columns x all K-chunks are issued together.
__global__ void __launch_bounds__(512)
hfin_kernel(const float *__restrict__ part, int n_kc, int n_entries, int I, const int32_t *__restrict__ sorted_tok,
            const float *__restrict__ xundo, int T, __half *__restrict__ h16, float *__restrict__ hundo,
            const uint32_t *__restrict__ hdr, int tc_order) {
    extern __shared__ float hbuf[];   // [2I]: the g and u sums, then h in the first I
    __shared__ float wmax[16];
    const int r = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    // every load that does not depend on another goes out first: the
    // entry's token and its x factor, the routing status and the sums
    const int tok = sorted_tok[r];
    const bool routed = *reinterpret_cast<const volatile int *>(hdr + kHdrNumPasses) != 0;
    const float xu = (unsigned)tok < (unsigned)T ? __ldg(xundo + tok) : 0.0f;
    const float *base = part + (size_t)r * 2 * I;
    const size_t kstride = (size_t)n_entries * 2 * I;
    if (n_kc == 1) {
        constexpr int kBatch = 8;
        for (int j0 = threadIdx.x; j0 < I; j0 += kBatch * blockDim.x) {
            float gv[kBatch], uv[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int j = j0 + q * blockDim.x;
                if (j < I) {
                    gv[q] = base[j];
                    uv[q] = base[I + j];
                }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int j = j0 + q * blockDim.x;
                if (j < I) {
                    hbuf[j] = gv[q];
                    hbuf[I + j] = uv[q];
                }
            }
        }
    } else {
        for (int j0 = threadIdx.x; j0 < I; j0 += 2 * blockDim.x) {
            float gv[2][kMaxKChunks], uv[2][kMaxKChunks];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int j = j0 + q * blockDim.x;
#pragma unroll
                for (int kc = 0; kc < kMaxKChunks; ++kc) {
                    if (j < I && kc < n_kc) {
                        gv[q][kc] = base[kc * kstride + j];
                        uv[q][kc] = base[kc * kstride + I + j];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int j = j0 + q * blockDim.x;
                if (j < I) {
                    float G = 0.0f, U = 0.0f;
#pragma unroll
                    for (int kc = 0; kc < kMaxKChunks; ++kc)
                        if (kc < n_kc) {
                            G += gv[q][kc];
                            U += uv[q][kc];
                        }
                    hbuf[j] = G;
                    hbuf[I + j] = U;
                }
            }
        }
    }
    if (!routed)
        return;                       // grouping rejected the routing
    // h from this thread's own sums (the same j as above: no barrier)
    float mx = 0.0f;
    for (int j = threadIdx.x; j < I; j += blockDim.x) {
        const float G = hbuf[j] * xu, U = hbuf[I + j] * xu;
        const float h = G / (1.0f + expf(-G)) * U;
        hbuf[j] = h;
        mx = fmaxf(mx, fabsf(h));
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, d));
    if ((threadIdx.x & 31) == 0)
        wmax[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = wmax[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
        mx = fmaxf(mx, wmax[w]);
    const int sh = f16_shift_for_max(mx);
    const float sc = exp2i(sh);
    __half *hi = h16 + (size_t)r * 2 * I, *lo = hi + I;
    for (int j = threadIdx.x; j < I; j += blockDim.x) {
        const float v = hbuf[j] * sc;
        const __half a = __float2half_rn(v);
        // tensor-memory K order: element k of a 64-element step at position
        // (k & 0x23) | (bit 2 of k at bit 4) | (bits 3-4 of k at bits 2-3)
        const int k = j & 63;
        const int pos = tc_order ? (j & ~63) | (k & 0x23) | (((k >> 2) & 1) << 4) | (((k >> 3) & 3) << 2) : j;
        hi[pos] = a;
        lo[pos] = __float2half_rn(v - __half2float(a));
    }
    if (threadIdx.x == 0)
        hundo[r] = exp2i(-sh);
}

// y[t] = bf16_rn( sum over slots s in order of w[t,s] * sum over K-chunks of Y ).
// A CTA covers 256 outputs of one token; the positions and weights of the
// token's slots are read once per CTA, then all partial loads of a thread are
// issued before they are summed.
__global__ void __launch_bounds__(256)
combine_kernel(const float *__restrict__ part, int n_kc, int n_entries, const int32_t *__restrict__ inv_pos,
               const float *__restrict__ topk_w, int T, int kps, int H, uint16_t *__restrict__ y,
               const uint32_t *__restrict__ hdr) {
    __shared__ int spos[kMaxSlots];
    __shared__ float sw[kMaxSlots];
    const int per_tok = (H + 255) / 256;
    const int t = blockIdx.x / per_tok;
    const int n = (blockIdx.x % per_tok) * 256 + threadIdx.x;
    pdl_wait();
    pdl_trigger();
    int bad = 0;
    if (threadIdx.x == 0)             // grouping rejected the routing
        bad = *reinterpret_cast<const volatile int *>(hdr + kHdrNumPasses) == 0;
    if (threadIdx.x < kps) {
        const int pos = inv_pos[t * kps + threadIdx.x];
        spos[threadIdx.x] = pos;
        sw[threadIdx.x] = topk_w[t * kps + threadIdx.x];
        bad |= pos < 0 || pos >= n_entries;
    }
    if (__syncthreads_or(bad) || n >= H)
        return;
    const size_t kstride = (size_t)n_entries * H;
    float s = 0.0f;
    if (n_kc == 1) {                  // one partial per slot: all loads in flight at once
        float v[kMaxSlots];
#pragma unroll
        for (int i = 0; i < kMaxSlots; ++i)
            if (i < kps)
                v[i] = part[(size_t)spos[i] * H + n];
#pragma unroll
        for (int i = 0; i < kMaxSlots; ++i)
            if (i < kps)
                s = fmaf(sw[i], v[i], s);
        const __nv_bfloat16 b = __float2bfloat16_rn(s);
        y[(size_t)t * H + n] = *reinterpret_cast<const uint16_t *>(&b);
        return;
    }
    for (int s0 = 0; s0 < kps; s0 += 4) {
        float v[4][kMaxKChunks];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int kc = 0; kc < kMaxKChunks; ++kc)
                if (s0 + i < kps && kc < n_kc)
                    v[i][kc] = part[(size_t)spos[s0 + i] * H + n + kc * kstride];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (s0 + i < kps) {
                float a = 0.0f;
#pragma unroll
                for (int kc = 0; kc < kMaxKChunks; ++kc)
                    if (kc < n_kc)
                        a += v[i][kc];
                s = fmaf(sw[s0 + i], a, s);
            }
        }
    }
    const __nv_bfloat16 b = __float2bfloat16_rn(s);
    y[(size_t)t * H + n] = *reinterpret_cast<const uint16_t *>(&b);
}

__global__ void __launch_bounds__(256) x16_kernel(const uint16_t *__restrict__ x, int H, __half *x16, float *xundo) {
    pdl_wait();
    pdl_trigger();
    convert_x_row(x, blockIdx.x, H, x16, xundo, 0, 8, 1);
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

bool ffn_shape_supported(int H, int I) { return H > 0 && I > 0 && H % 64 == 0 && I % 64 == 0 && I <= 16384; }

template <int MODE, bool WIN, bool ALIGNED>
static cudaError_t launch_one(const FfnArgs &a, int grid, size_t smem, cudaStream_t stream) {
    constexpr int NW = kFfnWarps, D = kFfnBatch;
    static std::atomic<int> set_bytes[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (smem > 48 * 1024 && set_bytes[dev & 63].load() < (int)smem) {
        err = cudaFuncSetAttribute(ffn_kernel<MODE, NW, D, WIN, ALIGNED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
        if (err != cudaSuccess)
            return err;
        set_bytes[dev & 63].store((int)smem);
    }
    return launch_pdl(ffn_kernel<MODE, NW, D, WIN, ALIGNED>, dim3(grid), dim3(NW * 32), smem, stream, a);
}

template <int MODE, bool WIN>
static cudaError_t launch_aligned(const FfnArgs &a, int grid, size_t smem, cudaStream_t stream) {
    if (a.steps / a.n_kc == kFfnBatch)
        return launch_one<MODE, WIN, true>(a, grid, smem, stream);
    return launch_one<MODE, WIN, false>(a, grid, smem, stream);
}

// Chooses the shared-memory window when the B rows a CTA can need fit.
template <int MODE>
static cudaError_t launch_mode(FfnArgs &a, int grid, int cache_passes, int window_rows, cudaStream_t stream) {
    const size_t cache_bytes = align_up((size_t)cache_passes * kCacheInts * sizeof(int), 16);
    a.win_offset = (int)cache_bytes;
    a.win_row = a.b_row + 32;
    const size_t win_bytes = (size_t)window_rows * a.win_row * sizeof(__half);
    if (cache_bytes + win_bytes <= (size_t)kWindowBudget)
        return launch_aligned<MODE, true>(a, grid, cache_bytes + win_bytes, stream);
    a.win_row = a.b_row;
    return launch_aligned<MODE, false>(a, grid, cache_bytes, stream);
}

cudaError_t launch_ffn(const FfnProblem &pr, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                       cudaEvent_t ev_after_gateup) {
    const moe_mxfp4_bank_t &b = *pr.bank;
    const int H = b.hidden, I = b.inter, T = pr.T, kps = pr.kps;
    const int n_tot = b.num_experts + b.has_shared;
    const int entries = T * kps;
    const PackedLayout PL = packed_layout(H, I, n_tot);
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    if (T >= kTiledMinTokens && tc_shape_supported(H, I) && L.xs16 != 0)
        return launch_ffn_tc(pr, ws, L, num_sms, stream, ev_after_gateup);
    // passes a CTA can touch: its share of all passes plus both boundary passes
    const int cache_passes = max_passes(T, kps, n_tot) / num_sms + 3;
    const int cache_passes4 = max_passes(T, kps, n_tot, kPassEntries) / num_sms + 3;
    cudaError_t err;

    FfnArgs g{};
    g.packed = b.packed + PL.gu_offset;
    g.unit_bytes = PL.gu_unit_bytes;
    g.units_per_expert = PL.gu_units_per_expert;
    g.steps = H / 64;
    g.n_kc = L.n_kc_gu;
    g.b16 = ws_at<__half>(ws, L.x16);
    g.b_row = H;
    g.passes = ws_at<Pass>(ws, L.passes);
    g.passes_word = kHdrNumPasses;
    g.sorted_tok = ws_at<int32_t>(ws, L.sorted_tok);
    g.hdr = hdr;
    g.part = ws_at<float>(ws, L.gpart);
    g.n_entries = entries;
    g.out_len = I;
    g.T = T;
    if ((err = launch_mode<kFfnGateUp>(g, num_sms, cache_passes, T, stream)) != cudaSuccess)
        return err;

    const size_t hsmem = 2 * (size_t)I * sizeof(float);
    if (hsmem > 48 * 1024 &&
        (err = cudaFuncSetAttribute(hfin_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsmem)) !=
            cudaSuccess)
        return err;
    err = launch_pdl(hfin_kernel, dim3(entries), dim3(512), hsmem, stream, (const float *)ws_at<float>(ws, L.gpart),
                     L.n_kc_gu, entries, I, (const int32_t *)ws_at<int32_t>(ws, L.sorted_tok),
                     (const float *)ws_at<float>(ws, L.xundo), T, ws_at<__half>(ws, L.h16), ws_at<float>(ws, L.hundo),
                     (const uint32_t *)hdr, 0);
    if (err != cudaSuccess)
        return err;
    if (ev_after_gateup &&
        (err = cudaEventRecord(ev_after_gateup, stream)) != cudaSuccess)
        return err;

    FfnArgs d{};
    d.packed = b.packed + PL.dn_offset;
    d.unit_bytes = PL.dn_unit_bytes;
    d.units_per_expert = PL.dn_units_per_expert;
    d.steps = I / 64;
    d.n_kc = L.n_kc_dn;
    d.b16 = ws_at<__half>(ws, L.h16);
    d.b_row = I;
    d.passes = ws_at<Pass>(ws, L.passes4);
    d.passes_word = kHdrNumPasses4;
    d.sorted_tok = g.sorted_tok;
    d.hdr = hdr;
    d.part = ws_at<float>(ws, L.ypart);
    d.n_entries = entries;
    d.out_len = H;
    d.bundo = ws_at<float>(ws, L.hundo);
    d.T = T;
    // entries a CTA's passes can hold: at most 4 per cached pass
    const int down_rows = 2 * (entries < kPassEntries * cache_passes4 ? entries : kPassEntries * cache_passes4);
    if ((err = launch_mode<kFfnDown>(d, num_sms, cache_passes4, down_rows, stream)) != cudaSuccess)
        return err;

    return launch_pdl(combine_kernel, dim3(T * ((H + 255) / 256)), dim3(256), 0, stream,
                      (const float *)ws_at<float>(ws, L.ypart), L.n_kc_dn, entries,
                      (const int32_t *)ws_at<int32_t>(ws, L.inv_pos), pr.topk_w, T, kps, H, pr.y,
                      (const uint32_t *)hdr);
}

cudaError_t launch_combine(const float *yent, int entries, const int32_t *inv_pos, const float *topk_w, int T, int kps,
                           int H, uint16_t *y, const uint32_t *hdr, cudaStream_t stream) {
    return launch_pdl(combine_kernel, dim3(T * ((H + 255) / 256)), dim3(256), 0, stream, yent, 1, entries, inv_pos,
                      topk_w, T, kps, H, y, hdr);
}

cudaError_t launch_hfin(void *ws, const WsLayout &L, int T, int entries, int I, bool tc_order, cudaStream_t stream) {
    const size_t hsmem = 2 * (size_t)I * sizeof(float);
    cudaError_t err;
    if (hsmem > 48 * 1024 &&
        (err = cudaFuncSetAttribute(hfin_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)hsmem)) !=
            cudaSuccess)
        return err;
    return launch_pdl(hfin_kernel, dim3(entries), dim3(512), hsmem, stream, (const float *)ws_at<float>(ws, L.gpart),
                      1, entries, I, (const int32_t *)ws_at<int32_t>(ws, L.sorted_tok),
                      (const float *)ws_at<float>(ws, L.xundo), T, ws_at<__half>(ws, L.h16), ws_at<float>(ws, L.hundo),
                      (const uint32_t *)ws_at<uint32_t>(ws, 0), tc_order ? 1 : 0);
}

cudaError_t launch_x16(const uint16_t *x, int T, int H, void *ws, const WsLayout &L, cudaStream_t stream) {
    return launch_pdl(x16_kernel, dim3(T), dim3(256), 0, stream, x, H, ws_at<__half>(ws, L.x16),
                      ws_at<float>(ws, L.xundo));
}

cudaError_t launch_selftest_decode(const uint8_t *codes, uint16_t *out, int n, cudaStream_t stream) {
    const int threads = 128, items = (n + 3) / 4;
    selftest_decode_kernel<<<(items + threads - 1) / threads, threads, 0, stream>>>(codes, out, n);
    return cudaGetLastError();
}

}  // namespace moe
