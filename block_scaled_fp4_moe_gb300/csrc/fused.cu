// fused.cu -- the whole MoE layer as one persistent kernel for decode-sized
// token counts (T <= 8), sm_103a.
//
// At a few tokens the layer is a chain of small dependent steps around two
// weight streams (GLM-5.2 on B300, d9249.github.io, "What it sets out to
// solve": decode is bound by streaming the active expert weights; the pages'
// kernel sections name launch gaps and too few CTAs as what kept the first
// batch-1 GEMMs at a quarter of peak).  Here one cooperative launch of one CTA
// per SM runs the chain, with three grid-wide waits:
//
//  R  router partial dot products (Dot2, error-free) over tiles of the router
//     matrix; meanwhile the shared expert's gate/up weights, which every token
//     uses, are prefetched into L2.
//  -- grid wait 1
//  T  every CTA sums the partials, selects the top k of each token (shared
//     expert as slot k), groups the (token, slot) entries by expert and
//     converts x to f16, all in its own shared memory (the same arithmetic
//     in every CTA, so every CTA holds the same routing).
//  G  gate/up: each CTA streams a contiguous range of whole 16-row blocks of
//     the active experts; its warps split the range's 64-element steps, sum
//     their partial results in shared memory in warp order and write
//     h = silu(gate) * up in fp32.  Before the second wait each warp already
//     issues the loads of its first down batch.
//  -- grid wait 2
//  D  down: each CTA converts the h rows of its entries to f16 hi + lo terms
//     (per-entry power-of-two scale), streams whole 16-row blocks of H, and
//     writes the per-entry outputs Y.
//  -- grid wait 3
//  C  every CTA combines an equal share of the outputs:
//     y = bf16(sum over slots in order of w * Y).
//
// A second instantiation (ROUTE_ONLY) runs phases R and T alone and writes the
// grouping to the workspace: the MXFP8 variant (mx8.cu) routes with it for
// T <= 8 and runs the expert projections itself.
//
// Waits spin on a counter in the workspace with a time limit; a wait that runs
// out records MOE_ERR_DEVICE_TIMEOUT and every CTA leaves without writing y.
// The cooperative launch guarantees that all CTAs are resident, so a wait can
// only end that way through a fault elsewhere.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

struct FusedArgs {
    const uint16_t *x;           // [T, H] bf16
    const float *wr;             // [H, E] router
    const float *bias;           // [E] or null
    const uint8_t *gu, *dn;      // packed gate/up and down sections
    uint16_t *y;                 // [T, H] bf16
    int32_t *ids_out;            // [T, kps] or null
    float *w_out;                // [T, kps] or null
    uint32_t *hdr;               // workspace header
    float2 *rpart;               // [kRouterCopies][r_chunks][T][E] router partial pairs
    float *h32;                  // [entries][I] h in sorted entry order
    float *yent;                 // [entries][H] per-entry outputs
    unsigned long long *cstamps; // [grid][4] per-CTA phase-end times (diagnostics)
    int T, H, E, k, S, I;
    float shared_weight;
    int r_groups, r_chunks, r_rows;   // router tiles: 32 experts x r_rows rows
    int r_final;                 // 1: the router phase sums each group's chunks (else every CTA does)
    int r_vec;                   // 1: router rows are 16-byte aligned (E % 4 == 0): asynchronous tile copies
    unsigned gu_unit, dn_unit;        // bytes of one packed row block
    int xwin_row, hwin_row;           // window row strides (elements)
    int win_entries;                  // entries the down window holds
    int off_hundo, off_b;             // dynamic shared-memory offsets (bytes)
    const uint8_t *next_pf[3];        // next layer: router, shared gate/up, shared down (nullable)
    size_t next_pf_bytes[3];
    Pass *x_passes;                   // routing only: the gate/up passes (one per active expert, <= 8 entries)
    // the grouping every CTA derived, written by CTA 0 (the layout of the
    // multi-launch grouping): sorted position -> token and slot, entry ->
    // sorted position, per-expert offsets [n_tot + 1], active experts
    int32_t *x_sorted_tok, *x_sorted_slot, *x_inv_pos, *x_offsets, *x_active;
    uint8_t *x_q, *x_qs;              // routing only, nullable: x as MXFP8 codes [T][H] and scales [T][H/32]
};

namespace {

constexpr int NW = kFusedWarps;
constexpr int NT = NW * 32;
constexpr int SB = 8;                 // steps per batch of loads
constexpr int NBUF = 2;               // register buffers of one batch; NBUF - 1 batches stay in flight
constexpr int kBatchBytes = SB * kStepBytes;
constexpr int kMaxEntries = kFusedMaxTokens * kMaxSlots;
constexpr unsigned long long kWaitLimitNs = 200ull * 1000 * 1000;

// Routing results every CTA derives for itself in phase T.
struct RouteState {
    int n_gu, n_dn, bad, pad;
    float xundo[kFusedMaxTokens];  // 2^-s of token t's f16 scaling
    float xscale[kFusedMaxTokens]; // 2^s
    int sel_id[kMaxEntries];       // entry t*kps+s -> expert
    float sel_w[kMaxEntries];      // entry -> combine weight
    int inv_pos[kMaxEntries];      // entry -> sorted position
    int sorted_ent[kMaxEntries];   // sorted position -> entry
    int sorted_tok[kMaxEntries];   // sorted position -> token
    Pass pgu[kMaxEntries];         // gate/up passes: one per active expert (T <= 8)
    Pass pdn[kMaxEntries];         // down passes of <= 4 entries
};

// The kernel's shared memory: the dynamic region (windows, scratch) and the
// routing state, declared here so that every function addresses them as
// shared memory.
extern __shared__ __align__(16) uint8_t fz_smem[];
__shared__ RouteState fz_rs;

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void prefetch_l2_line(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void stamp(const FusedArgs &a, int i) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
        reinterpret_cast<unsigned long long *>(a.hdr + kHdrStamps)[i] = globaltimer_ns();
}

__device__ __forceinline__ void cta_stamp(const FusedArgs &a, int i) {
    if (threadIdx.x == 0 && blockIdx.x < kFusedMaxCtaStamps)
        a.cstamps[blockIdx.x * 4 + i] = globaltimer_ns();
}

// Grid-wide wait in two halves.  grid_arrive: after the CTA barrier, one
// thread issues a release fence (cumulative: it covers the writes the barrier
// ordered before it) and adds its arrival to the counter.  grid_wait: until `target` (= waits so far
// x CTAs) arrivals are counted.  Work that needs nobody else's results can
// run in between.  A wait gives up after kWaitLimitNs (or when another CTA's
// wait gave up) and returns false.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ void grid_arrive(const FusedArgs &a) {
    __syncthreads();
    if (threadIdx.x == 0) {
        fence_acq_rel_gpu();
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;" ::"l"(a.hdr + kHdrBarrier) : "memory");
    }
}

__device__ bool grid_wait(const FusedArgs &a, unsigned target) {
    __shared__ int ok;
    if (threadIdx.x == 0) {
        const unsigned long long t0 = globaltimer_ns();
        int r = 1;
        for (unsigned it = 0; ld_acquire_u32(a.hdr + kHdrBarrier) < target; ++it) {
            __nanosleep(32);              // let the arrivals through to the counter's line
            if ((it & 15) != 15)
                continue;
            if (ld_acquire_u32(a.hdr + kHdrAbort)) {
                r = 0;
                break;
            }
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_status(a.hdr, MOE_ERR_DEVICE_TIMEOUT);
                atomicExch(a.hdr + kHdrAbort, 1u);
                r = 0;
                break;
            }
        }
        ok = r;                           // the acquiring load orders what follows the barrier below
    }
    __syncthreads();
    return ok != 0;
}

// ------------------------------------------------------------- phase R

// Dot2 sums of one warp's rows of a router tile for TT token columns (x rows
// staged as xs[row][TT], zero past T): each weight is loaded once and feeds TT
// independent compensated sums.  The weights come in register batches of B
// rows, the next batch in flight while the current one is summed.
template <int TT>
__device__ __forceinline__ void router_row(const float *xs, int row, float wv, float (&p)[kFusedMaxTokens],
                                           float (&q)[kFusedMaxTokens]) {
    const float *xr = xs + (size_t)row * TT;
    float xv[TT];
    if (TT == 1) {
        xv[0] = xr[0];
    } else if (TT == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(xr);
        xv[0] = v.x;
        xv[1 % TT] = v.y;
    } else {
#pragma unroll
        for (int h = 0; h < TT / 4; ++h) {
            const float4 v = *reinterpret_cast<const float4 *>(xr + 4 * h);
            xv[(4 * h) % TT] = v.x;
            xv[(4 * h + 1) % TT] = v.y;
            xv[(4 * h + 2) % TT] = v.z;
            xv[(4 * h + 3) % TT] = v.w;
        }
    }
#pragma unroll
    for (int t = 0; t < TT; ++t) {
        float hp, er, s;
        two_prod(xv[t], wv, hp, er);
        two_sum(p[t], hp, p[t], s);
        q[t] = __fadd_rn(q[t], __fadd_rn(s, er));
    }
}

template <int TT, int B>
__device__ __forceinline__ void router_load(float (&w)[B], const float *wp, size_t wstride, int j0, int nrw,
                                            bool live) {
#pragma unroll
    for (int u = 0; u < B; ++u)
        w[u] = live && j0 + u < nrw ? wp[(size_t)(j0 + u) * wstride] : 0.0f;
}

template <int TT, int B>
__device__ __forceinline__ void router_sum(const float (&w)[B], const float *xs, int j0, int nrw,
                                           float (&p)[kFusedMaxTokens], float (&q)[kFusedMaxTokens]) {
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int u = 0; u < B; ++u)
        if (j0 + u < nrw)
            router_row<TT>(xs, (j0 + u) * NW + warp, w[u], p, q);
}

template <int TT>
__device__ __forceinline__ void router_rows(const float *xs, const float *wp, size_t wstride, int nrw, bool live,
                                            float (&p)[kFusedMaxTokens], float (&q)[kFusedMaxTokens]) {
    constexpr int B = TT <= 2 ? 8 : 4;
    float wa[B], wb[B];
    router_load<TT, B>(wa, wp, wstride, 0, nrw, live);
#pragma unroll 1
    for (int j0 = 0; j0 < nrw; j0 += 2 * B) {
        router_load<TT, B>(wb, wp, wstride, j0 + B, nrw, live);
        router_sum<TT, B>(wa, xs, j0, nrw, p, q);
        router_load<TT, B>(wa, wp, wstride, j0 + 2 * B, nrw, live);
        router_sum<TT, B>(wb, xs, j0 + B, nrw, p, q);
    }
}

// The CTA that completes the last chunk of an expert group sums the group's
// chunk partials in chunk order (the chunk range split into parts that are
// then added in part order) and leaves the logit pairs in chunk 0's slots.
// Every CTA's partial writes are released before its ticket; the last CTA
// acquires them after its own.
__device__ void router_finish_group(const FusedArgs &a, int gi, float2 *red) {
    __shared__ int last;
    const int tid = threadIdx.x, T = a.T, E = a.E, chunks = a.r_chunks;
    __syncthreads();
    if (tid == 0) {
        fence_acq_rel_gpu();                       // release this CTA's partials
        const unsigned tk = atomicAdd(a.hdr + kHdrRouterTickets + gi, 1u);
        last = tk == (unsigned)chunks - 1u;
        if (last) {
            fence_acq_rel_gpu();                   // acquire the other CTAs' partials
            a.hdr[kHdrRouterTickets + gi] = 0u;    // ready for the next launch
        }
    }
    __syncthreads();
    if (!last)
        return;
    const int e0 = gi * 32, ne = min(E, e0 + 32) - e0, items = T * 32;
    const int parts = max(1, NT / items), cpp = (chunks + parts - 1) / parts;
    const int item = tid / parts, part = tid - item * parts, t = item >> 5, el = item & 31;
    const bool live = item < items && el < ne;
    float P = 0.0f, Q = 0.0f;
    if (live) {
        const float2 *src = a.rpart + (size_t)t * E + e0 + el;
        const size_t cstride = (size_t)T * E;
        const int c_lo = part * cpp, c_hi = min(chunks, c_lo + cpp);
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
            float2 v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c0 + c < c_hi)
                    v[c] = __ldcg(src + (size_t)(c0 + c) * cstride);
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (c0 + c < c_hi)
                    pair_add(P, Q, v[c].x, v[c].y);
        }
    }
    if (item < items)
        red[tid] = make_float2(P, Q);
    __syncthreads();
    if (live && part == 0) {
        for (int q = 1; q < parts; ++q)
            pair_add(P, Q, red[tid + q].x, red[tid + q].y);
        a.rpart[(size_t)t * E + e0 + el] = make_float2(P, Q);
    }
}

// Router tile (32 experts x r_rows rows): each warp pulls its rows (every
// NW-th row) into L1 while the tile's x rows are staged, then accumulates one
// Dot2 pair per token and lane (expert); the CTA sums the warps' pairs in warp
// order.
__device__ void phase_router(const FusedArgs &a, uint8_t *sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, H = a.H, E = a.E;
    const int TT = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;      // token columns of the x rows
    float *wt = reinterpret_cast<float *>(sm);                                    // [r_rows][32] weights
    float *xs = reinterpret_cast<float *>(sm + (size_t)a.r_rows * 128);          // [r_rows][TT]
    float2 *red = reinterpret_cast<float2 *>(sm + (size_t)a.r_rows * 128 + align_up(TT * a.r_rows * 4, 16));
    const int tiles = a.r_groups * a.r_chunks;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int gi = tile % a.r_groups, ci = tile / a.r_groups;
        const int r0 = ci * a.r_rows, nr = min(H - r0, a.r_rows);
        const int e0 = gi * 32, e1 = min(E, e0 + 32);       // experts [e0, e1) of this tile
        const int nrw = nr > warp ? (nr - warp + NW - 1) / NW : 0;
        __syncthreads();                                     // the previous tile's readers are done
        // the tile's weights into shared memory, all rows at once: 16-byte
        // asynchronous copies when rows are 16-byte aligned, else words
        if (a.r_vec) {
            const int nch = (e1 - e0) >> 2;                  // 16-byte chunks per row
            for (int i = threadIdx.x; i < nr * 8; i += NT) {
                const int row = i >> 3, ch = i & 7;
                if (ch < nch)
                    cp_async16(wt + row * 32 + 4 * ch, a.wr + (size_t)(r0 + row) * E + e0 + 4 * ch);
            }
            cp_async_commit();
        } else {
            for (int i = threadIdx.x; i < nr * 32; i += NT) {
                const int row = i >> 5, col = i & 31;
                if (e0 + col < e1)
                    wt[row * 32 + col] = __ldg(a.wr + (size_t)(r0 + row) * E + e0 + col);
            }
        }
        for (int i = threadIdx.x; i < TT * (nr / 8); i += NT) {
            const int c8 = i / TT, t = i - c8 * TT;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (t < T)
                v = __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * H + r0) + c8);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            float *d = xs + (size_t)c8 * 8 * TT + t;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                d[(2 * j) * TT] = __uint_as_float(w4[j] << 16);
                d[(2 * j + 1) * TT] = __uint_as_float(w4[j] & 0xFFFF0000u);
            }
        }
        if (a.r_vec)
            cp_async_wait<0>();
        __syncthreads();
        stamp(a, 8);
        const bool live = e0 + lane < e1;
        float p[kFusedMaxTokens], q[kFusedMaxTokens];
#pragma unroll
        for (int t = 0; t < kFusedMaxTokens; ++t)
            p[t] = q[t] = 0.0f;
        const float *w0 = wt + warp * 32 + lane;             // this warp's rows: warp, warp + NW, ...
        const size_t wstride = (size_t)NW * 32;
        if (TT == 1)
            router_rows<1>(xs, w0, wstride, nrw, live, p, q);
        else if (TT == 2)
            router_rows<2>(xs, w0, wstride, nrw, live, p, q);
        else if (TT == 4)
            router_rows<4>(xs, w0, wstride, nrw, live, p, q);
        else
            router_rows<8>(xs, w0, wstride, nrw, live, p, q);
#pragma unroll
        for (int t = 0; t < kFusedMaxTokens; ++t)
            if (t < T)
                red[(warp * T + t) * 32 + lane] = make_float2(p[t], q[t]);
        __syncthreads();
        for (int t = warp; t < T; t += NW) {
            float P = red[t * 32 + lane].x, Q = red[t * 32 + lane].y;
            for (int w2 = 1; w2 < NW; ++w2) {
                const float2 v = red[(w2 * T + t) * 32 + lane];
                pair_add(P, Q, v.x, v.y);
            }
            if (live) {
                const size_t o = ((size_t)ci * T + t) * E + e0 + lane;
                if (a.r_final) {
                    a.rpart[o] = make_float2(P, Q);
                } else {
                    const size_t copy = (size_t)a.r_chunks * T * E;
#pragma unroll
                    for (int r = 0; r < kRouterCopies; ++r)
                        a.rpart[o + r * copy] = make_float2(P, Q);
                }
            }
        }
        if (a.r_final)
            router_finish_group(a, gi, red);
    }
}

// This CTA's first router tile into L2 (a hint on read-only data: may run
// before the previous kernel on the stream has finished).
__device__ void prefetch_router_tile(const FusedArgs &a) {
    const int tile = blockIdx.x;
    if (tile >= a.r_groups * a.r_chunks)
        return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = tile % a.r_groups, ci = tile / a.r_groups;
    const int r0 = ci * a.r_rows, nr = min(a.H - r0, a.r_rows);
    const int e0 = gi * 32, e1 = min(a.E, e0 + 32);
    const int nrw = nr > warp ? (nr - warp + NW - 1) / NW : 0;
    const float *wrow = a.wr + (size_t)(r0 + warp) * a.E;
    const size_t wstride = (size_t)NW * a.E;
    for (int j = lane; j < nrw; j += 32) {
        prefetch_l2_line(wrow + j * wstride + e0);
        prefetch_l2_line(wrow + j * wstride + e1 - 1);
    }
}

// The shared expert's gate/up weights do not depend on the routing: pull
// this CTA's slice of them into L2 while the router runs.
__device__ void prefetch_shared_expert(const FusedArgs &a) {
    if (!a.S || threadIdx.x != 0)
        return;
    const size_t total = (size_t)(a.I / 8) * a.gu_unit;
    const uint8_t *base = a.gu + (size_t)a.E * total;
    const size_t piece = align_up((total + gridDim.x - 1) / gridDim.x, 16);
    const size_t lo = (size_t)blockIdx.x * piece;
    const size_t hi = lo + piece < total ? lo + piece : total;
    for (size_t o = lo; o < hi; o += 16384) {
        const size_t n = hi - o < 16384 ? hi - o : 16384;
        prefetch_l2(base + o, (uint32_t)n);
    }
}

// ------------------------------------------------------------- phase T

// x -> the f16 window: x[t] scaled by 2^s[t] so that max |x[t]| lies in
// [2^14, 2^15) (rs.xundo[t] = 2^-s[t]).  Every CTA reads all of x itself, so
// this needs nobody else's results; the kernel runs it while it waits for the
// other CTAs' router partials.
__device__ void x_window_local(const FusedArgs &a, RouteState &rs, __half *xwin) {
    __shared__ unsigned xm[kFusedMaxTokens];
    const int H = a.H, n8 = H / 8, total = a.T * n8;
    if (threadIdx.x < kFusedMaxTokens)
        xm[threadIdx.x] = 0u;
    __syncthreads();
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * NT) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * NT;
            if (i < total)
                v[j] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * NT;
            if (i < total) {
                const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                float m = 0.0f;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[k] << 16)), fabsf(__uint_as_float(w4[k] & 0xFFFF0000u))));
                atomicMax(&xm[i / n8], __float_as_uint(m));
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < a.T) {
        const int sh = f16_shift_for_max(__uint_as_float(xm[threadIdx.x]));
        rs.xundo[threadIdx.x] = exp2i(-sh);
        rs.xscale[threadIdx.x] = exp2i(sh);
    }
    __syncthreads();
    for (int i0 = threadIdx.x; i0 < total; i0 += 4 * NT) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * NT;
            if (i < total)
                v[j] = __ldg(reinterpret_cast<const uint4 *>(a.x) + i);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * NT;
            if (i < total) {
                const int t = i / n8, c = i - t * n8;
                const float sc = rs.xscale[t];
                const uint32_t w4[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    __half2 h2 = __floats2half2_rn(__uint_as_float(w4[k] << 16) * sc,
                                                   __uint_as_float(w4[k] & 0xFFFF0000u) * sc);
                    o[k] = *reinterpret_cast<uint32_t *>(&h2);
                }
                *reinterpret_cast<uint4 *>(xwin + (size_t)t * a.xwin_row + 8 * c) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

// Order key of a normalised logit pair (hi, lo): larger value -> larger key.
// lo is below half an ulp of hi, so (hi, lo) order is the order of the sums.

// The next layer's router weights and shared expert into L2: this CTA's
// slice of each region, issued once its own weight streams are done.
__device__ void prefetch_next_layer(const FusedArgs &a) {
    if (threadIdx.x != 0)
        return;
    for (int r = 0; r < 3; ++r) {
        const uint8_t *base = a.next_pf[r];
        const size_t total = a.next_pf_bytes[r];
        if (!base || total == 0 || (reinterpret_cast<uintptr_t>(base) & 15))   // bulk prefetches want 16-byte alignment
            continue;
        const size_t piece = align_up((total + gridDim.x - 1) / gridDim.x, 16);
        const size_t lo = (size_t)blockIdx.x * piece;
        const size_t hi = lo + piece < total ? lo + piece : total;
        for (size_t o = lo; o + 16 <= hi; o += 16384) {
            const size_t n = hi - o < 16384 ? (hi - o) & ~(size_t)15 : 16384;
            prefetch_l2(base + o, (uint32_t)n);
        }
    }
}


// Order key of logit + bias from its (P, Q) pair.
__device__ __forceinline__ void put_key(const FusedArgs &a, RouteState &rs, unsigned long long *key, int t, int e,
                                        float P, float Q) {
    pair_add(P, Q, a.bias ? __ldg(a.bias + e) : 0.0f, 0.0f);
    float hi, lo;
    two_sum(P, Q, hi, lo);
    if (!isfinite(hi))
        rs.bad = 1;                                  // non-finite router logits
    key[t * ((a.E + 31) & ~31) + e] = logit_order_key(hi, lo);
}

// Logit keys.  With r_final the router phase left each logit's pair in chunk
// 0's slot.  Otherwise every CTA sums the chunk pairs itself, from one of
// kRouterCopies copies (spreading the CTAs' reads of the same lines): S
// consecutive threads share a logit's chunks, each summing its range in chunk
// order, and combine in a fixed tree.
__device__ void route_logits(const FusedArgs &a, RouteState &rs, unsigned long long *key) {
    const int tid = threadIdx.x, T = a.T, E = a.E;
    if (a.r_final) {
#pragma unroll 4
        for (int i = tid; i < T * E; i += NT) {
            const float2 v = __ldcg(a.rpart + i);
            put_key(a, rs, key, i / E, i % E, v.x, v.y);
        }
        return;
    }
    const float2 *src = a.rpart + (size_t)(blockIdx.x % kRouterCopies) * a.r_chunks * T * E;
    int S = 1;
    while (S < 8 && 2 * S * T * E <= NT)
        S *= 2;
    const int cps = (a.r_chunks + S - 1) / S;
    for (int i0 = 0; i0 < T * E * S; i0 += NT) {
        const int i = i0 + tid, item = i / S, part = i - item * S;
        const bool live = item < T * E;
        const int t = live ? item / E : 0, e = live ? item - t * E : 0;
        const int c_lo = part * cps, c_hi = min(a.r_chunks, c_lo + cps);
        float P = 0.0f, Q = 0.0f;
        for (int c0 = c_lo; c0 < c_hi; c0 += 16) {
            float2 v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (live && c0 + c < c_hi)
                    v[c] = __ldcg(src + ((size_t)(c0 + c) * T + t) * E + e);
#pragma unroll
            for (int c = 0; c < 16; ++c)
                if (live && c0 + c < c_hi)
                    pair_add(P, Q, v[c].x, v[c].y);
        }
        for (int d = 1; d < S; d *= 2) {            // S divides 32: groups stay inside a warp
            const float oP = __shfl_xor_sync(0xffffffffu, P, d), oQ = __shfl_xor_sync(0xffffffffu, Q, d);
            if ((part & d) == 0)
                pair_add(P, Q, oP, oQ);
        }
        if (live && part == 0)
            put_key(a, rs, key, t, e, P, Q);
    }
}

// Returns false when the routing selected an invalid expert (non-finite
// logits); every CTA reaches the same answer.
__device__ bool phase_route(const FusedArgs &a, RouteState &rs, uint8_t *smA, uint8_t *smB) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const int T = a.T, E = a.E, k = a.k, kps = a.k + a.S, n = T * kps, n_tot = a.E + a.S;
    const int Ep = (E + 31) & ~31;                  // experts padded to whole groups of 32
    const int cmax = (Ep / 32) * k;                  // sorted group lists: k entries per group
    unsigned long long *key = reinterpret_cast<unsigned long long *>(smB);          // [T][Ep]
    unsigned long long *ckey = key + (size_t)T * Ep;                                  // [T][cmax]
    int *cand = reinterpret_cast<int *>(ckey + (size_t)T * cmax);                     // [T][cmax]
    route_logits(a, rs, key);
    for (int i = tid; i < T * (Ep - E); i += NT)     // padding ranks below every real key
        key[(i / (Ep - E)) * Ep + E + i % (Ep - E)] = 0ull;
    __syncthreads();
    stamp(a, 9);
    // top k, stage 1: an expert ranked k or lower inside its group of 32
    // cannot be in the top k; the group's first k ranks fill its sorted list
    // (order: key descending, index ascending; padding carries index
    // 0x7fffffff and key 0 and never reaches the top k)
    for (int i = tid; i < T * Ep; i += NT) {
        const int t = i / Ep, e = i - t * Ep;
        const unsigned long long *g = key + t * Ep + (e & ~31);
        const unsigned long long my = g[e & 31];
        // rank by the high words, two keys per 16-byte load; a key sharing
        // the high word (besides the own one) sends the item to the full
        // 64-bit comparison with the index rule
        const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
        const uint32_t myhi = (uint32_t)(my >> 32);
        int r = 0, eq = 0;
#pragma unroll 8
        for (int j2 = 0; j2 < 16; ++j2) {
            const uint4 w = g4[j2];                 // key 2j2: (x lo, y hi), key 2j2+1: (z lo, w hi)
            r += (w.y > myhi) + (w.w > myhi);
            eq += (w.y == myhi) + (w.w == myhi);
        }
        if (eq > 1) {
            r = 0;
            for (int j = 0; j < 32; ++j) {
                const unsigned long long o = g[j];
                r += (o > my) | ((o == my) & (j < (e & 31)));
            }
        }
        if (r < k) {
            const int slot = t * cmax + (e >> 5) * k + r;
            ckey[slot] = my;
            cand[slot] = e < E ? e : 0x7fffffff;
        }
    }
    __syncthreads();
    // stage 2, one warp per token: lane g holds the head of group g's list;
    // each round takes the largest head (key, then lower index), and its lane
    // moves to the next entry of its list.  Slot r gets the r-th largest
    // logit.  The softmax over the kept logits is taken relative to the
    // largest, its denominator summed in slot order.
    if (warp < T) {
        const unsigned full = 0xffffffffu;
        const int t = warp, G = Ep >> 5;
        const unsigned long long *ck = ckey + t * cmax;
        const int *ce = cand + t * cmax;
        int pos = 0;
        unsigned long long hk = lane < G ? ck[lane * k] : 0ull;
        unsigned he = lane < G ? (unsigned)ce[lane * k] : 0xffffffffu;
        unsigned long long myk = 0ull;
        int myid = -1;
        for (int r = 0; r < k; ++r) {
            const uint32_t hh = (uint32_t)(hk >> 32), mh = __reduce_max_sync(full, hh);
            const uint32_t ml = __reduce_max_sync(full, hh == mh ? (uint32_t)hk : 0u);
            const unsigned we = __reduce_min_sync(full, (hh == mh && (uint32_t)hk == ml) ? he : 0xffffffffu);
            if (lane == r) {
                myk = ((unsigned long long)mh << 32) | ml;
                myid = (int)we;
            }
            if (lane < G && he == we && we < (unsigned)E) {
                ++pos;
                hk = pos < k ? ck[lane * k + pos] : 0ull;
                he = pos < k ? (unsigned)ce[lane * k + pos] : 0xffffffffu;
            }
        }
        const unsigned long long k0 = __shfl_sync(full, myk, 0);
        float ex = 0.0f;
        if (lane < k) {
            const float h0 = logit_from_key((uint32_t)(k0 >> 32)), l0 = logit_from_key((uint32_t)k0);
            const float hr = logit_from_key((uint32_t)(myk >> 32)), lr = logit_from_key((uint32_t)myk);
            ex = expf(__fadd_rn(__fsub_rn(hr, h0), __fsub_rn(lr, l0)));
        }
        float denom = 0.0f;
        for (int r = 0; r < k; ++r)
            denom += __shfl_sync(full, ex, r);
        if (lane < k) {
            const float w = ex / denom;
            rs.sel_id[t * kps + lane] = myid;
            rs.sel_w[t * kps + lane] = w;
            if (blockIdx.x == 0) {
                if (a.ids_out)
                    a.ids_out[t * kps + lane] = myid;
                if (a.w_out)
                    a.w_out[t * kps + lane] = w;
            }
        }
        if (a.S && lane == k) {
            rs.sel_id[t * kps + k] = E;
            rs.sel_w[t * kps + k] = a.shared_weight;
            if (blockIdx.x == 0) {
                if (a.ids_out)
                    a.ids_out[t * kps + k] = E;
                if (a.w_out)
                    a.w_out[t * kps + k] = a.shared_weight;
            }
        }
    }
    __syncthreads();
    stamp(a, 10);
    if (tid < n && (unsigned)rs.sel_id[tid] >= (unsigned)n_tot)
        rs.bad = 1;
    __syncthreads();
    if (rs.bad) {
        if (blockIdx.x == 0 && tid == 0)
            record_status(a.hdr, MOE_ERR_DEVICE_ASSERT);
        return false;
    }
    if (n <= 32) {
        // one warp: entry `lane` -> sorted position, group starts and sizes,
        // passes, with shuffles and ballots only
        if (warp == 0) {
            const unsigned full = 0xffffffffu;
            const int ei = lane < n ? rs.sel_id[lane] : 0x7fffffff;
            int pos = 0;
            for (int j = 0; j < n; ++j) {
                const int ej = __shfl_sync(full, ei, j);
                pos += (ej < ei) | ((ej == ei) & (j < lane));
            }
            if (lane < n) {
                rs.inv_pos[lane] = pos;
                rs.sorted_ent[pos] = lane;
                rs.sorted_tok[pos] = lane / kps;
            }
            __syncwarp();
            const int ex = lane < n ? rs.sel_id[rs.sorted_ent[lane]] : -1;
            const int prev = __shfl_up_sync(full, ex, 1);
            const bool start = lane < n && (lane == 0 || prev != ex);
            const unsigned starts = __ballot_sync(full, start);
            const unsigned later = lane == 31 ? 0u : starts & ~((2u << lane) - 1u);
            const int next = later ? __ffs(later) - 1 : n;
            const int size = start ? next - lane : 0;
            const int gi = __popc(starts & ((1u << lane) - 1u));
            const int d4 = (size + kPassEntries - 1) / kPassEntries;
            int incl = d4;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(full, incl, d);
                if (lane >= d)
                    incl += y;
            }
            if (start) {
                const int di = incl - d4;
                rs.pgu[gi] = Pass{ex, lane, size, 0};
                for (int q = 0; q < d4; ++q)
                    rs.pdn[di + q] = Pass{ex, lane + q * kPassEntries, min(kPassEntries, size - q * kPassEntries), 0};
            }
            if (lane == 31) {
                rs.n_gu = __popc(starts);
                rs.n_dn = incl;
            }
        }
        __syncthreads();
        return true;
    }
    // sorted position of entry i: entries with a smaller expert, or the same
    // expert and a smaller index, come first
    if (tid < n) {
        const int ei = rs.sel_id[tid];
        int pos = 0;
        for (int j = 0; j < n; ++j) {
            const int ej = rs.sel_id[j];
            pos += (ej < ei) || (ej == ei && j < tid);
        }
        rs.inv_pos[tid] = pos;
        rs.sorted_ent[pos] = tid;
        rs.sorted_tok[pos] = tid / kps;
    }
    __syncthreads();
    // by sorted position p = tid: group starts from one ballot per warp; the
    // group's size from the next start (this warp, else the first later warp
    // holding one); group and down-pass indices from per-warp counts
    {
        __shared__ int wstarts[NW], wfirst[NW], wd4[NW];
        const unsigned full = 0xffffffffu;
        const int p = tid;
        int ex = -1;
        bool start = false;
        if (p < n) {
            ex = rs.sel_id[rs.sorted_ent[p]];
            start = p == 0 || rs.sel_id[rs.sorted_ent[p - 1]] != ex;
        }
        const unsigned sm = __ballot_sync(full, start);
        if (lane == 0) {
            wstarts[warp] = __popc(sm);
            wfirst[warp] = sm ? 32 * warp + __ffs(sm) - 1 : 0x7fffffff;
        }
        __syncthreads();
        int size = 0;
        if (start) {
            const unsigned later = lane == 31 ? 0u : sm & ~((2u << lane) - 1u);
            int next = n;
            if (later) {
                next = 32 * warp + __ffs(later) - 1;
            } else {
                for (int w = warp + 1; w < NW; ++w)
                    if (wfirst[w] != 0x7fffffff) {
                        next = wfirst[w];
                        break;
                    }
            }
            size = next - p;
        }
        const int d4 = (size + kPassEntries - 1) / kPassEntries;
        int incl = d4;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(full, incl, d);
            if (lane >= d)
                incl += y;
        }
        if (lane == 31)
            wd4[warp] = incl;
        __syncthreads();
        if (start) {
            int gi = __popc(sm & ((1u << lane) - 1u)), di = incl - d4;
            for (int w = 0; w < warp; ++w) {
                gi += wstarts[w];
                di += wd4[w];
            }
            rs.pgu[gi] = Pass{ex, p, size, 0};
            for (int q = 0; q * kPassEntries < size; ++q)
                rs.pdn[di + q] = Pass{ex, p + q * kPassEntries, min(kPassEntries, size - q * kPassEntries), 0};
        }
        if (tid == 0) {
            int gi = 0, di = 0;
            for (int w = 0; w < NW; ++w) {
                gi += wstarts[w];
                di += wd4[w];
            }
            rs.n_gu = gi;
            rs.n_dn = di;
        }
    }
    __syncthreads();
    return true;
}

// ------------------------------------------------------- streaming (G, D)

struct UnitCursor {
    int ul, bi;      // CTA-local unit, batch within the unit
    int P, rb;       // pass and row block of the unit
};

__device__ __forceinline__ void cursor_set(UnitCursor &c, long long u0, int b, int nb, int upe) {
    c.ul = b / nb;
    c.bi = b - c.ul * nb;
    const long long u = u0 + c.ul;
    c.P = (int)(u / upe);
    c.rb = (int)(u - (long long)c.P * upe);
}

__device__ __forceinline__ void cursor_next(UnitCursor &c, int nb, int upe) {
    if (++c.bi == nb) {
        c.bi = 0;
        ++c.ul;
        if (++c.rb == upe) {
            c.rb = 0;
            ++c.P;
        }
    }
}

// Warp owning CTA-local batch b when Bc batches are split over NW warps as
// [w*Bc/NW, (w+1)*Bc/NW).
__device__ __forceinline__ int warp_of_batch(long long b, long long Bc) { return (int)(((b + 1) * NW - 1) / Bc); }

struct Phase {
    const uint8_t *sec;      // packed section
    unsigned unit_bytes;     // bytes of one row block
    int upe;                 // row blocks per expert
    int steps;               // 64-element steps per row block
    int nb;                  // batches per row block
    const Pass *passes;
    const __half *win;       // activation window in shared memory
    int win_row;
    int e_lo;                // down: first entry of the window
    const float *hundo;      // down: per window entry, undoes the h scaling
    int win_rows;            // rows the window holds (range checks of the debug build)
    const uint32_t *hdr;
};

template <bool FULL>
__device__ __forceinline__ void load_batch(uint4 (&q)[SB], uint32_t (&s)[SB], const Phase &ph, const UnitCursor &c,
                                           int lane, uint64_t pol) {
    const uint8_t *p = ph.sec + ((size_t)ph.passes[c.P].expert * ph.upe + c.rb) * ph.unit_bytes +
                       (size_t)c.bi * kBatchBytes;
    const int ns = FULL ? SB : min(SB, ph.steps - c.bi * SB);
#pragma unroll
    for (int j = 0; j < SB; ++j) {
        if (FULL || j < ns) {
            q[j] = ld_stream16(p + j * kStepBytes + lane * 16, pol);
            s[j] = ld_stream4(p + j * kStepBytes + 512 + (lane >> 2) * 4, pol);
        }
    }
}

// One 16 x 64 step: decode, two MMAs per 32-element block, block scales.
__device__ __forceinline__ void step_mma(const uint4 q, const uint32_t s, const __half *bp, float (&acc)[4]) {
    const uint4 b0 = *reinterpret_cast<const uint4 *>(bp);
    const uint4 b1 = *reinterpret_cast<const uint4 *>(bp + 32);
    uint32_t pa[4], qa[4];
    const float zero[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    float d[4], e[4];
    float sg0, sg1, sh0, sh1;       // rows g / g+8, blocks 2q / 2q+1
    e8m0x4_to_f32(s, sg0, sg1, sh0, sh1);
    decode_e2m1x8(q.x, pa);
    decode_e2m1x8(q.y, qa);
    mma_m16n8k16_f16(d, pa[0], qa[0], pa[1], qa[1], b0.x, b0.y, zero);
    mma_m16n8k16_f16(d, pa[2], qa[2], pa[3], qa[3], b0.z, b0.w, d);
    decode_e2m1x8(q.z, pa);
    decode_e2m1x8(q.w, qa);
    mma_m16n8k16_f16(e, pa[0], qa[0], pa[1], qa[1], b1.x, b1.y, zero);
    mma_m16n8k16_f16(e, pa[2], qa[2], pa[3], qa[3], b1.z, b1.w, e);
    acc[0] = fmaf(d[0], sg0, acc[0]);
    acc[1] = fmaf(d[1], sg0, acc[1]);
    acc[2] = fmaf(d[2], sh0, acc[2]);
    acc[3] = fmaf(d[3], sh0, acc[3]);
    acc[0] = fmaf(e[0], sg1, acc[0]);
    acc[1] = fmaf(e[1], sg1, acc[1]);
    acc[2] = fmaf(e[2], sh1, acc[2]);
    acc[3] = fmaf(e[3], sh1, acc[3]);
}

template <bool FULL>
__device__ __forceinline__ void compute_batch(const uint4 (&q)[SB], const uint32_t (&s)[SB], const Phase &ph,
                                              const UnitCursor &c, const __half *bp, float (&acc)[4]) {
    const int ns = FULL ? SB : min(SB, ph.steps - c.bi * SB);
    const __half *b = bp + c.bi * (SB * 64);
#pragma unroll
    for (int j = 0; j < SB; ++j)
        if (FULL || j < ns)
            step_mma(q[j], s[j], b + 64 * j, acc);
}

// This lane's B-operand pointer at the start of the unit under the cursor:
// gate/up reads the x row of the pass's token in MMA column g; down reads
// the hi (columns 0..3) or lo (4..7) row of the pass's entry g % 4.
__device__ __forceinline__ const __half *unit_bptr(int mode, const Phase &ph, const RouteState &rs,
                                                   const UnitCursor &c, int lane) {
    const Pass ps = ph.passes[c.P];
    const int g = lane >> 2, cc = lane & 3;
    int row = mode == kFfnGateUp ? rs.sorted_tok[ps.begin + min(g, ps.count - 1)]
                                 : 2 * (ps.begin + min(g & 3, ps.count - 1) - ph.e_lo) + (g >> 2);
    if (!MOE_DBG_IN_RANGE(row, ph.win_rows, ph.hdr))
        row = 0;
    return ph.win + (size_t)row * ph.win_row + 8 * cc;
}

// A unit's sums are complete: write h = silu(gate) * up (gate/up) or the
// per-entry outputs Y (down) of its real columns.
__device__ __forceinline__ void finish_unit(int mode, const FusedArgs *a, const RouteState *rs, const Pass *passes,
                                         int e_lo, const float *hundo, int P, int rb, float a0, float a1, float a2,
                                         float a3) {
    const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const Pass ps = passes[P];
    const int entries = a->T * (a->k + a->S);
    if (mode == kFfnGateUp) {
        const float acc[4] = {a0, a1, a2, a3};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = 2 * c + h;
            if (n < ps.count && MOE_DBG_IN_RANGE(ps.begin + n, entries, a->hdr) &&
                MOE_DBG_IN_RANGE(8 * rb + g, a->I, a->hdr)) {
                const float xu = rs->xundo[rs->sorted_tok[ps.begin + n]];
                const float G = acc[h] * xu, U = acc[2 + h] * xu;
                a->h32[(size_t)(ps.begin + n) * a->I + 8 * rb + g] = G / (1.0f + expf(-G)) * U;
            }
        }
    } else {
        float y[4] = {a0, a1, a2, a3};
#pragma unroll
        for (int i = 0; i < 4; ++i)   // add the lo column n+4 to the hi column n
            y[i] += __shfl_xor_sync(0xffffffffu, y[i], 2);
        if (c < 2) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = 2 * c + h;
                if (n < ps.count && MOE_DBG_IN_RANGE(ps.begin + n, entries, a->hdr) &&
                    MOE_DBG_IN_RANGE(ps.begin + n - e_lo, a->win_entries, a->hdr) &&
                    MOE_DBG_IN_RANGE(16 * rb + g + 8, a->H, a->hdr)) {
                    const int e = ps.begin + n;
                    const float u = hundo[e - e_lo];
                    float *dst = a->yent + (size_t)e * a->H + 16 * rb;
                    dst[g] = y[h] * u;
                    dst[g + 8] = y[2 + h] * u;
                }
            }
        }
    }
}

// h rows of window entries -> f16 hi + lo rows, scaled per entry by 2^s with
// max|h| in [2^14, 2^15); one warp per entry.
__device__ void h_to_window(const FusedArgs &a, int e_lo, int n_win, int win_row, __half *win, float *hundo) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, I = a.I;
    for (int ew = warp; ew < n_win; ew += NW) {
        const float4 *src = reinterpret_cast<const float4 *>(a.h32 + (size_t)(e_lo + ew) * I);
        float m = 0.0f;
        for (int i = lane; i < I / 4; i += 32) {
            const float4 v = __ldcg(src + i);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
        const int sh = f16_shift_for_max(m);
        const float sc = exp2i(sh);
        __half *hi = win + (size_t)(2 * ew) * win_row, *lo = hi + win_row;
        for (int i = lane; i < I / 4; i += 32) {
            const float4 v = __ldcg(src + i);
            const float vv[4] = {v.x * sc, v.y * sc, v.z * sc, v.w * sc};
            __half hv[4], lv[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                hv[j] = __float2half_rn(vv[j]);
                lv[j] = __float2half_rn(vv[j] - __half2float(hv[j]));
            }
            *reinterpret_cast<uint2 *>(hi + 4 * i) = *reinterpret_cast<const uint2 *>(hv);
            *reinterpret_cast<uint2 *>(lo + 4 * i) = *reinterpret_cast<const uint2 *>(lv);
        }
        if (lane == 0)
            hundo[ew] = exp2i(-sh);
    }
}

// One streaming phase, shared by gate/up and down so that the down phase runs
// the code the gate/up phase has just brought into the instruction cache.
// Each CTA takes a contiguous range of whole row-block units; its warps take
// contiguous ranges of the range's batches.  A warp finishes the units it
// streams completely; units shared between warps leave partial sums in slot
// 2*warp (the warp's first unit) or 2*warp+1 (its last unit), which the warp
// holding the unit's last batch adds up in warp order.  The first batch is
// issued before anything else; for the down phase that is before the wait for
// every CTA's h.  Returns false when that wait gave up.
template <bool FULL>
__device__ __forceinline__ bool stream_phase(const FusedArgs *ap, int mode) {
    const FusedArgs &a = *ap;
    RouteState &rs = fz_rs;
    uint8_t *smem = fz_smem;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x;
    const uint64_t pol = l2_evict_first_policy();
    float *hundo = reinterpret_cast<float *>(smem + a.off_hundo);
    float *slots = reinterpret_cast<float *>(smem + a.off_b);
    const bool down = mode == kFfnDown;
    Phase ph;
    ph.sec = down ? a.dn : a.gu;
    ph.unit_bytes = down ? a.dn_unit : a.gu_unit;
    ph.upe = down ? a.H / 16 : a.I / 8;
    ph.steps = down ? a.I / 64 : a.H / 64;
    ph.nb = (ph.steps + SB - 1) / SB;
    ph.passes = down ? rs.pdn : rs.pgu;
    ph.win = reinterpret_cast<const __half *>(smem);
    ph.win_row = down ? a.hwin_row : a.xwin_row;
    ph.e_lo = 0;
    ph.hundo = hundo;
    ph.win_rows = down ? 2 * a.win_entries : a.T;
    ph.hdr = a.hdr;
    const long long U = (long long)(down ? rs.n_dn : rs.n_gu) * ph.upe;
    const long long u0 = (long long)blockIdx.x * U / G, u1 = (long long)(blockIdx.x + 1) * U / G;
    const long long Bc = (u1 - u0) * ph.nb;
    const int bw0 = (int)((long long)warp * Bc / NW), bw1 = (int)((long long)(warp + 1) * Bc / NW);
    uint4 q[NBUF][SB];
    uint32_t s[NBUF][SB];
    UnitCursor cc, lc;
    int lb = bw0;                         // next batch to load into registers
    if (bw0 < bw1) {
        cursor_set(cc, u0, bw0, ph.nb, ph.upe);
        lc = cc;
#pragma unroll
        for (int i = 0; i < NBUF - 1; ++i) {
            if (lb < bw1) {
                load_batch<FULL>(q[i], s[i], ph, lc, lane, pol);
                cursor_next(lc, ph.nb, ph.upe);
                ++lb;
            }
        }
    }
    if (down) {
        if (!grid_wait(a, 2u * G))
            return false;
        stamp(a, 5);
        cta_stamp(a, 1);
        if (u1 > u0) {
            const int P0 = (int)(u0 / ph.upe), P1 = (int)((u1 - 1) / ph.upe);
            ph.e_lo = rs.pdn[P0].begin;
            const int n_win = rs.pdn[P1].begin + rs.pdn[P1].count - ph.e_lo;
            if (n_win > a.win_entries) {           // cannot happen for the sizes the host admits
                if (threadIdx.x == 0)
                    record_status(a.hdr, MOE_ERR_DEVICE_ASSERT);
                return true;
            }
            h_to_window(a, ph.e_lo, n_win, ph.win_row, reinterpret_cast<__half *>(smem), hundo);
        }
        __syncthreads();
    }
    if (bw0 < bw1) {
        const int ul_first = cc.ul;
        const __half *bp = unit_bptr(mode, ph, rs, cc, lane);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        int b = bw0;
        auto end_batch = [&]() {
            const bool unit_end = cc.bi == ph.nb - 1;
            const bool range_end = b + 1 == bw1;
            if (unit_end || range_end) {
                if (unit_end && cc.ul * ph.nb >= bw0) {
                    finish_unit(mode, &a, &rs, ph.passes, ph.e_lo, ph.hundo, cc.P, cc.rb, acc[0], acc[1], acc[2],
                                acc[3]);
                } else {
                    const int slot = cc.ul == ul_first ? 2 * warp : 2 * warp + 1;
                    *reinterpret_cast<float4 *>(slots + (slot * 32 + lane) * 4) =
                        make_float4(acc[0], acc[1], acc[2], acc[3]);
                }
                acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            }
            cursor_next(cc, ph.nb, ph.upe);
            if (cc.bi == 0 && !range_end)
                bp = unit_bptr(mode, ph, rs, cc, lane);
        };
        // ring of NBUF register buffers: buffer i holds batch b; the load of
        // batch b + NBUF - 1 goes into the buffer consumed last
        bool more = true;
        while (more) {
#pragma unroll
            for (int i = 0; i < NBUF; ++i) {
                if (lb < bw1) {
                    load_batch<FULL>(q[(i + NBUF - 1) % NBUF], s[(i + NBUF - 1) % NBUF], ph, lc, lane, pol);
                    cursor_next(lc, ph.nb, ph.upe);
                    ++lb;
                }
                compute_batch<FULL>(q[i], s[i], ph, cc, bp, acc);
                end_batch();
                if (++b >= bw1) {
                    more = false;
                    break;
                }
            }
        }
    }
    __syncthreads();
    cta_stamp(a, down ? 2 : 0);
    // units shared between warps, finished by the warp holding the last batch
    if (bw0 < bw1 && Bc > 0) {
        const long long ul = bw0 / ph.nb;
        const long long ue = min((ul + 1) * ph.nb, Bc) - 1;
        if (ul * ph.nb != bw0 && ue < bw1) {
            const int wf = warp_of_batch(ul * ph.nb, Bc);
            float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int w = wf; w <= warp; ++w) {
                const long long wb0 = (long long)w * Bc / NW, wb1 = (long long)(w + 1) * Bc / NW;
                if (wb0 >= wb1)
                    continue;
                const int slot = wb0 / ph.nb == ul ? 2 * w : 2 * w + 1;
                const float4 v = *reinterpret_cast<const float4 *>(slots + (slot * 32 + lane) * 4);
                acc[0] += v.x;
                acc[1] += v.y;
                acc[2] += v.z;
                acc[3] += v.w;
            }
            const long long u = u0 + ul;
            const int P = (int)(u / ph.upe), rb = (int)(u - (long long)P * ph.upe);
            finish_unit(mode, &a, &rs, ph.passes, ph.e_lo, ph.hundo, P, rb, acc[0], acc[1], acc[2], acc[3]);
        }
    }
    return true;
}

// y = bf16(sum over slots, in slot order, of w * Y) for this CTA's equal
// share of the T x H outputs, after every CTA's per-entry outputs Y are
// written (third grid wait).  All loads of a thread are issued first.
__device__ void combine_share(const FusedArgs &a, const RouteState &rs) {
    const int kps = a.k + a.S, TH = a.T * a.H, G = gridDim.x;
    const int o0 = (int)((long long)blockIdx.x * TH / G), o1 = (int)((long long)(blockIdx.x + 1) * TH / G);
    for (int o = o0 + threadIdx.x; o < o1; o += NT) {
        const int t = o / a.H, hcol = o - t * a.H;
        float v[kMaxSlots];
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s)
            if (s < kps)
                v[s] = MOE_DBG_IN_RANGE(rs.inv_pos[t * kps + s], a.T * kps, a.hdr)
                           ? __ldcg(a.yent + (size_t)rs.inv_pos[t * kps + s] * a.H + hcol)
                           : 0.0f;
        float acc = 0.0f;
#pragma unroll
        for (int s = 0; s < kMaxSlots; ++s)
            if (s < kps)
                acc = fmaf(rs.sel_w[t * kps + s], v[s], acc);
        const __nv_bfloat16 bv = __float2bfloat16_rn(acc);
        a.y[o] = *reinterpret_cast<const uint16_t *>(&bv);
    }
}

// CTA 0 writes the grouping every CTA derived: the sorted order (token and
// slot of each sorted position) and its inverse, the per-expert offsets
// (exclusive prefix of the counts, n_tot + 1 values), the active experts in
// ascending order and their count (header), and for the routing-only
// instantiation the passes of one expert's entries.  0 passes and 0 active
// experts when the routing was rejected.
__device__ void route_export(const FusedArgs &a, const RouteState &rs, bool ok, bool with_passes) {
    const int kps = a.k + a.S, n = a.T * kps, n_tot = a.E + a.S;
    if (ok) {
        for (int i = threadIdx.x; i < n; i += NT) {
            const int ent = rs.sorted_ent[i];
            a.x_sorted_tok[i] = rs.sorted_tok[i];
            a.x_sorted_slot[i] = ent - (ent / kps) * kps;
            a.x_inv_pos[i] = rs.inv_pos[i];
        }
        for (int p = threadIdx.x; p < rs.n_gu; p += NT) {
            a.x_active[p] = rs.pgu[p].expert;
            if (with_passes)
                a.x_passes[p] = rs.pgu[p];
        }
        // offsets[e]: the first sorted position whose expert is >= e, i.e. the
        // begin of the first pass (ascending experts) with expert >= e
        for (int e = threadIdx.x; e <= n_tot; e += NT) {
            int lo = 0, hi = rs.n_gu;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (rs.pgu[mid].expert < e)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            a.x_offsets[e] = lo < rs.n_gu ? rs.pgu[lo].begin : n;
        }
    }
    if (threadIdx.x == 0) {
        a.hdr[kHdrNumActive] = ok ? (uint32_t)rs.n_gu : 0u;
        if (with_passes) {
            a.hdr[kHdrNumPassesW4] = ok ? (uint32_t)rs.n_gu : 0u;
            a.hdr[kHdrNumPasses] = ok ? (uint32_t)rs.n_gu : 0u;
        }
    }
}

// ---------------------------------------------------------------- kernel

// ROUTE_ONLY: phases R and T, then the grouping is exported (route_export)
// and the CTAs leave; no expert weights are read.
template <bool FULL, bool ROUTE_ONLY>
__global__ void __launch_bounds__(NT, 1) fused_layer_kernel(const __grid_constant__ FusedArgs a) {
    uint8_t *smem = fz_smem;
    RouteState &rs = fz_rs;
    const int G = gridDim.x;

    // read-only prefetches, then wait until the previous kernel on the stream
    // has completed (its outputs and the workspace are then ours); the next
    // kernel may be scheduled from here on
    if constexpr (!ROUTE_ONLY)
        prefetch_shared_expert(a);
    prefetch_router_tile(a);
    pdl_wait();
    pdl_trigger();
    stamp(a, 0);
    if (blockIdx.x == 0 && threadIdx.x == 0)
        reinterpret_cast<unsigned long long *>(a.hdr + kHdrStamps)[12] = clock64();
    if (threadIdx.x == 0)
        rs.bad = 0;
    phase_router(a, smem);                  // nothing else lives in shared memory yet
    stamp(a, 1);
    grid_arrive(a);
    if constexpr (!ROUTE_ONLY) {
        x_window_local(a, rs, reinterpret_cast<__half *>(smem));
    } else if (a.x_q) {
        // while the routing waits: x to MXFP8, one warp per block of 32
        const int nblk = a.T * (a.H / 32);
        for (int b = blockIdx.x * NW + (threadIdx.x >> 5); b < nblk; b += G * NW) {
            const size_t i = (size_t)b * 32 + (threadIdx.x & 31);
            mxfp8_quant_block(__uint_as_float((uint32_t)a.x[i] << 16), a.x_q + i, a.x_qs + b);
        }
    }
    bool ok = grid_wait(a, (unsigned)G);
    stamp(a, 2);
    if (ok)
        ok = phase_route(a, rs, smem, smem + a.off_b);
    stamp(a, 3);
    if constexpr (ROUTE_ONLY) {
        if (blockIdx.x == 0)
            route_export(a, rs, ok, true);
    } else if (ok) {
        // gate/up, then down: one copy of the streaming code runs both
#pragma unroll 1
        for (int mode = kFfnGateUp; mode <= kFfnDown; ++mode) {
            if (mode == kFfnDown) {
                stamp(a, 4);
                grid_arrive(a);
                if (blockIdx.x == 0)        // while CTA 0 waits for the other CTAs' h
                    route_export(a, rs, true, false);
            }
            if (!stream_phase<FULL>(&a, mode)) {
                ok = false;
                break;
            }
        }
        // every CTA's per-entry outputs, then the combine
        if (ok) {
            stamp(a, 11);
            cta_stamp(a, 3);
            prefetch_next_layer(a);
            grid_arrive(a);
            if (grid_wait(a, 3u * G)) {
                stamp(a, 14);
                combine_share(a, rs);
            }
        }
        stamp(a, 6);
        if (blockIdx.x == 0 && threadIdx.x == 0)
            reinterpret_cast<unsigned long long *>(a.hdr + kHdrStamps)[13] = clock64();
    }
    // the last CTA to leave resets the wait counters for the next call
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.hdr + kHdrDone, 1u) == (unsigned)G - 1) {
            a.hdr[kHdrBarrier] = 0;
            a.hdr[kHdrAbort] = 0;
            a.hdr[kHdrDone] = 0;
            reinterpret_cast<unsigned long long *>(a.hdr + kHdrStamps)[7] = globaltimer_ns();
            __threadfence();
        }
    }
}

// Self-test of the bounded grid wait: one CTA arrives and waits for an
// arrival that never comes; the wait gives up after kWaitLimitNs, records
// MOE_ERR_DEVICE_TIMEOUT, and the CTA leaves the way the layer kernel does.
__global__ void wait_selftest_kernel(const __grid_constant__ FusedArgs a) {
    grid_arrive(a);
    grid_wait(a, gridDim.x + 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(a.hdr + kHdrDone, 1u) == gridDim.x - 1) {
            a.hdr[kHdrBarrier] = 0;
            a.hdr[kHdrAbort] = 0;
            a.hdr[kHdrDone] = 0;
            __threadfence();
        }
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t *hdr, cudaStream_t stream) {
    FusedArgs a{};
    a.hdr = hdr;
    wait_selftest_kernel<<<1, 32, 0, stream>>>(a);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- host side

FusedPlan fused_plan(int T, int H, int I, int E, int k, int S, int grid) {
    FusedPlan p{};
    p.ok = false;
    if (T < 1 || T > kFusedMaxTokens || grid < 1 || H % 64 || I % 64)
        return p;
    const int kps = k + S, n = T * kps, n_tot = E + S;
    fused_router_tiling(H, E, &p.r_groups, &p.r_chunks, &p.r_rows);
    // past ~48 KB of chunk pairs per CTA, summing each group once in the
    // router phase (a ticket and one more dependent step) beats every CTA
    // reading them all
    p.r_final = (long long)T * E * p.r_chunks * 8 > 48 * 1024;
    p.xwin_row = H + 32;
    p.hwin_row = I + 32;
    // down units a CTA can own, and the entries their passes can span
    const int active = n < n_tot ? n : n_tot;
    const long long max_pdn = (n + (long long)(kPassEntries - 1) * active) / kPassEntries;
    const int upe_dn = H / 16;
    const long long nu_dn = (max_pdn * upe_dn + grid - 1) / grid;
    const long long spanned = (nu_dn + upe_dn - 1) / upe_dn + 1;
    long long we = spanned * kPassEntries;
    if (we > n)
        we = n;
    p.win_entries = (int)we;
    const size_t a_x = (size_t)T * p.xwin_row * 2;
    const size_t a_h = (size_t)p.win_entries * 2 * p.hwin_row * 2;
    const size_t szA = align_up(a_x > a_h ? a_x : a_h, 16);
    p.off_hundo = szA;
    const size_t sz_hundo = align_up((size_t)p.win_entries * sizeof(float), 16);
    p.off_b = p.off_hundo + sz_hundo;
    const int Ep = (E + 31) / 32 * 32;
    const size_t b_logits = (size_t)T * Ep * sizeof(unsigned long long) +
                            (size_t)T * (Ep / 32) * k * (sizeof(unsigned long long) + sizeof(int));
    const int TT = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    const size_t b_router = (size_t)p.r_rows * 128 + align_up((size_t)TT * p.r_rows * 4, 16) +
                            (size_t)kFusedWarps * T * 32 * sizeof(float2);
    const size_t b_slots = (size_t)2 * kFusedWarps * 32 * 4 * sizeof(float) + (size_t)(nu_dn + 1) * sizeof(int);
    size_t szB = b_logits;
    if (b_slots > szB)
        szB = b_slots;
    p.smem = p.off_b + align_up(szB, 16);
    if (b_router > p.smem)                  // the router phase runs first and may use all of it
        p.smem = align_up(b_router, 16);
    p.ok = p.smem <= kFusedSmemBudget;
    return p;
}

template <bool FULL, bool ROUTE_ONLY>
static cudaError_t launch_fused_t(const FusedArgs &args, int grid, size_t smem, cudaStream_t stream) {
    static std::atomic<int> set_bytes[64];
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    if (set_bytes[dev & 63].load() < (int)smem) {
        err = cudaFuncSetAttribute(fused_layer_kernel<FULL, ROUTE_ONLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem);
        if (err != cudaSuccess)
            return err;
        set_bytes[dev & 63].store((int)smem);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fused_layer_kernel<FULL, ROUTE_ONLY>, args);
}

cudaError_t launch_fused(const FusedProblem &pr, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                         const GroupOut *route_only) {
    const moe_mxfp4_bank_t &b = *pr.bank;
    const int H = b.hidden, I = b.inter, E = b.num_experts, S = b.has_shared;
    const FusedPlan plan = fused_plan(pr.T, H, I, E, pr.top_k, S, num_sms);
    if (!plan.ok)
        return cudaErrorInvalidValue;
    const PackedLayout PL = packed_layout(H, I, E + S);
    FusedArgs a{};
    a.x = pr.x;
    a.wr = pr.router_w;
    a.bias = pr.bias;
    a.gu = b.packed ? b.packed + PL.gu_offset : nullptr;     // routing only: no expert weights are read
    a.dn = b.packed ? b.packed + PL.dn_offset : nullptr;
    a.y = pr.y;
    a.ids_out = pr.ids_out;
    a.w_out = pr.w_out;
    a.hdr = ws_at<uint32_t>(ws, 0);
    a.rpart = ws_at<float2>(ws, L.fz_rpart);
    a.cstamps = ws_at<unsigned long long>(ws, kCtaStampOffset);
    a.h32 = ws_at<float>(ws, L.fz_h32);
    a.yent = ws_at<float>(ws, L.fz_yent);
    a.T = pr.T;
    a.H = H;
    a.E = E;
    a.k = pr.top_k;
    a.S = S;
    a.I = I;
    a.shared_weight = pr.shared_weight;
    a.r_groups = plan.r_groups;
    a.r_chunks = plan.r_chunks;
    a.r_rows = plan.r_rows;
    a.r_final = plan.r_final ? 1 : 0;
    a.r_vec = (E % 4 == 0 && (reinterpret_cast<uintptr_t>(pr.router_w) & 15) == 0) ? 1 : 0;
    a.gu_unit = (unsigned)PL.gu_unit_bytes;
    a.dn_unit = (unsigned)PL.dn_unit_bytes;
    a.xwin_row = plan.xwin_row;
    a.hwin_row = plan.hwin_row;
    a.win_entries = plan.win_entries;
    a.off_hundo = (int)plan.off_hundo;
    a.off_b = (int)plan.off_b;
    a.next_pf[0] = static_cast<const uint8_t *>(pr.next_router);
    a.next_pf_bytes[0] = pr.next_router_bytes;
    a.next_pf[1] = static_cast<const uint8_t *>(pr.next_shared_gu);
    a.next_pf_bytes[1] = pr.next_shared_gu_bytes;
    a.next_pf[2] = static_cast<const uint8_t *>(pr.next_shared_dn);
    a.next_pf_bytes[2] = pr.next_shared_dn_bytes;
    a.x_sorted_tok = ws_at<int32_t>(ws, L.sorted_tok);
    a.x_sorted_slot = ws_at<int32_t>(ws, L.sorted_slot);
    a.x_inv_pos = ws_at<int32_t>(ws, L.inv_pos);
    a.x_offsets = ws_at<int32_t>(ws, L.offsets);
    a.x_active = ws_at<int32_t>(ws, L.active);
    if (route_only) {
        a.x_passes = route_only->passesw4;
        a.x_q = pr.mx_xq;
        a.x_qs = pr.mx_xs;
        return launch_fused_t<false, true>(a, num_sms, plan.smem, stream);
    }
    if (!b.packed)
        return cudaErrorInvalidValue;
    if (H % (64 * SB) == 0 && I % (64 * SB) == 0)
        return launch_fused_t<true, false>(a, num_sms, plan.smem, stream);
    return launch_fused_t<false, false>(a, num_sms, plan.smem, stream);
}

}  // namespace moe
