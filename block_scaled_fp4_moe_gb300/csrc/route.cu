// route.cu -- router logits, top-k selection with the fused shared slot, and
// token-to-expert grouping (sm_103a).
//
// Router logits l[t,e] = sum_h x[t,h] Wr[h,e] + b[e] decide which experts a
// token visits, so the kernels evaluate them with error-free transformations:
// each product is split exactly into p + e with one FMA, and the running sum
// is kept as an unevaluated pair (Dot2 of Ogita, Rump and Oishi, "Accurate sum
// and dot product", SIAM J. Sci. Comput. 26(6), 2005).  The result carries
// about twice fp32 precision, so the chosen experts and their order match the
// exact logits except for near-ties far below anything the workloads produce.
//
// Top-k semantics: the k largest logits (equal logits: the lower expert index
// first), ordered by descending logit; softmax over the k kept logits; the
// shared expert, always selected, appended as slot k ("Optimizing GLM4-MoE for
// production", section 1 "Shared experts fusion": top-9 of 161, the shared
// expert always in the 9th position).
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ------------------------------------------------------------ router GEMV

// Grid (ceil(E/32), ceil(H/512), ceil(T/8)); CTA (bx, by, bz) owns experts
// [32bx, 32bx+32) (one per lane), router rows [512by, 512by+512) (64 per
// warp, summed in four interleaved Dot2 chains for instruction-level
// parallelism) and tokens [8bz, 8bz+8), and writes the partial pairs
// part[by][t][e].  The router weights do
// not depend on earlier kernels, so they are loaded before the wait on the
// preceding grid.
__global__ void __launch_bounds__(kRouteThreads)
route_partial_kernel(const uint16_t *__restrict__ x, const float *__restrict__ wr, int T, int H, int E,
                     float2 *__restrict__ part, uint32_t *__restrict__ hdr) {
    constexpr int kWarps = kRouteThreads / 32;
    constexpr int kRowsPerWarp = kRouteRows / kWarps;
    constexpr int kTok = 8;
    __shared__ float xs[kTok][kRouteRows];
    __shared__ float2 red[kWarps][kTok][32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kRouteCols + lane;
    const int h0 = blockIdx.y * kRouteRows;
    const int hw = h0 + warp * kRowsPerWarp;

    float w[kRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) {
        const int h = hw + i;
        w[i] = (e < E && h < H) ? __ldg(wr + (size_t)h * E + e) : 0.0f;
    }
    pdl_wait();
    pdl_trigger();
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        hdr[kHdrRouteTicket] = 0;

    for (int t0 = blockIdx.z * kTok; t0 < T && t0 < (int)(blockIdx.z + 1) * kTok; t0 += kTok) {
        const int tn = min(kTok, T - t0);
        __syncthreads();
        // tn tokens x 512 rows of bf16 in chunks of 8 elements, two per thread
#pragma unroll
        for (int i = threadIdx.x; i < kTok * kRouteRows / 8; i += kRouteThreads) {
            const int tt = i / (kRouteRows / 8), h8 = (i % (kRouteRows / 8)) * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tt < tn && h0 + h8 < H)      // H % 8 == 0: a chunk is either inside or outside
                v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(t0 + tt) * H + h0 + h8));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xs[tt][h8 + 2 * j] = __uint_as_float(w4[j] << 16);
                xs[tt][h8 + 2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
            }
        }
        __syncthreads();
        for (int tt = 0; tt < tn; ++tt) {
            const float *xr = &xs[tt][warp * kRowsPerWarp];
            float p[4], q4[4];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                two_prod(xr[c], w[c], p[c], q4[c]);
#pragma unroll
            for (int i = 4; i < kRowsPerWarp; i += 4) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float hp, r, q;
                    two_prod(xr[i + c], w[i + c], hp, r);
                    two_sum(p[c], hp, p[c], q);
                    q4[c] = __fadd_rn(q4[c], __fadd_rn(q, r));
                }
            }
            pair_add(p[0], q4[0], p[1], q4[1]);
            pair_add(p[2], q4[2], p[3], q4[3]);
            pair_add(p[0], q4[0], p[2], q4[2]);
            red[warp][tt][lane] = make_float2(p[0], q4[0]);
        }
        __syncthreads();
        const int tt = warp;   // one warp per token of the chunk
        if (tt < tn && e < E) {
            float p = red[0][tt][lane].x, q = red[0][tt][lane].y;
#pragma unroll
            for (int w2 = 1; w2 < kWarps; ++w2)
                pair_add(p, q, red[w2][tt][lane].x, red[w2][tt][lane].y);
            part[((size_t)blockIdx.y * T + t0 + tt) * E + e] = make_float2(p, q);
        }
    }
}

// ------------------------------------------------------------------ grouping

// Grouping of ids [T*kps] (entry i = t*kps + s) by one CTA of kGroupThreads:
// per-expert counts, exclusive offsets, the stable scatter of entries sorted
// by (expert, entry), the ascending list of active experts, the passes (runs
// of up to kPassTokens entries of one expert) and the reset of the down-kernel
// row-block counters.
__device__ void group_block(const int32_t *ids, int T, int kps, int n_tot, const GroupOut &o, uint32_t *hdr,
                            bool ids_in_smem = false) {
    __shared__ int cnt[kMaxExperts];
    __shared__ int cursor[kMaxExperts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = T * kps;

    for (int e = tid; e < n_tot; e += blockDim.x)
        cnt[e] = 0;
    for (int i = tid; i < o.n_counters; i += blockDim.x)
        o.counters[i] = 0;
    __syncthreads();
    int bad = 0;
    auto id_at = [&](int i) { return ids_in_smem ? ids[i] : __ldcg(ids + i); };
    for (int i = tid; i < n; i += blockDim.x) {
        const int e = id_at(i);
        if (e < 0 || e >= n_tot)
            bad = 1;
        else
            atomicAdd(&cnt[e], 1);
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (tid == 0) {
            record_status(hdr, MOE_ERR_DEVICE_ASSERT);
            hdr[kHdrNumActive] = 0;
            hdr[kHdrNumPasses] = 0;
            hdr[kHdrNumPasses4] = 0;
            hdr[kHdrNumPassesW] = 0;
            hdr[kHdrNumPassesW4] = 0;
            if (o.num_active)
                *o.num_active = 0;
        }
        return;
    }

    if (warp == 0) {
        // pass lists: caps kPassTokens (gate/up), kPassEntries (down) and the
        // wide caps of the tiled kernels
        constexpr int NL = 4;
        const int caps[NL] = {kPassTokens, kPassEntries, kWidePassTokens, kWidePassEntries};
        Pass *const lists[NL] = {o.passes, o.passes4, o.passesw, o.passesw4};
        int run = 0, na = 0;
        int np[NL] = {0, 0, 0, 0};
        for (int base = 0; base < n_tot; base += 32) {
            const int e = base + lane;
            const int v = e < n_tot ? cnt[e] : 0;
            int incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d)
                    incl += y;
            }
            const int excl = run + incl - v;
            const unsigned act = __ballot_sync(0xffffffffu, v > 0);
            const int rank = __popc(act & ((1u << lane) - 1u));
            if (e < n_tot) {
                cursor[e] = excl;
                o.offsets[e] = excl;
                if (v > 0)
                    o.active[na + rank] = e;
            }
#pragma unroll
            for (int li = 0; li < NL; ++li) {
                const int npass = (v + caps[li] - 1) / caps[li];
                int pincl = npass;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, pincl, d);
                    if (lane >= d)
                        pincl += y;
                }
                const int pexcl = np[li] + pincl - npass;
                if (o.passes && e < n_tot)
                    for (int p = 0; p < npass; ++p)
                        lists[li][pexcl + p] = Pass{e, excl + p * caps[li], min(caps[li], v - p * caps[li]), 0};
                np[li] += __shfl_sync(0xffffffffu, pincl, 31);
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            na += __popc(act);
        }
        if (lane == 0) {
            o.offsets[n_tot] = run;
            hdr[kHdrNumActive] = na;
            hdr[kHdrNumPasses] = np[0];
            hdr[kHdrNumPasses4] = np[1];
            hdr[kHdrNumPassesW] = np[2];
            hdr[kHdrNumPassesW4] = np[3];
            if (o.num_active)
                *o.num_active = na;
        }
        __syncwarp();
        // stable scatter in entry order, 32 entries at a time
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            const int e = i < n ? id_at(i) : -1;
            const unsigned same = __match_any_sync(0xffffffffu, e);
            if (i < n) {
                const int pos = cursor[e] + __popc(same & ((1u << lane) - 1u));
                if (MOE_DBG_IN_RANGE(pos, n, hdr)) {
                    o.sorted_tok[pos] = i / kps;
                    o.sorted_slot[pos] = i % kps;
                    if (o.inv_pos)
                        o.inv_pos[i] = pos;
                }
            }
            __syncwarp();
            if (i < n && lane == 31 - __clz(same))
                cursor[e] += __popc(same);
            __syncwarp();
        }
    }
}

__global__ void __launch_bounds__(kGroupThreads)
group_kernel(const int32_t *ids, int T, int kps, int n_tot, GroupOut o, uint32_t *hdr) {
    pdl_wait();
    pdl_trigger();
    group_block(ids, T, kps, n_tot, o, hdr);
}

// ------------------------------------------------------- top-k + shared slot

// Entries the grouping CTA copies into shared memory (32 KB: with the static
// arrays this stays under the 48 KB that need no opt-in).
constexpr int kGroupSmemIds = 8 * 1024;

// One CTA per token.  All threads sum the partial pairs of the experts in a
// fixed order (the loads of one expert issued together) and add the bias;
// then warp 0 selects the top k (warp-wide argmax over (hi, lo, -index)) and
// writes ids, softmax weights and the shared slot while, with do_group, warps
// 1..7 write the f16 copy of the token's x.  With do_group the last CTA to
// finish (atomic ticket; the only CTA when T = 1) groups all tokens.
__global__ void __launch_bounds__(256)
route_finish_kernel(const float2 *__restrict__ part, int nh, const float *__restrict__ bias, int T, int E, int k,
                    int has_shared, float shared_weight, int32_t *__restrict__ ids_out, float *__restrict__ w_out,
                    uint32_t *__restrict__ hdr, int do_group, GroupOut go, const uint16_t *__restrict__ x, int H,
                    __half *x16, float *xundo) {
    extern __shared__ float2 L[];   // [E] normalised (hi, lo) logits
    __shared__ int last_cta;
    __shared__ int sids[kMaxSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int kps = k + has_shared;
    pdl_wait();
    pdl_trigger();

    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float p = 0.0f, s = 0.0f;
        float2 v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)             // issue the loads of all chunks first
            if (c < nh)
                v[c] = part[((size_t)c * T + t) * E + e];
        const float b = bias ? bias[e] : 0.0f;
#pragma unroll
        for (int c = 0; c < 16; ++c)
            if (c < nh)
                pair_add(p, s, v[c].x, v[c].y);
        for (int c = 16; c < nh; ++c) {          // H > 8192
            const float2 u = part[((size_t)c * T + t) * E + e];
            pair_add(p, s, u.x, u.y);
        }
        pair_add(p, s, b, 0.0f);
        float hi, lo;
        two_sum(p, s, hi, lo);
        L[e] = make_float2(hi, lo);
    }
    __syncthreads();

    if (warp == 0) {
        const int per_lane = (E + 31) / 32;   // <= 32 (E <= 1024)
        unsigned taken = 0;
        float sel_num = 0.0f, top_hi = 0.0f, top_lo = 0.0f, denom = 0.0f;
        int sel_id = 0;
        for (int r = 0; r < k; ++r) {
            float bh = -INFINITY, bl = -INFINITY;
            int bi = 0x7fffffff;
            for (int j = 0; j < per_lane; ++j) {
                const int e = lane + 32 * j;
                if (e >= E || ((taken >> j) & 1u))
                    continue;
                const float2 v = L[e];
                if (v.x > bh || (v.x == bh && (v.y > bl || (v.y == bl && e < bi)))) {
                    bh = v.x;
                    bl = v.y;
                    bi = e;
                }
            }
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) {
                const float oh = __shfl_xor_sync(0xffffffffu, bh, d);
                const float ol = __shfl_xor_sync(0xffffffffu, bl, d);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, d);
                if (oh > bh || (oh == bh && (ol > bl || (ol == bl && oi < bi)))) {
                    bh = oh;
                    bl = ol;
                    bi = oi;
                }
            }
            if (bi < E && (bi & 31) == lane)
                taken |= 1u << (bi >> 5);
            if (r == 0) {
                top_hi = bh;
                top_lo = bl;
            }
            // softmax numerator relative to the largest logit
            const float dlt = __fadd_rn(__fsub_rn(bh, top_hi), __fsub_rn(bl, top_lo));
            const float ex = expf(dlt);
            denom += ex;
            if (lane == r) {
                sel_num = ex;
                sel_id = bi;
            }
        }
        if (lane < k) {
            ids_out[(size_t)t * kps + lane] = sel_id;
            w_out[(size_t)t * kps + lane] = sel_num / denom;
            sids[lane] = sel_id;
        }
        if (has_shared && lane == k) {
            ids_out[(size_t)t * kps + k] = E;
            w_out[(size_t)t * kps + k] = shared_weight;
            sids[k] = E;
        }
    } else if (do_group && x16) {
        convert_x_row(x, t, H, x16, xundo, 1, 7, 1);
    }
    if (!do_group)
        return;
    __syncthreads();
    if (gridDim.x == 1) {                        // a single token: group from shared memory
        group_block(sids, T, kps, E + has_shared, go, hdr, true);
        return;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(hdr + kHdrRouteTicket, 1u);
        last_cta = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last_cta)
        return;
    __threadfence();
    const int n = T * kps;
    if (n <= kGroupSmemIds) {
        // every token's ids into shared memory first: the grouping then reads
        // them without a global round trip per step
        int *sm_ids = reinterpret_cast<int *>(L);
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            sm_ids[i] = __ldcg(ids_out + i);
        __syncthreads();
        group_block(sm_ids, T, kps, E + has_shared, go, hdr, true);
    } else {
        group_block(ids_out, T, kps, E + has_shared, go, hdr);
    }
    if (threadIdx.x == 0)
        hdr[kHdrRouteTicket] = 0;
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_route(const uint16_t *x, const float *wr, const float *bias, int T, int H, int E, int k,
                         int has_shared, float shared_weight, int32_t *ids, float *w, void *ws,
                         const WsLayout &L, bool do_group, const GroupOut &go, cudaStream_t stream,
                         cudaEvent_t ev_after_partial) {
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    float2 *part = ws_at<float2>(ws, L.route_part);
    const int nh = (H + kRouteRows - 1) / kRouteRows;
    dim3 g1((E + kRouteCols - 1) / kRouteCols, nh, (T + 7) / 8);   // one CTA per 8 tokens of a tile
    cudaError_t err = launch_pdl(route_partial_kernel, g1, dim3(kRouteThreads), 0, stream, x, wr, T, H, E, part, hdr);
    if (err != cudaSuccess)
        return err;
    if (ev_after_partial &&
        (err = cudaEventRecord(ev_after_partial, stream)) != cudaSuccess)
        return err;
    const size_t n_ids = (size_t)T * (k + has_shared);
    size_t smem = (size_t)E * sizeof(float2);
    if (do_group && T > 1 && n_ids <= (size_t)kGroupSmemIds && n_ids * sizeof(int) > smem)
        smem = n_ids * sizeof(int);
    __half *x16 = do_group ? ws_at<__half>(ws, L.x16) : nullptr;
    float *xundo = do_group ? ws_at<float>(ws, L.xundo) : nullptr;
    return launch_pdl(route_finish_kernel, dim3(T), dim3(256), smem, stream, part, nh, bias, T, E, k, has_shared,
                      shared_weight, ids, w, hdr, do_group ? 1 : 0, go, x, H, x16, xundo);
}

cudaError_t launch_group(const int32_t *ids, int T, int kps, int n_tot, const GroupOut &go, uint32_t *hdr,
                         cudaStream_t stream) {
    return launch_pdl(group_kernel, dim3(1), dim3(kGroupThreads), 0, stream, ids, T, kps, n_tot, go, hdr);
}

}  // namespace moe
