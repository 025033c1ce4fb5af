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
// expert always in the 9th position).  For T > 8 the selection is the one the
// single-launch kernel uses: each group of 32 experts keeps its first k ranks
// as a sorted candidate list, and one warp merges the lists.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// ------------------------------------------------------------ router GEMV

// Grid (ceil(E/32), ceil(H/512), ceil(T/TOK)); CTA (bx, by, bz) owns experts
// [32bx, 32bx+32) (one per lane), router rows [512by, 512by+512) (64 per
// warp, summed in four interleaved Dot2 chains for instruction-level
// parallelism) and tokens [TOK bz, TOK bz + TOK), and writes the partial pairs
// part[by][t][e].  TOK (2, 4 or 8) only spreads the tokens over more CTAs at
// small T: each token's sums are the same for every TOK.  The router weights
// do not depend on earlier kernels, so they are loaded before the wait on
// the preceding grid.
template <int TOK>
__global__ void __launch_bounds__(kRouteThreads)
route_partial_kernel(const uint16_t *__restrict__ x, const float *__restrict__ wr, int T, int H, int E,
                     float2 *__restrict__ part, uint32_t *__restrict__ hdr) {
    constexpr int kWarps = kRouteThreads / 32;
    constexpr int kRowsPerWarp = kRouteRows / kWarps;
    constexpr int kTok = TOK;
    static_assert(kTok <= kWarps, "one warp per token of the chunk");
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

// Grouping of ids [T*kps] (entry i = t*kps + s) by one CTA of kGroupThreads
// (8 warps): per-expert counts, exclusive offsets, the stable scatter of
// entries sorted by (expert, entry), the ascending list of active experts, the
// pass lists (runs of up to kPassTokens, kPassEntries, kWidePassTokens and
// kWidePassEntries entries of one expert) and the reset of the down-kernel
// row-block counters.  A counting sort done by the whole CTA: the entries are
// cut into 8 contiguous segments, one per warp; each warp counts its segment
// per expert; one block-wide scan gives the offsets, the active list and the
// four pass lists; a warp's cursor for expert e starts at the offset of e plus
// the counts of e in the earlier segments, so the warps scatter their
// segments concurrently and the order stays the entry order.  Past
// kGroupParExperts experts the per-warp counts do not fit and one warp
// scatters all entries in order.
constexpr int kGroupParExperts = 512;

__device__ void group_block(const int32_t *ids, int T, int kps, int n_tot, const GroupOut &o, uint32_t *hdr,
                            bool ids_in_smem = false) {
    constexpr int kW = kGroupThreads / 32;
    __shared__ int cnt[kMaxExperts];
    __shared__ int wbase[kW][kGroupParExperts];       // per-warp counts, then per-warp cursors
    constexpr int kScanPerLane = kGroupThreads / 32;
    __shared__ int sscan[6][kGroupThreads];          // per-thread values, then their exclusive scans
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = T * kps;
    const bool par = n_tot <= kGroupParExperts;
    const int seg = (n + kW - 1) / kW;                 // entries of a warp's segment

    for (int e = tid; e < n_tot; e += blockDim.x)
        cnt[e] = 0;
    if (par)
        for (int i = tid; i < kW * n_tot; i += blockDim.x)
            wbase[i / n_tot][i % n_tot] = 0;
    for (int i = tid; i < o.n_counters; i += blockDim.x)
        o.counters[i] = 0;
    __syncthreads();
    int bad = 0;
    auto id_at = [&](int i) { return ids_in_smem ? ids[i] : __ldcg(ids + i); };
    // counts, 32 entries at a time, one update per distinct expert (its
    // lowest lane adds the group's size): into the warp's own row (no other
    // warp writes it; the rows are added per expert below), or with one
    // shared-memory atomic per group when the experts are too many for rows
    {
        const int i1 = min(n, (warp + 1) * seg);
        for (int base = warp * seg; base < i1; base += 32) {
            const int i = base + lane;
            int e = i < i1 ? id_at(i) : -1;
            if (i < i1 && (e < 0 || e >= n_tot)) {
                bad = 1;
                e = -1;
            }
            const unsigned same = __match_any_sync(0xffffffffu, e);
            if (e >= 0 && lane == __ffs(same) - 1) {
                if (par)
                    wbase[warp][e] += __popc(same);
                else
                    atomicAdd(&cnt[e], __popc(same));
            }
        }
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

    // block-wide exclusive scan of (count, active, passes of the four caps):
    // thread tid owns experts [per tid, per tid + per)
    const int caps[4] = {kPassTokens, kPassEntries, kWidePassTokens, kWidePassEntries};
    Pass *const lists[4] = {o.passes, o.passes4, o.passesw, o.passesw4};
    const int per = (n_tot + kGroupThreads - 1) / kGroupThreads;
    const int e0 = tid * per, e1 = min(n_tot, e0 + per);
    int loc[6] = {0, 0, 0, 0, 0, 0};
    for (int e = e0; e < e1; ++e) {
        int v = cnt[e];
        if (par) {
#pragma unroll
            for (int w2 = 0; w2 < kW; ++w2)
                v += wbase[w2][e];
            cnt[e] = v;                                // only this thread reads it again
        }
        loc[0] += v;
        loc[1] += v > 0;
#pragma unroll
        for (int l = 0; l < 4; ++l)
            loc[2 + l] += (v + caps[l] - 1) / caps[l];
    }
    // the six exclusive scans, one warp each over the threads' values (8
    // per lane, in loops: this runs once per call on one CTA, where compact
    // code matters more than unrolling)
#pragma unroll
    for (int q = 0; q < 6; ++q)
        sscan[q][tid] = loc[q];
    __syncthreads();
    if (warp < 6) {
        int *row = sscan[warp] + kScanPerLane * lane;
        int run = 0;
#pragma unroll 1
        for (int j = 0; j < kScanPerLane; ++j)
            run += row[j];
        int inc = run;
#pragma unroll 1
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, inc, d);
            if (lane >= d)
                inc += y;
        }
        int ex = inc - run;
#pragma unroll 1
        for (int j = 0; j < kScanPerLane; ++j) {
            const int v = row[j];
            row[j] = ex;
            ex += v;
        }
    }
    __syncthreads();
    int ex[6];
#pragma unroll
    for (int q = 0; q < 6; ++q)
        ex[q] = sscan[q][tid];
    for (int e = e0; e < e1; ++e) {
        const int v = cnt[e];
        o.offsets[e] = ex[0];
        cnt[e] = ex[0];                                // the offset, for the cursors below
        if (v > 0)
            o.active[ex[1]++] = e;
#pragma unroll
        for (int l = 0; l < 4; ++l) {
            const int np = (v + caps[l] - 1) / caps[l];
            if (o.passes)
                for (int p = 0; p < np; ++p)
                    lists[l][ex[2 + l] + p] = Pass{e, ex[0] + p * caps[l], min(caps[l], v - p * caps[l]), 0};
            ex[2 + l] += np;
        }
        ex[0] += v;
    }
    if (tid == kGroupThreads - 1) {                    // the totals
        o.offsets[n_tot] = ex[0];
        hdr[kHdrNumActive] = ex[1];
        hdr[kHdrNumPasses] = ex[2];
        hdr[kHdrNumPasses4] = ex[3];
        hdr[kHdrNumPassesW] = ex[4];
        hdr[kHdrNumPassesW4] = ex[5];
        if (o.num_active)
            *o.num_active = ex[1];
    }
    __syncthreads();                                   // offsets in cnt

    // cursors: per warp, the offset of the expert plus its counts in the
    // earlier segments
    if (par) {
        for (int e = tid; e < n_tot; e += blockDim.x) {
            int run = cnt[e];
#pragma unroll
            for (int w2 = 0; w2 < kW; ++w2) {
                const int h = wbase[w2][e];
                wbase[w2][e] = run;
                run += h;
            }
        }
        __syncthreads();
    }
    // stable scatter, 32 entries at a time: every warp its own segment, or
    // warp 0 all entries
    if (par || warp == 0) {
        int *cur = par ? wbase[warp] : cnt;
        const int i0 = par ? warp * seg : 0, i1 = par ? min(n, (warp + 1) * seg) : n;
        for (int base = i0; base < i1; base += 32) {
            const int i = base + lane;
            const int e = i < i1 ? id_at(i) : -1;
            const unsigned same = __match_any_sync(0xffffffffu, e);
            if (i < i1) {
                const int pos = cur[e] + __popc(same & ((1u << lane) - 1u));
                if (MOE_DBG_IN_RANGE(pos, n, hdr)) {
                    o.sorted_tok[pos] = i / kps;
                    o.sorted_slot[pos] = i % kps;
                    if (o.inv_pos)
                        o.inv_pos[i] = pos;
                }
            }
            __syncwarp();
            if (i < i1 && lane == 31 - __clz(same))
                cur[e] += __popc(same);
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

// Entries the grouping CTA copies into shared memory (16 KB: with the static
// arrays this stays under the 48 KB that need no opt-in).
constexpr int kGroupSmemIds = 4 * 1024;


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
    // [Ep] order keys of the logits, then the groups' candidate lists (keys,
    // then expert ids); later the grouping's ids
    extern __shared__ unsigned long long rkey[];
    __shared__ int last_cta;
    __shared__ int sids[kMaxSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x;
    const int kps = k + has_shared;
    const int Ep = (E + 31) & ~31, G = Ep >> 5;        // experts padded to whole groups of 32
    unsigned long long *ckey = rkey + Ep;               // [G][k]
    int *cand = reinterpret_cast<int *>(ckey + (size_t)G * k);
    pdl_wait();
    pdl_trigger();

    for (int e = threadIdx.x; e < Ep; e += blockDim.x) {
        if (e >= E) {
            rkey[e] = 0ull;                               // padding: below every real key
            continue;
        }
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
        if (hi != hi)                            // a NaN logit counts as -inf
            hi = lo = -INFINITY;
        rkey[e] = logit_order_key(hi, lo);
    }
    __syncthreads();

    // Top k in the order (logit pair descending, equal pairs: the lower index
    // first).  Stage 1: an expert ranked k or lower inside its group of 32
    // cannot be in the top k, so each group's first k ranks form its sorted
    // candidate list.  Ranks come from the keys' high words (two keys per
    // 16-byte load); a key whose high word another key shares is ranked by
    // the full keys and the index rule.
    for (int e = threadIdx.x; e < Ep; e += blockDim.x) {
        const unsigned long long *g = rkey + (e & ~31);
        const unsigned long long my = g[e & 31];
        const uint4 *g4 = reinterpret_cast<const uint4 *>(g);
        const uint32_t myhi = (uint32_t)(my >> 32);
        int r = 0, eq = 0;
#pragma unroll 8
        for (int j2 = 0; j2 < 16; ++j2) {
            const uint4 w = g4[j2];              // key 2 j2: (x lo, y hi), key 2 j2 + 1: (z lo, w hi)
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
            ckey[(e >> 5) * k + r] = my;
            cand[(e >> 5) * k + r] = e < E ? e : 0x7fffffff;
        }
    }
    __syncthreads();
    // Stage 2, warp 0: lane g holds the head of group g's list; each round
    // takes the largest head (key, then the lower index) and that lane moves
    // to its next entry, so slot r gets the r-th largest logit.  The softmax
    // over the kept logits is taken relative to the largest, its denominator
    // summed in slot order.
    if (warp == 0) {
        const unsigned full = 0xffffffffu;
        int pos = 0;
        unsigned long long hk = lane < G ? ckey[lane * k] : 0ull;
        unsigned he = lane < G ? (unsigned)cand[lane * k] : 0xffffffffu;
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
                hk = pos < k ? ckey[lane * k + pos] : 0ull;
                he = pos < k ? (unsigned)cand[lane * k + pos] : 0xffffffffu;
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
            ids_out[(size_t)t * kps + lane] = myid;
            w_out[(size_t)t * kps + lane] = ex / denom;
            sids[lane] = myid;
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
    // the CTA barrier orders this CTA's ids before thread 0's acquire-release
    // add (cumulative); the add that finds every other CTA counted acquires
    // their ids for the whole CTA through the barrier after it
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned ticket;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                     : "=r"(ticket)
                     : "l"(hdr + kHdrRouteTicket)
                     : "memory");
        last_cta = ticket == gridDim.x - 1;
    }
    __syncthreads();
    if (!last_cta)
        return;
    const int n = T * kps;
    if (n <= kGroupSmemIds) {
        // every token's ids into shared memory first: the grouping then reads
        // them without a global round trip per step
        int *sm_ids = reinterpret_cast<int *>(rkey);
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            sm_ids[i] = __ldcg(ids_out + i);
        __syncthreads();
        group_block(sm_ids, T, kps, E + has_shared, go, hdr, true);
        __syncthreads();
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
    // tokens per CTA: fewer at small T, so that the grid covers the SMs
    const int tok = 8;
    dim3 g1((E + kRouteCols - 1) / kRouteCols, nh, (T + tok - 1) / tok);
    cudaError_t err =
        tok == 8   ? launch_pdl(route_partial_kernel<8>, g1, dim3(kRouteThreads), 0, stream, x, wr, T, H, E, part, hdr)
        : tok == 4 ? launch_pdl(route_partial_kernel<4>, g1, dim3(kRouteThreads), 0, stream, x, wr, T, H, E, part, hdr)
                   : launch_pdl(route_partial_kernel<2>, g1, dim3(kRouteThreads), 0, stream, x, wr, T, H, E, part, hdr);
    if (err != cudaSuccess)
        return err;
    if (ev_after_partial &&
        (err = cudaEventRecord(ev_after_partial, stream)) != cudaSuccess)
        return err;
    const size_t n_ids = (size_t)T * (k + has_shared);
    const int Ep = (E + 31) & ~31;
    size_t smem = (size_t)Ep * sizeof(unsigned long long) + (size_t)(Ep / 32) * k * (sizeof(unsigned long long) + sizeof(int));
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
