// kernels.h -- launch functions of the MoE kernels (internal to the library).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moe {

// Where grouping writes its results (device pointers; nullable where noted).
struct GroupOut {
    int32_t *offsets;      // [n_tot + 1]
    int32_t *sorted_tok;   // [T*kps]
    int32_t *sorted_slot;  // [T*kps]
    int32_t *inv_pos;      // [T*kps] nullable: sorted position of entry t*kps+s
    int32_t *active;       // [n_tot]
    int32_t *num_active;   // [1] nullable (the header always gets it)
    Pass *passes;          // nullable: passes of <= 8 entries (gate/up)
    Pass *passes4;         // with passes: passes of <= 4 entries (down)
    Pass *passesw;         // with passes: wide passes of <= kWidePassTokens (tiled gate/up)
    Pass *passesw4;        // with passes: wide passes of <= kWidePassEntries (tiled down)
    uint32_t *counters;    // down-kernel row-block counters to zero
    int n_counters;
};

// Launch with programmatic stream serialization, so the kernel can be
// scheduled while its predecessor on the stream is still running; the kernel
// itself waits (pdl_wait) before it reads anything the predecessor writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// static shared memory of the grouping code (two int arrays of kMaxExperts)
constexpr size_t kGroupStaticSmem = 2 * kMaxExperts * sizeof(int) + 64;

// Router logits + top-k (+ grouping and the f16 copy of x when do_group).
cudaError_t launch_route(const uint16_t *x, const float *wr, const float *bias, int T, int H, int E, int k,
                         int has_shared, float shared_weight, int32_t *ids, float *w, void *ws,
                         const WsLayout &L, bool do_group, const GroupOut &go, cudaStream_t stream,
                         cudaEvent_t ev_after_partial = nullptr);

cudaError_t launch_group(const int32_t *ids, int T, int kps, int n_tot, const GroupOut &go, uint32_t *hdr,
                         cudaStream_t stream);

// Expert FFN: gate/up + SiLU*up (writes h), then down + weighted combine
// (writes y).  Grouping results must already be in the workspace.
struct FfnProblem {
    const uint16_t *x;       // [T, H] bf16
    const moe_mxfp4_bank_t *bank;
    const float *topk_w;     // [T, kps]
    uint16_t *y;             // [T, H] bf16
    int T, kps;
};

cudaError_t launch_ffn(const FfnProblem &p, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                       cudaEvent_t ev_after_gateup);
// y = bf16(sum over slots of w * Y), Y [entries][H] in sorted entry order.
cudaError_t launch_combine(const float *yent, int entries, const int32_t *inv_pos, const float *topk_w, int T, int kps,
                           int H, uint16_t *y, const uint32_t *hdr, cudaStream_t stream);

// MXFP8 live-activation-quantisation variant (mx8.cu): after routing and
// grouping, x and h are quantised to MXFP8 and both projections run as
// block-scaled tcgen05 MMAs on the canonical bank arrays.
struct Mx8Problem {
    const uint16_t *x;       // [T, H] bf16
    const moe_mxfp4_bank_t *bank;
    const uint8_t *packed_mx;   // the variant's bank (launch_mx8_pack)
    const float *topk_w;     // [T, kps]
    uint16_t *y;             // [T, H] bf16
    int T, kps;
    bool x_quantised;        // x's MXFP8 codes are already in the workspace
};
bool mx8_shape_supported(int H, int I);
size_t mx8_packed_size(int H, int I, int n_tot);
cudaError_t launch_mx8_pack(const moe_mxfp4_bank_t &b, uint8_t *out, cudaStream_t stream);
// ev (nullable): two events, recorded after the x quantisation and after the gate/up GEMM.
cudaError_t launch_mx8_ffn(const Mx8Problem &p, void *ws, const WsLayout &L, cudaStream_t stream,
                           cudaEvent_t *ev = nullptr);

// f16 copy of x with per-token power-of-two scaling (x16, xundo regions).
cudaError_t launch_x16(const uint16_t *x, int T, int H, void *ws, const WsLayout &L, cudaStream_t stream);

// The whole layer in one cooperative launch for T <= kFusedMaxTokens (fused.cu).
struct FusedProblem {
    const uint16_t *x;
    const float *router_w;
    const float *bias;
    const moe_mxfp4_bank_t *bank;
    float shared_weight;
    uint16_t *y;
    int32_t *ids_out;        // nullable
    float *w_out;            // nullable
    int T, top_k;
    // L2 prefetch hint for the next layer (nullable; sizes in bytes)
    const void *next_router;
    size_t next_router_bytes;
    const void *next_shared_gu, *next_shared_dn;
    size_t next_shared_gu_bytes, next_shared_dn_bytes;
    // routing only (launch_fused with route_only), nullable: x as MXFP8
    uint8_t *mx_xq = nullptr, *mx_xs = nullptr;
};

// Shared-memory plan of the single-launch kernel; ok = the shape fits.
struct FusedPlan {
    bool ok;
    int r_groups, r_chunks, r_rows;
    bool r_final;
    int xwin_row, hwin_row, win_entries;
    size_t off_hundo, off_b, smem;
};
FusedPlan fused_plan(int T, int H, int I, int E, int k, int S, int grid);
// route_only (nullable): run only the routing phases and write the grouping
// (passes of one expert's entries into route_only->passesw4, the sorted order
// and its inverse, the pass count in the header) instead of the whole layer.
cudaError_t launch_fused(const FusedProblem &p, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                         const GroupOut *route_only = nullptr);
cudaError_t launch_wait_selftest(uint32_t *hdr, cudaStream_t stream);

// Byte offsets inside a repacked bank (pack.cu).
struct PackedLayout {
    size_t gu_unit_bytes, dn_unit_bytes, gu_offset, dn_offset, gu_rowexp, dn_rowexp, total;
    int gu_units_per_expert, dn_units_per_expert;
};
PackedLayout packed_layout(int H, int I, int n_experts_total);
cudaError_t launch_pack(const moe_mxfp4_bank_t &b, uint8_t *out, cudaStream_t stream);

cudaError_t launch_selftest_decode(const uint8_t *codes, uint16_t *out, int n, cudaStream_t stream);

// Shape rules shared by validation and the kernels' staging choices.
bool ffn_shape_supported(int H, int I);

// A tiled tensor map (tc.cu): dims / strides / box innermost first, strides
// in bytes (rank - 1 of them); the driver's encoder is looked up at run time.
cudaError_t encode_tiled(CUtensorMap *m, CUtensorMapDataType type, int rank, const void *base, const uint64_t *dims,
                         const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle);

// Tensor-memory expert FFN for T > 8 (tc.cu): H and I multiples of 512.
bool tc_shape_supported(int H, int I);
// Exponent base per weight row into the packed bank's two row sections.
cudaError_t launch_rowexp(const moe_mxfp4_bank_t &b, uint8_t *packed, cudaStream_t stream);
// x gathered per sorted entry, the tensor-core gate/up, h finalisation, the
// tensor-core down and the combine.  Grouping results (passes of <= 32
// tokens and <= 16 entries) and x16 must already be in the workspace.
cudaError_t launch_ffn_tc(const FfnProblem &p, void *ws, const WsLayout &L, int num_sms, cudaStream_t stream,
                          cudaEvent_t ev_after_gateup);
// h = silu(g) u from the gate/up sums (one K chunk) into h16 (hi, lo) and
// hundo; tc_order: each 64-element step of h16 in the tensor-memory K order.
cudaError_t launch_hfin(void *ws, const WsLayout &L, int T, int entries, int I, bool tc_order, cudaStream_t stream);

}  // namespace moe
