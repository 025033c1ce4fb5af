// capi.cu -- the extern "C" boundary of the MoE library: argument checks,
// workspace layout and the launch sequence on the caller's stream.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

std::atomic<int> g_sms[64];

__global__ void set_word_kernel(uint32_t *p, uint32_t v) { *p = v; }

// Streaming-multiprocessor count of the current device; rejects devices the
// library was not built for.
moe_status_t current_device_sms(int *sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int cached = g_sms[dev & 63].load(std::memory_order_relaxed);
    if (cached > 0) {
        *sms = cached;
        return MOE_OK;
    }
    int major = 0, minor = 0, n = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3)
        return MOE_ERR_UNSUPPORTED_DEVICE;
    g_sms[dev & 63].store(n, std::memory_order_relaxed);
    *sms = n;
    return MOE_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_routing_shape(int T, int H, int E, int k, int S) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || (S != 0 && S != 1))
        return MOE_ERR_INVALID_ARG;
    if (T > kMaxTokens || k > E || E + S > kMaxExperts || k + S > kMaxSlots)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((long long)T * H >= (1LL << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// The kernels address activation rows with 32-bit element offsets.
moe_status_t check_ffn_extent(int T, int kps, int H, int I) {
    if ((long long)T * kps * 2 * I >= (1LL << 31) || (long long)T * kps * H >= (1LL << 31))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

moe_status_t check_bank_dims(const moe_mxfp4_bank_t *b) {
    if (!b)
        return MOE_ERR_INVALID_ARG;
    if (b->hidden <= 0 || b->inter <= 0 || b->num_experts <= 0 || (b->has_shared != 0 && b->has_shared != 1))
        return MOE_ERR_INVALID_ARG;
    if (!ffn_shape_supported(b->hidden, b->inter) || b->hidden > 65536 || b->num_experts + b->has_shared > kMaxExperts)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    return MOE_OK;
}

// The expert-FFN calls read only the repacked bank.
moe_status_t check_bank(const moe_mxfp4_bank_t *b) {
    moe_status_t st = check_bank_dims(b);
    if (st != MOE_OK)
        return st;
    if (!b->packed)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(b->packed, 16))
        return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

GroupOut group_out_for(void *ws, const WsLayout &L, int H) {
    GroupOut go{};
    go.offsets = ws_at<int32_t>(ws, L.offsets);
    go.sorted_tok = ws_at<int32_t>(ws, L.sorted_tok);
    go.sorted_slot = ws_at<int32_t>(ws, L.sorted_slot);
    go.inv_pos = ws_at<int32_t>(ws, L.inv_pos);
    go.active = ws_at<int32_t>(ws, L.active);
    go.num_active = nullptr;
    go.passes = ws_at<Pass>(ws, L.passes);
    go.passes4 = ws_at<Pass>(ws, L.passes4);
    go.passesw = ws_at<Pass>(ws, L.passesw);
    go.passesw4 = ws_at<Pass>(ws, L.passesw4);
    go.counters = ws_at<uint32_t>(ws, L.counters);
    go.n_counters = 0;
    return go;
}

// Shared body of the full-layer entry points.
moe_status_t layer_forward(const uint16_t *x, const float *router_w, const float *logit_bias, int T, int top_k,
                           const moe_mxfp4_bank_t *bank, float shared_weight, uint16_t *y, int32_t *ids_out,
                           float *w_out, void *ws, size_t ws_bytes, cudaEvent_t *ev, cudaStream_t stream,
                           const float *next_router_w = nullptr, const moe_mxfp4_bank_t *next_bank = nullptr) {
    moe_status_t st = check_bank(bank);
    if (st != MOE_OK)
        return st;
    const int H = bank->hidden, I = bank->inter, E = bank->num_experts, S = bank->has_shared;
    if ((st = check_routing_shape(T, H, E, top_k, S)) != MOE_OK ||
        (st = check_ffn_extent(T, top_k + S, H, I)) != MOE_OK)
        return st;
    if (T == 0)
        return MOE_OK;
    if (!x || !router_w || !y || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !aligned(router_w, 4) ||
        !aligned(logit_bias, 4) || !aligned(ids_out, 4) || !aligned(w_out, 4))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = WsLayout::make(T, H, I, E, top_k, S);
    if (ws_bytes < L.total)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    if (T == 0)
        return MOE_OK;
    if (T <= kFusedMaxTokens && fused_plan(T, H, I, E, top_k, S, sms).ok) {
        // decode-sized T: the whole layer in one cooperative launch
        if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess)
            return MOE_ERR_CUDA;
        FusedProblem fp{x, router_w, logit_bias, bank, shared_weight, y, ids_out, w_out, T, top_k,
                        nullptr, 0, nullptr, nullptr, 0, 0};
        if (next_bank && next_bank->hidden > 0 && next_bank->num_experts > 0 && next_bank->inter > 0) {
            const int nH = next_bank->hidden, nI = next_bank->inter, nE = next_bank->num_experts;
            if (next_router_w) {
                fp.next_router = next_router_w;
                fp.next_router_bytes = (size_t)nH * nE * sizeof(float);
            }
            if (next_bank->has_shared && next_bank->packed && nH % 64 == 0 && nI % 64 == 0) {
                const PackedLayout NL = packed_layout(nH, nI, nE + 1);
                fp.next_shared_gu = next_bank->packed + NL.gu_offset +
                                    (size_t)nE * NL.gu_units_per_expert * NL.gu_unit_bytes;
                fp.next_shared_gu_bytes = (size_t)NL.gu_units_per_expert * NL.gu_unit_bytes;
                fp.next_shared_dn = next_bank->packed + NL.dn_offset +
                                    (size_t)nE * NL.dn_units_per_expert * NL.dn_unit_bytes;
                fp.next_shared_dn_bytes = (size_t)NL.dn_units_per_expert * NL.dn_unit_bytes;
            }
        }
        const cudaError_t ferr = launch_fused(fp, ws, L, sms, stream);
        if (ferr == cudaSuccess) {
            for (int i = 1; ev && i < 5; ++i)
                if (cudaEventRecord(ev[i], stream) != cudaSuccess)
                    return MOE_ERR_CUDA;
            return MOE_OK;
        }
        // not all CTAs can be resident (e.g. a partitioned device): use the
        // multi-launch sequence below
        if (ferr != cudaErrorCooperativeLaunchTooLarge)
            return MOE_ERR_CUDA;
        (void)cudaGetLastError();
    }
    int32_t *ids = ids_out ? ids_out : ws_at<int32_t>(ws, L.topk_ids);
    float *w = w_out ? w_out : ws_at<float>(ws, L.topk_w);
    const GroupOut go = group_out_for(ws, L, H);
    if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    cudaError_t err = launch_route(x, router_w, logit_bias, T, H, E, top_k, S, shared_weight, ids, w, ws, L,
                                   true, go, stream, ev ? ev[1] : nullptr);
    if (err != cudaSuccess)
        return MOE_ERR_CUDA;
    if (ev && cudaEventRecord(ev[2], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    FfnProblem pr{x, bank, w, y, T, top_k + S};
    err = launch_ffn(pr, ws, L, sms, stream, ev ? ev[3] : nullptr);
    if (err != cudaSuccess)
        return MOE_ERR_CUDA;
    if (ev && cudaEventRecord(ev[4], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

// ------------------------------------------------------------ static scratch

// Scratch of moe_layer_forward_noalloc.  Every device that loads the library
// keeps this array until the process exits; its size bounds the problem sizes
// that entry point accepts.
constexpr size_t kStaticScratchBytes = 16u << 20;
__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::atomic<uintptr_t> g_static_addr[64];
std::mutex g_static_mu;

// Device address of the static scratch on the current device.  The first call
// on a device looks it up (the host-side name of the array is not a device
// address) and keeps it for the life of the process.  The array needs no
// clearing: a __device__ array without an initialiser is zero-filled when the
// module loads, and every call leaves the header's counters at zero again.
moe_status_t static_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dev < 0 || dev >= 64)
        return MOE_ERR_UNSUPPORTED_DEVICE;
    uintptr_t p = g_static_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        std::lock_guard<std::mutex> lock(g_static_mu);
        p = g_static_addr[dev].load(std::memory_order_acquire);
        if (!p) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr)
                return MOE_ERR_CUDA;
            p = reinterpret_cast<uintptr_t>(ptr);
            g_static_addr[dev].store(p, std::memory_order_release);
        }
    }
    *out = reinterpret_cast<void *>(p);
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_offset(int T, int H, int I, int E, int top_k, int has_shared, const char *region) {
    if (!region || T < 0 || H <= 0 || I <= 0 || E <= 0 || top_k <= 0 || (has_shared != 0 && has_shared != 1))
        return (size_t)-1;
    const WsLayout L = WsLayout::make(T, H, I, E, top_k, has_shared);
    const struct {
        const char *name;
        size_t off;
    } regions[] = {{"topk_ids", L.topk_ids}, {"topk_w", L.topk_w}, {"inv_pos", L.inv_pos},
                   {"sorted_tok", L.sorted_tok}, {"sorted_slot", L.sorted_slot}, {"offsets", L.offsets},
                   {"active", L.active}, {"num_active", kHdrNumActive * sizeof(uint32_t)},
                   {"h", T <= kFusedMaxTokens ? L.fz_h32 : (size_t)-1},
                   {"y_entries", T <= kFusedMaxTokens ? L.fz_yent : (size_t)-1},
                   {"mx_xq", L.mx_xq}, {"mx_xs", L.mx_xs},
                   {"mx_h32", L.mx_h32}, {"mx_hq", L.mx_hq}, {"mx_hs", L.mx_hs}, {"mx_y", L.mx_y}};
    for (const auto &r : regions)
        if (std::strcmp(r.name, region) == 0)
            return r.off;
    return (size_t)-1;
}

size_t moe_workspace_size(int T, int H, int I, int E, int top_k, int has_shared) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || top_k <= 0 || (has_shared != 0 && has_shared != 1))
        return 0;
    return WsLayout::make(T, H, I, E, top_k, has_shared).total;
}

size_t moe_packed_bank_size(int H, int I, int E, int has_shared) {
    if (H <= 0 || I <= 0 || E <= 0 || (has_shared != 0 && has_shared != 1) || H % 64 || I % 64)
        return 0;
    return packed_layout(H, I, E + has_shared).total;
}

moe_status_t moe_pack_bank(const moe_mxfp4_bank_t *bank, void *packed, size_t packed_bytes, cudaStream_t stream) {
    moe_status_t st = check_bank_dims(bank);
    if (st != MOE_OK)
        return st;
    if (!bank->w13 || !bank->s13 || !bank->w2 || !bank->s2 || !packed)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(bank->w13, 16) || !aligned(bank->s13, 16) || !aligned(bank->w2, 16) || !aligned(bank->s2, 16) ||
        !aligned(packed, 256))
        return MOE_ERR_MISALIGNED;
    if (packed_bytes < packed_layout(bank->hidden, bank->inter, bank->num_experts + bank->has_shared).total)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    return from_cuda(launch_pack(*bank, static_cast<uint8_t *>(packed), stream));
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < kHdrWords * sizeof(uint32_t))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes < kHeaderBytes ? ws_bytes : kHeaderBytes, stream));
}

moe_status_t moe_route_topk(const uint16_t *x, const float *router_w, const float *logit_bias, int T, int H, int E,
                            int top_k, int has_shared, float shared_weight, int32_t *topk_ids, float *topk_w,
                            void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status_t st = check_routing_shape(T, H, E, top_k, has_shared);
    if (st != MOE_OK)
        return st;
    if (T == 0)
        return MOE_OK;
    if (!x || !router_w || !topk_ids || !topk_w || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 2) || !aligned(router_w, 4) || !aligned(logit_bias, 4) || !aligned(topk_ids, 4) ||
        !aligned(topk_w, 4) || !aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = WsLayout::make(T, H, 64, E, top_k, has_shared);
    if (ws_bytes < L.topk_ids)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    if (T == 0)
        return MOE_OK;
    const GroupOut none{};
    return from_cuda(launch_route(x, router_w, logit_bias, T, H, E, top_k, has_shared, shared_weight, topk_ids,
                                  topk_w, ws, L, false, none, stream));
}

moe_status_t moe_group_tokens(const int32_t *topk_ids, int T, int k_plus_s, int n_experts_total,
                              int32_t *expert_offsets, int32_t *sorted_tok, int32_t *sorted_slot,
                              int32_t *active_experts, int32_t *num_active, void *ws, size_t ws_bytes,
                              cudaStream_t stream) {
    if (T < 0 || k_plus_s <= 0 || n_experts_total <= 0)
        return MOE_ERR_INVALID_ARG;
    if (T > kMaxTokens || k_plus_s > kMaxSlots || n_experts_total > kMaxExperts)
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!topk_ids || !expert_offsets || !sorted_tok || !sorted_slot || !active_experts || !num_active || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(topk_ids, 4) || !aligned(expert_offsets, 4) || !aligned(sorted_tok, 4) ||
        !aligned(sorted_slot, 4) || !aligned(active_experts, 4) || !aligned(num_active, 4) || !aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < kHdrWords * sizeof(uint32_t))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    moe_status_t st = current_device_sms(&sms);
    if (st != MOE_OK)
        return st;
    (void)cudaGetLastError();
    GroupOut go{};
    go.offsets = expert_offsets;
    go.sorted_tok = sorted_tok;
    go.sorted_slot = sorted_slot;
    go.inv_pos = nullptr;
    go.active = active_experts;
    go.num_active = num_active;
    go.passes = nullptr;
    go.passes4 = nullptr;
    go.passesw = nullptr;
    go.passesw4 = nullptr;
    go.counters = nullptr;
    go.n_counters = 0;
    return from_cuda(launch_group(topk_ids, T, k_plus_s, n_experts_total, go, ws_at<uint32_t>(ws, 0), stream));
}

moe_status_t moe_expert_ffn_mxfp4(const uint16_t *x, const int32_t *topk_ids, const float *topk_w, int T, int top_k,
                                  const moe_mxfp4_bank_t *bank, uint16_t *y, void *ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    moe_status_t st = check_bank(bank);
    if (st != MOE_OK)
        return st;
    const int H = bank->hidden, I = bank->inter, E = bank->num_experts, S = bank->has_shared;
    if ((st = check_routing_shape(T, H, E, top_k, S)) != MOE_OK ||
        (st = check_ffn_extent(T, top_k + S, H, I)) != MOE_OK)
        return st;
    if (T == 0)
        return MOE_OK;
    if (!x || !topk_ids || !topk_w || !y || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = WsLayout::make(T, H, I, E, top_k, S);
    if (ws_bytes < L.total)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    if (T == 0)
        return MOE_OK;
    const GroupOut go = group_out_for(ws, L, H);
    cudaError_t err = launch_group(topk_ids, T, top_k + S, E + S, go, ws_at<uint32_t>(ws, 0), stream);
    if (err == cudaSuccess)
        err = launch_x16(x, T, H, ws, L, stream);
    if (err != cudaSuccess)
        return MOE_ERR_CUDA;
    FfnProblem pr{x, bank, topk_w, y, T, top_k + S};
    return from_cuda(launch_ffn(pr, ws, L, sms, stream, nullptr));
}

moe_status_t moe_layer_forward(const uint16_t *x, const float *router_w, const float *logit_bias, int T, int top_k,
                               const moe_mxfp4_bank_t *bank, float shared_weight, uint16_t *y,
                               int32_t *topk_ids_out, float *topk_w_out, void *ws, size_t ws_bytes,
                               cudaStream_t stream) {
    return layer_forward(x, router_w, logit_bias, T, top_k, bank, shared_weight, y, topk_ids_out, topk_w_out, ws,
                         ws_bytes, nullptr, stream);
}

moe_status_t moe_layer_forward_next(const uint16_t *x, const float *router_w, const float *logit_bias, int T,
                                    int top_k, const moe_mxfp4_bank_t *bank, float shared_weight, uint16_t *y,
                                    int32_t *topk_ids_out, float *topk_w_out, void *ws, size_t ws_bytes,
                                    const float *next_router_w, const moe_mxfp4_bank_t *next_bank,
                                    cudaStream_t stream) {
    if (next_bank && check_bank(next_bank) != MOE_OK)
        return MOE_ERR_INVALID_ARG;
    if (next_router_w && !aligned(next_router_w, 4))
        return MOE_ERR_MISALIGNED;
    return layer_forward(x, router_w, logit_bias, T, top_k, bank, shared_weight, y, topk_ids_out, topk_w_out, ws,
                         ws_bytes, nullptr, stream, next_router_w, next_bank);
}

size_t moe_packed_mx_bank_size(int H, int I, int E, int has_shared) {
    if (E <= 0 || (has_shared != 0 && has_shared != 1) || !mx8_shape_supported(H, I))
        return 0;
    return mx8_packed_size(H, I, E + has_shared);
}

moe_status_t moe_pack_bank_mx(const moe_mxfp4_bank_t *bank, void *packed_mx, size_t packed_mx_bytes,
                              cudaStream_t stream) {
    moe_status_t st = check_bank_dims(bank);
    if (st != MOE_OK)
        return st;
    if (!mx8_shape_supported(bank->hidden, bank->inter))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!bank->w13 || !bank->s13 || !bank->w2 || !bank->s2 || !packed_mx)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(bank->w13, 16) || !aligned(bank->w2, 16) || !aligned(bank->s13, 4) || !aligned(bank->s2, 4) ||
        !aligned(packed_mx, 256))
        return MOE_ERR_MISALIGNED;
    if (packed_mx_bytes < mx8_packed_size(bank->hidden, bank->inter, bank->num_experts + bank->has_shared))
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    return from_cuda(launch_mx8_pack(*bank, static_cast<uint8_t *>(packed_mx), stream));
}

}  // extern "C"

namespace {

// Body of the MXFP8 entry points; ev (nullable): 5 events recorded before the
// routing, after it, after the x quantisation, after the gate/up GEMM and at
// the end.
moe_status_t layer_forward_mxfp8(const uint16_t *x, const float *router_w, const float *logit_bias, int T,
                                 int top_k, const moe_mxfp4_bank_t *bank, const void *packed_mx,
                                 float shared_weight, uint16_t *y, int32_t *topk_ids_out, float *topk_w_out,
                                 void *ws, size_t ws_bytes, cudaEvent_t *ev, cudaStream_t stream) {
    moe_status_t st = check_bank_dims(bank);
    if (st != MOE_OK)
        return st;
    if (!packed_mx)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(packed_mx, 256))
        return MOE_ERR_MISALIGNED;
    const int H = bank->hidden, I = bank->inter, E = bank->num_experts, S = bank->has_shared;
    if (!mx8_shape_supported(H, I))
        return MOE_ERR_UNSUPPORTED_SHAPE;
    if ((st = check_routing_shape(T, H, E, top_k, S)) != MOE_OK ||
        (st = check_ffn_extent(T, top_k + S, H, I)) != MOE_OK)
        return st;
    if (T == 0)
        return MOE_OK;
    if (!x || !router_w || !y || !ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16) || !aligned(ws, 256) || !aligned(router_w, 4) ||
        !aligned(logit_bias, 4) || !aligned(topk_ids_out, 4) || !aligned(topk_w_out, 4))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = WsLayout::make(T, H, I, E, top_k, S);
    if (ws_bytes < L.total)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    if ((st = current_device_sms(&sms)) != MOE_OK)
        return st;
    (void)cudaGetLastError();
    int32_t *ids = topk_ids_out ? topk_ids_out : ws_at<int32_t>(ws, L.topk_ids);
    float *w = topk_w_out ? topk_w_out : ws_at<float>(ws, L.topk_w);
    const GroupOut go = group_out_for(ws, L, H);
    if (ev && cudaEventRecord(ev[0], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    // routing and grouping: for decode-sized T the routing phases of the
    // single-launch kernel (one cooperative launch), else the two routing
    // launches of the multi-launch path
    cudaError_t err = cudaErrorCooperativeLaunchTooLarge;
    if (T <= kFusedMaxTokens && fused_plan(T, H, I, E, top_k, S, sms).ok) {
        FusedProblem fp{x, router_w, logit_bias, bank, shared_weight, nullptr, ids, w, T, top_k,
                        nullptr, 0, nullptr, nullptr, 0, 0, ws_at<uint8_t>(ws, L.mx_xq), ws_at<uint8_t>(ws, L.mx_xs)};
        err = launch_fused(fp, ws, L, sms, stream, &go);
        if (err != cudaSuccess && err != cudaErrorCooperativeLaunchTooLarge)
            return MOE_ERR_CUDA;
        (void)cudaGetLastError();
    }
    if (err != cudaSuccess &&
        launch_route(x, router_w, logit_bias, T, H, E, top_k, S, shared_weight, ids, w, ws, L, true, go, stream) !=
            cudaSuccess)
        return MOE_ERR_CUDA;
    if (ev && cudaEventRecord(ev[1], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    const Mx8Problem pr{x, bank, static_cast<const uint8_t *>(packed_mx), w, y, T, top_k + S, err == cudaSuccess};
    if ((err = launch_mx8_ffn(pr, ws, L, stream, ev ? ev + 2 : nullptr)) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (ev && cudaEventRecord(ev[4], stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status_t moe_layer_forward_mxfp8(const uint16_t *x, const float *router_w, const float *logit_bias, int T,
                                     int top_k, const moe_mxfp4_bank_t *bank, const void *packed_mx,
                                     float shared_weight, uint16_t *y, int32_t *topk_ids_out, float *topk_w_out,
                                     void *ws, size_t ws_bytes, cudaStream_t stream) {
    return layer_forward_mxfp8(x, router_w, logit_bias, T, top_k, bank, packed_mx, shared_weight, y, topk_ids_out,
                               topk_w_out, ws, ws_bytes, nullptr, stream);
}

moe_status_t moe_layer_forward_mxfp8_profiled(const uint16_t *x, const float *router_w, const float *logit_bias,
                                              int T, int top_k, const moe_mxfp4_bank_t *bank,
                                              const void *packed_mx, float shared_weight, uint16_t *y, void *ws,
                                              size_t ws_bytes, cudaEvent_t *events, int n_events,
                                              cudaStream_t stream) {
    if (!events || n_events < 5)
        return MOE_ERR_INVALID_ARG;
    return layer_forward_mxfp8(x, router_w, logit_bias, T, top_k, bank, packed_mx, shared_weight, y, nullptr,
                               nullptr, ws, ws_bytes, events, stream);
}

moe_status_t moe_layer_forward_noalloc(const uint16_t *x, const float *router_w, const float *logit_bias, int T,
                                      int top_k, const moe_mxfp4_bank_t *bank, float shared_weight, uint16_t *y,
                                      int32_t *topk_ids_out, float *topk_w_out, cudaStream_t stream) {
    moe_status_t st = check_bank(bank);
    if (st != MOE_OK)
        return st;
    if ((st = check_routing_shape(T, bank->hidden, bank->num_experts, top_k, bank->has_shared)) != MOE_OK)
        return st;
    const WsLayout L = WsLayout::make(T, bank->hidden, bank->inter, bank->num_experts, top_k, bank->has_shared);
    if (L.total > kStaticScratchBytes)
        return MOE_ERR_WORKSPACE_TOO_SMALL;     // more scratch than the built-in array holds
    if (T == 0)
        return MOE_OK;
    if (!x || !router_w || !y)
        return MOE_ERR_INVALID_ARG;
    void *ws = nullptr;
    if ((st = static_scratch(&ws)) != MOE_OK)
        return st;
    return layer_forward(x, router_w, logit_bias, T, top_k, bank, shared_weight, y, topk_ids_out, topk_w_out, ws,
                         kStaticScratchBytes, nullptr, stream);
}

moe_status_t moe_layer_forward_profiled(const uint16_t *x, const float *router_w, const float *logit_bias, int T,
                                        int top_k, const moe_mxfp4_bank_t *bank, float shared_weight, uint16_t *y,
                                        void *ws, size_t ws_bytes, cudaEvent_t *events, int n_events,
                                        cudaStream_t stream) {
    if (!events || n_events != 5)
        return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 5; ++i)
        if (!events[i])
            return MOE_ERR_INVALID_ARG;
    return layer_forward(x, router_w, logit_bias, T, top_k, bank, shared_weight, y, nullptr, nullptr, ws, ws_bytes,
                         events, stream);
}

moe_status_t moe_layer_forward_hostio(const uint16_t *x_host, const float *router_w, const float *logit_bias, int T,
                                      int top_k, const moe_mxfp4_bank_t *bank, float shared_weight,
                                      uint16_t *y_host, void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status_t st = check_bank(bank);
    if (st != MOE_OK)
        return st;
    if (!x_host || !y_host || !ws || T < 0)
        return MOE_ERR_INVALID_ARG;
    const int H = bank->hidden;
    if ((st = check_routing_shape(T, H, bank->num_experts, top_k, bank->has_shared)) != MOE_OK)
        return st;
    if (!aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    const WsLayout L = WsLayout::make(T, H, bank->inter, bank->num_experts, top_k, bank->has_shared);
    if (ws_bytes < L.total)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    if (T == 0)
        return MOE_OK;
    uint16_t *xd = ws_at<uint16_t>(ws, L.xstage);
    uint16_t *yd = ws_at<uint16_t>(ws, L.ystage);
    const size_t bytes = (size_t)T * H * sizeof(uint16_t);
    (void)cudaGetLastError();
    if (cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    st = layer_forward(xd, router_w, logit_bias, T, top_k, bank, shared_weight, yd, nullptr, nullptr, ws, ws_bytes,
                       nullptr, stream);
    if (st != MOE_OK)
        return st;
    if (cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return from_cuda(cudaStreamSynchronize(stream));
}

int moe_layer_launches(int T, int H, int I, int E, int top_k, int has_shared) {
    if (T < 0 || H <= 0 || I <= 0 || E <= 0 || top_k <= 0 || (has_shared != 0 && has_shared != 1))
        return -1;
    if (T == 0)
        return 0;
    int sms = 0;
    if (current_device_sms(&sms) != MOE_OK)
        return -1;
    return (T <= kFusedMaxTokens && fused_plan(T, H, I, E, top_k, has_shared, sms).ok) ? 1 : 6;
}

moe_status_t moe_read_phase_times(void *ws, float *out_us, int n_out, cudaStream_t stream) {
    if (!ws || !out_us || n_out < 8)
        return MOE_ERR_INVALID_ARG;
    unsigned long long st[8];
    const uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    if (cudaMemcpyAsync(st, hdr + kHdrStamps, sizeof st, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    for (int i = 0; i < 6; ++i)
        out_us[i] = (float)((double)(long long)(st[i + 1] - st[i]) * 1e-3);
    out_us[6] = (float)((double)(long long)(st[7] - st[6]) * 1e-3);
    out_us[7] = (float)((double)(long long)(st[7] - st[0]) * 1e-3);
    return MOE_OK;
}

moe_status_t moe_check_device_status(void *ws, cudaStream_t stream) {
    if (!ws)
        return MOE_ERR_INVALID_ARG;
    uint32_t word = 0;
    uint32_t *hdr = ws_at<uint32_t>(ws, 0);
    if (cudaMemcpyAsync(&word, hdr + kHdrStatus, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (word != 0) {
        set_word_kernel<<<1, 1, 0, stream>>>(hdr + kHdrStatus, 0u);
        if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    return static_cast<moe_status_t>(word);
}

moe_status_t moe_selftest_decode_e2m1(const uint8_t *codes, uint16_t *out, int n, cudaStream_t stream) {
    if (!codes || !out || n < 0)
        return MOE_ERR_INVALID_ARG;
    int sms = 0;
    moe_status_t st = current_device_sms(&sms);
    if (st != MOE_OK)
        return st;
    if (n == 0)
        return MOE_OK;
    return from_cuda(launch_selftest_decode(codes, out, n, stream));
}

moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(ws, 256))
        return MOE_ERR_MISALIGNED;
    if (ws_bytes < kHeaderBytes)
        return MOE_ERR_WORKSPACE_TOO_SMALL;
    int sms = 0;
    moe_status_t st = current_device_sms(&sms);
    if (st != MOE_OK)
        return st;
    (void)cudaGetLastError();
    return from_cuda(launch_wait_selftest(ws_at<uint32_t>(ws, 0), stream));
}

const char *moe_status_string(moe_status_t s) {
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "misaligned pointer";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_ASSERT: return "device-side input check failed";
    case MOE_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    }
    return "unknown status";
}

}  // extern "C"
