/*
 * moe_fp4.h -- C ABI of the GB300 (sm_103a) small-T Mixture-of-Experts FFN
 * layer with MXFP4 expert weights.
 *
 * The layer (for each of T tokens with hidden state x[t], a bf16 row of H):
 *   a1  router logits      l[t,e] = sum_h x[t,h] * Wr[h,e] + b[e]      (e < E)
 *   a2  top-k + shared     the k largest logits (ties to the lower expert
 *                          index), ordered by descending logit; softmax over
 *                          the k kept logits; the shared expert (index E) is
 *                          appended as slot k with weight shared_weight.
 *   a3  grouping           (token, slot) pairs sorted by (expert, token).
 *   a4  gate/up + SiLU*up  h = silu(Wg x) * (Wu x),  silu(z) = z/(1+e^-z)
 *   a5  down               Y = Wd h
 *   a6  combine            y[t] = bf16_rn( sum_{s=0..k} w[t,s] * Y_s ),
 *                          summed in slot order in fp32.
 *
 * Where the definition comes from:
 *   - the shared expert merged into the routed MoE as one more expert that is
 *     always chosen (top-9 of 161 for GLM, shared expert in the 9th slot),
 *     with all expert outputs weighted and aggregated: "Optimizing GLM4-MoE
 *     for production" (blogs.novita.ai), section 1 "Shared experts fusion";
 *   - experts stored as MXFP4, 32-element blocks sharing one exponent:
 *     "How Xiaomi reached 1,000 tokens/s on a 1T-parameter model"
 *     (molayo1419.me), section 2 "MXFP4 with QAT" (element format E2M1 and
 *     scale format E8M0 of the OCP MX v1.0 specification);
 *   - top-8 routed experts per token, batch-1 decode being bound by streaming
 *     each active expert's weights from HBM once: GLM-5.2 on B300
 *     (d9249.github.io), sections "What it solves" and "1. ... Split-K".
 *
 * Data formats (all tensors row-major, all pointers DEVICE pointers owned by
 * the caller unless stated otherwise):
 *   x, y            bf16 bit patterns (uint16_t) [T, H]
 *   router_w        float [H, E]; logit_bias float [E] or NULL
 *   topk_ids        int32 [T, k+S]  (S = has_shared), routed ids in 0..E-1,
 *                   slot k = E when S = 1
 *   topk_w          float [T, k+S]
 *   bank.w13        uint8 [E+S, 2I, H/2]: rows 0..I-1 gate, I..2I-1 up; two
 *                   E2M1 codes per byte, element 2j in the low nibble
 *   bank.s13        uint8 [E+S, 2I, H/32]: E8M0 exponent of each 32-element
 *                   block along a row, value 2^(s-127)
 *   bank.w2         uint8 [E+S, H, I/2];  bank.s2 uint8 [E+S, H, I/32]
 *
 * Shapes supported: H and I multiples of 64, I <= 16384, H <= 65536;
 * 1 <= k <= E <= 1024; k + S <= 32; 0 <= T <= 4096.  E8M0 exponent 255 (NaN
 * in the MX specification) is not supported.
 * Pointers: x, y, bank arrays and the workspace 16-byte aligned; router_w,
 * logit_bias, topk_ids, topk_w 4-byte aligned.
 *
 * Execution: every call enqueues kernels on `stream` and returns without
 * synchronising (moe_check_device_status and the *_hostio call excepted).
 * Calls that share one workspace must not overlap on the GPU.
 *
 * Errors: calls return a moe_status_t.  Argument errors are found on the host
 * before anything is enqueued.  MOE_ERR_CUDA reports a failed launch (the
 * sticky-free CUDA error is cleared).  An expert id outside 0..E+S-1 in
 * caller-supplied topk_ids (or produced from non-finite router logits) is
 * found on the device: it is recorded in a status word inside the workspace,
 * the remaining kernels of the call do no work and leave y untouched, and
 * moe_check_device_status reports and clears the word.
 *
 * Waits: for T <= 8, moe_layer_forward runs the whole layer as one
 * cooperative launch (all CTAs resident at once) whose CTAs wait three times
 * for one another on a counter in the workspace.  Each wait gives up after
 * 200 ms (the cooperative launch makes that happen only after a fault
 * elsewhere): the call then records MOE_ERR_DEVICE_TIMEOUT and y is
 * undefined; the counters are reset when the kernel ends, so the workspace
 * stays usable.  No other kernel waits on another CTA or on a flag.
 */
#ifndef MOE_FP4_H
#define MOE_FP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, bad flag */
    MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* H, I, E, k outside the supported set */
    MOE_ERR_MISALIGNED = 3,         /* a pointer breaks its alignment rule */
    MOE_ERR_WORKSPACE_TOO_SMALL = 4,/* ws_bytes < moe_workspace_size(...) */
    MOE_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = 6,     /* a device-side wait gave up (see Waits) */
    MOE_ERR_DEVICE_ASSERT = 7,      /* device-side input check failed */
    MOE_ERR_UNSUPPORTED_DEVICE = 8  /* current device is not sm_103 */
} moe_status_t;

/* MXFP4 expert bank.  Expert index E is the shared expert when has_shared =
 * 1; it has the same shapes as the routed experts.  w13/s13/w2/s2 are the
 * canonical arrays described above, the input of moe_pack_bank; `packed` is
 * the repacked copy moe_pack_bank writes, which the expert-FFN calls read (the
 * canonical pointers may be NULL there). */
typedef struct {
    const uint8_t *w13;    /* [E+S, 2I, H/2]  */
    const uint8_t *s13;    /* [E+S, 2I, H/32] */
    const uint8_t *w2;     /* [E+S, H, I/2]   */
    const uint8_t *s2;     /* [E+S, H, I/32]  */
    const uint8_t *packed; /* moe_packed_bank_size(...) bytes, 256-byte aligned */
    int32_t num_experts;   /* E, routed experts */
    int32_t has_shared;    /* S, 0 or 1 */
    int32_t hidden;        /* H */
    int32_t inter;         /* I */
} moe_mxfp4_bank_t;

/* Bytes of a repacked bank (same bytes as the canonical arrays, permuted),
 * 0 for unsupported sizes. */
size_t moe_packed_bank_size(int H, int I, int E, int has_shared);

/*
 * Repacks the canonical arrays of `bank` into `packed` (device, 256-byte
 * aligned, moe_packed_bank_size bytes): a pure permutation of the E2M1 code
 * bytes and E8M0 exponent bytes into the order in which the expert-FFN
 * kernels stream them.  For each expert and each block of 16 weight rows
 * (gate/up: 8 gate rows with their 8 up rows; down: 16 consecutive rows) and
 * each 64-element step along K, 544 bytes: lane l = 4g + c of a warp finds at
 * bytes [16l, 16l+16) the 4-byte words c of blocks 2q, 2q of row g+8, 2q+1
 * of row g and 2q+1 of row g+8; bytes [512 + 4g, 516 + 4g) hold the
 * exponents of blocks 2q, 2q+1 of row g and of row g+8.  Gate/up section
 * first, then the down section at a 256-byte aligned offset.  Done once when
 * the weights are loaded; enqueued on `stream`.
 */
moe_status_t moe_pack_bank(const moe_mxfp4_bank_t *bank, void *packed, size_t packed_bytes,
                           cudaStream_t stream);

/* Bytes of device workspace the calls below need for these sizes (a caller
 * may pass a larger one).  The pages describe no such buffer: it holds the
 * intermediate results of a1..a6 (router partials, the grouping of a3, h and
 * the per-entry outputs of a4/a5) so that the library allocates nothing.  The workspace carries no state between calls
 * except its header: the device status word and the counters of the
 * single-launch layer kernel, which every completed call leaves at zero. */
size_t moe_workspace_size(int T, int H, int I, int E, int top_k, int has_shared);

/*
 * Diagnostics: byte offset inside the workspace of a named region of the
 * T-token layout.  After moe_layer_forward (either launch form) the
 * grouping of a3 lies there, as moe_group_tokens returns it: "offsets"
 * int32 [E+S+1], "sorted_tok" / "sorted_slot" int32 [T*(k+S)], "active"
 * int32 [E+S] (the first num_active entries), "num_active" one uint32, and
 * "inv_pos" int32 [T*(k+S)] (entry t*(k+S)+s -> its sorted position).
 * When moe_layer_forward ran as one launch (T <= 8): "h" fp32 [T*(k+S)][I]
 * (silu(gate) * up of each entry) and "y_entries" fp32 [T*(k+S)][H] (each
 * entry's down projection, before the weighted combine), rows in sorted
 * order.  Also "topk_ids", "topk_w" (when the call was not given output
 * arrays) and the MXFP8 variant's "mx_xq" [T][H] E4M3 codes of x, "mx_xs" [T][H/32] their
 * E8M0 scales, "mx_h32" [T*(k+S)][I] fp32 h, "mx_hq" / "mx_hs" its MXFP8
 * codes and scales, "mx_y" [T*(k+S)][H] fp32 per-entry outputs; entry rows in
 * grouped order).  (size_t)-1 for an unknown name or invalid sizes.
 */
size_t moe_workspace_offset(int T, int H, int I, int E, int top_k, int has_shared, const char *region);

/* Clears the workspace header (status word, counters and diagnostics, the
 * first 8,704 bytes or ws_bytes if smaller) on `stream`.  Call it once on a newly
 * allocated workspace before its first use (a zero-filled workspace needs no
 * call), and after a call that reported MOE_ERR_DEVICE_TIMEOUT.  ws: device
 * pointer, 256-byte aligned; ws_bytes at least 512. */
moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * a1 + a2: router logits, top-k selection, softmax weights and the shared
 * slot.  Logits are evaluated with error-free products and compensated
 * summation (Dot2 of Ogita, Rump and Oishi, "Accurate sum and dot product",
 * 2005), so the selection equals that of the exact logits unless two of them
 * differ by less than about 2^-40 times the sum of the |x*w| terms.
 * x [T,H] bf16; router_w [H,E]; logit_bias [E] or NULL; outputs topk_ids and
 * topk_w [T, k+S] (device).  ws: device workspace of
 * moe_workspace_size(T, H, 64, E, top_k, has_shared) bytes or more.
 */
moe_status_t moe_route_topk(const uint16_t *x, const float *router_w, const float *logit_bias,
                            int T, int H, int E, int top_k, int has_shared, float shared_weight,
                            int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                            cudaStream_t stream);

/*
 * a3: token-to-expert grouping of caller-supplied topk_ids [T, k_plus_s] --
 * the step that turns "top-9 of 161 with the shared expert always 9th" into
 * per-expert batches ("Optimizing GLM4-MoE for production", section 1
 * "Shared experts fusion").
 * Outputs (device): expert_offsets [n_experts_total+1] (exclusive prefix of
 * per-expert counts), sorted_tok and sorted_slot [T*k_plus_s] (pairs sorted
 * by expert, then token, then slot), active_experts [n_experts_total]
 * (experts with a nonzero count, ascending; entries past *num_active are
 * unspecified), num_active [1].  An id outside 0..n_experts_total-1 sets
 * MOE_ERR_DEVICE_ASSERT in the status word.
 */
moe_status_t moe_group_tokens(const int32_t *topk_ids, int T, int k_plus_s, int n_experts_total,
                              int32_t *expert_offsets, int32_t *sorted_tok, int32_t *sorted_slot,
                              int32_t *active_experts, int32_t *num_active, void *ws,
                              size_t ws_bytes, cudaStream_t stream);

/*
 * a3..a6 for a given routing: grouping, gate/up + SiLU*up, down and the
 * weighted combine -- each token's experts (the shared one included, with
 * the same tensor shapes) evaluated on MXFP4 weights and their outputs
 * weighted and summed ("Optimizing GLM4-MoE for production", section 1;
 * MXFP4 blocks of 32 with one shared exponent: the 1T-model article,
 * section 2).  topk_ids / topk_w [T, top_k + bank->has_shared] (device;
 * the shared slot, if any, must name expert E).  bank: host pointer to the
 * descriptor (its arrays are device memory).  y [T,H] bf16 (device).
 */
moe_status_t moe_expert_ffn_mxfp4(const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                                  int T, int top_k, const moe_mxfp4_bank_t *bank, uint16_t *y,
                                  void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * The whole layer a1..a6.  topk_ids_out / topk_w_out [T, top_k+S] are
 * optional (NULL: not returned).  For T <= 8 (and shapes whose staging fits
 * in shared memory) the layer is one cooperative kernel launch; otherwise a
 * sequence of six launches.  Both compute the same definition; they may
 * differ in the last bits of y through a different fp32 summation order.
 */
moe_status_t moe_layer_forward(const uint16_t *x, const float *router_w, const float *logit_bias,
                               int T, int top_k, const moe_mxfp4_bank_t *bank, float shared_weight,
                               uint16_t *y, int32_t *topk_ids_out, float *topk_w_out, void *ws,
                               size_t ws_bytes, cudaStream_t stream);

/*
 * One layer of a chain of MoE layers: moe_layer_forward, plus a hint naming
 * the layer that runs next on the same stream (next_router_w [H', E'] and
 * next_bank; either may be NULL).  When the layer runs as one launch (T <= 8)
 * its CTAs, once their last expert weights have been streamed, ask L2 to hold
 * the next layer's router weights and its shared expert (gate/up and down),
 * so that the next layer's router phase and shared expert read L2 instead of
 * HBM.  The hint changes no result: outputs are bit-identical to
 * moe_layer_forward.  It moves no data the next layer would not read anyway;
 * with T > 8 it is ignored.  The motivation is the cost the pages put on
 * operator and layer boundaries: the execution gap between operators (the
 * 1T-model article, section 1, "the problem") and the runtime row of the
 * GLM-5.2-on-B300 article's table of optimisation axes (launch, graph and
 * synchronisation overhead).
 */
moe_status_t moe_layer_forward_next(const uint16_t *x, const float *router_w, const float *logit_bias,
                                    int T, int top_k, const moe_mxfp4_bank_t *bank, float shared_weight,
                                    uint16_t *y, int32_t *topk_ids_out, float *topk_w_out, void *ws,
                                    size_t ws_bytes, const float *next_router_w,
                                    const moe_mxfp4_bank_t *next_bank, cudaStream_t stream);

/*
 * The MXFP8 live-activation-quantisation variant of the layer (the pages'
 * live FP8 activation quantisation in front of the GEMM and its tcgen05/TMEM
 * path: GLM-5.2 on B300, d9249.github.io, kernel sections 1 and 2).  Routing
 * and grouping are those of moe_layer_forward (bit-identical ids and
 * weights).  Then x[t] (blocks of 32 along H) and each entry's h (blocks of
 * 32 along I) are converted to MXFP8 -- E4M3 elements with one E8M0 scale per
 * block, the OCP MX v1.0 conversion: shared exponent floor(log2(max|v|)) - 8,
 * elements rounded to nearest even and saturated at 448 -- and both
 * projections run as block-scaled tensor-core MMAs with the MXFP4 weights.
 * This is a different, lossier definition than moe_layer_forward: y differs
 * from it by the activation quantisation (a few 1e-2 of max|y| at the
 * shapes tested), and it is compared against its own oracle mode.
 *
 * bank gives the dimensions only (its arrays are not read); the weights are
 * read from packed_mx, the copy moe_pack_bank_mx writes
 * (256-byte aligned).  H and I must be multiples of 128
 * (MOE_ERR_UNSUPPORTED_SHAPE).  Workspace:
 * moe_workspace_size(T, ...) bytes, as for moe_layer_forward.  Five
 * launches for T <= 8 (the routing phases of the single-launch kernel, which
 * also quantise x; the gate/up GEMM; the h finalisation and quantisation;
 * the down GEMM; the combine), seven above (two routing launches and a
 * separate x quantisation); asynchronous on `stream`, graph-capturable.
 */
moe_status_t moe_layer_forward_mxfp8(const uint16_t *x, const float *router_w, const float *logit_bias,
                                     int T, int top_k, const moe_mxfp4_bank_t *bank, const void *packed_mx,
                                     float shared_weight, uint16_t *y, int32_t *topk_ids_out,
                                     float *topk_w_out, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Bytes of the bank of the MXFP8 variant (0 when H or I is not a multiple of
 * 128): the same codes and scales as the canonical arrays, K-chunk major.
 * Four sections, each at a 256-byte aligned offset: gate/up codes
 * [E+S][H/128][2I][64 bytes], down codes [E+S][I/128][H][64 bytes], gate/up
 * scales [E+S][H/128][2I][4 bytes], down scales [E+S][I/128][H][4 bytes] --
 * for each expert and each chunk of 128 K elements, every weight row's bytes
 * of that chunk in row order.  The GEMMs read the codes with tensor copies
 * (16 E2M1 codes per 16-byte shared-memory slot, 128-byte swizzle), a
 * 64-row copy being 4 KB of consecutive bytes.
 */
/*
 * Diagnostics: moe_layer_forward_mxfp8 with CUDA events recorded on `stream`
 * between its steps: events[0] before the routing, [1] after it, [2] after
 * the x quantisation, [3] after the gate/up GEMM, [4] at the end (n_events
 * >= 5, else MOE_ERR_INVALID_ARG).  topk ids and weights are not returned.
 */
moe_status_t moe_layer_forward_mxfp8_profiled(const uint16_t *x, const float *router_w,
                                              const float *logit_bias, int T, int top_k,
                                              const moe_mxfp4_bank_t *bank, const void *packed_mx,
                                              float shared_weight, uint16_t *y, void *ws,
                                              size_t ws_bytes, cudaEvent_t *events, int n_events,
                                              cudaStream_t stream);

size_t moe_packed_mx_bank_size(int H, int I, int E, int has_shared);

/*
 * Fill packed_mx (moe_packed_mx_bank_size bytes, 256-byte aligned) from the
 * bank's canonical arrays (w13, s13, w2, s2: non-NULL, w13 / w2 16-byte and
 * s13 / s2 4-byte aligned) in the order above.  One-time, load-time work;
 * asynchronous on `stream`; the canonical arrays may be freed once it has
 * completed.
 */
moe_status_t moe_pack_bank_mx(const moe_mxfp4_bank_t *bank, void *packed_mx, size_t packed_mx_bytes,
                              cudaStream_t stream);

/*
 * The whole layer without a caller-provided workspace.  The pages have no
 * counterpart of this call; it exists for callers that cannot allocate device
 * memory themselves, such as plugins whose host application owns every device
 * allocation, or runtimes whose device-memory budget is fixed at start-up.
 * Its scratch is one array of 16 MiB compiled into the library, which every
 * GPU that loads the library holds until the process exits; problem sizes
 * whose workspace (moe_workspace_size) exceeds it are rejected with
 * MOE_ERR_WORKSPACE_TOO_SMALL.  The call allocates nothing (no cudaMalloc or
 * cudaFree).  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and keeps it for the life of the process; make that
 * first call before any stream capture, and do not use this entry point
 * across a cudaDeviceReset or from a context other than the device's primary
 * context (the kept address would be stale there).  The array needs no
 * clearing: it is zero-filled when the library's device code loads, and
 * every call leaves its counters at zero.  All calls on a device share the
 * array and it keeps the last call's contents: calls that overlap on the GPU
 * (other streams, other host threads) race and must be serialised by the
 * caller.  Arguments and outputs as in moe_layer_forward.  A device-side
 * routing error leaves y untouched; it is recorded in the array's status
 * word, which no call can read or clear (the first such error stays latched
 * for the life of the process): callers that need device-side error reports
 * use moe_layer_forward with a workspace of their own.
 */
moe_status_t moe_layer_forward_noalloc(const uint16_t *x, const float *router_w, const float *logit_bias,
                                       int T, int top_k, const moe_mxfp4_bank_t *bank,
                                       float shared_weight, uint16_t *y, int32_t *topk_ids_out,
                                       float *topk_w_out, cudaStream_t stream);

/*
 * The whole layer with the activations in HOST memory: copies x_host [T,H]
 * to the workspace, runs moe_layer_forward, copies y back to y_host [T,H]
 * and waits for the stream.  x_host / y_host should be pinned
 * (cudaHostAlloc) for asynchronous copies.  The weights, router and
 * workspace are device memory as above.
 */
moe_status_t moe_layer_forward_hostio(const uint16_t *x_host, const float *router_w,
                                      const float *logit_bias, int T, int top_k,
                                      const moe_mxfp4_bank_t *bank, float shared_weight,
                                      uint16_t *y_host, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * Self-test of the device-side wait limit: launches one CTA that waits on
 * the workspace's grid-wait counter for an arrival that never comes.  After
 * the 200 ms limit the wait gives up and records MOE_ERR_DEVICE_TIMEOUT in
 * the status word (read it with moe_check_device_status); the counters are
 * left at zero, so the workspace stays usable.  ws_bytes >= 8,704.
 */
moe_status_t moe_selftest_wait_timeout(void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Number of kernel launches moe_layer_forward makes for these sizes on the
 * current device: 1 when the layer runs as one cooperative launch, 6 for the
 * multi-launch sequence, 0 for T = 0, -1 on invalid sizes or when the device
 * cannot be queried.  Host-only; enqueues nothing.
 */
int moe_layer_launches(int T, int H, int I, int E, int top_k, int has_shared);

/*
 * Diagnostic: the phase durations (microseconds, from the GPU's global timer)
 * of the last single-launch layer call that used `ws`, as seen by its first
 * CTA: out_us[0] router partials, [1] first grid wait, [2] top-k and
 * grouping, [3] gate/up, [4] second grid wait, [5] down and combine, [6] time
 * from the first CTA's end to the last CTA's end, [7] whole kernel.
 * n_out >= 8.  Synchronises `stream`.  Values are meaningless after a
 * multi-launch call.
 */
moe_status_t moe_read_phase_times(void *ws, float *out_us, int n_out, cudaStream_t stream);

/*
 * Diagnostic form of moe_layer_forward: records events[0] before the first
 * kernel, events[1] after the router GEMV, events[2] after top-k/grouping,
 * events[3] after gate/up + h finalize and events[4] after down + combine, so
 * n_events must be 5.  Events are created by the caller.  When the layer runs
 * as one launch (T <= 8), events[1..4] are all recorded after it.
 */
moe_status_t moe_layer_forward_profiled(const uint16_t *x, const float *router_w,
                                        const float *logit_bias, int T, int top_k,
                                        const moe_mxfp4_bank_t *bank, float shared_weight,
                                        uint16_t *y, void *ws, size_t ws_bytes,
                                        cudaEvent_t *events, int n_events, cudaStream_t stream);

/* Waits for `stream`, then returns and clears the device status word of the
 * workspace (MOE_OK when no device-side error was recorded). */
moe_status_t moe_check_device_status(void *ws, cudaStream_t stream);

/* Self-test of the in-register E2M1 decode: out[2i], out[2i+1] (fp16 bit
 * patterns) are the elements held in the low and high nibble of codes[i].
 * n bytes; device pointers. */
moe_status_t moe_selftest_decode_e2m1(const uint8_t *codes, uint16_t *out, int n,
                                      cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char *moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP4_H */
