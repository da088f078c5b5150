/*
 * moe_b300.h -- C ABI of the DeepSeekMoE layer forward on one B300 (sm_103a).
 *
 * The layer (source: "【推理llm論文精讀】DeepSeek V3技術論文", section 2.2
 * "DeepSeekMoE"; the bias step also "AI新顶流-DeepSeek 技术大揭秘", section
 * 无辅助损失的负载均衡策略):
 *
 *   s_{i,t} = Sigmoid(u_t . e_i)                      affinity equation
 *   top-K_r experts of token t by s_{i,t} + b_i       biased selection
 *   g_{i,t} = s_{i,t} on those experts, else 0        routing-weight equation
 *   h_t = u_t + sum_{s<N_s} FFN^(s)_s(u_t)
 *             + sum_{i<N_r} g_{i,t} FFN^(r)_i(u_t)    FFN-output equation
 *   after the step: b_i -= gamma if expert i is overloaded,
 *                   b_i += gamma if it is underloaded
 *
 * FFN(x) = W_down (SiLU(W_gate x) * (W_up x)) (SwiGLU; the pages give no FFN
 * form).  Ties in the top-K go to the lower expert index.  No gate
 * renormalisation.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers, row-major, owned by the caller.
 *    The library allocates nothing; scratch lives in the caller's workspace
 *    (size from moe_workspace_size).
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  Argument errors are returned immediately and
 *    nothing is launched.  Errors found on the device (a pipeline wait that
 *    timed out, an index out of range) are recorded in a device error word
 *    and reported by moe_get_device_error.
 *  - Pointers must be 16-byte aligned.  d and d_ff must be multiples of 64,
 *    d a multiple of 128; n_routed <= 256 and a multiple of 16 for bf16
 *    (<= 1024 for fp32); 1 <= top_k <= min(16, n_routed); 0 <= n_shared <= 8.
 *    Violations return MOE_ERR_UNSUPPORTED (shape) or MOE_ERR_INVALID_ARG.
 *  - Element type of u, E, weights and x_perm: shape->dtype.  y_perm and
 *    y_shared are fp16 when dtype is bf16 and fp32 when dtype is fp32.
 *    bias and topk_gate are fp32; indices and counts int32.
 *  - MOE_FP8: activations (u, h) and the router stay bf16; the expert GEMMs
 *    run on e4m3 codes with power-of-two block scales (see
 *    moe_pack_weights_fp8); x_perm is an e4m3 buffer (moe_x_perm_bytes);
 *    y_perm and y_shared are fp16.  d_ff must be a multiple of 128.
 *  - The library never aborts the process.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad value        */
  MOE_ERR_UNSUPPORTED = 2,   /* shape outside the supported range           */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing or too small              */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call failed                  */
  MOE_ERR_TIMEOUT = 5,       /* a device pipeline wait gave up (no hang)    */
  MOE_ERR_DEVICE_CHECK = 6   /* a device-side bounds check failed           */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8 = 2 } moe_dtype;

typedef struct {
  int T;          /* tokens in the batch                                    */
  int d;          /* hidden size (length of u_t and e_i)                    */
  int n_routed;   /* N_r, routed experts                                    */
  int top_k;      /* K_r, routed experts per token                          */
  int n_shared;   /* N_s, shared experts (every token, weight 1)            */
  int d_ff;       /* I, intermediate size of every expert FFN               */
  moe_dtype dtype;/* element type of activations and weights                */
} moe_shape;

/* Bytes of workspace every call below needs for this shape (one buffer
 * serves all calls; it holds per-block histograms and the intermediate
 * activations H).  No alignment beyond 256 bytes is required.            */
MOE_API moe_status moe_workspace_size(const moe_shape* shape, size_t* bytes);

/* One-time weight repack (not part of the per-step path).
 *  w_gate, w_up   [n_routed, d_ff, d]   -> w_gu_packed  [n_routed, 2*d_ff, d]
 *  ws_gate, ws_up [n_shared, d_ff, d]   -> ws_gu_packed [2*n_shared*d_ff, d]
 *  ws_down        [n_shared, d, d_ff]   -> ws_down_packed [d, n_shared*d_ff]
 * Packed gate/up rows come in blocks of 128: 64 gate rows then the 64 up
 * rows of the same intermediate columns, so one 128-row weight tile yields
 * 64 columns of SiLU(gate)*up.  The shared experts are concatenated along
 * the intermediate dimension, so sum_s FFN_s(u) is one wider FFN.
 * Routed w_down [n_routed, d, d_ff] is used as is.  ws_* may be NULL when
 * n_shared == 0.                                                          */
MOE_API moe_status moe_pack_weights(const moe_shape* shape,
                            const void* w_gate, const void* w_up,
                            const void* ws_gate, const void* ws_up,
                            const void* ws_down,
                            void* w_gu_packed, void* ws_gu_packed,
                            void* ws_down_packed, void* stream);

/* FP8 expert weights (MOE_FP8).  The pages run most GEMMs on FP8 inputs
 * with activations and weights grouped into blocks that are scaled on their
 * own, and promote the tensor cores' partial sums to FP32 every 128
 * elements of the reduction (DeepSeek-V3 report commentary,
 * cooktownmusic.com, FP8 training-framework part, Fig. 7a/7b).  The
 * library's reading of the unstated details:
 *   element e4m3 (largest finite 448), round to nearest even, saturating;
 *   weight blocks 128 x 128, activation blocks 1 x 128 along the reduction;
 *   scale 2^e with e the smallest integer such that the block's largest
 *   magnitude is <= 448 * 2^e (0 for an all-zero block), stored as fp32;
 *   codes = e4m3(x * 2^-e).  H = SiLU(G) * U is requantized the same way
 *   (1 x 128 along d_ff) before the down projection.
 * moe_fp8_weight_bytes gives the size of each packed buffer (which: 0
 * routed gate/up, 1 routed down, 2 shared gate/up, 3 shared down); each
 * holds the codes followed, at the next 256-byte boundary, by the fp32
 * scales.  moe_pack_weights_fp8 quantizes the bf16 weights (layouts as in
 * moe_pack_weights, plus w_down [n_routed, d, d_ff]) into them; the shared
 * arguments may be NULL when n_shared == 0.  Layouts inside the packed
 * buffers are private to the library.                                    */
MOE_API moe_status moe_fp8_weight_bytes(const moe_shape* shape, int which,
                                        size_t* bytes);
MOE_API moe_status moe_pack_weights_fp8(const moe_shape* shape,
                                        const void* w_gate, const void* w_up,
                                        const void* w_down,
                                        const void* ws_gate, const void* ws_up,
                                        const void* ws_down, void* w_gu8,
                                        void* w_down8, void* ws_gu8,
                                        void* ws_down8, void* stream);

/* Bytes of the x_perm buffer of moe_permute / moe_expert_ffn: T*top_k*d
 * elements of shape->dtype, or for MOE_FP8 the e4m3 codes [T*top_k, d]
 * followed, at the next 256-byte boundary, by fp32 scales
 * [d/128][T*top_k].                                                       */
MOE_API moe_status moe_x_perm_bytes(const moe_shape* shape, size_t* bytes);

/* Routing (affinity equation, biased selection, routing-weight equation).
 *  u [T, d], centroids E [n_routed, d] (row i = e_i), bias b [n_routed] fp32
 *  -> topk_idx [T, top_k] int32: the selected experts of each token, by
 *     s+b descending, lower index first on ties;
 *     topk_gate [T, top_k] fp32: g = s (never s+b) of those experts;
 *     counts [n_routed] int32: tokens routed to each expert in this batch.
 * s = 1/(1+exp(-z)) with z accumulated in fp32 (bf16 inputs: on the tensor
 * cores; fp32 inputs: fp32 FMA).  The bias only selects.                  */
MOE_API moe_status moe_route(const moe_shape* shape, const void* u,
                     const void* centroids, const float* bias,
                     int32_t* topk_idx, float* topk_gate, int32_t* counts,
                     void* workspace, size_t workspace_bytes, void* stream);

/* Group-limited routing.  The pages name node-limited routing (a token's
 * experts drawn from at most a few nodes: "解码DeepSeek创新之道：三代模型
 * 演进路线图", V3 part; at most 4 nodes, the cooktownmusic.com report
 * commentary, training-framework part) but give no rule for choosing the
 * nodes.  The rule implemented: the n_routed experts form n_groups groups of
 * n_routed/n_groups consecutive indices; a group's score is the largest
 * s+b among its experts; each token keeps the topk_groups best groups (lower
 * group index first on ties) and takes its top_k experts, by s+b, among the
 * experts of the kept groups only.  Gates are s, as in moe_route.
 *  1 <= topk_groups <= n_groups <= 64, n_routed % n_groups == 0,
 *  top_k <= topk_groups * n_routed / n_groups; else MOE_ERR_INVALID_ARG and
 *  nothing is launched.
 * topk_groups == n_groups (e.g. 1, 1) is exactly moe_route.  Other
 * arguments, outputs and workspace as moe_route.                          */
MOE_API moe_status moe_route_grouped(const moe_shape* shape, int n_groups,
                                     int topk_groups, const void* u,
                                     const void* centroids, const float* bias,
                                     int32_t* topk_idx, float* topk_gate,
                                     int32_t* counts, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* Dispatch: expert-contiguous copy of the token rows.
 *  offsets [n_routed+1]: exclusive prefix sum of counts (offsets[N] = T*K);
 *  perm [T*K]: token filling each slot; slots of expert e are
 *     [offsets[e], offsets[e+1]) in ascending token order (deterministic);
 *  inv [T, top_k]: slot of assignment (t, k);
 *  x_perm [T*K, d]: x_perm[slot] = u[perm[slot]] (MOE_FP8: its e4m3 codes
 *     and 1 x 128 block scales, layout of moe_x_perm_bytes).              */
MOE_API moe_status moe_permute(const moe_shape* shape, const void* u,
                       const int32_t* topk_idx, const int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv,
                       void* x_perm, void* workspace, size_t workspace_bytes,
                       void* stream);

/* Expert FFNs (the two sums of the FFN-output equation, before weighting).
 *  y_perm [T*K, d]: rows [offsets[e], offsets[e+1]) = FFN^(r)_e of those
 *     x_perm rows, from w_gu_packed and w_down [n_routed, d, d_ff];
 *  y_shared [T, d] = sum_s FFN^(s)_s(u) (not written when n_shared == 0).
 * bf16: tcgen05 tensor-core GEMMs, fp32 accumulation in TMEM, H =
 * SiLU(gate)*up rounded to bf16 in the workspace (the second GEMM's
 * operand), y rounded once to fp16 (11 significant bits); an output
 * outside the fp16 range is reported as MOE_ERR_DEVICE_CHECK by
 * moe_get_device_error, never stored silently as inf.  fp32: fp32 FMA and
 * fp32 y.  MOE_FP8: x_perm from moe_permute, w_gu_packed / w_down /
 * ws_gu_packed / ws_down_packed are the four moe_pack_weights_fp8 buffers,
 * u (bf16) is quantized in the workspace for the shared experts; e4m3
 * tensor-core GEMMs with the block scales applied to the partial sum of
 * every 128-wide block of the reduction in fp32; H requantized to e4m3 in
 * the workspace; y fp16 as for bf16.                                      */
MOE_API moe_status moe_expert_ffn(const moe_shape* shape, const void* x_perm,
                          const int32_t* offsets, const void* w_gu_packed,
                          const void* w_down, const void* u,
                          const void* ws_gu_packed, const void* ws_down_packed,
                          void* y_perm, void* y_shared, void* workspace,
                          size_t workspace_bytes, void* stream);

/* One part of moe_expert_ffn: part 1 = the routed experts only (y_perm),
 * part 2 = the shared experts only (y_shared; x_perm, offsets, w_gu_packed,
 * w_down and y_perm may be NULL), part 0 = both (moe_expert_ffn).  A part-2
 * call uses its own item counters and workspace regions, so it may run on
 * another stream at the same time as the routing, the permute and a part-1
 * call on the same workspace (the shared experts need no routing).  bf16
 * and fp32 shapes; MOE_FP8 takes part 0 only (MOE_ERR_UNSUPPORTED).      */
MOE_API moe_status moe_expert_ffn_part(const moe_shape* shape, int part,
                                       const void* x_perm,
                                       const int32_t* offsets,
                                       const void* w_gu_packed,
                                       const void* w_down, const void* u,
                                       const void* ws_gu_packed,
                                       const void* ws_down_packed,
                                       void* y_perm, void* y_shared,
                                       void* workspace,
                                       size_t workspace_bytes, void* stream);

/* moe_expert_ffn for a training step (bf16 layers only, else
 * MOE_ERR_UNSUPPORTED): the same outputs, bit for bit, and the gate and up
 * pre-activations a = W_gate x, c = W_up x of every row, rounded to fp16
 * (11 significant bits, the precision of the recomputing path to within
 * its other roundings; a value outside the fp16 range is reported as
 * MOE_ERR_DEVICE_CHECK by moe_get_device_error), for moe_backward, which
 * then skips recomputing them.
 *  act [T*K, 2*d_ff] fp16: row = x_perm slot; act_shared [T, 2*S*d_ff]
 *  fp16: row = token (may be NULL when n_shared == 0).  Columns are in the
 *  packed order of moe_pack_weights (blocks of 64 gate then 64 up values);
 *  the layout is for moe_backward only.  The caller owns both buffers and
 *  keeps them until the backward has read them.  act NULL ->
 *  MOE_ERR_INVALID_ARG.                                                   */
MOE_API moe_status moe_expert_ffn_train(const moe_shape* shape,
                                        const void* x_perm,
                                        const int32_t* offsets,
                                        const void* w_gu_packed,
                                        const void* w_down, const void* u,
                                        const void* ws_gu_packed,
                                        const void* ws_down_packed,
                                        void* y_perm, void* y_shared,
                                        void* act, void* act_shared,
                                        void* workspace,
                                        size_t workspace_bytes, void* stream);

/* Combine (FFN-output equation):
 *  h[t] = u[t] + y_shared[t] + sum_k topk_gate[t,k] * y_perm[inv[t,k]],
 * accumulated in fp32 in that order; h is written as h_dtype.  y_shared may
 * be NULL when n_shared == 0.                                             */
MOE_API moe_status moe_combine(const moe_shape* shape, const void* u,
                       const void* y_perm, const void* y_shared,
                       const int32_t* inv, const float* topk_gate, void* h,
                       moe_dtype h_dtype, void* stream);

/* Auxiliary-loss-free bias step after a batch (section 2.2 of the notes;
 * load counted over the whole step):
 *   counts[i]*n_routed >  total_assign  (overloaded):  b_i = fl32(b_i - gamma)
 *   counts[i]*n_routed <  total_assign  (underloaded): b_i = fl32(b_i + gamma)
 *   otherwise unchanged.  total_assign = T*K.  gamma is rounded to fp32.    */
MOE_API moe_status moe_update_bias(int n_routed, const int32_t* counts,
                           long long total_assign, float gamma, float* bias,
                           void* stream);

/* Synchronises `stream`, reads and clears the device error word of the
 * current device.  MOE_OK, MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK.       */
MOE_API moe_status moe_get_device_error(void* stream);

/* Self-test of the device-side failure detection: launches one kernel whose
 * single thread waits on a barrier that nothing signals, with a limit of
 * limit_us microseconds (1 .. 1000000) instead of the pipelines' 2 s.  The
 * wait gives up, records a timeout in the device error word and the kernel
 * returns, so the next moe_get_device_error(stream) returns MOE_ERR_TIMEOUT
 * and the context stays usable.  Every pipeline wait of the library uses
 * the same bounded-wait routine.                                          */
MOE_API moe_status moe_selftest_wait_timeout(unsigned limit_us, void* stream);

/* Static description of a status code; detail of the last host-side error
 * of the calling thread.                                                  */
MOE_API const char* moe_status_string(moe_status status);
MOE_API const char* moe_last_error_detail(void);

/* Number of kernel launches the previous successful call on this thread
 * issued (for launch accounting).                                         */
MOE_API int moe_last_launch_count(void);

/* ----------------------------------------------------------------------
 * Backward pass (training): the gradients of the layer output h with
 * respect to u, the centroids E and every expert weight, for an upstream
 * gradient dh = dL/dh.  The three GEMMs of each linear operator (forward,
 * activation gradient "Dgrad", weight gradient "Wgrad"): "AI新顶流-DeepSeek
 * 技术大揭秘" (blog.csdn.net), section "FP8混合精度训练框架"; the layer whose
 * derivative is taken is the FFN-output equation above.  The chain rule,
 * per selected expert e of token t (g = topk_gate, x = u_t):
 *   dY = g dh_t;   dW_down += dY H^T;   dH = W_down^T dY;
 *   da = dH c SiLU'(a), dc = dH SiLU(a)  (a = W_gate x, c = W_up x);
 *   dW_gate += da x^T;  dW_up += dc x^T;  du_t += W_gate^T da + W_up^T dc;
 *   dz = (dh_t . y) g (1 - g)  (y = FFN_e(x), z = u_t . e_e);
 *   du_t += dz e_e;  dE_e += dz u_t;
 * shared experts the same with g = 1 and no gate term; du_t += dh_t.  The
 * selection is piecewise constant and the bias receives no gradient.
 *
 * Inputs: the forward's own tensors: u [T, d], centroids [N, d] (bf16),
 * topk_idx / topk_gate [T, K] (moe_route), offsets [N+1] and inv [T, K]
 * (moe_permute), y_perm [T*K, d] fp16 (moe_expert_ffn), the packed weights
 * of moe_pack_weights and w_down; dh [T, d] bf16.  act / act_shared: the
 * pre-activations saved by moe_expert_ffn_train on the same batch, or both
 * NULL; with them the SwiGLU backward runs in the epilogue of the dH GEMM
 * from the saved a, c (and dH in fp32), without them a and c are recomputed
 * by a third gate/up GEMM.
 * Outputs (overwritten, not accumulated): du [T, d] fp32, dE [N, d] fp32;
 * dw_gate / dw_up [N, d_ff, d], dw_down [N, d, d_ff] and, when
 * n_shared > 0, dws_gate / dws_up [S, d_ff, d], dws_down [S, d, d_ff] in
 * the canonical (unpacked) layouts, as grad_dtype (MOE_F32 or MOE_BF16).
 * Arithmetic: bf16 GEMM operands (x, dY, H, dA rounded to bf16; a, c
 * saved in fp16 or recomputed in fp32), fp32 accumulation in TMEM; the
 * recomputing path keeps dH in fp16 between its GEMMs, and both keep the
 * input-side products in fp16 (range checked).  Every call is
 * asynchronous on `stream`; the workspace (moe_backward_workspace_size,
 * 256-byte aligned) holds the per-assignment operands in a layout whose
 * expert segments are padded to 16 rows.
 * Supported: dtype MOE_BF16 and d_ff a multiple of 128 (else
 * MOE_ERR_UNSUPPORTED); every pointer 16-byte aligned (else
 * MOE_ERR_INVALID_ARG).                                                   */
MOE_API moe_status moe_backward_workspace_size(const moe_shape* shape,
                                               size_t* bytes);
MOE_API moe_status moe_backward(
    const moe_shape* shape, const void* dh, const void* u,
    const void* centroids, const int32_t* topk_idx, const float* topk_gate,
    const int32_t* offsets, const int32_t* inv, const void* y_perm,
    const void* act, const void* act_shared,
    const void* w_gu_packed, const void* w_down, const void* ws_gu_packed,
    const void* ws_down_packed, float* du, float* dE, void* dw_gate,
    void* dw_up, void* dw_down, void* dws_gate, void* dws_up, void* dws_down,
    moe_dtype grad_dtype, void* workspace, size_t workspace_bytes,
    void* stream);

/* moe_route without a workspace, for callers that cannot allocate device
 * memory at the point of the call: for example a plugin inside an inference
 * engine that is handed only its input and output buffers and may not
 * allocate while the engine runs (cudaMalloc can synchronise the device and
 * break the engine's memory plan), or code running where allocating CUDA
 * calls are not allowed at all.  The layer equations have no counterpart of
 * this call; it exists only for such callers.
 *
 * Arguments and results are those of moe_route (same kernels).  The router's
 * per-block histograms go to a library-owned array in device memory of
 * MOE_ROUTE_NOALLOC_MAX_ENTRIES int32 (1 MiB), which every GPU that loads
 * the library holds until the process exits.  A call needs n_routed
 * entries per router CTA: ceil(T/128) CTAs, or up to 8 per 128-token tile
 * while the grid stays within one wave of the GPU's SMs (for example T up to
 * 131072 tokens with 256 experts); larger shapes return MOE_ERR_UNSUPPORTED
 * and launch nothing.
 * The call allocates nothing (no cudaMalloc, no cudaFree).  Its first call
 * on a device looks up that array's device address (cudaGetSymbolAddress)
 * with the device current; make that first call before any stream capture.
 * All calls share the one array and it keeps the last call's contents:
 * each call writes every entry it later reads, so nothing needs clearing,
 * but calls that overlap on the GPU (other streams, other threads) race on
 * it and must be serialised by the caller.                                */
#define MOE_ROUTE_NOALLOC_MAX_ENTRIES (1 << 18)
MOE_API moe_status moe_route_noalloc(const moe_shape* shape, const void* u,
                                     const void* centroids, const float* bias,
                                     int32_t* topk_idx, float* topk_gate,
                                     int32_t* counts, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_B300_H */
