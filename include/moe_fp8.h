/*
 * moe_fp8.h - C ABI of the routed FP8 Mixture-of-Experts FFN forward for
 * sm_103a (GB300).
 *
 * The layer (Kimi K2 MoE block FFN):
 *   scores  s = sigmoid(x W_g^T)                    "Kimi-K2-Base", Mixture of experts: Router score
 *   choice  c = s + b  (bias used only to choose)    same section: Load balancing (e_score_correction_bias)
 *   I       = top-k of c per token (one group)       same section: Experts per token, Group-limited routing none
 *   w_j     = s_{I_j} / sum_j s_{I_j} * 2.827        same section: Renormalize top-k, Routed scaling factor
 *   E_e(x)  = down(silu(gate x) * up x), no bias     "Kimi-K2-Base", Feed-forward: Activation, FFN bias
 *   y       = shared(x) + sum_j w_j E_{I_j}(x)       "Kimi K2 · Architecture", Fact sheet: 384 routed + 1 shared
 * Weights are e4m3 with one fp32 scale per 128x128 block ("Kimi K2 ·
 * Architecture", config.json quantization_config); activations entering each
 * projection are quantised dynamically to e4m3 in 1x128 groups with an fp32
 * scale amax/448 ("Kimi-K2-Base", Pretraining recipe: Training precision).
 *
 * Conventions for every call:
 *  - Memory: every pointer is DEVICE memory allocated and owned by the caller,
 *    except `cfg` (host). The library never allocates or frees and never
 *    synchronises the stream. Device buffers must be 16-byte aligned.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream). Every
 *    call only enqueues work on it and returns. The kernels are launched with
 *    programmatic dependent launch allowed: each waits for the stream's
 *    preceding kernel to complete before it touches global memory, and lets
 *    the next kernel start launching at once. Ordinary launches, copies and
 *    events after a call keep plain stream order. A kernel the caller launches
 *    after a call with the programmatic-serialisation attribute must itself
 *    wait (cudaGridDependencySynchronize) before it reads the call's outputs.
 *  - Errors: every call returns a moe_status_t. Arguments are checked on the
 *    host before anything is enqueued; on an error nothing is enqueued.
 *    moe_last_error_string() describes the last error of the calling thread.
 *  - T = 0 is legal for every call and enqueues nothing.
 *  - Layouts are row-major. Weight matrices use the nn.Linear layout
 *    [out_features, in_features]. Scales of 1x128 activation groups are stored
 *    K-block-major ("transposed"): scale of row r, group g at [g * rows + r]
 *    unless a call says otherwise.
 *  - Shapes: d and H multiples of 128; 1 <= topk <= 32, topk <= E <= 1024;
 *    0 <= n_shared <= 4.
 */
#ifndef MOE_FP8_H
#define MOE_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_ARG = -1,          /* null pointer, misaligned pointer, bad size or short workspace */
    MOE_ERR_UNSUPPORTED = -2,  /* shape outside the supported range */
    MOE_ERR_CUDA = -3,         /* a CUDA call or launch failed; see moe_last_error_string() */
    MOE_ERR_TIMEOUT = -4,      /* a bounded device wait gave up (reported by moe_check_device_error) */
    MOE_ERR_INDEX = -5         /* a device-side index check failed and its access was skipped
                                  (reported by moe_check_device_error) */
} moe_status_t;

/* Shape of one MoE layer. */
typedef struct {
    int d;              /* model width (hidden_size) */
    int E;              /* routed experts (n_routed_experts) */
    int topk;           /* experts chosen per token (num_experts_per_tok) */
    int H;              /* hidden features of one expert (moe_intermediate_size) */
    int n_shared;       /* always-on shared experts (n_shared_experts) */
    float route_scale;  /* routed_scaling_factor */
    int w_tiled;        /* 0: expert weights row-major (w13 [E+S, 2, H, d], w2 [E+S, d, H]);
                           1: the same bytes in 128 x 128 tiles, as moe_pack_weights_fp8 writes
                           them (the GEMMs then read each 16 KB tile in one sequential run) */
} moe_cfg_t;

/* Rows of the permuted activation buffer: topk*T routed rows, then n_shared*T
 * shared-expert rows (row topk*T + s*T + t holds token t for shared expert s). */
int64_t moe_permuted_rows(const moe_cfg_t *cfg, int T);

/* Bytes of caller-provided workspace needed by moe_route, moe_permute,
 * moe_expert_gemm_fp8 and moe_layer_forward for T tokens (one size fits all
 * of them). Returns 0 for an invalid cfg. Host only. */
size_t moe_workspace_bytes(const moe_cfg_t *cfg, int T);

/* Dynamic 1x128 quantisation ("Kimi-K2-Base", Pretraining recipe: Training
 * precision; scale = amax / 448).
 * in      [rows, cols] bf16 (in_is_bf16 = 1) or fp32 (in_is_bf16 = 0)
 * q       [rows, cols] e4m3 codes (uint8)
 * s       [rows, cols/128] fp32, ROW-major (s_transposed = 0) or
 *         [cols/128, rows] (s_transposed = 1)
 * Per group of 128 columns: s = fp32(amax) / 448 (IEEE division);
 * q = e4m3(fp32(x) / s) (the correctly rounded fp32 quotient, as IEEE division
 * gives it; then round to nearest even, saturate to +-448); a group with
 * amax = 0 gets s = 0 and codes 0x00. cols % 128 == 0. */
int moe_quant_fp8_1x128(const void *in, int in_is_bf16, int64_t rows, int cols,
                        uint8_t *q, float *s, int s_transposed, void *stream);

/* Router ("Kimi-K2-Base", Mixture of experts: Router score, Load balancing,
 * Renormalize top-k, Routed scaling factor).
 * x         [T, d] bf16;  w_gate [E, d] bf16;  bias [E] fp32
 * topk_idx  [T, topk] int32: chosen experts, descending biased score, equal
 *           scores ordered by the lower expert id
 * topk_w    [T, topk] fp32: s_I / sum(s_I) * route_scale (unbiased scores)
 * scores    [T, E] fp32 sigmoid scores, or NULL
 * Logits accumulate in fp32 on the tensor cores; sigmoid, bias and weights in fp32. */
int moe_route(const void *x, const void *w_gate, const float *bias, const moe_cfg_t *cfg, int T,
              int32_t *topk_idx, float *topk_w, float *scores,
              void *workspace, size_t workspace_bytes, void *stream);

/* Token permutation into contiguous per-expert segments (deterministic).
 * topk_idx   [T, topk] int32 (each row distinct ids < E)
 * xq, sx     [T, d] e4m3 and [T, d/128] fp32 ROW-major (moe_quant_fp8_1x128, s_transposed = 0)
 * offsets    [E + 1] int32: exclusive prefix sum of per-expert counts, offsets[E] = topk*T
 * sorted_tok [topk*T] int32: segment e = [offsets[e], offsets[e+1]) holds its tokens ascending
 * inv_pos    [T, topk] int32: position of assignment (t, topk_idx[t, j]) in sorted_tok
 * xq_perm    [moe_permuted_rows, d] e4m3: row p < topk*T is xq[sorted_tok[p]];
 *            then n_shared copies of xq in token order
 * sx_perm    [d/128, moe_permuted_rows] fp32 (K-block-major) scales of xq_perm's rows */
int moe_permute(const int32_t *topk_idx, const uint8_t *xq, const float *sx,
                const moe_cfg_t *cfg, int T,
                int32_t *offsets, int32_t *sorted_tok, int32_t *inv_pos,
                uint8_t *xq_perm, float *sx_perm,
                void *workspace, size_t workspace_bytes, void *stream);

/* The tiled weight layout (cfg->w_tiled = 1): w [groups, rows, cols] e4m3,
 * row-major, becomes w_tiled [groups, rows/128, cols/128, 128, 128] with
 *   w_tiled[g][rb][cb][r][c] = w[g][rb*128 + r][cb*128 + c],
 * so every 128 x 128 block of a weight matrix (one 128-row block of one 128-wide
 * K block, the unit the GEMMs load) is 16 KB of contiguous memory. For the
 * expert weights: w13 [E+S, 2, H, d] with groups = 2(E+S), rows = H, cols = d;
 * w2 [E+S, d, H] with groups = E+S, rows = d, cols = H. The block scales keep
 * their layout. A one-time transformation of the weights; w and w_tiled must not
 * overlap. rows % 128 == 0, cols % 128 == 0; groups == 0 is a no-op. Pointers
 * 16-byte aligned. */
int moe_pack_weights_fp8(const uint8_t *w, int64_t groups, int rows, int cols, uint8_t *w_tiled,
                         void *stream);

/* moe_quant_fp8_1x128 of x (in_is_bf16 = 1, s_transposed = 0) followed by
 * moe_permute, in one pass over x: each token's 1x128 codes and scales are
 * computed once and written straight to its permuted rows, and the unpermuted
 * codes are never stored.
 * x [T, d] bf16; every other argument and output as moe_permute's. The outputs
 * equal those of the two calls bit for bit. Pointers 16-byte aligned. */
int moe_quant_permute_fp8(const int32_t *topk_idx, const void *x,
                          const moe_cfg_t *cfg, int T,
                          int32_t *offsets, int32_t *sorted_tok, int32_t *inv_pos,
                          uint8_t *xq_perm, float *sx_perm,
                          void *workspace, size_t workspace_bytes, void *stream);

/* moe_permute without a caller workspace. The pages have no counterpart: this
 * entry point exists for callers that cannot provide scratch memory, such as a
 * plugin inside a host application that owns every device allocation, or a
 * serving loop that may not call cudaMalloc after start-up (cudaMalloc
 * synchronises the device and can fail when memory is tight).
 * Arguments and outputs are those of moe_permute, minus the workspace. The
 * scratch lives in one fixed device array inside the library (about 1.3 MB,
 * held on every GPU that loads the library until the process exits), so:
 *  - limits: T <= 8192 tokens, T * topk <= 65536 assignments, E <= 1024,
 *    n_shared <= 4; larger calls return MOE_ERR_UNSUPPORTED and enqueue nothing;
 *  - the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture. The address is kept for the rest of the
 *    process: calls after a cudaDeviceReset of that device are not supported
 *    (the array may then live elsewhere);
 *  - every call on a device shares the array: calls that may run at the same
 *    time on the GPU (different streams without ordering) race and give wrong
 *    results. Nothing in the array needs to be zero between calls;
 *  - it allocates nothing and calls no allocating routine. */
int moe_permute_noalloc(const int32_t *topk_idx, const uint8_t *xq, const float *sx,
                        const moe_cfg_t *cfg, int T,
                        int32_t *offsets, int32_t *sorted_tok, int32_t *inv_pos,
                        uint8_t *xq_perm, float *sx_perm, void *stream);

/* Grouped expert SwiGLU over FP8 weights ("Kimi-K2-Base", Feed-forward):
 * for each expert segment, o = down(silu(gate x) * up x), with h = silu(g) * u
 * quantised 1x128 between the two projections. Runs on the tcgen05 tensor
 * cores; the 128x128 weight scales and the 1x128 activation scales are applied
 * per 128-wide K block in fp32.
 * xq_perm, sx_perm  as written by moe_permute; offsets [E+1] (device)
 * w13    [E+S, 2, H, d] e4m3 (index 0 gate_proj, 1 up_proj); w13_s [E+S, 2, H/128, d/128] fp32
 * w2     [E+S, d, H] e4m3 (down_proj); w2_s [E+S, d/128, H/128] fp32
 *        (w13 and w2 in the tiled layout of moe_pack_weights_fp8 when cfg->w_tiled = 1)
 * o      [moe_permuted_rows, d] bf16, same row order as xq_perm
 * Routed experts come first, shared experts last. */
int moe_expert_gemm_fp8(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets,
                        const uint8_t *w13, const float *w13_s, const uint8_t *w2, const float *w2_s,
                        const moe_cfg_t *cfg, int T, void *o,
                        void *workspace, size_t workspace_bytes, void *stream);

/* The two halves of moe_expert_gemm_fp8, for callers that schedule them apart.
 * moe_expert_gateup_fp8: h = silu(gate x) * up x per expert segment, quantised 1x128:
 *   hq [moe_permuted_rows, H] e4m3, hs [H/128, moe_permuted_rows] fp32 (K-block-major).
 * moe_expert_down_fp8: o = down(h) per expert segment from hq/hs; o as in moe_expert_gemm_fp8.
 * Other arguments as in moe_expert_gemm_fp8. */
int moe_expert_gateup_fp8(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets,
                          const uint8_t *w13, const float *w13_s, const moe_cfg_t *cfg, int T,
                          uint8_t *hq, float *hs, void *workspace, size_t workspace_bytes, void *stream);
int moe_expert_down_fp8(const uint8_t *hq, const float *hs, const int32_t *offsets,
                        const uint8_t *w2, const float *w2_s, const moe_cfg_t *cfg, int T, void *o,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Weighted combine: y[t] = sum_s o[topk*T + s*T + t] + sum_j topk_w[t, j] * o[inv_pos[t, j]],
 * in fp32 in that order, rounded to bf16.
 * o [moe_permuted_rows, d] bf16; topk_w, inv_pos [T, topk]; y [T, d] bf16. */
int moe_combine(const void *o, const float *topk_w, const int32_t *inv_pos,
                const moe_cfg_t *cfg, int T, void *y, void *stream);

/* The block's pieces next to the layer ("Kimi K2 · Dense transformer block",
 * Sources: residual = h; h = post_attention_layernorm(h); h = mlp(h);
 * h = residual + h; "Kimi-K2-Base", Normalization and stability: RMSNorm, pre-norm,
 * epsilon 1e-06). RMSNorm of a bf16 row: y = bf16(h * gamma / sqrt(mean(h^2) + eps)),
 * the sum of squares in fp32 (fixed order), IEEE square root and division.
 *
 * moe_rmsnorm_quant_fp8: the layer input from the residual stream in one pass:
 *   h [rows, cols] bf16; gamma [cols] bf16; y [rows, cols] bf16 (may be NULL: not
 *   written); q, s the 1x128 quantisation of the bf16 y values, bit-identical to
 *   moe_quant_fp8_1x128 applied to y (s layout as there). cols % 128 == 0.
 *   Pointers 16-byte aligned; rows == 0 is a no-op. */
int moe_rmsnorm_quant_fp8(const void *h, const void *gamma, float eps, int rows, int cols,
                          void *y, uint8_t *q, float *s, int s_transposed, void *stream);

/* moe_combine_residual_rmsnorm: moe_combine (same summation order) rounded to bf16
 * as the FFN output y, then h_out = bf16(residual + y) (the block's second residual
 * addition), and, when gamma is not NULL, x_next = the next block's input RMSNorm
 * of h_out (gamma and x_next both given or both NULL).
 * o, topk_w, inv_pos as in moe_combine; residual, h_out, x_next [T, d] bf16;
 * gamma [d] bf16. */
int moe_combine_residual_rmsnorm(const void *o, const float *topk_w, const int32_t *inv_pos,
                                 const moe_cfg_t *cfg, int T, const void *residual, const void *gamma,
                                 float eps, void *h_out, void *x_next, void *stream);

/* The whole layer: route, quantise x, permute, grouped expert GEMMs, combine
 * (the quantisation runs inside the permutation, as in moe_quant_permute_fp8).
 * x [T, d] bf16; w_gate [E, d] bf16; bias [E] fp32; weights as in
 * moe_expert_gemm_fp8; y [T, d] bf16. topk_idx / topk_w [T, topk] receive the
 * routing when not NULL. workspace: moe_workspace_bytes(cfg, T) bytes. y equals
 * the chain moe_route, moe_quant_fp8_1x128, moe_permute, moe_expert_gemm_fp8,
 * moe_combine on the same inputs bit for bit. The call only enqueues kernels on
 * the stream (no allocation, synchronisation or host read of device data), so it
 * can be captured in a CUDA graph. */
int moe_layer_forward(const void *x, const void *w_gate, const float *bias,
                      const uint8_t *w13, const float *w13_s, const uint8_t *w2, const float *w2_s,
                      const moe_cfg_t *cfg, int T, void *y, int32_t *topk_idx, float *topk_w,
                      void *workspace, size_t workspace_bytes, void *stream);

/* The FFN half of a MoE block in one call ("Kimi K2 · Dense transformer block",
 * Sources: residual = h; h = post_attention_layernorm(h); h = mlp(h);
 * h = residual + h; "Kimi-K2-Base", Normalization and stability: RMSNorm, eps):
 *   x      = RMSNorm_post(h) = bf16(gamma_post * h / sqrt(mean(h^2) + eps)),
 *            with its 1x128 e4m3 codes and scales formed in the same pass (the
 *            layer's input quantisation, bit for bit that of moe_quant_fp8_1x128
 *            on x; no second pass over x);
 *   y      = the MoE layer of moe_layer_forward on x (route on x, permute the codes);
 *   h_out  = bf16(h + bf16(y));
 *   x_next = RMSNorm_next(h_out) when gamma_next is given (the next block's input).
 * h [T, d] bf16 (the residual stream), gamma_post / gamma_next [d] bf16, eps >= 0;
 * h_out, x_next [T, d] bf16 (gamma_next and x_next both given or both NULL);
 * other arguments as in moe_layer_forward; workspace: moe_workspace_bytes(cfg, T). */
int moe_block_ffn_forward(const void *h, const void *gamma_post, float eps, const void *w_gate, const float *bias,
                          const uint8_t *w13, const float *w13_s, const uint8_t *w2, const float *w2_s,
                          const moe_cfg_t *cfg, int T, const void *gamma_next, void *h_out, void *x_next,
                          int32_t *topk_idx, float *topk_w, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace for dense_swiglu_fp8. Host only. */
size_t dense_swiglu_workspace_bytes(int d, int H, int T);

/* Dense SwiGLU FFN of the first block ("Kimi K2 · Dense transformer block",
 * Parameters: SwiGLU MLP; "Kimi K2 · Architecture", config.json
 * intermediate_size): y = down(silu(gate x) * up x) with FP8 weights,
 * x and h quantised 1x128.
 * x [T, d] bf16; w13 [2, H, d] e4m3, w13_s [2, H/128, d/128]; w2 [d, H] e4m3,
 * w2_s [d/128, H/128]; y [T, d] bf16. */
int dense_swiglu_fp8(const void *x, const uint8_t *w13, const float *w13_s,
                     const uint8_t *w2, const float *w2_s, int d, int H, int T, void *y,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Reads and clears the device error word of the current device after
 * synchronising `stream`. MOE_ERR_TIMEOUT if a kernel's bounded wait on an
 * mbarrier gave up since the last check (bits 0x01..0x10, 0x40; its outputs are
 * then invalid); otherwise MOE_ERR_INDEX if an index check failed and the
 * access was skipped (0x20: a GEMM work item outside the schedule; 0x80, the
 * bounds-checked build only: an expert id, a permuted position or an item's
 * rows outside their buffer); MOE_OK if no bit is set. *detail (may be NULL)
 * receives the raw error bits. */
int moe_check_device_error(void *stream, uint32_t *detail);

/* Self-test of the kernels' bounded waits (test only; the pages have no
 * counterpart). Enqueues one small kernel whose two warps wait, through the
 * grouped GEMMs' own wait routine, on a barrier that nothing ever completes: one
 * with limit_ns (1000 .. 1e9 nanoseconds), the other with the kernels' usual 1 s
 * limit. The first gives up after limit_ns, raises the CTA's abort word and sets
 * bit 0x40 of the device error word; the second sees the abort word and returns.
 * Nothing faults or traps and the context stays usable: the following
 * moe_check_device_error returns MOE_ERR_TIMEOUT with detail 0x40, the one after
 * it MOE_OK. MOE_ERR_ARG for a limit outside the range (nothing enqueued). */
int moe_test_wait_timeout(uint64_t limit_ns, void *stream);

/* Description of the calling thread's last error (static storage). */
const char *moe_last_error_string(void);

/* Number of kernels the last successful call enqueued (calling thread). */
int moe_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FP8_H */
