// Launchers of the quantise / top-k / permutation / combine kernels.
#include "kernels.cuh"
#include "internal.h"
#include "gemm.cuh"

namespace moe {

cudaError_t launch_quant(const void *in, bool bf16, int64_t rows, int cols, uint8_t *q, float *s,
                         bool s_transposed, int num_sms, cudaStream_t stream) {
    const int64_t groups = rows * (cols / 128);
    const int threads = 256;   // eight warps, each with 2 * kQuantPairs groups per trip
    int64_t blocks = (groups + 8 * 2 * kQuantPairs - 1) / (8 * 2 * kQuantPairs);
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    const int st = s_transposed ? 1 : 0;
    if (bf16)
        return launch_pdl(quant_1x128_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, in,
                          rows, cols, q, s, st);
    return launch_pdl(quant_1x128_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, in,
                      rows, cols, q, s, st);
}

cudaError_t launch_topk(const float *logits, int splits, const float *bias, int T, int E, int k, float scale,
                        int32_t *idx, float *w, float *scores, cudaStream_t stream) {
    const int threads = 64;   // 2 tokens per block: a 256-token batch spreads over 128 blocks
    const dim3 grid((T + 1) / 2);
    const int nper = (E + 31) / 32;   // E <= 1024
    if (nper <= 4)
        return launch_pdl(topk_kernel<4>, grid, dim3(threads), 0, stream, logits, splits, bias, T, E, k, scale, idx, w,
                          scores);
    if (nper <= 8)
        return launch_pdl(topk_kernel<8>, grid, dim3(threads), 0, stream, logits, splits, bias, T, E, k, scale, idx, w,
                          scores);
    if (nper <= 12)
        return launch_pdl(topk_kernel<12>, grid, dim3(threads), 0, stream, logits, splits, bias, T, E, k, scale, idx, w,
                          scores);
    if (nper <= 16)
        return launch_pdl(topk_kernel<16>, grid, dim3(threads), 0, stream, logits, splits, bias, T, E, k, scale, idx, w,
                          scores);
    return launch_pdl(topk_kernel<32>, grid, dim3(threads), 0, stream, logits, splits, bias, T, E, k, scale, idx, w,
                      scores);
}

cudaError_t launch_permute(const int32_t *idx, const uint8_t *xq, const float *sx, int T, int k, int S, int E,
                           int d, int tile_a, int tile_b, int32_t *rank, int32_t *cnt, int32_t *counts,
                           int32_t *offsets, int32_t *row_start, int32_t *tile_prefix_a, int32_t *tile_prefix_b,
                           int32_t *counters, int32_t *sorted_tok, int32_t *inv_pos, uint8_t *xq_perm,
                           float *sx_perm, int *launches,
                           cudaStream_t stream, bool copy_rows, const void *x_bf16, uint8_t *xq_out,
                           float *sx_out) {
    const int C = (T + 31) / 32;
    const size_t smem = sizeof(uint32_t) * kPermWarps * E;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(perm_rank_kernel, dim3((C + kPermWarps - 1) / kPermWarps), dim3(kPermWarps * 32), smem, stream, idx,
                   T, k, E, C, rank, cnt, err);
    if (e != cudaSuccess) return e;
    e = launch_pdl(perm_scan_kernel, dim3(E), dim3(256), 0, stream, cnt, C, counts);
    if (e != cudaSuccess) return e;
    e = launch_pdl(perm_offsets_kernel, dim3(1), dim3(1024), 0, stream, counts, E, S, T, k, tile_a, tile_b, offsets,
                   row_start, tile_prefix_a, tile_prefix_b, counters);
    if (e != cudaSuccess) return e;
    if (x_bf16) {
        // kScatterUnits 8-element units per thread: 224 threads at d = 7168
        const int per = (d / 8 + kScatterUnits - 1) / kScatterUnits;
        const int threads = (min(1024, max(64, per)) + 31) / 32 * 32;
        e = launch_pdl(perm_quant_scatter_kernel, dim3(T), dim3(threads), 0, stream, idx, rank, cnt, offsets,
                       static_cast<const __nv_bfloat16 *>(x_bf16), T, k, S, E, d, C, sorted_tok, inv_pos, xq_perm,
                       sx_perm, copy_rows ? 1 : 0, xq_out, sx_out, err);
    } else {
        const int threads = min(1024, max(64, d / 16));
        e = launch_pdl(perm_scatter_kernel, dim3(T), dim3(threads), 0, stream, idx, rank, cnt, offsets, xq, sx, T, k,
                       S, E, d, C, sorted_tok, inv_pos, xq_perm, sx_perm, err, copy_rows ? 1 : 0);
    }
    *launches += 4;
    return e;
}

cudaError_t launch_pack_tiles(const uint8_t *w, int64_t groups, int rows, int cols, uint8_t *w_tiled, int num_sms,
                              cudaStream_t stream) {
    const int64_t units = groups * (rows / 128) * (cols / 128) * 1024;
    int64_t blocks = (units + 255) / 256;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pack_tiles_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, w, groups, rows,
                      cols, w_tiled);
}

cudaError_t launch_sched(const int32_t *offsets, int E, int S, int T, int k, int tile_a, int tile_b,
                         int32_t *row_start, int32_t *tile_prefix_a, int32_t *tile_prefix_b, int32_t *counters,
                         cudaStream_t stream) {
    return launch_pdl(sched_kernel, dim3(1), dim3(1024), 0, stream, offsets, E, S, T, k, tile_a, tile_b, row_start,
                      tile_prefix_a, tile_prefix_b, counters);
}

cudaError_t launch_combine(const void *o, const float *w, const int32_t *inv_pos, int T, int k, int S, int d,
                           void *y, cudaStream_t stream) {
    // 128 threads x 8 features per block: a d=7168 token spans 7 blocks
    const int units = d / 8;
    const int threads = 128;
    const dim3 grid(T, (units + threads - 1) / threads);
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    return launch_pdl(combine_kernel, grid, dim3(threads), 0, stream, static_cast<const __nv_bfloat16 *>(o), w,
                      inv_pos, T, k, S, d, static_cast<__nv_bfloat16 *>(y), err);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    return launch_pdl(wait_selftest_kernel, dim3(1), dim3(64), 0, stream, err, limit_ns);
}

// Threads of a one-row-per-CTA kernel: kRowUnits 8-element units each, a multiple
// of 32, at most 1024 (longer rows loop). A d = 7168 row: 224 threads.
static int row_threads(int cols) {
    const int units = cols / 8;
    const int t = ((units + kRowUnits - 1) / kRowUnits + 31) / 32 * 32;
    return t < 1024 ? t : 1024;
}

cudaError_t launch_rmsnorm_quant(const void *h, const void *gamma, float eps, int rows, int cols, void *y,
                                 uint8_t *q, float *s, bool s_transposed, cudaStream_t stream) {
    return launch_pdl(rmsnorm_quant_kernel, dim3(rows), dim3(row_threads(cols)), 0, stream,
                      static_cast<const __nv_bfloat16 *>(h), static_cast<const __nv_bfloat16 *>(gamma), eps, cols,
                      static_cast<__nv_bfloat16 *>(y), q, s, rows, s_transposed ? 1 : 0);
}

cudaError_t launch_combine_residual_rmsnorm(const void *o, const float *w, const int32_t *inv_pos, int T, int k,
                                            int S, int d, const void *residual, const void *gamma, float eps,
                                            void *h_out, void *x_next, cudaStream_t stream) {
    // batched row loads for small batches (a decode step's 256 tokens: 15 -> 10 us);
    // at a 4096-token batch the 64-register variant's occupancy wins (192 vs 204 us)
    const int threads = row_threads(d);
    auto kernel = (threads <= 256 && T <= 512) ? combine_residual_rmsnorm_kernel<true>
                                                : combine_residual_rmsnorm_kernel<false>;
    unsigned int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(T), dim3(threads), 0, stream, static_cast<const __nv_bfloat16 *>(o), w, inv_pos, T,
                      k, S, d, static_cast<const __nv_bfloat16 *>(residual), static_cast<const __nv_bfloat16 *>(gamma),
                      eps, static_cast<__nv_bfloat16 *>(h_out), static_cast<__nv_bfloat16 *>(x_next), err);
}

}  // namespace moe
