// Host-side interfaces shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#include <utility>

namespace moe {

struct GemmArgs;
enum class Kind;

// Tensor maps of one activation matrix with box heights 16, 32, 64, 96 and 128
// rows (128-byte swizzle; one K block, or a pair of K blocks for the K-pair
// kind): a token tile is loaded with the smallest single box that covers its rows.
constexpr int kActBoxes = 5;
struct ActMaps {
    CUtensorMap box[kActBoxes];
};

// Launches `kernel` on `stream` with programmatic dependent launch allowed: its
// CTAs may be scheduled while the stream's preceding kernel finishes. Every kernel
// of the library starts with pdl_trigger() and calls pdl_wait() before its first
// global-memory access, so the stream order of all memory effects is kept.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Grouped tcgen05 GEMM launch (gemm.cu). Returns a cudaError_t.
cudaError_t launch_grouped_gemm(Kind kind, int bn, const CUtensorMap &map_a, const ActMaps &map_b,
                                GemmArgs &args, int grid, cudaStream_t stream);
// Address of the device error word on the current device (gemm.cu).
cudaError_t device_error_word(unsigned int **ptr);

// Small kernels (kernels.cu).
cudaError_t launch_quant(const void *in, bool bf16, int64_t rows, int cols, uint8_t *q, float *s,
                         bool s_transposed, int num_sms, cudaStream_t stream);
cudaError_t launch_topk(const float *logits, int splits, const float *bias, int T, int E, int k, float scale,
                        int32_t *idx, float *w, float *scores, cudaStream_t stream);
cudaError_t launch_permute(const int32_t *idx, const uint8_t *xq, const float *sx, int T, int k, int S, int E,
                           int d, int tile_a, int tile_b, int32_t *rank, int32_t *cnt, int32_t *counts,
                           int32_t *offsets, int32_t *row_start, int32_t *tile_prefix_a, int32_t *tile_prefix_b,
                           int32_t *counters, int32_t *sorted_tok, int32_t *inv_pos, uint8_t *xq_perm,
                           float *sx_perm, int *launches,
                           cudaStream_t stream, bool copy_rows = true, const void *x_bf16 = nullptr,
                           uint8_t *xq_out = nullptr, float *sx_out = nullptr);
cudaError_t launch_pack_tiles(const uint8_t *w, int64_t groups, int rows, int cols, uint8_t *w_tiled, int num_sms,
                              cudaStream_t stream);
cudaError_t launch_sched(const int32_t *offsets, int E, int S, int T, int k, int tile_a, int tile_b,
                         int32_t *row_start, int32_t *tile_prefix_a, int32_t *tile_prefix_b, int32_t *counters,
                         cudaStream_t stream);
cudaError_t launch_combine(const void *o, const float *w, const int32_t *inv_pos, int T, int k, int S, int d,
                           void *y, cudaStream_t stream);
cudaError_t launch_rmsnorm_quant(const void *h, const void *gamma, float eps, int rows, int cols, void *y,
                                 uint8_t *q, float *s, bool s_transposed, cudaStream_t stream);
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);
cudaError_t launch_combine_residual_rmsnorm(const void *o, const float *w, const int32_t *inv_pos, int T, int k,
                                            int S, int d, const void *residual, const void *gamma, float eps,
                                            void *h_out, void *x_next, cudaStream_t stream);

// Record the calling thread's last error text / launch count (api.cu), for
// entry points defined in other translation units. report_error returns code.
int report_error(int code, const char *msg);
void report_launches(int n);

}  // namespace moe
