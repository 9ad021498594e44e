// Instantiations and launcher of the grouped tcgen05 GEMM.
#include "gemm.cuh"
#include "internal.h"

namespace moe {

__device__ unsigned int g_moe_device_error = 0;

cudaError_t device_error_word(unsigned int **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_moe_device_error);
}

template <Kind KIND>
static cudaError_t launch_kind(const CUtensorMap &map_a, const CUtensorMap &map_b, const GemmArgs &args,
                               int grid, cudaStream_t stream) {
    constexpr size_t smem = gemm_smem_bytes<KIND>();
    static_assert(smem <= 232448, "shared memory budget");
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    grouped_gemm_kernel<KIND><<<grid, kThreads, smem, stream>>>(map_a, map_b, args);
    return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(Kind kind, const CUtensorMap &map_a, const CUtensorMap &map_b, GemmArgs &args,
                                int grid, cudaStream_t stream) {
    cudaError_t e = device_error_word(&args.err);
    if (e != cudaSuccess) return e;
    switch (kind) {
        case Kind::GateUp: return launch_kind<Kind::GateUp>(map_a, map_b, args, grid, stream);
        case Kind::Down: return launch_kind<Kind::Down>(map_a, map_b, args, grid, stream);
        case Kind::Router: return launch_kind<Kind::Router>(map_a, map_b, args, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
