// Instantiations and launcher of the grouped tcgen05 GEMM.
#include "gemm.cuh"
#include "internal.h"

namespace moe {

__device__ unsigned int g_moe_device_error = 0;

cudaError_t device_error_word(unsigned int **ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(ptr), g_moe_device_error);
}

template <Kind KIND, int BN>
static cudaError_t launch_kind(const CUtensorMap &map_a, const ActMaps &map_b, const GemmArgs &args,
                               int grid, cudaStream_t stream) {
    constexpr size_t smem = gemm_smem_bytes<KIND, BN>();
    void (*kernel)(const CUtensorMap, const ActMaps, const GemmArgs);
    if constexpr (KindCfg<KIND, BN>::kWide) kernel = grouped_gemm_wide_kernel<KIND, BN>;
    else kernel = grouped_gemm_kernel<KIND, BN>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, dim3(grid), dim3(KindCfg<KIND, BN>::kThreads), smem, stream, map_a, map_b, args);
}

// Token-tile widths compiled per kind: the swap-AB kinds serve decode-sized
// tiles (32 tokens; the router also 128), the token-major kinds 128-token tiles.
template <Kind KIND>
static cudaError_t launch_bn(int bn, const CUtensorMap &map_a, const ActMaps &map_b, const GemmArgs &args,
                             int grid, cudaStream_t stream) {
    constexpr bool kTokenMajor = (KIND == Kind::Down || KIND == Kind::GateUpWide || KIND == Kind::DownWide);
    switch (bn) {
        case 32:
            if constexpr (!kTokenMajor) return launch_kind<KIND, 32>(map_a, map_b, args, grid, stream);
            break;
        case 128:
            if constexpr (kTokenMajor || KIND == Kind::Router)
                return launch_kind<KIND, 128>(map_a, map_b, args, grid, stream);
            break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_grouped_gemm(Kind kind, int bn, const CUtensorMap &map_a, const ActMaps &map_b,
                                GemmArgs &args, int grid, cudaStream_t stream) {
    cudaError_t e = device_error_word(&args.err);
    if (e != cudaSuccess) return e;
    switch (kind) {
        case Kind::GateUp: return launch_bn<Kind::GateUp>(bn, map_a, map_b, args, grid, stream);
        case Kind::Down: return launch_bn<Kind::Down>(bn, map_a, map_b, args, grid, stream);
        case Kind::Router: return launch_bn<Kind::Router>(bn, map_a, map_b, args, grid, stream);
        case Kind::DownPair: return launch_bn<Kind::DownPair>(bn, map_a, map_b, args, grid, stream);
        case Kind::GateUpWide: return launch_bn<Kind::GateUpWide>(bn, map_a, map_b, args, grid, stream);
        case Kind::DownWide: return launch_bn<Kind::DownWide>(bn, map_a, map_b, args, grid, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace moe
