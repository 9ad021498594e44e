// moe_permute_noalloc: the token permutation without a caller workspace.
//
// Some callers cannot hand this library a scratch buffer: for example a plugin
// running inside a host application that owns every device allocation, or a
// serving loop that must not call cudaMalloc once it is running (cudaMalloc
// synchronises the device and can fail when memory is tight). For them this
// entry point keeps the permutation's scratch (per-assignment ranks, per-chunk
// expert counts, the expert counts and the GEMM schedule tables) in one
// file-scope device array of fixed size, which every GPU that loads the
// library holds until the process exits.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "internal.h"
#include "moe_fp8.h"

namespace {

// Limits of the static scratch: T tokens, T * topk assignments, E experts.
constexpr int kMaxTokens = 8192;
constexpr int kMaxAssignments = 65536;
constexpr int kMaxExperts = 1024;
constexpr int kMaxShared = 4;
constexpr int kMaxChunks = kMaxTokens / 32;

// Scratch layout in int32 words; each region starts on a 64-word (256-byte) boundary.
constexpr size_t align64(size_t w) { return (w + 63) / 64 * 64; }
constexpr size_t kRankOff = 0;
constexpr size_t kCntOff = kRankOff + align64(kMaxAssignments);
constexpr size_t kCountsOff = kCntOff + align64(static_cast<size_t>(kMaxExperts) * kMaxChunks);
constexpr size_t kRowStartOff = kCountsOff + align64(kMaxExperts);
constexpr size_t kTileAOff = kRowStartOff + align64(kMaxExperts + kMaxShared + 1);
constexpr size_t kTileBOff = kTileAOff + align64(2 * (kMaxExperts + kMaxShared + 1));
constexpr size_t kCountersOff = kTileBOff + align64(2 * (kMaxExperts + kMaxShared + 1));
constexpr size_t kScratchWords = kCountersOff + 64;   // about 1.3 MB

}  // namespace

static __device__ __align__(256) int32_t g_permute_scratch[kScratchWords];

namespace {

// Device address of the scratch array on the current device, looked up once
// per device and kept for the process (after a cudaDeviceReset the module, and
// the array with it, may load elsewhere: calls after one are not supported). The
// host-side name g_permute_scratch is only a stand-in for the address.
int32_t *scratch_on_current_device() {
    static std::mutex mu;
    static int32_t *addr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return nullptr;
        addr[dev] = static_cast<int32_t *>(p);
    }
    return addr[dev];
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t *topk_idx, const uint8_t *xq, const float *sx,
                                   const moe_cfg_t *cfg, int T, int32_t *offsets, int32_t *sorted_tok,
                                   int32_t *inv_pos, uint8_t *xq_perm, float *sx_perm, void *stream) {
    moe::report_launches(0);
    if (!cfg) return moe::report_error(MOE_ERR_ARG, "cfg is NULL");
    if (cfg->d <= 0 || cfg->d % 128 || cfg->d > 16384)
        return moe::report_error(MOE_ERR_UNSUPPORTED, "d must be a multiple of 128 in [128, 16384]");
    if (cfg->topk < 1 || cfg->topk > 32 || cfg->E < cfg->topk || cfg->E > kMaxExperts || cfg->n_shared < 0 ||
        cfg->n_shared > kMaxShared)
        return moe::report_error(MOE_ERR_UNSUPPORTED, "topk, E or n_shared outside the supported range");
    if (T < 0) return moe::report_error(MOE_ERR_ARG, "T is negative");
    if (T > kMaxTokens || static_cast<long long>(T) * cfg->topk > kMaxAssignments) {
        char msg[160];
        snprintf(msg, sizeof(msg),
                 "moe_permute_noalloc handles at most %d tokens and %d token-expert assignments "
                 "(got T=%d, topk=%d); use moe_permute with a workspace",
                 kMaxTokens, kMaxAssignments, T, cfg->topk);
        return moe::report_error(MOE_ERR_UNSUPPORTED, msg);
    }
    if (T == 0) return MOE_OK;
    if (!aligned16(topk_idx) || !aligned16(xq) || !aligned16(sx) || !aligned16(offsets) || !aligned16(sorted_tok) ||
        !aligned16(inv_pos) || !aligned16(xq_perm) || !aligned16(sx_perm))
        return moe::report_error(MOE_ERR_ARG, "a pointer is NULL or not 16-byte aligned");
    int32_t *scratch = scratch_on_current_device();
    if (!scratch) return moe::report_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the permutation scratch failed");
    int n = 0;
    const cudaError_t e = moe::launch_permute(
        topk_idx, xq, sx, T, cfg->topk, cfg->n_shared, cfg->E, cfg->d, 64, 64, scratch + kRankOff,
        scratch + kCntOff, scratch + kCountsOff, offsets, scratch + kRowStartOff, scratch + kTileAOff,
        scratch + kTileBOff, scratch + kCountersOff, sorted_tok, inv_pos, xq_perm, sx_perm, &n,
        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, cudaGetErrorString(e));
    moe::report_launches(n);
    return MOE_OK;
}
