// C ABI of the routed FP8 MoE FFN forward (declared in include/moe_fp8.h).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gemm.cuh"
#include "internal.h"
#include "moe_fp8.h"

using namespace moe;

namespace {

thread_local char t_err[512] = "no error";
thread_local int t_launches = 0;

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define MOE_CUDA(call, what)                            \
    do {                                                \
        cudaError_t e_ = (call);                        \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

#define MOE_CHECK(expr)             \
    do {                            \
        int s_ = (expr);            \
        if (s_ != MOE_OK) return s_; \
    } while (0)

constexpr int kMaxT = 1 << 20;

int check_cfg(const moe_cfg_t *c) {
    if (!c) return fail(MOE_ERR_ARG, "cfg is NULL");
    if (c->d <= 0 || c->d % 128 || c->d > 16384)
        return fail(MOE_ERR_UNSUPPORTED, "d=%d must be a multiple of 128 in [128, 16384]", c->d);
    if (c->H <= 0 || c->H % 128 || c->H > 65536)
        return fail(MOE_ERR_UNSUPPORTED, "H=%d must be a multiple of 128 in [128, 65536]", c->H);
    if (c->topk < 1 || c->topk > 32) return fail(MOE_ERR_UNSUPPORTED, "topk=%d must be in [1, 32]", c->topk);
    if (c->E < c->topk || c->E > 1024)
        return fail(MOE_ERR_UNSUPPORTED, "E=%d must be in [topk, 1024]", c->E);
    if (c->n_shared < 0 || c->n_shared > 4) return fail(MOE_ERR_UNSUPPORTED, "n_shared=%d must be in [0, 4]", c->n_shared);
    if (!std::isfinite(c->route_scale)) return fail(MOE_ERR_ARG, "route_scale is not finite");
    if (c->w_tiled != 0 && c->w_tiled != 1) return fail(MOE_ERR_ARG, "w_tiled=%d must be 0 or 1", c->w_tiled);
    return MOE_OK;
}

int check_T(int T) {
    if (T < 0) return fail(MOE_ERR_ARG, "T=%d is negative", T);
    if (T > kMaxT) return fail(MOE_ERR_UNSUPPORTED, "T=%d exceeds %d", T, kMaxT);
    return MOE_OK;
}

int check_ptr(const void *p, const char *name) {
    if (!p) return fail(MOE_ERR_ARG, "%s is NULL", name);
    if (reinterpret_cast<uintptr_t>(p) & 15) return fail(MOE_ERR_ARG, "%s is not 16-byte aligned", name);
    return MOE_OK;
}

int num_sms() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// Token-tile width of the expert GEMMs: expected rows per routed expert k*T/E
// decides.
//
// Decode regime (<= 12 expected rows per expert): 32-token tiles in the swap-AB
// kernels (weight rows on the MMA M dimension), the fused gate/up kernel and the
// two-block down kernel, which stream the weights at the HBM rate. Beyond it:
// 128-token tiles in the token-major kernels (tokens on M): gate/up items hold the
// gate and up blocks of 128 features (N = 256) with the fused SiLU*mul and h
// quantisation; down items hold two adjacent 128-row output blocks.
bool decode_regime(const moe_cfg_t &c, int T) { return static_cast<double>(c.topk) * T / c.E <= 12.0; }

int expert_bn(const moe_cfg_t &c, int T) { return decode_regime(c, T) ? 32 : 128; }

// The decode down projection pairs two 128-row weight blocks per item, which
// needs an even number of them; otherwise the token-major kernel runs.
bool down_pair(const moe_cfg_t &c, int T) { return decode_regime(c, T) && (c.d / 128) % 2 == 0; }

int down_bn(const moe_cfg_t &c, int T) { return down_pair(c, T) ? 32 : 128; }

int router_bn(int T) { return T <= 512 ? 32 : 128; }

// Deterministic split-K of the router GEMM: the split count (1..4, at least 4 K
// blocks of 64 elements per split, at most two waves of items) that minimises
// waves x K blocks per split, the smaller count on ties. Each split adds a plane
// of partial logits that the top-k kernel reads in turn, so few splits pay: at a
// 256-token batch 4 splits (one wave of 96 items) route 4.5 us faster than 6
// (144 items). Past 512 tokens an item holds every 128-expert block (up to three),
// so a 4096-token batch runs 32 token tiles x 4 splits in one wave.
int router_splits(const moe_cfg_t &c, int T) {
    const int bn = router_bn(T);
    const int blocks = (c.E + 127) / 128;
    const int items = std::max(1, ((T + bn - 1) / bn) * ((bn == 128 && blocks <= 3) ? 1 : blocks));
    const int num_kb = c.d / 64;
    const int max_s = std::max(1, std::min(4, num_kb / 4));
    const int sms = 148;   // work items per wave (the GPU's SMs less a small margin)
    int best = 1;
    long best_cost = -1;
    // splits only while the split items fit two waves: beyond that each split adds a
    // plane of partial logits for the top-k kernel to read and nothing to balance
    for (int s = 1; s <= max_s && (s == 1 || items * s <= 2 * sms); ++s) {
        const long waves = (static_cast<long>(items) * s + sms - 1) / sms;
        const long cost = waves * ((num_kb + s - 1) / s);
        if (best_cost < 0 || cost < best_cost) { best_cost = cost; best = s; }
    }
    return best;
}

// ---------------------------------------------------------------- workspace

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Carver {
    uint8_t *base;
    size_t off = 0;
    template <typename P> P *take(size_t bytes) {
        off = align_up(off, 1024);
        P *p = base ? reinterpret_cast<P *>(base + off) : nullptr;
        off += bytes;
        return p;
    }
};

struct LayerWs {
    float *logits;
    uint8_t *xq;
    float *sx;
    int32_t *idx;
    float *w;
    int32_t *rank, *cnt, *counts, *offsets, *sorted_tok, *inv_pos, *row_start, *tile_prefix, *tile_prefix_dn;
    int32_t *counters;  // [2] dynamic scheduler counters of the gate/up and down GEMMs
    uint8_t *xq_perm;
    float *sx_perm;
    uint8_t *hq;
    float *hs_t;
    __nv_bfloat16 *o;
    __nv_bfloat16 *xn;   // moe_block_ffn_forward: the post-attention RMSNorm of h (bf16)
    size_t bytes;
};

LayerWs carve_layer(const moe_cfg_t &c, int T, void *base) {
    Carver cv{static_cast<uint8_t *>(base)};
    const size_t Tz = static_cast<size_t>(T);
    const size_t R = static_cast<size_t>(c.topk + c.n_shared) * Tz;
    const size_t C = (Tz + 31) / 32;
    const size_t G = static_cast<size_t>(c.E + c.n_shared);
    LayerWs w{};
    w.logits = cv.take<float>(static_cast<size_t>(router_splits(c, T)) * Tz * c.E * 4);
    w.xq = cv.take<uint8_t>(Tz * c.d);
    w.sx = cv.take<float>(Tz * (c.d / 128) * 4);
    w.idx = cv.take<int32_t>(Tz * c.topk * 4);
    w.w = cv.take<float>(Tz * c.topk * 4);
    w.rank = cv.take<int32_t>(Tz * c.topk * 4);
    w.cnt = cv.take<int32_t>(std::max<size_t>(C, 1) * c.E * 4);
    w.counts = cv.take<int32_t>(static_cast<size_t>(c.E) * 4);
    w.offsets = cv.take<int32_t>(static_cast<size_t>(c.E + 1) * 4);
    w.sorted_tok = cv.take<int32_t>(Tz * c.topk * 4);
    w.inv_pos = cv.take<int32_t>(Tz * c.topk * 4);
    w.row_start = cv.take<int32_t>((G + 1) * 4);
    // [2][G+1]: all groups' tiles, then those of the groups of two or more tiles
    w.tile_prefix = cv.take<int32_t>(2 * (G + 1) * 4);
    w.tile_prefix_dn = cv.take<int32_t>(2 * (G + 1) * 4);
    w.counters = cv.take<int32_t>(2 * 4);
    w.xq_perm = cv.take<uint8_t>(R * c.d);
    w.sx_perm = cv.take<float>(R * (c.d / 128) * 4);
    w.hq = cv.take<uint8_t>(R * c.H);
    w.hs_t = cv.take<float>(R * (c.H / 128) * 4);
    w.o = cv.take<__nv_bfloat16>(R * c.d * 2);
    w.xn = cv.take<__nv_bfloat16>(Tz * c.d * 2);
    w.bytes = align_up(cv.off, 1024);
    return w;
}

int check_ws(const void *ws, size_t have, size_t need) {
    if (have < need) return fail(MOE_ERR_ARG, "workspace of %zu bytes is smaller than the %zu needed", have, need);
    return check_ptr(ws, "workspace");
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2D row-major matrix [rows, cols] of 1- or 2-byte elements; box = 128 bytes x box_rows,
// 128-byte swizzle (the canonical K-major layout of the MMA operands).
int make_map(CUtensorMap *m, const void *ptr, int elem_bytes, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const CUtensorMapDataType dt = elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * elem_bytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MOE_OK;
}

// The gate/up weights [G][2][H][d] as a 3D map (x = d, y = H, z = 2G) whose box
// {128 bytes, 128 rows, 2} holds one row block of gate_proj and the same rows of
// up_proj: one request per K block.
int make_map_gateup(CUtensorMap *m, const void *ptr, uint64_t G, uint64_t H, uint64_t d) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {d, H, 2 * G};
    cuuint64_t strides[2] = {d, H * d};
    cuuint32_t box[3] = {128, 128, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (3D) failed (%d)", static_cast<int>(r));
    return MOE_OK;
}

// Activation maps with box heights 16, 32, 64, 96 and 128 rows.
int make_act_maps(ActMaps *m, const void *ptr, int elem_bytes, uint64_t rows, uint64_t cols) {
    const uint32_t heights[kActBoxes] = {16, 32, 64, 96, 128};
    for (int i = 0; i < kActBoxes; ++i) MOE_CHECK(make_map(&m->box[i], ptr, elem_bytes, rows, cols, heights[i]));
    return MOE_OK;
}

// An FP8 matrix [rows][cols] viewed as 3D (x = byte inside a 128-byte K block,
// y = row, z = K block) so that one box {128, box_rows, 2} holds two consecutive
// K blocks of box_rows rows: in shared memory, two 128-byte-swizzled K-major
// tiles one after the other. A box that starts at the last K block of an odd
// count reads zeros for the second.
int make_map_kpair(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[3] = {128, rows, cols / 128};
    cuuint64_t strides[2] = {cols, 128};
    cuuint32_t box[3] = {128, box_rows, 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (K pairs) failed (%d)", static_cast<int>(r));
    return MOE_OK;
}

int make_act_maps_kpair(ActMaps *m, const void *ptr, uint64_t rows, uint64_t cols) {
    const uint32_t heights[kActBoxes] = {16, 32, 64, 96, 128};
    for (int i = 0; i < kActBoxes; ++i) MOE_CHECK(make_map_kpair(&m->box[i], ptr, rows, cols, heights[i]));
    return MOE_OK;
}

// The tiled weight layout [groups][rows/128][cols/128][128][128] as a map whose two
// innermost dimensions are one 128 x 128 tile (x = the 128 bytes of a tile row,
// y = its 128 rows, z = the K block, w = the row block over all groups).
// pair_rows: box {128, 128, 1, 2}, two row blocks of a K block (256-row items);
// otherwise box {128, 128, 2, 1}, two K blocks of a row block (the K-pair kind).
int make_map_tiled_w2(CUtensorMap *m, const void *ptr, uint64_t groups, uint64_t rows, uint64_t cols,
                      bool pair_rows) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[4] = {128, 128, cols / 128, groups * (rows / 128)};
    cuuint64_t strides[3] = {128, 16384, 16384 * (cols / 128)};
    cuuint32_t box[4] = {128, 128, pair_rows ? 1u : 2u, pair_rows ? 2u : 1u};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (tiled 4D) failed (%d)", static_cast<int>(r));
    return MOE_OK;
}

// The tiled gate/up weights [2G][H/128][d/128][128][128] as a 5D map (x, y = a
// tile's bytes and rows, z = K block, w = row block, v = 2g + gate/up) whose box
// {128, 128, 1, 1, 2} holds a gate tile and the up tile of the same rows.
int make_map_tiled_gateup(CUtensorMap *m, const void *ptr, uint64_t G, uint64_t H, uint64_t d) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    cuuint64_t dims[5] = {128, 128, d / 128, H / 128, 2 * G};
    cuuint64_t strides[4] = {128, 16384, 16384 * (d / 128), 16384 * (d / 128) * (H / 128)};
    cuuint32_t box[5] = {128, 128, 1, 1, 2};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (tiled 5D) failed (%d)", static_cast<int>(r));
    return MOE_OK;
}

int gateup_map(CUtensorMap *m, const void *w13, const moe_cfg_t &c, uint64_t G) {
    return c.w_tiled ? make_map_tiled_gateup(m, w13, G, c.H, c.d) : make_map_gateup(m, w13, G, c.H, c.d);
}

// ---------------------------------------------------------------- steps

int route_impl(const void *x, const void *wg, const float *bias, const moe_cfg_t &c, int T, int32_t *idx,
               float *w, float *scores, float *logits, cudaStream_t st) {
    const int bn = router_bn(T);
    CUtensorMap ma;
    ActMaps mb;
    MOE_CHECK(make_map(&ma, wg, 2, c.E, c.d, kBM));
    MOE_CHECK(make_act_maps(&mb, x, 2, T, c.d));
    GemmArgs a{};
    a.G = 1;
    a.num_kb = c.d / 64;
    a.num_mb = (c.E + kBM - 1) / kBM;
    a.total_rows = T;
    a.single_rows = T;
    a.logits = logits;
    a.n_valid = c.E;
    a.k_splits = router_splits(c, T);
    if (bn == 128 && a.num_mb <= 3) {
        // each item covers every expert block, so the token tile is read once instead
        // of once per block: the 16,384-token route 181 -> 152 us on one GB300
        a.a_tiles = a.num_mb;
        a.num_mb = 1;
    }
    const int items = a.num_mb * ((T + bn - 1) / bn) * a.k_splits;
    MOE_CUDA(launch_grouped_gemm(Kind::Router, bn, ma, mb, a, std::min(items, num_sms()), st), "router GEMM launch");
    MOE_CUDA(launch_topk(logits, a.k_splits, bias, T, c.E, c.topk, c.route_scale, idx, w, scores, st), "top-k launch");
    t_launches += 2;
    return MOE_OK;
}

// Activation rows gathered by the decode gate/up kernel itself (instead of the
// permuted copy): the unpermuted codes [T][d] and scales [T][d/128] and sorted_tok.
struct Gather {
    const uint8_t *xq;
    const float *sx;
    const int32_t *sorted_tok;
};

// L2 prefetch of the decode GEMMs' first-round items on the tiled weights, bytes per
// weight run: 152 items x 2 runs x 320 KB = 97 MB of gate/up weights, under L2's
// 129 MB; 152 x 512 KB = 78 MB of down weights. HBM idles while the routing and the
// permutation run: an A/B on one GB300 gave the decode step 2.299 -> 2.284 ms
constexpr uint64_t kGateUpPrefetch = 320 * 1024;
constexpr uint64_t kDownPrefetch = 512 * 1024;

int gateup_impl(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets, const uint8_t *w13,
                const float *w13_s, const moe_cfg_t &c, int T, uint8_t *hq, float *hs, const LayerWs &ws,
                bool run_sched, cudaStream_t st, const Gather *gather = nullptr) {
    const int G = c.E + c.n_shared;
    const int64_t R = static_cast<int64_t>(c.topk + c.n_shared) * T;
    const int bn = expert_bn(c, T);
    if (run_sched) {
        MOE_CUDA(launch_sched(offsets, c.E, c.n_shared, T, c.topk, bn, down_bn(c, T), ws.row_start, ws.tile_prefix,
                              ws.tile_prefix_dn, ws.counters, st),
                 "schedule launch");
        t_launches += 1;
    }
    CUtensorMap m13;
    ActMaps mx;
    MOE_CHECK(gateup_map(&m13, w13, c, G));
    MOE_CHECK(make_act_maps(&mx, xq_perm, 1, R, c.d));
    GemmArgs gu{};
    gu.G = G;
    gu.num_kb = c.d / 128;
    gu.num_mb = c.H / 128;
    gu.total_rows = static_cast<int>(R);
    gu.single_rows = -1;
    gu.row_start = ws.row_start;
    gu.tile_prefix = ws.tile_prefix;
    gu.act_scale_t = sx_perm;
    gu.w_scale = w13_s;
    gu.a_rows_per_group = 2 * c.H;
    gu.w_tiled = c.w_tiled;
    if (decode_regime(c, T)) {
        // fused gate/up + SiLU*mul + h quantisation; items handed out by the global
        // counter (one atomic per 56-K-block item), so the CTAs that finish early
        // share the last partial round
        gu.hq = hq;
        gu.hs_t = hs;
        gu.item_counter = ws.counters;
        if (gather) {
            gu.gather_rows = gather->xq;
            gu.gather_scales = gather->sx;
            gu.row_token = gather->sorted_tok;
            gu.n_routed = c.topk * T;
            gu.n_tok = T;
        }
        if (c.w_tiled) {
            // the first round's items: their gate and up runs, kGateUpPrefetch bytes each
            gu.pf_base = w13;
            gu.pf_group_bytes = 2ull * c.H * c.d;
            gu.pf_item_bytes = 128ull * c.d;
            gu.pf_second = static_cast<uint64_t>(c.H) * c.d;
            gu.pf_len = static_cast<uint32_t>(std::min<uint64_t>(kGateUpPrefetch, 128ull * c.d));
            gu.pf_items = c.H / 128;
        }
        MOE_CUDA(launch_grouped_gemm(Kind::GateUp, bn, m13, mx, gu, num_sms(), st), "gate/up GEMM launch");
        t_launches += 1;
        return MOE_OK;
    }
    // 128-token tiles, token-major: the gate and up blocks of 128 features per
    // item (N = 256) with the fused SiLU*mul and h quantisation
    gu.hq = hq;
    gu.hs_t = hs;
    gu.item_counter = ws.counters;
    // the items of multi-tile experts (tensor-bound) and one-tile experts (weight
    // streaming) interleaved: skewed batch 4.65 -> 4.48 ms, prefill 1.88 -> 1.85 ms
    gu.interleave = 1;
    MOE_CUDA(launch_grouped_gemm(Kind::GateUpWide, bn, m13, mx, gu, num_sms(), st), "gate/up GEMM launch");
    t_launches += 1;
    return MOE_OK;
}

int down_impl(const uint8_t *hq, const float *hs, const int32_t *offsets, const uint8_t *w2, const float *w2_s,
              const moe_cfg_t &c, int T, void *o, const LayerWs &ws, bool run_sched, cudaStream_t st) {
    const int G = c.E + c.n_shared;
    const int64_t R = static_cast<int64_t>(c.topk + c.n_shared) * T;
    const int bn = down_bn(c, T);
    if (run_sched) {
        MOE_CUDA(launch_sched(offsets, c.E, c.n_shared, T, c.topk, expert_bn(c, T), bn, ws.row_start,
                              ws.tile_prefix, ws.tile_prefix_dn, ws.counters, st),
                 "schedule launch");
        t_launches += 1;
    }
    CUtensorMap m2;
    ActMaps mh;
    MOE_CHECK(make_map(&m2, w2, 1, static_cast<uint64_t>(G) * c.d, c.H, kBM));
    MOE_CHECK(make_act_maps(&mh, hq, 1, R, c.H));
    GemmArgs dn{};
    dn.G = G;
    dn.num_kb = c.H / 128;
    dn.num_mb = c.d / 128;
    dn.total_rows = static_cast<int>(R);
    dn.single_rows = -1;
    dn.row_start = ws.row_start;
    dn.tile_prefix = ws.tile_prefix_dn;
    dn.item_counter = ws.counters + 1;   // items handed out by the global counter
    dn.act_scale_t = hs;
    dn.w_scale = w2_s;
    dn.a_rows_per_group = c.d;
    dn.out = static_cast<__nv_bfloat16 *>(o);
    dn.w_tiled = c.w_tiled;
    if (down_pair(c, T)) {
        // decode: two adjacent 128-row blocks per item, one 256-row box (32 KB of
        // weights per K block and request)
        if (c.w_tiled) MOE_CHECK(make_map_tiled_w2(&m2, w2, G, c.d, c.H, true));
        else MOE_CHECK(make_map(&m2, w2, 1, static_cast<uint64_t>(G) * c.d, c.H, 2 * kBM));
        dn.num_mb = c.d / 256;
        if (c.w_tiled && kDownPrefetch > 0) {
            // the first round's items: their 256-row runs, kDownPrefetch bytes of each
            dn.pf_base = w2;
            dn.pf_group_bytes = static_cast<uint64_t>(c.d) * c.H;
            dn.pf_item_bytes = 256ull * c.H;
            dn.pf_second = 0;
            dn.pf_len = static_cast<uint32_t>(std::min<uint64_t>(kDownPrefetch, 256ull * c.H));
            dn.pf_items = c.d / 256;
        }
        MOE_CUDA(launch_grouped_gemm(Kind::DownPair, bn, m2, mh, dn, num_sms(), st), "down GEMM launch");
    } else if ((c.d / 128) % 2 == 0) {
        // 128-token tiles, token-major, two 128-row blocks per item (N = 256)
        if (c.w_tiled) MOE_CHECK(make_map_tiled_w2(&m2, w2, G, c.d, c.H, true));
        else MOE_CHECK(make_map(&m2, w2, 1, static_cast<uint64_t>(G) * c.d, c.H, 2 * kBM));
        dn.num_mb = c.d / 256;
        // on the tiled weights the multi-tile and one-tile experts' items interleaved, as
        // in the gate/up GEMM (skewed down 2.835 -> 2.70 ms, prefill 0.980 -> 0.959 ms);
        // on the row-major weights the plain order, 3% faster there
        dn.interleave = c.w_tiled;
        MOE_CUDA(launch_grouped_gemm(Kind::DownWide, bn, m2, mh, dn, num_sms(), st), "down GEMM launch");
    } else {
        if (c.w_tiled) MOE_CHECK(make_map_tiled_w2(&m2, w2, G, c.d, c.H, false));
        else MOE_CHECK(make_map_kpair(&m2, w2, static_cast<uint64_t>(G) * c.d, c.H, kBM));
        MOE_CHECK(make_act_maps_kpair(&mh, hq, R, c.H));
        MOE_CUDA(launch_grouped_gemm(Kind::Down, bn, m2, mh, dn, num_sms(), st), "down GEMM launch");
    }
    t_launches += 1;
    return MOE_OK;
}

int experts_impl(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets, const uint8_t *w13,
                 const float *w13_s, const uint8_t *w2, const float *w2_s, const moe_cfg_t &c, int T, void *o,
                 const LayerWs &ws, bool run_sched, cudaStream_t st, const Gather *gather = nullptr) {
    MOE_CHECK(gateup_impl(xq_perm, sx_perm, offsets, w13, w13_s, c, T, ws.hq, ws.hs_t, ws, run_sched, st, gather));
    return down_impl(ws.hq, ws.hs_t, offsets, w2, w2_s, c, T, o, ws, false, st);
}

}  // namespace

namespace moe {
int report_error(int code, const char *msg) { return fail(code, "%s", msg); }
void report_launches(int n) { t_launches = n; }
}  // namespace moe

extern "C" {

int64_t moe_permuted_rows(const moe_cfg_t *cfg, int T) {
    if (!cfg || T < 0) return 0;
    return static_cast<int64_t>(cfg->topk + cfg->n_shared) * T;
}

size_t moe_workspace_bytes(const moe_cfg_t *cfg, int T) {
    if (check_cfg(cfg) != MOE_OK || check_T(T) != MOE_OK) return 0;
    return carve_layer(*cfg, T, nullptr).bytes;
}

int moe_quant_fp8_1x128(const void *in, int in_is_bf16, int64_t rows, int cols, uint8_t *q, float *s,
                        int s_transposed, void *stream) {
    t_launches = 0;
    if (rows < 0) return fail(MOE_ERR_ARG, "rows=%lld is negative", static_cast<long long>(rows));
    if (cols <= 0 || cols % 128) return fail(MOE_ERR_UNSUPPORTED, "cols=%d must be a positive multiple of 128", cols);
    if (rows == 0) return MOE_OK;
    MOE_CHECK(check_ptr(in, "in"));
    MOE_CHECK(check_ptr(q, "q"));
    if (!s) return fail(MOE_ERR_ARG, "s is NULL");
    MOE_CUDA(launch_quant(in, in_is_bf16 != 0, rows, cols, q, s, s_transposed != 0, num_sms(),
                          static_cast<cudaStream_t>(stream)),
             "quantise launch");
    t_launches = 1;
    return MOE_OK;
}

int moe_pack_weights_fp8(const uint8_t *w, int64_t groups, int rows, int cols, uint8_t *w_tiled, void *stream) {
    t_launches = 0;
    if (groups < 0) return fail(MOE_ERR_ARG, "groups=%lld is negative", static_cast<long long>(groups));
    if (rows <= 0 || rows % 128 || cols <= 0 || cols % 128)
        return fail(MOE_ERR_UNSUPPORTED, "rows=%d and cols=%d must be positive multiples of 128", rows, cols);
    if (groups == 0) return MOE_OK;
    MOE_CHECK(check_ptr(w, "w"));
    MOE_CHECK(check_ptr(w_tiled, "w_tiled"));
    const uint64_t bytes = static_cast<uint64_t>(groups) * rows * cols;
    const uintptr_t a = reinterpret_cast<uintptr_t>(w), b = reinterpret_cast<uintptr_t>(w_tiled);
    if (a < b + bytes && b < a + bytes) return fail(MOE_ERR_ARG, "w and w_tiled overlap");
    MOE_CUDA(launch_pack_tiles(w, groups, rows, cols, w_tiled, num_sms(), static_cast<cudaStream_t>(stream)),
             "weight tiling launch");
    t_launches = 1;
    return MOE_OK;
}

int moe_route(const void *x, const void *w_gate, const float *bias, const moe_cfg_t *cfg, int T, int32_t *topk_idx,
              float *topk_w, float *scores, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(x, "x"));
    MOE_CHECK(check_ptr(w_gate, "w_gate"));
    if (!bias) return fail(MOE_ERR_ARG, "bias is NULL");
    MOE_CHECK(check_ptr(topk_idx, "topk_idx"));
    MOE_CHECK(check_ptr(topk_w, "topk_w"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    return route_impl(x, w_gate, bias, *cfg, T, topk_idx, topk_w, scores, ws.logits, static_cast<cudaStream_t>(stream));
}

int moe_permute(const int32_t *topk_idx, const uint8_t *xq, const float *sx, const moe_cfg_t *cfg, int T,
                int32_t *offsets, int32_t *sorted_tok, int32_t *inv_pos, uint8_t *xq_perm, float *sx_perm,
                void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(topk_idx, "topk_idx"));
    MOE_CHECK(check_ptr(xq, "xq"));
    MOE_CHECK(check_ptr(sx, "sx"));
    MOE_CHECK(check_ptr(offsets, "offsets"));
    MOE_CHECK(check_ptr(sorted_tok, "sorted_tok"));
    MOE_CHECK(check_ptr(inv_pos, "inv_pos"));
    MOE_CHECK(check_ptr(xq_perm, "xq_perm"));
    MOE_CHECK(check_ptr(sx_perm, "sx_perm"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    int n = 0;
    MOE_CUDA(launch_permute(topk_idx, xq, sx, T, cfg->topk, cfg->n_shared, cfg->E, cfg->d, expert_bn(*cfg, T),
                            down_bn(*cfg, T), ws.rank, ws.cnt, ws.counts, offsets, ws.row_start, ws.tile_prefix,
                            ws.tile_prefix_dn, ws.counters, sorted_tok, inv_pos, xq_perm, sx_perm, &n,
                            static_cast<cudaStream_t>(stream)),
             "permutation launch");
    t_launches = n;
    return MOE_OK;
}

int moe_quant_permute_fp8(const int32_t *topk_idx, const void *x, const moe_cfg_t *cfg, int T, int32_t *offsets,
                          int32_t *sorted_tok, int32_t *inv_pos, uint8_t *xq_perm, float *sx_perm, void *workspace,
                          size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(topk_idx, "topk_idx"));
    MOE_CHECK(check_ptr(x, "x"));
    MOE_CHECK(check_ptr(offsets, "offsets"));
    MOE_CHECK(check_ptr(sorted_tok, "sorted_tok"));
    MOE_CHECK(check_ptr(inv_pos, "inv_pos"));
    MOE_CHECK(check_ptr(xq_perm, "xq_perm"));
    MOE_CHECK(check_ptr(sx_perm, "sx_perm"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    int n = 0;
    MOE_CUDA(launch_permute(topk_idx, nullptr, nullptr, T, cfg->topk, cfg->n_shared, cfg->E, cfg->d,
                            expert_bn(*cfg, T), down_bn(*cfg, T), ws.rank, ws.cnt, ws.counts, offsets, ws.row_start,
                            ws.tile_prefix, ws.tile_prefix_dn, ws.counters, sorted_tok, inv_pos, xq_perm, sx_perm, &n,
                            static_cast<cudaStream_t>(stream), true, x),
             "quantise + permutation launch");
    t_launches = n;
    return MOE_OK;
}

int moe_expert_gemm_fp8(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets, const uint8_t *w13,
                        const float *w13_s, const uint8_t *w2, const float *w2_s, const moe_cfg_t *cfg, int T,
                        void *o, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(xq_perm, "xq_perm"));
    MOE_CHECK(check_ptr(sx_perm, "sx_perm"));
    MOE_CHECK(check_ptr(offsets, "offsets"));
    MOE_CHECK(check_ptr(w13, "w13"));
    MOE_CHECK(check_ptr(w13_s, "w13_s"));
    MOE_CHECK(check_ptr(w2, "w2"));
    MOE_CHECK(check_ptr(w2_s, "w2_s"));
    MOE_CHECK(check_ptr(o, "o"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    return experts_impl(xq_perm, sx_perm, offsets, w13, w13_s, w2, w2_s, *cfg, T, o, ws, true,
                        static_cast<cudaStream_t>(stream));
}

int moe_expert_gateup_fp8(const uint8_t *xq_perm, const float *sx_perm, const int32_t *offsets,
                          const uint8_t *w13, const float *w13_s, const moe_cfg_t *cfg, int T, uint8_t *hq,
                          float *hs, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(xq_perm, "xq_perm"));
    MOE_CHECK(check_ptr(sx_perm, "sx_perm"));
    MOE_CHECK(check_ptr(offsets, "offsets"));
    MOE_CHECK(check_ptr(w13, "w13"));
    MOE_CHECK(check_ptr(w13_s, "w13_s"));
    MOE_CHECK(check_ptr(hq, "hq"));
    MOE_CHECK(check_ptr(hs, "hs"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    return gateup_impl(xq_perm, sx_perm, offsets, w13, w13_s, *cfg, T, hq, hs, ws, true,
                       static_cast<cudaStream_t>(stream));
}

int moe_expert_down_fp8(const uint8_t *hq, const float *hs, const int32_t *offsets, const uint8_t *w2,
                        const float *w2_s, const moe_cfg_t *cfg, int T, void *o, void *workspace,
                        size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(hq, "hq"));
    MOE_CHECK(check_ptr(hs, "hs"));
    MOE_CHECK(check_ptr(offsets, "offsets"));
    MOE_CHECK(check_ptr(w2, "w2"));
    MOE_CHECK(check_ptr(w2_s, "w2_s"));
    MOE_CHECK(check_ptr(o, "o"));
    const LayerWs need = carve_layer(*cfg, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(*cfg, T, workspace);
    return down_impl(hq, hs, offsets, w2, w2_s, *cfg, T, o, ws, true, static_cast<cudaStream_t>(stream));
}

int moe_combine(const void *o, const float *topk_w, const int32_t *inv_pos, const moe_cfg_t *cfg, int T, void *y,
                void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(o, "o"));
    MOE_CHECK(check_ptr(topk_w, "topk_w"));
    MOE_CHECK(check_ptr(inv_pos, "inv_pos"));
    MOE_CHECK(check_ptr(y, "y"));
    MOE_CUDA(launch_combine(o, topk_w, inv_pos, T, cfg->topk, cfg->n_shared, cfg->d, y,
                            static_cast<cudaStream_t>(stream)),
             "combine launch");
    t_launches = 1;
    return MOE_OK;
}

int moe_rmsnorm_quant_fp8(const void *h, const void *gamma, float eps, int rows, int cols, void *y, uint8_t *q,
                          float *s, int s_transposed, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_T(rows));
    if (cols <= 0 || cols % 128 || cols > 65536)
        return fail(MOE_ERR_UNSUPPORTED, "cols=%d must be a positive multiple of 128 (at most 65536)", cols);
    if (!(eps >= 0.f)) return fail(MOE_ERR_ARG, "eps must be a non-negative number");
    if (rows == 0) return MOE_OK;
    MOE_CHECK(check_ptr(h, "h"));
    MOE_CHECK(check_ptr(gamma, "gamma"));
    if (y) MOE_CHECK(check_ptr(y, "y"));
    MOE_CHECK(check_ptr(q, "q"));
    if (!s) return fail(MOE_ERR_ARG, "s is NULL");
    MOE_CUDA(launch_rmsnorm_quant(h, gamma, eps, rows, cols, y, q, s, s_transposed != 0,
                                  static_cast<cudaStream_t>(stream)),
             "RMSNorm quantise launch");
    t_launches = 1;
    return MOE_OK;
}

int moe_combine_residual_rmsnorm(const void *o, const float *topk_w, const int32_t *inv_pos, const moe_cfg_t *cfg,
                                 int T, const void *residual, const void *gamma, float eps, void *h_out,
                                 void *x_next, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (!(eps >= 0.f)) return fail(MOE_ERR_ARG, "eps must be a non-negative number");
    if ((gamma == nullptr) != (x_next == nullptr))
        return fail(MOE_ERR_ARG, "gamma and x_next are both given or both NULL");
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(o, "o"));
    MOE_CHECK(check_ptr(topk_w, "topk_w"));
    MOE_CHECK(check_ptr(inv_pos, "inv_pos"));
    MOE_CHECK(check_ptr(residual, "residual"));
    MOE_CHECK(check_ptr(h_out, "h_out"));
    if (gamma) {
        MOE_CHECK(check_ptr(gamma, "gamma"));
        MOE_CHECK(check_ptr(x_next, "x_next"));
    }
    MOE_CUDA(launch_combine_residual_rmsnorm(o, topk_w, inv_pos, T, cfg->topk, cfg->n_shared, cfg->d, residual,
                                             gamma, eps, h_out, x_next, static_cast<cudaStream_t>(stream)),
             "combine + residual + RMSNorm launch");
    t_launches = 1;
    return MOE_OK;
}

int moe_layer_forward(const void *x, const void *w_gate, const float *bias, const uint8_t *w13, const float *w13_s,
                      const uint8_t *w2, const float *w2_s, const moe_cfg_t *cfg, int T, void *y, int32_t *topk_idx,
                      float *topk_w, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(x, "x"));
    MOE_CHECK(check_ptr(w_gate, "w_gate"));
    if (!bias) return fail(MOE_ERR_ARG, "bias is NULL");
    MOE_CHECK(check_ptr(w13, "w13"));
    MOE_CHECK(check_ptr(w13_s, "w13_s"));
    MOE_CHECK(check_ptr(w2, "w2"));
    MOE_CHECK(check_ptr(w2_s, "w2_s"));
    MOE_CHECK(check_ptr(y, "y"));
    if (topk_idx) MOE_CHECK(check_ptr(topk_idx, "topk_idx"));
    if (topk_w) MOE_CHECK(check_ptr(topk_w, "topk_w"));
    const moe_cfg_t &c = *cfg;
    const LayerWs need = carve_layer(c, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(c, T, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *idx = topk_idx ? topk_idx : ws.idx;
    float *w = topk_w ? topk_w : ws.w;
    int n = 0;
    MOE_CHECK(route_impl(x, w_gate, bias, c, T, idx, w, nullptr, ws.logits, st));
    n += t_launches;
    // the permutation quantises x on the way (one pass over x). Decode regime: the
    // gate/up kernel gathers the activation rows by sorted_tok, so the permutation
    // writes the unpermuted codes and no permuted copy
    const bool gather = decode_regime(c, T);
    const Gather g{ws.xq, ws.sx, ws.sorted_tok};
    int np = 0;
    MOE_CUDA(launch_permute(idx, nullptr, nullptr, T, c.topk, c.n_shared, c.E, c.d, expert_bn(c, T), down_bn(c, T),
                            ws.rank, ws.cnt, ws.counts, ws.offsets, ws.row_start, ws.tile_prefix, ws.tile_prefix_dn,
                            ws.counters, ws.sorted_tok, ws.inv_pos, ws.xq_perm, ws.sx_perm, &np, st, !gather, x,
                            gather ? ws.xq : nullptr, gather ? ws.sx : nullptr),
             "quantise + permutation launch");
    n += np;
    t_launches = 0;
    // the permutation already wrote the GEMM schedule into the workspace
    MOE_CHECK(experts_impl(ws.xq_perm, ws.sx_perm, ws.offsets, w13, w13_s, w2, w2_s, c, T, ws.o, ws, false, st,
                           gather ? &g : nullptr));
    n += t_launches;
    MOE_CUDA(launch_combine(ws.o, w, ws.inv_pos, T, c.topk, c.n_shared, c.d, y, st), "combine launch");
    n += 1;
    t_launches = n;
    return MOE_OK;
}

int moe_block_ffn_forward(const void *h, const void *gamma_post, float eps, const void *w_gate, const float *bias,
                          const uint8_t *w13, const float *w13_s, const uint8_t *w2, const float *w2_s,
                          const moe_cfg_t *cfg, int T, const void *gamma_next, void *h_out, void *x_next,
                          int32_t *topk_idx, float *topk_w, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    MOE_CHECK(check_cfg(cfg));
    MOE_CHECK(check_T(T));
    if (!(eps >= 0.f)) return fail(MOE_ERR_ARG, "eps must be a non-negative number");
    if ((gamma_next == nullptr) != (x_next == nullptr))
        return fail(MOE_ERR_ARG, "gamma_next and x_next are both given or both NULL");
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(h, "h"));
    MOE_CHECK(check_ptr(gamma_post, "gamma_post"));
    MOE_CHECK(check_ptr(w_gate, "w_gate"));
    if (!bias) return fail(MOE_ERR_ARG, "bias is NULL");
    MOE_CHECK(check_ptr(w13, "w13"));
    MOE_CHECK(check_ptr(w13_s, "w13_s"));
    MOE_CHECK(check_ptr(w2, "w2"));
    MOE_CHECK(check_ptr(w2_s, "w2_s"));
    MOE_CHECK(check_ptr(h_out, "h_out"));
    if (gamma_next) {
        MOE_CHECK(check_ptr(gamma_next, "gamma_next"));
        MOE_CHECK(check_ptr(x_next, "x_next"));
    }
    if (topk_idx) MOE_CHECK(check_ptr(topk_idx, "topk_idx"));
    if (topk_w) MOE_CHECK(check_ptr(topk_w, "topk_w"));
    const moe_cfg_t &c = *cfg;
    const LayerWs need = carve_layer(c, T, nullptr);
    MOE_CHECK(check_ws(workspace, workspace_bytes, need.bytes));
    const LayerWs ws = carve_layer(c, T, workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *idx = topk_idx ? topk_idx : ws.idx;
    float *w = topk_w ? topk_w : ws.w;
    int n = 0;
    // x = RMSNorm_post(h) in bf16 for the router, and its 1x128 codes and scales in
    // the same pass: the layer's input quantisation, not repeated
    MOE_CUDA(launch_rmsnorm_quant(h, gamma_post, eps, T, c.d, ws.xn, ws.xq, ws.sx, false, st),
             "RMSNorm quantise launch");
    n += 1;
    MOE_CHECK(route_impl(ws.xn, w_gate, bias, c, T, idx, w, nullptr, ws.logits, st));
    n += t_launches;
    const bool gather = decode_regime(c, T);   // as in moe_layer_forward
    const Gather g{ws.xq, ws.sx, ws.sorted_tok};
    int np = 0;
    MOE_CUDA(launch_permute(idx, ws.xq, ws.sx, T, c.topk, c.n_shared, c.E, c.d, expert_bn(c, T), down_bn(c, T),
                            ws.rank, ws.cnt, ws.counts, ws.offsets, ws.row_start, ws.tile_prefix, ws.tile_prefix_dn,
                            ws.counters, ws.sorted_tok, ws.inv_pos, ws.xq_perm, ws.sx_perm, &np, st, !gather),
             "permutation launch");
    n += np;
    t_launches = 0;
    MOE_CHECK(experts_impl(ws.xq_perm, ws.sx_perm, ws.offsets, w13, w13_s, w2, w2_s, c, T, ws.o, ws, false, st,
                           gather ? &g : nullptr));
    n += t_launches;
    // h_out = h + y (y rounded to bf16), x_next = RMSNorm_next(h_out)
    MOE_CUDA(launch_combine_residual_rmsnorm(ws.o, w, ws.inv_pos, T, c.topk, c.n_shared, c.d, h, gamma_next, eps,
                                             h_out, x_next, st),
             "combine + residual + RMSNorm launch");
    n += 1;
    t_launches = n;
    return MOE_OK;
}

size_t dense_swiglu_workspace_bytes(int d, int H, int T) {
    if (d <= 0 || d % 128 || H <= 0 || H % 128 || T < 0 || T > kMaxT) return 0;
    Carver cv{nullptr};
    const size_t Tz = static_cast<size_t>(T);
    cv.take<uint8_t>(Tz * d);
    cv.take<float>(Tz * (d / 128) * 4);
    cv.take<uint8_t>(Tz * H);
    cv.take<float>(Tz * (H / 128) * 4);
    return align_up(cv.off, 1024);
}

int dense_swiglu_fp8(const void *x, const uint8_t *w13, const float *w13_s, const uint8_t *w2, const float *w2_s,
                     int d, int H, int T, void *y, void *workspace, size_t workspace_bytes, void *stream) {
    t_launches = 0;
    if (d <= 0 || d % 128 || d > 65536) return fail(MOE_ERR_UNSUPPORTED, "d=%d must be a multiple of 128", d);
    if (H <= 0 || H % 128 || H > 65536) return fail(MOE_ERR_UNSUPPORTED, "H=%d must be a multiple of 128", H);
    MOE_CHECK(check_T(T));
    if (T == 0) return MOE_OK;
    MOE_CHECK(check_ptr(x, "x"));
    MOE_CHECK(check_ptr(w13, "w13"));
    MOE_CHECK(check_ptr(w13_s, "w13_s"));
    MOE_CHECK(check_ptr(w2, "w2"));
    MOE_CHECK(check_ptr(w2_s, "w2_s"));
    MOE_CHECK(check_ptr(y, "y"));
    MOE_CHECK(check_ws(workspace, workspace_bytes, dense_swiglu_workspace_bytes(d, H, T)));
    Carver cv{static_cast<uint8_t *>(workspace)};
    const size_t Tz = static_cast<size_t>(T);
    uint8_t *xq = cv.take<uint8_t>(Tz * d);
    float *sx_t = cv.take<float>(Tz * (d / 128) * 4);
    uint8_t *hq = cv.take<uint8_t>(Tz * H);
    float *hs_t = cv.take<float>(Tz * (H / 128) * 4);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    MOE_CUDA(launch_quant(x, true, T, d, xq, sx_t, true, num_sms(), st), "quantise launch");
    CUtensorMap m13, m2;
    ActMaps mx, mh;
    const bool down_wide = (d / 128) % 2 == 0;
    MOE_CHECK(make_map_gateup(&m13, w13, 1, H, d));
    MOE_CHECK(make_act_maps(&mx, xq, 1, T, d));
    if (down_wide) {
        MOE_CHECK(make_map(&m2, w2, 1, d, H, 2 * kBM));
        MOE_CHECK(make_act_maps(&mh, hq, 1, T, H));
    } else {
        MOE_CHECK(make_map_kpair(&m2, w2, d, H, kBM));
        MOE_CHECK(make_act_maps_kpair(&mh, hq, T, H));
    }
    GemmArgs gu{};
    gu.G = 1;
    gu.num_kb = d / 128;
    gu.num_mb = H / 128;
    gu.total_rows = T;
    gu.single_rows = T;
    gu.act_scale_t = sx_t;
    gu.w_scale = w13_s;
    gu.a_rows_per_group = 2 * H;
    gu.hq = hq;
    gu.hs_t = hs_t;
    MOE_CUDA(launch_grouped_gemm(Kind::GateUpWide, 128, m13, mx, gu, num_sms(), st), "gate/up GEMM launch");
    GemmArgs dn{};
    dn.G = 1;
    dn.num_kb = H / 128;
    dn.num_mb = d / 128;
    dn.total_rows = T;
    dn.single_rows = T;
    dn.act_scale_t = hs_t;
    dn.w_scale = w2_s;
    dn.a_rows_per_group = d;
    dn.out = static_cast<__nv_bfloat16 *>(y);
    if (down_wide) {
        dn.num_mb = d / 256;
        MOE_CUDA(launch_grouped_gemm(Kind::DownWide, 128, m2, mh, dn, num_sms(), st), "down GEMM launch");
    } else {
        MOE_CUDA(launch_grouped_gemm(Kind::Down, 128, m2, mh, dn, num_sms(), st), "down GEMM launch");
    }
    t_launches = 3;
    return MOE_OK;
}

int moe_check_device_error(void *stream, uint32_t *detail) {
    unsigned int *word = nullptr;
    MOE_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronise");
    MOE_CUDA(device_error_word(&word), "error word address");
    unsigned int v = 0;
    MOE_CUDA(cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost), "error word read");
    if (v) MOE_CUDA(cudaMemset(word, 0, sizeof(v)), "error word clear");
    if (detail) *detail = v;
    if (v & (ERR_WAIT_TMA_FULL | ERR_WAIT_SMEM_EMPTY | ERR_WAIT_PART_FULL | ERR_WAIT_PART_EMPTY | ERR_WAIT_DRAIN |
             ERR_WAIT_SELFTEST))
        return fail(MOE_ERR_TIMEOUT, "device error bits 0x%x (a bounded wait gave up)", v);
    if (v) return fail(MOE_ERR_INDEX, "device error bits 0x%x (an index check failed; its access was skipped)", v);
    return MOE_OK;
}

int moe_test_wait_timeout(uint64_t limit_ns, void *stream) {
    t_launches = 0;
    if (limit_ns < 1000 || limit_ns > 1000000000ull)
        return fail(MOE_ERR_ARG, "limit_ns=%llu must be in [1000, 1e9]", static_cast<unsigned long long>(limit_ns));
    MOE_CUDA(launch_wait_selftest(limit_ns, static_cast<cudaStream_t>(stream)), "wait self-test launch");
    t_launches = 1;
    return MOE_OK;
}

const char *moe_last_error_string(void) { return t_err; }

int moe_last_launch_count(void) { return t_launches; }

}  // extern "C"
