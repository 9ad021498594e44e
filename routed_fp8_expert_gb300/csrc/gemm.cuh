// Persistent grouped GEMM on the tcgen05 tensor cores (sm_103a).
//
// A "work item" is (group g, 128-row weight block mb, token tile nt); items of
// one group are ordered mb-major so that the token tiles sharing a weight block
// run at the same time on neighbouring CTAs. Two orientations:
//   swap-AB (decode-sized tiles: GateUp, DownPair, Router): the block's weight
//     rows are the MMA M dimension (TMEM lanes) and the tile's tokens the N
//     dimension (TMEM columns), so a handful of tokens costs an N=16 MMA;
//   token-major (128-token tiles: GateUpWide, DownWide, Down): the tile's 128 tokens are M and
//     the block's 128 weight rows N. Each epilogue thread then owns one token,
//     and the per-K-block scale s_w[mb,kb] * s_x[token,kb] is one scalar per
//     thread instead of one value per column.
//
// Roles (one CTA per SM):
//   warp 0      producer: takes work items from the tile scheduler, issues the
//               TMA tile loads (weight tile(s) + activation rows per 128-byte K
//               block, or per pair of K blocks for the token-major kinds)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..9  epilogue: 2 column groups of four warps; each warp reads its
//               32-lane quarter of TMEM for its group's columns
//   last warp   (FP8 kinds) copies each K block's activation and weight scales
//
// Tile scheduler: for expert groups the producer takes the next item from a
// global counter (atomicAdd), so token tiles that share a weight block start
// within a microsecond of each other on whichever CTAs are free (their weight
// tiles are then read from HBM once), and unequal items balance themselves.
// Single-group GEMMs (router, dense FFN) use a static round-robin order. The
// item index reaches the MMA and epilogue warps through a shared-memory queue.
//
// FP8 kinds (gate/up and down): e4m3 x e4m3 -> fp32 with one partial product
// per 128-wide K block, because the weight scale (per 128x128 block) and the
// activation scale (per token and 128-wide K block) both change at every K
// block. The epilogue promotes each partial into fp32 registers:
//     acc[j] += (s_w[mb, kb] * s_x[row_j, kb]) * partial[j]
// TMEM holds two to four partial buffers so the MMAs of the next K blocks run
// while block kb is promoted.
//
// Router kind: bf16 x bf16 -> fp32, accumulated in TMEM over the whole K
// range; the epilogue writes fp32 logits. With 128-token tiles an item holds up to
// three 128-expert blocks (three MMAs on one token tile per K step, 384 TMEM columns).
#pragma once
#include "internal.h"
#include "ptx.cuh"

namespace moe {

// GateUp: gate and up projections of one weight block, fused SiLU*mul and h quantisation.
// Down:   token-major down projection with one 128-row block per item, bf16
//         output (the wide-tile down projection when the output has an odd
//         number of 128-row blocks).
// DownPair: down projection with two adjacent 128-row weight blocks per item
//         (like GateUp's two tiles): twice the weight bytes per K block for the
//         same per-K-block fixed costs; used for decode-sized tiles.
// Router: bf16 router logits.
// GateUpWide: token-major, the gate and up blocks of the same 128 features as one
//         N = 256 item, with the fused SiLU*mul and h quantisation.
// DownWide: token-major down projection with two adjacent 128-row blocks (N = 256).
enum class Kind { GateUp, Down, Router, DownPair, GateUpWide, DownWide };

// Column groups of the 256-row token-major kinds' epilogue: 2 gives eight epilogue
// warps of 128 accumulators a thread (eleven warps, 168 registers a thread), 4
// gives sixteen warps of 64 (nineteen warps, 96 registers).
constexpr int kWideGroups = 2;

constexpr int kBM = 128;                    // weight rows per tile (MMA M)
constexpr int kKBytes = 128;                // bytes of K per stage (= one swizzle row)
constexpr int kATileBytes = kBM * kKBytes;  // 16 KB
constexpr int kActBoxRows = 16;             // smallest activation TMA box height
__device__ constexpr int kActBoxHeights[kActBoxes] = {16, 32, 64, 96, 128};
constexpr int kMaxGroups = 1032;            // routed + shared experts, padded
constexpr int kItemQ = 4;                   // depth of the producer -> consumers item queue
constexpr int kItemWords = 8;               // a queue entry: the item index and its decoded Item

constexpr int kStageBudget = 200 * 1024;    // shared memory for the operand ring
constexpr int kPrefetchReps = 4;            // first-round items whose weights a CTA prefetches

constexpr int pow2_at_least(int v, int lo) { return v <= lo ? lo : 2 * pow2_at_least((v + 1) / 2, lo); }

// Per-kind, per-tile-width configuration. BN = tokens per tile (MMA N upper bound).
template <Kind K, int BN> struct KindCfg {
    // token-major with 256 weight rows per item (two 128-row tiles per K block)
    static constexpr bool kWide = (K == Kind::GateUpWide || K == Kind::DownWide);
    // weight tiles per K block: gate and up, or two row blocks
    // the 128-token router reads up to three 128-row blocks of W_g per stage (all
    // the experts of a 384-expert router: the token tile is read once, not per block)
    static constexpr bool kRouterAll = (K == Kind::Router && BN == 128);
    static constexpr int kATiles = kRouterAll ? 3 : (K == Kind::GateUp || K == Kind::DownPair || kWide) ? 2 : 1;
    static constexpr bool kPromote = (K != Kind::Router);         // per-128-K fp32 promotion
    static constexpr bool kBf16 = (K == Kind::Router);
    // token-major: tokens on the TMEM lanes (M = 128), weight rows on the columns
    static constexpr bool kTM = (K == Kind::Down || kWide);
    // K blocks per stage: the single-tile token-major kind loads two consecutive K
    // blocks per TMA request (3D maps with a K-block dimension)
    static constexpr int kKPS = (K == Kind::Down) ? 2 : 1;
    static constexpr int kBTileBytes = BN * kKBytes;
    static constexpr int kAStageBytes = kKPS * kATiles * kATileBytes;   // weight part of a stage
    static constexpr int kStageBytes = kAStageBytes + kKPS * kBTileBytes;
    static constexpr int kStages = (kStageBudget / kStageBytes) > 12 ? 12 : (kStageBudget / kStageBytes);
    static constexpr int kPartCols = kATiles * (kTM ? kBM : BN);  // one TMEM partial buffer
    // partial buffers in flight between the MMA issuer and the epilogue: as
    // many as TMEM holds, up to 4, so the MMAs run ahead of the promotion
    static constexpr int kNumPart = (512 / kPartCols) >= 4 ? 4 : (512 / kPartCols);
    static constexpr int kTmemCols = pow2_at_least(kNumPart * kPartCols, 32);
    // scale slots: their own ring, released by the epilogue, so operand stages
    // are released by the MMA alone and the producer keeps kStages ahead of it
    static constexpr int kScaleSlots = kPromote ? (kStages + kNumPart + 2) : 1;
    // epilogue column groups: token columns (swap-AB) or weight rows (token-major);
    // kWideGroups for the 256-row items, each thread holding 256 / kWideGroups
    // accumulators
    static constexpr int kGroups = kWide ? kWideGroups : 2;
    static constexpr int kHalfCols = kWide ? 256 / kWideGroups : (kTM ? kBM : BN) / kGroups;  // accumulators per thread
    static constexpr int kChunks = kHalfCols / 16;
    static constexpr int kEpiWarps = 4 * kGroups;                 // one warp per TMEM lane quarter and group
    // the K blocks' scales are copied by a warp of their own, beside the producer
    static constexpr bool kScaleWarpOwn = kPromote;
    static constexpr int kScaleWarp = 2 + kEpiWarps;
    static constexpr int kThreads = 64 + 32 * kEpiWarps + (kScaleWarpOwn ? 32 : 0);
    // h amax exchange barriers: GateUp [groups][2 buffers]; wide [4 lane quarters][2]
    static constexpr int kAmaxBars = kWide ? 8 : 2 * kGroups;
    // registers a thread of the wide kinds may use: the register file is split over
    // the four sub-partitions (16,384 each), which hold the CTA's warps round-robin
    static constexpr int kWideRegs = (16384 / ((kThreads / 32 + 3) / 4 * 32)) / 8 * 8;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 128, "tile width");
    static_assert(!kTM || BN == 128, "token-major tiles hold 128 tokens (the MMA M dimension)");
    static_assert((kStages * kKPS >= 4 || kRouterAll) && kStages >= 3, "pipeline depth");
    static_assert(kKPS == 1 || kATiles == 1, "K-pair stages hold one weight tile per K block");
};

struct GemmArgs {
    int G;                    // groups (experts, routed first, shared last)
    int num_kb;               // K blocks of 128 bytes
    int num_mb;               // 128-row blocks of weight rows per group (output features / 128)
    int total_rows;           // rows of the activation buffer
    int single_rows;          // >= 0: one group of that many rows (row_start / tile_prefix unused)
    const int *row_start;     // [G+1] first activation row of each group's segment
    const int *tile_prefix;   // [2][G+1] prefix sums of ceil(rows_g / BN): all groups, then those
                              // of two or more tiles only
    int interleave;           // merge the items of multi-tile groups with those of one-tile groups
    const float *act_scale_t; // [num_kb][total_rows]  (FP8 kinds)
    const float *w_scale;     // GateUp: [G][2][num_mb][num_kb]; Down: [G][num_mb][num_kb]
    int w_tiled;              // map_a is over the tiled weight layout (128 x 128 tiles): gate/up 5D
                              // {128 B, 128 rows, K block, row block, 2G}; down 4D {128 B, 128 rows,
                              // K block, row block} (expert kinds only)
    int a_rows_per_group;     // weight rows of one group in the A tensor map (GateUp: 2*H, Down: d_out)
    // L2 prefetch of weights while the preceding kernel still runs (a hint; null: none).
    // Item j of the first round is taken to be (group j / pf_items, block j % pf_items),
    // as it is when the first groups are all routed to; its weight run(s) start at
    // pf_base + g * pf_group_bytes + i * pf_item_bytes (and pf_second bytes further on,
    // if non-zero), of which pf_len bytes are prefetched. Every address stays inside
    // the weights.
    const uint8_t *pf_base;
    uint64_t pf_group_bytes;
    uint64_t pf_item_bytes;
    uint64_t pf_second;
    uint32_t pf_len;          // a multiple of 16 KB
    int pf_items;
    uint8_t *hq;              // GateUp: [total_rows][num_mb*128]
    float *hs_t;              // GateUp: [num_mb][total_rows]
    __nv_bfloat16 *out;       // Down: [total_rows][num_mb*128]
    float *logits;            // Router: [k_splits][total_rows][n_valid] partial logits
    int n_valid;              // Router: valid weight rows (experts)
    int k_splits;             // Router: K range split into this many partial sums (>= 1)
    int a_tiles;              // 128-token router: weight blocks per item (num_mb is then 1), or 0
    unsigned int *err;        // device error word (bounded waits that gave up)
    int *item_counter;        // dynamic scheduler counter (zero at launch), or null for static order
    // GateUp gathering its activation rows (null: rows of the permuted copy by TMA):
    // permuted row p holds token tok(p) = row_token[p] for p < n_routed, else
    // (p - n_routed) % n_tok (the shared experts' rows); its codes are
    // gather_rows[tok][num_kb * 128] and its scales gather_scales[tok][num_kb]
    const uint8_t *gather_rows;
    const float *gather_scales;
    const int *row_token;
    int n_routed;
    int n_tok;
};

// Token of permuted row p in the gathering mode.
__device__ __forceinline__ int gather_token(const GemmArgs &a, int p) {
    return p < a.n_routed ? a.row_token[p] : (p - a.n_routed) % a.n_tok;
}

// 16-byte asynchronous global -> shared copy (L2 only).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Orders this thread's later async-proxy reads of shared memory (the MMAs) after
// the generic-proxy writes it has observed complete (cp.async copies).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct Item {
    int g, mb, row0, n, ks;
    int ntiles;   // token tiles of the item's group (tiles sharing its weight block)
};

// Items of a group are ordered (weight block, token tile) with the token tile
// fastest, so the tiles that share a weight block are adjacent.
//
// Interleaved order (a.interleave): the items of groups with two or more token
// tiles (weight blocks re-read from L2 by every tile: tensor-bound) and those of
// one-tile groups (weights streamed from HBM once) form two streams, each in the
// order above, merged evenly: item i is the m-th of the multi-tile stream when
// floor((i+1) NM / N) > floor(i NM / N) = m (NM of N items multi-tile), else
// the (i - m)-th single-tile item. Under skewed routing the HBM streaming of the
// cold experts then overlaps the hot experts' MMAs instead of alternating with them.
// s_tpm[g] is the multi-tile prefix; the single-tile prefix is s_tp[g] - s_tpm[g].
// Called by a whole warp (the producer's), all lanes with the same it; they
// return the same item. The group search takes two rounds of 32 parallel
// shared-memory reads and a ballot each, not a binary search of dependent reads.
template <int BN>
__device__ __forceinline__ bool decode_item(int it, const GemmArgs &a, const int *s_tp,
                                            const int *s_rs, const int *s_tpm, Item &o, int lane) {
    const int nblk = a.num_mb;   // weight blocks per group
    int mbx;
    if (a.single_rows >= 0) {
        // items = (block, token tile, K split) with the split fastest
        const int nt_total = (a.single_rows + BN - 1) / BN;
        const int splits = a.k_splits > 0 ? a.k_splits : 1;
        o.ks = it % splits;
        const int rest = it / splits;
        o.g = 0;
        mbx = rest / nt_total;
        const int nt = rest - mbx * nt_total;
        o.row0 = nt * BN;
        o.n = min(BN, a.single_rows - o.row0);
        o.ntiles = nt_total;
    } else {
        o.ks = 0;
        int idx = it;          // index inside the item's stream
        int stream = 0;        // 0: all groups (plain order), 1: multi-tile, 2: one-tile
        if (a.interleave) {
            const long long n_all = static_cast<long long>(nblk) * s_tp[a.G];
            const long long n_multi = static_cast<long long>(nblk) * s_tpm[a.G];
            const long long num = static_cast<long long>(it) * n_multi;
            const long long m0 = num / n_all;
            // floor((it + 1) NM / N) = m0 + [r + NM >= N] with r = it NM - m0 N < N, as NM <= N
            if (num - m0 * n_all + n_multi >= n_all) { idx = static_cast<int>(m0); stream = 1; }
            else { idx = it - static_cast<int>(m0); stream = 2; }
        }
        // the stream's tile prefix at group g
        auto prefix = [&](int g) -> int { return stream == 0 ? s_tp[g] : stream == 1 ? s_tpm[g] : s_tp[g] - s_tpm[g]; };
        const int key = idx / nblk;
        // the last g < G with prefix(g) <= key (a group of the stream): prefix rises from
        // prefix(0) = 0, so the lanes whose candidate passes form a run from lane 0.
        // First the chunk of 32 groups (chunk 32 only when G > 1024), then the group
        const unsigned m1 = __ballot_sync(0xffffffffu, 32 * lane < a.G && prefix(32 * lane) <= key);
        int c = 31 - __clz(m1);
        if (c == 31 && a.G > 1024 && prefix(1024) <= key) c = 32;
        const int g0 = 32 * c;
        const unsigned m2 = __ballot_sync(0xffffffffu, g0 + lane < a.G && prefix(g0 + lane) <= key);
        const int g = g0 + 31 - __clz(m2);
        const int nt_g = prefix(g + 1) - prefix(g);
        if (nt_g <= 0) return false;
        const int li = idx - nblk * prefix(g);
        o.g = g;
        mbx = li / nt_g;
        const int nt = li - mbx * nt_g;
        o.row0 = s_rs[g] + nt * BN;
        o.n = min(BN, s_rs[g + 1] - o.row0);
        o.ntiles = s_tp[g + 1] - s_tp[g];
    }
    o.mb = mbx;
    // (bounds-checked build: an item's rows inside the activation buffer)
    if (kDebugBounds && (o.row0 < 0 || o.row0 + o.n > a.total_rows)) return false;
    return o.n > 0 && o.mb < a.num_mb;
}

template <int BN>
__device__ __forceinline__ int total_items(const GemmArgs &a, const int *s_tp) {
    const int nblk = a.num_mb;
    if (a.single_rows >= 0)
        return nblk * ((a.single_rows + BN - 1) / BN) * (a.k_splits > 0 ? a.k_splits : 1);
    return nblk * s_tp[a.G];
}

// K blocks [kb0, kb1) of one item.
__device__ __forceinline__ void kb_range(const GemmArgs &a, const Item &I, int &kb0, int &kb1) {
    const int splits = a.k_splits > 0 ? a.k_splits : 1;
    kb0 = (a.num_kb * I.ks) / splits;
    kb1 = (a.num_kb * (I.ks + 1)) / splits;
}

// Index into kActBoxHeights of the activation box of a tile of n rows: the
// smallest that covers them. A token-major MMA still reads 128 rows (its M
// dimension); the rows past the box hold an earlier stage's activations, and
// their output rows (tokens past the tile's end) are never stored.
__device__ __forceinline__ int act_box_index(int n) {
    return (n <= 16) ? 0 : (n <= 32) ? 1 : (n <= 64) ? 2 : (n <= 96) ? 3 : 4;
}

// Two floats as round-to-nearest bf16, the first in the low half (lower address).
__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division intrinsics
// (__expf, __fdividef: a few ulp of fp32, far inside the h quantiser's rounding
// step); IEEE division here made the per-item epilogue tail a tenth of the
// wide gate/up kernel's time, with the tensor pipe idle behind it. For g below
// about -87, e^-g overflows and the quotient is 0, silu's limit.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// acc[i] += s * p[i], i < 16, as eight two-lane packed FMAs: each lane is an
// ordinary fma.rn, so the sums equal fmaf's bit for bit with half the issue slots
__device__ __forceinline__ void fold16(float *acc, const float *p, float s) {
    const float2 s2 = make_float2(s, s);
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float2 r = __ffma2_rn(s2, make_float2(p[i], p[i + 1]), make_float2(acc[i], acc[i + 1]));
        acc[i] = r.x;
        acc[i + 1] = r.y;
    }
}

// Shared-memory carve-up of one CTA (offsets from a 1024-byte aligned base).
template <Kind KIND, int BN> struct SmemLayout {
    using C = KindCfg<KIND, BN>;
    static constexpr int kNumBars = 2 * C::kStages + 2 * C::kNumPart + 1 + C::kAmaxBars + 2 * kItemQ +
                                    2 * C::kScaleSlots;
    static constexpr size_t kBars = static_cast<size_t>(C::kStages) * C::kStageBytes;
    static constexpr size_t kMisc = (kBars + kNumBars * 8 + 15) & ~size_t(15);
    static constexpr size_t kItems = kMisc + 16;                                // [kItemQ][kItemWords] int
    static constexpr size_t kTp = kItems + kItemQ * kItemWords * 4;
    static constexpr size_t kRs = kTp + kMaxGroups * 4;
    static constexpr size_t kTpm = kRs + kMaxGroups * 4;                       // [kMaxGroups] multi-tile prefix
    static constexpr int kScaleStride = BN + 4;                                // floats per stage: BN act + 2 weight
    static constexpr size_t kScale = kTpm + kMaxGroups * 4;                    // [kScaleSlots][kScaleStride]
    static constexpr size_t kCs = kScale + C::kScaleSlots * kScaleStride * 4;  // [warps][2][kATiles][HC], swap-AB
    static constexpr size_t kAmax = kCs + (C::kTM ? 0 : C::kEpiWarps * 2 * C::kATiles * C::kHalfCols * 4);
    // the h amax exchange: GateUp [groups][2][4][HC]; GateUpWide [2][4 groups][128 rows]
    static constexpr size_t kAmaxBytes = (KIND == Kind::GateUp)       ? C::kGroups * 2 * 4 * C::kHalfCols * 4
                                         : (KIND == Kind::GateUpWide) ? 2 * 4 * kBM * 4
                                                                      : 0;
    // DownWide: a slot of eight output rows per epilogue warp to turn its rows into
    // whole-line stores
    static constexpr size_t kXpose = kAmax + kAmaxBytes;
    static constexpr size_t kEnd = kXpose + ((KIND == Kind::DownWide) ? C::kEpiWarps * 8 * C::kHalfCols * 2 : 0);
    static constexpr size_t kLaunchBytes = kEnd + 1024;  // + alignment slack of the dynamic base
    static_assert(kBars % 1024 == 0 && kScale % 16 == 0 && kCs % 16 == 0 && kXpose % 16 == 0, "alignment");
    static_assert(kLaunchBytes <= 232448, "shared memory budget");
};

// The kernel body; map_a and map_b are the kernels' grid-constant parameters,
// whose addresses the TMA instructions take.
template <Kind KIND, int BN>
__device__ __forceinline__ void grouped_gemm_body(const CUtensorMap &map_a, const ActMaps &map_b,
                                                  const GemmArgs &args) {
    using C = KindCfg<KIND, BN>;
    using L = SmemLayout<KIND, BN>;
    constexpr int kStageBytes = C::kStageBytes;
    constexpr int kKbElems = C::kBf16 ? 64 : 128;
    constexpr uint32_t kFmt = C::kBf16 ? 1u : 0u;
    constexpr int HC = C::kHalfCols;
    constexpr int kEpi = C::kEpiWarps;
    // arrivals that release a partial buffer or a scale slot: one per epilogue warp,
    // or one per epilogue thread in the 256-row kinds
    constexpr int kRelease = C::kWide ? kEpi * 32 : kEpi;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *full = bars;
    uint64_t *empty = full + C::kStages;
    uint64_t *pfull = empty + C::kStages;
    uint64_t *pempty = pfull + C::kNumPart;
    uint64_t *mma_done = pempty + C::kNumPart;
    uint64_t *amax_bar = mma_done + 1;                  // [kAmaxBars]
    uint64_t *item_full = amax_bar + C::kAmaxBars;       // [kItemQ]
    uint64_t *item_empty = item_full + kItemQ;           // [kItemQ]
    uint64_t *sfull = item_empty + kItemQ;               // [kScaleSlots]
    uint64_t *sempty = sfull + C::kScaleSlots;           // [kScaleSlots]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_word = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    const uint32_t abort_flag = smem_u32(smem + L::kMisc + 4);   // shared address of the abort word
    volatile int *s_items = reinterpret_cast<volatile int *>(smem + L::kItems);
    int *s_tp = reinterpret_cast<int *>(smem + L::kTp);
    int *s_rs = reinterpret_cast<int *>(smem + L::kRs);
    int *s_tpm = reinterpret_cast<int *>(smem + L::kTpm);
    float *s_scale = reinterpret_cast<float *>(smem + L::kScale);  // scale slots
    float *s_cs = reinterpret_cast<float *>(smem + L::kCs);        // per-warp combined scales
    float *s_amax = reinterpret_cast<float *>(smem + L::kAmax);
    uint8_t *s_xpose = smem + L::kXpose;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    pdl_trigger();
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            // the producer's expect_tx arrival (+ TMA bytes); gathering GateUp: plus one
            // cp.async arrival per producer lane
            mbar_init(smem_u32(&full[s]), (KIND == Kind::GateUp && args.gather_rows) ? 33 : 1);
            mbar_init(smem_u32(&empty[s]), 1);   // the MMA commit
        }
        for (int s = 0; s < C::kScaleSlots; ++s) {
            mbar_init(smem_u32(&sfull[s]), 32);    // one cp.async arrival per scale-warp lane
            mbar_init(smem_u32(&sempty[s]), kRelease);
        }
        for (int b = 0; b < C::kNumPart; ++b) {
            mbar_init(smem_u32(&pfull[b]), 1);
            mbar_init(smem_u32(&pempty[b]), kRelease);
        }
        mbar_init(smem_u32(mma_done), 1);
        for (int b = 0; b < C::kAmaxBars; ++b) mbar_init(smem_u32(&amax_bar[b]), C::kWide ? C::kGroups : 4);
        for (int b = 0; b < kItemQ; ++b) {
            mbar_init(smem_u32(&item_full[b]), 1);
            mbar_init(smem_u32(&item_empty[b]), 1 + kEpi + (C::kScaleWarpOwn ? 1 : 0));
        }
        *abort_word = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map_a);
        for (int i = 0; i < kActBoxes; ++i) tma_prefetch_desc(&map_b.box[i]);
    }
    if (warp == 1) tmem_alloc<C::kTmemCols>(smem_u32(tmem_slot));
    // weights are not written by the preceding kernels: their first bytes may be on
    // their way to L2 before it completes (HBM is idle during the routing and the
    // permutation, and partly so during the previous GEMM's last items)
    // CTA b prefetches the first-round items b + r n / kPrefetchReps (mod n, n CTAs):
    // each item is prefetched by several CTAs, so that those resident early (on the SMs
    // the router GEMM leaves free) cover the whole first round
    if (warp == 0 && args.pf_base != nullptr) {
        for (int r = 0; r < kPrefetchReps; ++r) {
            const int item = static_cast<int>((blockIdx.x + r * (gridDim.x / kPrefetchReps)) % gridDim.x);
            const int g = item / args.pf_items, i = item % args.pf_items;
            if (g >= args.G) continue;
            const uint8_t *run = args.pf_base + static_cast<uint64_t>(g) * args.pf_group_bytes +
                                 static_cast<uint64_t>(i) * args.pf_item_bytes;
            const int chunks = static_cast<int>(args.pf_len >> 14);
            const int total = args.pf_second ? 2 * chunks : chunks;
            for (int c = lane; c < total; c += 32)
                l2_prefetch_bulk(run + (c >= chunks ? args.pf_second : 0) + (static_cast<uint64_t>(c % chunks) << 14),
                                 16384u);
        }
    }
    // the set-up above touches only shared memory, TMEM and the kernel's parameters,
    // so it overlaps the preceding kernel's tail; the global inputs come after it
    pdl_wait();
    if (args.single_rows < 0) {
        for (int i = threadIdx.x; i <= args.G; i += blockDim.x) {
            s_tp[i] = args.tile_prefix[i];
            s_rs[i] = args.row_start[i];
            if (args.interleave) s_tpm[i] = args.tile_prefix[args.G + 1 + i];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = total_items<BN>(args, s_tp);

    // Next item for a consumer: wait for the producer's queue slot, read the index
    // and the item the producer decoded, release the slot. Called by lane 0; returns
    // -1 on give-up, n_items at the end.
    auto take_item = [&](int &q, uint32_t &qphase, Item &I) -> int {
        if (!mbar_wait(smem_u32(&item_full[q]), qphase, abort_flag, args.err, ERR_WAIT_TMA_FULL)) return -1;
        const volatile int *e = s_items + q * kItemWords;
        const int it = e[0];
        I.g = e[1];
        I.mb = e[2];
        I.row0 = e[3];
        I.n = e[4];
        I.ks = e[5];
        I.ntiles = e[6];
        mbar_arrive(smem_u32(&item_empty[q]));
        if (++q == kItemQ) { q = 0; qphase ^= 1; }
        return it;
    };
    // lane 0's item to the whole warp
    auto bcast_item = [&](Item &I) {
        I.g = __shfl_sync(0xffffffffu, I.g, 0);
        I.mb = __shfl_sync(0xffffffffu, I.mb, 0);
        I.row0 = __shfl_sync(0xffffffffu, I.row0, 0);
        I.n = __shfl_sync(0xffffffffu, I.n, 0);
        I.ks = __shfl_sync(0xffffffffu, I.ks, 0);
        I.ntiles = __shfl_sync(0xffffffffu, I.ntiles, 0);
    };

    // The weight-scale rows [num_kb] of an item's block(s).
    auto weight_scale_rows = [&](const Item &I, const float *&ws0, const float *&ws1) {
        ws1 = nullptr;
        if constexpr (KIND == Kind::GateUp || KIND == Kind::GateUpWide) {
            ws0 = args.w_scale + (static_cast<size_t>(I.g * 2 + 0) * args.num_mb + I.mb) * args.num_kb;
            ws1 = args.w_scale + (static_cast<size_t>(I.g * 2 + 1) * args.num_mb + I.mb) * args.num_kb;
        } else if constexpr (KIND == Kind::DownPair || KIND == Kind::DownWide) {
            // row blocks 2mb and 2mb+1 of the group's [2 * num_mb][num_kb] scale grid
            ws0 = args.w_scale + (static_cast<size_t>(I.g) * 2 * args.num_mb + 2 * I.mb) * args.num_kb;
            ws1 = ws0 + args.num_kb;
        } else {
            ws0 = args.w_scale + (static_cast<size_t>(I.g) * args.num_mb + I.mb) * args.num_kb;
        }
    };
    // K block kb's scales into slot `slot`: the activation scales of the tile's
    // tokens and the weight scale(s) of the block (cp.async, 4 bytes per lane and
    // copy); the slot's full barrier counts one arrival per lane.
    auto copy_scales = [&](const Item &I, int kb, int slot, const float *ws0, const float *ws1) {
        const uint32_t sdst = smem_u32(s_scale + slot * L::kScaleStride);
        if (KIND == Kind::GateUp && args.gather_rows) {
            // the tile's tokens' scales straight from the unpermuted [T][num_kb] array
            for (int i = lane; i < I.n; i += 32)
                cp_async_4(sdst + 4 * i, args.gather_scales + static_cast<size_t>(gather_token(args, I.row0 + i)) * args.num_kb + kb);
        } else {
            const float *src = args.act_scale_t + static_cast<size_t>(kb) * args.total_rows + I.row0;
            for (int i = lane; i < I.n; i += 32) cp_async_4(sdst + 4 * i, src + i);
        }
        if (lane == 0) {
            cp_async_4(sdst + 4 * BN, ws0 + kb);
            if constexpr (C::kATiles == 2) cp_async_4(sdst + 4 * (BN + 1), ws1 + kb);
        }
        cp_async_arrive_noinc(smem_u32(&sfull[slot]));
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // lane 0 fetches items and issues the TMA tile loads
        // weights read by one token tile only are streamed (evict first); a weight
        // block shared by several token tiles, which run at the same time, stays
        // in L2 for them (normal policy)
        const uint64_t pol_stream = policy_evict_first();
        const uint64_t pol_shared = policy_evict_normal();
        const uint64_t pol_x = policy_evict_last();
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_parity = 0;
        int q = 0;
        uint32_t qphase = 0;
        int next_static = blockIdx.x;
        while (true) {
            int it = 0, got = 1;
            Item I{};
            if (lane == 0) got = mbar_wait(smem_u32(&item_empty[q]), qphase ^ 1, abort_flag, args.err, ERR_WAIT_SMEM_EMPTY);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) break;
            // the item is decoded here, once, by the whole warp, and handed to the other
            // roles with its index; one that does not decode is recorded and skipped
            while (true) {
                if (lane == 0) {
                    if (args.item_counter) it = atomicAdd(args.item_counter, 1);
                    else { it = next_static; next_static += gridDim.x; }
                }
                it = __shfl_sync(0xffffffffu, it, 0);
                if (it >= n_items) { it = n_items; break; }
                if (decode_item<BN>(it, args, s_tp, s_rs, s_tpm, I, lane)) break;
                if (lane == 0) record_error(args.err, ERR_BAD_TILE);
            }
            if (lane == 0) {
                volatile int *e = s_items + q * kItemWords;
                e[0] = it;
                e[1] = I.g;
                e[2] = I.mb;
                e[3] = I.row0;
                e[4] = I.n;
                e[5] = I.ks;
                e[6] = I.ntiles;
                mbar_arrive(smem_u32(&item_full[q]));
            }
            if (it >= n_items) break;
            if (++q == kItemQ) { q = 0; qphase ^= 1; }
            int kb0, kb1;
            kb_range(args, I, kb0, kb1);
            // one activation box per stage
            const int box_i = act_box_index(I.n);
            // full boxes count toward the transaction bytes, including rows and a
            // K block beyond the tensor, which the TMA unit fills with zeros
            uint32_t bytes = C::kKPS * (C::kATiles * kATileBytes + kActBoxHeights[box_i] * kKBytes);
            if constexpr (C::kRouterAll)   // the weight blocks actually loaded: a_tiles, or one
                bytes = (args.a_tiles > 0 ? args.a_tiles : 1) * kATileBytes + kActBoxHeights[box_i] * kKBytes;
            // gathering GateUp: lane i copies the tile's row i (one token's 128-byte K
            // block, eight 16-byte copies into its 128-byte-swizzled place); only the
            // weights come by TMA. Rows past the tile's end stay as they are: their
            // output columns are never stored, and no column depends on another row
            const bool gather = (KIND == Kind::GateUp) && args.gather_rows != nullptr;
            const uint8_t *grow = nullptr;
            if (gather) {
                bytes = C::kATiles * kATileBytes;
                if (lane < I.n)
                    grow = args.gather_rows + static_cast<size_t>(gather_token(args, I.row0 + lane)) * args.num_kb * kKBytes;
            }
            const uint64_t pol_w = (I.ntiles > 1) ? pol_shared : pol_stream;
            int arow0;
            if constexpr (KIND == Kind::Router) {
                arow0 = I.mb * kBM;
            } else {
                constexpr int kRowsPerBlock = (KIND == Kind::DownPair || KIND == Kind::DownWide) ? 2 * kBM : kBM;
                arow0 = I.g * args.a_rows_per_group + I.mb * kRowsPerBlock;
            }
            bool ok = true;
            for (int kb = kb0; kb < kb1; kb += C::kKPS) {
                int w = 1;
                if (lane == 0) w = mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, args.err, ERR_WAIT_SMEM_EMPTY);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) { ok = false; break; }
                const uint32_t fb = smem_u32(&full[stage]);
                const uint32_t sbase = smem_u32(stages + stage * kStageBytes);
                if (gather) {
                    if (grow) {
                        const uint32_t dst = sbase + C::kAStageBytes + lane * kKBytes;
                        const uint8_t *src = grow + static_cast<size_t>(kb) * kKBytes;
#pragma unroll
                        for (int c = 0; c < kKBytes / 16; ++c) cp_async_16(dst + ((c ^ (lane & 7)) << 4), src + 16 * c);
                    }
                    cp_async_arrive_noinc(fb);
                    if (lane == 0) {
                        mbar_arrive_expect_tx(fb, bytes);
                        if (args.w_tiled) tma_load_5d(sbase, &map_a, fb, 0, 0, kb, I.mb, 2 * I.g, pol_w);
                        else tma_load_3d(sbase, &map_a, fb, kb * kKbElems, I.mb * kBM, 2 * I.g, pol_w);
                    }
                } else if (lane == 0) {
                    mbar_arrive_expect_tx(fb, bytes);
                    // weight tiles in one request (the TMA unit's request rate, not its
                    // bytes, bounds an SM's loads): GateUp's gate and up tiles as one
                    // 3D box, DownPair's two row blocks as one 256-row box
                    // K-pair kinds: K blocks kb and kb+1 of the weight rows and of the
                    // activation rows, one request each (x = 0, y = row, z = K block)
                    if constexpr (C::kKPS == 2) {
                        // tiled: box {128, 128, 2 K blocks, 1}, two consecutive tiles
                        if (args.w_tiled) tma_load_4d(sbase, &map_a, fb, 0, 0, kb, arow0 / kBM, pol_w);
                        else tma_load_3d(sbase, &map_a, fb, 0, arow0, kb, pol_w);
                        tma_load_3d(sbase + C::kAStageBytes, &map_b.box[box_i], fb, 0, I.row0, kb, pol_x);
                    } else {
                        const int kx = kb * kKbElems;
                        if constexpr (KIND == Kind::GateUp || KIND == Kind::GateUpWide) {
                            // tiled: box {128, 128, 1, 1, 2}, the gate and up tiles
                            if (args.w_tiled) tma_load_5d(sbase, &map_a, fb, 0, 0, kb, I.mb, 2 * I.g, pol_w);
                            else tma_load_3d(sbase, &map_a, fb, kx, I.mb * kBM, 2 * I.g, pol_w);
                        } else if constexpr (KIND == Kind::DownPair || KIND == Kind::DownWide) {
                            // tiled: box {128, 128, 1, 2}, two row blocks' tiles
                            if (args.w_tiled) tma_load_4d(sbase, &map_a, fb, 0, 0, kb, arow0 / kBM, pol_w);
                            else tma_load_2d(sbase, &map_a, fb, kx, arow0, pol_w);
                        } else if constexpr (C::kRouterAll) {
                            if (args.a_tiles > 0) {
                                for (int t = 0; t < args.a_tiles; ++t)
                                    tma_load_2d(sbase + t * kATileBytes, &map_a, fb, kx, t * kBM, pol_w);
                            } else {
                                tma_load_2d(sbase, &map_a, fb, kx, arow0, pol_w);
                            }
                        } else {
                            tma_load_2d(sbase, &map_a, fb, kx, arow0, pol_w);
                        }
                        tma_load_2d(sbase + C::kAStageBytes, &map_b.box[box_i], fb, kx, I.row0, pol_x);
                    }
                }
                issued_mask |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
        // every issued copy must land before the CTA may exit
        cp_async_wait_all();
        if (lane == 0)
            for (int s = 0; s < C::kStages; ++s)
                if (issued_mask & (1u << s)) mbar_wait_drain(smem_u32(&full[s]), (issued_parity >> s) & 1u, args.err);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pbuf = 0;
            uint32_t pphase = 0;
            int q = 0;
            uint32_t qphase = 0;
            bool ok = true;
            while (ok) {
                Item I;
                const int it = take_item(q, qphase, I);
                if (it < 0 || it >= n_items) break;
                int kb0, kb1;
                kb_range(args, I, kb0, kb1);
                // swap-AB: M = 128 weight rows, N = the tile's tokens rounded up to 16;
                // token-major: M = 128 tokens, N = 128 weight rows
                const int n_mma = C::kTM ? C::kPartCols : ((I.n + 15) & ~15);
                const uint32_t idesc = idesc_make(kFmt, kFmt, kBM, n_mma);
                // bytes of one K block's activation sub-tile inside a K-pair box
                const uint32_t b_kb_bytes = kActBoxHeights[act_box_index(I.n)] * kKBytes;
                for (int kb = kb0; kb < kb1; kb += C::kKPS) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err, ERR_WAIT_TMA_FULL)) { ok = false; break; }
                    // gathered rows were written by cp.async (generic proxy): order them
                    // before the MMAs' reads
                    if (KIND == Kind::GateUp && args.gather_rows) fence_proxy_async_smem();
                    const uint32_t sbase = smem_u32(stages + stage * kStageBytes);
#pragma unroll
                    for (int h = 0; h < C::kKPS; ++h) {
                        const int kbh = kb + h;
                        if (kbh >= kb1) break;   // odd K-block count: the pair's second half is padding
                        if (C::kPromote || kbh == kb0) {
                            if (!mbar_wait(smem_u32(&pempty[pbuf]), pphase ^ 1, abort_flag, args.err, ERR_WAIT_PART_EMPTY)) {
                                ok = false;
                                break;
                            }
                        }
                        tc_fence_after();
                        const uint32_t abase = sbase + h * C::kATiles * kATileBytes;
                        const uint32_t bbase = sbase + C::kAStageBytes + h * b_kb_bytes;
                        const uint32_t dcol = tmem_base + pbuf * C::kPartCols;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t acc = C::kPromote ? (k > 0) : (kbh > kb0 || k > 0);
                            const uint64_t bdesc = sdesc_sw128(bbase + k * 32);   // activations
                            const uint64_t adesc = sdesc_sw128(abase + k * 32);   // weights
                            if constexpr (C::kRouterAll) {
                                const int nt = args.a_tiles > 0 ? args.a_tiles : 1;
                                for (int t = 0; t < nt; ++t)
                                    mma_bf16(dcol + t * BN, sdesc_sw128(abase + t * kATileBytes + k * 32), bdesc, idesc, acc);
                            } else if constexpr (C::kBf16) mma_bf16(dcol, adesc, bdesc, idesc, acc);
                            else if constexpr (C::kTM) mma_f8(dcol, bdesc, adesc, idesc, acc);
                            else mma_f8(dcol, adesc, bdesc, idesc, acc);
                            if constexpr (C::kATiles == 2 && !C::kTM)
                                mma_f8(dcol + BN, sdesc_sw128(abase + kATileBytes + k * 32), bdesc, idesc, acc);
                        }
                        if (C::kPromote || kbh == kb1 - 1) {
                            mma_commit(smem_u32(&pfull[pbuf]));
                            if (++pbuf == C::kNumPart) { pbuf = 0; pphase ^= 1; }
                        }
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&empty[stage]));
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
            // all MMAs must finish before TMEM is released
            mma_commit(smem_u32(mma_done));
            mbar_wait_drain(smem_u32(mma_done), 0, args.err);
        }
    } else if (C::kScaleWarpOwn && warp == C::kScaleWarp) {
        // ------------------------------------------------------------ scale copier
        // per K block, the scales into the next scale slot; runs beside the producer
        // so the TMA issue never waits on these copies
        int sslot = 0;
        uint32_t sphase = 0;
        int q = 0;
        uint32_t qphase = 0;
        bool ok = true;
        while (ok) {
            int it = 0;
            Item I{};
            if (lane == 0) it = take_item(q, qphase, I);
            it = __shfl_sync(0xffffffffu, it, 0);
            if (it < 0 || it >= n_items) break;
            bcast_item(I);
            const float *ws0, *ws1;
            weight_scale_rows(I, ws0, ws1);
            for (int kb = 0; kb < args.num_kb; ++kb) {
                int w = 1;
                if (lane == 0) w = mbar_wait(smem_u32(&sempty[sslot]), sphase ^ 1, abort_flag, args.err, ERR_WAIT_SMEM_EMPTY);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) { ok = false; break; }
                copy_scales(I, kb, sslot, ws0, ws1);
                if (++sslot == C::kScaleSlots) { sslot = 0; sphase ^= 1; }
            }
        }
        cp_async_wait_all();   // the copies must land before the CTA may exit
    } else if (warp >= 2 && warp < 2 + kEpi) {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int quad = warp & 3;           // TMEM lane quarter this warp may access
        const int grp = ew >> 2;             // token columns [HC*grp, HC*grp + HC)
        const int col_base = grp * HC;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        int sslot = 0;                       // scale slot of the K block being promoted
        uint32_t sphase = 0;
        int pbuf = 0;
        uint32_t pphase = 0;
        int q = 0;
        uint32_t qphase = 0;
        int item_count = 0;
        uint32_t kb_done = 0;                // wide kinds: K blocks promoted so far (both rings)
        bool ok = true;
        while (ok) {
            int it = 0;
            Item I{};
            if (lane == 0) it = take_item(q, qphase, I);
            it = __shfl_sync(0xffffffffu, it, 0);
            if (it < 0 || it >= n_items) break;
            bcast_item(I);
            const int n_my = max(0, min(HC, I.n - col_base));
            if constexpr (C::kWide) {
                // token-major, 256 weight rows: thread = token row r; its HC accumulators are
                //   GateUpWide: gate [0, FPT) and up [FPT, HC) of features FPT*grp ..
                //   DownWide:   the HC output rows HC*grp .. of the item's 256
                constexpr int FPT = HC / 2;          // GateUpWide: features per thread
                constexpr int kHalfChunks = C::kChunks / 2;
                const int r = quad * 32 + lane;
                const bool quad_live = quad * 32 < I.n;   // warp-uniform
                float acc[HC];
#pragma unroll
                for (int j = 0; j < HC; ++j) acc[j] = 0.f;
                // TMEM column of 16-column chunk c inside a partial buffer
                auto chunk_col = [&](int c) -> uint32_t {
                    if constexpr (KIND == Kind::GateUpWide)
                        return (c / kHalfChunks) * kBM + grp * FPT + (c % kHalfChunks) * 16;
                    else return grp * HC + c * 16;
                };
                // the partial ring and the scale ring advance together, one entry per K
                // block, so one counter gives both positions
                static_assert((C::kNumPart & (C::kNumPart - 1)) == 0 && (C::kScaleSlots & (C::kScaleSlots - 1)) == 0,
                              "ring sizes are powers of two");
                for (int kb = 0; kb < args.num_kb; ++kb, ++kb_done) {
                    const uint32_t pb = kb_done & (C::kNumPart - 1), pph = (kb_done / C::kNumPart) & 1;
                    const uint32_t ss = kb_done & (C::kScaleSlots - 1), sph = (kb_done / C::kScaleSlots) & 1;
                    // the scales first (copied well ahead, so this wait seldom blocks): no
                    // TMEM load is in flight across it, which keeps the registers free
                    if (!mbar_wait(smem_u32(&sfull[ss]), sph, abort_flag, args.err, ERR_WAIT_TMA_FULL)) { ok = false; break; }
                    // this token's scales for the K block: s_w[block, kb] * s_x[row r, kb]
                    // (rows beyond the tile's end compute on stale slot entries, never stored)
                    const float *sc = s_scale + ss * L::kScaleStride;
                    const float sx = sc[r];
                    float s_lo, s_hi;
                    if constexpr (KIND == Kind::GateUpWide) {
                        s_lo = sc[BN] * sx;       // gate block
                        s_hi = sc[BN + 1] * sx;   // up block
                    } else {
                        s_lo = sc[BN + ((grp * HC) >> 7)] * sx;   // the group's 128-row block
                        s_hi = s_lo;
                    }
                    if (!mbar_wait(smem_u32(&pfull[pb]), pph, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t tpart = t_lane + pb * C::kPartCols;
                    float p[16];
                    // one 16-column chunk in flight at a time (the accumulators and 16
                    // partials fill the thread's registers); a lane quarter wholly past
                    // the tile's last token has nothing to fold
                    if (quad_live) {
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c) {
                            tmem_ld16(tpart + chunk_col(c), p);
                            tmem_wait_ld();
                            const float s_c = (c < kHalfChunks) ? s_lo : s_hi;
                            fold16(acc + c * 16, p, s_c);
                        }
                    }
                    // every thread releases the partial and the scale slot itself: no
                    // warp barrier and no single-lane branch in the K loop
                    tc_fence_before();
                    mbar_arrive(smem_u32(&pempty[pb]));
                    mbar_arrive(smem_u32(&sempty[ss]));
                }
                if (!ok) break;
                const size_t row = static_cast<size_t>(I.row0 + r);
                if constexpr (KIND == Kind::GateUpWide) {
                    // h = silu(g) * u for the token's FPT features, then the 1x128 amax
                    // over the block's 128 features, held by the column-group warps of
                    // this lane quarter: exchanged through shared memory
                    const int H = args.num_mb * kBM;
                    const int buf = item_count & 1;
                    const uint32_t ab = smem_u32(&amax_bar[quad * 2 + buf]);
                    float *xch = s_amax + buf * 4 * kBM;   // [group][token row]
                    float am = 0.f;
                    if (quad_live) {
#pragma unroll
                        for (int j = 0; j < FPT; ++j) {
                            acc[j] = silu_f(acc[j]) * acc[FPT + j];
                            am = fmaxf(am, fabsf(acc[j]));
                        }
                    }
                    xch[grp * kBM + r] = am;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ab);
                    if (!mbar_wait(ab, (item_count >> 1) & 1, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                    if (r < I.n) {
                        float amax = xch[r];
#pragma unroll
                        for (int g = 1; g < C::kGroups; ++g) amax = fmaxf(amax, xch[g * kBM + r]);
                        const float sq = amax / 448.0f;
                        // codes in feature order, four to a word (the first in the low byte);
                        // an all-zero group has scale 0 and codes 0. The quotients h / sq
                        // are correctly rounded by Markstein's correction step (P. Markstein,
                        // IBM J. Res. Develop. 34(1), 1990): q0 = h r with r = 1 / sq
                        // correctly rounded, then q0 + (h - sq q0) r, the inner term exact
                        // by FMA. For sq >= 2^-80 an underflowing term can only touch
                        // quotients below 2^-11, under every e4m3 rounding boundary, so the
                        // codes are those of IEEE division; smaller scales, and an
                        // infinite or NaN one, divide.
                        uint32_t w[FPT / 4];
                        if (sq >= 8.27180613e-25f && sq <= 3.40282347e38f) {   // 2^-80 <= sq <= FLT_MAX
                            const float rq = 1.0f / sq;
                            auto qd = [&](float x) -> float {
                                const float q0 = x * rq;
                                return copysignf(fmaf(fmaf(-q0, sq, x), rq, q0), x);
                            };
#pragma unroll
                            for (int v = 0; v < FPT / 4; ++v) {
                                const uint32_t lo = e4m3x2(qd(acc[4 * v]), qd(acc[4 * v + 1]));
                                const uint32_t hi = e4m3x2(qd(acc[4 * v + 2]), qd(acc[4 * v + 3]));
                                w[v] = lo | (hi << 16);
                            }
                        } else {
#pragma unroll
                            for (int v = 0; v < FPT / 4; ++v) {
                                const uint32_t lo = e4m3x2(acc[4 * v] / sq, acc[4 * v + 1] / sq);
                                const uint32_t hi = e4m3x2(acc[4 * v + 2] / sq, acc[4 * v + 3] / sq);
                                w[v] = (amax == 0.f) ? 0u : (lo | (hi << 16));
                            }
                        }
                        uint4 *h4 = reinterpret_cast<uint4 *>(args.hq + row * H + I.mb * kBM + grp * FPT);
#pragma unroll
                        for (int v = 0; v < FPT / 16; ++v)
                            h4[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
                        if (grp == 0) args.hs_t[static_cast<size_t>(I.mb) * args.total_rows + row] = sq;
                    }
                } else {
                    // each lane holds its token's HC outputs (2 HC bytes of bf16). Stored
                    // directly, one 16-byte store instruction would touch 32 rows; instead
                    // eight rows at a time pass through this warp's slot (16-byte chunk v
                    // of slot row q at chunk v ^ q: conflict-free both ways) and leave as
                    // stores of whole row segments.
                    const int nout = args.num_mb * 2 * kBM;   // output features per row
                    uint4 w[HC / 8];
#pragma unroll
                    for (int v = 0; v < HC / 8; ++v) {
                        w[v].x = bf16x2_bits(acc[8 * v + 0], acc[8 * v + 1]);
                        w[v].y = bf16x2_bits(acc[8 * v + 2], acc[8 * v + 3]);
                        w[v].z = bf16x2_bits(acc[8 * v + 4], acc[8 * v + 5]);
                        w[v].w = bf16x2_bits(acc[8 * v + 6], acc[8 * v + 7]);
                    }
                    constexpr int kRowBytes = HC * 2;         // one slot row
                    constexpr int kRowChunks = HC / 8;        // its 16-byte chunks
                    uint8_t *slot = s_xpose + ew * 8 * kRowBytes;
                    if (quad_live) {
                    __nv_bfloat16 *obase = args.out + static_cast<size_t>(I.mb) * 2 * kBM + grp * HC;
#pragma unroll
                    for (int pass = 0; pass < 4; ++pass) {
                        if ((lane >> 3) == pass) {
                            const int q = lane & 7;
#pragma unroll
                            for (int v = 0; v < kRowChunks; ++v)
                                *reinterpret_cast<uint4 *>(slot + q * kRowBytes + ((v ^ q) << 4)) = w[v];
                        }
                        __syncwarp();
#pragma unroll
                        for (int part = 0; part < kRowChunks / 4; ++part) {
                            const int idx = part * 32 + lane;
                            const int q = idx / kRowChunks, c = idx % kRowChunks;
                            const uint4 v4 = *reinterpret_cast<const uint4 *>(slot + q * kRowBytes + ((c ^ q) << 4));
                            const int tr = quad * 32 + pass * 8 + q;   // token row in the tile
                            if (tr < I.n)
                                *reinterpret_cast<uint4 *>(obase + static_cast<size_t>(I.row0 + tr) * nout + c * 8) = v4;
                        }
                        __syncwarp();
                    }
                    }
                }
            } else if constexpr (C::kTM) {
                // token-major: this thread's TMEM lane is token row r of the tile, its
                // columns the weight rows [col_base, col_base + 64) of block mb
                const int r = quad * 32 + lane;
                float acc[HC];
#pragma unroll
                for (int j = 0; j < HC; ++j) acc[j] = 0.f;
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&pfull[pbuf]), pphase, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t tcol = t_lane + pbuf * C::kPartCols + col_base;
                    float p[C::kChunks][16];
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) tmem_ld16(tcol + c * 16, p[c]);
                    // while the loads are in flight: this token's scale for the K block,
                    // s_w[mb, kb] * s_x[row r, kb] (rows beyond the tile's end compute on
                    // stale slot entries and are never stored)
                    if (!mbar_wait(smem_u32(&sfull[sslot]), sphase, abort_flag, args.err, ERR_WAIT_TMA_FULL)) {
                        tmem_wait_ld();
                        ok = false;
                        break;
                    }
                    const float *sc = s_scale + sslot * L::kScaleStride;
                    const float s_kb = sc[BN] * sc[r];
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) fold16(acc + c * 16, p[c], s_kb);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&pempty[pbuf]));
                        mbar_arrive(smem_u32(&sempty[sslot]));
                    }
                    if (++pbuf == C::kNumPart) { pbuf = 0; pphase ^= 1; }
                    if (++sslot == C::kScaleSlots) { sslot = 0; sphase ^= 1; }
                }
                if (!ok) break;
                if (r < I.n) {
                    // one token's 64 consecutive outputs: 16-byte stores
                    const size_t row = static_cast<size_t>(I.row0 + r);
                    const int nout = args.num_mb * kBM;   // output features per row
                    const size_t col = static_cast<size_t>(I.mb) * kBM + col_base;
                    uint4 *o4 = reinterpret_cast<uint4 *>(args.out + row * nout + col);
#pragma unroll
                    for (int v = 0; v < HC / 8; ++v) {
                        uint4 w;
                        w.x = bf16x2_bits(acc[8 * v + 0], acc[8 * v + 1]);
                        w.y = bf16x2_bits(acc[8 * v + 2], acc[8 * v + 3]);
                        w.z = bf16x2_bits(acc[8 * v + 4], acc[8 * v + 5]);
                        w.w = bf16x2_bits(acc[8 * v + 6], acc[8 * v + 7]);
                        o4[v] = w;
                    }
                }
            } else if constexpr (C::kPromote) {
                constexpr bool kTwo = (C::kATiles == 2);
                float acc0[HC], acc1[kTwo ? HC : 1];
#pragma unroll
                for (int j = 0; j < HC; ++j) acc0[j] = 0.f;
                if constexpr (kTwo) {
#pragma unroll
                    for (int j = 0; j < HC; ++j) acc1[j] = 0.f;
                }
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    // 1. wait for this K block's partial products, start loading them
                    if (!mbar_wait(smem_u32(&pfull[pbuf]), pphase, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t tcol = t_lane + pbuf * C::kPartCols + col_base;
                    // the partial's 16-column chunks (gate first, then up for the
                    // two-tile kinds) are loaded kLd at a time: all of them when the
                    // registers allow, one at a time in the wide (16-warp) epilogue
                    constexpr int kTot = C::kATiles * C::kChunks;
                    constexpr int kLd = (C::kThreads > 384) ? 2 : kTot;
                    float p[kLd][16];
                    auto load_batch = [&](int t0) {
#pragma unroll
                        for (int b = 0; b < kLd; ++b) {
                            const int t = t0 + b;
                            tmem_ld16(tcol + (t / C::kChunks) * BN + (t % C::kChunks) * 16, p[b]);
                        }
                    };
                    if (n_my > 0) load_batch(0);
                    // 2. while they are in flight: the combined scales
                    //    s_w[mb, kb] * s_x[row_j, kb] of this warp's columns, once per
                    //    K block, into a warp-private slot
                    if (!mbar_wait(smem_u32(&sfull[sslot]), sphase, abort_flag, args.err, ERR_WAIT_TMA_FULL)) {
                        tmem_wait_ld();
                        ok = false;
                        break;
                    }
                    const float *sc = s_scale + sslot * L::kScaleStride;
                    float *cs = s_cs + (ew * 2 + (kb & 1)) * C::kATiles * HC;
                    {
                        const float sw0 = sc[BN];
                        const float sw1 = kTwo ? sc[BN + 1] : 0.f;
#pragma unroll
                        for (int j = lane; j < HC; j += 32) {
                            const float a = sc[col_base + j];
                            cs[j] = sw0 * a;
                            if constexpr (kTwo) cs[HC + j] = sw1 * a;
                        }
                    }
                    __syncwarp();
                    // 3. fold the partials into the fp32 accumulators
                    if (n_my > 0) {
#pragma unroll
                        for (int t0 = 0; t0 < kTot; t0 += kLd) {
                            if (t0 > 0) load_batch(t0);
                            tmem_wait_ld();
#pragma unroll
                            for (int b = 0; b < kLd; ++b) {
                                const int t = t0 + b;
                                const int pass = t / C::kChunks, c = t % C::kChunks;
                                float *acc = (pass == 0) ? acc0 : acc1;
                                const float4 *s4 = reinterpret_cast<const float4 *>(cs + pass * HC + c * 16);
#pragma unroll
                                for (int v = 0; v < 4; ++v) {
                                    const float4 a4 = s4[v];
                                    const int j = c * 16 + v * 4;
                                    acc[j + 0] = fmaf(a4.x, p[b][v * 4 + 0], acc[j + 0]);
                                    acc[j + 1] = fmaf(a4.y, p[b][v * 4 + 1], acc[j + 1]);
                                    acc[j + 2] = fmaf(a4.z, p[b][v * 4 + 2], acc[j + 2]);
                                    acc[j + 3] = fmaf(a4.w, p[b][v * 4 + 3], acc[j + 3]);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(smem_u32(&pempty[pbuf]));
                        mbar_arrive(smem_u32(&sempty[sslot]));
                    }
                    if (++pbuf == C::kNumPart) { pbuf = 0; pphase ^= 1; }
                    if (++sslot == C::kScaleSlots) { sslot = 0; sphase ^= 1; }
                }
                if (!ok) break;
                const int wrow = quad * 32 + lane;  // weight row inside the 128-row block
                if constexpr (KIND == Kind::GateUp) {
                    // h = silu(g) * u, then 1x128 quantisation over the block's 128 rows
                    const int H = args.num_mb * kBM;
                    const int buf = item_count & 1;
                    const uint32_t ab = smem_u32(&amax_bar[grp * 2 + buf]);
                    float *xch = s_amax + (grp * 2 + buf) * 4 * HC;
                    if (n_my > 0) {
#pragma unroll
                        for (int j = 0; j < HC; ++j) {
                            acc0[j] = silu_f(acc0[j]) * acc1[j];
                            const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(acc0[j])));
                            if (lane == 0) xch[quad * HC + j] = __uint_as_float(m);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ab);
                    if (!mbar_wait(ab, (item_count >> 1) & 1, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
#pragma unroll
                    for (int j = 0; j < HC; ++j) {
                        if (j < n_my) {
                            const float amax = fmaxf(fmaxf(xch[j], xch[HC + j]), fmaxf(xch[2 * HC + j], xch[3 * HC + j]));
                            const float s = amax / 448.0f;
                            const uint8_t code = (amax == 0.f) ? uint8_t(0) : e4m3(acc0[j] / s);
                            const size_t row = static_cast<size_t>(I.row0 + col_base + j);
                            args.hq[row * H + I.mb * kBM + wrow] = code;
                            if (wrow == 0) args.hs_t[static_cast<size_t>(I.mb) * args.total_rows + row] = s;
                        }
                    }
                } else {
                    static_assert(KIND == Kind::DownPair, "swap-AB promoted kinds: GateUp, DownPair");
                    const int dout = args.num_mb * 2 * kBM;
#pragma unroll
                    for (int j = 0; j < HC; ++j) {
                        if (j < n_my) {
                            const size_t row = static_cast<size_t>(I.row0 + col_base + j);
                            __nv_bfloat16 *o = args.out + row * dout + I.mb * 2 * kBM + wrow;
                            o[0] = __float2bfloat16_rn(acc0[j]);
                            o[kBM] = __float2bfloat16_rn(acc1[j]);
                        }
                    }
                }
            } else {
                // Router: one accumulator per item (one K split)
                if (!mbar_wait(smem_u32(&pfull[pbuf]), pphase, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                tc_fence_after();
                float *dst = args.logits + static_cast<size_t>(I.ks) * args.total_rows * args.n_valid;
                const int nt = (C::kRouterAll && args.a_tiles > 0) ? args.a_tiles : 1;
                for (int t = 0; t < nt; ++t) {
                    const uint32_t tcol = t_lane + pbuf * C::kPartCols + t * BN + col_base;
                    const int e = (nt > 1 ? t : I.mb) * kBM + quad * 32 + lane;
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        if (c * 16 < n_my) {
                            float p0[16];
                            tmem_ld16(tcol + c * 16, p0);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int j = c * 16 + i;
                                if (j < n_my && e < args.n_valid)
                                    dst[static_cast<size_t>(I.row0 + col_base + j) * args.n_valid + e] = p0[i];
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pempty[pbuf]));
                if (++pbuf == C::kNumPart) { pbuf = 0; pphase ^= 1; }
            }
            ++item_count;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<C::kTmemCols>(tmem_base);
}

template <Kind KIND, int BN>
__global__ void __launch_bounds__(KindCfg<KIND, BN>::kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ ActMaps map_b,
                    const GemmArgs args) {
    grouped_gemm_body<KIND, BN>(map_a, map_b, args);
}

// The CTAs of the 256-row token-major kinds: the register cap is what each
// sub-partition's register file (16,384 registers) allows for its share of the
// warps, enough for the epilogue's accumulators and a 16-column TMEM chunk.
template <Kind KIND, int BN>
__global__ void __maxnreg__((KindCfg<KIND, BN>::kWideRegs))
grouped_gemm_wide_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ ActMaps map_b,
                         const GemmArgs args) {
    grouped_gemm_body<KIND, BN>(map_a, map_b, args);
}

template <Kind KIND, int BN>
constexpr size_t gemm_smem_bytes() { return SmemLayout<KIND, BN>::kLaunchBytes; }

}  // namespace moe
