// Persistent grouped GEMM on the tcgen05 tensor cores (sm_103a).
//
// Swap-AB formulation: the weight rows of one 128-row block are the MMA M
// dimension (TMEM lanes) and the tokens of one segment tile are the MMA N
// dimension (TMEM columns). A "work item" is (group g, 128-row weight block mb,
// token tile nt); items of one group are ordered mb-major so that the token
// tiles sharing a weight block run at the same time on neighbouring CTAs.
//
// Roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: weight tile(s) + activation rows per 128-byte K block
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2..9  epilogue: two groups of four warps, one per half of the token
//               columns; each warp reads its 32-lane quarter of TMEM
//
// FP8 kinds (gate/up and down): e4m3 x e4m3 -> fp32 with one partial product
// per 128-wide K block, because the weight scale (per 128x128 block) and the
// activation scale (per token and 128-wide K block) both change at every K
// block. The epilogue promotes each partial into fp32 registers:
//     acc[j] += (s_w[mb, kb] * s_x[row_j, kb]) * partial[j]
// TMEM holds two partial buffers so the MMAs of K block kb+1 run while block
// kb is promoted.
//
// Router kind: bf16 x bf16 -> fp32, accumulated in TMEM over the whole K
// range; the epilogue writes fp32 logits.
#pragma once
#include "ptx.cuh"

namespace moe {

enum class Kind { GateUp, Down, Router };

constexpr int kBN = 128;                    // max tokens per tile (MMA N)
constexpr int kBM = 128;                    // weight rows per tile (MMA M)
constexpr int kKBytes = 128;                // bytes of K per stage (= one swizzle row)
constexpr int kATileBytes = kBM * kKBytes;  // 16 KB
constexpr int kBTileBytes = kBN * kKBytes;  // 16 KB
constexpr int kActBoxRows = 16;             // activation TMA box height
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kMaxGroups = 1032;            // routed + shared experts, padded

template <Kind K> struct KindCfg;
template <> struct KindCfg<Kind::GateUp> {
    static constexpr int kATiles = 2, kStages = 4, kTmemCols = 512, kPartCols = 256;
    static constexpr bool kPromote = true, kBf16 = false;
};
template <> struct KindCfg<Kind::Down> {
    static constexpr int kATiles = 1, kStages = 6, kTmemCols = 256, kPartCols = 128;
    static constexpr bool kPromote = true, kBf16 = false;
};
template <> struct KindCfg<Kind::Router> {
    static constexpr int kATiles = 1, kStages = 6, kTmemCols = 256, kPartCols = 128;
    static constexpr bool kPromote = false, kBf16 = true;
};

struct GemmArgs {
    int G;                    // groups (experts, routed first, shared last)
    int num_kb;               // K blocks of 128 bytes
    int num_mb;               // 128-row blocks of weight rows per group (output features / 128)
    int total_rows;           // rows of the activation buffer
    int single_rows;          // >= 0: one group of that many rows (row_start / tile_prefix unused)
    const int *row_start;     // [G+1] first activation row of each group's segment
    const int *tile_prefix;   // [G+1] prefix sum of ceil(rows_g / kBN)
    const float *act_scale_t; // [num_kb][total_rows]  (FP8 kinds)
    const float *w_scale;     // GateUp: [G][2][num_mb][num_kb]; Down: [G][num_mb][num_kb]
    int a_rows_per_group;     // weight rows of one group in the A tensor map (GateUp: 2*H, Down: d_out)
    int a_second_offset;      // GateUp: row offset of up_proj inside a group (H)
    uint8_t *hq;              // GateUp: [total_rows][num_mb*128]
    float *hs_t;              // GateUp: [num_mb][total_rows]
    __nv_bfloat16 *out;       // Down: [total_rows][num_mb*128]
    float *logits;            // Router: [total_rows][n_valid]
    int n_valid;              // Router: valid weight rows (experts)
    unsigned int *err;        // device error word (bounded waits that gave up)
};

struct Item {
    int g, mb, row0, n;
};

__device__ __forceinline__ bool decode_item(int it, const GemmArgs &a, const int *s_tp,
                                            const int *s_rs, Item &o) {
    if (a.single_rows >= 0) {
        const int nt_total = (a.single_rows + kBN - 1) / kBN;
        o.g = 0;
        o.mb = it / nt_total;
        const int nt = it - o.mb * nt_total;
        o.row0 = nt * kBN;
        o.n = min(kBN, a.single_rows - o.row0);
        return o.n > 0 && o.mb < a.num_mb;
    }
    const int key = it / a.num_mb;
    int lo = 0, hi = a.G;  // find the last g with tile_prefix[g] <= key
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_tp[mid] <= key) lo = mid; else hi = mid;
    }
    const int g = lo;
    const int nt_g = s_tp[g + 1] - s_tp[g];
    if (nt_g <= 0) return false;
    const int li = it - a.num_mb * s_tp[g];
    o.g = g;
    o.mb = li / nt_g;
    const int nt = li - o.mb * nt_g;
    o.row0 = s_rs[g] + nt * kBN;
    o.n = min(kBN, s_rs[g + 1] - o.row0);
    return o.n > 0 && o.mb < a.num_mb;
}

__device__ __forceinline__ int total_items(const GemmArgs &a, const int *s_tp) {
    if (a.single_rows >= 0) return a.num_mb * ((a.single_rows + kBN - 1) / kBN);
    return a.num_mb * s_tp[a.G];
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Shared-memory carve-up of one CTA (offsets from a 1024-byte aligned base).
template <Kind KIND> struct SmemLayout {
    using C = KindCfg<KIND>;
    static constexpr int kStageBytes = C::kATiles * kATileBytes + kBTileBytes;
    static constexpr int kNumBars = 2 * C::kStages + 2 + 2 + 1 + 4;
    static constexpr size_t kBars = static_cast<size_t>(C::kStages) * kStageBytes;
    static constexpr size_t kMisc = (kBars + kNumBars * 8 + 15) & ~size_t(15);
    static constexpr size_t kTp = kMisc + 16;
    static constexpr size_t kRs = kTp + kMaxGroups * 4;
    static constexpr size_t kScale = kRs + kMaxGroups * 4;
    static constexpr size_t kAmax = kScale + kEpiWarps * 2 * 64 * 4;
    static constexpr size_t kEnd = kAmax + 2 * 2 * 4 * 64 * 4;
    static constexpr size_t kLaunchBytes = kEnd + 1024;  // + alignment slack of the dynamic base
    static_assert(kBars % 1024 == 0 && kScale % 16 == 0, "alignment");
};

template <Kind KIND>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const GemmArgs args) {
    using C = KindCfg<KIND>;
    constexpr int kStageBytes = SmemLayout<KIND>::kStageBytes;
    constexpr int kKbElems = C::kBf16 ? 64 : 128;
    constexpr uint32_t kFmt = C::kBf16 ? 1u : 0u;

    extern __shared__ uint8_t smem_raw[];
    using L = SmemLayout<KIND>;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kBars);
    uint64_t *full = bars;
    uint64_t *empty = full + C::kStages;
    uint64_t *pfull = empty + C::kStages;
    uint64_t *pempty = pfull + 2;
    uint64_t *mma_done = pempty + 2;
    uint64_t *amax_bar = mma_done + 1;  // [2 halves][2 buffers]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
    int *s_tp = reinterpret_cast<int *>(smem + L::kTp);
    int *s_rs = reinterpret_cast<int *>(smem + L::kRs);
    float *s_scale = reinterpret_cast<float *>(smem + L::kScale);  // [8 warps][2][64]
    float *s_amax = reinterpret_cast<float *>(smem + L::kAmax);    // [2 halves][2 bufs][4 quads][64]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (args.single_rows < 0) {
        for (int i = threadIdx.x; i <= args.G; i += blockDim.x) {
            s_tp[i] = args.tile_prefix[i];
            s_rs[i] = args.row_start[i];
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&pfull[b]), 1);
            mbar_init(smem_u32(&pempty[b]), kEpiWarps);
        }
        mbar_init(smem_u32(mma_done), 1);
        for (int b = 0; b < 4; ++b) mbar_init(smem_u32(&amax_bar[b]), 4);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map_a);
        tma_prefetch_desc(&map_b);
    }
    if (warp == 1) tmem_alloc<C::kTmemCols>(smem_u32(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int n_items = total_items(args, s_tp);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                Item I;
                if (!decode_item(it, args, s_tp, s_rs, I)) { record_error(args.err, ERR_BAD_TILE); continue; }
                const int nb16 = (I.n + kActBoxRows - 1) / kActBoxRows;
                const uint32_t bytes = C::kATiles * kATileBytes + nb16 * kActBoxRows * kKBytes;
                int arow0, arow1 = 0;
                if (KIND == Kind::Router) {
                    arow0 = I.mb * kBM;
                } else {
                    arow0 = I.g * args.a_rows_per_group + I.mb * kBM;
                    arow1 = arow0 + args.a_second_offset;
                }
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1, abort_flag, args.err, ERR_WAIT_SMEM_EMPTY)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, bytes);
                    const uint32_t sbase = smem_u32(stages + stage * kStageBytes);
                    const int kx = kb * kKbElems;
                    tma_load_2d(sbase, &map_a, fb, kx, arow0, pol_w);
                    if (C::kATiles == 2) tma_load_2d(sbase + kATileBytes, &map_a, fb, kx, arow1, pol_w);
                    const uint32_t bdst = sbase + C::kATiles * kATileBytes;
                    for (int i = 0; i < nb16; ++i)
                        tma_load_2d(bdst + i * kActBoxRows * kKBytes, &map_b, fb, kx, I.row0 + i * kActBoxRows, pol_x);
                    issued_mask |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
            // every issued copy must land before the CTA may exit
            for (int s = 0; s < C::kStages; ++s)
                if (issued_mask & (1u << s)) mbar_wait_drain(smem_u32(&full[s]), (issued_parity >> s) & 1u, args.err);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int pbuf = 0;
            uint32_t pphase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                Item I;
                if (!decode_item(it, args, s_tp, s_rs, I)) continue;
                const int n_mma = (I.n + 15) & ~15;
                const uint32_t idesc = idesc_make(kFmt, kFmt, kBM, n_mma);
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, args.err, ERR_WAIT_TMA_FULL)) { ok = false; break; }
                    if (C::kPromote || kb == 0) {
                        if (!mbar_wait(smem_u32(&pempty[pbuf]), pphase ^ 1, abort_flag, args.err, ERR_WAIT_PART_EMPTY)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    const uint32_t sbase = smem_u32(stages + stage * kStageBytes);
                    const uint32_t bbase = sbase + C::kATiles * kATileBytes;
                    const uint32_t dcol = tmem_base + pbuf * C::kPartCols;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = C::kPromote ? (k > 0) : (kb > 0 || k > 0);
                        const uint64_t bdesc = sdesc_sw128(bbase + k * 32);
                        const uint64_t adesc = sdesc_sw128(sbase + k * 32);
                        if constexpr (C::kBf16) mma_bf16(dcol, adesc, bdesc, idesc, acc);
                        else mma_f8(dcol, adesc, bdesc, idesc, acc);
                        if constexpr (C::kATiles == 2)
                            mma_f8(dcol + kBN, sdesc_sw128(sbase + kATileBytes + k * 32), bdesc, idesc, acc);
                    }
                    mma_commit(smem_u32(&empty[stage]));
                    if (C::kPromote || kb == args.num_kb - 1) {
                        mma_commit(smem_u32(&pfull[pbuf]));
                        pbuf ^= 1;
                        if (pbuf == 0) pphase ^= 1;
                    }
                    if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                }
            }
            // all MMAs must finish before TMEM is released
            mma_commit(smem_u32(mma_done));
            mbar_wait_drain(smem_u32(mma_done), 0, args.err);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int ew = warp - 2;
        const int quad = warp & 3;           // TMEM lane quarter this warp may access
        const int half = ew >> 2;            // token columns [64*half, 64*half + 64)
        const int col_base = half * 64;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
        float *my_scale = s_scale + ew * 2 * 64;
        int pbuf = 0;
        uint32_t pphase = 0;
        int item_count = 0;
        bool ok = true;
        for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            Item I;
            if (!decode_item(it, args, s_tp, s_rs, I)) continue;
            const int n_my = max(0, min(64, I.n - col_base));
            if constexpr (C::kPromote) {
                constexpr bool kTwo = (KIND == Kind::GateUp);
                float acc0[64], acc1[kTwo ? 64 : 1];
#pragma unroll
                for (int j = 0; j < 64; ++j) acc0[j] = 0.f;
#pragma unroll
                for (int j = 0; j < (kTwo ? 64 : 1); ++j) acc1[j] = 0.f;
                const float *ws0, *ws1;
                if constexpr (kTwo) {
                    ws0 = args.w_scale + (static_cast<size_t>(I.g * 2 + 0) * args.num_mb + I.mb) * args.num_kb;
                    ws1 = args.w_scale + (static_cast<size_t>(I.g * 2 + 1) * args.num_mb + I.mb) * args.num_kb;
                } else {
                    ws0 = args.w_scale + (static_cast<size_t>(I.g) * args.num_mb + I.mb) * args.num_kb;
                    ws1 = ws0;
                }
                const float *sa_col = args.act_scale_t + I.row0 + col_base;
                const size_t sa_stride = static_cast<size_t>(args.total_rows);
                float pf0 = (lane < n_my) ? sa_col[lane] : 0.f;
                float pf1 = (lane + 32 < n_my) ? sa_col[lane + 32] : 0.f;
                float wr0 = 0.f, wr1 = 0.f;
                for (int kb = 0; kb < args.num_kb; ++kb) {
                    float *slot = my_scale + (kb & 1) * 64;
                    slot[lane] = pf0;
                    slot[lane + 32] = pf1;
                    if ((kb & 31) == 0) {
                        wr0 = (kb + lane < args.num_kb) ? ws0[kb + lane] : 0.f;
                        wr1 = (kb + lane < args.num_kb) ? ws1[kb + lane] : 0.f;
                    }
                    __syncwarp();
                    if (kb + 1 < args.num_kb) {
                        const float *nxt = sa_col + (kb + 1) * sa_stride;
                        pf0 = (lane < n_my) ? nxt[lane] : 0.f;
                        pf1 = (lane + 32 < n_my) ? nxt[lane + 32] : 0.f;
                    }
                    const float sw0 = __shfl_sync(0xffffffffu, wr0, kb & 31);
                    const float sw1 = __shfl_sync(0xffffffffu, wr1, kb & 31);
                    if (!mbar_wait(smem_u32(&pfull[pbuf]), pphase, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t tcol = t_lane + pbuf * C::kPartCols + col_base;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c * 16 < n_my) {
                            float p0[16], p1[16];
                            tmem_ld16(tcol + c * 16, p0);
                            if constexpr (kTwo) tmem_ld16(tcol + kBN + c * 16, p1);
                            tmem_wait_ld();
                            const float4 *sv = reinterpret_cast<const float4 *>(slot + c * 16);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                const float4 s4 = sv[v];
                                const float sa[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int j = c * 16 + v * 4 + i;
                                    acc0[j] = fmaf(sw0 * sa[i], p0[v * 4 + i], acc0[j]);
                                    if constexpr (kTwo) acc1[j] = fmaf(sw1 * sa[i], p1[v * 4 + i], acc1[j]);
                                }
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&pempty[pbuf]));
                    pbuf ^= 1;
                    if (pbuf == 0) pphase ^= 1;
                }
                if (!ok) break;
                const int wrow = quad * 32 + lane;  // weight row inside the 128-row block
                if constexpr (KIND == Kind::GateUp) {
                    // h = silu(g) * u, then 1x128 quantisation over the block's 128 rows
                    const int H = args.num_mb * kBM;
                    const int buf = item_count & 1;
                    const uint32_t ab = smem_u32(&amax_bar[half * 2 + buf]);
                    float *xch = s_amax + (half * 2 + buf) * 4 * 64;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c * 16 < n_my) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int j = c * 16 + i;
                                acc0[j] = silu_f(acc0[j]) * acc1[j];
                                const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(acc0[j])));
                                if (lane == 0) xch[quad * 64 + j] = __uint_as_float(m);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ab);
                    if (!mbar_wait(ab, (item_count >> 1) & 1, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c * 16 < n_my) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int j = c * 16 + i;
                                if (j < n_my) {
                                    const float amax = fmaxf(fmaxf(xch[j], xch[64 + j]), fmaxf(xch[128 + j], xch[192 + j]));
                                    const float s = amax / 448.0f;
                                    const uint8_t code = (amax == 0.f) ? uint8_t(0) : e4m3(acc0[j] / s);
                                    const size_t row = static_cast<size_t>(I.row0 + col_base + j);
                                    args.hq[row * H + I.mb * kBM + wrow] = code;
                                    if (wrow == 0) args.hs_t[static_cast<size_t>(I.mb) * args.total_rows + row] = s;
                                }
                            }
                        }
                    }
                } else {
                    const int dout = args.num_mb * kBM;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c * 16 < n_my) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int j = c * 16 + i;
                                if (j < n_my) {
                                    const size_t row = static_cast<size_t>(I.row0 + col_base + j);
                                    args.out[row * dout + I.mb * kBM + wrow] = __float2bfloat16_rn(acc0[j]);
                                }
                            }
                        }
                    }
                }
            } else {
                // Router: one accumulator per item
                if (!mbar_wait(smem_u32(&pfull[pbuf]), pphase, abort_flag, args.err, ERR_WAIT_PART_FULL)) { ok = false; break; }
                tc_fence_after();
                const uint32_t tcol = t_lane + pbuf * C::kPartCols + col_base;
                const int e = I.mb * kBM + quad * 32 + lane;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c * 16 < n_my) {
                        float p0[16];
                        tmem_ld16(tcol + c * 16, p0);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int j = c * 16 + i;
                            if (j < n_my && e < args.n_valid)
                                args.logits[static_cast<size_t>(I.row0 + col_base + j) * args.n_valid + e] = p0[i];
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&pempty[pbuf]));
                pbuf ^= 1;
                if (pbuf == 0) pphase ^= 1;
            }
            ++item_count;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc<C::kTmemCols>(tmem_base);
}

template <Kind KIND>
constexpr size_t gemm_smem_bytes() { return SmemLayout<KIND>::kLaunchBytes; }

}  // namespace moe
