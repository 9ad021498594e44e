// Bandwidth- and latency-bound kernels of the MoE layer: 1x128 activation
// quantisation, router top-k, token permutation and the weighted combine, and
// the block pieces around the layer (RMSNorm + quantisation of its input; the
// combine fused with the residual addition and the next block's RMSNorm).
#pragma once
#include "ptx.cuh"

namespace moe {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void unpack_bf16x8(const uint4 &raw, float (&v)[8]) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __low2float(h[i]);
        v[2 * i + 1] = __high2float(h[i]);
    }
}

// ------------------------------------------------------------------ quantise
// The quotients x / s of one group, correctly rounded as IEEE division rounds
// them, by Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1),
// 1990): with r = 1 / s correctly rounded, q0 = x r, e = x - s q0 (exact, one
// FMA) and q = q0 + e r, each rounded to nearest, q is the correctly rounded
// x / s when no step over- or underflows. The quotients here are at most 448 in
// magnitude. For s >= 2^-80, e can lose bits to underflow only where the quotient
// lies below 2^-11, under every e4m3 rounding boundary, so the codes equal those
// of IEEE division. A zero quotient takes x's sign, as x / s does. Smaller scales,
// and an infinite or NaN scale (a group holding an infinity or a NaN, where the
// correction term would be NaN), fall back to the division.
template <int N>
__device__ __forceinline__ void div_by_scale(const float (&x)[N], float s, float (&q)[N]) {
    if (s >= 8.27180613e-25f && s <= 3.40282347e38f) {   // 2^-80 <= s <= FLT_MAX
        const float r = 1.0f / s;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float q0 = x[i] * r;
            q[i] = copysignf(fmaf(fmaf(-q0, s, x[i]), r, q0), x[i]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) q[i] = x[i] / s;
    }
}

// Half a warp per 128-wide group (lane l of the half holds elements 8l..8l+7, one
// 16-byte load of bf16), two groups per warp and kQuantPairs pairs per loop trip, so
// each warp has eight groups' loads in flight. Groups are numbered row-major (group g
// of row r is r * cols/128 + g), so a run of groups is a run of memory; each warp
// takes an equal contiguous run of trips (eight groups each) and first sends its
// whole input run towards L2 with one bulk prefetch. Against a grid-strided order
// with the same loads: 62.1 -> 53.9 us for 8192 x 7168 bf16 on one GB300.
// s = amax / 448 (IEEE fp32 division), q = e4m3(x / s) (x / s correctly rounded,
// RNE to e4m3, saturating); amax = 0 gives s = 0 and zero codes.
constexpr int kQuantPairs = 4;

template <bool kBf16In>
__global__ void quant_1x128_kernel(const void *__restrict__ in, int64_t rows, int cols,
                                   uint8_t *__restrict__ q, float *__restrict__ s, int s_transposed) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int half = lane >> 4, l16 = lane & 15;
    const int gpr = cols / 128;
    const int64_t n_groups = rows * gpr;
    const int64_t n_chunks = (n_groups + 2 * kQuantPairs - 1) / (2 * kQuantPairs);   // 2 kQuantPairs groups each
    const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // warp w takes the contiguous chunks [c0, c1): its (row, group) then advances by
    // two groups a pair, with no division past the first
    const int64_t per = (n_chunks + nwarps - 1) / nwarps;
    const int64_t c0 = warp0 * per, c1 = (c0 + per < n_chunks) ? c0 + per : n_chunks;
    if (c0 >= c1) return;
    {
        // the warp's whole input range (contiguous: groups are row-major) on its way to L2
        const int64_t eb = kBf16In ? 256 : 512;
        const int64_t gfirst = c0 * 2 * kQuantPairs;
        const int64_t glast = (c1 * 2 * kQuantPairs < n_groups) ? c1 * 2 * kQuantPairs : n_groups;
        if (lane == 0 && glast > gfirst)
            l2_prefetch_bulk(static_cast<const uint8_t *>(in) + gfirst * eb, static_cast<uint32_t>((glast - gfirst) * eb));
    }
    int64_t gi0 = c0 * 2 * kQuantPairs + half;
    int64_t r = gi0 / gpr;
    int g = static_cast<int>(gi0 - r * gpr);
    const int64_t gend = c1 * 2 * kQuantPairs;
    for (int64_t gb = c0 * 2 * kQuantPairs; gb < gend; gb += 2 * kQuantPairs) {
        float v[kQuantPairs][8];
        int64_t base[kQuantPairs], gi[kQuantPairs], rr[kQuantPairs];
        int gg[kQuantPairs];
#pragma unroll
        for (int u = 0; u < kQuantPairs; ++u) {
            gi[u] = gb + 2 * u + half;
            rr[u] = r;
            gg[u] = g;
            base[u] = r * cols + g * 128 + l16 * 8;
            g += 2;
            while (g >= gpr) { g -= gpr; ++r; }
#pragma unroll
            for (int i = 0; i < 8; ++i) v[u][i] = 0.f;
            if (gi[u] < n_groups) {
                if constexpr (kBf16In) {
                    unpack_bf16x8(*reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(in) + base[u]), v[u]);
                } else {
                    const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(in) + base[u]);
                    const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(in) + base[u] + 4);
                    v[u][0] = a.x; v[u][1] = a.y; v[u][2] = a.z; v[u][3] = a.w;
                    v[u][4] = b.x; v[u][5] = b.y; v[u][6] = b.z; v[u][7] = b.w;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kQuantPairs; ++u) {
            unsigned m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, __float_as_uint(fabsf(v[u][i])));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off, 16));
            if (gi[u] >= n_groups) continue;
            const float amax = __uint_as_float(m);
            const float sc = amax / 448.0f;
            uint2 packed = make_uint2(0u, 0u);
            if (amax != 0.f) {
                float d8[8];
                div_by_scale(v[u], sc, d8);
                packed.x = static_cast<uint32_t>(e4m3x2(d8[0], d8[1])) | (static_cast<uint32_t>(e4m3x2(d8[2], d8[3])) << 16);
                packed.y = static_cast<uint32_t>(e4m3x2(d8[4], d8[5])) | (static_cast<uint32_t>(e4m3x2(d8[6], d8[7])) << 16);
            }
            *reinterpret_cast<uint2 *>(q + base[u]) = packed;
            if (l16 == 0) s[s_transposed ? (static_cast<int64_t>(gg[u]) * rows + rr[u]) : gi[u]] = sc;
        }
    }
}

// ------------------------------------------------------------------ top-k
// One warp per token; lane l holds experts l + 32 i, i < NPER (NPER >= ceil(E / 32)).
// The logit is the sum of the router GEMM's K-split partials, added in split order;
// scores s = sigmoid(logit) in fp32; choice c = s + bias. Each lane keeps the best
// of its own choices (c desc, expert id asc: its ids ascend with i, so the first
// strict maximum); each of the k rounds takes the warp's best of the lanes' bests,
// and only the lane that owned it strikes it out and rescans its own NPER values.
// Weights come from s.
template <int NPER>
__global__ void topk_kernel(const float *__restrict__ logits, int splits, const float *__restrict__ bias,
                            int T, int E, int k, float route_scale, int32_t *__restrict__ topk_idx,
                            float *__restrict__ topk_w, float *__restrict__ scores) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (t >= T) return;
    const float *lrow = logits + static_cast<size_t>(t) * E;
    const size_t split_stride = static_cast<size_t>(T) * E;
    float sv[NPER], cv[NPER];
    // logits: the split partials added in split order; the loads of the first
    // kGather splits are all issued before the first addition
    constexpr int kGather = (NPER <= 12) ? 4 : 1;
#pragma unroll
    for (int i = 0; i < NPER; ++i) sv[i] = (lane + 32 * i < E) ? lrow[lane + 32 * i] : 0.f;
    if constexpr (kGather > 1) {
        float pv[kGather - 1][NPER];
#pragma unroll
        for (int sp = 1; sp < kGather; ++sp) {
            const float *prow = lrow + sp * split_stride;
#pragma unroll
            for (int i = 0; i < NPER; ++i)
                pv[sp - 1][i] = (sp < splits && lane + 32 * i < E) ? prow[lane + 32 * i] : 0.f;
        }
#pragma unroll
        for (int sp = 1; sp < kGather; ++sp)
            if (sp < splits) {
#pragma unroll
                for (int i = 0; i < NPER; ++i) sv[i] += pv[sp - 1][i];
            }
    }
    for (int sp = kGather; sp < splits; ++sp) {
        const float *prow = lrow + sp * split_stride;
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) sv[i] += prow[lane + 32 * i];
    }
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        if (e < E) {
            const float sc = 1.0f / (1.0f + expf(-sv[i]));
            sv[i] = sc;
            cv[i] = sc + bias[e];
            if (scores) scores[static_cast<size_t>(t) * E + e] = sc;
        } else {
            sv[i] = 0.f;
            cv[i] = -INFINITY;
        }
    }
    float lb;   // the lane's best remaining choice and its expert id
    int le;
    auto rescan = [&]() {
        lb = -INFINITY;
        le = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (cv[i] > lb) { lb = cv[i]; le = lane + 32 * i; }
    };
    rescan();
    int my_idx = 0;
    float my_s = 0.f;
    for (int r = 0; r < k; ++r) {
        float best = lb;
        int best_e = le;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ob = __shfl_xor_sync(kFull, best, off);
            const int oe = __shfl_xor_sync(kFull, best_e, off);
            if (ob > best || (ob == best && oe < best_e)) { best = ob; best_e = oe; }
        }
        const int owner = best_e & 31;
        const int slot = best_e >> 5;
        float mine = 0.f;
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i < NPER; ++i)
                if (i == slot) { mine = sv[i]; cv[i] = -INFINITY; }
            rescan();
        }
        const float s_sel = __shfl_sync(kFull, mine, owner);
        if (lane == r) { my_idx = best_e; my_s = s_sel; }
    }
    float sum = (lane < k) ? my_s : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < k) {
        topk_idx[static_cast<size_t>(t) * k + lane] = my_idx;
        topk_w[static_cast<size_t>(t) * k + lane] = my_s / sum * route_scale;
    }
}

// ------------------------------------------------------------------ permutation
// Tokens are processed in chunks of 32 (one warp). For assignment (t, j) to
// expert e:
//   rank[t, j]   = number of tokens t' < t in t's chunk that also chose e
//   cnt[e][c]    = number of tokens of chunk c that chose e
// then cnt is scanned over chunks (per expert) and over experts, giving
//   position(t, j) = offsets[e] + sum_{c' < c} cnt[e][c'] + rank[t, j],
// the ascending-token order inside every expert segment.
constexpr int kPermWarps = 8;

// One warp per chunk: a shared-memory word per expert collects the chunk's
// lanes that chose it; ranks and counts are population counts of those words.
// Ids outside [0, E) are skipped (rank -1), so bad input cannot write out of bounds.
__global__ void perm_rank_kernel(const int32_t *__restrict__ idx, int T, int k, int E, int C,
                                 int32_t *__restrict__ rank, int32_t *__restrict__ cnt, unsigned int *err) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ uint32_t s_bits[];  // [kPermWarps][E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * kPermWarps + warp;
    if (c >= C) return;
    uint32_t *bits = s_bits + warp * E;
    for (int e = lane; e < E; e += 32) bits[e] = 0u;
    __syncwarp();
    const int t = c * 32 + lane;
    const int32_t *row = idx + static_cast<size_t>(t) * k;
    if (t < T) {
        for (int j = 0; j < k; ++j) {
            const int e = row[j];
            if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) atomicOr(&bits[e], 1u << lane);
            else if (kDebugBounds) record_error(err, ERR_BAD_INDEX);
        }
    }
    __syncwarp();
    if (t < T) {
        const uint32_t below = (1u << lane) - 1u;
        for (int j = 0; j < k; ++j) {
            const int e = row[j];
            rank[static_cast<size_t>(t) * k + j] =
                (static_cast<unsigned>(e) < static_cast<unsigned>(E)) ? __popc(bits[e] & below) : -1;
        }
    }
    for (int e = lane; e < E; e += 32) cnt[static_cast<size_t>(e) * C + c] = __popc(bits[e]);
}

// Exclusive scan of one expert's per-chunk counts (in place); total -> counts[e].
__global__ void perm_scan_kernel(int32_t *__restrict__ cnt, int C, int32_t *__restrict__ counts) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_warp[32];
    __shared__ int32_t s_carry;
    const int e = blockIdx.x;
    int32_t *row = cnt + static_cast<size_t>(e) * C;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) s_carry = 0;
    __syncthreads();
    for (int base = 0; base < C; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const int v = (i < C) ? row[i] : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) s_warp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < nw) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, w, off);
                if (lane >= off) w += o;
            }
            s_warp[lane] = w;  // inclusive scan of warp totals
        }
        __syncthreads();
        const int carry = s_carry;
        const int excl = carry + (warp > 0 ? s_warp[warp - 1] : 0) + incl - v;
        if (i < C) row[i] = excl;
        __syncthreads();
        if (threadIdx.x == 0) s_carry = carry + s_warp[nw - 1];
        __syncthreads();
    }
    if (threadIdx.x == 0) counts[e] = s_carry;
}

// Block-wide exclusive scan of up to blockDim.x * kItems values (single block).
template <int kItems>
__device__ void block_exclusive_scan(const int32_t *in, int n, int32_t *out, int32_t *total) {
    __shared__ int32_t s_warp[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int v[kItems];
    int local = 0;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const int idx = threadIdx.x * kItems + i;
        v[i] = (idx < n) ? in[idx] : 0;
        local += v[i];
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < nw) ? s_warp[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, w, off);
            if (lane >= off) w += o;
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    int run = (warp > 0 ? s_warp[warp - 1] : 0) + incl - local;
#pragma unroll
    for (int i = 0; i < kItems; ++i) {
        const int idx = threadIdx.x * kItems + i;
        if (idx < n) out[idx] = run;
        run += v[i];
    }
    if (total && threadIdx.x == 0) *total = s_warp[nw - 1];
    __syncthreads();
}

// Segment table of the grouped GEMMs from the routed offsets: groups 0..E-1
// are the routed experts' segments, groups E..E+S-1 the shared experts' T rows.
//   row_start[g]              first activation row of group g; row_start[E+S] = (k+S)*T
//   tile_prefix_a/b[g]        prefix sums of ceil(rows_g / tile_a) and ceil(rows_g / tile_b)
//   tile_prefix_a/b[G+1+g]    the same over the groups of two or more tiles only
// (the gate/up and the down GEMM may use different token-tile widths; each array
// holds 2 (G+1) entries), and the two GEMMs' dynamic scheduler counters are reset
// to zero. Called by a whole block of 1024 threads (E + S <= 1028).
__device__ void schedule_block(const int32_t *offsets, int E, int S, int T, int k, int tile_a, int tile_b,
                               int32_t *row_start, int32_t *tile_prefix_a, int32_t *tile_prefix_b,
                               int32_t *counters) {
    __shared__ int32_t s_rows[2048];
    const int G = E + S;
    const int kT = k * T;
    if (threadIdx.x < 2) counters[threadIdx.x] = 0;   // the two GEMMs' dynamic scheduler counters
    for (int g = threadIdx.x; g <= G; g += blockDim.x) row_start[g] = (g <= E) ? offsets[g] : kT + (g - E) * T;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int a = (g < E) ? offsets[g] : kT + (g - E) * T;
        const int b = (g < E) ? offsets[g + 1] : kT + (g - E + 1) * T;
        s_rows[g] = (b - a + tile_a - 1) / tile_a;
    }
    __syncthreads();
    block_exclusive_scan<2>(s_rows, G, tile_prefix_a, tile_prefix_a + G);
    for (int g = threadIdx.x; g < G; g += blockDim.x) s_rows[g] = (s_rows[g] >= 2) ? s_rows[g] : 0;
    __syncthreads();
    block_exclusive_scan<2>(s_rows, G, tile_prefix_a + G + 1, tile_prefix_a + 2 * G + 1);
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        const int a = (g < E) ? offsets[g] : kT + (g - E) * T;
        const int b = (g < E) ? offsets[g + 1] : kT + (g - E + 1) * T;
        s_rows[g] = (b - a + tile_b - 1) / tile_b;
    }
    __syncthreads();
    block_exclusive_scan<2>(s_rows, G, tile_prefix_b, tile_prefix_b + G);
    for (int g = threadIdx.x; g < G; g += blockDim.x) s_rows[g] = (s_rows[g] >= 2) ? s_rows[g] : 0;
    __syncthreads();
    block_exclusive_scan<2>(s_rows, G, tile_prefix_b + G + 1, tile_prefix_b + 2 * G + 1);
}

// offsets[0..E] from counts[0..E-1], then the GEMM schedules. Single block of 1024 threads.
__global__ void perm_offsets_kernel(const int32_t *__restrict__ counts, int E, int S, int T, int k, int tile_a,
                                    int tile_b, int32_t *__restrict__ offsets, int32_t *__restrict__ row_start,
                                    int32_t *__restrict__ tile_prefix_a, int32_t *__restrict__ tile_prefix_b,
                                    int32_t *__restrict__ counters) {
    pdl_trigger();
    pdl_wait();
    block_exclusive_scan<1>(counts, E, offsets, offsets + E);
    schedule_block(offsets, E, S, T, k, tile_a, tile_b, row_start, tile_prefix_a, tile_prefix_b, counters);
}

__global__ void sched_kernel(const int32_t *__restrict__ offsets, int E, int S, int T, int k, int tile_a, int tile_b,
                             int32_t *__restrict__ row_start, int32_t *__restrict__ tile_prefix_a,
                             int32_t *__restrict__ tile_prefix_b, int32_t *__restrict__ counters) {
    pdl_trigger();
    pdl_wait();
    schedule_block(offsets, E, S, T, k, tile_a, tile_b, row_start, tile_prefix_a, tile_prefix_b, counters);
}

// Token t's destinations, by the block's first k + S threads: assignment j < k
// goes to offsets[e] + cnt_scan[e][t / 32] + rank[t, j] (written to inv_pos, and t
// to sorted_tok there; an id outside [0, E) or a position outside [0, kT) gives -1
// and no write), shared expert s to row kT + sT + t. s_pos[j] holds them.
__device__ __forceinline__ void scatter_positions(const int32_t *__restrict__ idx, const int32_t *__restrict__ rank,
                                                  const int32_t *__restrict__ cnt_scan,
                                                  const int32_t *__restrict__ offsets, int t, int T, int k, int S,
                                                  int E, int C, int32_t *__restrict__ sorted_tok,
                                                  int32_t *__restrict__ inv_pos, int32_t *s_pos, unsigned int *err) {
    if (threadIdx.x < k) {
        const int j = threadIdx.x;
        const int e = idx[static_cast<size_t>(t) * k + j];
        int pos = -1;
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
            pos = offsets[e] + cnt_scan[static_cast<size_t>(e) * C + (t >> 5)] + rank[static_cast<size_t>(t) * k + j];
            if (pos < 0 || pos >= k * T) {
                if (kDebugBounds) record_error(err, ERR_BAD_INDEX);
                pos = -1;
            }
        }
        s_pos[j] = pos;
        inv_pos[static_cast<size_t>(t) * k + j] = pos;
        if (pos >= 0) sorted_tok[pos] = t;
    } else if (threadIdx.x < k + S) {
        s_pos[threadIdx.x] = k * T + (threadIdx.x - k) * T + t;
    }
}

// One block per token: writes sorted_tok / inv_pos and, when copy_rows, copies the
// token's quantised row and scales to its k routed positions and its S shared rows
// (a caller whose GEMM gathers the rows by sorted_tok skips the copy).
// sx is row-major [T, d/128]; sx_perm is K-block-major [d/128, R].
__global__ void perm_scatter_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ rank,
                                    const int32_t *__restrict__ cnt_scan, const int32_t *__restrict__ offsets,
                                    const uint8_t *__restrict__ xq, const float *__restrict__ sx, int T, int k,
                                    int S, int E, int d, int C, int32_t *__restrict__ sorted_tok,
                                    int32_t *__restrict__ inv_pos, uint8_t *__restrict__ xq_perm,
                                    float *__restrict__ sx_perm, unsigned int *err, int copy_rows) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_pos[40];
    const int t = blockIdx.x;
    const int64_t R = static_cast<int64_t>(k + S) * T;
    const int ndst = k + S;
    scatter_positions(idx, rank, cnt_scan, offsets, t, T, k, S, E, C, sorted_tok, inv_pos, s_pos, err);
    if (!copy_rows) return;   // uniform over the block
    __syncthreads();
    const uint4 *src = reinterpret_cast<const uint4 *>(xq + static_cast<size_t>(t) * d);
    const int nvec = d / 16;
    for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
        const uint4 val = src[v];
        for (int j = 0; j < ndst; ++j)
            if (s_pos[j] >= 0) reinterpret_cast<uint4 *>(xq_perm + static_cast<size_t>(s_pos[j]) * d)[v] = val;
    }
    const int gpr = d / 128;
    for (int g = threadIdx.x; g < gpr; g += blockDim.x) {
        const float sc = sx[static_cast<size_t>(t) * gpr + g];
        for (int j = 0; j < ndst; ++j)
            if (s_pos[j] >= 0) sx_perm[static_cast<size_t>(g) * R + s_pos[j]] = sc;
    }
}

// perm_scatter_kernel with the 1x128 quantisation of the bf16 row on the way, in
// quant_1x128_kernel's arithmetic: one block per token; thread i holds the 8-element
// units u = i + blockDim * n of the row (elements 8u..8u+7), kScatterUnits of them
// loaded together. A 128-wide group is 16
// consecutive units, held by a half-warp (blockDim a multiple of 32, d a multiple
// of 128). Codes and scale go to the token's k routed positions and S shared rows
// when copy_rows, and to the unpermuted xq_out [T, d] / sx_out [T, d/128]
// (row-major) when xq_out is given.
constexpr int kScatterUnits = 4;

__global__ void perm_quant_scatter_kernel(const int32_t *__restrict__ idx, const int32_t *__restrict__ rank,
                                          const int32_t *__restrict__ cnt_scan, const int32_t *__restrict__ offsets,
                                          const __nv_bfloat16 *__restrict__ x, int T, int k, int S, int E, int d,
                                          int C, int32_t *__restrict__ sorted_tok, int32_t *__restrict__ inv_pos,
                                          uint8_t *__restrict__ xq_perm, float *__restrict__ sx_perm, int copy_rows,
                                          uint8_t *__restrict__ xq_out, float *__restrict__ sx_out,
                                          unsigned int *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_pos[40];
    const int t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const unsigned half_mask = 0xffffu << (lane & 16);
    const int64_t R = static_cast<int64_t>(k + S) * T;
    const int ndst = copy_rows ? k + S : 0;
    const int nunits = d / 8;
    const int gpr = d / 128;
    const int nthr = static_cast<int>(blockDim.x);
    const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(t) * d);
    uint4 raw[kScatterUnits];
    auto load_batch = [&](int base) {
#pragma unroll
        for (int i = 0; i < kScatterUnits; ++i) {
            const int u = base + static_cast<int>(threadIdx.x) + i * nthr;
            raw[i] = u < nunits ? xr[u] : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    scatter_positions(idx, rank, cnt_scan, offsets, t, T, k, S, E, C, sorted_tok, inv_pos, s_pos, err);
    __syncthreads();
    for (int base = 0; base < nunits; base += kScatterUnits * nthr) {
        load_batch(base);
#pragma unroll
        for (int i = 0; i < kScatterUnits; ++i) {
            const int u = base + static_cast<int>(threadIdx.x) + i * nthr;
            if (u >= nunits) continue;   // whole half-warps: nunits and nthr are multiples of 16
            float v[8];
            unpack_bf16x8(raw[i], v);
            unsigned m = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) m = max(m, __float_as_uint(fabsf(v[q])));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(half_mask, m, off, 16));
            const float amax = __uint_as_float(m);
            const float sc = amax / 448.0f;
            uint2 codes = make_uint2(0u, 0u);
            if (amax != 0.f) {
                float d8[8];
                div_by_scale(v, sc, d8);
                codes.x = static_cast<uint32_t>(e4m3x2(d8[0], d8[1])) | (static_cast<uint32_t>(e4m3x2(d8[2], d8[3])) << 16);
                codes.y = static_cast<uint32_t>(e4m3x2(d8[4], d8[5])) | (static_cast<uint32_t>(e4m3x2(d8[6], d8[7])) << 16);
            }
            for (int j = 0; j < ndst; ++j)
                if (s_pos[j] >= 0) reinterpret_cast<uint2 *>(xq_perm + static_cast<size_t>(s_pos[j]) * d)[u] = codes;
            if (xq_out) reinterpret_cast<uint2 *>(xq_out + static_cast<size_t>(t) * d)[u] = codes;
            if ((lane & 15) == 0) {
                const int g = u >> 4;
                for (int j = 0; j < ndst; ++j)
                    if (s_pos[j] >= 0) sx_perm[static_cast<size_t>(g) * R + s_pos[j]] = sc;
                if (sx_out) sx_out[static_cast<size_t>(t) * gpr + g] = sc;
            }
        }
    }
}

// ------------------------------------------------------------------ combine
// y[t] = sum_s o[kT + sT + t] + sum_j w[t, j] * o[inv_pos[t, j]] (fp32, fixed order) -> bf16.
// Block (t, slice): blockDim.x threads, each owning 8 consecutive features of
// the slice [slice * 8 * blockDim.x, ...) of token t.
__global__ void combine_kernel(const __nv_bfloat16 *__restrict__ o, const float *__restrict__ w,
                               const int32_t *__restrict__ inv_pos, int T, int k, int S, int d,
                               __nv_bfloat16 *__restrict__ y, unsigned int *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_pos[32];
    __shared__ float s_w[32];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        int p = inv_pos[static_cast<size_t>(t) * k + threadIdx.x];
        if (kDebugBounds && (p < -1 || p >= k * T)) {   // a routed row is one of the k*T
            record_error(err, ERR_BAD_INDEX);
            p = -1;
        }
        s_pos[threadIdx.x] = p;
        s_w[threadIdx.x] = w[static_cast<size_t>(t) * k + threadIdx.x];
    }
    __syncthreads();
    const int v = blockIdx.y * blockDim.x + threadIdx.x;   // 8-feature unit of token t
    if (v >= d / 8) return;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    // the routed slots' rows are loaded a batch at a time before any of them is
    // added, so their loads are in flight together; the sums keep the fixed order
    // (shared experts, then slots j = 0, 1, ...)
    constexpr int kBatch = 8;
    uint4 raw[kBatch];
    auto load_batch = [&](int j0) {
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
            const int j = j0 + jj;
            raw[jj] = make_uint4(0u, 0u, 0u, 0u);
            if (j < k && s_pos[j] >= 0) raw[jj] = reinterpret_cast<const uint4 *>(o + static_cast<size_t>(s_pos[j]) * d)[v];
        }
    };
    load_batch(0);
    for (int s = 0; s < S; ++s) {
        const uint4 rs = reinterpret_cast<const uint4 *>(o + (static_cast<size_t>(k) * T + static_cast<size_t>(s) * T + t) * d)[v];
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&rs);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i] += __low2float(h[i]);
            acc[2 * i + 1] += __high2float(h[i]);
        }
    }
    for (int j0 = 0; j0 < k; j0 += kBatch) {
        if (j0 > 0) load_batch(j0);
#pragma unroll
        for (int jj = 0; jj < kBatch; ++jj) {
            const int j = j0 + jj;
            if (j >= k || s_pos[j] < 0) continue;
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw[jj]);
            const float wj = s_w[j];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[2 * i] = fmaf(wj, __low2float(h[i]), acc[2 * i]);
                acc[2 * i + 1] = fmaf(wj, __high2float(h[i]), acc[2 * i + 1]);
            }
        }
    }
    uint4 out;
    __nv_bfloat162 *oh = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) oh[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    reinterpret_cast<uint4 *>(y + static_cast<size_t>(t) * d)[v] = out;
}

// ------------------------------------------------------------------ weight tiling
// w [groups][rows][cols] -> w_tiled [groups][rows/128][cols/128][128][128]:
// w_tiled[g][rb][cb][r][c] = w[g][rb*128 + r][cb*128 + c]. Grid-stride over the
// 16-byte units of the output (8 per tile row), read from the input row.
__global__ void pack_tiles_kernel(const uint8_t *__restrict__ w, int64_t groups, int rows, int cols,
                                  uint8_t *__restrict__ w_tiled) {
    pdl_trigger();
    pdl_wait();
    const int rbs = rows / 128, cbs = cols / 128;
    const int64_t units = groups * rbs * cbs * 128 * 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < units; u += stride) {
        const int c16 = static_cast<int>(u & 7);
        const int r = static_cast<int>((u >> 3) & 127);
        const int64_t tile = u >> 10;   // [g][rb][cb]
        const int cb = static_cast<int>(tile % cbs);
        const int64_t grb = tile / cbs;  // g * rbs + rb
        const int rb = static_cast<int>(grb % rbs);
        const int64_t g = grb / rbs;
        const uint8_t *src = w + (g * rows + static_cast<int64_t>(rb) * 128 + r) * cols + static_cast<int64_t>(cb) * 128 + c16 * 16;
        reinterpret_cast<uint4 *>(w_tiled)[u] = *reinterpret_cast<const uint4 *>(src);
    }
}

// ------------------------------------------------------------------ bounded-wait self-test
// One CTA of two warps whose lane 0s wait on an mbarrier that nothing arrives at,
// through the GEMMs' own bounded wait: warp 0 with the given limit, warp 1 with the
// kernels' usual limit. Warp 0 gives up, raises the CTA's abort word and records
// ERR_WAIT_SELFTEST; warp 1 sees the abort word and returns without recording.
// No trap, no fault: the context stays usable.
__global__ void wait_selftest_kernel(unsigned int *err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_word;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_word = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        mbar_wait_for(smem_u32(&bar), 0, smem_u32(&abort_word), err, ERR_WAIT_SELFTEST,
                      warp == 0 ? limit_ns : kWaitLimitNs);
    __syncthreads();
}

// ------------------------------------------------------------------ block pieces
// Sum of one float per thread over the CTA (blockDim a multiple of 32), in a fixed
// order: lanes by xor butterfly, then the warps' sums by warp 0. Every thread gets
// the total.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = (lane < static_cast<int>(blockDim.x >> 5)) ? red[lane] : 0.f;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(kFull, t, off);
        if (lane == 0) red[32] = t;
    }
    __syncthreads();
    return red[32];
}

// 1 / sqrt(mean of squares + eps), with IEEE square root and division.
__device__ __forceinline__ float rms_inverse(float sum_sq, int n, float eps) {
    return 1.0f / sqrtf(sum_sq / static_cast<float>(n) + eps);
}


__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
    uint4 out;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return out;
}

// Units (8 bf16 each) of a row that a thread of the one-row-per-CTA kernels loads
// up front and keeps in registers between their two passes; longer rows loop and
// re-read.
constexpr int kRowUnits = 4;

// RMSNorm of one bf16 row per CTA, y = bf16(h * inv * gamma) with
// inv = 1 / sqrt(mean(h^2) + eps), followed by the 1x128 quantisation of the bf16
// y values with the arithmetic of quant_1x128_kernel. Thread t holds units
// t + i * blockDim (i < kRowUnits): pass 1 sums h^2 in fp32 in that fixed order;
// pass 2 normalises, and each 128-wide group is 16 consecutive units held by a
// half-warp (blockDim a multiple of 32, cols a multiple of 128, so a half-warp is
// wholly inside or outside the row).
__global__ void __launch_bounds__(1024) rmsnorm_quant_kernel(const __nv_bfloat16 *__restrict__ h,
                                                             const __nv_bfloat16 *__restrict__ gamma, float eps,
                                                             int cols, __nv_bfloat16 *__restrict__ y,
                                                             uint8_t *__restrict__ q, float *__restrict__ s, int rows,
                                                             int s_transposed) {
    pdl_trigger();
    pdl_wait();
    __shared__ float red[33];
    const int r = blockIdx.x;
    const int lane = threadIdx.x & 31;
    const int nunits = cols / 8;
    const int nthr = static_cast<int>(blockDim.x);
    const bool cached = nunits <= kRowUnits * nthr;
    const uint4 *hr = reinterpret_cast<const uint4 *>(h + static_cast<size_t>(r) * cols);
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
    uint4 row[kRowUnits];
    float ss = 0.f;
    auto accumulate = [&](const uint4 &raw) {
        float v[8];
        unpack_bf16x8(raw, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    };
    if (cached) {
#pragma unroll
        for (int i = 0; i < kRowUnits; ++i) {
            const int u = threadIdx.x + i * nthr;
            if (u < nunits) row[i] = hr[u];
        }
#pragma unroll
        for (int i = 0; i < kRowUnits; ++i)
            if (threadIdx.x + i * nthr < nunits) accumulate(row[i]);
    } else {
        for (int u = threadIdx.x; u < nunits; u += nthr) accumulate(hr[u]);
    }
    const float inv = rms_inverse(block_sum(ss, red), cols, eps);
    const unsigned half_mask = 0xffffu << (lane & 16);
    auto emit = [&](int u, const uint4 &raw) {
        float v[8], g[8];
        unpack_bf16x8(raw, v);
        unpack_bf16x8(gr[u], g);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = v[i] * inv * g[i];
        const uint4 packed = pack_bf16x8(v);
        if (y) reinterpret_cast<uint4 *>(y + static_cast<size_t>(r) * cols)[u] = packed;
        unpack_bf16x8(packed, v);   // the bf16 values are what gets quantised
        unsigned m = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = max(m, __float_as_uint(fabsf(v[i])));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(half_mask, m, off, 16));
        const float amax = __uint_as_float(m);
        const float sc = amax / 448.0f;
        uint2 codes = make_uint2(0u, 0u);
        if (amax != 0.f) {
            float d8[8];
            div_by_scale(v, sc, d8);
            codes.x = static_cast<uint32_t>(e4m3x2(d8[0], d8[1])) | (static_cast<uint32_t>(e4m3x2(d8[2], d8[3])) << 16);
            codes.y = static_cast<uint32_t>(e4m3x2(d8[4], d8[5])) | (static_cast<uint32_t>(e4m3x2(d8[6], d8[7])) << 16);
        }
        reinterpret_cast<uint2 *>(q + static_cast<size_t>(r) * cols)[u] = codes;
        if ((lane & 15) == 0) {
            const int g128 = u >> 4;
            s[s_transposed ? (static_cast<size_t>(g128) * rows + r) : (static_cast<size_t>(r) * (cols / 128) + g128)] = sc;
        }
    };
    if (cached) {
#pragma unroll
        for (int i = 0; i < kRowUnits; ++i) {
            const int u = threadIdx.x + i * nthr;
            if (u < nunits) emit(u, row[i]);
        }
    } else {
        for (int u = threadIdx.x; u < nunits; u += nthr) emit(u, hr[u]);
    }
}

// The combine of combine_kernel (same summation order, rounded to bf16 as the FFN
// output), plus the block's residual addition h = bf16(residual + y), and, when
// gamma is given, the next block's input RMSNorm x = bf16(h * inv * gamma) of that
// bf16 row. One CTA per token; thread t holds units t + i * blockDim as above.
// kBatch: load a token's routed rows eight slots at a time (more loads in flight
// per thread, for batches too small to fill the GPU with CTAs); it needs rows of
// at most 256 threads (d <= 8192), for the register room (up to 128 a thread).
// Without it the launch bound is 1024 threads and 64 registers, for the occupancy
// that large batches want, and the rows are loaded four slots at a time.
template <bool kBatch>
__global__ void __launch_bounds__(kBatch ? 256 : 1024, kBatch ? 2 : 1) combine_residual_rmsnorm_kernel(
    const __nv_bfloat16 *__restrict__ o, const float *__restrict__ w, const int32_t *__restrict__ inv_pos, int T,
    int k, int S, int d, const __nv_bfloat16 *__restrict__ residual, const __nv_bfloat16 *__restrict__ gamma,
    float eps, __nv_bfloat16 *__restrict__ h_out, __nv_bfloat16 *__restrict__ x_next, unsigned int *err) {
    pdl_trigger();
    pdl_wait();
    __shared__ int32_t s_pos[32];
    __shared__ float s_w[32];
    __shared__ float red[33];
    const int t = blockIdx.x;
    if (threadIdx.x < k) {
        int p = inv_pos[static_cast<size_t>(t) * k + threadIdx.x];
        if (kDebugBounds && (p < -1 || p >= k * T)) {   // a routed row is one of the k*T
            record_error(err, ERR_BAD_INDEX);
            p = -1;
        }
        s_pos[threadIdx.x] = p;
        s_w[threadIdx.x] = w[static_cast<size_t>(t) * k + threadIdx.x];
    }
    __syncthreads();
    const int nunits = d / 8;
    const int nthr = static_cast<int>(blockDim.x);
    const bool cached = nunits <= kRowUnits * nthr;
    const uint4 *rr = reinterpret_cast<const uint4 *>(residual + static_cast<size_t>(t) * d);
    uint4 *hr = reinterpret_cast<uint4 *>(h_out + static_cast<size_t>(t) * d);
    uint4 row[kRowUnits];
    float ss = 0.f;
    auto make_h = [&](int v) -> uint4 {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
        for (int sh = 0; sh < S; ++sh) {
            float e[8];
            unpack_bf16x8(reinterpret_cast<const uint4 *>(o + (static_cast<size_t>(k) * T + static_cast<size_t>(sh) * T + t) * d)[v], e);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += e[i];
        }
        if constexpr (kBatch) {
            // the rows of eight slots are loaded before they are added; the order of
            // the sums is that of combine_kernel
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 raw[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    raw[jj] = make_uint4(0u, 0u, 0u, 0u);
                    if (j < k && s_pos[j] >= 0)
                        raw[jj] = reinterpret_cast<const uint4 *>(o + static_cast<size_t>(s_pos[j]) * d)[v];
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int j = j0 + jj;
                    if (j >= k || s_pos[j] < 0) continue;
                    float e[8];
                    unpack_bf16x8(raw[jj], e);
                    const float wj = s_w[j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, e[i], acc[i]);
                }
            }
        } else {
            // four slots at a time within the 64-register budget of this variant
            for (int j0 = 0; j0 < k; j0 += 4) {
                uint4 raw[4];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = j0 + jj;
                    raw[jj] = make_uint4(0u, 0u, 0u, 0u);
                    if (j < k && s_pos[j] >= 0)
                        raw[jj] = reinterpret_cast<const uint4 *>(o + static_cast<size_t>(s_pos[j]) * d)[v];
                }
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = j0 + jj;
                    if (j >= k || s_pos[j] < 0) continue;
                    float e[8];
                    unpack_bf16x8(raw[jj], e);
                    const float wj = s_w[j];
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, e[i], acc[i]);
                }
            }
        }
        float yb[8], res[8];
        unpack_bf16x8(pack_bf16x8(acc), yb);   // the FFN output is a bf16 tensor
        unpack_bf16x8(rr[v], res);
#pragma unroll
        for (int i = 0; i < 8; ++i) yb[i] = res[i] + yb[i];
        const uint4 hp = pack_bf16x8(yb);
        hr[v] = hp;
        if (gamma) {
            unpack_bf16x8(hp, yb);
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(yb[i], yb[i], ss);
        }
        return hp;
    };
    if (cached) {
#pragma unroll
        for (int i = 0; i < kRowUnits; ++i) {
            const int v = threadIdx.x + i * nthr;
            if (v < nunits) row[i] = make_h(v);
        }
    } else {
        for (int v = threadIdx.x; v < nunits; v += nthr) make_h(v);
    }
    if (!gamma) return;   // uniform over the CTA
    const float inv = rms_inverse(block_sum(ss, red), d, eps);
    const uint4 *gr = reinterpret_cast<const uint4 *>(gamma);
    auto emit = [&](int v, const uint4 &hp) {
        float hv[8], g[8];
        unpack_bf16x8(hp, hv);
        unpack_bf16x8(gr[v], g);
#pragma unroll
        for (int i = 0; i < 8; ++i) hv[i] = hv[i] * inv * g[i];
        reinterpret_cast<uint4 *>(x_next + static_cast<size_t>(t) * d)[v] = pack_bf16x8(hv);
    };
    if (cached) {
#pragma unroll
        for (int i = 0; i < kRowUnits; ++i) {
            const int v = threadIdx.x + i * nthr;
            if (v < nunits) emit(v, row[i]);
        }
    } else {
        for (int v = threadIdx.x; v < nunits; v += nthr) emit(v, hr[v]);
    }
}

}  // namespace moe
