// fused_fma.cuh -- the fused decode MoE layer on CUDA cores (dequant-GEMV).
//
// One persistent cooperative launch computes the whole layer ("Daily AI
// Hotspot 2026-08-21", section "Most Worth Your Attention Today": shared
// gate/up, routed experts, shared down and the residual add in one pass,
// FP32 accumulation, the BF16 output written once), over the deduplicated
// groups of the step (PR #27 "each expert once", "Motivation" and
// "Modifications"): every group's weights stream from HBM once, and all the
// rows that use the group are its columns.
//
// Phases, separated by grid barriers:
//   A  gate/up + SwiGLU: one warp per (group, intermediate row i): the gate
//      row i and up row i of the group's expert are dotted with every column's
//      activation row; mid[c][i] = silu(gate) * up (fp32, workspace).
//   B  down: one warp per (group, hidden row h): y[c][h] = Wd[h] . mid[c].
//   C  combine: out[t][h] = bf16(x + y[shared] + sum_p w[t,p] y[pick p]) in
//      that order.
// The arithmetic of a column does not depend on which group it sits in or
// on its position in the group, so the dedup and one-row forms agree bit for
// bit. Dequantisation is exact (E2M1 and E4M3 values are exact in fp32); the
// NVFP4 block scale multiplies each 16-element partial sum, the FP8 block
// scale each 16-element partial sum, the NVFP4 tensor scale the row total.
#pragma once

#include "group_table.cuh"
#include "moe_common.cuh"
#include "router.cuh"
#include "sm100.cuh"

namespace moe {

struct FusedParams {
    const __nv_bfloat16 *x;
    const int32_t *ids;
    const float *topk_w;
    WeightsDev routed, shared;
    __nv_bfloat16 *out;
    int T, H, I, Is, E, K;
    unsigned flags;
    WsHeader *hdr;
    float *mid;  // [Ucap][Imax]
    float *y;    // [Ucap][H]
    int Imax;
    int route_mode;  // 1: the picks and weights come from the router below, not ids/topk_w
    RouterDev router;
};

constexpr int kFmaThreads = 256;
constexpr int kFmaNcb = 4;  // columns per pass over a weight row

// ---- activation loaders: EPC consecutive elements of one column as fp32 ----

template <int EPC>
__device__ __forceinline__ void load_act(const __nv_bfloat16 *row, int k0, float (&a)[EPC]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(row + k0);
#pragma unroll
    for (int v = 0; v < EPC / 8; ++v) {
        const uint4 q = __ldg(src + v);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            a[v * 8 + 2 * k] = bf16_bits_to_float(w[k] & 0xffffu);
            a[v * 8 + 2 * k + 1] = bf16_bits_to_float(w[k] >> 16);
        }
    }
}

template <int EPC>
__device__ __forceinline__ void load_act(const float *row, int k0, float (&a)[EPC]) {
    const float4 *src = reinterpret_cast<const float4 *>(row + k0);
#pragma unroll
    for (int v = 0; v < EPC / 4; ++v) {
        const float4 q = __ldcg(src + v);
        a[4 * v] = q.x;
        a[4 * v + 1] = q.y;
        a[4 * v + 2] = q.z;
        a[4 * v + 3] = q.w;
    }
}

template <int N>
__device__ __forceinline__ float dot_seq(const float *w, const float *a) {
    float p = __fmul_rn(w[0], a[0]);
#pragma unroll
    for (int k = 1; k < N; ++k) p = __fmaf_rn(w[k], a[k], p);
    return p;
}

// ---- one weight row dotted with up to kFmaNcb activation columns -----------
// Lane l takes the row's 16-byte chunks l, l+32, ...; returns per-lane partial
// sums (not yet reduced across the warp, tensor scale not yet applied).

template <int FMT>
struct FmtTraits;
template <>
struct FmtTraits<kFmtNvfp4> {
    static constexpr int kEpc = 32;
};
template <>
struct FmtTraits<kFmtFp8B128> {
    static constexpr int kEpc = 16;
};
template <>
struct FmtTraits<kFmtBf16> {
    static constexpr int kEpc = 8;
};

// q: the row's element bytes; sc: NVFP4 -> the row's E4M3 block scales;
// FP8 -> the fp32 scales of the row's 128-row block (one per 128 columns).
template <int FMT, typename ACT>
__device__ __forceinline__ void row_dot(const uint8_t *__restrict__ q, const void *__restrict__ sc,
                                        int L, const ACT *const (&act)[kFmaNcb], int nc,
                                        float (&acc)[kFmaNcb]) {
    constexpr int EPC = FmtTraits<FMT>::kEpc;
    const int lane = threadIdx.x & 31;
    const int nchunks = L / EPC;
#pragma unroll
    for (int c = 0; c < kFmaNcb; ++c) acc[c] = 0.0f;
    for (int j = lane; j < nchunks; j += 32) {
        const uint4 raw = ld_stream_v4(q + (size_t)j * 16);
        const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
        float w[EPC];
        float s0 = 1.0f, s1 = 1.0f;
        if constexpr (FMT == kFmtNvfp4) {
#pragma unroll
            for (int b = 0; b < 16; ++b) {
                const __half2 h = e2m1x2_to_half2((wd[b >> 2] >> (8 * (b & 3))) & 0xffu);
                w[2 * b] = __low2float(h);
                w[2 * b + 1] = __high2float(h);
            }
            const uint32_t sb = *reinterpret_cast<const uint16_t *>(
                static_cast<const uint8_t *>(sc) + (size_t)j * 2);
            const __half2 hs = e4m3x2_to_half2(sb);
            s0 = __low2float(hs);
            s1 = __high2float(hs);
        } else if constexpr (FMT == kFmtFp8B128) {
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                const __half2 h = e4m3x2_to_half2((wd[b >> 1] >> (16 * (b & 1))) & 0xffffu);
                w[2 * b] = __low2float(h);
                w[2 * b + 1] = __high2float(h);
            }
            s0 = static_cast<const float *>(sc)[(j * EPC) / 128];
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                w[2 * b] = bf16_bits_to_float(wd[b] & 0xffffu);
                w[2 * b + 1] = bf16_bits_to_float(wd[b] >> 16);
            }
        }
#pragma unroll
        for (int c = 0; c < kFmaNcb; ++c) {
            if (c < nc) {
                float a[EPC];
                load_act<EPC>(act[c], j * EPC, a);
                if constexpr (FMT == kFmtNvfp4) {
                    const float p0 = dot_seq<16>(w, a);
                    const float p1 = dot_seq<16>(w + 16, a + 16);
                    acc[c] = __fmaf_rn(p0, s0, acc[c]);
                    acc[c] = __fmaf_rn(p1, s1, acc[c]);
                } else if constexpr (FMT == kFmtFp8B128) {
                    acc[c] = __fmaf_rn(dot_seq<16>(w, a), s0, acc[c]);
                } else {
                    acc[c] = __fadd_rn(acc[c], dot_seq<8>(w, a));
                }
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Locate weight row `r` of matrix `mat` (0 = w13 [2Ig][Lin], 1 = w2 [H][Ig]) of
// expert e and dot it with the columns. Returns warp-reduced, fully scaled dots.
template <typename ACT>
__device__ __forceinline__ void weight_row_dots(const WeightsDev &w, int mat, int e, int rows,
                                                int L, int r, const ACT *const (&act)[kFmaNcb],
                                                int nc, float (&out)[kFmaNcb]) {
    const size_t ri = (size_t)e * rows + r;
    const uint8_t *q = mat ? w.w2 : w.w13;
    const uint8_t *sc = mat ? w.w2_scale : w.w13_scale;
    float acc[kFmaNcb];
    float gs = 1.0f;
    switch (w.fmt) {
        case kFmtNvfp4:
            row_dot<kFmtNvfp4>(q + ri * (L / 2), sc + ri * (L / 16), L, act, nc, acc);
            gs = (mat ? w.w2_gscale : w.w13_gscale)[e];
            break;
        case kFmtFp8B128: {
            const float *s = reinterpret_cast<const float *>(sc) +
                             ((size_t)e * (rows / 128) + r / 128) * (L / 128);
            row_dot<kFmtFp8B128>(q + ri * L, s, L, act, nc, acc);
            break;
        }
        default:
            row_dot<kFmtBf16>(q + ri * L * 2, nullptr, L, act, nc, acc);
            break;
    }
#pragma unroll
    for (int c = 0; c < kFmaNcb; ++c) {
        out[c] = warp_sum(acc[c]);
        if (w.fmt == kFmtNvfp4) out[c] = __fmul_rn(out[c], gs);
    }
}

__global__ void __launch_bounds__(kFmaThreads) fused_fma_kernel(FusedParams p) {
    extern __shared__ int4 smem_i4[];
    int32_t *tbl = reinterpret_cast<int32_t *>(smem_i4);
    const int T = p.T, K = p.K, H = p.H;
    const bool no_dedup = (p.flags & kFlagNoDedup) != 0;
    GroupTable tab{tbl, T * (K + 1), T * (K + 1)};
    int *scr = tbl + group_table_ints(T, K);
    float *tw_s = reinterpret_cast<float *>(scr + group_table_scratch_ints(T, K, p.E));  // [T][K] routed weights
    const int lane = threadIdx.x & 31;
    const int nwarps_cta = blockDim.x >> 5;
    const int gw = blockIdx.x * nwarps_cta + (threadIdx.x >> 5);
    const int nw = gridDim.x * nwarps_cta;
    sm100::griddep_wait();  // a chained launch: the previous grid's writes first

    // ---- phase R (routed launches): partial logits over every warp of the
    // grid, then each CTA picks every row's experts on chip ----------------
    if (p.route_mode) {
        router_logits(p.router, p.x, T, H, p.E, gw, nw);
        if (!grid_barrier(p.hdr, gridDim.x, false)) return;
        router_picks(p.router, T, p.E, K, threadIdx.x >> 5, nwarps_cta, group_table_picks(scr, p.E), tw_s, K,
                     blockIdx.x == 0);
    }
    group_table_cta(p.route_mode ? nullptr : p.ids, T, K, p.E, no_dedup, tab, scr,
                    blockIdx.x == 0 ? &p.hdr->err : nullptr, 0, blockDim.x, 0);
    const float *topk_w = p.route_mode ? tw_s : p.topk_w;
    sm100::griddep_launch_dependents();

    const int G = tab.G();
    const int32_t *gexp = tab.gexp(), *gn = tab.gncols(), *g0 = tab.gcol0(),
                  *crow = tab.col_row(), *rcol = tab.row_col();
    const int n_shared_groups = no_dedup ? T : (T > 0 ? 1 : 0);

    // ---- phase A: gate/up + SwiGLU --------------------------------------
    {
        const int NA = n_shared_groups * p.Is + (G - n_shared_groups) * p.I;
        int g = 0, gstart = 0;
        for (int task = gw; task < NA; task += nw) {
            int rows_g = gexp[g] < 0 ? p.Is : p.I;
            while (task >= gstart + rows_g) {
                gstart += rows_g;
                ++g;
                rows_g = gexp[g] < 0 ? p.Is : p.I;
            }
            const int i = task - gstart;
            const bool sh = gexp[g] < 0;
            const WeightsDev &w = sh ? p.shared : p.routed;
            const int e = sh ? 0 : gexp[g];
            const int Ig = rows_g;
            for (int cb = 0; cb < gn[g]; cb += kFmaNcb) {
                const int nc = min(kFmaNcb, gn[g] - cb);
                const __nv_bfloat16 *act[kFmaNcb];
#pragma unroll
                for (int c = 0; c < kFmaNcb; ++c)
                    act[c] = p.x + (size_t)crow[g0[g] + cb + (c < nc ? c : 0)] * H;
                float gate[kFmaNcb], up[kFmaNcb];
                weight_row_dots(w, 0, e, 2 * Ig, H, i, act, nc, gate);
                weight_row_dots(w, 0, e, 2 * Ig, H, Ig + i, act, nc, up);
#pragma unroll
                for (int c = 0; c < kFmaNcb; ++c)
                    if (c < nc && lane == c)
                        p.mid[(size_t)(g0[g] + cb + c) * p.Imax + i] = silu_f32(gate[c]) * up[c];
            }
        }
    }
    const bool drop = (p.flags & kFlagDebugDropArrive) && blockIdx.x == 0;
    if (!grid_barrier(p.hdr, gridDim.x, drop)) return;

    // ---- phase B: down ----------------------------------------------------
    {
        const int NB = G * H;
        for (int task = gw; task < NB; task += nw) {
            const int g = task / H, h = task - g * H;
            const bool sh = gexp[g] < 0;
            const WeightsDev &w = sh ? p.shared : p.routed;
            const int e = sh ? 0 : gexp[g];
            const int Ig = sh ? p.Is : p.I;
            for (int cb = 0; cb < gn[g]; cb += kFmaNcb) {
                const int nc = min(kFmaNcb, gn[g] - cb);
                const float *act[kFmaNcb];
#pragma unroll
                for (int c = 0; c < kFmaNcb; ++c)
                    act[c] = p.mid + (size_t)(g0[g] + cb + (c < nc ? c : 0)) * p.Imax;
                float yv[kFmaNcb];
                weight_row_dots(w, 1, e, H, Ig, h, act, nc, yv);
#pragma unroll
                for (int c = 0; c < kFmaNcb; ++c)
                    if (c < nc && lane == c) p.y[(size_t)(g0[g] + cb + c) * H + h] = yv[c];
            }
        }
    }
    if (!grid_barrier(p.hdr, gridDim.x, false)) return;

    // ---- phase C: combine, one bf16 write per output element -------------
    {
        const size_t n = (size_t)T * H;
        for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n;
             idx += (size_t)gridDim.x * blockDim.x) {
            const int t = (int)(idx / H), h = (int)(idx - (size_t)t * H);
            const int32_t *rc = rcol + t * (K + 1);
            float acc = __bfloat162float(p.x[idx]);
            acc = __fadd_rn(acc, __ldcg(p.y + (size_t)rc[0] * H + h));
            for (int q = 0; q < K; ++q) {
                const int c = rc[1 + q];
                if (c >= 0) acc = __fmaf_rn(topk_w[t * K + q], __ldcg(p.y + (size_t)c * H + h), acc);
            }
            p.out[idx] = __float2bfloat16_rn(acc);
        }
    }
}

// Standalone table kernel (one CTA), for moe_group_table.
__global__ void __launch_bounds__(256) group_table_kernel(const int32_t *ids, int T, int K, int E,
                                                          unsigned flags, int32_t *out,
                                                          uint32_t *err_word) {
    extern __shared__ int4 smem_i4[];
    int32_t *tbl = reinterpret_cast<int32_t *>(smem_i4);
    GroupTable tab{tbl, T * (K + 1), T * (K + 1)};
    int *scr = tbl + group_table_ints(T, K);
    group_table_cta(ids, T, K, E, (flags & kFlagNoDedup) != 0, tab, scr, err_word, 0, blockDim.x, 0);
    for (int i = threadIdx.x; i < group_table_ints(T, K); i += blockDim.x) out[i] = tbl[i];
}

}  // namespace moe
