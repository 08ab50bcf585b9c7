// router.cuh -- the routing front end: topk_ids and topk_w from the layer
// input, inside the fused launch.
//
// "Daily AI Hotspot 2026-08-21", section "Most Worth Your Attention Today"
// (the SGLang #32340 paragraph): the shared-expert fusion has to handle a bf16
// correction bias and a top-k whose K is not a power of two. PR #27 "each
// expert once", "Reviewer notes": every CTA routes all rows itself, so no
// cross-CTA hand-off of the routing decision is needed, and the tie order is
// the usual one. Scoring as in DeepSeek-V3: for row t and routed expert e
//   logit = x[t] . Wr[e]                     (bf16 inputs, fp32 sums)
//   s     = 1 / (1 + exp(-logit))            (sigmoid)
//   key   = s + bias[e]                      (bf16 bias, or 0)
//   picks = the K largest keys, largest first; equal keys: lower e first
//   w[p]  = scale * s[p] / sum_q s[q]        (renormalised; or scale * s[p])
//
// The router GEMM is shared out over the warps of the grid: each (t, e, part)
// is one warp's dot product over one of kRouterParts slices of H, written to
// the workspace, so every load a warp needs is in flight at once. Every CTA
// then waits for all partial logits and selects the picks of every row on
// chip (each logit the sum of its parts in part order).
#pragma once

#include "moe_common.cuh"

namespace moe {

constexpr int kRouterParts = 8;   // slices of H per logit
constexpr int kRouterMaxE = 1024;

struct RouterDev {
    const __nv_bfloat16 *wr;    // [E][H] router weights, H contiguous
    const __nv_bfloat16 *bias;  // [E] correction bias, or null
    float scale;                // routed scaling factor
    int renorm;                 // 1: weights renormalised over the picks
    float *part;                // workspace [T][E][kRouterParts] partial logits
    int32_t *ids_out;           // [T][K] or null: the picks, written by CTA 0
    float *w_out;               // [T][K] or null: the weights, written by CTA 0
};

// x[t] . Wr[e] over H slice `part` by one whole warp: lane l takes the
// 8-element chunks l, l+32, ... of the slice, each summed in order with fp32
// FMAs (the bf16 x bf16 products are exact in fp32), then a fixed butterfly
// over the lanes. Every lane returns the same value.
__device__ __forceinline__ float router_part_dot(const __nv_bfloat16 *__restrict__ xr,
                                                 const __nv_bfloat16 *__restrict__ wr, int H, int part) {
    const int lane = threadIdx.x & 31;
    const int nch = H / 8 / kRouterParts, c0 = part * nch;
    const uint4 *xq = reinterpret_cast<const uint4 *>(xr) + c0;
    const uint4 *wq = reinterpret_cast<const uint4 *>(wr) + c0;
    float acc = 0.0f;
#pragma unroll 4
    for (int c = lane; c < nch; c += 32) {
        const uint4 a = __ldg(xq + c), b = ld_stream_v4(wq + c);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc = __fmaf_rn(bf16_bits_to_float(av[k] & 0xffffu), bf16_bits_to_float(bv[k] & 0xffffu), acc);
            acc = __fmaf_rn(bf16_bits_to_float(av[k] >> 16), bf16_bits_to_float(bv[k] >> 16), acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
    return acc;
}

// The partial logits of the (t, e, part) items dealt to this warp: item i =
// gw, gw + nw, ... (part fastest, then e, then t).
__device__ __forceinline__ void router_logits(const RouterDev &r, const __nv_bfloat16 *x, int T, int H,
                                              int E, int gw, int nw) {
    const int lane = threadIdx.x & 31;
    const int n = T * E * kRouterParts;
    for (int i = gw; i < n; i += nw) {
        const int te = i / kRouterParts, part = i - te * kRouterParts;
        const int t = te / E, e = te - t * E;
        const float v = router_part_dot(x + (size_t)t * H, r.wr + (size_t)e * H, H, part);
        if (lane == 0) r.part[i] = v;
    }
}

__device__ __forceinline__ float router_score(float logit) { return 1.0f / (1.0f + expf(-logit)); }

__device__ __forceinline__ float router_logit(const float *part) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(part));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(part) + 1);
    float v = a.x;
    v = __fadd_rn(v, a.y);
    v = __fadd_rn(v, a.z);
    v = __fadd_rn(v, a.w);
    v = __fadd_rn(v, b.x);
    v = __fadd_rn(v, b.y);
    v = __fadd_rn(v, b.z);
    return __fadd_rn(v, b.w);
}
static_assert(kRouterParts == 8, "router_logit sums eight parts");

// The K picks of row t by one whole warp. Lane l holds the keys of experts
// l, l+32, ... (NJ per lane, E <= 32*NJ); each of the K passes takes the
// largest remaining key (equal keys: the lower expert) with a fixed butterfly
// of (key, expert) comparisons. Lane p < K returns pick p and its weight.
template <int NJ>
__device__ __forceinline__ void router_topk_row_n(const RouterDev &r, int t, int E, int K, int &id_out,
                                                  float &w_out) {
    const int lane = threadIdx.x & 31;
    float key[NJ], sc[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
        const int e = lane + 32 * j;
        key[j] = -INFINITY;
        sc[j] = 0.0f;
        if (e < E) {
            sc[j] = router_score(router_logit(r.part + ((size_t)t * E + e) * kRouterParts));
            key[j] = r.bias ? __fadd_rn(sc[j], __bfloat162float(r.bias[e])) : sc[j];
        }
    }
    int pick = -1;
    float my_s = 0.0f, sum = 0.0f;
    for (int p = 0; p < K; ++p) {
        float bk = -INFINITY, bs = 0.0f;
        int be = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            const int e = lane + 32 * j;
            if (e < E && (key[j] > bk || (key[j] == bk && e < be))) {
                bk = key[j];
                be = e;
                bs = sc[j];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ok = __shfl_xor_sync(0xffffffffu, bk, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            if (ok > bk || (ok == bk && oe < be)) {
                bk = ok;
                be = oe;
                bs = os;
            }
        }
#pragma unroll
        for (int j = 0; j < NJ; ++j)
            if (lane + 32 * j == be) key[j] = -INFINITY;  // taken
        sum = __fadd_rn(sum, bs);
        if (lane == p) {
            pick = be;
            my_s = bs;
        }
    }
    id_out = pick;
    w_out = r.renorm ? __fmul_rn(r.scale, __fdiv_rn(my_s, sum)) : __fmul_rn(r.scale, my_s);
}

// Row t's picks by one whole warp: lane p < K gets pick p and its weight.
__device__ __forceinline__ void router_topk_row(const RouterDev &r, int t, int E, int K, int &id, float &w) {
    if (E <= 256) router_topk_row_n<8>(r, t, E, K, id, w);
    else if (E <= 512) router_topk_row_n<16>(r, t, E, K, id, w);
    else router_topk_row_n<32>(r, t, E, K, id, w);
}

// Every row's picks, rows dealt over `nwarps` warps of one CTA (this warp:
// wi): picks [T][K] and weights written with the given stride per row.
__device__ __forceinline__ void router_picks(const RouterDev &r, int T, int E, int K, int wi, int nwarps,
                                             int32_t *picks, float *wts, int wstride, bool write_out) {
    const int lane = threadIdx.x & 31;
    for (int t = wi; t < T; t += nwarps) {
        int id;
        float w;
        router_topk_row(r, t, E, K, id, w);
        if (lane < K) {
            picks[t * K + lane] = id;
            wts[t * wstride + lane] = w;
            if (write_out) {
                if (r.ids_out) r.ids_out[t * K + lane] = id;
                if (r.w_out) r.w_out[t * K + lane] = w;
            }
        }
    }
}

// Standalone router launch (cooperative): the partial logits over every warp
// of the grid, a grid barrier, then each warp of the grid picks one row's
// experts at a time and writes them out.
__global__ void __launch_bounds__(256) route_kernel(const __nv_bfloat16 *x, RouterDev r, int T, int H, int E,
                                                    int K, WsHeader *hdr) {
    const int nwc = blockDim.x >> 5, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = (int)blockIdx.x * nwc + warp, nw = (int)gridDim.x * nwc;
    router_logits(r, x, T, H, E, gw, nw);
    if (!grid_barrier(hdr, gridDim.x, false)) return;
    for (int t = gw; t < T; t += nw) {
        int id;
        float w;
        router_topk_row(r, t, E, K, id, w);
        if (lane < K) {
            r.ids_out[t * K + lane] = id;
            r.w_out[t * K + lane] = w;
        }
    }
}

}  // namespace moe
