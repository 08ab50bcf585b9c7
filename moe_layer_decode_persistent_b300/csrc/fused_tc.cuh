// fused_tc.cuh -- the fused decode MoE layer on the tcgen05 tensor cores.
//
// One persistent cooperative launch, one CTA per SM, computes the whole layer
// ("Daily AI Hotspot 2026-08-21", section "Most Worth Your Attention Today":
// shared gate/up, routed experts, shared down and the residual add in one
// pass, FP32 accumulation, BF16 written once) over the step's deduplicated
// groups (PR #27 "each expert once", "Motivation"/"Modifications": each
// distinct expert streams its weights once, with every row that uses it as an
// MMA column; jobs are the intermediate tiles of each group, dealt over the
// CTAs; a row's output is summed in a fixed order so the dedup form is bitwise
// equal to the one-row form).
//
// Work items ("jobs"); CTA b takes job b first, later jobs are claimed in list
// order from one global counter:
//   gate/up job (group g, column tile ct, 128-row tile rt, K chunk kc):
//     tile0 = gate rows rt*128.., tile1 = up rows I+rt*128.., K = H chunk
//   down job (g, ct, 256-row tile ht, K chunk kc):
//     tile0 = rows ht*256.., tile1 = rows ht*256+128.., K = I chunk
// Both tiles of a job share the B operand (the group's activation columns).
// The K chunks depend on the launch's shape only (the dedup and one-row forms
// split work alike). The launch-wide counters (job claims, ready counts) come
// in two sets that alternate by launch parity, each launch zeroing the other.
//
// Per CTA the roles are warp-specialised (18 warps; 26 with the two-parity
// dequant build option):
//   warp 0      producer: claims jobs, TMA-loads 128-byte-wide weight boxes
//               (SWIZZLE_128B) and NVFP4 block scales into a ring of 2 to 6
//               stages (as many as shared memory holds next to the tables),
//               the first ones before the group table is built where the
//               shape alone defines the first job; at the end it watches the
//               output tiles for the combine
//   warp 1      B stager: copies the job's B tile per 128-K unit with
//               cp.async (not the TMA queue, which is full of weight boxes):
//               gate/up gathers each column from its row of the f16
//               activations (converted once per launch at the start, spread
//               over all CTAs); down copies the f16 intermediate. It first
//               waits for the operand's producers.
//   warps 2-5   MMA issuers: tcgen05.mma kind::f16, M=128, N=16|32, K=16,
//               A from TMEM, B from shared memory. One issuing thread sustains
//               one MMA per ~120 cycles whatever N is, so four issuers split
//               each unit: issuer q takes tile q&1, K-steps of half q>>1, into
//               its own accumulator (the halves are added in a fixed order)
//   warps 6-13  dequant, one warpgroup per tile: one thread per weight row,
//               E2M1*E4M3 -> exact f16 (or E4M3 -> f16), written to TMEM as the
//               MMA's A operand (the weights never touch shared memory as f16)
//   warps 14-17 epilogue: TMEM accumulators -> registers; FP8 128x128 block
//               scales applied per 128-K block in fp32; partial sums, the
//               fixed-order reductions, SwiGLU, the f16 intermediate, the down
//               partials
//   all warps   the final combine (fixed-order sum, single bf16 write), each
//               warp as soon as its role is done
//
// Precision: weights dequantise exactly to f16 (e2m1*e4m3 has <= 6
// significant bits); activations bf16 -> f16, each row scaled by a power of
// two that keeps its largest element below 16 (exact wherever f16 holds the
// scaled value); the fp32 SwiGLU intermediate is
// rounded once to f16 for the down MMA (relative error <= 2^-12 per element,
// about 1.4e-4 |y| rms on the down output); every accumulation is fp32.
#pragma once

#include <cuda.h>
#include <cuda_fp8.h>

#include "group_table.cuh"
#include "moe_common.cuh"
#include "router.cuh"
#include "sm100.cuh"

namespace moe {

#ifndef MOE_TC_DQ_PARITIES
#define MOE_TC_DQ_PARITIES 1
#endif
// Dequant warpgroups per tile: 1, or 2 taking alternate units (a build option
// that measured slower: 26 warps leave 72 registers and crowd the issuers).
constexpr int kDqPar = MOE_TC_DQ_PARITIES;
constexpr int kDqWarps = 8 * kDqPar;
constexpr int kTcThreads = 32 * (2 + 4 + kDqWarps + 4);
constexpr int kTcMaxT = 256;
constexpr int kNt = 32;               // columns per job at most (NVFP4, T > 16)
constexpr int kNtSmall = 16;          // columns per job when T <= 16, and for FP8 jobs
constexpr int kUnitK = 128;           // K elements of one TMEM A unit per tile
constexpr int kRawStagesMax = 6;      // raw weight ring: as many stages as shared memory holds, 2..6
constexpr int kRawStagesMin = 2;
constexpr int kRawTileBytes = 16384;  // 128 rows x 128 bytes
constexpr int kRawScaleOff = 2 * kRawTileBytes;
constexpr int kRawStageBytes = 2 * kRawTileBytes + 2 * 2048;  // + NVFP4 scales
constexpr int kBUnitBytes = kNt * kUnitK * 2;  // one B buffer: [32][128] f16 at most
constexpr int kASlotsMax = 3;         // TMEM A slots (each with its B buffer): 3 when jobs have 16 columns, else 2
constexpr int kIssuers = 4;
constexpr int kJobSlots = 4;
constexpr int kTmemCols = 512;
// Columns per job. Depends on the launch (T) and the format only, never on a
// group's size, so the dedup and one-row forms split work the same way.
__host__ __device__ constexpr int tc_nt(int fmt, int T) {
    return (fmt == kFmtFp8B128 || T <= 16) ? kNtSmall : kNt;
}
// TMEM: nA A slots of 128 columns, then two D sets of 4 x ntmax columns.
__host__ __device__ constexpr int tc_ntmax(int T) { return T <= 16 ? kNtSmall : kNt; }
__host__ __device__ constexpr int tc_aslots(int T) { return T <= 16 ? 3 : 2; }
constexpr int kKcNvfp4 = 1792;
constexpr int kKcFp8 = 1024;
constexpr int kKcDown = 1024;
constexpr int kSplitMaxT = 16;
constexpr int kCombBatch = 20;  // combine: partial sums loaded per batch (18 for DSv3 shapes at T <= 16)
// Launch-wide counters, two sets used in alternate launches (by parity).
constexpr int kTcReadyCap = 256 * 17;  // (group, column tile) pairs: at most T*(K+1)
constexpr int kTcHtileCap = 64;        // 256-row output tiles: H / 256 at most
constexpr int kTcMaxGrid = 1024;       // CTAs (SMs) a launch may have: one parity word each

struct TcMaps {
    CUtensorMap r13, r13s, r2, r2s, s13, s13s, s2, s2s;
};

// Job-list constants of one expert set (index 0: the shared expert, 1: the
// routed experts), fixed by the launch's shape and computed on the host, so
// the per-group bookkeeping at the start of a launch needs no division.
struct TcFmt {
    int nt, nt_shift;  // columns per job and log2 of it
    int tiles;         // 128-row tiles of the intermediate (Ig / 128)
    int nkc_gu, kc_gu; // gate/up K chunks and their length
    int nkc_dn, kc_dn; // down K chunks and their length
};

struct TcParams {
    TcMaps maps;
    const __nv_bfloat16 *x;
    const int32_t *ids;
    const float *topk_w;
    WeightsDev routed, shared;
    __nv_bfloat16 *out;
    int T, H, I, Is, E, K;
    int nR;  // raw weight ring stages (kRawStagesMin..kRawStagesMax)
    unsigned flags;
    WsHeader *hdr;
    uint32_t *group_ready;  // [2][kTcReadyCap], per parity, per (group, column tile)
    uint32_t *tile_cnt;     // per (group, column tile, 128-row tile); each launch leaves it zero
    uint32_t *htile_cnt;    // [2][kTcHtileCap], per parity, per 256-row output tile
    uint32_t *cta_par;      // [kTcMaxGrid]: CTA b's parity of its next launch, toggled by CTA b alone
    float *P;               // gate/up partials [kc][2][Ucap][Imax]
    float *Y;               // down partials [kc][Ucap][H]
    uint8_t *midB;          // f16 intermediate in MMA B layout
    __half *xh;             // the activations as f16 [T][H], each row scaled by 2^-xs[t]
    int32_t *xs;            // [T] the rows' activation scale exponents (0 <= xs <= 63)
    int Ucap, Imax;
    int route_mode;         // 1: the picks and weights come from the router, not ids/topk_w
    RouterDev router;
    TcFmt fc[2];            // 0: shared expert, 1: routed experts
    const uint8_t *nx13;    // or null: the next layer's shared gate/up weights (same shape and format),
    const uint8_t *nx13s;   // and their NVFP4 block scales; their first stages are requested into L2
};

struct TcJob {
    int kind;  // 0 gate/up, 1 down, -1 end
    int g, ct, tile, kc, nkc;
    int e, shared, fmt, Ig;
    int n, npad, col0;
    int k0, nunits;
    int rows0, rows1;
    int tile_id, pair;
    long long mid_off;  // bytes into midB of this (group, column tile)
};

// ---- per-launch constants shared by host and device -----------------------

// K chunks of the jobs up to kSplitMaxT rows. A launch with more rows streams
// more distinct experts per CTA, so its jobs are made twice as long: every job
// boundary costs a hand-off, while the last jobs' length sets how far apart the
// CTAs finish, which matters most when there are few jobs per CTA. The chunks
// depend on the launch's shape alone, never on its groups.
constexpr int kShortJobsMaxT = 2;
__host__ __device__ inline int tc_kc_gu(int fmt, int H, int T) {
    if (T > kSplitMaxT) return H;
    return (fmt == kFmtNvfp4 ? kKcNvfp4 : kKcFp8) * (T > kShortJobsMaxT ? 2 : 1);
}
__host__ __device__ inline int tc_nkc_gu(int fmt, int H, int T) {
    const int kc = tc_kc_gu(fmt, H, T);
    return (H + kc - 1) / kc;
}
__host__ __device__ inline int tc_kc_dn(int Ig, int T) {
    return T > kSplitMaxT ? Ig : kKcDown * (T > kShortJobsMaxT ? 2 : 1);
}
__host__ __device__ inline int tc_nkc_dn(int Ig, int T) {
    const int kc = tc_kc_dn(Ig, T);
    return (Ig + kc - 1) / kc;
}

// B-operand layout of a [n][128] f16 unit: core matrices of 8 columns x 8 K.
__device__ __forceinline__ uint32_t b_off(int n, int k) {
    return (uint32_t)(((n >> 3) * 16 + (k >> 3)) * 128 + (n & 7) * 16 + (k & 7) * 2);
}

// Shared-memory layout of the fused kernel (dynamic, 1024-aligned base): B
// buffers, job slots, barriers, small words, the group table with its per-group
// arrays, and last the raw weight ring (1024-aligned, for the 128-byte swizzle).
struct TcSmem {
    static constexpr int bbuf = 0;
    static constexpr int jobs = bbuf + kASlotsMax * kBUnitBytes;
    static constexpr int bars = jobs + kJobSlots * (int)sizeof(TcJob);
    // jfull, jempty, rfull, rempty, sfull, sempty, dfull, dempty, drain[4], coef, xs
    static constexpr int nbars = 2 * kJobSlots + 2 * kRawStagesMax + 2 * kASlotsMax + 2 * 2 + kIssuers + 2;
    static constexpr int misc = bars + nbars * 8;  // tmem addr, abort, down jobs per tile, parity
    static constexpr int tile_ready = misc + 64;   // per 256-row output tile: combine may start (64 max)
    static constexpr int red = tile_ready + 256;     // row-maximum reduction scratch (32 ints)
    static constexpr int tables = red + 128;         // group table, then per-group arrays
};
constexpr int kTcGroupArrays = 5;  // gu, dn, tile, mid and pair prefix sums

// The group table (per-group arrays of capacity gcap), the per-group prefix
// sums (gcap + 1 each), then two float arrays of C = T*(K+1): each (row, slot)'s
// combine weight and down global scale (slot 0 = shared expert), then the T
// rows' activation scale exponents. Up to
// kTcFullTablesMaxT rows the per-group arrays hold C entries (the compiler then
// sees a fixed layout); above, they hold the group capacity so the tables fit.
constexpr int kTcFullTablesMaxT = 64;
__host__ __device__ inline bool tc_capped_tables(int T) { return T > kTcFullTablesMaxT; }
__host__ __device__ inline int tc_gcap(int T, int K, int E, bool no_dedup) {
    return tc_capped_tables(T) ? group_capacity(T, K, E, no_dedup) : T * (K + 1);
}
__host__ __device__ inline int tc_raw_offset(int T, int K, int gcap) {
    const int C = T * (K + 1);
    const int end = TcSmem::tables + 4 * (group_table_ints_cap(T, K, gcap) + kTcGroupArrays * (gcap + 1) + 2 * C + T + 1);
    return (end + 1023) & ~1023;
}
// Dynamic shared memory for nR raw stages (+1024 to align the base).
__host__ __device__ inline int tc_smem_bytes(int T, int K, int E, bool no_dedup, int nR) {
    return tc_raw_offset(T, K, tc_gcap(T, K, E, no_dedup)) + nR * kRawStageBytes + 1024;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// group of column c: the last g with g0[g] <= c
__device__ __forceinline__ int group_of_col(const int32_t *g0, int G, int c) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g0[mid] <= c) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The activations -> f16 [T][H], the gate/up MMA's B operand, each row t
// scaled by an exact power of two 2^-s_t: s_t = 0 while the row's largest
// magnitude is below 16, else the shift that brings it into [8, 16) (at most
// 63). Rows without a shift convert exactly as bf16 -> f16 (exact for |x| in
// [2^-17, 65504]); a shifted row keeps f16's 11 bits for everything within
// 2^-24 of its largest element. The gate/up epilogue undoes the shift inside
// the SwiGLU and the combine undoes its square, so results are unchanged
// except where f16 would have overflowed (MOE_DEV_RANGE is left for
// non-finite inputs and intermediates).
//
// Rows are shared out over the CTAs: with T < grid, the CTAs b = t + T*k
// (k < grid / T) split row t's 16-byte items between them; with T >= grid,
// CTA b converts rows b, b + grid, ... whole. Each CTA finds the maximum of
// the rows it touches itself (a reduction over the converting warps behind
// named barrier `bar`), so the shift needs no exchange between CTAs; the CTA holding a
// row's first slice writes s_t.
constexpr int kMaxActShift = 63;
constexpr int kWarpTablePicks = 32;  // up to this many picks, warp 1 alone builds the group table
constexpr int kWarpPicks = 128;      // up to this many picks, warp 1 alone loads them
// The raw stages that CTA b requests before its group table is built: its
// first job, when that is one of the shared expert's gate/up jobs (the shared
// expert is group 0 in either form and its gate/up jobs come first in the
// list), which the launch's shape alone defines. Returns how many stages (0:
// the first job is another one), with the job's 128-row tile and first K
// element.
__device__ __forceinline__ int tc_first_stages(const TcParams &p, bool no_dedup, int nR, int *tile, int *k0) {
    const TcFmt &f0 = p.fc[0];
    const int n0 = no_dedup ? 1 : p.T;
    const int tiles0 = f0.tiles, nkc0 = f0.nkc_gu, b = (int)blockIdx.x;
    if (b >= ((n0 + f0.nt - 1) >> f0.nt_shift) * tiles0 * nkc0) return 0;
    const int rem = b % (tiles0 * nkc0), kc = rem % nkc0;
    *tile = rem / nkc0;
    *k0 = kc * f0.kc_gu;
    const bool fp4 = p.shared.fmt == kFmtNvfp4;
    const int nst = (min(f0.kc_gu, p.H - *k0) / kUnitK) / (fp4 ? 2 : 1);
    return min(nst, nR - 1);
}

__device__ __forceinline__ int act_shift(uint32_t max_abs_bits) {
    const int e = (int)(max_abs_bits >> 7) - 127;  // bf16 exponent of the largest magnitude
    return (max_abs_bits >= 0x7f80u) ? 0 : max(0, min(e - 3, kMaxActShift));
}

__device__ __forceinline__ bool tc_convert_rows(const TcParams &p, int tid1, int nthr1, int bar, uint32_t *red_s) {
    constexpr int kMaxItems = 4;  // 16-byte items of a row a thread holds: H <= 16384, 16 warps
    const int T = p.T, G = (int)gridDim.x, b = (int)blockIdx.x;
    const int n8 = p.H / 8;  // 16-byte items per row
    const int nsl = T < G ? G / T : 1;  // CTAs per row
    const int t0 = T < G ? b % T : b, dt = T < G ? T : G;
    const int sl = T < G ? b / T : 0;
    bool shifted = false;  // some row of this CTA's share is shifted (meaningful on tid1 0)
    if (sl >= nsl) return shifted;  // no slice for this CTA
    uint4 *dst = reinterpret_cast<uint4 *>(p.xh);
    uint32_t range_bad = 0;
    for (int t = t0; t < T; t += dt) {
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x) + (size_t)t * n8;
        // the row's largest magnitude (bf16 bits without sign: monotone); the
        // items stay in registers for the conversion below
        uint4 v[kMaxItems];
        uint32_t mx = 0;
#pragma unroll
        for (int k = 0; k < kMaxItems; ++k) {
            const int i = tid1 + k * nthr1;
            v[k] = i < n8 ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kMaxItems; ++k) {
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) mx = max(mx, max(w4[q] & 0x7fffu, (w4[q] >> 16) & 0x7fffu));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if ((tid1 & 31) == 0) red_s[tid1 >> 5] = mx;
        sm100::named_bar_sync(bar, nthr1);
        uint32_t rowmax = 0;
        for (int w = 0; w < nthr1 / 32; ++w) rowmax = max(rowmax, red_s[w]);
        sm100::named_bar_sync(bar, nthr1);  // red_s may be reused for the next row
        const int sh = act_shift(rowmax);
        const float f = __uint_as_float((uint32_t)(127 - sh) << 23);  // 2^-sh, exact
        if (sl == 0 && tid1 == 0) p.xs[t] = sh;
        shifted |= sh != 0;
        // this CTA's slice of the row's items
        const int i0 = (int)((long long)n8 * sl / nsl), i1 = (int)((long long)n8 * (sl + 1) / nsl);
#pragma unroll
        for (int k = 0; k < kMaxItems; ++k) {
            const int i = tid1 + k * nthr1;
            if (i < i0 || i >= i1) continue;
            const uint32_t w4[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const __half2 h = __floats2half2_rn(__fmul_rn(bf16_bits_to_float(w4[q] & 0xffffu), f),
                                                    __fmul_rn(bf16_bits_to_float(w4[q] >> 16), f));
                if (__hisinf(__low2half(h)) || __hisinf(__high2half(h))) range_bad = 1;
                o[q] = pack_h2(h);
            }
            dst[(size_t)t * n8 + i] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    if (range_bad) atomicOr(&p.hdr->err, kErrRange);
    return shifted;
}
static_assert(16384 / 8 <= 4 * (kTcThreads - 64), "a row's items fit the converting threads' registers");

// This CTA's slice of the activations (and its shifted-row flag) goes out to
// the grid: a release after the barrier that ordered the converting warps'
// stores.
__device__ __forceinline__ void tc_publish_x(const TcParams &p, int par, bool shifted) {
    if (shifted) atomicOr(&p.hdr->x_scaled[par], 1u);
    __threadfence();
    red_add_release_gpu(&p.hdr->x_ready[par], 1u);
}

// SwiGLU of a column whose activations were scaled by 2^-s (g, u: the scaled
// gate and up sums, global scales applied; fs = 2^s, fis = 2^-s): the true
// silu(g 2^s) (u 2^s), scaled by 2^-2s. With s = 0 it is silu(g) u exactly.
__device__ __forceinline__ float swiglu_scaled(float g, float u, float fs, float fis) {
    return __fmul_rn(__fmul_rn(silu_f32(__fmul_rn(g, fs)), fis), u);
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }  // |e| <= 126

// FP8 intermediate blocks (MOE_FLAG_FP8_MID; PR #27 "each expert once",
// "Modifications": FP8 mid blocks). The warp's 32 values of one column (one
// per lane: 32 consecutive intermediate rows) share the smallest power-of-two
// scale 2^k with max|m| <= 448 * 2^k (k >= -126), and each becomes its nearest
// E4M3 value (ties to even) times 2^k, which f16 then holds exactly. 448 is
// 1.75 * 2^8, so with max|m| = f 2^E (f in [1, 2)) k = E - 8, plus one when
// f > 1.75. Warp-collective; an all-zero or non-finite block is left as it is
// (the range check flags the latter).
__device__ __forceinline__ float fp8_mid_q(float m) {
    float a = fabsf(m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const uint32_t b = __float_as_uint(a);
    if (a == 0.0f || b >= 0x7f800000u) return m;
    const int k = max((int)(b >> 23) - 127 - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0), -126);
    const __nv_fp8_storage_t q = __nv_cvt_float_to_fp8(__fmul_rn(m, pow2f(-k)), __NV_SATFINITE, __NV_E4M3);
    return __fmul_rn(__half2float(__half(__nv_cvt_fp8_to_halfraw(q, __NV_E4M3))), pow2f(k));
}

// kRouted: the picks and weights come from the router inside the launch (a
// separate instantiation, so the router's registers never weigh on the
// unrouted kernel's hot loops).
// kFp8Mid: the opt-in FP8 intermediate blocks, an instantiation of its own so
// the default kernels' code is unchanged by it.
template <bool kCappedTables, bool kRouted, bool kFp8Mid>
__global__ void __launch_bounds__(kTcThreads, 1) fused_tc_kernel(const __grid_constant__ TcParams p) {
    using namespace sm100;
    extern __shared__ __align__(1024) uint8_t smem_raw_[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw_) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = p.T, K = p.K, H = p.H;
    const bool no_dedup = (p.flags & kFlagNoDedup) != 0;
    const int nA = tc_aslots(T), ntmax = tc_ntmax(T), nR = p.nR;
    const int dcol0 = nA * 128, dset = 4 * ntmax;  // TMEM D set base and size

    const int C = T * (K + 1), gcap = kCappedTables ? group_capacity(T, K, p.E, no_dedup) : C;
    uint8_t *raw = smem + tc_raw_offset(T, K, gcap);
    uint8_t *bbuf = smem + TcSmem::bbuf;
    TcJob *jobs = reinterpret_cast<TcJob *>(smem + TcSmem::jobs);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + TcSmem::bars);
    uint64_t *jfull = bars, *jempty = jfull + kJobSlots;
    uint64_t *rfull = jempty + kJobSlots, *rempty = rfull + kRawStagesMax;
    // a unit slot = one TMEM A slot + one B buffer, filled by the dequant
    // warps and the B stager together and released by one commit per issuer
    uint64_t *sfull = rempty + kRawStagesMax, *sempty = sfull + kASlotsMax;
    uint64_t *dfull = sempty + kASlotsMax, *dempty = dfull + 2;
    uint64_t *drain = dempty + 2;
    uint64_t *coef_bar = drain + kIssuers;  // the combine coefficients are filled
    uint64_t *xs_bar = coef_bar + 1;        // the rows' activation scales are in xs_s
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(smem + TcSmem::misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + TcSmem::misc + 4);
    int *dn_per_ht_s = reinterpret_cast<int *>(smem + TcSmem::misc + 8);
    int *par_s = reinterpret_cast<int *>(smem + TcSmem::misc + 12);
    int *shifted_s = reinterpret_cast<int *>(smem + TcSmem::misc + 16);  // some row of this CTA's share is shifted
    uint32_t *tile_ready_s = reinterpret_cast<uint32_t *>(smem + TcSmem::tile_ready);
    int32_t *tbl = reinterpret_cast<int32_t *>(smem + TcSmem::tables);
    GroupTable tab{tbl, C, gcap};
    int *gu_prefix = tbl + tab.ints();
    int *dn_prefix = gu_prefix + (gcap + 1);
    int *tile_prefix = dn_prefix + (gcap + 1);
    int *mid_prefix = tile_prefix + (gcap + 1);
    int *pair_prefix = mid_prefix + (gcap + 1);
    float *comb_w = reinterpret_cast<float *>(pair_prefix + (gcap + 1));  // [T][K+1]
    float *comb_g = comb_w + C;                                        // [T][K+1]
    int32_t *xs_s = reinterpret_cast<int32_t *>(comb_g + C);           // [T + 1]
    uint32_t *err = &p.hdr->err;

    // ---- prologue -----------------------------------------------------------
    // Warp 0 (the producer) sets up the barriers, helps build the group table,
    // sums the per-group job counts and starts streaming weights at once; the
    // other warps convert the activations meanwhile, then fill the combine
    // coefficients, then take up their roles.
    const int nw1 = kTcThreads - 32;  // threads of warps 1..
    // one raw stage: tile0 and tile1 boxes of 128 bytes x 128 rows at byte
    // column kb (and their NVFP4 scale boxes at column ks), completing on rfull
    auto tma_stage = [&](int st, const CUtensorMap *mc, const CUtensorMap *ms, bool fp4, int kb, int ks, int rows0,
                         int rows1, int e, uint64_t pol) {
        uint8_t *dst = raw + st * kRawStageBytes;
        mbar_arrive_expect_tx(&rfull[st], fp4 ? kRawStageBytes : 2 * kRawTileBytes);
        tma_load_3d_hint(dst, mc, kb, rows0, e, &rfull[st], pol);
        tma_load_3d_hint(dst + kRawTileBytes, mc, kb, rows1, e, &rfull[st], pol);
        if (fp4) {
            tma_load_3d_hint(dst + kRawScaleOff, ms, ks, rows0, e, &rfull[st], pol);
            tma_load_3d_hint(dst + kRawScaleOff + 2048, ms, ks, rows1, e, &rfull[st], pol);
        }
    };
    int npre = 0;  // stages of this CTA's first job issued before the group table
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < kJobSlots; ++i) {
            mbar_init(&jfull[i], 1);
            mbar_init(&jempty[i], 1 + kIssuers + kDqWarps + 4);  // stager, issuers, dequant, epilogue
        }
        for (int i = 0; i < kRawStagesMax; ++i) {
            mbar_init(&rfull[i], 1);
            mbar_init(&rempty[i], kDqWarps);
        }
        for (int i = 0; i < kASlotsMax; ++i) {
            mbar_init(&sfull[i], 8 + 32);  // 8 dequant warps + one cp.async arrival per stager lane
            mbar_init(&sempty[i], kIssuers);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&dfull[i], kIssuers);
            mbar_init(&dempty[i], 4);
        }
        for (int i = 0; i < kIssuers; ++i) mbar_init(&drain[i], 1);
        mbar_init(coef_bar, 4);  // one arrival per epilogue warp
        mbar_init(xs_bar, 1);    // the first epilogue warp
        for (int i = 0; i < 64; ++i) tile_ready_s[i] = 0;
        *abort_flag = 0;
        fence_mbar_init();
        // When this CTA's first job is one of the shared expert's gate/up jobs,
        // its first stages stream in while the group table is built (the
        // table's scratch sits in the ring's last stage). Weights only: they
        // are constant, so a chained launch may request them at once.
        int tile0 = 0, k00 = 0;
        npre = tc_first_stages(p, no_dedup, nR, &tile0, &k00);
        if (npre) {
            fence_proxy_async_smem();
            const bool fp4 = p.shared.fmt == kFmtNvfp4;
            const uint64_t pol = l2_evict_first_policy();
            for (int st = 0; st < npre; ++st)
                tma_stage(st, &p.maps.s13, &p.maps.s13s, fp4, (fp4 ? k00 / 2 : k00) + st * 128, k00 / 16 + st * 16,
                          tile0 * 128, p.Is + tile0 * 128, 0, pol);
        }
    }
    if (warp != 1) griddep_wait();
    // A chained launch may have started under the previous kernel on the
    // stream: up to here it has touched only its own shared memory, TMEM and
    // constant weights. Inputs and the workspace are read after the previous
    // grid has completed.
    uint32_t start_no = 0;
    if (warp == 1) {
        griddep_wait();
        // this launch's parity: every CTA keeps its own word, flipped once per
        // launch, so all CTAs of a launch read the same value without a shared
        // counter. Only tid 32 uses it, when it publishes this CTA's
        // activations, so the load's round trip overlaps the TMEM allocation,
        // the picks and the conversion.
        if (lane == 0) {
            uint32_t *cp = p.cta_par + blockIdx.x;
            start_no = __ldcg(cp);
            __stcg(cp, start_no ^ 1u);
        }
        __syncwarp();
        tmem_alloc(tmem_base_s, kTmemCols);
        tc_fence_before();
    }
    int *gt_scr = reinterpret_cast<int *>(raw + (nR - 1) * kRawStageBytes);  // group table scratch
    // The step's picks and router weights go first, ahead of the conversion
    // and the weight stream: the picks into the group table's scratch, the
    // weights into the pick slots of the combine weights (a routed launch
    // computes both on chip below). Up to kWarpPicks picks, warp 1 alone
    // loads them (warps 2.. start converting at once); up to kWarpTablePicks,
    // warp 1 also builds the group table while warps 2.. convert (the table
    // is short, once-per-launch code whose instruction fetches dominate it);
    // above, warps 1.. share both, the table after the conversion.
    const bool warp_table = !kRouted && T * K <= kWarpTablePicks;
    const int nT = warp_table ? 32 : nw1;  // threads that build the table
    if (!kRouted && T * K <= kWarpPicks) {
        if (warp == 1) {  // all loads in flight at once, then the stores
            int32_t *picks = group_table_picks(gt_scr, p.E);
            int32_t v[kWarpPicks / 32];
            float w[kWarpPicks / 32];
#pragma unroll
            for (int r = 0; r < kWarpPicks / 32; ++r) {
                const int j = lane + 32 * r;
                v[r] = j < T * K ? __ldg(p.ids + j) : 0;
                w[r] = j < T * K ? __ldg(p.topk_w + j) : 0.0f;
            }
#pragma unroll
            for (int r = 0; r < kWarpPicks / 32; ++r) {
                const int j = lane + 32 * r;
                if (j < T * K) {
                    picks[j] = v[r];
                    comb_w[j + j / K + 1] = w[r];  // [t][1 + q]
                }
            }
        }
    } else if (!kRouted && warp >= 1) {
        int32_t *picks = group_table_picks(gt_scr, p.E);
        for (int j = tid - 32; j < T * K; j += nw1) {
            picks[j] = __ldg(p.ids + j);
            comb_w[j + j / K + 1] = __ldg(p.topk_w + j);
        }
    }
    // warps 2.. convert (warp 1 allocates TMEM, reads the parity and builds
    // a small table meanwhile, so the row maxima's barrier does not wait for it)
    if (warp >= 2) {
        const bool shifted = tc_convert_rows(p, tid - 64, nw1 - 32, 3, reinterpret_cast<uint32_t *>(smem + TcSmem::red));
        if (tid == 64) *shifted_s = shifted ? 1 : 0;  // read after the CTA barrier below
    }

    // routed launches: warps 1.. of every CTA compute their share of the
    // router's partial logits (warp 0 streams the first weights meanwhile),
    // then every CTA waits for all of them and picks every row's experts on
    // chip: the picks go to the group table's scratch, the weights to the
    // combine weights of the pick slots
    if (kRouted && warp >= 1) {
        const int ncw = kTcThreads / 32 - 1;
        router_logits(p.router, p.x, T, H, p.E, (warp - 1) * (int)gridDim.x + (int)blockIdx.x,
                      ncw * (int)gridDim.x);
        named_bar_sync(2, nw1);
        if (tid == 32) {
            __threadfence();
            uint32_t *rr = &p.hdr->route_ready[start_no];
            red_add_release_gpu(rr, 1u);
            const unsigned long long t0 = globaltimer_ns();
            while (ld_acquire_gpu(rr) < gridDim.x) {
                if (globaltimer_ns() - t0 > kWaitBudgetNs) {
                    atomicOr(err, kErrWaitTimeout);
                    *abort_flag = 1;
                    break;
                }
                __nanosleep(64);
            }
        }
        named_bar_sync(2, nw1);
        int32_t *picks = group_table_picks(gt_scr, p.E);
        if (*abort_flag) {
            for (int j = tid - 32; j < T * K; j += nw1) picks[j] = -1;
        } else {
            router_picks(p.router, T, p.E, K, warp - 1, ncw, picks, comb_w + 1, K + 1, blockIdx.x == 0);
        }
    }

    // the group table, by the threads that loaded the picks, behind named
    // barrier 1 (warp 0 streams meanwhile; the table's scratch is the raw
    // ring's last stage); one CTA barrier then publishes the mbarriers, the
    // TMEM address, the parity, the table and this CTA's activation slice
    if (warp >= 1 && tid - 32 < nT)
        group_table_cta(nullptr, T, K, p.E, no_dedup, tab, gt_scr, blockIdx.x == 0 ? err : nullptr, 32, nT, 1);
    // This CTA's activation slice goes out to the grid from tid 32 once a
    // barrier has ordered the converting warps' stores: with a one-warp table
    // after the CTA barrier (so no warp waits for the fence), else right after
    // the table's own barriers, which the converting warps take part in.
    if (tid == 32) {
        *par_s = (int)start_no;
        if (!warp_table) tc_publish_x(p, (int)start_no, *shifted_s != 0);
    }
    __syncthreads();
    tc_fence_after();
    griddep_launch_dependents();  // a chained next launch may now take each SM this grid leaves
    if (tid == 32 && warp_table) tc_publish_x(p, (int)start_no, *shifted_s != 0);
    const int G = tab.G();
    const int32_t *gexp = tab.gexp(), *gn = tab.gncols(), *g0 = tab.gcol0(), *rcol = tab.row_col();
    const int *crow = tab.col_row();
    const int par = *par_s;
    uint32_t *group_ready = p.group_ready + par * kTcReadyCap;
    uint32_t *htile_cnt = p.htile_cnt + par * kTcHtileCap;
    if (warp == 0) {
        // per-group job counts and their prefix sums, 32 groups per round:
        // gate/up jobs, down jobs, (column tile, row tile) pairs, padded
        // intermediate columns x row tiles, column tiles, and down jobs per
        // 256-row output tile
        int run[6] = {0, 0, 0, 0, 0, 0};
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int v[6] = {0, 0, 0, 0, 0, 0};
            if (g < G) {
                const TcFmt &f = p.fc[gexp[g] < 0 ? 0 : 1];
                const int n = gn[g], nct = (n + f.nt - 1) >> f.nt_shift;
                const int last = n - (nct - 1) * f.nt;  // columns of the last column tile
                const int np = (nct - 1) * f.nt + ((last + 15) & ~15);
                v[0] = nct * f.tiles * f.nkc_gu;
                v[1] = nct * (H >> 8) * f.nkc_dn;
                v[2] = nct * f.tiles;
                v[3] = np * f.tiles;
                v[4] = nct;
                v[5] = nct * f.nkc_dn;
            }
            int sc[6];
#pragma unroll
            for (int a = 0; a < 6; ++a) sc[a] = v[a];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
                for (int a = 0; a < 6; ++a) {
                    const int y = __shfl_up_sync(0xffffffffu, sc[a], o);
                    if (lane >= o) sc[a] += y;
                }
            }
            if (g < G) {
                gu_prefix[g] = run[0] + sc[0] - v[0];
                dn_prefix[g] = run[1] + sc[1] - v[1];
                tile_prefix[g] = run[2] + sc[2] - v[2];
                mid_prefix[g] = run[3] + sc[3] - v[3];
                pair_prefix[g] = run[4] + sc[4] - v[4];
            }
#pragma unroll
            for (int a = 0; a < 6; ++a) run[a] += __shfl_sync(0xffffffffu, sc[a], 31);
        }
        if (lane == 0) {
            gu_prefix[G] = run[0];
            dn_prefix[G] = run[1];
            tile_prefix[G] = run[2];
            mid_prefix[G] = run[3];
            pair_prefix[G] = run[4];
            // down jobs that write one 256-row output tile; read by the other
            // warps after their first job-slot wait
            *dn_per_ht_s = run[5];
        }
        __syncwarp();
    } else {
        // zero the other parity's counters for the next launch (the launch
        // before this one was their last user)
        {
            const int opar = par ^ 1;
            const int gt = (int)blockIdx.x * nw1 + (tid - 32);
            const int nz = kTcReadyCap + kTcHtileCap + 4;
            for (int i = gt; i < nz; i += nw1 * (int)gridDim.x) {
                if (i < kTcReadyCap) p.group_ready[opar * kTcReadyCap + i] = 0u;
                else if (i < kTcReadyCap + kTcHtileCap) p.htile_cnt[opar * kTcHtileCap + i - kTcReadyCap] = 0u;
                else if (i == kTcReadyCap + kTcHtileCap) p.hdr->job_next[opar] = 0u;
                else if (i == kTcReadyCap + kTcHtileCap + 1) p.hdr->x_ready[opar] = 0u;
                else if (i == kTcReadyCap + kTcHtileCap + 2) p.hdr->route_ready[opar] = 0u;
                else p.hdr->x_scaled[opar] = 0u;
            }
        }
    }
    const uint32_t tmem = *tmem_base_s;

    auto job_at = [&](int slot) -> TcJob { return jobs[slot]; };

    if (warp == 0) {
        // ===================== producer =====================
        if (lane == 0) {
            const int NGU = gu_prefix[G], njobs = NGU + dn_prefix[G];
            int js = 0, jph = 0, rs = npre, rph = 0;  // npre < nR
            int cur_gu = 0, cur_dn = 0;
            int skip = npre;                         // the first job's stages already issued
            uint32_t armed = (1u << npre) - 1u;     // raw stages with a TMA in flight not yet seen consumed
            // CTA b takes job b first, with no claim; later jobs come from the counter.
            // The next job is claimed just before the current job's last stage
            // waits for its slot, so the claim's round trip overlaps that wait.
            int j = (int)blockIdx.x;
            for (;;) {
                TcJob d;
                if (*abort_flag || j >= njobs) {
                    d.kind = -1;
                } else {
                    const bool gu = j < NGU;
                    int g, local;
                    if (gu) {
                        while (gu_prefix[cur_gu + 1] <= j) ++cur_gu;
                        g = cur_gu;
                        local = j - gu_prefix[g];
                    } else {
                        const int jd = j - NGU;
                        while (dn_prefix[cur_dn + 1] <= jd) ++cur_dn;
                        g = cur_dn;
                        local = jd - dn_prefix[g];
                    }
                    const bool sh = gexp[g] < 0;
                    const TcFmt &f = p.fc[sh ? 0 : 1];
                    d.g = g;
                    d.shared = sh;
                    d.e = sh ? 0 : gexp[g];
                    d.fmt = sh ? p.shared.fmt : p.routed.fmt;
                    d.Ig = sh ? p.Is : p.I;
                    const int tiles = f.tiles;
                    const int nt = f.nt;
                    if (gu) {
                        d.kind = 0;
                        d.nkc = f.nkc_gu;
                        const int per_ct = tiles * d.nkc;
                        d.ct = local / per_ct;
                        const int rem = local - d.ct * per_ct;
                        d.tile = rem / d.nkc;
                        d.kc = rem - d.tile * d.nkc;
                        const int kc_len = f.kc_gu;
                        d.k0 = d.kc * kc_len;
                        d.nunits = min(kc_len, H - d.k0) / kUnitK;
                        d.rows0 = d.tile * 128;
                        d.rows1 = d.Ig + d.tile * 128;
                    } else {
                        d.kind = 1;
                        d.nkc = f.nkc_dn;
                        const int per_ct = (H >> 8) * d.nkc;
                        d.ct = local / per_ct;
                        const int rem = local - d.ct * per_ct;
                        d.tile = rem / d.nkc;
                        d.kc = rem - d.tile * d.nkc;
                        const int kc_len = f.kc_dn;
                        d.k0 = d.kc * kc_len;
                        d.nunits = min(kc_len, d.Ig - d.k0) / kUnitK;
                        d.rows0 = d.tile * 256;
                        d.rows1 = d.tile * 256 + 128;
                    }
                    d.n = min(nt, gn[g] - d.ct * nt);
                    d.npad = ((d.n + 15) / 16) * 16;
                    d.col0 = g0[g] + d.ct * nt;
                    d.tile_id = tile_prefix[g] + d.ct * tiles + (d.kind == 0 ? d.tile : 0);
                    d.pair = pair_prefix[g] + d.ct;
                    d.mid_off = ((long long)mid_prefix[g] + (long long)d.ct * tiles * nt) * 256ll;
                }
                if (!mbar_wait(&jempty[js], jph ^ 1, abort_flag, err)) break;
                jobs[js] = d;
                mbar_arrive(&jfull[js]);
                if (++js == kJobSlots) {
                    js = 0;
                    jph ^= 1;
                }
                if (d.kind < 0) break;
                // weight boxes for the job: 128-byte-wide slices of tile0 and tile1 rows
                const CUtensorMap *mc, *ms;
                if (d.kind == 0) {
                    mc = d.shared ? &p.maps.s13 : &p.maps.r13;
                    ms = d.shared ? &p.maps.s13s : &p.maps.r13s;
                } else {
                    mc = d.shared ? &p.maps.s2 : &p.maps.r2;
                    ms = d.shared ? &p.maps.s2s : &p.maps.r2s;
                }
                const bool fp4 = d.fmt == kFmtNvfp4;
                const int upst = fp4 ? 2 : 1;
                const int nst = d.nunits / upst;
                const int kb0 = fp4 ? d.k0 / 2 : d.k0;
                const uint64_t pol = l2_evict_first_policy();  // weights are read once
                bool ok = true;
                int next = -1;
                for (int s = skip; s < nst; ++s) {
                    if (s == nst - 1) next = (int)gridDim.x + (int)atomicAdd(&p.hdr->job_next[par], 1u);
                    if (!mbar_wait(&rempty[rs], rph ^ 1, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    armed &= ~(1u << rs);
                    tma_stage(rs, mc, ms, fp4, kb0 + s * 128, d.k0 / 16 + s * 16, d.rows0, d.rows1, d.e, pol);
                    armed |= 1u << rs;
                    if (++rs == nR) {
                        rs = 0;
                        rph ^= 1;
                    }
                }
                skip = 0;
                if (!ok) break;
                j = next >= 0 ? next : (int)gridDim.x + (int)atomicAdd(&p.hdr->job_next[par], 1u);
            }
            // never leave with a TMA write into shared memory still in flight
            if (*abort_flag && armed) {
                for (int s = 0; s < nR; ++s) {
                    if (!(armed >> s & 1u)) continue;
                    // the phase armed last for slot s has parity rph if s < rs, else rph ^ 1
                    const uint32_t par = (s < rs) ? (uint32_t)rph : (uint32_t)(rph ^ 1);
                    const unsigned long long t0 = globaltimer_ns();
                    while (!mbar_try_wait(&rfull[s], par) && globaltimer_ns() - t0 < kWaitBudgetNs) {
                    }
                }
            }
        }
        // Every job is claimed: while this launch drains and combines, the
        // stages that CTA b of the next launch (same shape, the next layer's
        // shared expert) requests first are brought into L2, so they arrive
        // from L2 instead of HBM when that launch starts.
        __syncwarp();
        if (p.nx13 && !*abort_flag) {
            int tile = 0, k0 = 0;
            const int n = tc_first_stages(p, no_dedup, nR, &tile, &k0);
            if (n) {
                const bool fp4 = p.shared.fmt == kFmtNvfp4;
                const size_t rb = fp4 ? (size_t)H / 2 : (size_t)H, sb = (size_t)H / 16;  // bytes per row
                for (int r = lane; r < 256; r += 32) {
                    const size_t row = (size_t)(r < 128 ? tile * 128 + r : p.Is + tile * 128 + (r - 128));
                    prefetch_l2_bulk(p.nx13 + row * rb + (fp4 ? k0 / 2 : k0), (uint32_t)n * 128u);
                    if (fp4) prefetch_l2_bulk(p.nx13s + row * sb + k0 / 16, (uint32_t)n * 16u);
                }
            }
        }
    } else if (warp == 1) {
        // ===================== B stager =====================
        int js = 0, jph = 0, bs = 0, bph = 0;  // unit slot ring position
        const uint32_t bunit = (uint32_t)ntmax * kUnitK * 2;  // bytes of one B buffer
        const int nl = lane & 7, kq = lane >> 3;  // gather: column within an 8-column block, K quarter
        bool x_seen = false;
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait(&jfull[js], jph, abort_flag, err))) break;
            const TcJob d = job_at(js);
            __syncwarp();
            if (lane == 0) mbar_arrive(&jempty[js]);
            if (++js == kJobSlots) {
                js = 0;
                jph ^= 1;
            }
            if (d.kind < 0) break;
            // wait until the B operand's producers are done: every CTA's slice
            // of the activations (gate/up; once per launch) or every quarter of
            // every row tile of the group's intermediate (down)
            int okl = 1;
            if (lane == 0 && !(d.kind == 0 && x_seen)) {
                const uint32_t need = d.kind == 0 ? gridDim.x : (uint32_t)(4 * (d.Ig / 128));
                const uint32_t *flag = d.kind == 0 ? &p.hdr->x_ready[par] : group_ready + d.pair;
                if (ld_acquire_gpu(flag) < need) {
                    const unsigned long long t0 = globaltimer_ns();
                    while (ld_acquire_gpu(flag) < need) {
                        if (*abort_flag) {
                            okl = 0;
                            break;
                        }
                        if (globaltimer_ns() - t0 > kWaitBudgetNs) {
                            atomicOr(err, kErrWaitTimeout);
                            *abort_flag = 1;
                            okl = 0;
                            break;
                        }
                        __nanosleep(64);
                    }
                }
            }
            // the other lanes' copies below are ordered after lane 0's acquire
            bool ok = __shfl_sync(0xffffffffu, okl, 0) != 0;
            __syncwarp();
            if (d.kind == 0) x_seen = true;
            // gate/up: this lane's columns nb*8 + nl (nb < npad/8) come from
            // their rows of xh and the padding columns are zero-filled without
            // a read (many lanes reading one address slows the copies down);
            // down: the contiguous intermediate
            const __half *xrow[kNt / 8];
#pragma unroll
            for (int nb = 0; nb < kNt / 8; ++nb)
                xrow[nb] = p.xh + (size_t)crow[d.col0 + min(nb * 8 + nl, d.n - 1)] * H + kq * 8;
            const uint32_t bytes = (uint32_t)d.npad * 256u;
            const uint8_t *mid0 = p.midB + d.mid_off;
            for (int u = 0; u < d.nunits && ok; ++u) {
                if (!__all_sync(0xffffffffu, mbar_wait(&sempty[bs], bph ^ 1, abort_flag, err))) {
                    ok = false;
                    break;
                }
                {
                    const int ku = d.k0 / kUnitK + u;  // global K unit index
                    uint8_t *dst = bbuf + bs * bunit;
                    if (d.kind == 0) {
                        // B layout: core matrices of 8 columns x 8 K, 2048 B per 8 columns
                        uint8_t *dl = dst + kq * 128 + nl * 16;
#pragma unroll
                        for (int nb = 0; nb < kNt / 8; ++nb)
                            if (nb < d.npad / 8)
#pragma unroll
                                for (int m = 0; m < 4; ++m)
                                    cp_async16_zfill(dl + nb * 2048 + m * 512, xrow[nb] + ku * kUnitK + m * 32,
                                                     nb * 8 + nl < d.n ? 16u : 0u);
                    } else {
                        const uint8_t *src = mid0 + (long long)ku * bytes;
                        for (uint32_t o = (uint32_t)lane * 16; o < bytes; o += 32 * 16) cp_async16(dst + o, src + o);
                    }
                    cp_async_arrive_noinc(&sfull[bs]);
                }
                if (++bs == nA) {
                    bs = 0;
                    bph ^= 1;
                }
            }
            if (!ok) break;
        }
        cp_async_wait_all();  // no copy into shared memory outlives the role
    } else if (warp < 2 + kIssuers) {
        // ===================== MMA issuers (warps 2-5) =====================
        if (lane == 0) {
            const int q = warp - 2, tile = q & 1, kh = q >> 1;
            int js = 0, jph = 0, as = 0, aph = 0, ds = 0, dph = 0;
            const uint32_t bunit = (uint32_t)ntmax * kUnitK * 2;
            bool issued = false;
            for (;;) {
                if (!mbar_wait(&jfull[js], jph, abort_flag, err)) break;
                const TcJob d = job_at(js);
                mbar_arrive(&jempty[js]);
                if (++js == kJobSlots) {
                    js = 0;
                    jph ^= 1;
                }
                if (d.kind < 0) break;
                const uint32_t idesc = idesc_f16(128, d.npad);
                const bool fp8 = d.fmt == kFmtFp8B128;
                bool ok = true;
                for (int u = 0; u < d.nunits && ok; ++u) {
                    const bool fresh = fp8 || u == 0;
                    if (fresh && !mbar_wait(&dempty[ds], dph ^ 1, abort_flag, err)) ok = false;
                    if (ok && !mbar_wait(&sfull[as], aph, abort_flag, err)) ok = false;
                    if (!ok) break;
                    fence_proxy_async_smem();  // B arrived through the generic proxy (cp.async)
                    tc_fence_after();
                    const uint32_t a = tmem + as * 128 + tile * 64;
                    const uint32_t dd = tmem + dcol0 + ds * dset + (tile * 2 + kh) * ntmax;
                    const uint32_t bb = smem_u32(bbuf + as * bunit);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int ks = kh * 4 + k;
                        mma_f16_ats(dd, a + ks * 8, smem_desc_noswz(bb + ks * 256, 128, 2048), idesc,
                                    !(fresh && k == 0));
                    }
                    issued = true;
                    mma_commit(&sempty[as]);
                    if (fp8 || u == d.nunits - 1) {
                        mma_commit(&dfull[ds]);
                        if (++ds == 2) {
                            ds = 0;
                            dph ^= 1;
                        }
                    }
                    if (++as == nA) {
                        as = 0;
                        aph ^= 1;
                    }
                }
                if (!ok) break;
            }
            if (issued) {  // all of this thread's MMAs retired before TMEM is released
                mma_commit(&drain[q]);
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_try_wait(&drain[q], 0) && globaltimer_ns() - t0 < kWaitBudgetNs) {
                }
            }
        }
    } else if (warp < 2 + kIssuers + kDqWarps) {
        // ===================== dequant (warps 6 .. 6+kDqWarps-1) =====================
        // warpgroup dq = (warp - 6) / 4: tile = dq & 1, parity = dq >> 1. A
        // warpgroup converts its tile's rows of the units whose running index
        // has its parity; it still steps through every unit and stage so its
        // ring positions stay in step with the others.
        const int dq = (warp - 6) >> 2;
        const int wg = dq & 1, par = dq >> 1;  // par < kDqPar
        const int r = ((warp & 3) << 5) | lane;  // row of the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int js = 0, jph = 0, rs = 0, rph = 0, as = 0, aph = 0, ucount = 0;
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait(&jfull[js], jph, abort_flag, err))) break;
            const TcJob d = job_at(js);
            __syncwarp();
            if (lane == 0) mbar_arrive(&jempty[js]);
            if (++js == kJobSlots) {
                js = 0;
                jph ^= 1;
            }
            if (d.kind < 0) break;
            const bool fp4 = d.fmt == kFmtNvfp4;
            const int upst = fp4 ? 2 : 1;
            const int nst = d.nunits / upst;
            bool ok = true;
            for (int s = 0; s < nst && ok; ++s) {
                // every dequant warp waits for every stage, converting or not, so
                // no warp can arrive on a stage's release twice in one phase
                if (!__all_sync(0xffffffffu, mbar_wait(&rfull[rs], rph, abort_flag, err))) {
                    ok = false;
                    break;
                }
                const uint8_t *row = raw + rs * kRawStageBytes + wg * kRawTileBytes + r * 128;
                const int sw = r & 7;
                // With three or more A slots a warp converts all of its units of
                // the stage, then waits once for its TMEM stores and publishes them
                // together; with two, each unit is published as soon as it is stored
                // (the next unit's slot is the one the MMA is still reading).
                const bool batch = nA >= 3;
                int pend[2], npend = 0;
                for (int uu = 0; uu < upst; ++uu, ++ucount) {
                    const int cur = as;
                    if (++as == nA) {
                        as = 0;
                        aph ^= 1;
                    }
                    if ((ucount % kDqPar) != par) continue;
                    const int cur_ph = (as == 0) ? (aph ^ 1) : aph;  // phase of slot `cur`
                    if (!__all_sync(0xffffffffu, mbar_wait(&sempty[cur], cur_ph ^ 1, abort_flag, err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tcol = tmem + lane_base + cur * 128 + wg * 64;
                    if (fp4) {
                        const uint2 sc = *reinterpret_cast<const uint2 *>(
                            raw + rs * kRawStageBytes + kRawScaleOff + wg * 2048 + r * 16 + uu * 8);
                        const uint32_t scw[2] = {sc.x, sc.y};
                        const uint32_t row_s = sm100::smem_u32(row);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // 16 B = 32 codes = 2 scale blocks
                            const uint32_t ca = row_s + (((uu * 4 + q) ^ sw) << 4);
                            uint32_t hs0, hs1;  // the two block scales as f16, each in both halves
                            e4m3x4_to_half2x2(scw[q >> 1] >> (16 * (q & 1)), hs0, hs1);
                            const __half2 s2 = u32_h2(hs0);
                            const __half2 slo = __low2half2(s2), shi = __high2half2(s2);
                            uint32_t o[16];
#pragma unroll
                            for (int b = 0; b < 16; b += 4) {
                                uint32_t h0, h1, h2, h3;
                                e2m1x8_from_smem(ca + b, h0, h1, h2, h3);
                                const __half2 sb = b < 8 ? slo : shi;
                                o[b] = pack_h2(__hmul2(u32_h2(h0), sb));
                                o[b + 1] = pack_h2(__hmul2(u32_h2(h1), sb));
                                o[b + 2] = pack_h2(__hmul2(u32_h2(h2), sb));
                                o[b + 3] = pack_h2(__hmul2(u32_h2(h3), sb));
                            }
                            tmem_st16(tcol + q * 16, o);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t o[16];
#pragma unroll
                            for (int hq = 0; hq < 2; ++hq) {
                                const uint4 vv = *reinterpret_cast<const uint4 *>(row + (((q * 2 + hq) ^ sw) << 4));
                                e4m3x4_to_half2x2(vv.x, o[hq * 8 + 0], o[hq * 8 + 1]);
                                e4m3x4_to_half2x2(vv.y, o[hq * 8 + 2], o[hq * 8 + 3]);
                                e4m3x4_to_half2x2(vv.z, o[hq * 8 + 4], o[hq * 8 + 5]);
                                e4m3x4_to_half2x2(vv.w, o[hq * 8 + 6], o[hq * 8 + 7]);
                            }
                            tmem_st16(tcol + q * 16, o);
                        }
                    }
                    if (batch) {
                        pend[npend++] = cur;
                    } else {
                        tmem_wait_st();
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sfull[cur]);
                    }
                }
                if (!ok) break;
                // the stage's shared memory has been read (its values are in the
                // TMEM stores' registers): release it before waiting for the stores
                __syncwarp();
                if (lane == 0) mbar_arrive(&rempty[rs]);
                if (++rs == nR) {
                    rs = 0;
                    rph ^= 1;
                }
                if (npend) {
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0)
                        for (int i = 0; i < npend; ++i) mbar_arrive(&sfull[pend[i]]);
                }
            }
            if (!ok) break;
        }
        tmem_wait_st();  // an aborted stage may leave TMEM stores in flight
    } else {
        // ===================== epilogue (the last 4 warps) =====================
        // Each warp owns 32 rows of the tile (its TMEM lane quarter) and runs
        // the reductions for those rows on its own: counters are kept per
        // (tile, quarter), so no warp ever waits for another.
        const int quarter = warp & 3;
        const int r = (quarter << 5) | lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        int js = 0, jph = 0, ds = 0, dph = 0;
        // The combine coefficients of every (row, slot), filled here while
        // the first MMAs are still ahead (the combine waits for coef_bar):
        // weight 1 and the shared down scale for slot 0, the expert's down
        // scale for pick slots (their router weights are in place already).
        {
            const int etid = (warp - 2 - kIssuers - kDqWarps) * 32 + lane;
            for (int i = etid; i < C; i += 128) {
                const int q = i % (K + 1);
                float gsc = 1.0f;
                if (q == 0) {
                    comb_w[i] = 1.0f;
                    if (p.shared.fmt == kFmtNvfp4) gsc = __ldg(p.shared.w2_gscale);
                } else {
                    const int c = rcol[i];
                    if (c >= 0 && p.routed.fmt == kFmtNvfp4)
                        gsc = __ldg(p.routed.w2_gscale + gexp[group_of_col(g0, G, c)]);
                }
                comb_g[i] = gsc;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(coef_bar);
        }
        // the rows' activation scale exponents into shared memory, once every
        // CTA's share of the activations is converted, by the first epilogue
        // warp (idle until the first MMAs complete); xs_s[T] holds 1 when some
        // row is shifted, so launches without shifted rows skip the rescaling
        if (warp == 2 + kIssuers + kDqWarps) {
            int okx = 1;
            if (lane == 0) {
                const unsigned long long t0 = globaltimer_ns();
                while (ld_acquire_gpu(&p.hdr->x_ready[par]) < gridDim.x) {
                    if (*abort_flag || globaltimer_ns() - t0 > kWaitBudgetNs) {
                        if (!*abort_flag) atomicOr(err, kErrWaitTimeout);
                        *abort_flag = 1;
                        okx = 0;
                        break;
                    }
                    __nanosleep(128);
                }
            }
            okx = __shfl_sync(0xffffffffu, okx, 0);
            const int any = okx ? (int)__ldcg(&p.hdr->x_scaled[par]) : 0;
            for (int t = lane; t < T; t += 32) xs_s[t] = any ? __ldcg(p.xs + t) : 0;
            if (lane == 0) xs_s[T] = any ? 1 : 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(xs_bar);
        }
        (void)__all_sync(0xffffffffu, mbar_wait(xs_bar, 0, abort_flag, err));
        const bool xsc = xs_s[T] != 0;  // some activation row is shifted
        // fault injection (MOE_FLAG_DEBUG_DROP_ARRIVE): CTA 0's first quarter
        // skips its first intermediate-ready arrival, so the down jobs of that
        // (group, column tile) wait out their budget and the launch aborts
        bool drop_next = (p.flags & kFlagDebugDropArrive) && blockIdx.x == 0 && quarter == 0;
        constexpr bool fp8mid = kFp8Mid;
        for (;;) {
            if (!__all_sync(0xffffffffu, mbar_wait(&jfull[js], jph, abort_flag, err))) break;
            const TcJob d = job_at(js);
            __syncwarp();
            if (lane == 0) mbar_arrive(&jempty[js]);
            if (++js == kJobSlots) {
                js = 0;
                jph ^= 1;
            }
            if (d.kind < 0) break;
            const bool fp8 = d.fmt == kFmtFp8B128;
            const WeightsDev &W = d.shared ? p.shared : p.routed;
            const int i = d.tile * 128 + r;                      // gate/up: intermediate row
            const int h0 = d.rows0 + r, h1 = d.rows1 + r;        // down: output rows
            const float gs13 = (d.kind == 0 && !fp8) ? __ldg(W.w13_gscale + d.e) : 1.0f;
            uint8_t *mb = p.midB + d.mid_off + (long long)d.tile * d.npad * 256;
            uint32_t range_bad = 0;

            // phase 1, one column at a time (a loop the compiler keeps rolled, so the
            // epilogue's code stays small next to the dequant and MMA loops): the
            // column's (gate, up) or (row h0, row h1) values from the D set -> partial
            // sums, the intermediate, or the down output. With two K-halves per tile
            // (NVFP4) they are added in a fixed order; FP8 jobs leave their promoted
            // sum in K-half 0.
            auto drain = [&](uint32_t dcol, bool halves) {
#pragma unroll 1
                for (int c = 0; c < d.n; ++c) {
                    const uint32_t a0 = tmem_ld1(dcol + c), b0 = tmem_ld1(dcol + 2 * ntmax + c);
                    uint32_t a1 = 0u, b1 = 0u;
                    if (halves) {
                        a1 = tmem_ld1(dcol + ntmax + c);
                        b1 = tmem_ld1(dcol + 3 * ntmax + c);
                    }
                    tmem_wait_ld();
                    const float v0 = halves ? __fadd_rn(__uint_as_float(a0), __uint_as_float(a1)) : __uint_as_float(a0);
                    const float v1 = halves ? __fadd_rn(__uint_as_float(b0), __uint_as_float(b1)) : __uint_as_float(b0);
                    const size_t col = (size_t)(d.col0 + c);
                    if (d.kind == 0) {
                        if (d.nkc > 1) {
                            p.P[(((size_t)d.kc * 2 + 0) * p.Ucap + col) * p.Imax + i] = v0;
                            p.P[(((size_t)d.kc * 2 + 1) * p.Ucap + col) * p.Imax + i] = v1;
                        } else {
                            const int sx = xsc ? xs_s[crow[col]] : 0;
                            const float m = swiglu_scaled(__fmul_rn(v0, gs13), __fmul_rn(v1, gs13), pow2f(sx), pow2f(-sx));
                            const __half hm = __float2half_rn(fp8mid ? fp8_mid_q(m) : m);
                            if (__hisinf(hm) || !(fabsf(m) == fabsf(m))) range_bad = 1;
                            *reinterpret_cast<__half *>(mb + b_off(c, r)) = hm;
                        }
                    } else {
                        float *y = p.Y + ((size_t)d.kc * p.Ucap + col) * H;
                        if (h0 < H) y[h0] = v0;
                        if (h1 < H) y[h1] = v1;
                    }
                }
            };

            bool ok = true;
            if (fp8) {
                // per 128-K unit: fresh accumulators, fp32 block scale, running sum
                float acc0[16], acc1[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) acc0[j] = acc1[j] = 0.0f;
                const float *sc = reinterpret_cast<const float *>(d.kind == 0 ? W.w13_scale : W.w2_scale);
                const int rows = d.kind == 0 ? 2 * d.Ig : H;
                const int cols_blk = (d.kind == 0 ? H : d.Ig) / 128;
                const size_t sbase = (size_t)d.e * (rows / 128);
                // the two tiles' block scales of a unit, loaded one unit ahead so
                // the load is off the path from the unit's MMAs to the D release
                const float *sc0 = sc + (sbase + d.rows0 / 128) * cols_blk + d.k0 / kUnitK;
                const float *sc1 = sc + (sbase + d.rows1 / 128) * cols_blk + d.k0 / kUnitK;
                const bool has1 = d.rows1 < rows;
                float s0n = __ldg(sc0), s1n = has1 ? __ldg(sc1) : 0.0f;
                for (int u = 0; u < d.nunits; ++u) {
                    const float s0 = s0n, s1 = s1n;
                    if (u + 1 < d.nunits) {
                        s0n = __ldg(sc0 + u + 1);
                        s1n = has1 ? __ldg(sc1 + u + 1) : 0.0f;
                    }
                    if (!__all_sync(0xffffffffu, mbar_wait(&dfull[ds], dph, abort_flag, err))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t dcol = tmem + lane_base + dcol0 + ds * dset;
#pragma unroll
                    for (int h8 = 0; h8 < 16; h8 += 8) {
                        if (h8 >= d.n) break;  // columns past the job's last one stay 0
                        uint32_t x0[8], x1[8];
                        tmem_ld8(dcol + h8, x0);
                        tmem_ld8(dcol + ntmax + h8, x1);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            acc0[h8 + j] = __fmaf_rn(s0, __fadd_rn(__uint_as_float(x0[j]), __uint_as_float(x1[j])), acc0[h8 + j]);
                        tmem_ld8(dcol + 2 * ntmax + h8, x0);
                        tmem_ld8(dcol + 3 * ntmax + h8, x1);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            acc1[h8 + j] = __fmaf_rn(s1, __fadd_rn(__uint_as_float(x0[j]), __uint_as_float(x1[j])), acc1[h8 + j]);
                    }
                    if (u == d.nunits - 1) {
                        // the promoted sums go back to K-half 0 of this D set and are
                        // drained from there before the set is released
                        uint32_t o0[16], o1[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            o0[j] = __float_as_uint(acc0[j]);
                            o1[j] = __float_as_uint(acc1[j]);
                        }
                        tmem_st16(dcol, o0);
                        tmem_st16(dcol + 2 * ntmax, o1);
                        tmem_wait_st();
                        drain(dcol, false);
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&dempty[ds]);
                    if (++ds == 2) {
                        ds = 0;
                        dph ^= 1;
                    }
                }
                if (!ok) break;
            } else {
                if (!__all_sync(0xffffffffu, mbar_wait(&dfull[ds], dph, abort_flag, err))) break;
                tc_fence_after();
                drain(tmem + lane_base + dcol0 + ds * dset, true);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[ds]);
                if (++ds == 2) {
                    ds = 0;
                    dph ^= 1;
                }
            }

            if (d.kind == 0) {
                // ---- gate/up phase 2: the last K chunk reduces in kc order, SwiGLU ----
                bool have_mid = d.nkc == 1;
                if (d.nkc > 1) {
                    __threadfence();
                    __syncwarp();
                    int l = 0;
                    if (lane == 0)
                        l = atom_add_acq_rel_gpu(p.tile_cnt + (size_t)d.tile_id * 4 + quarter, 1u) ==
                            (uint32_t)d.nkc - 1;
                    if (__shfl_sync(0xffffffffu, l, 0)) {
                        __threadfence();
                        for (int c = 0; c < d.n; ++c) {
                            const size_t col = (size_t)(d.col0 + c);
                            float sg = __ldcg(p.P + ((size_t)0 * p.Ucap + col) * p.Imax + i);
                            float su = __ldcg(p.P + ((size_t)1 * p.Ucap + col) * p.Imax + i);
                            for (int kc = 1; kc < d.nkc; ++kc) {
                                sg = __fadd_rn(sg, __ldcg(p.P + (((size_t)kc * 2 + 0) * p.Ucap + col) * p.Imax + i));
                                su = __fadd_rn(su, __ldcg(p.P + (((size_t)kc * 2 + 1) * p.Ucap + col) * p.Imax + i));
                            }
                            const int sx = xsc ? xs_s[crow[col]] : 0;
                            const float m = swiglu_scaled(__fmul_rn(sg, gs13), __fmul_rn(su, gs13), pow2f(sx), pow2f(-sx));
                            const __half hm = __float2half_rn(fp8mid ? fp8_mid_q(m) : m);
                            if (__hisinf(hm) || !(fabsf(m) == fabsf(m))) range_bad = 1;
                            *reinterpret_cast<__half *>(mb + b_off(c, r)) = hm;
                        }
                        if (lane == 0) p.tile_cnt[(size_t)d.tile_id * 4 + quarter] = 0;
                        have_mid = true;
                    }
                }
                if (range_bad) atomicOr(err, kErrRange);
                if (have_mid) {
                    __threadfence();
                    __syncwarp();
                    if (lane == 0 && !drop_next) atom_add_acq_rel_gpu(group_ready + d.pair, 1u);
                    drop_next = false;
                }
            } else {
                // ---- down phase 2: count this (job, quarter) on its 256-row tile;
                // the tile is combined once every down job has arrived ----
                __threadfence();
                __syncwarp();
                if (lane == 0) atom_add_acq_rel_gpu(htile_cnt + d.tile, 1u);
            }
        }
    }

    // A warp whose role's loop ran on lane 0 alone reconverges here.
    __syncwarp();

    // ---- combine: every warp of the grid shares the output ------------------
    // A 256-row output tile is complete once all 4 * (down jobs per tile) (down job,
    // quarter) arrivals are in. Warp 0 (the producer, which finishes first)
    // watches every tile's counter with one load per lane per round and marks
    // the complete ones in shared memory; the other warps start on the combine
    // as soon as their role is done and wait on those marks, so the counters,
    // which the epilogues are still incrementing, see one reader per CTA.
    // A warp unit is 32 consecutive outputs of one row; units are dealt
    // round-robin over the CTAs first and then over warps 1.. of a CTA in role
    // order, so the warps that finish first take them first. Each lane sums its
    // output in the fixed order x + y_shared*gs + sum over picks of w*(y*gs),
    // each y the sum of its K-chunk partials in chunk order. The partials are
    // loaded kCombBatch at a time with no dependence between them, so a unit
    // costs about one memory round trip.
    const uint32_t tile_target = 4u * (uint32_t)*dn_per_ht_s;
    if (warp == 0) {
        const int nht = H / 256;  // <= 64
        uint32_t pending = (lane < nht ? 1u : 0u) | (lane + 32 < nht ? 2u : 0u);
        const unsigned long long t0 = globaltimer_ns();
        // one memory round trip per round: the error word (another CTA gave up)
        // and the clock are looked at every 8th round only
        for (unsigned round = 1; !*abort_flag; ++round) {
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if ((pending >> k) & 1u) {
                    const int ht = lane + 32 * k;
                    if (ld_acquire_gpu(htile_cnt + ht) >= tile_target) {
                        st_release_cta_shared(tile_ready_s + ht, 1u);
                        pending &= ~(1u << k);
                    }
                }
            if (!__any_sync(0xffffffffu, pending != 0u)) break;
            if ((round & 7u) == 0u && ((*reinterpret_cast<volatile uint32_t *>(err) & kErrWaitTimeout) ||
                                       globaltimer_ns() - t0 > kWaitBudgetNs)) {
                if (lane == 0) {
                    atomicOr(err, kErrWaitTimeout);
                    *abort_flag = 1;
                }
                break;
            }
            __nanosleep(128);
        }
        __syncwarp();
    } else if (!*abort_flag && __all_sync(0xffffffffu, mbar_wait(coef_bar, 0, abort_flag, err)) &&
               __all_sync(0xffffffffu, mbar_wait(xs_bar, 0, abort_flag, err))) {
        const int ncw = kTcThreads / 32 - 1, hw = H / 32;  // combine warps 1..
        const long long nwu = (long long)T * hw;
        const int nkc_s = tc_nkc_dn(p.Is, T), nkc_r = tc_nkc_dn(p.I, T);
        const int nterm = nkc_s + K * nkc_r;
        for (long long wu = (long long)(warp - 1) * gridDim.x + blockIdx.x; wu < nwu;
             wu += (long long)gridDim.x * ncw) {
            const int t = (int)(wu / hw), h = (int)(wu % hw) * 32 + lane, ht = h >> 8;
            float acc = __bfloat162float(p.x[(size_t)t * H + h]);  // the residual, before the wait
            if (!ld_acquire_cta_shared(tile_ready_s + ht)) {
                const unsigned long long t0 = globaltimer_ns();
                bool ready = false;
                while (!(ready = ld_acquire_cta_shared(tile_ready_s + ht) != 0u)) {
                    if (*abort_flag || globaltimer_ns() - t0 > kWaitBudgetNs) break;
                    __nanosleep(64);
                }
                if (!__all_sync(0xffffffffu, ready)) {
                    atomicOr(err, kErrWaitTimeout);
                    break;
                }
            }
            const int32_t *rc = rcol + t * (K + 1);
            const float *cw = comb_w + t * (K + 1), *cg = comb_g + t * (K + 1);
            const float fx = pow2f(2 * xs_s[t]);  // undoes the row's activation scale, squared (1 unless shifted)
            float y = 0.0f;
            int lq = 0, lk = 0;  // (slot, chunk) of the next term to load
            int aq = 0, ak = 0;  // ... and to add
            for (int b0 = 0; b0 < nterm; b0 += kCombBatch) {
                float v[kCombBatch];
#pragma unroll
                for (int u = 0; u < kCombBatch; ++u) {
                    v[u] = 0.0f;
                    if (b0 + u < nterm) {
                        const int c = rc[lq];
                        if (c >= 0) v[u] = __ldcg(p.Y + ((size_t)lk * p.Ucap + c) * H + h);
                        if (++lk == (lq == 0 ? nkc_s : nkc_r)) {
                            lk = 0;
                            ++lq;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kCombBatch; ++u) {
                    if (b0 + u < nterm) {
                        const int nk = aq == 0 ? nkc_s : nkc_r;
                        y = ak == 0 ? v[u] : __fadd_rn(y, v[u]);
                        if (ak == nk - 1) {
                            if (rc[aq] >= 0) acc = __fmaf_rn(cw[aq], __fmul_rn(__fmul_rn(y, cg[aq]), fx), acc);
                            ak = 0;
                            ++aq;
                        } else {
                            ++ak;
                        }
                    }
                }
            }
            p.out[(size_t)t * H + h] = __float2bfloat16_rn(acc);
        }
    }
    __syncwarp();

    // ---- teardown -----------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace moe
