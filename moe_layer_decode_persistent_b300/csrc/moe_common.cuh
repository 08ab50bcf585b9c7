// moe_common.cuh -- device-side definitions shared by the kernels of libmoe.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

// device error word bits (same values as MOE_DEV_* in include/moe.h)
constexpr uint32_t kErrBadExpert = 1u;
constexpr uint32_t kErrDupExpert = 2u;
constexpr uint32_t kErrWaitTimeout = 4u;
constexpr uint32_t kErrRange = 8u;

// shape flags (MOE_FLAG_* in include/moe.h)
constexpr unsigned kFlagNoDedup = 1u;
constexpr unsigned kFlagForceFma = 2u;
constexpr unsigned kFlagForceMma = 4u;
constexpr unsigned kFlagDebugDropArrive = 8u;

// weight formats (moe_wfmt)
constexpr int kFmtBf16 = 0;
constexpr int kFmtNvfp4 = 1;
constexpr int kFmtFp8B128 = 2;

// An inter-CTA wait gives up after this long (ns of %globaltimer). Normal
// waits in a launch last microseconds; this only bounds a broken launch.
constexpr unsigned long long kWaitBudgetNs = 400ull * 1000ull * 1000ull;

struct WeightsDev {
    int fmt;
    const uint8_t *w13;
    const uint8_t *w13_scale;
    const float *w13_gscale;
    const uint8_t *w2;
    const uint8_t *w2_scale;
    const float *w2_gscale;
};

// Workspace header, at the start of the caller's workspace (256 B).
// The tensor-core path keeps two sets of its launch-wide counters and uses
// them in alternate launches: a launch finds its own set zeroed by the launch
// before it and zeroes the other set, so no CTA has to reset anything at exit.
struct WsHeader {
    uint32_t err;          // device error word (MOE_DEV_* bits)
    uint32_t bar_count;    // grid barrier: arrivals in the current round
    uint32_t bar_gen;      // grid barrier: completed rounds (monotonic)
    uint32_t spare;        // unused
    uint32_t job_next[2];  // tensor-core path, per parity: jobs claimed past the first round
    uint32_t x_ready[2];   // tensor-core path, per parity: CTAs done converting their activation slice
    uint32_t route_ready[2];  // tensor-core path, per parity: CTAs done with their router partial logits
    uint32_t x_scaled[2];  // tensor-core path, per parity: nonzero when some activation row is shifted
    uint32_t pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header size");

// ---- small PTX helpers --------------------------------------------------

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_release_cta_shared(uint32_t *p, uint32_t v) {
    asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"((uint32_t)__cvta_generic_to_shared(p)), "r"(v)
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta_shared(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];"
                 : "=r"(v)
                 : "r"((uint32_t)__cvta_generic_to_shared(p))
                 : "memory");
    return v;
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16 bytes of streamed (read-once) weights: skip L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Two E2M1 codes (one byte, low nibble first) -> two exact halves.
__device__ __forceinline__ __half2 e2m1x2_to_half2(uint32_t byte) {
    uint32_t h;
    asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(h) : "r"(byte));
    return *reinterpret_cast<__half2 *>(&h);
}

// Two E4M3 bytes (low byte first) -> two exact halves.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t two_bytes) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)two_bytes));
    return *reinterpret_cast<__half2 *>(&h);
}

// Eight E2M1 codes at shared address `saddr` (4 bytes, low nibble first in
// each byte) -> four f16x2 words. The bytes are loaded straight into 8-bit
// registers, which feeds the conversion far more cheaply than extracting them
// from a 32-bit word.
__device__ __forceinline__ void e2m1x8_from_smem(uint32_t saddr, uint32_t &h0, uint32_t &h1, uint32_t &h2,
                                                 uint32_t &h3) {
    asm volatile(
        "{ .reg .b8 t0, t1, t2, t3;\n"
        " ld.shared.v4.b8 {t0, t1, t2, t3}, [%4];\n"
        " cvt.rn.f16x2.e2m1x2 %0, t0; cvt.rn.f16x2.e2m1x2 %1, t1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, t2; cvt.rn.f16x2.e2m1x2 %3, t3; }"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(saddr)
        : "memory");
}

// Four E4M3 bytes (a 32-bit word, low byte first) -> two f16x2 words; the
// 16-bit halves of the register are used as they are.
__device__ __forceinline__ void e4m3x4_to_half2x2(uint32_t w, uint32_t &h0, uint32_t &h1) {
    asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2; cvt.rn.f16x2.e4m3x2 %0, lo; cvt.rn.f16x2.e4m3x2 %1, hi; }"
        : "=r"(h0), "=r"(h1)
        : "r"(w));
}

__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
    return __low2float(e4m3x2_to_half2(byte & 0xffu));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
    return __uint_as_float(bits16 << 16);
}

__device__ __forceinline__ float silu_f32(float v) { return v / (1.0f + expf(-v)); }

// ---- grid barrier --------------------------------------------------------
// Sense by generation: the last arriver resets the count and bumps bar_gen.
// Every CTA of the (cooperative) grid must call it the same number of times.
// Returns false if the wait ran out of budget (error bit set; caller exits).
__device__ __forceinline__ bool grid_barrier(WsHeader *hdr, unsigned nblocks, bool skip_arrive) {
    __shared__ uint32_t s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t ok = 1;
        uint32_t gen = ld_acquire_gpu(&hdr->bar_gen);
        if (!skip_arrive) {
            __threadfence();
            uint32_t arrived = atom_add_acq_rel_gpu(&hdr->bar_count, 1u) + 1u;
            if (arrived == nblocks) {
                hdr->bar_count = 0;
                __threadfence();
                st_release_gpu(&hdr->bar_gen, gen + 1u);
            }
        }
        if (ld_acquire_gpu(&hdr->bar_gen) == gen) {
            unsigned long long t0 = globaltimer_ns();
            while (ld_acquire_gpu(&hdr->bar_gen) == gen) {
                __nanosleep(64);
                if (globaltimer_ns() - t0 > kWaitBudgetNs) {
                    atomicOr(&hdr->err, kErrWaitTimeout);
                    ok = 0;
                    break;
                }
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

}  // namespace moe
