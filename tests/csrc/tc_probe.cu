// tc_probe.cu -- test-only kernels that check the Blackwell building blocks the
// fused kernel relies on, one at a time, on a single CTA: the TMEM layout of a
// tcgen05.mma A operand, the shared-memory descriptor of the B operand, the
// instruction descriptor, mbarrier commit, and TMA swizzled tiles. Every wait
// is bounded. Built by tests/test_tcgen05_probe_gpu.py into tests/csrc/.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>

#include "../../moe_layer_decode_persistent_b300/csrc/sm100.cuh"

using namespace moe;
using namespace moe::sm100;

// B (or A) tile [rows][K] f16 in the no-swizzle K-major core-matrix layout:
// element (r, k) at ((r/8)*(K/8) + k/8)*128 + (r%8)*16 + (k%8)*2 bytes.
__device__ __forceinline__ uint32_t cm_off(int r, int k, int K) {
    return (uint32_t)(((r >> 3) * (K >> 3) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// D[128][N] = A[128][K] * B[N][K]^T with K in {16, 32, 64}, N in {16, 32, 64}.
__global__ void __launch_bounds__(128) probe_mma_kernel(const uint16_t *A, const uint16_t *B, int K,
                                                        int N, int a_in_tmem, float *D, uint32_t *err) {
    __shared__ __align__(1024) uint8_t sB[64 * 64 * 2];
    __shared__ __align__(1024) uint8_t sA[128 * 64 * 2];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t taddr_s;
    __shared__ int abort_flag;
    const int t = threadIdx.x, w = t >> 5;
    if (w == 0) tmem_alloc(&taddr_s, 256);
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    // B and (optionally) A into shared memory, core-matrix layout
    for (int i = t; i < N * K; i += 128) {
        const int n = i / K, k = i % K;
        *reinterpret_cast<uint16_t *>(sB + cm_off(n, k, K)) = B[i];
    }
    if (!a_in_tmem)
        for (int i = t; i < 128 * K; i += 128) {
            const int m = i / K, k = i % K;
            *reinterpret_cast<uint16_t *>(sA + cm_off(m, k, K)) = A[i];
        }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = taddr_s;
    const uint32_t d_col = 128;
    if (a_in_tmem) {
        // thread t owns row t = lane t; columns hold consecutive k pairs
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t r[16];
            for (int j = 0; j < 16; ++j) {
                const int c = c0 + j;
                r[j] = (c < K / 2) ? ((uint32_t)A[t * K + 2 * c] | ((uint32_t)A[t * K + 2 * c + 1] << 16)) : 0u;
            }
            tmem_st16(tmem_addr(taddr, 32 * w, c0), r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    if (t == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_f16(128, N);
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t bd = smem_desc_noswz(smem_u32(sB) + ks * 256, 128, (K / 8) * 128);
            if (a_in_tmem) {
                mma_f16_ats(taddr + d_col, taddr + ks * 8, bd, idesc, ks > 0);
            } else {
                const uint64_t ad = smem_desc_noswz(smem_u32(sA) + ks * 256, 128, (K / 8) * 128);
                mma_f16_ss(taddr + d_col, ad, bd, idesc, ks > 0);
            }
        }
        mma_commit(&bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&bar, 0, &abort_flag, err);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tmem_addr(taddr, 32 * w, d_col + c0), r);
            tmem_wait_ld();
            for (int j = 0; j < 16; ++j) D[t * N + c0 + j] = __uint_as_float(r[j]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0) tmem_dealloc(taddr, 256);
}

// TMEM round trip: every thread stores then loads 32 columns of its lane.
__global__ void __launch_bounds__(128) probe_tmem_kernel(uint32_t *out) {
    __shared__ uint32_t taddr_s;
    const int t = threadIdx.x, w = t >> 5;
    if (w == 0) tmem_alloc(&taddr_s, 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = taddr_s;
    for (int c0 = 0; c0 < 32; c0 += 16) {
        uint32_t r[16];
        for (int j = 0; j < 16; ++j) r[j] = (uint32_t)(t * 1000 + c0 + j);
        tmem_st16(tmem_addr(taddr, 32 * w, c0), r);
    }
    tmem_wait_st();
    for (int c0 = 0; c0 < 32; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_addr(taddr, 32 * w, c0), r);
        tmem_wait_ld();
        for (int j = 0; j < 16; ++j) out[t * 32 + c0 + j] = r[j];
    }
    tc_fence_before();
    __syncthreads();
    if (w == 0) tmem_dealloc(taddr, 32);
}

// One TMA 3-D box [box_c bytes][128 rows][1] into shared memory, copied out raw.
__global__ void __launch_bounds__(128) probe_tma_kernel(const __grid_constant__ CUtensorMap tm, int c0,
                                                        int c1, int c2, int box_bytes, uint8_t *out,
                                                        uint32_t *err) {
    __shared__ __align__(1024) uint8_t buf[128 * 128];
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int t = threadIdx.x;
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (t == 0) {
        mbar_arrive_expect_tx(&bar, (uint32_t)box_bytes);
        tma_load_3d(buf, &tm, c0, c1, c2, &bar);
    }
    const bool ok = mbar_wait(&bar, 0, &abort_flag, err);
    __syncthreads();
    if (ok)
        for (int i = t; i < box_bytes; i += 128) out[i] = buf[i];
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

extern "C" {

int probe_tmem(uint32_t *host_out) {
    uint32_t *d = nullptr;
    if (cudaMalloc(&d, 128 * 32 * 4) != cudaSuccess) return -1;
    probe_tmem_kernel<<<1, 128>>>(d);
    int rc = (int)cudaDeviceSynchronize();
    if (!rc) rc = (int)cudaMemcpy(host_out, d, 128 * 32 * 4, cudaMemcpyDeviceToHost);
    cudaFree(d);
    return rc;
}

int probe_mma(const uint16_t *hA, const uint16_t *hB, int K, int N, int a_in_tmem, float *hD,
              uint32_t *herr) {
    uint16_t *dA = nullptr, *dB = nullptr;
    float *dD = nullptr;
    uint32_t *derr = nullptr;
    cudaMalloc(&dA, 128 * K * 2);
    cudaMalloc(&dB, N * K * 2);
    cudaMalloc(&dD, 128 * N * 4);
    cudaMalloc(&derr, 4);
    cudaMemcpy(dA, hA, 128 * K * 2, cudaMemcpyHostToDevice);
    cudaMemcpy(dB, hB, N * K * 2, cudaMemcpyHostToDevice);
    cudaMemset(dD, 0xff, 128 * N * 4);
    cudaMemset(derr, 0, 4);
    probe_mma_kernel<<<1, 128>>>(dA, dB, K, N, a_in_tmem, dD, derr);
    int rc = (int)cudaDeviceSynchronize();
    if (!rc) {
        cudaMemcpy(hD, dD, 128 * N * 4, cudaMemcpyDeviceToHost);
        cudaMemcpy(herr, derr, 4, cudaMemcpyDeviceToHost);
    }
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dD);
    cudaFree(derr);
    return rc;
}

// src [E][R][Cb] uint8; box [box_c][128][1] at (c0, c1, c2); swz in {0, 64, 128}
int probe_tma(const uint8_t *hsrc, int E, int R, int Cb, int box_c, int swz, int c0, int c1, int c2,
              uint8_t *hout, uint32_t *herr) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return -2;
    uint8_t *dsrc = nullptr, *dout = nullptr;
    uint32_t *derr = nullptr;
    const size_t n = (size_t)E * R * Cb;
    cudaMalloc(&dsrc, n);
    cudaMalloc(&dout, box_c * 128);
    cudaMalloc(&derr, 4);
    cudaMemcpy(dsrc, hsrc, n, cudaMemcpyHostToDevice);
    cudaMemset(dout, 0, box_c * 128);
    cudaMemset(derr, 0, 4);
    CUtensorMap tm;
    cuuint64_t dims[3] = {(cuuint64_t)Cb, (cuuint64_t)R, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)Cb, (cuuint64_t)R * Cb};
    cuuint32_t box[3] = {(cuuint32_t)box_c, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUtensorMapSwizzle sw = swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                            : swz == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    CUresult cr = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dsrc, dims, strides, box, es,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    int rc = (int)cr ? 1000 + (int)cr : 0;
    if (!rc) {
        probe_tma_kernel<<<1, 128>>>(tm, c0, c1, c2, box_c * 128, dout, derr);
        rc = (int)cudaDeviceSynchronize();
    }
    if (!rc) {
        cudaMemcpy(hout, dout, box_c * 128, cudaMemcpyDeviceToHost);
        cudaMemcpy(herr, derr, 4, cudaMemcpyDeviceToHost);
    }
    cudaFree(dsrc);
    cudaFree(dout);
    cudaFree(derr);
    return rc;
}

}  // extern "C"
