// api.cu -- the C ABI of libmoe (declared in include/moe.h): argument
// validation, workspace layout, launch configuration and error reporting.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "../../include/moe.h"
#include "fused_fma.cuh"

namespace {

thread_local std::string g_detail;

moe_status fail(moe_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_detail = buf;
    return s;
}

moe_status cuda_fail(cudaError_t e, const char *what) {
    return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxT = 256, kMaxK = 16, kMaxE = 1024, kMaxDim = 16384;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace: header | mid fp32 [Ucap][Imax] | y fp32 [Ucap][H] | host staging.
struct WsLayout {
    size_t mid = 0, y = 0, dev_total = 0;
    size_t st_x = 0, st_ids = 0, st_w = 0, st_out = 0, host_total = 0;
};

WsLayout ws_layout(const moe_shape *s) {
    WsLayout L;
    const size_t T = (size_t)std::max(s->T, 0), K = (size_t)std::max(s->K, 0);
    const size_t Ucap = T * (K + 1);
    const size_t Imax = (size_t)std::max(s->I, s->I_shared);
    size_t off = sizeof(moe::WsHeader);
    L.mid = off = align_up(off, 256);
    off += Ucap * Imax * sizeof(float);
    L.y = off = align_up(off, 256);
    off += Ucap * (size_t)s->H * sizeof(float);
    L.dev_total = off = align_up(off, 256);
    L.st_x = off;
    off = align_up(off + T * (size_t)s->H * 2, 256);
    L.st_ids = off;
    off = align_up(off + T * K * 4, 256);
    L.st_w = off;
    off = align_up(off + T * K * 4, 256);
    L.st_out = off;
    off = align_up(off + T * (size_t)s->H * 2, 256);
    L.host_total = off;
    return L;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

moe_status check_shape(const moe_shape *s) {
    if (!s) return fail(MOE_ERR_INVALID_ARG, "shape is NULL");
    if (s->T < 0 || s->T > kMaxT) return fail(MOE_ERR_INVALID_ARG, "T=%d outside [0, %d]", s->T, kMaxT);
    if (s->K < 1 || s->K > kMaxK) return fail(MOE_ERR_INVALID_ARG, "K=%d outside [1, %d]", s->K, kMaxK);
    if (s->E < 1 || s->E > kMaxE) return fail(MOE_ERR_INVALID_ARG, "E=%d outside [1, %d]", s->E, kMaxE);
    if (s->K > s->E) return fail(MOE_ERR_INVALID_ARG, "K=%d > E=%d", s->K, s->E);
    const int dims[3] = {s->H, s->I, s->I_shared};
    const char *names[3] = {"H", "I", "I_shared"};
    for (int i = 0; i < 3; ++i) {
        if (dims[i] < 128 || dims[i] > kMaxDim)
            return fail(MOE_ERR_INVALID_ARG, "%s=%d outside [128, %d]", names[i], dims[i], kMaxDim);
        if (dims[i] % 128)
            return fail(MOE_ERR_UNSUPPORTED, "%s=%d is not a multiple of 128", names[i], dims[i]);
    }
    const unsigned known = MOE_FLAG_NO_DEDUP | MOE_FLAG_FORCE_FMA | MOE_FLAG_FORCE_MMA |
                           MOE_FLAG_DEBUG_DROP_ARRIVE;
    if (s->flags & ~known) return fail(MOE_ERR_INVALID_ARG, "unknown flag bits 0x%x", s->flags & ~known);
    if ((s->flags & MOE_FLAG_FORCE_FMA) && (s->flags & MOE_FLAG_FORCE_MMA))
        return fail(MOE_ERR_INVALID_ARG, "FORCE_FMA and FORCE_MMA both set");
    return MOE_OK;
}

moe_status check_weights(const moe_weights *w, const char *which) {
    if (!w) return fail(MOE_ERR_INVALID_ARG, "%s weights struct is NULL", which);
    if (w->fmt != MOE_W_BF16 && w->fmt != MOE_W_NVFP4 && w->fmt != MOE_W_FP8_B128)
        return fail(MOE_ERR_INVALID_ARG, "%s weights: unknown format %d", which, w->fmt);
    const void *need[4] = {w->w13, w->w2, nullptr, nullptr};
    int n = 2;
    if (w->fmt != MOE_W_BF16) {
        need[2] = w->w13_scale;
        need[3] = w->w2_scale;
        n = 4;
    }
    for (int i = 0; i < n; ++i) {
        if (!need[i]) return fail(MOE_ERR_INVALID_ARG, "%s weights: NULL pointer", which);
        if (!aligned(need[i], 16))
            return fail(MOE_ERR_INVALID_ARG, "%s weights: pointer not 16-byte aligned", which);
    }
    if (w->fmt == MOE_W_NVFP4 && (!w->w13_gscale || !w->w2_gscale))
        return fail(MOE_ERR_INVALID_ARG, "%s weights: NVFP4 needs both tensor scales", which);
    return MOE_OK;
}

moe::WeightsDev to_dev(const moe_weights *w) {
    moe::WeightsDev d;
    d.fmt = w->fmt;
    d.w13 = static_cast<const uint8_t *>(w->w13);
    d.w13_scale = static_cast<const uint8_t *>(w->w13_scale);
    d.w13_gscale = w->w13_gscale;
    d.w2 = static_cast<const uint8_t *>(w->w2);
    d.w2_scale = static_cast<const uint8_t *>(w->w2_scale);
    d.w2_gscale = w->w2_gscale;
    return d;
}

size_t table_smem_bytes(const moe_shape *s) {
    return sizeof(int32_t) * (size_t)(moe::group_table_ints(s->T, s->K) + moe::group_table_scratch_ints(s->E));
}

struct DevInfo {
    int nsm = 0;
    int max_smem_optin = 0;
};

std::mutex g_mu;
std::unordered_map<int, DevInfo> g_dev;

moe_status dev_info(DevInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it == g_dev.end()) {
        DevInfo d;
        e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
        it = g_dev.emplace(dev, d).first;
    }
    *out = it->second;
    return MOE_OK;
}

template <typename Kern>
moe_status set_smem(Kern k, size_t smem, const DevInfo &d) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, k);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
    const size_t limit = (size_t)d.max_smem_optin - fa.sharedSizeBytes;
    if (smem > limit)
        return fail(MOE_ERR_UNSUPPORTED, "needs %zu B dynamic shared memory, the device allows %zu",
                    smem, limit);
    // always the largest allowed size, so an attribute set for one launch
    // never undercuts a later, larger launch of the same kernel
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
    return MOE_OK;
}

// Blocks per SM of a kernel at a dynamic smem size, with the smem attribute
// set; cached per (device, kernel, smem) so a launch inside stream capture
// makes no other CUDA call.
template <typename Kern>
moe_status plan_occupancy(Kern k, int threads, size_t smem, const DevInfo &d, int *occ_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    static std::mutex mu;
    static std::unordered_map<std::string, int> cache;
    char key[128];
    snprintf(key, sizeof key, "%d/%p/%d/%zu", dev, (const void *)k, threads, smem);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *occ_out = it->second;
            return MOE_OK;
        }
    }
    moe_status st = set_smem(k, smem, d);
    if (st != MOE_OK) return st;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1) return fail(MOE_ERR_UNSUPPORTED, "kernel does not fit on an SM (%zu B smem)", smem);
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = occ;
    *occ_out = occ;
    return MOE_OK;
}

moe_status launch_fused_fma(const moe::FusedParams &p, const moe_shape *s, cudaStream_t stream) {
    DevInfo d;
    moe_status st = dev_info(&d);
    if (st != MOE_OK) return st;
    const size_t smem = table_smem_bytes(s);
    int occ = 0;
    st = plan_occupancy(moe::fused_fma_kernel, moe::kFmaThreads, smem, d, &occ);
    if (st != MOE_OK) return st;
    cudaError_t e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(d.nsm * occ));
    cfg.blockDim = dim3(moe::kFmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, moe::fused_fma_kernel, p);
    if (e != cudaSuccess) return cuda_fail(e, "launch fused_fma_kernel");
    return MOE_OK;
}

moe_status fused_decode_impl(const void *x, const int32_t *ids, const float *w,
                             const moe_weights *routed, const moe_weights *shared, void *out,
                             const moe_shape *s, void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    if ((st = check_weights(routed, "routed")) != MOE_OK) return st;
    if ((st = check_weights(shared, "shared")) != MOE_OK) return st;
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    const WsLayout L = ws_layout(s);
    if (ws_bytes < L.dev_total)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu B, needs %zu B", ws_bytes, L.dev_total);
    if (s->T == 0) return MOE_OK;
    if (!x || !out || !ids || !w) return fail(MOE_ERR_INVALID_ARG, "NULL x/out/topk_ids/topk_w");
    if (!aligned(x, 16) || !aligned(out, 16))
        return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (!aligned(ids, 4) || !aligned(w, 4))
        return fail(MOE_ERR_INVALID_ARG, "topk_ids and topk_w must be 4-byte aligned");
    const size_t act_bytes = (size_t)s->T * s->H * 2;
    const uintptr_t xa = (uintptr_t)x, oa = (uintptr_t)out;
    if (xa < oa + act_bytes && oa < xa + act_bytes)
        return fail(MOE_ERR_INVALID_ARG, "out overlaps x");

    moe::FusedParams p;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.ids = ids;
    p.topk_w = w;
    p.routed = to_dev(routed);
    p.shared = to_dev(shared);
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.T = s->T;
    p.H = s->H;
    p.I = s->I;
    p.Is = s->I_shared;
    p.E = s->E;
    p.K = s->K;
    p.flags = s->flags;
    p.hdr = static_cast<moe::WsHeader *>(ws);
    p.mid = reinterpret_cast<float *>(static_cast<char *>(ws) + L.mid);
    p.y = reinterpret_cast<float *>(static_cast<char *>(ws) + L.y);
    p.Imax = std::max(s->I, s->I_shared);
    return launch_fused_fma(p, s, stream);
}

}  // namespace

// ---- entry point for callers that cannot allocate device memory ----------
// Its scratch is this file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds it until the process exits. Device
// code could name it directly; host code only ever passes the address that
// cudaGetSymbolAddress returns for the current device (the array's name in
// host code is a host-side stand-in, not a device address).
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device; looked up once
// per device, with that device current, on its first call.
moe_status noalloc_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices)
        return fail(MOE_ERR_UNSUPPORTED, "device %d: the no-allocation entry handles devices 0..%d",
                    dev, kNoAllocMaxDevices - 1);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return ws_layout(s).dev_total;
}

size_t moe_workspace_bytes_host(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return ws_layout(s).host_total;
}

size_t moe_group_table_ints(int T, int K) {
    if (T < 0 || K < 1) return 0;
    return (size_t)moe::group_table_ints(T, K);
}

moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (workspace_bytes < sizeof(moe::WsHeader))
        return fail(MOE_ERR_WORKSPACE, "workspace smaller than its %zu-byte header", sizeof(moe::WsHeader));
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(moe::WsHeader), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    return MOE_OK;
}

moe_status moe_group_table(const int32_t *topk_ids, const moe_shape *s, int32_t *table_out,
                           void *workspace, size_t workspace_bytes, void *stream) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    if (!table_out) return fail(MOE_ERR_INVALID_ARG, "table_out is NULL");
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (workspace_bytes < sizeof(moe::WsHeader))
        return fail(MOE_ERR_WORKSPACE, "workspace smaller than its header");
    if (s->T > 0 && !topk_ids) return fail(MOE_ERR_INVALID_ARG, "topk_ids is NULL");
    DevInfo d;
    if ((st = dev_info(&d)) != MOE_OK) return st;
    const size_t smem = table_smem_bytes(s);
    if ((st = set_smem(moe::group_table_kernel, smem, d)) != MOE_OK) return st;
    moe::group_table_kernel<<<1, 256, smem, (cudaStream_t)stream>>>(
        topk_ids, s->T, s->K, s->E, s->flags, table_out,
        &static_cast<moe::WsHeader *>(workspace)->err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "launch group_table_kernel");
    return MOE_OK;
}

moe_status moe_fused_decode(const void *x, const int32_t *topk_ids, const float *topk_w,
                            const moe_weights *routed, const moe_weights *shared, void *out,
                            const moe_shape *s, void *workspace, size_t workspace_bytes,
                            void *stream) {
    return fused_decode_impl(x, topk_ids, topk_w, routed, shared, out, s, workspace,
                             workspace_bytes, (cudaStream_t)stream);
}

moe_status moe_fused_decode_host(const void *x_host, const int32_t *ids_host, const float *w_host,
                                 const moe_weights *routed, const moe_weights *shared,
                                 void *out_host, const moe_shape *s, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    const WsLayout L = ws_layout(s);
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (workspace_bytes < L.host_total)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu B, the host-buffer call needs %zu B",
                    workspace_bytes, L.host_total);
    if (s->T == 0) return MOE_OK;
    if (!x_host || !ids_host || !w_host || !out_host)
        return fail(MOE_ERR_INVALID_ARG, "NULL host buffer");
    cudaStream_t cs = (cudaStream_t)stream;
    char *ws = static_cast<char *>(workspace);
    const size_t xb = (size_t)s->T * s->H * 2, kb = (size_t)s->T * s->K * 4;
    cudaError_t e;
    if ((e = cudaMemcpyAsync(ws + L.st_x, x_host, xb, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
        return cuda_fail(e, "copy x to device");
    if ((e = cudaMemcpyAsync(ws + L.st_ids, ids_host, kb, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
        return cuda_fail(e, "copy topk_ids to device");
    if ((e = cudaMemcpyAsync(ws + L.st_w, w_host, kb, cudaMemcpyHostToDevice, cs)) != cudaSuccess)
        return cuda_fail(e, "copy topk_w to device");
    st = fused_decode_impl(ws + L.st_x, reinterpret_cast<const int32_t *>(ws + L.st_ids),
                           reinterpret_cast<const float *>(ws + L.st_w), routed, shared,
                           ws + L.st_out, s, workspace, workspace_bytes, cs);
    if (st != MOE_OK) return st;
    if ((e = cudaMemcpyAsync(out_host, ws + L.st_out, xb, cudaMemcpyDeviceToHost, cs)) != cudaSuccess)
        return cuda_fail(e, "copy out to host");
    if ((e = cudaStreamSynchronize(cs)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    return MOE_OK;
}

moe_status moe_fused_decode_noalloc(const void *x, const int32_t *topk_ids, const float *topk_w,
                                    const moe_weights *routed, const moe_weights *shared,
                                    void *out, const moe_shape *s, uint32_t *err_out,
                                    void *stream) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    const size_t need = ws_layout(s).dev_total;
    if (need > kNoAllocScratchBytes)
        return fail(MOE_ERR_WORKSPACE,
                    "this shape needs %zu B of scratch; the no-allocation entry's built-in "
                    "scratch holds %zu B (use moe_fused_decode with a workspace)",
                    need, kNoAllocScratchBytes);
    if (err_out && !aligned(err_out, 4)) return fail(MOE_ERR_INVALID_ARG, "err_out not 4-byte aligned");
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != MOE_OK) return st;
    cudaStream_t cs = (cudaStream_t)stream;
    // The header must be zero when the kernel starts. The array is zero when
    // the library loads, and every call below leaves it zero again.
    st = fused_decode_impl(x, topk_ids, topk_w, routed, shared, out, s, scratch,
                           kNoAllocScratchBytes, cs);
    if (st != MOE_OK) return st;
    cudaError_t e;
    if (err_out &&
        (e = cudaMemcpyAsync(err_out, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, cs)) !=
            cudaSuccess)
        return cuda_fail(e, "copy error word");
    if ((e = cudaMemsetAsync(scratch, 0, sizeof(moe::WsHeader), cs)) != cudaSuccess)
        return cuda_fail(e, "clear no-allocation scratch header");
    return MOE_OK;
}

moe_status moe_read_error(void *workspace, uint32_t *err_bits, void *stream) {
    if (!workspace || !err_bits) return fail(MOE_ERR_INVALID_ARG, "NULL workspace or err_bits");
    cudaStream_t cs = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t v = 0;
    if ((e = cudaMemcpy(&v, workspace, sizeof v, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "read error word");
    if ((e = cudaMemset(workspace, 0, sizeof v)) != cudaSuccess) return cuda_fail(e, "clear error word");
    *err_bits = v;
    return MOE_OK;
}

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: valid but not supported by this build";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
    }
    return "unknown moe_status";
}

const char *moe_last_error_detail(void) { return g_detail.c_str(); }

}  // extern "C"
