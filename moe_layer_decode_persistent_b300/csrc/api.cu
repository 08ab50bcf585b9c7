// api.cu -- the C ABI of libmoe (declared in include/moe.h): argument
// validation, workspace layout, launch configuration and error reporting.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "fused_fma.cuh"
#include "fused_tc.cuh"

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
static_assert(kMaxT * (kMaxK + 1) <= moe::kTcReadyCap, "group_ready capacity");
static_assert(kMaxE <= moe::kRouterMaxE, "the router's picks hold every expert");
static_assert(kMaxDim / 256 <= moe::kTcHtileCap, "htile_cnt capacity");
static_assert(moe::group_table_scratch_ints(kMaxT, kMaxK, kMaxE) * 4 <= moe::kRawStageBytes,
              "the group table scratch fits in one raw stage");

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Workspace. Both kernels share the 256-byte header (error word, counters),
// and the tensor path's counters come next in a region the CUDA-core path never
// writes, so they stay valid when the two paths take turns on one workspace:
//   header | group_ready [2][kTcReadyCap] | htile_cnt [2][kTcHtileCap] |
//   tile_cnt [kTcTileCntWords] | then
//   CUDA-core path : mid fp32 [Ucap][Imax] | y fp32 [Ucap][H]
//   tensor path    : P | Y | midB | xh f16 [T][H]
// followed by the host-buffer call's staging area. Ucap = C = T*(K+1). The
// counter region's size is a constant (sized from the largest T, K and
// intermediate the tensor path splits), so it sits at the same offsets for
// every shape: launches of different T, K, I or I_shared on one workspace
// never find their counters under another shape's scratch.
constexpr size_t kTcTileCntWords = (size_t)moe::kSplitMaxT * (kMaxK + 1) * (kMaxDim / 128) * 4;
struct WsLayout {
    size_t route = 0;  // router partial logits [T][E][kRouterParts] fp32 (routed launches)
    size_t mid = 0, y = 0, fma_end = 0;
    size_t tc_ready = 0, tc_htile = 0, tc_tile = 0, tc_par = 0, tc_ctrl_end = 0, tc_P = 0, tc_Y = 0, tc_midB = 0,
           tc_xh = 0, tc_xs = 0, tc_end = 0;
    size_t dev_total = 0;
    size_t st_x = 0, st_ids = 0, st_w = 0, st_out = 0, host_total = 0;
};

WsLayout ws_layout(const moe_shape *s) {
    WsLayout L;
    const size_t T = (size_t)std::max(s->T, 0), K = (size_t)std::max(s->K, 0);
    const size_t Ucap = T * (K + 1);
    const size_t Imax = (size_t)std::max(s->I, s->I_shared);
    const size_t H = (size_t)s->H;
    size_t off = sizeof(moe::WsHeader);
    L.tc_ready = off;
    off += 2 * (size_t)moe::kTcReadyCap * 4;
    L.tc_htile = off = align_up(off, 16);
    off += 2 * (size_t)moe::kTcHtileCap * 4;
    // tile_cnt: one word per (group, column tile, 128-row tile, quarter) of a
    // launch that splits K, i.e. at most kSplitMaxT*(K+1) column tiles times
    // Imax/128 row tiles; sized for the caps so the region never moves
    L.tc_tile = off = align_up(off, 16);
    off += kTcTileCntWords * 4;
    L.tc_par = off = align_up(off, 16);  // one launch-parity word per CTA
    off += (size_t)moe::kTcMaxGrid * 4;
    L.tc_ctrl_end = off = align_up(off, 256);

    L.mid = off;
    off += Ucap * Imax * sizeof(float);
    L.y = off = align_up(off, 256);
    off += Ucap * H * sizeof(float);
    L.fma_end = align_up(off, 256);

    off = L.tc_ctrl_end;
    // The K-chunk partials are sized for the most chunks any T' <= T uses (one
    // row, the shortest jobs, at up to kSplitMaxT rows), so the size for T also
    // serves every smaller T.
    const int Hi = (int)H;
    const size_t Tsplit = std::min(T, (size_t)moe::kSplitMaxT), Usplit = Tsplit * (K + 1);
    const size_t nkc_gu = (size_t)std::max(moe::tc_nkc_gu(moe::kFmtNvfp4, Hi, 1), moe::tc_nkc_gu(moe::kFmtFp8B128, Hi, 1));
    const size_t y_cols = std::max((size_t)moe::tc_nkc_dn((int)Imax, 1) * Usplit, Ucap);
    L.tc_P = off;
    off += nkc_gu * 2 * Usplit * Imax * sizeof(float);
    L.tc_Y = off = align_up(off, 256);
    off += y_cols * H * sizeof(float);
    // sum over (group, column tile) of the padded column counts: each group pads
    // its last column tile to a multiple of 16, so it is at most U + 15 * G <=
    // 16 * U in either form (the size does not depend on the flags)
    const size_t cols_padded = 16 * Ucap;
    L.tc_midB = off = align_up(off, 256);
    off += cols_padded * (Imax / 128) * 256;
    L.tc_xh = off = align_up(off, 256);
    off += T * H * 2;
    L.tc_xs = off = align_up(off, 256);
    off += T * 4;
    L.tc_end = align_up(off, 256);

    L.route = off = std::max(L.fma_end, L.tc_end);
    off = align_up(off + T * (size_t)std::max(s->E, 0) * moe::kRouterParts * sizeof(float), 256);
    L.dev_total = off;
    L.st_x = off;
    off = align_up(off + T * H * 2, 256);
    L.st_ids = off;
    off = align_up(off + T * K * 4, 256);
    L.st_w = off;
    off = align_up(off + T * K * 4, 256);
    L.st_out = off;
    off = align_up(off + T * H * 2, 256);
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
                           MOE_FLAG_DEBUG_DROP_ARRIVE | MOE_FLAG_CHAIN | MOE_FLAG_FP8_MID;
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

// CUDA-core kernel and standalone table: the table, its scratch, then the
// routed weights [T][K] (used by routed launches)
size_t table_smem_bytes(const moe_shape *s) {
    return sizeof(int32_t) * (size_t)(moe::group_table_ints(s->T, s->K) + moe::group_table_scratch_ints(s->T, s->K, s->E) +
                                      s->T * s->K);
}

struct DevInfo {
    int nsm = 0;
    int max_smem_optin = 0;
    int tc_static_smem = 0;  // static shared memory of the tensor-core kernel
};

// Per-device facts, filled once per device (under a lock) and read without one.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];
std::atomic<bool> g_dev_ready[kMaxDevices];

moe_status current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (*dev < 0 || *dev >= kMaxDevices)
        return fail(MOE_ERR_UNSUPPORTED, "device %d: the library handles devices 0..%d", *dev, kMaxDevices - 1);
    return MOE_OK;
}

moe_status dev_info(int dev, DevInfo *out) {
    if (g_dev_ready[dev].load(std::memory_order_acquire)) {
        *out = g_dev[dev];
        return MOE_OK;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev_ready[dev].load(std::memory_order_relaxed)) {
        DevInfo d;
        cudaError_t e = cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(smem)");
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, moe::fused_tc_kernel<false, false, false>);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes");
        d.tc_static_smem = (int)fa.sharedSizeBytes;
        g_dev[dev] = d;
        g_dev_ready[dev].store(true, std::memory_order_release);
    }
    *out = g_dev[dev];
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
// set; cached per (device, kernel, threads, smem) so a launch inside stream
// capture makes no other CUDA call.
template <typename Kern>
moe_status plan_occupancy(Kern k, int dev, int threads, size_t smem, const DevInfo &d, int *occ_out) {
    struct Entry {
        int dev;
        const void *k;
        int threads;
        size_t smem;
        int occ;
    };
    static std::mutex mu;
    static std::vector<Entry> cache;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (const Entry &c : cache)
            if (c.dev == dev && c.k == (const void *)k && c.threads == threads && c.smem == smem) {
                *occ_out = c.occ;
                return MOE_OK;
            }
    }
    moe_status st = set_smem(k, smem, d);
    if (st != MOE_OK) return st;
    int occ = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (occ < 1) return fail(MOE_ERR_UNSUPPORTED, "kernel does not fit on an SM (%zu B smem)", smem);
    std::lock_guard<std::mutex> lk(mu);
    cache.push_back({dev, (const void *)k, threads, smem, occ});
    *occ_out = occ;
    return MOE_OK;
}

// Launches a fused kernel cooperatively: every CTA resident at once, or the
// launch fails. A chained launch (MOE_FLAG_CHAIN) also carries programmatic
// stream serialization, so it may start while the previous kernel on the
// stream still runs. Where the runtime refuses the two attributes together,
// chained launches on that device go without the cooperative one: the grid is
// still one wave by the occupancy calculation, and every inter-CTA wait is
// bounded, so a grid that could not be all resident ends with
// MOE_DEV_WAIT_TIMEOUT instead of hanging.
std::atomic<int> g_chain_coop[kMaxDevices];  // 0 untried, 1 accepted, 2 refused

template <typename P>
moe_status launch_persistent(cudaLaunchConfig_t cfg, void (*kern)(P), const P &p, bool chain, int dev,
                             const char *what) {
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    const bool both = chain && g_chain_coop[dev].load(std::memory_order_relaxed) != 2;
    cfg.attrs = (chain && !both) ? attr + 1 : attr;
    cfg.numAttrs = both ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (both && (e == cudaErrorInvalidValue || e == cudaErrorNotSupported)) {
        (void)cudaGetLastError();  // a refused configuration, not a device error
        g_chain_coop[dev].store(2);
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, p);
    } else if (both && e == cudaSuccess) {
        g_chain_coop[dev].store(1, std::memory_order_relaxed);
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    return MOE_OK;
}

moe_status launch_fused_fma(const moe::FusedParams &p, const moe_shape *s, int dev, const DevInfo &d,
                            cudaStream_t stream) {
    const size_t smem = table_smem_bytes(s);
    int occ = 0;
    moe_status st = plan_occupancy(moe::fused_fma_kernel, dev, moe::kFmaThreads, smem, d, &occ);
    if (st != MOE_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(d.nsm * occ));
    cfg.blockDim = dim3(moe::kFmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return launch_persistent(cfg, moe::fused_fma_kernel, p, (s->flags & MOE_FLAG_CHAIN) != 0, dev,
                             "launch fused_fma_kernel");
}

// ---- tensor maps (cached: encoding costs microseconds of host time) ----------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

moe_status encode_fn(EncodeTiledFn *out) {
    static EncodeTiledFn fn = nullptr;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !ptr)
            return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        fn = (EncodeTiledFn)ptr;
    }
    *out = fn;
    return MOE_OK;
}

// 3-D uint8 map over [E][rows][cols] bytes; box [box_c][128][1].
moe_status tensor_map(CUtensorMap *out, const void *base, size_t cols, size_t rows, size_t E, int box_c,
                      bool swz128) {
    EncodeTiledFn enc;
    moe_status st = encode_fn(&enc);
    if (st != MOE_OK) return st;
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)E};
    cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)(cols * rows)};
    cuuint32_t box[3] = {(cuuint32_t)box_c, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swz128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return MOE_OK;
}

// codes and (NVFP4) block-scale maps of one expert set
moe_status set_maps(const moe_weights *w, int E, int H, int I, CUtensorMap *m13, CUtensorMap *m13s,
                    CUtensorMap *m2, CUtensorMap *m2s) {
    const bool fp4 = w->fmt == MOE_W_NVFP4;
    const size_t h_b = fp4 ? (size_t)H / 2 : (size_t)H, i_b = fp4 ? (size_t)I / 2 : (size_t)I;
    moe_status st = tensor_map(m13, w->w13, h_b, 2 * (size_t)I, E, 128, true);
    if (st == MOE_OK) st = tensor_map(m2, w->w2, i_b, (size_t)H, E, 128, true);
    if (st != MOE_OK) return st;
    if (fp4) {
        st = tensor_map(m13s, w->w13_scale, (size_t)H / 16, 2 * (size_t)I, E, 16, false);
        if (st == MOE_OK) st = tensor_map(m2s, w->w2_scale, (size_t)I / 16, (size_t)H, E, 16, false);
        return st;
    }
    *m13s = *m13;  // unused for FP8
    *m2s = *m2;
    return MOE_OK;
}

// The eight tensor maps of a (routed, shared, shape) triple, cached: encoding
// them costs microseconds of host time, and a caller typically cycles over a
// few resident weight sets (one per layer). Up to kMapsCache entries, replaced
// in turn.
moe_status tc_maps(const moe_weights *routed, const moe_weights *shared, const moe_shape *s, moe::TcMaps *out) {
    struct Key {
        const void *p[8];
        int fr, fs, E, H, I, Is;
        bool operator==(const Key &o) const { return memcmp(this, &o, sizeof(Key)) == 0; }
    };
    struct Entry {
        Key k;
        moe::TcMaps m;
    };
    constexpr int kMapsCache = 32;
    static std::mutex mu;
    static Entry cache[kMapsCache];
    static int used = 0, next = 0;
    Key key;
    memset(&key, 0, sizeof key);
    key.p[0] = routed->w13;
    key.p[1] = routed->w13_scale;
    key.p[2] = routed->w2;
    key.p[3] = routed->w2_scale;
    key.p[4] = shared->w13;
    key.p[5] = shared->w13_scale;
    key.p[6] = shared->w2;
    key.p[7] = shared->w2_scale;
    key.fr = routed->fmt;
    key.fs = shared->fmt;
    key.E = s->E;
    key.H = s->H;
    key.I = s->I;
    key.Is = s->I_shared;
    {
        std::lock_guard<std::mutex> lk(mu);
        for (int i = 0; i < used; ++i)
            if (cache[i].k == key) {
                *out = cache[i].m;
                return MOE_OK;
            }
    }
    moe::TcMaps m;
    moe_status st = set_maps(routed, s->E, s->H, s->I, &m.r13, &m.r13s, &m.r2, &m.r2s);
    if (st == MOE_OK) st = set_maps(shared, 1, s->H, s->I_shared, &m.s13, &m.s13s, &m.s2, &m.s2s);
    if (st != MOE_OK) return st;
    std::lock_guard<std::mutex> lk(mu);
    const int slot = used < kMapsCache ? used++ : (next++ % kMapsCache);
    cache[slot].k = key;
    cache[slot].m = m;
    *out = m;
    return MOE_OK;
}

// Whether the tensor-core path handles this launch (and why not).
bool tc_eligible(const moe_shape *s, const moe_weights *routed, const moe_weights *shared, const DevInfo &d,
                 const char **why) {
    if (routed->fmt == MOE_W_BF16 || shared->fmt == MOE_W_BF16) {
        *why = "bf16 weights use the CUDA-core path";
        return false;
    }
    if (s->H % 256 || s->I % 256 || s->I_shared % 256) {
        *why = "H, I and I_shared must be multiples of 256";
        return false;
    }
    if (s->T > moe::kTcMaxT) {
        *why = "T above 256";
        return false;
    }
    const bool nd = (s->flags & MOE_FLAG_NO_DEDUP) != 0;
    if (moe::tc_smem_bytes(s->T, s->K, s->E, nd, moe::kRawStagesMin) > d.max_smem_optin - d.tc_static_smem) {
        *why = "group tables do not fit in shared memory";
        return false;
    }
    return true;
}

moe_status launch_fused_tc(const moe::FusedParams &fp, const WsLayout &L, const moe_shape *s,
                           const moe_weights *routed, const moe_weights *shared, const moe_weights *next_shared,
                           int dev, const DevInfo &d, cudaStream_t stream) {
    moe::TcParams p;
    memset(&p, 0, sizeof p);
    moe_status st = tc_maps(routed, shared, s, &p.maps);
    if (st != MOE_OK) return st;
    p.x = fp.x;
    p.ids = fp.ids;
    p.topk_w = fp.topk_w;
    p.routed = fp.routed;
    p.shared = fp.shared;
    p.out = fp.out;
    p.T = s->T;
    p.H = s->H;
    p.I = s->I;
    p.Is = s->I_shared;
    p.E = s->E;
    p.K = s->K;
    p.flags = s->flags;
    if (next_shared) {
        p.nx13 = static_cast<const uint8_t *>(next_shared->w13);
        p.nx13s = static_cast<const uint8_t *>(next_shared->w13_scale);
    }
    char *ws = reinterpret_cast<char *>(fp.hdr);
    p.hdr = fp.hdr;
    p.group_ready = reinterpret_cast<uint32_t *>(ws + L.tc_ready);
    p.tile_cnt = reinterpret_cast<uint32_t *>(ws + L.tc_tile);
    p.htile_cnt = reinterpret_cast<uint32_t *>(ws + L.tc_htile);
    p.cta_par = reinterpret_cast<uint32_t *>(ws + L.tc_par);
    p.P = reinterpret_cast<float *>(ws + L.tc_P);
    p.Y = reinterpret_cast<float *>(ws + L.tc_Y);
    p.midB = reinterpret_cast<uint8_t *>(ws + L.tc_midB);
    p.xh = reinterpret_cast<__half *>(ws + L.tc_xh);
    p.xs = reinterpret_cast<int32_t *>(ws + L.tc_xs);
    p.Ucap = s->T * (s->K + 1);
    p.Imax = std::max(s->I, s->I_shared);
    p.route_mode = fp.route_mode;
    p.router = fp.router;
    for (int i = 0; i < 2; ++i) {  // 0: shared expert, 1: routed experts
        const int fmt = i == 0 ? shared->fmt : routed->fmt, Ig = i == 0 ? s->I_shared : s->I;
        moe::TcFmt &f = p.fc[i];
        f.nt = moe::tc_nt(fmt, s->T);
        f.nt_shift = f.nt == 32 ? 5 : 4;
        f.tiles = Ig / 128;
        f.nkc_gu = moe::tc_nkc_gu(fmt, s->H, s->T);
        f.kc_gu = moe::tc_kc_gu(fmt, s->H, s->T);
        f.nkc_dn = moe::tc_nkc_dn(Ig, s->T);
        f.kc_dn = moe::tc_kc_dn(Ig, s->T);
    }
    // the raw weight ring gets as many stages as shared memory holds
    const int smem_limit = d.max_smem_optin - d.tc_static_smem;
    const bool nd = (s->flags & MOE_FLAG_NO_DEDUP) != 0;
    int nR = moe::kRawStagesMax;
    while (nR > moe::kRawStagesMin && moe::tc_smem_bytes(s->T, s->K, s->E, nd, nR) > smem_limit) --nR;
    p.nR = nR;
    const size_t smem = (size_t)moe::tc_smem_bytes(s->T, s->K, s->E, nd, nR);
    int occ = 0;
    const bool capped = moe::tc_capped_tables(s->T);
    void (*kern)(const moe::TcParams) =
        !(s->flags & MOE_FLAG_FP8_MID)
            ? (p.route_mode ? (capped ? moe::fused_tc_kernel<true, true, false> : moe::fused_tc_kernel<false, true, false>)
                            : (capped ? moe::fused_tc_kernel<true, false, false> : moe::fused_tc_kernel<false, false, false>))
            : (p.route_mode ? (capped ? moe::fused_tc_kernel<true, true, true> : moe::fused_tc_kernel<false, true, true>)
                            : (capped ? moe::fused_tc_kernel<true, false, true> : moe::fused_tc_kernel<false, false, true>));
    if ((st = plan_occupancy(kern, dev, moe::kTcThreads, smem, d, &occ)) != MOE_OK) return st;
    cudaLaunchConfig_t cfg = {};
    if (d.nsm > moe::kTcMaxGrid)
        return fail(MOE_ERR_UNSUPPORTED, "%d SMs: the tensor-core path keeps parity words for %d", d.nsm,
                    moe::kTcMaxGrid);
    cfg.gridDim = dim3((unsigned)d.nsm);  // one CTA per SM: it holds all of TMEM
    cfg.blockDim = dim3(moe::kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return launch_persistent(cfg, kern, p, (s->flags & MOE_FLAG_CHAIN) != 0, dev, "launch fused_tc_kernel");
}

// CUDA-core scratch laid out straight after the header (no tensor-path
// counter region): for a scratch buffer that only the CUDA-core kernel ever
// uses. Returns its size; mid and y get their offsets.
size_t fma_compact_layout(const moe_shape *s, size_t *mid, size_t *y) {
    const size_t T = (size_t)std::max(s->T, 0), K = (size_t)std::max(s->K, 0), Ucap = T * (K + 1);
    const size_t Imax = (size_t)std::max(s->I, s->I_shared), H = (size_t)s->H;
    *mid = sizeof(moe::WsHeader);
    *y = align_up(*mid + Ucap * Imax * sizeof(float), 256);
    return align_up(*y + Ucap * H * sizeof(float), 256);
}

// fma_compact: the caller's buffer serves the CUDA-core kernel alone (the
// no-allocation entry), with its scratch laid out by fma_compact_layout.
moe_status check_router(const moe_router *r, const moe_shape *s) {
    if (!r) return fail(MOE_ERR_INVALID_ARG, "router struct is NULL");
    if (!r->wr) return fail(MOE_ERR_INVALID_ARG, "router weights are NULL");
    if (!aligned(r->wr, 16)) return fail(MOE_ERR_INVALID_ARG, "router weights not 16-byte aligned");
    if (r->bias && !aligned(r->bias, 2)) return fail(MOE_ERR_INVALID_ARG, "router bias not 2-byte aligned");
    if (!(r->scale == r->scale)) return fail(MOE_ERR_INVALID_ARG, "router scale is NaN");
    if (s->E > moe::kRouterMaxE) return fail(MOE_ERR_UNSUPPORTED, "the router handles E <= %d", moe::kRouterMaxE);
    return MOE_OK;
}

moe::RouterDev router_dev(const moe_router *r, const WsLayout &L, void *ws, int32_t *ids_out, float *w_out) {
    moe::RouterDev d;
    d.wr = static_cast<const __nv_bfloat16 *>(r->wr);
    d.bias = static_cast<const __nv_bfloat16 *>(r->bias);
    d.scale = r->scale;
    d.renorm = r->renorm ? 1 : 0;
    d.part = reinterpret_cast<float *>(static_cast<char *>(ws) + L.route);
    d.ids_out = ids_out;
    d.w_out = w_out;
    return d;
}

// router != null: a routed launch (the picks and weights come from the router
// inside the launch; ids and w are ignored, ids_out / w_out receive them).
moe_status fused_decode_impl(const void *x, const int32_t *ids, const float *w,
                             const moe_weights *routed, const moe_weights *shared, void *out,
                             const moe_shape *s, void *ws, size_t ws_bytes, cudaStream_t stream,
                             bool fma_compact = false, const moe_router *router = nullptr,
                             int32_t *ids_out = nullptr, float *w_out = nullptr,
                             const moe_weights *next_shared = nullptr) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    if ((st = check_weights(routed, "routed")) != MOE_OK) return st;
    if ((st = check_weights(shared, "shared")) != MOE_OK) return st;
    if (next_shared) {
        if ((st = check_weights(next_shared, "next shared")) != MOE_OK) return st;
        if (next_shared->fmt != shared->fmt)
            return fail(MOE_ERR_INVALID_ARG, "next shared weights: format %d, this layer's is %d", next_shared->fmt,
                        shared->fmt);
    }
    if (router && (st = check_router(router, s)) != MOE_OK) return st;
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    // host-only checks first: nothing below them touches the device until
    // the arguments are known to be valid
    const WsLayout L = ws_layout(s);
    size_t mid_off = L.mid, y_off = L.y, fma_need = L.fma_end;
    if (fma_compact) fma_need = fma_compact_layout(s, &mid_off, &y_off);
    const bool force_fma = fma_compact || (s->flags & MOE_FLAG_FORCE_FMA);
    size_t need_min = force_fma ? fma_need : std::min(fma_need, L.tc_end);
    if (router) need_min = L.dev_total;  // the router's partial logits sit past both paths' scratch
    if (ws_bytes < need_min)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu B, needs %zu B", ws_bytes, need_min);
    if (s->T == 0) return MOE_OK;
    if (!x || !out || (!router && (!ids || !w))) return fail(MOE_ERR_INVALID_ARG, "NULL x/out/topk_ids/topk_w");
    if (!aligned(x, 16) || !aligned(out, 16))
        return fail(MOE_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (!aligned(router ? ids_out : ids, 4) || !aligned(router ? w_out : w, 4))
        return fail(MOE_ERR_INVALID_ARG, "topk_ids and topk_w must be 4-byte aligned");
    const size_t act_bytes = (size_t)s->T * s->H * 2;
    const uintptr_t xa = (uintptr_t)x, oa = (uintptr_t)out;
    if (xa < oa + act_bytes && oa < xa + act_bytes)
        return fail(MOE_ERR_INVALID_ARG, "out overlaps x");
    // the path: tensor cores where eligible (a device fact: shared memory)
    int dev = 0;
    if ((st = current_device(&dev)) != MOE_OK) return st;
    DevInfo d;
    if ((st = dev_info(dev, &d)) != MOE_OK) return st;
    const char *why = "this entry runs the CUDA-core contraction";
    const bool tc_ok = !fma_compact && tc_eligible(s, routed, shared, d, &why);
    bool use_tc = tc_ok && !(s->flags & MOE_FLAG_FORCE_FMA);
    if ((s->flags & MOE_FLAG_FORCE_MMA) && !tc_ok)
        return fail(MOE_ERR_UNSUPPORTED, "tensor-core path requested but unavailable: %s", why);
    if ((s->flags & MOE_FLAG_FP8_MID) && !use_tc)
        return fail(MOE_ERR_UNSUPPORTED, "MOE_FLAG_FP8_MID needs the tensor-core path: %s",
                    tc_ok ? "MOE_FLAG_FORCE_FMA is set" : why);
    const size_t need = router ? L.dev_total : use_tc ? L.tc_end : fma_need;
    if (ws_bytes < need)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu B, needs %zu B", ws_bytes, need);

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
    p.mid = reinterpret_cast<float *>(static_cast<char *>(ws) + mid_off);
    p.y = reinterpret_cast<float *>(static_cast<char *>(ws) + y_off);
    p.Imax = std::max(s->I, s->I_shared);
    p.route_mode = router ? 1 : 0;
    memset(&p.router, 0, sizeof p.router);
    if (router) p.router = router_dev(router, L, ws, ids_out, w_out);
    if (use_tc) return launch_fused_tc(p, L, s, routed, shared, next_shared, dev, d, stream);
    return launch_fused_fma(p, s, dev, d, stream);
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

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

// Unique id of the CUDA context current on this thread (ids are never reused
// within a process, unlike context handles after a device reset).
moe_status current_context_id(unsigned long long *id) {
    static CtxGetCurrentFn get_cur = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!get_cur || !get_id) {
            cudaDriverEntryPointQueryResult q;
            void *p1 = nullptr, *p2 = nullptr;
            cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p1)
                return fail(MOE_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
            e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p2)
                return fail(MOE_ERR_CUDA, "cuCtxGetId is not available from the driver");
            get_cur = (CtxGetCurrentFn)p1;
            get_id = (CtxGetIdFn)p2;
        }
    }
    CUcontext ctx = nullptr;
    if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return fail(MOE_ERR_CUDA, "no current CUDA context");
    if (get_id(ctx, id) != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuCtxGetId failed");
    return MOE_OK;
}

// Device address of g_noalloc_scratch in the current context: looked up with
// cudaGetSymbolAddress the first time a context calls (its device current),
// then cached under the context's unique id, so a context created later (for
// example after a device reset) gets its own lookup.
moe_status noalloc_scratch(void **out) {
    struct Entry {
        unsigned long long ctx;
        void *addr;
    };
    constexpr int kEntries = 64;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    static std::mutex mu;
    unsigned long long ctx = 0;
    bool have_ctx = current_context_id(&ctx) == MOE_OK;
    std::lock_guard<std::mutex> lk(mu);
    if (have_ctx)
        for (int i = 0; i < used; ++i)
            if (cache[i].ctx == ctx) {
                *out = cache[i].addr;
                return MOE_OK;
            }
    // first call in this context (the lookup also makes the runtime's context
    // current when no context was)
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
    if (!have_ctx) {
        moe_status st = current_context_id(&ctx);
        if (st != MOE_OK) return st;
    }
    const int slot = used < kEntries ? used++ : (next++ % kEntries);
    cache[slot] = {ctx, p};
    *out = p;
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
    cudaError_t e = cudaMemsetAsync(workspace, 0, workspace_bytes, (cudaStream_t)stream);
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
    int dev = 0;
    if ((st = current_device(&dev)) != MOE_OK) return st;
    DevInfo d;
    if ((st = dev_info(dev, &d)) != MOE_OK) return st;
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

moe_status moe_fused_decode_next(const void *x, const int32_t *topk_ids, const float *topk_w,
                                 const moe_weights *routed, const moe_weights *shared,
                                 const moe_weights *next_shared, void *out, const moe_shape *s, void *workspace,
                                 size_t workspace_bytes, void *stream) {
    if (!next_shared) return fail(MOE_ERR_INVALID_ARG, "next shared weights struct is NULL");
    return fused_decode_impl(x, topk_ids, topk_w, routed, shared, out, s, workspace, workspace_bytes,
                             (cudaStream_t)stream, false, nullptr, nullptr, nullptr, next_shared);
}

moe_status moe_route(const void *x, const moe_router *router, int32_t *topk_ids, float *topk_w,
                     const moe_shape *s, void *workspace, size_t workspace_bytes, void *stream) {
    moe_status st = check_shape(s);
    if (st != MOE_OK) return st;
    if ((st = check_router(router, s)) != MOE_OK) return st;
    if (!workspace) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned(workspace, 256)) return fail(MOE_ERR_INVALID_ARG, "workspace not 256-byte aligned");
    const WsLayout L = ws_layout(s);
    if (workspace_bytes < L.dev_total)
        return fail(MOE_ERR_WORKSPACE, "workspace has %zu B, needs %zu B", workspace_bytes, L.dev_total);
    if (s->T == 0) return MOE_OK;
    if (!x || !topk_ids || !topk_w) return fail(MOE_ERR_INVALID_ARG, "NULL x/topk_ids/topk_w");
    if (!aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
    if (!aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(MOE_ERR_INVALID_ARG, "topk_ids and topk_w must be 4-byte aligned");
    int dev = 0;
    if ((st = current_device(&dev)) != MOE_OK) return st;
    DevInfo d;
    if ((st = dev_info(dev, &d)) != MOE_OK) return st;
    int occ = 0;
    if ((st = plan_occupancy(moe::route_kernel, dev, 256, 0, d, &occ)) != MOE_OK) return st;
    moe::RouterDev r = router_dev(router, L, workspace, topk_ids, topk_w);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    moe::WsHeader *hdr = static_cast<moe::WsHeader *>(workspace);
    int T = s->T, H = s->H, E = s->E, K = s->K;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(d.nsm * occ));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, moe::route_kernel, xb, r, T, H, E, K, hdr);
    if (e != cudaSuccess) return cuda_fail(e, "launch route_kernel");
    return MOE_OK;
}

moe_status moe_fused_decode_routed(const void *x, const moe_router *router, const moe_weights *routed,
                                   const moe_weights *shared, void *out, int32_t *topk_ids, float *topk_w,
                                   const moe_shape *s, void *workspace, size_t workspace_bytes, void *stream) {
    return fused_decode_impl(x, nullptr, nullptr, routed, shared, out, s, workspace, workspace_bytes,
                             (cudaStream_t)stream, false, router, topk_ids, topk_w);
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
    // the built-in scratch serves the CUDA-core contraction alone, laid out
    // straight after the header (its fp32 intermediates are the smaller scratch)
    moe_shape sf = *s;
    sf.flags = (sf.flags & ~(unsigned)MOE_FLAG_FORCE_MMA) | MOE_FLAG_FORCE_FMA;
    size_t mid_off = 0, y_off = 0;
    const size_t need = fma_compact_layout(&sf, &mid_off, &y_off);
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
    st = fused_decode_impl(x, topk_ids, topk_w, routed, shared, out, &sf, scratch,
                           kNoAllocScratchBytes, cs, true);
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
