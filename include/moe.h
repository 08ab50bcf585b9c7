/*
 * moe.h -- C ABI of the B300 fused decode MoE layer library (libmoe.so).
 *
 * The layer (one decode step, T token rows):
 *
 *   out[t] = bf16( x[t] + S(x[t]) + sum_p topk_w[t,p] * R_{topk_ids[t,p]}(x[t]) )
 *   F(x)   = Wd * ( silu(Wg x) .* (Wu x) )         (S = shared, R_e = routed e)
 *
 * Source: "Daily AI Hotspot 2026-08-21: Shared-Expert Fusion Lands on NVIDIA and
 * AMD the Same Day", section "Most Worth Your Attention Today" -- routed FP4
 * experts and an FP8 shared expert every token passes through, the four
 * unfused launches (routed MoE, shared gate/up, shared down, residual add)
 * replaced by one persistent pass with FP32 accumulation that writes the BF16
 * output exactly once. Expert dedup and the group table follow
 * MarloweAI/sgl-amd-mono-upstream PR #27 "each expert once", sections
 * "Motivation", "Modifications" and "Reviewer notes": the step's shared expert
 * and each distinct routed expert stream their weights once, with every row
 * that uses the expert batched as a column; the result is bitwise equal to the
 * one-row form.
 *
 * Conventions for every entry point:
 *   - All pointers except those documented as host pointers are DEVICE
 *     pointers, owned by the caller; the library allocates nothing per call
 *     and keeps no pointer after a call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous on that stream: the returned status covers argument
 *     validation and launch errors only. Problems found on the device set
 *     bits in the workspace's error word (MOE_DEV_*), read with
 *     moe_read_error(). No kernel traps.
 *   - A call that returns an error other than MOE_ERR_CUDA launched nothing.
 *   - moe_last_error_detail() describes the last failed call on this host
 *     thread in one line.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size, aliasing */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but outside what this build handles */
    MOE_ERR_WORKSPACE = 3,    /* workspace too small or not initialised */
    MOE_ERR_CUDA = 4          /* a CUDA runtime call failed */
} moe_status;

/* Bits of the device error word. */
enum {
    MOE_DEV_BAD_EXPERT = 1u,   /* a topk id outside [0, E): that pick adds 0 */
    MOE_DEV_DUP_EXPERT = 2u,   /* an id repeated within a row: both uses count */
    MOE_DEV_WAIT_TIMEOUT = 4u, /* an inter-CTA wait gave up; output invalid,
                                  call moe_workspace_init before reuse */
    MOE_DEV_RANGE = 8u         /* an intermediate left the range of the
                                  tensor-core operand type; output invalid */
};

/* moe_shape.flags */
enum {
    MOE_FLAG_NO_DEDUP = 1u,   /* one-row form: every (row, pick) and every
                                 row's shared use is its own 1-column group */
    MOE_FLAG_FORCE_FMA = 2u,  /* CUDA-core dequant-GEMV contraction */
    MOE_FLAG_FORCE_MMA = 4u,  /* tcgen05 tensor-core contraction */
    MOE_FLAG_DEBUG_DROP_ARRIVE = 8u, /* fault injection: one CTA skips one
                                 inter-CTA arrival, so the waits on it time out
                                 and set MOE_DEV_WAIT_TIMEOUT */
    MOE_FLAG_CHAIN = 16u,     /* layers back to back: the launch may start
                                 while the previous kernel on the stream still
                                 runs (programmatic dependent launch). Each CTA
                                 sets up its barriers and tensor memory and
                                 streams its first shared-expert weights, then
                                 waits for the previous grid to complete before
                                 it reads any input or the workspace, so the
                                 result is the same bits as without the flag
                                 and the previous kernel may produce this
                                 launch's inputs. Only weights must not be
                                 written by the previous kernel. */
    MOE_FLAG_FP8_MID = 32u    /* opt-in low-precision variant (PR #27 "each
                                 expert once", "Modifications": FP8 mid
                                 blocks): the SwiGLU intermediate goes
                                 through FP8 before down. Blocks of 32
                                 consecutive intermediate values of one
                                 column share the smallest power-of-two
                                 scale 2^k with max|mid| <= 448 * 2^k
                                 (k >= -126); each value becomes its nearest
                                 OCP E4M3FN value (ties to even) times 2^k.
                                 Tensor-core path only: with
                                 MOE_FLAG_FORCE_FMA, or where the tensor-core
                                 path is not eligible, the call fails with
                                 MOE_ERR_UNSUPPORTED. */
};

/* Weight storage formats. */
typedef enum {
    MOE_W_BF16 = 0,     /* bf16, no scales */
    MOE_W_NVFP4 = 1,    /* E2M1 codes, 2 per byte (low nibble = even element);
                           E4M3 scale per 16 elements along the input
                           (contiguous) dimension; fp32 scale per expert and
                           matrix */
    MOE_W_FP8_B128 = 2  /* E4M3FN bytes; fp32 scale per 128x128 block */
} moe_wfmt;

/*
 * One expert set: the E routed experts, or the shared expert (E = 1).
 * Row-major, the input dimension contiguous:
 *   w13  [E][2I][H]  rows 0..I-1 = gate (Wg), rows I..2I-1 = up (Wu)
 *   w2   [E][H][I]   down (Wd)
 * Element storage per fmt (H, I are the set's sizes):
 *   BF16 : w13 uint16 [E][2I][H]; w2 uint16 [E][H][I]; scales NULL
 *   NVFP4: w13 uint8 [E][2I][H/2]; w13_scale uint8 (E4M3) [E][2I][H/16];
 *          w13_gscale fp32 [E]; w2 uint8 [E][H][I/2]; w2_scale [E][H][I/16];
 *          w2_gscale fp32 [E].   Element = e2m1 * e4m3(block) * gscale.
 *   FP8  : w13 uint8 [E][2I][H]; w13_scale fp32 [E][2I/128][H/128];
 *          w2 uint8 [E][H][I]; w2_scale fp32 [E][H/128][I/128]; gscales NULL.
 *          Element = e4m3 * scale(block).
 * Every pointer 16-byte aligned. Device memory, read only.
 */
typedef struct {
    int fmt; /* moe_wfmt */
    const void *w13;
    const void *w13_scale;
    const float *w13_gscale;
    const void *w2;
    const void *w2_scale;
    const float *w2_gscale;
} moe_weights;

/*
 * T rows (0 <= T <= 256), hidden H, routed intermediate I, shared
 * intermediate I_shared, E routed experts (1 <= E <= 1024), K picks a row
 * (1 <= K <= 16, K <= E; K need not be a power of two). H, I and I_shared
 * must be multiples of 128 and at most 16384.
 */
typedef struct {
    int T, H, I, I_shared, E, K;
    unsigned flags; /* MOE_FLAG_* */
} moe_shape;

/* Bytes of device workspace moe_fused_decode needs for this shape (the
 * error word, inter-CTA counters and the fp32 intermediates). Sizes for a
 * larger T also serve any smaller T with the same other fields. One
 * workspace may serve launches of different shapes (T, K, I, I_shared) as
 * long as it is at least moe_workspace_bytes of each: the counters sit at
 * the same offsets for every shape. */
size_t moe_workspace_bytes(const moe_shape *s);

/* Zero a workspace (async on stream). Required once before first use and
 * after a MOE_DEV_WAIT_TIMEOUT. */
moe_status moe_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/* Number of int32 in a group table for T rows and K picks: 2 + 5*T*(K+1). */
size_t moe_group_table_ints(int T, int K);

/*
 * Distinct-expert group table of one step (PR #27 "each expert once",
 * "Modifications" commit 1 and "Reviewer notes": count, each group's expert,
 * each row's slot; found with a warp ballot over the picks).
 *
 *   topk_ids   int32 [T][K]   device
 *   table_out  int32 [moe_group_table_ints(T, K)]   device, written fully:
 *     [0] G (groups)  [1] U (columns = row uses)   then, with C = T*(K+1):
 *     group_expert[C]  expert of each group, -1 = the shared expert
 *     group_ncols[C]   columns of each group
 *     group_col0[C]    first column of each group (prefix sum)
 *     col_row[C]       row of each column
 *     row_col[T][K+1]  slot 0 = the row's shared column, 1+p = pick p's
 *                      column (-1 for an out-of-range id)
 *     entries past G (or U) are 0.
 *   Dedup order: group 0 = shared expert, then distinct in-range ids in order
 *   of first use scanning (t, p) row-major; columns in a group in that same
 *   order. With MOE_FLAG_NO_DEDUP in s->flags: per row, the shared use then
 *   each in-range pick, one group and one column each.
 *   workspace  receives MOE_DEV_BAD_EXPERT / MOE_DEV_DUP_EXPERT.
 */
moe_status moe_group_table(const int32_t *topk_ids, const moe_shape *s,
                           int32_t *table_out, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * The fused layer, one persistent launch.
 *   x         bf16 [T][H]        device, 16-byte aligned
 *   topk_ids  int32 [T][K]       device
 *   topk_w    fp32 [T][K]        device (used as given: no renormalising)
 *   routed    E experts, intermediate I      (struct in host memory)
 *   shared    1 expert, intermediate I_shared (struct in host memory)
 *   out       bf16 [T][H]        device, must not overlap x; written once
 *   workspace device, >= moe_workspace_bytes(s), initialised once with
 *             moe_workspace_init; one launch at a time per workspace
 * Each row's output is summed in a fixed order (residual, shared expert,
 * picks 0..K-1) in fp32, rounded to bf16 once. The result does not depend on
 * the dedup flag, the grid size or timing (bit for bit).
 */
moe_status moe_fused_decode(const void *x, const int32_t *topk_ids,
                            const float *topk_w, const moe_weights *routed,
                            const moe_weights *shared, void *out,
                            const moe_shape *s, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * moe_fused_decode for layers run back to back: the same computation and
 * arguments, plus next_shared, the shared expert of the layer launched next
 * with the same shape (same format, H and I_shared; device memory, not
 * written before that launch). Once this launch has handed out its last job,
 * each CTA requests into L2 the first weight stages of the next layer's
 * shared expert that the same CTA of that launch loads before its group
 * table, so those arrive from L2 while the next launch builds its table
 * ("Daily AI Hotspot 2026-08-21", "Most Worth Your Attention Today": the
 * persistent kernel's start-up cost; PR #27 "each expert once",
 * "Modifications": weight loads issued ahead of every wait). A prefetch moves
 * no result: the output is the same bits as moe_fused_decode's. The
 * CUDA-core contraction ignores the hint. Errors: those of moe_fused_decode,
 * and MOE_ERR_INVALID_ARG when next_shared is NULL, incomplete, misaligned or
 * of another format than `shared`.
 */
moe_status moe_fused_decode_next(const void *x, const int32_t *topk_ids,
                                 const float *topk_w, const moe_weights *routed,
                                 const moe_weights *shared,
                                 const moe_weights *next_shared, void *out,
                                 const moe_shape *s, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * The same layer called with HOST buffers for the step's inputs and output
 * (x_host bf16 [T][H], ids_host int32 [T][K], w_host fp32 [T][K],
 * out_host bf16 [T][H]; pinned memory makes the copies asynchronous).
 * Weights stay in device memory. The inputs are copied into the workspace's
 * staging area, the layer runs, the output is copied back, and the call
 * returns after `stream` has finished. Needs moe_workspace_bytes_host(s).
 */
size_t moe_workspace_bytes_host(const moe_shape *s);
moe_status moe_fused_decode_host(const void *x_host, const int32_t *ids_host,
                                 const float *w_host, const moe_weights *routed,
                                 const moe_weights *shared, void *out_host,
                                 const moe_shape *s, void *workspace,
                                 size_t workspace_bytes, void *stream);

/*
 * The fused layer for callers that cannot allocate device memory. The pages
 * have no counterpart to this entry point; it exists for callers that may not
 * call cudaMalloc: code that runs while a CUDA graph is being captured in
 * global mode (cudaMalloc is not permitted then), plugins whose host
 * framework owns every device allocation, and latency-critical paths that
 * cannot take cudaMalloc's implicit device-wide synchronisation.
 *
 * Same computation and arguments as moe_fused_decode, minus the workspace,
 * always on the CUDA-core contraction (MOE_FLAG_FORCE_FMA; its fp32
 * intermediates are the smaller scratch): the scratch is a file-scope device
 * array of 8 MiB inside the library, which
 * every GPU that loads the library holds until the process exits. Shapes
 * whose CUDA-core scratch, 256 + 4*T*(K+1)*(Imax + H) bytes (rounded up to
 * 256-byte boundaries) with Imax = max(I, I_shared), exceeds 8 MiB are
 * rejected with MOE_ERR_WORKSPACE before anything is launched (DeepSeek-V3
 * shapes: T <= 25).
 *   err_out  optional device uint32: receives the call's device error word
 *            (MOE_DEV_* bits); NULL to ignore it.
 * The first call in a CUDA context looks up the array's device address there
 * (with that context's device current) and keeps it under the context's
 * unique id, so a context created later (another driver-API context, or the
 * runtime's after cudaDeviceReset) gets its own lookup; make the first call
 * in each context before any stream capture.
 * All calls share the one array and it keeps the last call's contents; each
 * call leaves its header cleared for the next. Calls that overlap on the GPU
 * (different streams, or threads) race on it: serialise them. This entry
 * point calls no cudaMalloc or cudaFree.
 */
moe_status moe_fused_decode_noalloc(const void *x, const int32_t *topk_ids,
                                    const float *topk_w, const moe_weights *routed,
                                    const moe_weights *shared, void *out,
                                    const moe_shape *s, uint32_t *err_out,
                                    void *stream);

/*
 * The routing front end: topk_ids and topk_w computed from the layer input.
 * "Daily AI Hotspot 2026-08-21", section "Most Worth Your Attention Today"
 * (the SGLang #32340 paragraph): a bf16 correction bias and a top-k whose K is
 * not a power of two. PR #27 "each expert once", "Reviewer notes": every CTA
 * routes all rows itself and the tie order is unchanged. The pages give no
 * scoring formula; this library takes the DeepSeek-V3 one. For row t, expert e:
 *
 *   logit[t,e] = x[t] . wr[e]                 (fp32 sums of the bf16 products)
 *   s[t,e]     = 1 / (1 + exp(-logit[t,e]))   (sigmoid score)
 *   key[t,e]   = s[t,e] + bias[e]             (selection only)
 *   topk_ids   = the K experts of largest key, largest first; equal keys: the
 *                lower expert first
 *   topk_w[p]  = scale * s[ids[p]] / sum_q s[ids[q]]   (renorm = 1)
 *                scale * s[ids[p]]                     (renorm = 0)
 *
 *   wr    bf16 [E][H], H contiguous, 16-byte aligned (device)
 *   bias  bf16 [E] correction bias (device), or NULL for none
 * E <= 1024. The logits are summed in a fixed order, so the picks are the
 * same on every call; keys that differ by less than the fp32 rounding of the
 * logits may order differently from an exact computation.
 */
typedef struct {
    const void *wr;
    const void *bias;
    float scale;
    int renorm;
} moe_router;

/*
 * The router alone (one cooperative launch): writes topk_ids int32 [T][K] and
 * topk_w fp32 [T][K] (device). workspace as for moe_fused_decode
 * (>= moe_workspace_bytes(s), initialised once).
 */
moe_status moe_route(const void *x, const moe_router *router, int32_t *topk_ids,
                     float *topk_w, const moe_shape *s, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * The fused layer with the router inside the same launch: every CTA computes
 * its share of the router's logits, waits for all of them, picks every row's
 * experts on chip and builds its group table from them; the rest is
 * moe_fused_decode with those picks and weights (bit for bit the result of
 * moe_fused_decode given the topk_ids / topk_w this call returns).
 *   topk_ids, topk_w  optional device outputs [T][K] (NULL to skip)
 * Other arguments as for moe_fused_decode.
 */
moe_status moe_fused_decode_routed(const void *x, const moe_router *router,
                                   const moe_weights *routed, const moe_weights *shared,
                                   void *out, int32_t *topk_ids, float *topk_w,
                                   const moe_shape *s, void *workspace,
                                   size_t workspace_bytes, void *stream);

/* Synchronise `stream`, copy the device error word to *err_bits and clear it. */
moe_status moe_read_error(void *workspace, uint32_t *err_bits, void *stream);

/* Static description of a status code. */
const char *moe_status_string(moe_status s);

/* One-line description of the last failed call on this host thread. */
const char *moe_last_error_detail(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
