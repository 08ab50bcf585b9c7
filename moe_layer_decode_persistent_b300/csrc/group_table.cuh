// group_table.cuh -- the step's distinct-expert group table, built by one CTA.
//
// MarloweAI/sgl-amd-mono-upstream PR #27 "each expert once", "Modifications"
// (commit 1) and "Reviewer notes": every CTA finds the step's distinct routed
// experts from the rows' top-k picks with a ballot that marks first uses, and
// keeps the table (group count, each group's expert, each row's slot) on chip,
// so no cross-CTA hand-off is needed. Group 0 is the shared expert, which
// every row uses first; routed groups follow in order of first use, scanning
// the picks row-major. Columns of a group follow the same order.
//
// On sm_103a with 32-lane warps: lane j of a 32-pick chunk holds pick j; a
// __ballot_sync marks first uses (first use = the pick holding the minimum
// flat index of its expert, found with a shared-memory atomicMin), and
// __match_any_sync ranks equal experts inside the chunk so each pick gets its
// column within its group in one pass.
#pragma once

#include <limits.h>

#include "moe_common.cuh"

namespace moe {

// Table layout (int32), C = T*(K+1), gcap >= G the capacity of the per-group
// arrays: [0] G, [1] U, group_expert[gcap], group_ncols[gcap], group_col0[gcap],
// col_row[C], row_col[T][K+1]. The exported table (moe_group_table) has
// gcap = C; the tensor-core kernel keeps it on chip with gcap = min(E, T*K) + 1
// (dedup form) so large T still fits.
struct GroupTable {
    int32_t *base;
    int C;
    int gcap;
    __device__ __forceinline__ int32_t &G() const { return base[0]; }
    __device__ __forceinline__ int32_t &U() const { return base[1]; }
    __device__ __forceinline__ int32_t *gexp() const { return base + 2; }
    __device__ __forceinline__ int32_t *gncols() const { return base + 2 + gcap; }
    __device__ __forceinline__ int32_t *gcol0() const { return base + 2 + 2 * gcap; }
    __device__ __forceinline__ int32_t *col_row() const { return base + 2 + 3 * gcap; }
    __device__ __forceinline__ int32_t *row_col() const { return base + 2 + 3 * gcap + C; }
    __device__ __forceinline__ int ints() const { return 2 + 3 * gcap + 2 * C; }
};

__host__ __device__ constexpr int group_table_ints(int T, int K) { return 2 + 5 * T * (K + 1); }
__host__ __device__ constexpr int group_table_ints_cap(int T, int K, int gcap) {
    return 2 + 3 * gcap + 2 * T * (K + 1);
}
// Groups a launch can have: every (row, slot) use in the one-row form, else
// the shared expert plus at most min(E, T*K) distinct routed experts.
__host__ __device__ constexpr int group_capacity(int T, int K, int E, bool no_dedup) {
    return no_dedup ? T * (K + 1) : 1 + (E < T * K ? E : T * K);
}

// Shared-memory ints group_table_cta needs besides the table: three per-expert
// arrays of E ints and a copy of the T*K picks.
__host__ __device__ constexpr int group_table_scratch_ints(int T, int K, int E) { return 3 * E + T * K; }
// Where in that scratch the copy of the picks ([T][K]) sits.
__host__ __device__ inline int *group_table_picks(int *scr, int E) { return scr + 3 * E; }

// Build the table for ids [T][K] into `tab` (shared memory) using `scr`
// (shared, group_table_scratch_ints(T, K, E) ints). Error bits are OR-ed into
// *err_word when err_word != null.
// ids == null: the picks are already in the scratch's pick copy
// (group_table_picks(scr, E)), put there by the on-chip router.
// The participating threads are threadIdx.x in [tid0, tid0 + nthr) (whole
// warps), synchronised with named barrier `bar` (bar 0 with the whole CTA is
// __syncthreads); the last barrier leaves the table visible to them.
__device__ __forceinline__ void gt_sync(int bar, int nthr) {
    asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(nthr) : "memory");
}

__device__ void group_table_cta(const int32_t *__restrict__ ids, int T, int K, int E,
                                bool no_dedup, GroupTable tab, int *scr, uint32_t *err_word,
                                int tid0, int nthr, int bar) {
    const int C = T * (K + 1), n = T * K, K1 = K + 1;
    const int tid = (int)threadIdx.x - tid0;
    const int lane = tid & 31, warp = tid >> 5;
    int *e_first = scr, *e_group = scr + E, *e_count = scr + 2 * E;
    int *sid = group_table_picks(scr, E);  // the picks, read from global memory once
    int32_t *gexp = tab.gexp(), *gn = tab.gncols(), *g0 = tab.gcol0(), *crow = tab.col_row(),
            *rcol = tab.row_col();

    for (int i = tid; i < tab.ints(); i += nthr) tab.base[i] = 0;
    for (int e = tid; e < E; e += nthr) {
        e_first[e] = INT_MAX;
        e_count[e] = 0;
    }
    if (ids)
        for (int j = tid; j < n; j += nthr) sid[j] = ids[j];
    gt_sync(bar, nthr);

    uint32_t err = 0;
    for (int j = tid; j < n; j += nthr) {
        const int id = sid[j], t = j / K, p = j - t * K;
        if (id < 0 || id >= E) {
            err |= kErrBadExpert;
            continue;
        }
        atomicMin(&e_first[id], j);
        for (int q = 0; q < p; ++q)
            if (sid[t * K + q] == id) err |= kErrDupExpert;
    }
    if (err && err_word) atomicOr(err_word, err);
    gt_sync(bar, nthr);

    if (warp == 0) {
        const unsigned lt = (1u << lane) - 1u;
        if (no_dedup) {
            // one group per (row, slot) use, slots in order: shared, picks
            int run = 0;
            for (int base = 0; base < C; base += 32) {
                const int s = base + lane;
                const int t = s / K1, slot = s - t * K1;
                int id = -1;
                bool v = false;
                if (s < C) {
                    if (slot == 0) {
                        v = true;
                    } else {
                        id = sid[t * K + slot - 1];
                        v = id >= 0 && id < E;
                    }
                }
                const unsigned b = __ballot_sync(0xffffffffu, v);
                const int idx = run + __popc(b & lt);
                if (v) {
                    gexp[idx] = id;  // -1 for the shared slot
                    gn[idx] = 1;
                    g0[idx] = idx;
                    crow[idx] = t;
                    rcol[s] = idx;
                } else if (s < C) {
                    rcol[s] = -1;
                }
                run += __popc(b);
            }
            if (lane == 0) {
                tab.G() = run;
                tab.U() = run;
            }
        } else if (T > 0) {
            int ngroups = 1;
            if (lane == 0) {
                gexp[0] = -1;
                gn[0] = T;
                g0[0] = 0;
            }
            for (int base = 0; base < n; base += 32) {
                const int j = base + lane;
                const int id = j < n ? sid[j] : -1;
                const bool valid = j < n && id >= 0 && id < E;
                const bool first = valid && e_first[id] == j;
                const unsigned b = __ballot_sync(0xffffffffu, first);
                if (first) {
                    const int g = ngroups + __popc(b & lt);
                    e_group[id] = g;
                    gexp[g] = id;
                }
                ngroups += __popc(b);
                // rank of this pick among equal experts, in pick order
                const int key = valid ? id : -1 - lane;
                const unsigned m = __match_any_sync(0xffffffffu, key);
                int rank = 0;
                if (valid) rank = e_count[id] + __popc(m & lt);
                __syncwarp();
                if (valid && (m >> lane) == 1u) e_count[id] += __popc(m);  // highest lane of its set
                if (j < n) rcol[(j / K) * K1 + 1 + (j % K)] = valid ? rank : -1;
                __syncwarp();
            }
            // column counts and first columns (prefix sum in group order)
            int run = 0;
            for (int base = 0; base < ngroups; base += 32) {
                const int g = base + lane;
                int cnt = 0;
                if (g < ngroups) cnt = (g == 0) ? T : e_count[gexp[g]];
                int incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (g < ngroups) {
                    gn[g] = cnt;
                    g0[g] = run + incl - cnt;
                }
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                tab.G() = ngroups;
                tab.U() = run;
            }
        } else if (lane == 0) {
            tab.G() = 0;
            tab.U() = 0;
        }
    }
    gt_sync(bar, nthr);

    if (!no_dedup && T > 0) {
        for (int t = tid; t < T; t += nthr) {
            rcol[t * K1] = t;  // the shared group's columns are 0..T-1 in row order
            crow[t] = t;
        }
        for (int j = tid; j < n; j += nthr) {
            const int id = sid[j], t = j / K, p = j - t * K;
            if (id < 0 || id >= E) continue;
            const int c = g0[e_group[id]] + rcol[t * K1 + 1 + p];
            rcol[t * K1 + 1 + p] = c;
            crow[c] = t;
        }
    }
    gt_sync(bar, nthr);
}

}  // namespace moe
