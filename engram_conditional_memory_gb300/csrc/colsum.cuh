// Ordered column sums of partial rows: the reduction step shared by the gate's weight gradient, the
// short convolution's weight gradients and the Sinkhorn column step.
//
// For a row-major [P, d4] float4 array, column c's sum is taken in an order that depends on P only,
// so that it is bitwise reproducible on any grid and any device:
//   kColGroups row groups, group g summing rows [g R, min(P, (g + 1) R)), R = ceil(P / kColGroups),
//     in ascending order;
//   kColGroups / kColRun runs of kColRun consecutive group sums, each in ascending order;
//   the run sums in ascending order.
// A CTA of kColThreads threads, one per SM, owns a contiguous share of the columns (the shares differ
// by one column at most) and takes them up to kColCols at a time.  The (group, column) sums of a chunk
// are spread over the threads, item i being column i mod ncols of group i / ncols, and a thread walks
// its items' rows as one sequence in batches of kColBatch 16-byte loads that cross item boundaries:
// with few rows per group (small P) every load of a chunk is still in flight at once, and with many
// every SM keeps about 128 KB of partials in flight.  Which CTA owns a column, and which thread sums a
// group, does not change its sum.
#pragma once

#include "engram_internal.cuh"

namespace engram {

constexpr int kColGroups = 128;
constexpr int kColRun = 16;
constexpr int kColThreads = 1024;
constexpr int kColCols = 20;  // float4 columns per chunk (the chunk's group sums fill 40 KB of shared memory)
constexpr int kColBatch = 8;
static_assert(kColGroups % kColRun == 0, "runs of whole groups");

struct ColSumSmem {
    float4 group[kColGroups * kColCols];           // [group][column of the chunk]
    float4 run[(kColGroups / kColRun) * kColCols];  // [run][column of the chunk]
};

// This CTA's columns [c_begin, c_end) of d4 when the grid's CTAs split them evenly.
__device__ __forceinline__ void column_share(int d4, int &c_begin, int &c_end) {
    c_begin = static_cast<int>(static_cast<int64_t>(blockIdx.x) * d4 / gridDim.x);
    c_end = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * d4 / gridDim.x);
}

__device__ __forceinline__ void add4(float4 &t, const float4 &x) {
    t.x += x.x;
    t.y += x.y;
    t.z += x.z;
    t.w += x.w;
}

// The sums of this CTA's columns; epi(column, sum) is called once per column, by one thread.  Every
// thread of the CTA calls it (it synchronises the CTA).
template <typename Epi>
__device__ __forceinline__ void column_sums(const float4 *__restrict__ part, int P, int d4, ColSumSmem &sm,
                                            Epi &&epi) {
    const int tid = threadIdx.x;
    int c_begin, c_end;
    column_share(d4, c_begin, c_end);
    const int rows = (P + kColGroups - 1) / kColGroups;
    const int geff = rows > 0 ? (P + rows - 1) / rows : 0;  // groups with at least one row
    for (int cc = c_begin; cc < c_end; cc += kColCols) {
        const int ncols = c_end - cc < kColCols ? c_end - cc : kColCols;
        for (int i = geff * ncols + tid; i < kColGroups * ncols; i += kColThreads)  // groups without rows
            sm.group[(i / ncols) * kColCols + i % ncols] = make_float4(0.f, 0.f, 0.f, 0.f);
        const int nitems = geff * ncols;
        // issue cursor: item `it` = (group g, column j), next row p of [g rows, pend)
        int it = tid, g = it / ncols, j = it - g * ncols, p = g * rows;
        int pend = min(P, p + rows);
        // consume cursor: the same sequence, behind by the loads of one batch
        int cit = it, cg = g, cj = j, cp = p, cpend = pend;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        while (it < nitems) {
            float4 x[kColBatch];
#pragma unroll
            for (int b = 0; b < kColBatch; ++b) {
                if (it < nitems) {
                    x[b] = __ldcs(part + static_cast<size_t>(p) * d4 + cc + j);
                    if (++p == pend) {
                        it += kColThreads;
                        g = it / ncols;
                        j = it - g * ncols;
                        p = g * rows;
                        pend = min(P, p + rows);
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < kColBatch; ++b) {
                if (cit < nitems) {
                    add4(s, x[b]);
                    if (++cp == cpend) {
                        sm.group[cg * kColCols + cj] = s;
                        s = make_float4(0.f, 0.f, 0.f, 0.f);
                        cit += kColThreads;
                        cg = cit / ncols;
                        cj = cit - cg * ncols;
                        cp = cg * rows;
                        cpend = min(P, cp + rows);
                    }
                }
            }
        }
        __syncthreads();
        if (tid < ncols * (kColGroups / kColRun)) {
            const int u = tid / ncols;
            const int j = tid - u * ncols;
            float4 t = sm.group[(u * kColRun) * kColCols + j];
#pragma unroll
            for (int q = 1; q < kColRun; ++q) add4(t, sm.group[(u * kColRun + q) * kColCols + j]);
            sm.run[u * kColCols + j] = t;
        }
        __syncthreads();
        if (tid < ncols) {
            float4 t = sm.run[tid];
#pragma unroll
            for (int u = 1; u < kColGroups / kColRun; ++u) add4(t, sm.run[u * kColCols + tid]);
            epi(cc + tid, t);
        }
        __syncthreads();  // the chunk's sums are read before the next chunk's overwrite them
    }
}

// CTAs for column_sums over d4 columns: one per SM, no more than there are columns.
inline int column_sum_grid(int d4, int num_sms) { return static_cast<int>(cap_grid(d4 < num_sms ? (d4 > 0 ? d4 : 1) : num_sms)); }

}  // namespace engram
