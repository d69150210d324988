// The Engram Sinkhorn of the TileKernels release: row / column L2 scaling of a [rows, head_dim]
// fp32 matrix, as the four calls of the TileLang tutorial, ch. 34 "TileKernels: Engram and mHC",
// sec. 5.3 (the Engram version: four kernels for row/column L2 scaling).
//
//   momentum:  m = beta1 m + g (in place), input = g + beta1 m with Nesterov, else m.  The pages
//              name the call's arguments, not its update; this is the plainest momentum reading.
//   step:      x = row_scale[r] * matrix[r, :] (*) col_scale, row_norm[r] = ||x||, row_scale[r]
//              divided by (row_norm[r] + eps) in place, and per partial p the column sums of
//              squares of x / (row_norm + eps) over its rows, written to col_sumsq_partial[p, :].
//   reduce:    the partials summed in a fixed order; optionally the column step
//              col_scale /= sqrt(col_sumsq) + eps, which the sec. 5.3 walk-through alternates
//              with the row step, applied in the same pass.
//   finalize:  out[r, :] = alpha * x / (||x|| + eps).
//
// GB300 design.  The row kernels stream whole rows through a ring of shared-memory stages that a
// producer warp fills with 1-D bulk (TMA) copies.  Two consumer groups of four warps take
// alternate rows: a group works on one row at a time with all of its threads (as the pages' kernel
// does with the whole CTA), and the two groups' per-row reduction chains overlap, which a single
// row-at-a-time CTA cannot do.  A consumer thread owns the float4 column vectors gt, gt + 128, ...
// (gt its index in the group) of every row, so col_scale and the column accumulators stay in
// registers.  Each row costs one barrier of its group, which carries the row norm's cross-warp
// partials and the timeout consensus; the stage is then released to the producer.  The producer
// also delivers each row's row_scale next to its stage, so no consumer waits on a global load.
//
// Partial p holds rows [p * C, min(rows, (p + 1) * C)), C = ceil(rows / P).  Within a partial,
// group 0 sums the rows of even offset and group 1 those of odd offset, each in ascending order,
// and the partial is group 0's sum plus group 1's.  That order depends on rows and P only, so the
// partials and the reduced columns are bitwise reproducible for any grid.
#include <algorithm>

#include "colsum.cuh"
#include "gate_pipeline.cuh"

namespace engram {

constexpr int kSkGroupThreads = 128;                    // one consumer group: 4 warps
constexpr int kSkGroupWarps = kSkGroupThreads / 32;
constexpr int kSkConsumers = 2 * kSkGroupThreads;
constexpr int kSkThreads = kSkConsumers + 32;           // + the producer warp
constexpr int kSkMaxVpt = 16;                           // float4 vectors per thread: head_dim <= 4 * 16 * 128
constexpr int kSkMaxHeadDim = 4 * kSkMaxVpt * kSkGroupThreads;
constexpr int kSkMaxStages = 32;

struct SinkhornParams {
    const float *matrix;
    const float *row_scale_in;  // the step reads and rewrites row_scale: then row_scale_out == row_scale_in
    float *row_scale_out;
    const float *col_scale;
    float *row_norm;            // step, nullable
    float *partial;             // step: [P, d]
    float *out;                 // finalize: [rows, d]
    uint32_t *status;
    int64_t rows;
    int64_t chunk;              // step: rows per partial
    int32_t P;
    int32_t d;
    int32_t stages;
    float eps;
    float alpha;
};

// Shared memory: ring [S][row] | exchange row (step only) | full [S] | empty [S] |
// row_scale per stage [S] | row-norm partials [2 groups][2][4 warps].  S as large as fits.
inline int sk_smem_bytes(int stages, int64_t row_bytes, bool exchange) {
    return static_cast<int>(stages * row_bytes + (exchange ? row_bytes : 0)) + stages * 20 + 2 * 2 * kSkGroupWarps * 4;
}

inline int sk_stages(int64_t row_bytes, bool exchange, int smem_limit) {
    int s = kSkMaxStages;
    while (s > 2 && sk_smem_bytes(s, row_bytes, exchange) > smem_limit) --s;
    return s;
}

struct SkShared {
    uint8_t *ring;
    float4 *xrow;      // the step's exchange row for combining the two groups' partial sums
    uint64_t *full;
    uint64_t *empty;
    float *rs;         // row_scale of the row in each stage, written by the producer
    float *red;
    uint32_t row_bytes;
    int S;
};

__device__ __forceinline__ SkShared sk_carve(uint8_t *smem, const SinkhornParams &p, bool exchange) {
    SkShared sh;
    sh.row_bytes = static_cast<uint32_t>(p.d) * 4u;
    sh.S = p.stages;
    sh.ring = smem;
    uint8_t *q = smem + static_cast<size_t>(sh.S) * sh.row_bytes;
    sh.xrow = reinterpret_cast<float4 *>(q);
    if (exchange) q += sh.row_bytes;
    sh.full = reinterpret_cast<uint64_t *>(q);
    sh.empty = sh.full + sh.S;
    sh.rs = reinterpret_cast<float *>(sh.empty + sh.S);
    sh.red = sh.rs + sh.S;
    return sh;
}

// The producer warp: copies the CTA's n rows in order into the ring.  They start at row `first`
// and come in runs of run_rows consecutive rows, a run's end `gap` rows before the next run's
// start, so each row's address advances without a division.  The lanes also load row_scale for
// the rows, 32 at a time and one batch ahead (row_of maps the CTA's q-th row to its matrix row),
// and lane 0 parks each row's value next to its stage before arming the stage's barrier, whose
// completion publishes it.  A stage is refilled once the consumer group that read it has
// released it.  Before returning, lane 0 waits (bounded) for its copies still in flight, so none
// lands after the CTA has exited.
template <typename RowOf>
__device__ __forceinline__ void sk_produce(const SkShared &sh, const SinkhornParams &p, int64_t n, int64_t first,
                                           int64_t run_rows, int64_t gap, RowOf row_of) {
    const int lane = threadIdx.x & 31;
    const uint64_t pol = l2_evict_first_policy();
    const float *src = p.matrix + static_cast<size_t>(first) * p.d;
    int64_t left = run_rows, q = 0;
    int stage = 0;
    uint32_t round = 0;
    float rs_batch = 0.f, rs_next = lane < n ? p.row_scale_in[row_of(lane)] : 0.f;
    for (; q < n; ++q) {
        const int slot = static_cast<int>(q & 31);
        if (slot == 0) {
            rs_batch = rs_next;
            const int64_t qn = q + 32 + lane;
            rs_next = qn < n ? p.row_scale_in[row_of(qn)] : 0.f;
        }
        const bool ok = __all_sync(0xffffffffu, round == 0 || mbar_wait(&sh.empty[stage], (round - 1) & 1u));
        if (!ok) {
            if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        const float rs = __shfl_sync(0xffffffffu, rs_batch, slot);
        if (lane == 0) {
            sh.rs[stage] = rs;
            mbar_arrive_expect_tx(&sh.full[stage], sh.row_bytes);
            bulk_load(sh.ring + static_cast<size_t>(stage) * sh.row_bytes, src, sh.row_bytes, &sh.full[stage], pol);
        }
        src += p.d;
        if (--left == 0) {
            src += gap * p.d;
            left = run_rows;
        }
        if (++stage == sh.S) {
            stage = 0;
            ++round;
        }
    }
    if (lane == 0)
        for (int64_t k = q > sh.S ? q - sh.S : 0; k < q; ++k)
            if (!mbar_wait(&sh.full[k % sh.S], static_cast<uint32_t>((k / sh.S) & 1)))
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
}

// A consumer group's position in the ring: the stage and phase of the CTA's j-th row, moved
// forward by small steps.
struct SkSlot {
    int64_t j;
    int s;
    uint32_t phase;
    __device__ __forceinline__ void move_to(int64_t target, int S) {
        s += static_cast<int>(target - j);
        j = target;
        while (s >= S) {
            s -= S;
            phase ^= 1u;
        }
    }
};

// Loads stage s into x[] (scaled by rs and the column scales) and returns this thread's sum of
// squares; x is zero where the thread has no column or the wait failed.
template <int VPT>
__device__ __forceinline__ float sk_load_row(const SkShared &sh, int s, int gt, float rs, const float4 (&cs)[VPT],
                                             int d4, bool ok, float4 (&x)[VPT]) {
    const uint8_t *src = sh.ring + static_cast<size_t>(s) * sh.row_bytes;
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
        const int jj = gt + m * kSkGroupThreads;
        if (ok && jj < d4) {
            const uint4 u = ld_shared_v4(src + static_cast<size_t>(jj) * 16);
            x[m] = make_float4(__uint_as_float(u.x) * rs * cs[m].x, __uint_as_float(u.y) * rs * cs[m].y,
                               __uint_as_float(u.z) * rs * cs[m].z, __uint_as_float(u.w) * rs * cs[m].w);
        } else {
            x[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ss += fmaf(x[m].x, x[m].x, x[m].y * x[m].y) + fmaf(x[m].z, x[m].z, x[m].w * x[m].w);
    }
    return ss;
}

// The group-wide sum of the per-thread values, after the group barrier `id` (which also ORs the
// threads' failure flags).  Returns false when a thread of the group failed.
__device__ __forceinline__ bool sk_group_total(const SkShared &sh, int g, int gw, int lane, int parity, float ss,
                                               bool ok, float *total) {
    ss = warp_sum(ss);
    float *red = sh.red + (g * 2 + parity) * kSkGroupWarps;
    if (lane == 0) red[gw] = ss;
    if (named_sync_or(1 + g, kSkGroupThreads, !ok)) return false;
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < kSkGroupWarps; ++q) t += red[q];
    *total = t;
    return true;
}

template <int VPT>
__device__ __forceinline__ void sk_load_col_scale(const float *col_scale, int gt, int d4, float4 (&cs)[VPT]) {
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
        const int jj = gt + m * kSkGroupThreads;
        cs[m] = jj < d4 ? __ldg(reinterpret_cast<const float4 *>(col_scale) + jj) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// ------------------------------------------------------------------------------- the row step

template <int VPT>
__global__ void __launch_bounds__(kSkThreads, 1) sinkhorn_step_kernel(const __grid_constant__ SinkhornParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SkShared sh = sk_carve(smem, p, true);
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t G = gridDim.x, C = p.chunk;

    // This CTA owns the partials blockIdx.x, blockIdx.x + G, ...; all but the matrix's last
    // non-empty partial are full, so they are runs of C rows, (G - 1) C rows apart.
    int64_t n_my = 0;
    for (int64_t pp = blockIdx.x; pp < p.P; pp += G) {
        const int64_t t0 = pp * C;
        n_my += t0 >= p.rows ? 0 : (t0 + C < p.rows ? C : p.rows - t0);
    }
    if (tid == 0) {
        for (int q = 0; q < sh.S; ++q) {
            mbar_init(&sh.full[q], 1);
            mbar_init(&sh.empty[q], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();  // barriers initialised
    if (tid >= kSkConsumers) {
        sk_produce(sh, p, n_my, blockIdx.x * C, C, (G - 1) * C,
                   [&](int64_t q) { return (blockIdx.x + (q / C) * G) * C + q % C; });
        return;
    }

    const int g = tid / kSkGroupThreads, gt = tid % kSkGroupThreads, gw = gt >> 5;
    const int d4 = p.d >> 2;
    float4 cs[VPT];
    sk_load_col_scale<VPT>(p.col_scale, gt, d4, cs);

    SkSlot slot{0, 0, 0};
    int parity = 0;
    bool failed = false;
    int64_t jbase = 0;
    for (int64_t pp = blockIdx.x; pp < p.P; pp += G, jbase += C) {
        const int64_t t0 = pp * C;
        const int64_t len = t0 >= p.rows ? 0 : (t0 + C < p.rows ? C : p.rows - t0);
        float4 acc[VPT];
#pragma unroll
        for (int m = 0; m < VPT; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t i = g; i < len && !failed; i += 2) {
            slot.move_to(jbase + i, sh.S);
            const bool ok = mbar_wait(&sh.full[slot.s], slot.phase);
            const float rs = sh.rs[slot.s];
            float4 x[VPT];
            const float ss = sk_load_row<VPT>(sh, slot.s, gt, rs, cs, d4, ok, x);
            float tot;
            if (!sk_group_total(sh, g, gw, lane, parity, ss, ok, &tot)) {
                failed = true;
                break;
            }
            parity ^= 1;
            if (gt == 0) mbar_arrive(&sh.empty[slot.s]);  // the group holds the row in registers
            const float nrm = sqrtf(tot);
            const float inv = 1.0f / (nrm + p.eps);
            if (gt == 0) {
                if (p.row_norm) p.row_norm[t0 + i] = nrm;
                p.row_scale_out[t0 + i] = rs * inv;
            }
#pragma unroll
            for (int m = 0; m < VPT; ++m) {
                const float4 y = make_float4(x[m].x * inv, x[m].y * inv, x[m].z * inv, x[m].w * inv);
                acc[m].x = fmaf(y.x, y.x, acc[m].x);
                acc[m].y = fmaf(y.y, y.y, acc[m].y);
                acc[m].z = fmaf(y.z, y.z, acc[m].z);
                acc[m].w = fmaf(y.w, y.w, acc[m].w);
            }
        }
        // partial = (group 0's rows) + (group 1's rows): group 1 parks its sum in the exchange row,
        // group 0 adds its own and writes the partial; the second barrier frees the exchange row
        if (g == 1 && !failed) {
#pragma unroll
            for (int m = 0; m < VPT; ++m) {
                const int jj = gt + m * kSkGroupThreads;
                if (jj < d4) sh.xrow[jj] = acc[m];
            }
        }
        if (named_sync_or(3, kSkConsumers, failed)) {
            if (tid == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        if (g == 0) {
            float4 *prow = reinterpret_cast<float4 *>(p.partial + static_cast<size_t>(pp) * p.d);
#pragma unroll
            for (int m = 0; m < VPT; ++m) {
                const int jj = gt + m * kSkGroupThreads;
                if (jj < d4) {
                    const float4 o = sh.xrow[jj];
                    prow[jj] = make_float4(acc[m].x + o.x, acc[m].y + o.y, acc[m].z + o.z, acc[m].w + o.w);
                }
            }
        }
        named_sync(4, kSkConsumers);
    }
}

// ------------------------------------------------------------------------------- finalize

template <int VPT>
__global__ void __launch_bounds__(kSkThreads, 1) sinkhorn_finalize_kernel(const __grid_constant__ SinkhornParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const SkShared sh = sk_carve(smem, p, false);
    const int tid = threadIdx.x, lane = tid & 31;
    // a contiguous, balanced range of rows per CTA; the groups take alternate rows of it
    const int64_t r0 = p.rows * blockIdx.x / gridDim.x;
    const int64_t n_my = p.rows * (blockIdx.x + 1) / gridDim.x - r0;
    if (tid == 0) {
        for (int q = 0; q < sh.S; ++q) {
            mbar_init(&sh.full[q], 1);
            mbar_init(&sh.empty[q], 1);
        }
        mbar_init_fence();
    }
    __syncthreads();  // barriers initialised
    if (tid >= kSkConsumers) {
        sk_produce(sh, p, n_my, r0, n_my, 0, [&](int64_t q) { return r0 + q; });
        return;
    }

    const int g = tid / kSkGroupThreads, gt = tid % kSkGroupThreads, gw = gt >> 5;
    const int d4 = p.d >> 2;
    float4 cs[VPT];
    sk_load_col_scale<VPT>(p.col_scale, gt, d4, cs);

    SkSlot slot{0, 0, 0};
    int parity = 0;
    for (int64_t j = g; j < n_my; j += 2) {
        slot.move_to(j, sh.S);
        const bool ok = mbar_wait(&sh.full[slot.s], slot.phase);
        float4 x[VPT];
        const float ss = sk_load_row<VPT>(sh, slot.s, gt, sh.rs[slot.s], cs, d4, ok, x);
        float tot;
        if (!sk_group_total(sh, g, gw, lane, parity, ss, ok, &tot)) {
            if (gt == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        parity ^= 1;
        if (gt == 0) mbar_arrive(&sh.empty[slot.s]);
        const float f = p.alpha / (sqrtf(tot) + p.eps);
        float4 *orow = reinterpret_cast<float4 *>(p.out + static_cast<size_t>(r0 + j) * p.d);
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int jj = gt + m * kSkGroupThreads;
            if (jj < d4) __stcs(orow + jj, make_float4(x[m].x * f, x[m].y * f, x[m].z * f, x[m].w * f));
        }
    }
}

// ------------------------------------------------------------------------------- ordered reduction

// S = sum_p partial[p] (column_sums: an order that depends on P only).  With col_scale given,
// col_scale[c] /= sqrt(S[c]) + eps in place.
__global__ void __launch_bounds__(kColThreads, 1)
    sinkhorn_reduce_kernel(const float4 *__restrict__ part, int32_t P, int32_t d4, float4 *__restrict__ col_sumsq,
                           float4 *__restrict__ col_scale, float eps) {
    __shared__ ColSumSmem sm;
    column_sums(part, P, d4, sm, [&](int col, const float4 &t) {
        if (col_sumsq) col_sumsq[col] = t;
        if (col_scale) {
            float4 c = col_scale[col];
            c.x /= sqrtf(t.x) + eps;
            c.y /= sqrtf(t.y) + eps;
            c.z /= sqrtf(t.z) + eps;
            c.w /= sqrtf(t.w) + eps;
            col_scale[col] = c;
        }
    });
}

// ------------------------------------------------------------------------------- momentum

// Chunks of kMomChunk elements (grad and momentum) reach shared memory by two 1-D bulk (TMA) copies
// each, kMomStages chunks in flight per CTA, thread 0 issuing; a thread updates eight elements of a
// chunk and writes momentum and the Sinkhorn input straight to global memory.  Chunk c of the n8
// groups of eight goes to CTA c mod grid.  The n % 8 tail is done element by element.
constexpr int kMomChunk = 2048;   // elements per chunk: 256 threads x 8
constexpr int kMomStages = 4;

__host__ __device__ inline int sk_mom_smem(int gsize) { return kMomStages * kMomChunk * (gsize + 4) + kMomStages * 8; }

template <typename G>
__device__ __forceinline__ void sk_unpack8(const uint8_t *src, float (&g)[8]);

template <>
__device__ __forceinline__ void sk_unpack8<float>(const uint8_t *src, float (&g)[8]) {
    const uint4 a = ld_shared_v4(src), b = ld_shared_v4(src + 16);
    g[0] = __uint_as_float(a.x), g[1] = __uint_as_float(a.y), g[2] = __uint_as_float(a.z), g[3] = __uint_as_float(a.w);
    g[4] = __uint_as_float(b.x), g[5] = __uint_as_float(b.y), g[6] = __uint_as_float(b.z), g[7] = __uint_as_float(b.w);
}

template <>
__device__ __forceinline__ void sk_unpack8<__nv_bfloat16>(const uint8_t *src, float (&g)[8]) {
    Vec<__nv_bfloat16>::unpack(ld_shared_v4(src), g);
}

template <typename G>
__global__ void __launch_bounds__(256) sinkhorn_momentum_kernel(const G *__restrict__ grad, float *__restrict__ m,
                                                                float *__restrict__ out, int64_t n, float beta,
                                                                int nesterov, uint32_t *status) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int gsize = static_cast<int>(sizeof(G));
    const int tid = threadIdx.x;
    const size_t stage_bytes = static_cast<size_t>(kMomChunk) * (gsize + 4);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kMomStages * stage_bytes);
    const int64_t n8 = n >> 3;
    const int64_t nchunks = (n8 * 8 + kMomChunk - 1) / kMomChunk;
    const int64_t G_ = gridDim.x;
    const int64_t n_my = blockIdx.x < nchunks ? (nchunks - 1 - blockIdx.x) / G_ + 1 : 0;
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t k) {  // thread 0: this CTA's k-th chunk into stage k % kMomStages
        const int64_t c = blockIdx.x + k * G_;
        const int64_t e0 = c * kMomChunk;
        const int64_t cnt = n8 * 8 - e0 < kMomChunk ? n8 * 8 - e0 : kMomChunk;  // a multiple of 8
        uint8_t *dst = smem + static_cast<size_t>(k % kMomStages) * stage_bytes;
        uint64_t *bar = &full[k % kMomStages];
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt * (gsize + 4)));
        bulk_load(dst, grad + e0, static_cast<uint32_t>(cnt * gsize), bar, pol);
        bulk_load(dst + static_cast<size_t>(kMomChunk) * gsize, m + e0, static_cast<uint32_t>(cnt * 4), bar, pol);
    };
    int64_t issued = 0;
    if (tid == 0) {
        for (int q = 0; q < kMomStages; ++q) mbar_init(&full[q], 1);
        mbar_init_fence();
        for (; issued < kMomStages && issued < n_my; ++issued) issue(issued);
    }
    __syncthreads();
    int64_t k = 0;
    for (; k < n_my; ++k) {
        const int st = static_cast<int>(k % kMomStages);
        const bool ok = mbar_wait(&full[st], static_cast<uint32_t>((k / kMomStages) & 1));
        const int64_t e0 = (blockIdx.x + k * G_) * kMomChunk;
        const int64_t e = e0 + tid * 8;
        const uint8_t *stg = smem + static_cast<size_t>(st) * stage_bytes;
        if (ok && e < n8 * 8) {
            float g[8], mo[8];
            sk_unpack8<G>(stg + static_cast<size_t>(tid) * 8 * gsize, g);
            sk_unpack8<float>(stg + static_cast<size_t>(kMomChunk) * gsize + static_cast<size_t>(tid) * 32, mo);
            float mn[8], o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                mn[q] = fmaf(beta, mo[q], g[q]);
                o[q] = nesterov ? fmaf(beta, mn[q], g[q]) : mn[q];
            }
            float4 *mv = reinterpret_cast<float4 *>(m + e);
            float4 *ov = reinterpret_cast<float4 *>(out + e);
            mv[0] = make_float4(mn[0], mn[1], mn[2], mn[3]);
            mv[1] = make_float4(mn[4], mn[5], mn[6], mn[7]);
            __stcs(ov, make_float4(o[0], o[1], o[2], o[3]));
            __stcs(ov + 1, make_float4(o[4], o[5], o[6], o[7]));
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report(status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        // every thread has read its part of the stage: refill it
        if (tid == 0 && issued < n_my) issue(issued++);
    }
    if (tid == 0)  // copies issued but not consumed (after a timeout) land before the CTA leaves
        for (int64_t q = k; q < issued; ++q)
            if (!mbar_wait(&full[q % kMomStages], static_cast<uint32_t>((q / kMomStages) & 1)))
                report(status, nullptr, ENGRAM_DEVERR_TIMEOUT);
    if (blockIdx.x == 0 && tid < (n & 7)) {
        const int64_t i = (n8 << 3) + tid;
        const float g = static_cast<float>(grad[i]);
        const float mn = fmaf(beta, m[i], g);
        m[i] = mn;
        out[i] = nesterov ? fmaf(beta, mn, g) : mn;
    }
}

// ------------------------------------------------------------------------------- launchers

namespace {

engram_status sk_check_shape(const char *fn, int64_t rows, int32_t head_dim) {
    if (rows < 0 || head_dim <= 0)
        return fail(ENGRAM_ERR_SHAPE, "%s: rows = %lld, head_dim = %d", fn, (long long)rows, head_dim);
    if (head_dim % 4 != 0) return fail(ENGRAM_ERR_ALIGN, "%s: head_dim = %d is not a multiple of 4", fn, head_dim);
    if (head_dim > kSkMaxHeadDim)
        return fail(ENGRAM_ERR_SHAPE, "%s: head_dim = %d exceeds %d", fn, head_dim, kSkMaxHeadDim);
    return ENGRAM_OK;
}

// 16-byte alignment and device residency of the non-NULL pointers among the first `n_aligned`
// (which the kernels read or write as 16-byte vectors), device residency of the rest.
engram_status sk_check_ptrs(const char *fn, const void *const *ptrs, int n, int n_aligned, DeviceInfo *dev) {
    for (int i = 0; i < n_aligned; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(ENGRAM_ERR_ALIGN, "%s: pointer argument %d is not 16-byte aligned", fn, i);
    engram_status st = current_device(dev);
    if (st != ENGRAM_OK) return st;
    for (int i = 0; i < n; ++i)
        if (ptrs[i] && (st = check_device_ptr(ptrs[i], dev->device, fn)) != ENGRAM_OK) return st;
    return ENGRAM_OK;
}

using SkKernel = void (*)(SinkhornParams);

// VPT is instantiated for 1..6, 8, 10, 12 and 16 vectors per thread; a head_dim takes the
// smallest that covers it.
constexpr int kSkVpts[] = {1, 2, 3, 4, 5, 6, 8, 10, 12, 16};

int sk_vpt(int32_t head_dim) {
    const int need = (head_dim / 4 + kSkGroupThreads - 1) / kSkGroupThreads;
    for (int v : kSkVpts)
        if (v >= need) return v;
    return 0;
}

template <template <int> class Tag>
SkKernel sk_pick(int vpt);

template <int V>
struct StepTag {
    static constexpr SkKernel k = sinkhorn_step_kernel<V>;
};
template <int V>
struct FinTag {
    static constexpr SkKernel k = sinkhorn_finalize_kernel<V>;
};

template <template <int> class Tag>
SkKernel sk_pick(int vpt) {
    switch (vpt) {
        case 1: return Tag<1>::k;
        case 2: return Tag<2>::k;
        case 3: return Tag<3>::k;
        case 4: return Tag<4>::k;
        case 5: return Tag<5>::k;
        case 6: return Tag<6>::k;
        case 8: return Tag<8>::k;
        case 10: return Tag<10>::k;
        case 12: return Tag<12>::k;
        default: return Tag<16>::k;
    }
}

// Launches a row kernel on min(units, SMs) CTAs: one per SM, the ring takes most of its memory.
engram_status sk_launch(const char *fn, SkKernel kernel, SinkhornParams prm, bool exchange, int64_t units,
                        const DeviceInfo &dev, engram_stream_t stream) {
    const int64_t row_bytes = static_cast<int64_t>(prm.d) * 4;
    prm.stages = sk_stages(row_bytes, exchange, dev.smem_optin);
    const int smem = sk_smem_bytes(prm.stages, row_bytes, exchange);
    if (smem > dev.smem_optin)
        return fail(ENGRAM_ERR_SHAPE, "%s: %d bytes of shared memory exceed %d", fn, smem, dev.smem_optin);
    engram_status st = set_smem(reinterpret_cast<const void *>(kernel), smem);
    if (st != ENGRAM_OK) return st;
    const int64_t grid = cap_grid(std::min<int64_t>(units, dev.num_sms));
    kernel<<<static_cast<unsigned>(grid), kSkThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(prm);
    return check_launch(fn);
}



}  // namespace
}  // namespace engram

using namespace engram;

extern "C" engram_status engram_sinkhorn_momentum_update(const void *grad, engram_dtype dtype, float *momentum,
                                                         float *sinkhorn_input, int64_t n, float beta1,
                                                         int32_t nesterov, engram_stream_t stream) {
    const char *fn = "engram_sinkhorn_momentum_update";
    if (n < 0) return fail(ENGRAM_ERR_SHAPE, "%s: n = %lld", fn, (long long)n);
    if (dtype_size(dtype) == 0) return fail(ENGRAM_ERR_DTYPE, "%s: dtype %d", fn, (int)dtype);
    if (n == 0) return ENGRAM_OK;
    if (!grad || !momentum || !sinkhorn_input) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (sinkhorn_input == momentum) return fail(ENGRAM_ERR_SHAPE, "%s: sinkhorn_input may not alias momentum", fn);
    const void *ptrs[] = {grad, momentum, sinkhorn_input};
    DeviceInfo dev;
    engram_status st = sk_check_ptrs(fn, ptrs, 3, 3, &dev);
    if (st != ENGRAM_OK) return st;
    const int64_t nchunks = std::max<int64_t>(1, ((n >> 3) * 8 + kMomChunk - 1) / kMomChunk);
    const int64_t blocks = cap_grid(std::min<int64_t>(nchunks, static_cast<int64_t>(dev.num_sms) * 2));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == ENGRAM_F32) {
        const int smem = sk_mom_smem(4);
        if ((st = set_smem(reinterpret_cast<const void *>(sinkhorn_momentum_kernel<float>), smem)) != ENGRAM_OK)
            return st;
        sinkhorn_momentum_kernel<float><<<static_cast<unsigned>(blocks), 256, smem, s>>>(
            static_cast<const float *>(grad), momentum, sinkhorn_input, n, beta1, nesterov != 0, dev.status_word);
    } else {
        const int smem = sk_mom_smem(2);
        if ((st = set_smem(reinterpret_cast<const void *>(sinkhorn_momentum_kernel<__nv_bfloat16>), smem)) !=
            ENGRAM_OK)
            return st;
        sinkhorn_momentum_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, smem, s>>>(
            static_cast<const __nv_bfloat16 *>(grad), momentum, sinkhorn_input, n, beta1, nesterov != 0,
            dev.status_word);
    }
    return check_launch(fn);
}

extern "C" engram_status engram_sinkhorn_num_partials(int64_t rows, int32_t head_dim, int32_t *P) {
    if (!P) return fail(ENGRAM_ERR_NULL, "engram_sinkhorn_num_partials: NULL P");
    if (rows < 0 || head_dim <= 0)
        return fail(ENGRAM_ERR_SHAPE, "engram_sinkhorn_num_partials: rows = %lld, head_dim = %d", (long long)rows,
                    head_dim);
    // 16 or more rows per partial (a partial row costs 1/16 of their bytes or less) and at most
    // 1024 partials.
    const int64_t chunk = std::max<int64_t>(16, (rows + 1023) / 1024);
    *P = static_cast<int32_t>(std::max<int64_t>(1, (rows + chunk - 1) / chunk));
    return ENGRAM_OK;
}

extern "C" engram_status engram_sinkhorn_step(const float *matrix, float *row_scale, const float *col_scale,
                                              int64_t rows, int32_t head_dim, float eps, float *row_norm,
                                              float *col_sumsq_partial, int32_t P, engram_stream_t stream) {
    const char *fn = "engram_sinkhorn_step";
    engram_status st = sk_check_shape(fn, rows, head_dim);
    if (st != ENGRAM_OK) return st;
    if (P < 1) return fail(ENGRAM_ERR_SHAPE, "%s: P = %d", fn, P);
    if (!col_scale || !col_sumsq_partial || (rows > 0 && (!matrix || !row_scale)))
        return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    const void *ptrs[] = {matrix, col_scale, col_sumsq_partial, row_scale, row_norm};
    DeviceInfo dev;
    if ((st = sk_check_ptrs(fn, ptrs, 5, 3, &dev)) != ENGRAM_OK) return st;
    SinkhornParams prm{};
    prm.matrix = matrix;
    prm.row_scale_in = row_scale;
    prm.row_scale_out = row_scale;
    prm.col_scale = col_scale;
    prm.row_norm = row_norm;
    prm.partial = col_sumsq_partial;
    prm.status = dev.status_word;
    prm.rows = rows;
    prm.chunk = rows == 0 ? 1 : (rows + P - 1) / P;
    prm.P = P;
    prm.d = head_dim;
    prm.eps = eps;
    return sk_launch(fn, sk_pick<StepTag>(sk_vpt(head_dim)), prm, true, P, dev, stream);
}

extern "C" engram_status engram_sinkhorn_step_reduce(const float *col_sumsq_partial, int32_t P, int32_t head_dim,
                                                     float *col_sumsq, float *col_scale, float eps,
                                                     engram_stream_t stream) {
    const char *fn = "engram_sinkhorn_step_reduce";
    engram_status st = sk_check_shape(fn, 0, head_dim);
    if (st != ENGRAM_OK) return st;
    if (P < 1) return fail(ENGRAM_ERR_SHAPE, "%s: P = %d", fn, P);
    if (!col_sumsq_partial || (!col_sumsq && !col_scale)) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    const void *ptrs[] = {col_sumsq_partial, col_sumsq, col_scale};
    DeviceInfo dev;
    if ((st = sk_check_ptrs(fn, ptrs, 3, 3, &dev)) != ENGRAM_OK) return st;
    const int d4 = head_dim / 4;
    sinkhorn_reduce_kernel<<<column_sum_grid(d4, dev.num_sms), kColThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4 *>(col_sumsq_partial), P, d4, reinterpret_cast<float4 *>(col_sumsq),
        reinterpret_cast<float4 *>(col_scale), eps);
    return check_launch(fn);
}

extern "C" engram_status engram_sinkhorn_finalize(const float *matrix, const float *row_scale,
                                                  const float *col_scale, int64_t rows, int32_t head_dim, float eps,
                                                  float alpha, float *out, engram_stream_t stream) {
    const char *fn = "engram_sinkhorn_finalize";
    engram_status st = sk_check_shape(fn, rows, head_dim);
    if (st != ENGRAM_OK) return st;
    if (rows == 0) return ENGRAM_OK;
    if (!matrix || !row_scale || !col_scale || !out) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (out == matrix) return fail(ENGRAM_ERR_SHAPE, "%s: out may not alias matrix", fn);
    const void *ptrs[] = {matrix, col_scale, out, row_scale};
    DeviceInfo dev;
    if ((st = sk_check_ptrs(fn, ptrs, 4, 3, &dev)) != ENGRAM_OK) return st;
    SinkhornParams prm{};
    prm.matrix = matrix;
    prm.row_scale_in = row_scale;
    prm.col_scale = col_scale;
    prm.out = out;
    prm.status = dev.status_word;
    prm.rows = rows;
    prm.d = head_dim;
    prm.eps = eps;
    prm.alpha = alpha;
    return sk_launch(fn, sk_pick<FinTag>(sk_vpt(head_dim)), prm, false, rows, dev, stream);
}
