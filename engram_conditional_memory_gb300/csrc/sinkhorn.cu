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
// GB300 design.  The row kernels stream whole rows through a ring of shared-memory stages filled
// by 1-D bulk (TMA) copies that thread 0 issues; a CTA works on one row at a time with all of its
// threads (as the pages' kernel does) while the next rows land.  A thread owns the float4 column
// vectors tid, tid + 256, ... of every row, so the column accumulators and col_scale stay in
// registers for the CTA's whole life.  One barrier per row carries the row norm's cross-warp
// partials, the timeout consensus and the release of the stage.  Partial p holds rows
// [p * C, min(rows, (p + 1) * C)), C = ceil(rows / P), summed in ascending order by whichever CTA
// owns it, so the partials and the reduced columns are bitwise reproducible for any grid.
#include <algorithm>

#include "engram_internal.cuh"

namespace engram {

constexpr int kSkThreads = 256;               // threads per CTA of the row kernels
constexpr int kSkWarps = kSkThreads / 32;
constexpr int kSkMaxVpt = 8;                  // float4 vectors per thread: head_dim <= 4 * 8 * 256
constexpr int kSkMaxHeadDim = 4 * kSkMaxVpt * kSkThreads;
constexpr int kSkMaxStages = 32;
constexpr int kSkRingBytes = 192 * 1024;      // shared memory for the ring of row stages

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

inline int sk_stages(int64_t row_bytes) {
    const int64_t s = kSkRingBytes / row_bytes;
    return static_cast<int>(s < 2 ? 2 : (s > kSkMaxStages ? kSkMaxStages : s));
}

// ring | full barriers [S] | row-norm partials [2][warps] | row_scale windows [2][threads]
inline int sk_smem_bytes(int stages, int64_t row_bytes) {
    return static_cast<int>(stages * row_bytes) + stages * 8 + 2 * kSkWarps * 4 + 2 * kSkThreads * 4;
}

// The ring of row stages shared by the step and the finalize kernels.
struct SkRing {
    uint8_t *stages;
    uint64_t *full;
    float *red;
    float *rsw;
    uint32_t row_bytes;
    int S;
    uint64_t pol;

    // Thread 0 only: copy one row into the stage of the CTA's j-th row and arm its barrier.
    __device__ __forceinline__ void issue(int64_t j, const float *src) const {
        uint64_t *bar = &full[j % S];
        mbar_arrive_expect_tx(bar, row_bytes);
        bulk_load(stages + static_cast<size_t>(j % S) * row_bytes, src, row_bytes, bar, pol);
    }
};

// Loads stage s into x[] (scaled by rs and the column scales) and returns this thread's sum of
// squares; x is zero where the thread has no column or the wait failed.
template <int VPT>
__device__ __forceinline__ float sk_load_row(const SkRing &ring, int s, float rs, const float4 (&cs)[VPT], int d4,
                                             bool ok, float4 (&x)[VPT]) {
    const uint8_t *src = ring.stages + static_cast<size_t>(s) * ring.row_bytes;
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
        const int jj = threadIdx.x + m * kSkThreads;
        if (ok && jj < d4) {
            const uint4 u = ld_shared_v4(src + static_cast<size_t>(jj) * 16);
            x[m] = make_float4(__uint_as_float(u.x) * rs * cs[m].x, __uint_as_float(u.y) * rs * cs[m].y,
                               __uint_as_float(u.z) * rs * cs[m].z, __uint_as_float(u.w) * rs * cs[m].w);
        } else {
            x[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ss = fmaf(x[m].x, x[m].x, fmaf(x[m].y, x[m].y, fmaf(x[m].z, x[m].z, fmaf(x[m].w, x[m].w, ss))));
    }
    return ss;
}

// Common prologue of the row kernels: carve shared memory, initialise the barriers, issue the
// first stages (thread 0) and load the column scales.
template <int VPT, typename RowOf>
__device__ __forceinline__ SkRing sk_prologue(const SinkhornParams &p, uint8_t *smem, int64_t n_my, RowOf row_of,
                                              float4 (&cs)[VPT], int64_t *issued) {
    SkRing ring;
    ring.row_bytes = static_cast<uint32_t>(p.d) * 4u;
    ring.S = p.stages;
    ring.stages = smem;
    ring.full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(ring.S) * ring.row_bytes);
    ring.red = reinterpret_cast<float *>(ring.full + ring.S);
    ring.rsw = ring.red + 2 * kSkWarps;
    ring.pol = l2_evict_first_policy();
    *issued = 0;
    if (threadIdx.x == 0) {
        for (int q = 0; q < ring.S; ++q) mbar_init(&ring.full[q], 1);
        mbar_init_fence();
        for (; *issued < ring.S && *issued < n_my; ++*issued)
            ring.issue(*issued, p.matrix + static_cast<size_t>(row_of(*issued)) * p.d);
    }
    const int d4 = p.d >> 2;
#pragma unroll
    for (int m = 0; m < VPT; ++m) {
        const int jj = threadIdx.x + m * kSkThreads;
        cs[m] = jj < d4 ? __ldg(reinterpret_cast<const float4 *>(p.col_scale) + jj) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return ring;
}

// Thread 0 waits (bounded) for the copies it issued that nobody consumed, so that no bulk copy
// lands in shared memory after the CTA has exited.
__device__ __forceinline__ void sk_drain(const SkRing &ring, int64_t consumed, int64_t issued, uint32_t *status) {
    if (threadIdx.x != 0) return;
    for (int64_t q = consumed; q < issued; ++q)
        if (!mbar_wait(&ring.full[q % ring.S], static_cast<uint32_t>((q / ring.S) & 1)))
            report(status, nullptr, ENGRAM_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------------------------- the row step

template <int VPT>
__global__ void __launch_bounds__(kSkThreads, 1) sinkhorn_step_kernel(const __grid_constant__ SinkhornParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d4 = p.d >> 2;
    const int64_t G = gridDim.x, C = p.chunk;

    // This CTA owns the partials blockIdx.x, blockIdx.x + G, ...; every one but the last non-empty
    // partial of the matrix is full, so the CTA's j-th row is found without a table.
    int64_t n_my = 0;
    for (int64_t pp = blockIdx.x; pp < p.P; pp += G) {
        const int64_t t0 = pp * C;
        n_my += t0 >= p.rows ? 0 : (t0 + C < p.rows ? C : p.rows - t0);
    }
    auto row_of = [&](int64_t j) { return (blockIdx.x + (j / C) * G) * C + j % C; };

    float4 cs[VPT];
    int64_t issued;
    const SkRing ring = sk_prologue<VPT>(p, smem, n_my, row_of, cs, &issued);
    // row_scale of this CTA's rows, one window of kSkThreads rows at a time, the next window's
    // load in flight while the current one is used.  row_scale is rewritten in place, but a row
    // is written only after it has been read.
    float rs_next = tid < n_my ? p.row_scale_in[row_of(tid)] : 0.f;
    __syncthreads();  // barriers initialised

    int64_t j = 0;
    int s = 0;
    uint32_t phase = 0;
    bool failed = false;
    for (int64_t pp = blockIdx.x; pp < p.P && !failed; pp += G) {
        const int64_t t0 = pp * C;
        const int64_t t1 = t0 + C < p.rows ? t0 + C : p.rows;
        float4 acc[VPT];
#pragma unroll
        for (int m = 0; m < VPT; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int64_t r = t0; r < t1; ++r, ++j) {
            const int wpos = static_cast<int>(j % kSkThreads);
            float *win = ring.rsw + ((j / kSkThreads) & 1) * kSkThreads;
            if (wpos == 0) {
                win[tid] = rs_next;
                const int64_t jn = j + kSkThreads + tid;
                rs_next = jn < n_my ? p.row_scale_in[row_of(jn)] : 0.f;
                __syncthreads();
            }
            const bool ok = mbar_wait(&ring.full[s], phase);
            const float rs = win[wpos];
            float4 x[VPT];
            const float ss = warp_sum(sk_load_row<VPT>(ring, s, rs, cs, d4, ok, x));
            float *red = ring.red + (j & 1) * kSkWarps;
            if (lane == 0) red[warp] = ss;
            if (__syncthreads_or(!ok)) {
                if (tid == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
                break;
            }
            // every thread holds its part of row j in registers: stage s can be refilled
            if (tid == 0 && issued < n_my) {
                ring.issue(issued, p.matrix + static_cast<size_t>(row_of(issued)) * p.d);
                ++issued;
            }
            if (++s == ring.S) {
                s = 0;
                phase ^= 1u;
            }
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < kSkWarps; ++q) tot += red[q];
            const float nrm = sqrtf(tot);
            const float inv = 1.0f / (nrm + p.eps);
            if (tid == 0) {
                if (p.row_norm) p.row_norm[r] = nrm;
                p.row_scale_out[r] = rs * inv;
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
        if (failed) break;
        float4 *prow = reinterpret_cast<float4 *>(p.partial + static_cast<size_t>(pp) * p.d);
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int jj = tid + m * kSkThreads;
            if (jj < d4) prow[jj] = acc[m];
        }
    }
    sk_drain(ring, j, issued, p.status);
}

// ------------------------------------------------------------------------------- finalize

template <int VPT>
__global__ void __launch_bounds__(kSkThreads, 1) sinkhorn_finalize_kernel(const __grid_constant__ SinkhornParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d4 = p.d >> 2;
    // a contiguous, balanced range of rows per CTA
    const int64_t r0 = p.rows * blockIdx.x / gridDim.x;
    const int64_t n_my = p.rows * (blockIdx.x + 1) / gridDim.x - r0;
    auto row_of = [&](int64_t j) { return r0 + j; };

    float4 cs[VPT];
    int64_t issued;
    const SkRing ring = sk_prologue<VPT>(p, smem, n_my, row_of, cs, &issued);
    float rs_next = tid < n_my ? __ldg(p.row_scale_in + r0 + tid) : 0.f;
    __syncthreads();  // barriers initialised

    int64_t j = 0;
    int s = 0;
    uint32_t phase = 0;
    for (; j < n_my; ++j) {
        const int wpos = static_cast<int>(j % kSkThreads);
        float *win = ring.rsw + ((j / kSkThreads) & 1) * kSkThreads;
        if (wpos == 0) {
            win[tid] = rs_next;
            const int64_t jn = j + kSkThreads + tid;
            rs_next = jn < n_my ? __ldg(p.row_scale_in + r0 + jn) : 0.f;
            __syncthreads();
        }
        const bool ok = mbar_wait(&ring.full[s], phase);
        float4 x[VPT];
        const float ss = warp_sum(sk_load_row<VPT>(ring, s, win[wpos], cs, d4, ok, x));
        float *red = ring.red + (j & 1) * kSkWarps;
        if (lane == 0) red[warp] = ss;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        if (tid == 0 && issued < n_my) {
            ring.issue(issued, p.matrix + static_cast<size_t>(row_of(issued)) * p.d);
            ++issued;
        }
        if (++s == ring.S) {
            s = 0;
            phase ^= 1u;
        }
        float tot = 0.f;
#pragma unroll
        for (int q = 0; q < kSkWarps; ++q) tot += red[q];
        const float f = p.alpha / (sqrtf(tot) + p.eps);
        float4 *orow = reinterpret_cast<float4 *>(p.out + static_cast<size_t>(r0 + j) * p.d);
#pragma unroll
        for (int m = 0; m < VPT; ++m) {
            const int jj = tid + m * kSkThreads;
            if (jj < d4) __stcs(orow + jj, make_float4(x[m].x * f, x[m].y * f, x[m].z * f, x[m].w * f));
        }
    }
    sk_drain(ring, j, issued, p.status);
}

// ------------------------------------------------------------------------------- ordered reduction

constexpr int kSkRG = 64;  // row groups of the partials
constexpr int kSkCV = 4;   // float4 columns per CTA

// Column c of S = sum_p partial[p, c]: thread group r sums partials [r * R, (r + 1) * R) in
// ascending order, then the 64 group sums are added in ascending order.  The order depends on P
// only.  With col_scale given, col_scale[c] /= sqrt(S) + eps in place.
__global__ void __launch_bounds__(kSkRG *kSkCV)
    sinkhorn_reduce_kernel(const float4 *__restrict__ part, int32_t P, int32_t d4, float4 *__restrict__ col_sumsq,
                           float4 *__restrict__ col_scale, float eps) {
    __shared__ float4 sums[kSkRG][kSkCV];
    const int cv = threadIdx.x % kSkCV;
    const int r = threadIdx.x / kSkCV;
    const int col = blockIdx.x * kSkCV + cv;
    const int per = (P + kSkRG - 1) / kSkRG;
    const int p0 = r * per;
    const int p1 = p0 + per < P ? p0 + per : P;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < d4) {
        for (int q = p0; q < p1; ++q) {
            const float4 x = __ldcs(part + static_cast<size_t>(q) * d4 + col);
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
    }
    sums[r][cv] = s;
    __syncthreads();
    if (r == 0 && col < d4) {
        float4 t = sums[0][cv];
        for (int q = 1; q < kSkRG; ++q) {
            const float4 x = sums[q][cv];
            t.x += x.x;
            t.y += x.y;
            t.z += x.z;
            t.w += x.w;
        }
        if (col_sumsq) col_sumsq[col] = t;
        if (col_scale) {
            float4 c = col_scale[col];
            c.x /= sqrtf(t.x) + eps;
            c.y /= sqrtf(t.y) + eps;
            c.z /= sqrtf(t.z) + eps;
            c.w /= sqrtf(t.w) + eps;
            col_scale[col] = c;
        }
    }
}

// ------------------------------------------------------------------------------- momentum

// Eight elements per thread and iteration: 16- or 32-byte gradient loads, 2 x 16-byte momentum
// loads and 4 x 16-byte stores.  The n % 8 tail is done element by element.
template <typename G>
__device__ __forceinline__ void sk_load8(const G *grad, int64_t v, float (&g)[8]);

template <>
__device__ __forceinline__ void sk_load8<float>(const float *grad, int64_t v, float (&g)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4 *>(grad) + 2 * v);
    const float4 b = __ldcs(reinterpret_cast<const float4 *>(grad) + 2 * v + 1);
    g[0] = a.x, g[1] = a.y, g[2] = a.z, g[3] = a.w, g[4] = b.x, g[5] = b.y, g[6] = b.z, g[7] = b.w;
}

template <>
__device__ __forceinline__ void sk_load8<__nv_bfloat16>(const __nv_bfloat16 *grad, int64_t v, float (&g)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(grad) + v);
    Vec<__nv_bfloat16>::unpack(u, g);
}

template <typename G>
__global__ void __launch_bounds__(256) sinkhorn_momentum_kernel(const G *__restrict__ grad, float *__restrict__ m,
                                                                float *__restrict__ out, int64_t n, float beta,
                                                                int nesterov) {
    const int64_t n8 = n >> 3;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < n8; v += stride) {
        float g[8];
        sk_load8<G>(grad, v, g);
        float4 *mv = reinterpret_cast<float4 *>(m) + 2 * v;
        float4 *ov = reinterpret_cast<float4 *>(out) + 2 * v;
        const float4 m0 = mv[0], m1 = mv[1];
        const float mo[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
        float mn[8], o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            mn[e] = fmaf(beta, mo[e], g[e]);
            o[e] = nesterov ? fmaf(beta, mn[e], g[e]) : mn[e];
        }
        mv[0] = make_float4(mn[0], mn[1], mn[2], mn[3]);
        mv[1] = make_float4(mn[4], mn[5], mn[6], mn[7]);
        __stcs(ov, make_float4(o[0], o[1], o[2], o[3]));
        __stcs(ov + 1, make_float4(o[4], o[5], o[6], o[7]));
    }
    if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
        const int64_t i = (n8 << 3) + threadIdx.x;
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

SkKernel sk_step_kernel(int vpt) {
    static const SkKernel k[kSkMaxVpt] = {sinkhorn_step_kernel<1>, sinkhorn_step_kernel<2>, sinkhorn_step_kernel<3>,
                                          sinkhorn_step_kernel<4>, sinkhorn_step_kernel<5>, sinkhorn_step_kernel<6>,
                                          sinkhorn_step_kernel<7>, sinkhorn_step_kernel<8>};
    return k[vpt - 1];
}

SkKernel sk_finalize_kernel(int vpt) {
    static const SkKernel k[kSkMaxVpt] = {
        sinkhorn_finalize_kernel<1>, sinkhorn_finalize_kernel<2>, sinkhorn_finalize_kernel<3>,
        sinkhorn_finalize_kernel<4>, sinkhorn_finalize_kernel<5>, sinkhorn_finalize_kernel<6>,
        sinkhorn_finalize_kernel<7>, sinkhorn_finalize_kernel<8>};
    return k[vpt - 1];
}

// Launches a row kernel on min(units, SMs) CTAs: one per SM, the ring takes most of its memory.
engram_status sk_launch(const char *fn, SkKernel kernel, const SinkhornParams &prm, int64_t units,
                        const DeviceInfo &dev, engram_stream_t stream) {
    const int smem = sk_smem_bytes(prm.stages, static_cast<int64_t>(prm.d) * 4);
    if (smem > dev.smem_optin)
        return fail(ENGRAM_ERR_SHAPE, "%s: %d bytes of shared memory exceed %d", fn, smem, dev.smem_optin);
    engram_status st = set_smem(reinterpret_cast<const void *>(kernel), smem);
    if (st != ENGRAM_OK) return st;
    const int64_t grid = cap_grid(std::min<int64_t>(units, dev.num_sms));
    kernel<<<static_cast<unsigned>(grid), kSkThreads, smem, reinterpret_cast<cudaStream_t>(stream)>>>(prm);
    return check_launch(fn);
}

int sk_vpt(int32_t head_dim) { return (head_dim / 4 + kSkThreads - 1) / kSkThreads; }

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
    const int threads = 256;
    const int64_t vecs = std::max<int64_t>(1, n >> 3);
    const int64_t blocks =
        cap_grid(std::min<int64_t>((vecs + threads - 1) / threads, static_cast<int64_t>(dev.num_sms) * 8));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == ENGRAM_F32)
        sinkhorn_momentum_kernel<float><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            static_cast<const float *>(grad), momentum, sinkhorn_input, n, beta1, nesterov != 0);
    else
        sinkhorn_momentum_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), threads, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(grad), momentum, sinkhorn_input, n, beta1, nesterov != 0);
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
    prm.stages = sk_stages(static_cast<int64_t>(head_dim) * 4);
    prm.eps = eps;
    return sk_launch(fn, sk_step_kernel(sk_vpt(head_dim)), prm, P, dev, stream);
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
    sinkhorn_reduce_kernel<<<(d4 + kSkCV - 1) / kSkCV, kSkRG * kSkCV, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
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
    prm.stages = sk_stages(static_cast<int64_t>(head_dim) * 4);
    prm.eps = eps;
    prm.alpha = alpha;
    return sk_launch(fn, sk_finalize_kernel(sk_vpt(head_dim)), prm, rows, dev, stream);
}
