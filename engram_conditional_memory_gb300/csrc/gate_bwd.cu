// B2 gate backward and B3 deterministic weight-gradient reduction.
//
// TileLang tutorial, ch. 34 "TileKernels: Engram and mHC":
//   sec. 4.1  fused_weight / gate_fwd / gate_bwd / grad_w_reduce division of work;
//   sec. 4.2  the backward: dL/dalpha = sum_i dout_i v_i first, then through the
//             sigmoid to dL/d dot, then the RMSNorm chain rule for the inputs and
//             the per-block partial of dL/dw_fused = c * x * k;
//   sec. 4.3  why the parameter gradient needs a separate cross-block reduction,
//             and its accumulate semantics (grad_w_h += S * w_k, grad_w_k += S * w_h);
// and the TileLang DSL article (DeepSeek-V4 determinism): replace concurrent
// atomic accumulation by partitioned partial writes plus one ordered reduction.
//
// Partition: partial p covers tokens [p*C, min(T, (p+1)*C)), C = ceil(T / P).
// The P recommended by engram_gate_bwd_num_partials depends on T only, and a
// CTA's consumer thread owns the same columns whatever the grid, summing its
// tokens in ascending order, so every partial -- and the reduced gradient -- is
// bitwise identical on any GPU and for any grid size.
#include <algorithm>
#include <mutex>

#include "colsum.cuh"
#include "gate_pipeline.cuh"

namespace engram {

struct GateBwdParams {
    const uint8_t *g, *h, *k, *v;
    const float *w, *alpha, *rstd_h, *rstd_k, *dot;
    uint8_t *dh, *dk, *dv;
    float *dw_partial;
    uint32_t *status;
    int64_t T;
    int64_t chunk;  // C
    int32_t P;
    int32_t d;
    uint32_t row_bytes;
    int32_t stages;
    int32_t accumulate;  // 1: each partial row adds its tokens' terms onto the row's current contents
    float scale;  // 1/sqrt(d)
};

// ACC: each partial row adds its tokens' terms onto the row's current contents (p.accumulate).
template <typename T, int NCW, bool ACC>
__global__ void __launch_bounds__((NCW + 1) * 32) gate_bwd_kernel(const __grid_constant__ GateBwdParams p) {
    pdl_wait();              // the previous kernel's writes are complete and visible
    using V = Vec<T>;
    constexpr int EV = V::N;
    constexpr int NC = NCW * 32;
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rb = p.row_bytes;
    const int S = p.stages;
    const int nvec = static_cast<int>(rb / 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * 4 * rb);
    uint64_t *empty = full + S;
    float *red = reinterpret_cast<float *>(empty + S);  // [2][NCW] (4 floats reserved per warp)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == NCW) {  // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int64_t it = 0;
            bool failed = false;
            for (int64_t pp = blockIdx.x; pp < p.P && !failed; pp += gridDim.x) {
                const int64_t t0 = pp * p.chunk;
                const int64_t t1 = t0 + p.chunk < p.T ? t0 + p.chunk : p.T;
                for (int64_t t = t0; t < t1; ++t, ++it) {
                    const int s = static_cast<int>(it % S);
                    if (it >= S && !mbar_wait(&empty[s], static_cast<uint32_t>((it / S) & 1) ^ 1u)) {
                        report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                        failed = true;
                        break;
                    }
                    uint8_t *dst = smem + static_cast<size_t>(s) * 4 * rb;
                    const size_t off = static_cast<size_t>(t) * rb;
                    mbar_arrive_expect_tx(&full[s], 4 * rb);
                    bulk_load(dst, p.g + off, rb, &full[s], pol);
                    bulk_load(dst + rb, p.v + off, rb, &full[s], pol);
                    bulk_load(dst + 2 * rb, p.h + off, rb, &full[s], pol);
                    bulk_load(dst + 3 * rb, p.k + off, rb, &full[s], pol);
                }
            }
            const int64_t issued = it;
            for (int64_t q = issued > S ? issued - S : 0; q < issued; ++q)
                if (!mbar_wait(&full[q % S], static_cast<uint32_t>((q / S) & 1)))
                    report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
        }
        return;
    }

    // ------------------------------------------------------------------------------------ consumers
    const int c = threadIdx.x;
    float w[kVPT][EV];
#pragma unroll
    for (int m = 0; m < kVPT; ++m) {
        const int j = c + m * NC;
#pragma unroll
        for (int e = 0; e < EV; ++e) w[m][e] = 0.f;
        if (j < nvec) {
#pragma unroll
            for (int e = 0; e < EV; e += 4) {
                const float4 q = __ldg(reinterpret_cast<const float4 *>(p.w + j * EV + e));
                w[m][e] = q.x;
                w[m][e + 1] = q.y;
                w[m][e + 2] = q.z;
                w[m][e + 3] = q.w;
            }
        }
    }
    const float inv_d = 1.0f / static_cast<float>(p.d);

    int64_t it = 0;
    bool failed = false;
    for (int64_t pp = blockIdx.x; pp < p.P && !failed; pp += gridDim.x) {
        const int64_t t0 = pp * p.chunk;
        const int64_t t1 = t0 + p.chunk < p.T ? t0 + p.chunk : p.T;
        // the partial row's accumulators: zero, or (accumulate) the row as a previous call left it, its
        // load overlapping the first stage's wait
        float *prow = p.dw_partial + static_cast<size_t>(pp) * p.d;
        float acc[kVPT][EV];
#pragma unroll
        for (int m = 0; m < kVPT; ++m) {
            const int j = c + m * NC;
#pragma unroll
            for (int e = 0; e < EV; e += 4) {
                float4 q = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ACC && j < nvec) q = *reinterpret_cast<const float4 *>(prow + j * EV + e);
                acc[m][e] = q.x;
                acc[m][e + 1] = q.y;
                acc[m][e + 2] = q.z;
                acc[m][e + 3] = q.w;
            }
        }

        for (int64_t t = t0; t < t1; ++t, ++it) {
            const int s = static_cast<int>(it % S);
            // saved statistics of this token (plain loads; their latency overlaps the stage wait)
            const float a = __ldg(p.alpha + t);
            const float rh = __ldg(p.rstd_h + t);
            const float rk = __ldg(p.rstd_k + t);
            const float dt = __ldg(p.dot + t);
            const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1));
            const uint8_t *st = smem + static_cast<size_t>(s) * 4 * rb;
            const size_t roff = static_cast<size_t>(t) * rb;

            // pass 1: dalpha partial = sum g*v; dv = alpha * g
            float da = 0.f;
            if (ok) {
#pragma unroll
                for (int m = 0; m < kVPT; ++m) {
                    const int j = c + m * NC;
                    if (j < nvec) {
                        float gx[EV], vx[EV];
                        V::unpack(*reinterpret_cast<const uint4 *>(st + j * 16), gx);
                        V::unpack(*reinterpret_cast<const uint4 *>(st + rb + j * 16), vx);
#pragma unroll
                        for (int e = 0; e < EV; ++e) {
                            da = fmaf(gx[e], vx[e], da);
                            gx[e] *= a;
                        }
                        st_global_v4(p.dv + roff + j * 16, V::pack(gx));
                    }
                }
            }
            da = warp_sum(da);
            float *rbuf = red + (it & 1) * NCW * 4;
            if (lane == 0) rbuf[warp * 4] = da;
            if (named_sync_or(1, NC, !ok)) {
                if (c == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
                break;
            }
            float DA = 0.f;
#pragma unroll
            for (int q = 0; q < NCW; ++q) DA += rbuf[q * 4];

            // dL/d dot through the sigmoid and the scaling
            const float cc = DA * a * (1.0f - a) * p.scale * rh * rk;
            const float ch = cc * dt * rh * rh * inv_d;
            const float ck = cc * dt * rk * rk * inv_d;

            // pass 2: dh, dk and the weight-gradient accumulators
#pragma unroll
            for (int m = 0; m < kVPT; ++m) {
                const int j = c + m * NC;
                if (j < nvec) {
                    float hx[EV], kx[EV], oh[EV], ok2[EV];
                    V::unpack(*reinterpret_cast<const uint4 *>(st + 2 * rb + j * 16), hx);
                    V::unpack(*reinterpret_cast<const uint4 *>(st + 3 * rb + j * 16), kx);
#pragma unroll
                    for (int e = 0; e < EV; ++e) {
                        const float cw = cc * w[m][e];
                        oh[e] = fmaf(cw, kx[e], -ch * hx[e]);
                        ok2[e] = fmaf(cw, hx[e], -ck * kx[e]);
                        acc[m][e] = fmaf(cc * hx[e], kx[e], acc[m][e]);
                    }
                    st_global_v4(p.dh + roff + j * 16, V::pack(oh));
                    st_global_v4(p.dk + roff + j * 16, V::pack(ok2));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (failed) break;

        // this partial's row of dw_partial (zeros, or the row unchanged, for a partial with no token)
#pragma unroll
        for (int m = 0; m < kVPT; ++m) {
            const int j = c + m * NC;
            if (j < nvec) {
#pragma unroll
                for (int e = 0; e < EV; e += 4)
                    *reinterpret_cast<float4 *>(prow + j * EV + e) =
                        make_float4(acc[m][e], acc[m][e + 1], acc[m][e + 2], acc[m][e + 3]);
            }
        }
    }
}

// S = sum_p partial[p] (column_sums: an order that depends on P only), then the accumulate.
__global__ void __launch_bounds__(kColThreads, 1)
    grad_w_reduce_kernel(const float4 *__restrict__ part, int32_t P, int32_t d4, float4 *__restrict__ dweight,
                         const float4 *__restrict__ w_h, const float4 *__restrict__ w_k, float4 *__restrict__ g_h,
                         float4 *__restrict__ g_k) {
    pdl_wait();
    __shared__ ColSumSmem sm;
    column_sums(part, P, d4, sm, [&](int col, const float4 &t) {
        if (dweight) dweight[col] = t;
        if (g_h) {
            const float4 a = w_k[col], b = w_h[col];
            float4 gh = g_h[col], gk = g_k[col];
            gh.x += t.x * a.x; gh.y += t.y * a.y; gh.z += t.z * a.z; gh.w += t.w * a.w;
            gk.x += t.x * b.x; gk.y += t.y * b.y; gk.z += t.z * b.z; gk.w += t.w * b.w;
            g_h[col] = gh;
            g_k[col] = gk;
        }
    });
}

namespace {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <typename T, int NCW>
engram_status launch_bwd(const GateBwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    const auto kern = p.accumulate ? gate_bwd_kernel<T, NCW, true> : gate_bwd_kernel<T, NCW, false>;
    const PipelineShape shape = pick_bwd_pipeline(4 * static_cast<int>(p.row_bytes), NCW, dev.smem_optin);
    if (shape.stages == 0) return fail(ENGRAM_ERR_SHAPE, "engram_gate_bwd: row of %u bytes does not fit", p.row_bytes);
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), shape.smem_bytes);
    if (st != ENGRAM_OK) return st;
    GateBwdParams q = p;
    q.stages = shape.stages;
    // One CTA per partial (the kernel's partial loop then runs once per CTA).
    const int64_t grid = cap_grid(p.P);
    cudaError_t e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3((NCW + 1) * 32), shape.smem_bytes,
                                  stream, q);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_gate_bwd launch: %s", cudaGetErrorString(e));
    return check_launch("engram_gate_bwd");
}

template <typename T>
engram_status dispatch_bwd(const GateBwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    switch (pick_consumer_warps(static_cast<int>(p.row_bytes))) {
        case 1: return launch_bwd<T, 1>(p, dev, stream);
        case 2: return launch_bwd<T, 2>(p, dev, stream);
        case 4: return launch_bwd<T, 4>(p, dev, stream);
        default: return launch_bwd<T, 8>(p, dev, stream);
    }
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" engram_status engram_gate_bwd_num_partials(int64_t T, int32_t d, int32_t *P) {
    if (!P) return fail(ENGRAM_ERR_NULL, "engram_gate_bwd_num_partials: NULL P");
    if (T < 0 || d <= 0) return fail(ENGRAM_ERR_SHAPE, "engram_gate_bwd_num_partials: T = %lld, d = %d", (long long)T, d);
    // About 16 or more tokens per partial (a partial row costs 8d bytes of traffic,
    // under 4 % of 16 tokens' 14d + 16 bytes each) and at most 1024 partials.
    const int64_t chunk = std::max<int64_t>(16, ceil_div(T, 1024));
    *P = static_cast<int32_t>(std::max<int64_t>(1, ceil_div(T, chunk)));
    return ENGRAM_OK;
}

namespace {

engram_status gate_bwd_call(const char *fn, int accumulate, const void *dout, const void *h, const void *k,
                            const void *v, engram_dtype dtype, const float *w_fused, const float *alpha,
                            const float *rstd_h, const float *rstd_k, const float *dot, int64_t T, int32_t d,
                            void *dh, void *dk, void *dv, float *dw_partial, int32_t P, engram_stream_t stream) {
    // Per-token tensors may be NULL only when there is no token; dw_partial is always written.
    if (!w_fused || !dw_partial ||
        (T > 0 && (!dout || !h || !k || !v || !alpha || !rstd_h || !rstd_k || !dot || !dh || !dk || !dv)))
        return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    const int es = dtype_size(dtype);
    if (es == 0) return fail(ENGRAM_ERR_DTYPE, "%s: dtype %d", fn, (int)dtype);
    if (T < 0 || d <= 0 || P < 1)
        return fail(ENGRAM_ERR_SHAPE, "%s: T = %lld, d = %d, P = %d", fn, (long long)T, d, P);
    const int64_t row_bytes = static_cast<int64_t>(d) * es;
    if (row_bytes % 16 != 0) return fail(ENGRAM_ERR_ALIGN, "%s: row of %lld bytes", fn, (long long)row_bytes);
    if (row_bytes > ENGRAM_MAX_ROW_BYTES)
        return fail(ENGRAM_ERR_SHAPE, "%s: row of %lld bytes exceeds %d", fn, (long long)row_bytes,
                    ENGRAM_MAX_ROW_BYTES);
    if (!aligned16(dout) || !aligned16(h) || !aligned16(k) || !aligned16(v) || !aligned16(w_fused) ||
        !aligned16(dh) || !aligned16(dk) || !aligned16(dv) || !aligned16(dw_partial))
        return fail(ENGRAM_ERR_ALIGN, "%s: tensor not 16-byte aligned", fn);
    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    const void *ptrs[] = {dout, h, k, v, w_fused, alpha, rstd_h, rstd_k, dot, dh, dk, dv, dw_partial};
    const char *names[] = {"dout", "h", "k", "v", "w_fused", "alpha", "rstd_h", "rstd_k", "dot", "dh", "dk", "dv",
                           "dw_partial"};
    for (int i = 0; i < 13; ++i)
        if ((st = check_device_ptr(ptrs[i], dev.device, names[i])) != ENGRAM_OK) return st;

    GateBwdParams p{};
    p.g = static_cast<const uint8_t *>(dout);
    p.h = static_cast<const uint8_t *>(h);
    p.k = static_cast<const uint8_t *>(k);
    p.v = static_cast<const uint8_t *>(v);
    p.w = w_fused;
    p.alpha = alpha;
    p.rstd_h = rstd_h;
    p.rstd_k = rstd_k;
    p.dot = dot;
    p.dh = static_cast<uint8_t *>(dh);
    p.dk = static_cast<uint8_t *>(dk);
    p.dv = static_cast<uint8_t *>(dv);
    p.dw_partial = dw_partial;
    p.status = dev.status_word;
    p.T = T;
    p.P = P;
    p.chunk = ceil_div(T, P);
    p.d = d;
    p.row_bytes = static_cast<uint32_t>(row_bytes);
    p.accumulate = accumulate;
    p.scale = 1.0f / sqrtf(static_cast<float>(d));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dtype == ENGRAM_F32 ? dispatch_bwd<float>(p, dev, s) : dispatch_bwd<__nv_bfloat16>(p, dev, s);
}

}  // namespace

extern "C" engram_status engram_gate_bwd(const void *dout, const void *h, const void *k, const void *v,
                                         engram_dtype dtype, const float *w_fused, const float *alpha,
                                         const float *rstd_h, const float *rstd_k, const float *dot, int64_t T,
                                         int32_t d, void *dh, void *dk, void *dv, float *dw_partial, int32_t P,
                                         engram_stream_t stream) {
    return gate_bwd_call("engram_gate_bwd", 0, dout, h, k, v, dtype, w_fused, alpha, rstd_h, rstd_k, dot, T, d, dh,
                         dk, dv, dw_partial, P, stream);
}

extern "C" engram_status engram_gate_bwd_accumulate(const void *dout, const void *h, const void *k, const void *v,
                                                    engram_dtype dtype, const float *w_fused, const float *alpha,
                                                    const float *rstd_h, const float *rstd_k, const float *dot,
                                                    int64_t T, int32_t d, void *dh, void *dk, void *dv,
                                                    float *dw_partial, int32_t P, engram_stream_t stream) {
    return gate_bwd_call("engram_gate_bwd_accumulate", 1, dout, h, k, v, dtype, w_fused, alpha, rstd_h, rstd_k, dot,
                         T, d, dh, dk, dv, dw_partial, P, stream);
}

extern "C" engram_status engram_grad_w_reduce(const float *dw_partial, int32_t P, int32_t d, float *dweight_fused,
                                              const float *w_h, const float *w_k, float *grad_w_h, float *grad_w_k,
                                              engram_stream_t stream) {
    if (!dw_partial && P > 0) return fail(ENGRAM_ERR_NULL, "engram_grad_w_reduce: NULL dw_partial");
    const int nw = (w_h != nullptr) + (w_k != nullptr) + (grad_w_h != nullptr) + (grad_w_k != nullptr);
    if (nw != 0 && nw != 4)
        return fail(ENGRAM_ERR_NULL, "engram_grad_w_reduce: w_h, w_k, grad_w_h, grad_w_k must be given together");
    if (!dweight_fused && nw == 0) return fail(ENGRAM_ERR_NULL, "engram_grad_w_reduce: no output");
    if (P < 0 || d <= 0) return fail(ENGRAM_ERR_SHAPE, "engram_grad_w_reduce: P = %d, d = %d", P, d);
    if (d % 4 != 0) return fail(ENGRAM_ERR_ALIGN, "engram_grad_w_reduce: d = %d not a multiple of 4", d);
    const void *ptrs[] = {dw_partial, dweight_fused, w_h, w_k, grad_w_h, grad_w_k};
    const char *names[] = {"dw_partial", "dweight_fused", "w_h", "w_k", "grad_w_h", "grad_w_k"};
    for (int i = 0; i < 6; ++i)
        if (ptrs[i] && !aligned16(ptrs[i])) return fail(ENGRAM_ERR_ALIGN, "engram_grad_w_reduce: %s unaligned", names[i]);
    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    for (int i = 0; i < 6; ++i)
        if ((st = check_device_ptr(ptrs[i], dev.device, names[i])) != ENGRAM_OK) return st;
    const int d4 = d / 4;
    // one CTA per SM, no more than there are columns
    cudaError_t e = launch_kernel(
        grad_w_reduce_kernel, dim3(column_sum_grid(d4, dev.num_sms)), dim3(kColThreads), 0,
        reinterpret_cast<cudaStream_t>(stream),
        reinterpret_cast<const float4 *>(dw_partial), P, d4, reinterpret_cast<float4 *>(dweight_fused),
        reinterpret_cast<const float4 *>(w_h), reinterpret_cast<const float4 *>(w_k),
        reinterpret_cast<float4 *>(grad_w_h), reinterpret_cast<float4 *>(grad_w_k));
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_grad_w_reduce launch: %s", cudaGetErrorString(e));
    return check_launch("engram_grad_w_reduce");
}

// ---------------------------------------------------------------------------------------------
// Allocation-free backward + reduction for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: an embedding that has handed the whole device to a
// framework's caching allocator or to a fixed arena reserved at start-up (a raw allocation
// would fail or fragment it), or a serving loop that forbids allocation after start-up
// (cudaMalloc / cudaFree may synchronise the device and stall every stream).  For them,
// engram_gate_bwd_reduce_noalloc keeps the [P, d] weight-gradient partials in the library's
// own file-scope device array instead of a caller buffer.
// ---------------------------------------------------------------------------------------------

// 16 MiB of partials, held on every device that loads the library until the process exits.
static __device__ __align__(256) float g_noalloc_partials[ENGRAM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mutex;
float *g_noalloc_addr[kNoallocMaxDevices];

// The array's device address on `device` (which must be current).  The symbol's host-side
// name is only a stand-in; the address is looked up once per device and cached.
engram_status noalloc_scratch(int device, float **out) {
    if (device < 0 || device >= kNoallocMaxDevices)
        return fail(ENGRAM_ERR_CUDA, "engram_gate_bwd_reduce_noalloc: device %d out of range", device);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[device]) {
        float *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_partials);
        if (e != cudaSuccess || !p)
            return fail(ENGRAM_ERR_CUDA, "engram_gate_bwd_reduce_noalloc: scratch address on device %d: %s", device,
                        cudaGetErrorString(e));
        g_noalloc_addr[device] = p;
    }
    *out = g_noalloc_addr[device];
    return ENGRAM_OK;
}

}  // namespace

extern "C" engram_status engram_gate_bwd_reduce_noalloc(
    const void *dout, const void *h, const void *k, const void *v, engram_dtype dtype, const float *w_fused,
    const float *alpha, const float *rstd_h, const float *rstd_k, const float *dot, int64_t T, int32_t d,
    void *dh, void *dk, void *dv, float *dweight_fused, const float *w_h, const float *w_k, float *grad_w_h,
    float *grad_w_k, engram_stream_t stream) {
    const char *fn = "engram_gate_bwd_reduce_noalloc";
    const int nw = (w_h != nullptr) + (w_k != nullptr) + (grad_w_h != nullptr) + (grad_w_k != nullptr);
    if (nw != 0 && nw != 4) return fail(ENGRAM_ERR_NULL, "%s: w_h, w_k, grad_w_h, grad_w_k must be given together", fn);
    if (!dweight_fused && nw == 0) return fail(ENGRAM_ERR_NULL, "%s: no weight-gradient output", fn);
    if (!w_fused || (T > 0 && (!dout || !h || !k || !v || !alpha || !rstd_h || !rstd_k || !dot || !dh || !dk || !dv)))
        return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    const int es = dtype_size(dtype);
    if (es == 0) return fail(ENGRAM_ERR_DTYPE, "%s: dtype %d", fn, (int)dtype);
    if (T < 0 || d <= 0) return fail(ENGRAM_ERR_SHAPE, "%s: T = %lld, d = %d", fn, (long long)T, d);
    const int64_t row_bytes = static_cast<int64_t>(d) * es;
    if (row_bytes % 16 != 0) return fail(ENGRAM_ERR_ALIGN, "%s: row of %lld bytes", fn, (long long)row_bytes);
    if (row_bytes > ENGRAM_MAX_ROW_BYTES)
        return fail(ENGRAM_ERR_SHAPE, "%s: row of %lld bytes exceeds %d", fn, (long long)row_bytes,
                    ENGRAM_MAX_ROW_BYTES);
    int32_t P = 0;
    engram_status st = engram_gate_bwd_num_partials(T, d, &P);
    if (st != ENGRAM_OK) return st;
    const int64_t need = static_cast<int64_t>(P) * d * static_cast<int64_t>(sizeof(float));
    if (need > static_cast<int64_t>(ENGRAM_NOALLOC_SCRATCH_BYTES))
        return fail(ENGRAM_ERR_SHAPE,
                    "%s: T = %lld, d = %d needs %lld bytes of weight-gradient partials (P = %d), more than the %u "
                    "bytes this entry point holds; call engram_gate_bwd with a caller-allocated buffer instead",
                    fn, (long long)T, d, (long long)need, P, (unsigned)ENGRAM_NOALLOC_SCRATCH_BYTES);
    const void *ptrs[] = {dout, h, k, v, w_fused, dh, dk, dv, dweight_fused, w_h, w_k, grad_w_h, grad_w_k};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return fail(ENGRAM_ERR_ALIGN, "%s: tensor not 16-byte aligned", fn);
    DeviceInfo dev;
    if ((st = current_device(&dev)) != ENGRAM_OK) return st;
    const void *dptrs[] = {dout, h, k, v, w_fused, alpha, rstd_h, rstd_k, dot, dh, dk, dv, dweight_fused, w_h, w_k,
                           grad_w_h, grad_w_k};
    for (const void *q : dptrs)
        if ((st = check_device_ptr(q, dev.device, fn)) != ENGRAM_OK) return st;
    float *scratch = nullptr;
    if ((st = noalloc_scratch(dev.device, &scratch)) != ENGRAM_OK) return st;

    // Backward into the scratch partials.  Every one of the P rows is written (rows of
    // partials without tokens are written as zeros), so nothing needs clearing first.
    GateBwdParams p{};
    p.g = static_cast<const uint8_t *>(dout);
    p.h = static_cast<const uint8_t *>(h);
    p.k = static_cast<const uint8_t *>(k);
    p.v = static_cast<const uint8_t *>(v);
    p.w = w_fused;
    p.alpha = alpha;
    p.rstd_h = rstd_h;
    p.rstd_k = rstd_k;
    p.dot = dot;
    p.dh = static_cast<uint8_t *>(dh);
    p.dk = static_cast<uint8_t *>(dk);
    p.dv = static_cast<uint8_t *>(dv);
    p.dw_partial = scratch;
    p.status = dev.status_word;
    p.T = T;
    p.P = P;
    p.chunk = ceil_div(T, P);
    p.d = d;
    p.row_bytes = static_cast<uint32_t>(row_bytes);
    p.scale = 1.0f / sqrtf(static_cast<float>(d));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = dtype == ENGRAM_F32 ? dispatch_bwd<float>(p, dev, s) : dispatch_bwd<__nv_bfloat16>(p, dev, s);
    if (st != ENGRAM_OK) return st;

    // Ordered reduction of the partials, on the same stream.
    const int d4 = d / 4;
    grad_w_reduce_kernel<<<column_sum_grid(d4, dev.num_sms), kColThreads, 0, s>>>(
        reinterpret_cast<const float4 *>(scratch), P, d4, reinterpret_cast<float4 *>(dweight_fused),
        reinterpret_cast<const float4 *>(w_h), reinterpret_cast<const float4 *>(w_k),
        reinterpret_cast<float4 *>(grad_w_h), reinterpret_cast<float4 *>(grad_w_k));
    return check_launch(fn);
}
