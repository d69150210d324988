// B0 weight fold and B1 context-aware gate forward.
//
// TileLang tutorial, ch. 34 "TileKernels: Engram and mHC":
//   sec. 1.2 item 3  alpha_t = sigmoid(RMSNorm(h_t)^T RMSNorm(k_t) / sqrt(d)), output alpha_t * v_t;
//   sec. 3.1         RMSNorm(x; w_h)^T RMSNorm(k; w_k) = rstd_x * rstd_k * sum_i x_i (w_h (*) w_k)_i k_i,
//                    so with w_fused precomputed one pass yields sum x^2, sum k^2 and sum x*w*k;
//   sec. 3.2         the saved per-token statistics dot, alpha, rstd_x, rstd_k.
// The pages' kernel keeps the whole x row on chip because its output is
// x + alpha * v; the paper form alpha * v needs h and k only for the three
// sums, so here h, k and v are each streamed through shared memory once.
#include "gate_pipeline.cuh"

namespace engram {

struct GateFwdParams {
    const uint8_t *h, *k, *v;
    const float *w;
    // fold: with w_h and w_k given (w unused), each thread forms its slice of w_h (*) w_k itself, as
    // engram_fuse_weight rounds it, and CTA 0 writes the whole fold to w_out (nullable)
    const void *w_h, *w_k;
    float *w_out;
    int32_t w_bf16;
    uint8_t *out;
    float *alpha, *rstd_h, *rstd_k, *dot;
    float *out_rstd;  // with RMS: 1/sqrt(mean(out_t^2) + out_eps) of each stored output row
    uint32_t *status;
    int64_t T;
    int32_t d;
    uint32_t row_bytes;
    int32_t stages;
    float eps;
    float out_eps;
    float scale;  // 1/sqrt(d)
};

// RMS: also the RMS statistic of each output row as stored (rounded to `T`), the input of an RMSNorm
// that reads this output next: every warp adds its part of sum(out^2) to its slot of the token's
// reduction buffer in the output pass, and thread 0 sums the warps' parts in warp order once the
// next token's reduction barrier (or, for the last token, one more barrier) shows them complete.
template <typename T, int NCW, bool RMS>
__global__ void __launch_bounds__((NCW + 1) * 32) gate_fwd_kernel(const __grid_constant__ GateFwdParams p) {
    pdl_wait();              // the previous kernel's writes are complete and visible
    using V = Vec<T>;
    constexpr int EV = V::N;
    constexpr int NC = NCW * 32;
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rb = p.row_bytes;
    const int S = p.stages;
    const int nvec = static_cast<int>(rb / 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * 3 * rb);
    uint64_t *empty = full + S;
    float *red = reinterpret_cast<float *>(empty + S);  // [2][NCW][4]

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

    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t n_my = first < p.T ? (p.T - 1 - first) / stride + 1 : 0;

    if (warp == NCW) {  // ---------------------------------------------------------------- producer
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int64_t issued = 0;
            for (int64_t it = 0; it < n_my; ++it) {
                const int s = static_cast<int>(it % S);
                if (it >= S && !mbar_wait(&empty[s], static_cast<uint32_t>((it / S) & 1) ^ 1u)) {
                    report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                    break;
                }
                const int64_t tok = first + it * stride;
                uint8_t *dst = smem + static_cast<size_t>(s) * 3 * rb;
                const size_t off = static_cast<size_t>(tok) * rb;
                mbar_arrive_expect_tx(&full[s], 3 * rb);
                bulk_load(dst, p.h + off, rb, &full[s], pol);
                bulk_load(dst + rb, p.k + off, rb, &full[s], pol);
                bulk_load(dst + 2 * rb, p.v + off, rb, &full[s], pol);
                issued = it + 1;
            }
            // Never leave while a copy into this CTA's shared memory may be in flight.
            for (int64_t it = issued > S ? issued - S : 0; it < issued; ++it)
                if (!mbar_wait(&full[it % S], static_cast<uint32_t>((it / S) & 1)))
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
                const int i = j * EV + e;
                float4 q;
                if (p.w_h == nullptr) {
                    q = __ldg(reinterpret_cast<const float4 *>(p.w + i));
                } else {
                    float a[4], b[4];
                    if (p.w_bf16) {
                        const uint2 ua = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.w_h) + i));
                        const uint2 ub = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p.w_k) + i));
                        a[0] = __uint_as_float(ua.x << 16), a[1] = __uint_as_float(ua.x & 0xffff0000u);
                        a[2] = __uint_as_float(ua.y << 16), a[3] = __uint_as_float(ua.y & 0xffff0000u);
                        b[0] = __uint_as_float(ub.x << 16), b[1] = __uint_as_float(ub.x & 0xffff0000u);
                        b[2] = __uint_as_float(ub.y << 16), b[3] = __uint_as_float(ub.y & 0xffff0000u);
                    } else {
                        const float4 fa = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.w_h) + i));
                        const float4 fb = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p.w_k) + i));
                        a[0] = fa.x, a[1] = fa.y, a[2] = fa.z, a[3] = fa.w;
                        b[0] = fb.x, b[1] = fb.y, b[2] = fb.z, b[3] = fb.w;
                    }
                    q = make_float4(__fmul_rn(a[0], b[0]), __fmul_rn(a[1], b[1]), __fmul_rn(a[2], b[2]),
                                    __fmul_rn(a[3], b[3]));
                    if (p.w_out && blockIdx.x == 0) *reinterpret_cast<float4 *>(p.w_out + i) = q;
                }
                w[m][e] = q.x;
                w[m][e + 1] = q.y;
                w[m][e + 2] = q.z;
                w[m][e + 3] = q.w;
            }
        }
    }
    const float inv_d = 1.0f / static_cast<float>(p.d);
    // (thread 0) the statistic of token `it`, from the warps' parts in its buffer's fourth slots
    auto out_stat = [&](int64_t it) {
        const float *buf = red + (it & 1) * NCW * 4;
        float so = 0.f;
#pragma unroll
        for (int q = 0; q < NCW; ++q) so += buf[q * 4 + 3];
        p.out_rstd[first + it * stride] = 1.0f / sqrtf(so * inv_d + p.out_eps);
    };
    bool completed = true;

    for (int64_t it = 0; it < n_my; ++it) {
        const int s = static_cast<int>(it % S);
        const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1));
        const uint8_t *st = smem + static_cast<size_t>(s) * 3 * rb;

        // pass 1: sum h^2, sum k^2, sum h*w*k over this thread's vectors
        float sh = 0.f, sk = 0.f, sd = 0.f;
        if (ok) {
#pragma unroll
            for (int m = 0; m < kVPT; ++m) {
                const int j = c + m * NC;
                if (j < nvec) {
                    float hx[EV], kx[EV];
                    V::unpack(*reinterpret_cast<const uint4 *>(st + j * 16), hx);
                    V::unpack(*reinterpret_cast<const uint4 *>(st + rb + j * 16), kx);
#pragma unroll
                    for (int e = 0; e < EV; ++e) {
                        sh = fmaf(hx[e], hx[e], sh);
                        sk = fmaf(kx[e], kx[e], sk);
                        sd = fmaf(hx[e] * w[m][e], kx[e], sd);
                    }
                }
            }
        }
        sh = warp_sum(sh);
        sk = warp_sum(sk);
        sd = warp_sum(sd);
        float *rb_buf = red + (it & 1) * NCW * 4;
        if (lane == 0) {
            rb_buf[warp * 4 + 0] = sh;
            rb_buf[warp * 4 + 1] = sk;
            rb_buf[warp * 4 + 2] = sd;
        }
        if (named_sync_or(1, NC, !ok)) {
            if (c == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            completed = false;
            break;
        }
        // every warp has finished the previous token's output pass
        if (RMS && c == 0 && it > 0) out_stat(it - 1);
        float SH = 0.f, SK = 0.f, SD = 0.f;
#pragma unroll
        for (int q = 0; q < NCW; ++q) {
            SH += rb_buf[q * 4 + 0];
            SK += rb_buf[q * 4 + 1];
            SD += rb_buf[q * 4 + 2];
        }
        const float rh = 1.0f / sqrtf(SH * inv_d + p.eps);
        const float rk = 1.0f / sqrtf(SK * inv_d + p.eps);
        const float z = SD * rh * rk * p.scale;
        const float a = 1.0f / (1.0f + expf(-z));

        // pass 2: out = alpha * v
        const int64_t tok = first + it * stride;
        uint8_t *orow = p.out + static_cast<size_t>(tok) * rb;
        float so = 0.f;
#pragma unroll
        for (int m = 0; m < kVPT; ++m) {
            const int j = c + m * NC;
            if (j < nvec) {
                float vx[EV];
                V::unpack(*reinterpret_cast<const uint4 *>(st + 2 * rb + j * 16), vx);
#pragma unroll
                for (int e = 0; e < EV; ++e) vx[e] *= a;
                const uint4 packed = V::pack(vx);
                st_global_v4(orow + j * 16, packed);
                if (RMS) {  // the squares of the values as stored
                    float ox[EV];
                    V::unpack(packed, ox);
#pragma unroll
                    for (int e = 0; e < EV; ++e) so = fmaf(ox[e], ox[e], so);
                }
            }
        }
        if (RMS) {
            so = warp_sum(so);
            if (lane == 0) rb_buf[warp * 4 + 3] = so;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (c == 0) {
            if (p.alpha) p.alpha[tok] = a;
            if (p.rstd_h) p.rstd_h[tok] = rh;
            if (p.rstd_k) p.rstd_k[tok] = rk;
            if (p.dot) p.dot[tok] = SD;
        }
    }
    if (RMS && completed && n_my > 0) {
        named_sync_or(1, NC, false);  // every warp has finished the last token's output pass
        if (c == 0) out_stat(n_my - 1);
    }
}

template <typename T>
__global__ void fuse_weight_kernel(const T *__restrict__ w_h, const T *__restrict__ w_k, float *__restrict__ w,
                                   int32_t d) {
    pdl_wait();
    for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < d; i += gridDim.x * blockDim.x)
        w[i] = static_cast<float>(w_h[i]) * static_cast<float>(w_k[i]);
}

namespace {

template <typename T, int NCW>
engram_status launch_fwd(const GateFwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    const auto kern = p.out_rstd ? gate_fwd_kernel<T, NCW, true> : gate_fwd_kernel<T, NCW, false>;
    const PipelineShape shape = pick_fwd_pipeline(3 * static_cast<int>(p.row_bytes), NCW, dev.smem_optin);
    if (shape.stages == 0) return fail(ENGRAM_ERR_SHAPE, "engram_gate_fwd: row of %u bytes does not fit", p.row_bytes);
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), shape.smem_bytes);
    if (st != ENGRAM_OK) return st;
    GateFwdParams q = p;
    q.stages = shape.stages;
    int64_t grid = static_cast<int64_t>(dev.num_sms) * shape.blocks_per_sm;
    if (grid > p.T) grid = p.T;
    grid = cap_grid(grid);
    cudaError_t e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3((NCW + 1) * 32), shape.smem_bytes,
                                  stream, q);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_gate_fwd launch: %s", cudaGetErrorString(e));
    return check_launch("engram_gate_fwd");
}

template <typename T>
engram_status dispatch_fwd(const GateFwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    switch (pick_consumer_warps(static_cast<int>(p.row_bytes))) {
        case 1: return launch_fwd<T, 1>(p, dev, stream);
        case 2: return launch_fwd<T, 2>(p, dev, stream);
        case 4: return launch_fwd<T, 4>(p, dev, stream);
        default: return launch_fwd<T, 8>(p, dev, stream);
    }
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" engram_status engram_fuse_weight(const void *w_h, const void *w_k, engram_dtype dtype, float *w_fused,
                                            int32_t d, engram_stream_t stream) {
    if (!w_h || !w_k || !w_fused) return fail(ENGRAM_ERR_NULL, "engram_fuse_weight: NULL pointer");
    if (dtype_size(dtype) == 0) return fail(ENGRAM_ERR_DTYPE, "engram_fuse_weight: dtype %d", (int)dtype);
    if (d <= 0) return fail(ENGRAM_ERR_SHAPE, "engram_fuse_weight: d = %d", d);
    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    if ((st = check_device_ptr(w_h, dev.device, "w_h")) || (st = check_device_ptr(w_k, dev.device, "w_k")) ||
        (st = check_device_ptr(w_fused, dev.device, "w_fused")))
        return st;
    const int threads = 256;
    int blocks = (d + threads - 1) / threads;
    if (blocks > 4 * dev.num_sms) blocks = 4 * dev.num_sms;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == ENGRAM_F32)
        e = launch_kernel(fuse_weight_kernel<float>, dim3(blocks), dim3(threads), 0, s,
                          static_cast<const float *>(w_h), static_cast<const float *>(w_k), w_fused, d);
    else
        e = launch_kernel(fuse_weight_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, s,
                          static_cast<const __nv_bfloat16 *>(w_h), static_cast<const __nv_bfloat16 *>(w_k), w_fused, d);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_fuse_weight launch: %s", cudaGetErrorString(e));
    return check_launch("engram_fuse_weight");
}

namespace {

// The forward; with fold != nullptr (w_fused unused) the weights are fold->w_h and fold->w_k, multiplied in
// the kernel, and the fold is written to fold->w_out.
struct FoldArgs {
    const void *w_h, *w_k;
    engram_dtype w_dtype;
    float *w_out;
};

engram_status gate_fwd_impl(const void *h, const void *k, const void *v, engram_dtype dtype, const float *w_fused,
                            int64_t T, int32_t d, float eps, void *out, float *alpha, float *rstd_h, float *rstd_k,
                            float *dot, float *out_rstd, float out_eps, engram_stream_t stream,
                            const FoldArgs *fold = nullptr) {
    // Per-token tensors may be NULL only when there is no token (an empty tensor has no storage).
    if ((!fold && !w_fused) || (T > 0 && (!h || !k || !v || !out)))
        return fail(ENGRAM_ERR_NULL, "engram_gate_fwd: NULL pointer");
    const int es = dtype_size(dtype);
    if (es == 0) return fail(ENGRAM_ERR_DTYPE, "engram_gate_fwd: dtype %d", (int)dtype);
    if (T < 0 || d <= 0) return fail(ENGRAM_ERR_SHAPE, "engram_gate_fwd: T = %lld, d = %d", (long long)T, d);
    const int64_t row_bytes = static_cast<int64_t>(d) * es;
    if (row_bytes % 16 != 0) return fail(ENGRAM_ERR_ALIGN, "engram_gate_fwd: row of %lld bytes", (long long)row_bytes);
    if (row_bytes > ENGRAM_MAX_ROW_BYTES)
        return fail(ENGRAM_ERR_SHAPE, "engram_gate_fwd: row of %lld bytes exceeds %d", (long long)row_bytes,
                    ENGRAM_MAX_ROW_BYTES);
    if (!aligned16(h) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(w_fused))
        return fail(ENGRAM_ERR_ALIGN, "engram_gate_fwd: tensor not 16-byte aligned");
    DeviceInfo dev;
    engram_status st = current_device(&dev);
    if (st != ENGRAM_OK) return st;
    if (fold) {
        if (!aligned16(fold->w_h) || !aligned16(fold->w_k) || !aligned16(fold->w_out))
            return fail(ENGRAM_ERR_ALIGN, "engram_gate_fwd_fold: weight not 16-byte aligned");
        if ((st = check_device_ptr(fold->w_h, dev.device, "w_h")) ||
            (st = check_device_ptr(fold->w_k, dev.device, "w_k")) ||
            (st = check_device_ptr(fold->w_out, dev.device, "w_fused_out")))
            return st;
        if (T == 0)  // no token, so no forward to fold it in: the fold alone, for the backward
            return fold->w_out ? engram_fuse_weight(fold->w_h, fold->w_k, fold->w_dtype, fold->w_out, d, stream)
                               : ENGRAM_OK;
    }
    if ((st = check_device_ptr(h, dev.device, "h")) || (st = check_device_ptr(k, dev.device, "k")) ||
        (st = check_device_ptr(v, dev.device, "v")) || (st = check_device_ptr(w_fused, dev.device, "w_fused")) ||
        (st = check_device_ptr(out, dev.device, "out")) || (st = check_device_ptr(alpha, dev.device, "alpha")) ||
        (st = check_device_ptr(rstd_h, dev.device, "rstd_h")) ||
        (st = check_device_ptr(rstd_k, dev.device, "rstd_k")) || (st = check_device_ptr(dot, dev.device, "dot")) ||
        (st = check_device_ptr(out_rstd, dev.device, "out_rstd")))
        return st;
    if (T == 0) return ENGRAM_OK;

    GateFwdParams p{};
    p.h = static_cast<const uint8_t *>(h);
    p.k = static_cast<const uint8_t *>(k);
    p.v = static_cast<const uint8_t *>(v);
    p.w = w_fused;
    p.out = static_cast<uint8_t *>(out);
    p.alpha = alpha;
    p.rstd_h = rstd_h;
    p.rstd_k = rstd_k;
    p.dot = dot;
    p.out_rstd = out_rstd;
    p.out_eps = out_eps;
    p.status = dev.status_word;
    p.T = T;
    p.d = d;
    p.row_bytes = static_cast<uint32_t>(row_bytes);
    p.eps = eps;
    p.scale = 1.0f / sqrtf(static_cast<float>(d));
    if (fold) {
        p.w = nullptr;
        p.w_h = fold->w_h;
        p.w_k = fold->w_k;
        p.w_bf16 = fold->w_dtype == ENGRAM_BF16;
        p.w_out = fold->w_out;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dtype == ENGRAM_F32 ? dispatch_fwd<float>(p, dev, s) : dispatch_fwd<__nv_bfloat16>(p, dev, s);
}

}  // namespace

extern "C" engram_status engram_gate_fwd(const void *h, const void *k, const void *v, engram_dtype dtype,
                                         const float *w_fused, int64_t T, int32_t d, float eps, void *out,
                                         float *alpha, float *rstd_h, float *rstd_k, float *dot,
                                         engram_stream_t stream) {
    return gate_fwd_impl(h, k, v, dtype, w_fused, T, d, eps, out, alpha, rstd_h, rstd_k, dot, nullptr, 0.f, stream);
}

extern "C" engram_status engram_gate_fwd_rms(const void *h, const void *k, const void *v, engram_dtype dtype,
                                             const float *w_fused, int64_t T, int32_t d, float eps, void *out,
                                             float *alpha, float *rstd_h, float *rstd_k, float *dot, float *out_rstd,
                                             float out_eps, engram_stream_t stream) {
    if (!out_rstd && T > 0) return fail(ENGRAM_ERR_NULL, "engram_gate_fwd_rms: NULL out_rstd");
    return gate_fwd_impl(h, k, v, dtype, w_fused, T, d, eps, out, alpha, rstd_h, rstd_k, dot, out_rstd, out_eps,
                         stream);
}

extern "C" engram_status engram_gate_fwd_fold(const void *h, const void *k, const void *v, engram_dtype dtype,
                                              const void *w_h, const void *w_k, engram_dtype w_dtype, int64_t T,
                                              int32_t d, float eps, void *out, float *alpha, float *rstd_h,
                                              float *rstd_k, float *dot, float *w_fused_out, engram_stream_t stream) {
    if (!w_h || !w_k) return fail(ENGRAM_ERR_NULL, "engram_gate_fwd_fold: NULL weight");
    if (dtype_size(w_dtype) == 0) return fail(ENGRAM_ERR_DTYPE, "engram_gate_fwd_fold: weight dtype %d", (int)w_dtype);
    const FoldArgs fold{w_h, w_k, w_dtype, w_fused_out};
    return gate_fwd_impl(h, k, v, dtype, nullptr, T, d, eps, out, alpha, rstd_h, rstd_k, dot, nullptr, 0.f, stream,
                         &fold);
}
