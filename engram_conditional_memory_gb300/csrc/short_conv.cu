// The short convolution after the gate (NEXT-2): Y = SiLU(Conv1D(RMSNorm(V~))) + V~, H <- H + Y,
// a depthwise causal convolution of `width` taps (at most 4) with a dilation, per sequence
// (TileLang tutorial, ch. 34 "TileKernels: Engram and mHC", sec. 1.2 item 4: kernel size 4,
// dilation the largest N-gram order).  Tap i multiplies the token (width - 1 - i) * dilation steps
// back, so tap width - 1 is the current token (torch's depthwise conv1d layout with left padding).
//
// GB300 design.  The convolution couples tokens only along time, one channel at a time, and the
// RMSNorm couples channels only within a token, through one scalar.  So:
//   * conv_rstd_kernel: a warp per token computes rstd = 1/sqrt(mean(V~^2) + eps);
//   * conv_stencil_kernel: a warp owns 128 channels of one residue class t = r (mod dilation):
//     every tap of a class token lies in the same class, so the warp sweeps its tokens in time
//     order keeping the last three taps' inputs in registers, with no other warp involved.  Each
//     warp streams its rows (V~ and H, or V~ and dout) through its own ring of shared-memory
//     stages filled by 1-D bulk (TMA) copies that its lane 0 issues, so the bytes in flight do not
//     depend on occupancy.  Per-token scalars (rstd, and the backward's row dots) come 64 tokens at
//     a time, two per lane, one window ahead, and reach a token by a shuffle.
// The backward is two sweeps: the first gives each token's partial dot s = sum_j norm_w du V~ over
// the warp's channels, the second the full dV~ = dout + rstd norm_w du - rstd^3 V~ s / d with s
// summed over the warps in a fixed order, and the weight-gradient partials of its (time chunk,
// residue) work item.  conv_grad_reduce_kernel sums those partials in a fixed order.  The time
// chunks depend on T only, so the weight gradients are bitwise reproducible on any GPU.
#include <algorithm>

#include "engram_internal.cuh"

namespace engram {

constexpr int kScWarps = 8;             // warps per CTA, each an independent work item
constexpr int kScEV = 4;                // channels per lane
constexpr int kScCols = 32 * kScEV;     // channels per warp
constexpr int kScAges = 4;              // taps: width <= 4
constexpr int kScRingBytes = 8192;      // per warp: stages x (V~ segment + second segment)
constexpr int kScMaxBlocks = 64;        // channel blocks per row: d <= 64 * 128

enum ScMode { kScFwd = 0, kScBwdDot = 1, kScBwdFinal = 2 };

struct ScParams {
    const uint8_t *v;          // V~ [T, d]
    const uint8_t *x2;         // forward: H (nullable); backward: dout
    const float *norm_w;       // [d]
    const float *conv_w;       // [d, width]
    const float *bias;         // [d] nullable
    const float *rstd;         // [T]
    const int64_t *offs;       // [num_seqs + 1]
    const float *token_dot;    // final backward: [T, nb] partial dots
    float *token_dot_out;      // first backward sweep: [T, nb]
    uint8_t *out;              // forward: out; final backward: dv
    float *partial;            // final backward: [nchunks * dil, width + 2, d]
    uint32_t *status;
    int64_t T;
    int64_t chunk;             // tokens per time chunk
    int64_t nchunks;
    int32_t num_seqs;
    int32_t d;
    int32_t width;
    int32_t dil;
    int32_t nb;                // channel blocks of kScCols
    int32_t stages;
};

// ---- four channels per lane: 8 bytes of bf16 or 16 bytes of fp32

template <typename E>
struct Ev4;

template <>
struct Ev4<float> {
    static constexpr int kBytes = 16;
    __device__ __forceinline__ static void load_smem(const uint8_t *p, float (&x)[4]) {
        const uint4 u = ld_shared_v4(p);
        x[0] = __uint_as_float(u.x), x[1] = __uint_as_float(u.y), x[2] = __uint_as_float(u.z),
        x[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static void store(uint8_t *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <>
struct Ev4<__nv_bfloat16> {
    static constexpr int kBytes = 8;
    __device__ __forceinline__ static void load_smem(const uint8_t *p, float (&x)[4]) {
        uint32_t a, b;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(smem_addr(p)) : "memory");
        x[0] = __uint_as_float(a << 16), x[1] = __uint_as_float(a & 0xffff0000u);
        x[2] = __uint_as_float(b << 16), x[3] = __uint_as_float(b & 0xffff0000u);
    }
    __device__ __forceinline__ static void store(uint8_t *p, const float (&x)[4]) {
        *reinterpret_cast<uint2 *>(p) =
            make_uint2(Vec<__nv_bfloat16>::pack2(x[0], x[1]), Vec<__nv_bfloat16>::pack2(x[2], x[3]));
    }
};

__device__ __forceinline__ float sc_sigmoid(float c) { return 1.0f / (1.0f + expf(-c)); }

// Index of the sequence holding token t: the largest s with offs[s] <= t (offsets assumed sorted).
__device__ __forceinline__ int sc_seq_of(const int64_t *offs, int num_seqs, int64_t t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offs + mid) <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------------------------------- rstd

template <typename E>
__global__ void __launch_bounds__(256) conv_rstd_kernel(const uint8_t *__restrict__ v, int64_t T, int32_t d,
                                                        float eps, float *__restrict__ rstd) {
    using V = Vec<E>;
    const int lane = threadIdx.x & 31;
    const int nvec = d / V::N;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const uint4 *row = reinterpret_cast<const uint4 *>(v + static_cast<size_t>(t) * d * sizeof(E));
        float ss = 0.f;
#pragma unroll 4
        for (int j = lane; j < nvec; j += 32) {
            float x[V::N];
            V::unpack(__ldcs(row + j), x);
#pragma unroll
            for (int e = 0; e < V::N; ++e) ss = fmaf(x[e], x[e], ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) rstd[t] = rsqrtf(ss / static_cast<float>(d) + eps);
    }
}

// ------------------------------------------------------------------------------- the stencil sweep

// Per-token scalars of the warp's sweep (indexed by the sweep position q), 64 at a time: lane l
// holds positions w0 + l and w0 + 32 + l of the current window and the next window's two.
struct ScWindow {
    float lo, hi, nlo, nhi;
    int64_t w0;
};

// The row-dot total of token t: the nb partials in ascending order.
__device__ __forceinline__ float sc_dot_total(const ScParams &p, int64_t t) {
    const float *row = p.token_dot + static_cast<size_t>(t) * p.nb;
    float s = 0.f;
    for (int b = 0; b < p.nb; ++b) s += __ldg(row + b);
    return s;
}

template <typename E, int MODE>
__global__ void __launch_bounds__(kScWarps * 32) conv_stencil_kernel(const __grid_constant__ ScParams p) {
    using EV = Ev4<E>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.stages;
    const int seg_max = kScCols * static_cast<int>(sizeof(E));
    uint8_t *ring = smem + static_cast<size_t>(warp) * kScRingBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(kScWarps) * kScRingBytes) + warp * S;

    const int64_t item = static_cast<int64_t>(blockIdx.x) * kScWarps + warp;
    const int cb = static_cast<int>(item % p.nb);
    const int64_t kr = item / p.nb;
    const int r = static_cast<int>(kr % p.dil);
    const int64_t k = kr / p.dil;
    if (k >= p.nchunks) return;  // whole warp: no shared state with the other warps

    const int64_t t_lo = k * p.chunk;
    const int64_t t_hi = t_lo + p.chunk < p.T ? t_lo + p.chunk : p.T;
    const int c0 = cb * kScCols;
    const int ncols = p.d - c0 < kScCols ? p.d - c0 : kScCols;
    const uint32_t seg = static_cast<uint32_t>(ncols) * sizeof(E);
    const bool active = lane * kScEV < ncols;
    const size_t row_bytes = static_cast<size_t>(p.d) * sizeof(E);
    const int dil = p.dil;
    auto first_class = [&](int64_t x) { return x + ((r - x % dil) % dil + dil) % dil; };

    // per-lane constants: taps by age (age a multiplies the token a * dil back), norm weight, bias
    float K[kScAges][kScEV], nw[kScEV], bias[kScEV];
#pragma unroll
    for (int e = 0; e < kScEV; ++e) {
        const int c = c0 + lane * kScEV + e;
        const bool ok = active && c < p.d;
        nw[e] = ok ? __ldg(p.norm_w + c) : 0.f;
        bias[e] = ok && p.bias ? __ldg(p.bias + c) : 0.f;
#pragma unroll
        for (int a = 0; a < kScAges; ++a)
            K[a][e] = ok && a < p.width ? __ldg(p.conv_w + static_cast<size_t>(c) * p.width + (p.width - 1 - a)) : 0.f;
    }

    // the sweep: class tokens from up to three taps before the chunk (their inputs only) to the
    // chunk's end, or three taps past it for the backward (their dc completes the chunk's du)
    const int64_t t_first = first_class(t_lo);
    float dK[kScAges][kScEV], db[kScEV], dnw[kScEV];
#pragma unroll
    for (int e = 0; e < kScEV; ++e) {
        db[e] = dnw[e] = 0.f;
#pragma unroll
        for (int a = 0; a < kScAges; ++a) dK[a][e] = 0.f;
    }
    int64_t n_sw = 0, t_a = t_first;
    int s = 0;
    if (t_first < t_hi) {
        s = sc_seq_of(p.offs, p.num_seqs, t_first);
        const int64_t hist = t_first - static_cast<int64_t>(kScAges - 1) * dil;
        const int64_t s0 = __ldg(p.offs + s);
        t_a = first_class(hist > s0 ? hist : s0);
        int64_t t_b = MODE == kScFwd ? t_hi : t_hi + static_cast<int64_t>(kScAges - 1) * dil;
        if (t_b > p.T) t_b = p.T;
        n_sw = (t_b - t_a + dil - 1) / dil;
    }

    const uint64_t pol = l2_evict_first_policy();
    const bool two = MODE != kScFwd || p.x2 != nullptr;
    // lane 0: sweep position q into stage q % S; a lead-in token (before the chunk) needs V~ only
    auto issue = [&](int64_t q) {
        const int st = static_cast<int>(q % S);
        const int64_t t = t_a + q * dil;
        const bool second = two && t >= t_lo;
        uint8_t *dst = ring + static_cast<size_t>(st) * 2 * seg_max;
        mbar_arrive_expect_tx(&full[st], second ? 2 * seg : seg);
        bulk_load(dst, p.v + static_cast<size_t>(t) * row_bytes + static_cast<size_t>(c0) * sizeof(E), seg, &full[st],
                  pol);
        if (second)
            bulk_load(dst + seg_max, p.x2 + static_cast<size_t>(t) * row_bytes + static_cast<size_t>(c0) * sizeof(E),
                      seg, &full[st], pol);
    };
    int64_t issued = 0;
    if (lane == 0) {
        for (int q = 0; q < S; ++q) mbar_init(&full[q], 1);
        mbar_init_fence();
        for (; issued < S && issued < n_sw; ++issued) issue(issued);
    }
    __syncwarp();

    // scalar windows: rstd, and the backward's row-dot totals in the final sweep
    auto scalar_at = [&](int64_t q, bool dot) -> float {
        const int64_t t = t_a + q * dil;
        if (q >= n_sw) return 0.f;
        return dot ? sc_dot_total(p, t) : __ldg(p.rstd + t);
    };
    ScWindow wr{0.f, 0.f, scalar_at(lane, false), scalar_at(32 + lane, false), -64};
    ScWindow ws{0.f, 0.f, 0.f, 0.f, -64};
    if (MODE == kScBwdFinal) ws.nlo = scalar_at(lane, true), ws.nhi = scalar_at(32 + lane, true);

    // histories by age (1..3): the RMSNorm output u, the raw inputs and scalars of those tokens,
    // and (backward) the du still collecting contributions and the token it belongs to
    float u1[kScEV] = {}, u2[kScEV] = {}, u3[kScEV] = {};
    float x1[kScEV] = {}, x2[kScEV] = {}, x3[kScEV] = {};
    float g1[kScEV] = {}, g2[kScEV] = {}, g3[kScEV] = {};
    float P1[kScEV] = {}, P2[kScEV] = {}, P3[kScEV] = {};
    float r1 = 0.f, r2 = 0.f, r3 = 0.f, sd1 = 0.f, sd2 = 0.f, sd3 = 0.f;
    int64_t pend1 = -1, pend2 = -1, pend3 = -1;
    int64_t seq_end = n_sw > 0 ? __ldg(p.offs + s + 1) : 0;

    // backward: a token's du is complete -> its row-dot partial, or its dv and dnorm_w share
    auto emit = [&](int64_t te, const float (&du)[kScEV], const float (&x)[kScEV], const float (&g)[kScEV], float rt,
                    float sd) {
        if (MODE == kScBwdDot) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kScEV; ++e) acc = fmaf(nw[e] * du[e], x[e], acc);
            acc = warp_sum(acc);
            if (lane == 0) p.token_dot_out[static_cast<size_t>(te) * p.nb + cb] = acc;
        } else if (MODE == kScBwdFinal) {
            const float k3 = rt * rt * rt * sd / static_cast<float>(p.d);
            float o[kScEV];
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                o[e] = g[e] + rt * nw[e] * du[e] - k3 * x[e];
                dnw[e] = fmaf(du[e] * x[e], rt, dnw[e]);
            }
            if (active) EV::store(p.out + static_cast<size_t>(te) * row_bytes + (c0 + lane * kScEV) * sizeof(E), o);
        }
    };
    auto flush = [&]() {
        if (pend3 >= 0) emit(pend3, P3, x3, g3, r3, sd3);
        if (pend2 >= 0) emit(pend2, P2, x2, g2, r2, sd2);
        if (pend1 >= 0) emit(pend1, P1, x1, g1, r1, sd1);
        pend1 = pend2 = pend3 = -1;
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            u1[e] = u2[e] = u3[e] = 0.f;
            P1[e] = P2[e] = P3[e] = 0.f;
        }
    };

    bool failed = false;
    int64_t q = 0;
    for (; q < n_sw; ++q) {
        const int64_t t = t_a + q * dil;
        // a new sequence: the taps reach back no further, and the pending du are complete
        if (t >= seq_end) {
            if (MODE != kScFwd) flush();
            else {
#pragma unroll
                for (int e = 0; e < kScEV; ++e) u1[e] = u2[e] = u3[e] = 0.f;
            }
            if (t >= t_hi) break;  // the backward's look-ahead stays in the chunk's last sequence
            while (s + 1 < p.num_seqs && t >= __ldg(p.offs + s + 1)) ++s;
            seq_end = __ldg(p.offs + s + 1);
        }
        // scalars of position q
        if (q - wr.w0 >= 64) {
            wr.w0 += 64;
            wr.lo = wr.nlo, wr.hi = wr.nhi;
            wr.nlo = scalar_at(wr.w0 + 64 + lane, false), wr.nhi = scalar_at(wr.w0 + 96 + lane, false);
            if (MODE == kScBwdFinal) {
                ws.w0 = wr.w0;
                ws.lo = ws.nlo, ws.hi = ws.nhi;
                ws.nlo = scalar_at(wr.w0 + 64 + lane, true), ws.nhi = scalar_at(wr.w0 + 96 + lane, true);
            }
        }
        const int wq = static_cast<int>(q - wr.w0);
        const float rt = __shfl_sync(0xffffffffu, wq < 32 ? wr.lo : wr.hi, wq & 31);
        const float sdt = MODE == kScBwdFinal ? __shfl_sync(0xffffffffu, wq < 32 ? ws.lo : ws.hi, wq & 31) : 0.f;

        // the row segments of token t
        const int st = static_cast<int>(q % S);
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[st], static_cast<uint32_t>((q / S) & 1)));
        if (!ok) {
            if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            failed = true;
            break;
        }
        const uint8_t *stage = ring + static_cast<size_t>(st) * 2 * seg_max;
        float x0[kScEV] = {}, y0[kScEV] = {};
        if (active) {
            EV::load_smem(stage + lane * EV::kBytes, x0);
            if (two && t >= t_lo) EV::load_smem(stage + seg_max + lane * EV::kBytes, y0);
        }
        __syncwarp();
        if (lane == 0 && issued < n_sw) issue(issued++);  // every lane holds its part of the stage

        float u0[kScEV], c[kScEV];
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            u0[e] = x0[e] * rt * nw[e];
            c[e] = bias[e] + K[0][e] * u0[e] + K[1][e] * u1[e] + K[2][e] * u2[e] + K[3][e] * u3[e];
        }
        const bool in_chunk = t >= t_lo && t < t_hi;
        if (MODE == kScFwd) {
            if (in_chunk && active) {
                float o[kScEV];
#pragma unroll
                for (int e = 0; e < kScEV; ++e) o[e] = c[e] * sc_sigmoid(c[e]) + x0[e] + y0[e];
                EV::store(p.out + static_cast<size_t>(t) * row_bytes + (c0 + lane * kScEV) * sizeof(E), o);
            }
        } else {
            // dc = dout SiLU'(c) for the chunk's tokens and the look-ahead; 0 for the lead-in
            float dc[kScEV];
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                const float sg = sc_sigmoid(c[e]);
                dc[e] = t >= t_lo ? y0[e] * sg * (1.0f + c[e] * (1.0f - sg)) : 0.f;
            }
            if (MODE == kScBwdFinal && in_chunk) {
#pragma unroll
                for (int e = 0; e < kScEV; ++e) {
                    db[e] += dc[e];
                    dK[0][e] = fmaf(dc[e], u0[e], dK[0][e]);
                    dK[1][e] = fmaf(dc[e], u1[e], dK[1][e]);
                    dK[2][e] = fmaf(dc[e], u2[e], dK[2][e]);
                    dK[3][e] = fmaf(dc[e], u3[e], dK[3][e]);
                }
            }
            // the token three taps back has all its contributions
            if (pend3 >= 0) {
                float du[kScEV];
#pragma unroll
                for (int e = 0; e < kScEV; ++e) du[e] = fmaf(K[3][e], dc[e], P3[e]);
                emit(pend3, du, x3, g3, r3, sd3);
            }
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                P3[e] = fmaf(K[2][e], dc[e], P2[e]);
                P2[e] = fmaf(K[1][e], dc[e], P1[e]);
                P1[e] = K[0][e] * dc[e];
            }
            pend3 = pend2, pend2 = pend1, pend1 = in_chunk ? t : -1;
        }
        // age the histories
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            u3[e] = u2[e], u2[e] = u1[e], u1[e] = u0[e];
            x3[e] = x2[e], x2[e] = x1[e], x1[e] = x0[e];
            g3[e] = g2[e], g2[e] = g1[e], g1[e] = y0[e];
        }
        r3 = r2, r2 = r1, r1 = rt;
        sd3 = sd2, sd2 = sd1, sd1 = sdt;
    }
    if (MODE != kScFwd && !failed) flush();

    if (MODE == kScBwdFinal && !failed) {
        // this work item's weight-gradient partial row: taps (by tap index), bias, norm weight
        float *prow = p.partial + static_cast<size_t>(k * dil + r) * (p.width + 2) * p.d;
        if (active) {
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                const int c = c0 + lane * kScEV + e;
                for (int i = 0; i < p.width; ++i) prow[static_cast<size_t>(i) * p.d + c] = dK[p.width - 1 - i][e];
                prow[static_cast<size_t>(p.width) * p.d + c] = db[e];
                prow[static_cast<size_t>(p.width + 1) * p.d + c] = dnw[e];
            }
        }
    }
    // copies issued but never consumed (the backward stops its look-ahead at a sequence end)
    if (lane == 0)
        for (int64_t qq = q; qq < issued; ++qq)
            if (!mbar_wait(&full[qq % S], static_cast<uint32_t>((qq / S) & 1)))
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
}

// ------------------------------------------------------------------------------- weight-gradient reduction

constexpr int kScRG = 64;
constexpr int kScCV = 4;

// S[j] = sum_p partial[p, j] over the (width + 2) * d columns: 64 groups of consecutive partials,
// each summed in ascending order, then the groups in ascending order.  Then
// dconv_w[c, i] = S[i * d + c], dbias[c] = S[width * d + c], dnorm_w[c] = S[(width + 1) * d + c].
__global__ void __launch_bounds__(kScRG *kScCV)
    conv_grad_reduce_kernel(const float *__restrict__ part, int32_t P, int32_t width, int32_t d,
                            float *__restrict__ dconv_w, float *__restrict__ dbias, float *__restrict__ dnorm_w) {
    __shared__ float sums[kScRG][kScCV];
    const int64_t ncol = static_cast<int64_t>(width + 2) * d;
    const int cv = threadIdx.x % kScCV;
    const int g = threadIdx.x / kScCV;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * kScCV + cv;
    const int per = (P + kScRG - 1) / kScRG;
    const int p0 = g * per;
    const int p1 = p0 + per < P ? p0 + per : P;
    float s = 0.f;
    if (col < ncol)
        for (int q = p0; q < p1; ++q) s += __ldcs(part + static_cast<size_t>(q) * ncol + col);
    sums[g][cv] = s;
    __syncthreads();
    if (g == 0 && col < ncol) {
        float t = sums[0][cv];
        for (int q = 1; q < kScRG; ++q) t += sums[q][cv];
        const int row = static_cast<int>(col / d), c = static_cast<int>(col % d);
        if (row < width) dconv_w[static_cast<size_t>(c) * width + row] = t;
        else if (row == width) {
            if (dbias) dbias[c] = t;
        } else dnorm_w[c] = t;
    }
}

// ------------------------------------------------------------------------------- host side

namespace {

int64_t sc_chunk(int64_t T) { return std::max<int64_t>(256, (T + 255) / 256); }

engram_status sc_check(const char *fn, engram_dtype dtype, int64_t T, int32_t d, int32_t width, int32_t dil,
                       int32_t num_seqs) {
    if (dtype_size(dtype) == 0) return fail(ENGRAM_ERR_DTYPE, "%s: dtype %d", fn, (int)dtype);
    if (T < 0 || d <= 0 || num_seqs < 1)
        return fail(ENGRAM_ERR_SHAPE, "%s: T = %lld, d = %d, num_seqs = %d", fn, (long long)T, d, num_seqs);
    if (width < 1 || width > kScAges) return fail(ENGRAM_ERR_SHAPE, "%s: width = %d (1..%d)", fn, width, kScAges);
    if (dil < 1) return fail(ENGRAM_ERR_SHAPE, "%s: dilation = %d", fn, dil);
    if ((static_cast<int64_t>(d) * dtype_size(dtype)) % 16 != 0)
        return fail(ENGRAM_ERR_ALIGN, "%s: a row of d = %d elements is not a multiple of 16 bytes", fn, d);
    if (d > kScMaxBlocks * kScCols) return fail(ENGRAM_ERR_SHAPE, "%s: d = %d exceeds %d", fn, d, kScMaxBlocks * kScCols);
    return ENGRAM_OK;
}

engram_status sc_ptrs(const char *fn, const void *const *ptrs, int n, int n_aligned, DeviceInfo *dev) {
    for (int i = 0; i < n_aligned; ++i)
        if (ptrs[i] && !aligned16(ptrs[i]))
            return fail(ENGRAM_ERR_ALIGN, "%s: pointer argument %d is not 16-byte aligned", fn, i);
    engram_status st = current_device(dev);
    if (st != ENGRAM_OK) return st;
    for (int i = 0; i < n; ++i)
        if (ptrs[i] && (st = check_device_ptr(ptrs[i], dev->device, fn)) != ENGRAM_OK) return st;
    return ENGRAM_OK;
}

template <typename E, int MODE>
engram_status sc_launch(const char *fn, ScParams prm, cudaStream_t s) {
    prm.stages = kScRingBytes / (2 * kScCols * static_cast<int>(sizeof(E)));
    const int smem = kScWarps * kScRingBytes + kScWarps * prm.stages * 8;
    engram_status st = set_smem(reinterpret_cast<const void *>(conv_stencil_kernel<E, MODE>), smem);
    if (st != ENGRAM_OK) return st;
    const int64_t items = prm.nchunks * prm.dil * prm.nb;
    const int64_t grid = (items + kScWarps - 1) / kScWarps;
    if (grid > 0x7fffffff) return fail(ENGRAM_ERR_SHAPE, "%s: too many work items", fn);
    conv_stencil_kernel<E, MODE><<<static_cast<unsigned>(grid), kScWarps * 32, smem, s>>>(prm);
    return check_launch(fn);
}

template <int MODE>
engram_status sc_dispatch(const char *fn, engram_dtype dtype, const ScParams &prm, cudaStream_t s) {
    return dtype == ENGRAM_F32 ? sc_launch<float, MODE>(fn, prm, s) : sc_launch<__nv_bfloat16, MODE>(fn, prm, s);
}

ScParams sc_params(const void *v, const float *norm_w, const float *conv_w, const float *bias, const float *rstd,
                   const int64_t *offs, int32_t num_seqs, int64_t T, int32_t d, int32_t width, int32_t dil,
                   const DeviceInfo &dev) {
    ScParams prm{};
    prm.v = static_cast<const uint8_t *>(v);
    prm.norm_w = norm_w;
    prm.conv_w = conv_w;
    prm.bias = bias;
    prm.rstd = rstd;
    prm.offs = offs;
    prm.status = dev.status_word;
    prm.T = T;
    prm.chunk = sc_chunk(T);
    prm.nchunks = (T + prm.chunk - 1) / prm.chunk;
    prm.num_seqs = num_seqs;
    prm.d = d;
    prm.width = width;
    prm.dil = dil;
    prm.nb = (d + kScCols - 1) / kScCols;
    return prm;
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" engram_status engram_short_conv_num_partials(int64_t T, int32_t dilation, int32_t *P) {
    if (!P) return fail(ENGRAM_ERR_NULL, "engram_short_conv_num_partials: NULL P");
    if (T < 0 || dilation < 1)
        return fail(ENGRAM_ERR_SHAPE, "engram_short_conv_num_partials: T = %lld, dilation = %d", (long long)T, dilation);
    const int64_t chunk = sc_chunk(T);
    const int64_t p = ((T + chunk - 1) / chunk) * dilation;
    if (p > 0x7fffffff) return fail(ENGRAM_ERR_SHAPE, "engram_short_conv_num_partials: too many partials");
    *P = static_cast<int32_t>(p);
    return ENGRAM_OK;
}

extern "C" engram_status engram_short_conv_dot_blocks(int32_t d, int32_t *nb) {
    if (!nb) return fail(ENGRAM_ERR_NULL, "engram_short_conv_dot_blocks: NULL nb");
    if (d <= 0) return fail(ENGRAM_ERR_SHAPE, "engram_short_conv_dot_blocks: d = %d", d);
    *nb = (d + kScCols - 1) / kScCols;
    return ENGRAM_OK;
}

extern "C" engram_status engram_short_conv_fwd(const void *v, const void *h, engram_dtype dtype, const float *norm_w,
                                               const float *conv_w, const float *bias, const int64_t *seq_offsets,
                                               int32_t num_seqs, int64_t T, int32_t d, int32_t width,
                                               int32_t dilation, float eps, void *out, float *rstd,
                                               engram_stream_t stream) {
    const char *fn = "engram_short_conv_fwd";
    engram_status st = sc_check(fn, dtype, T, d, width, dilation, num_seqs);
    if (st != ENGRAM_OK) return st;
    if (!norm_w || !conv_w || !seq_offsets) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (T == 0) return ENGRAM_OK;
    if (!v || !out || !rstd) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (out == v) return fail(ENGRAM_ERR_SHAPE, "%s: out may not alias V~ (later tokens read it as taps)", fn);
    const void *ptrs[] = {v, h, out, norm_w, conv_w, bias, seq_offsets, rstd};
    DeviceInfo dev;
    if ((st = sc_ptrs(fn, ptrs, 8, 3, &dev)) != ENGRAM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t grid = cap_grid(std::min<int64_t>((T + 7) / 8, static_cast<int64_t>(dev.num_sms) * 8));
    if (dtype == ENGRAM_F32)
        conv_rstd_kernel<float><<<static_cast<unsigned>(grid), 256, 0, s>>>(static_cast<const uint8_t *>(v), T, d,
                                                                            eps, rstd);
    else
        conv_rstd_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, 0, s>>>(static_cast<const uint8_t *>(v),
                                                                                    T, d, eps, rstd);
    if ((st = check_launch(fn)) != ENGRAM_OK) return st;
    ScParams prm = sc_params(v, norm_w, conv_w, bias, rstd, seq_offsets, num_seqs, T, d, width, dilation, dev);
    prm.x2 = static_cast<const uint8_t *>(h);
    prm.out = static_cast<uint8_t *>(out);
    return sc_dispatch<kScFwd>(fn, dtype, prm, s);
}

extern "C" engram_status engram_short_conv_bwd(const void *dout, const void *v, engram_dtype dtype,
                                               const float *norm_w, const float *conv_w, const float *bias,
                                               const float *rstd, const int64_t *seq_offsets, int32_t num_seqs,
                                               int64_t T, int32_t d, int32_t width, int32_t dilation, void *dv,
                                               float *token_dot, float *dw_partial, int32_t P,
                                               engram_stream_t stream) {
    const char *fn = "engram_short_conv_bwd";
    engram_status st = sc_check(fn, dtype, T, d, width, dilation, num_seqs);
    if (st != ENGRAM_OK) return st;
    int32_t want = 0;
    if ((st = engram_short_conv_num_partials(T, dilation, &want)) != ENGRAM_OK) return st;
    if (P != want) return fail(ENGRAM_ERR_SHAPE, "%s: P = %d, engram_short_conv_num_partials gives %d", fn, P, want);
    if (!norm_w || !conv_w || !seq_offsets) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (T == 0) return ENGRAM_OK;
    if (!dout || !v || !rstd || !dv || !token_dot || !dw_partial) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (dv == v || dv == dout) return fail(ENGRAM_ERR_SHAPE, "%s: dv may not alias V~ or dout", fn);
    const void *ptrs[] = {dout, v, dv, norm_w, conv_w, bias, rstd, seq_offsets, token_dot, dw_partial};
    DeviceInfo dev;
    if ((st = sc_ptrs(fn, ptrs, 10, 3, &dev)) != ENGRAM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ScParams prm = sc_params(v, norm_w, conv_w, bias, rstd, seq_offsets, num_seqs, T, d, width, dilation, dev);
    prm.x2 = static_cast<const uint8_t *>(dout);
    prm.token_dot_out = token_dot;
    if ((st = sc_dispatch<kScBwdDot>(fn, dtype, prm, s)) != ENGRAM_OK) return st;
    prm.token_dot = token_dot;
    prm.token_dot_out = nullptr;
    prm.out = static_cast<uint8_t *>(dv);
    prm.partial = dw_partial;
    return sc_dispatch<kScBwdFinal>(fn, dtype, prm, s);
}

extern "C" engram_status engram_short_conv_grad_reduce(const float *dw_partial, int32_t P, int32_t width, int32_t d,
                                                       float *dconv_w, float *dbias, float *dnorm_w,
                                                       engram_stream_t stream) {
    const char *fn = "engram_short_conv_grad_reduce";
    if (P < 0 || d <= 0 || width < 1 || width > kScAges)
        return fail(ENGRAM_ERR_SHAPE, "%s: P = %d, d = %d, width = %d", fn, P, d, width);
    if ((!dw_partial && P > 0) || !dconv_w || !dnorm_w) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    const void *ptrs[] = {dw_partial, dconv_w, dbias, dnorm_w};
    DeviceInfo dev;
    engram_status st = sc_ptrs(fn, ptrs, 4, 0, &dev);
    if (st != ENGRAM_OK) return st;
    const int64_t ncol = static_cast<int64_t>(width + 2) * d;
    conv_grad_reduce_kernel<<<static_cast<unsigned>((ncol + kScCV - 1) / kScCV), kScRG * kScCV, 0,
                              reinterpret_cast<cudaStream_t>(stream)>>>(dw_partial, P, width, d, dconv_w, dbias,
                                                                         dnorm_w);
    return check_launch(fn);
}
