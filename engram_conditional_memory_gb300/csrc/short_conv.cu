// The short convolution after the gate (NEXT-2): Y = SiLU(Conv1D(RMSNorm(V~))) + V~, H <- H + Y,
// a depthwise causal convolution of `width` taps (at most 4) with a dilation, per sequence
// (TileLang tutorial, ch. 34 "TileKernels: Engram and mHC", sec. 1.2 item 4: kernel size 4,
// dilation the largest N-gram order).  Tap i multiplies the token (width - 1 - i) * dilation steps
// back, so tap width - 1 is the current token (torch's depthwise conv1d layout with left padding).
//
// GB300 design.  The convolution couples tokens only along time, one channel at a time, and the
// RMSNorm couples channels only within a token, through one scalar.  So:
//   * conv_rstd_kernel: a warp per token computes rstd = 1/sqrt(mean(V~^2) + eps);
//   * conv_fwd_kernel: persistent CTAs, each on one 512-byte channel block, stream tiles of 64
//     tokens plus the taps' halo into shared memory with 1-D bulk (TMA) copies, two or three tiles
//     in flight, and compute every output from the tile: the taps are read back from shared memory
//     instead of being carried along time, so there is no per-token bookkeeping;
//   * conv_stencil_kernel (the backward): a warp owns 128 channels of one residue class
//     t = r (mod dilation).  Every tap of a class token lies in the same class, so the warp sweeps
//     its tokens in time order carrying the last three taps' inputs and the du still collecting
//     contributions in registers.  Each warp streams its rows (V~ and dout) through its own ring of
//     shared-memory stages filled by bulk copies that its lane 0 issues, and keeps a stage resident
//     for the three tokens that read it back.  Per-token scalars (rstd, the row dots) come 64
//     tokens at a time, two per lane, one window ahead, and reach a token by a shuffle.
// The backward is two sweeps: the first gives each token's partial dot s = sum_j norm_w du V~ over
// the warp's channels and the taps' and bias's gradient partials of its (time chunk, residue) work
// item, the second the full dV~ = dout + rstd norm_w du - rstd^3 V~ s / d with s summed over the
// channel blocks in a fixed order, and the norm weight's partials.  conv_grad_reduce_kernel sums
// the partials in a fixed order.  The time chunks depend on T only, so the weight gradients are
// bitwise reproducible on any GPU.
#include <algorithm>

#include "engram_internal.cuh"

namespace engram {

constexpr int kScWarps = 8;             // warps per CTA, each an independent work item
constexpr int kScEV = 4;                // channels per lane
constexpr int kScCols = 32 * kScEV;     // channels per warp
constexpr int kScAges = 4;              // taps: width <= 4
constexpr int kScRingBytes = 8192;      // per warp: stages x (V~ segment + second segment)
constexpr int kScMaxBlocks = 64;        // channel blocks per row: d <= 64 * 128

enum ScMode { kScBwdDot = 1, kScBwdFinal = 2 };  // the backward sweeps

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
        uint4 u;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                     : "r"(smem_addr(p)));
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
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(smem_addr(p)));
        x[0] = __uint_as_float(a << 16), x[1] = __uint_as_float(a & 0xffff0000u);
        x[2] = __uint_as_float(b << 16), x[3] = __uint_as_float(b & 0xffff0000u);
    }
    __device__ __forceinline__ static void store(uint8_t *p, const float (&x)[4]) {
        *reinterpret_cast<uint2 *>(p) =
            make_uint2(Vec<__nv_bfloat16>::pack2(x[0], x[1]), Vec<__nv_bfloat16>::pack2(x[2], x[3]));
    }
};

// SiLU's sigmoid with the fast exponential and division (a few ulp; the outputs are rounded far
// coarser, and the tolerances carry the bound).
__device__ __forceinline__ float sc_sigmoid_fast(float c) { return __fdividef(1.0f, 1.0f + __expf(-c)); }

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
#pragma unroll 8
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

// ------------------------------------------------------------------------------- forward

constexpr int kScTileTokens = 64;       // tokens per forward tile
constexpr int kScMaxDil = 32;           // forward: the halo of (width - 1) * dilation rows stays small

// Shared memory of one tile buffer: rows [rows_max][32] uint4, rstd [rows_max], sequence starts
// [kScTileTokens] int64; two buffers, then two mbarriers.
__host__ __device__ inline int sc_fwd_buf_bytes(int width, int dil) {
    const int rows = kScTileTokens + (width - 1) * dil;
    // rounded to 128 bytes: the second buffer's rows are bulk-copy destinations (16-byte aligned)
    return (rows * 512 + ((rows + 1) & ~1) * 4 + kScTileTokens * 8 + 127) & ~127;
}
// three tile buffers where they fit two CTAs per SM, else two
inline int sc_fwd_nbuf(int width, int dil) { return 3 * sc_fwd_buf_bytes(width, dil) + 24 <= 113 * 1024 ? 3 : 2; }
inline int sc_fwd_smem(int width, int dil) { return sc_fwd_nbuf(width, dil) * (sc_fwd_buf_bytes(width, dil) + 8); }

struct ScFwdParams {
    const uint8_t *v, *h;
    const float *norm_w, *conv_w, *bias, *rstd;
    const int64_t *offs;
    uint8_t *out;
    uint32_t *status;
    int64_t T;
    int32_t num_seqs, d, width, dil, nblk, ntiles, nbuf;
};

// Persistent CTAs, each on one channel block of 512 bytes (its taps, folded with norm_w, loaded
// once) and the tiles j, j + J, ... of kScTileTokens tokens (J CTAs per block).  A tile's V~ rows and
// the halo of (width - 1) * dilation rows before it reach shared memory by 1-D bulk (TMA) copies,
// one row segment per lane of warp 0, completing on the buffer's mbarrier; the next one or two
// tiles' copies are in flight while this one is computed.  Lane l of warp w computes channel vector l of the
// tile's tokens w, w + 8, ...:
//   conv = bias + sum_a (conv_w[width-1-a] norm_w) rstd[t - a dil] V~[t - a dil],
//   out  = H + SiLU(conv) + V~,
// with taps before the token's sequence start left out.
template <typename E>
__global__ void __launch_bounds__(256, 2) conv_fwd_kernel(const __grid_constant__ ScFwdParams p) {
    using V = Vec<E>;
    constexpr int N = V::N;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int width = p.width, dil = p.dil;
    const int halo = (width - 1) * dil;
    const int rows_max = kScTileTokens + halo;
    const int buf_bytes = sc_fwd_buf_bytes(width, dil);
    const int nbuf = p.nbuf;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(nbuf) * buf_bytes);
    const int nvec = p.d / N;
    const int cb = static_cast<int>(blockIdx.x % p.nblk);
    const int J = static_cast<int>(gridDim.x / p.nblk);
    const int j0 = static_cast<int>(blockIdx.x / p.nblk);
    if (j0 >= J) return;  // whole CTA: a grid that is not a multiple of the block count
    const int jv = cb * 32 + lane;
    const bool active = jv < nvec;
    const int jv_c = active ? jv : 0;
    const int nv_blk = nvec - cb * 32 < 32 ? nvec - cb * 32 : 32;
    const uint32_t seg = static_cast<uint32_t>(nv_blk) * 16u;
    const size_t row_bytes = static_cast<size_t>(nvec) * 16;

    auto tile_rows = [&](int b) { return reinterpret_cast<uint4(*)[32]>(smem + static_cast<size_t>(b) * buf_bytes); };
    auto tile_rs = [&](int b) {
        return reinterpret_cast<float *>(smem + static_cast<size_t>(b) * buf_bytes + static_cast<size_t>(rows_max) * 512);
    };
    auto tile_ss = [&](int b) {
        return reinterpret_cast<int64_t *>(smem + static_cast<size_t>(b) * buf_bytes +
                                           static_cast<size_t>(rows_max) * 512 + ((rows_max + 1) & ~1) * 4);
    };
    // tile j covers tokens [j K, min(T, (j + 1) K)) and buffers rows from max(0, j K - halo)
    auto first_row = [&](int j) {
        const int64_t t0 = static_cast<int64_t>(j) * kScTileTokens;
        return t0 - halo > 0 ? t0 - halo : static_cast<int64_t>(0);
    };
    auto tile_end = [&](int j) {
        const int64_t t1 = (static_cast<int64_t>(j) + 1) * kScTileTokens;
        return t1 < p.T ? t1 : p.T;
    };
    // start tile j's copies into buffer b (warp 0), and its rstd and sequence starts (all threads)
    auto stage_tile = [&](int j, int b) {
        const int64_t r0 = first_row(j), t0 = static_cast<int64_t>(j) * kScTileTokens, t1 = tile_end(j);
        const int nrows = static_cast<int>(t1 - r0);
        if (warp == 0) {
            if (lane == 0) mbar_arrive_expect_tx(&bars[b], seg * static_cast<uint32_t>(nrows));
            __syncwarp();
            uint4(*rows)[32] = tile_rows(b);
            for (int i = lane; i < nrows; i += 32)
                bulk_load_plain(&rows[i][0], p.v + static_cast<size_t>(r0 + i) * row_bytes + static_cast<size_t>(cb) * 512,
                                seg, &bars[b]);
        }
        float *rs = tile_rs(b);
        for (int i = threadIdx.x; i < nrows; i += blockDim.x) rs[i] = __ldg(p.rstd + r0 + i);
        if (threadIdx.x < t1 - t0) tile_ss(b)[threadIdx.x] = __ldg(p.offs + sc_seq_of(p.offs, p.num_seqs, t0 + threadIdx.x));
    };

    // this lane's channels: the taps by age folded with norm_w, and the bias (16-byte loads)
    float KW[kScAges][N], bv[N];
    {
        float nw[N], cw[N][kScAges];
        const float4 *nw4 = reinterpret_cast<const float4 *>(p.norm_w + static_cast<size_t>(jv_c) * N);
        const float4 *b4 = p.bias ? reinterpret_cast<const float4 *>(p.bias + static_cast<size_t>(jv_c) * N) : nullptr;
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 a = __ldg(nw4 + q);
            nw[4 * q] = a.x, nw[4 * q + 1] = a.y, nw[4 * q + 2] = a.z, nw[4 * q + 3] = a.w;
            const float4 bb = b4 ? __ldg(b4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
            bv[4 * q] = bb.x, bv[4 * q + 1] = bb.y, bv[4 * q + 2] = bb.z, bv[4 * q + 3] = bb.w;
        }
#pragma unroll
        for (int e = 0; e < N; ++e) {
            const size_t c = static_cast<size_t>(jv_c) * N + e;
            if (width == kScAges) {
                const float4 w4 = __ldg(reinterpret_cast<const float4 *>(p.conv_w + c * kScAges));
                cw[e][0] = w4.x, cw[e][1] = w4.y, cw[e][2] = w4.z, cw[e][3] = w4.w;
            } else {
#pragma unroll
                for (int i = 0; i < kScAges; ++i) cw[e][i] = i < width ? __ldg(p.conv_w + c * width + i) : 0.f;
            }
#pragma unroll
            for (int a = 0; a < kScAges; ++a) KW[a][e] = a < width ? cw[e][width - 1 - a] * nw[e] : 0.f;
        }
    }
    const uint4 *h4 = p.h ? reinterpret_cast<const uint4 *>(p.h) + jv_c : nullptr;
    uint4 *o4 = reinterpret_cast<uint4 *>(p.out) + jv_c;

    if (threadIdx.x == 0) {
        for (int q = 0; q < nbuf; ++q) mbar_init(&bars[q], 1);
        mbar_init_fence();
    }
    __syncthreads();
    for (int q = 0; q < nbuf - 1 && j0 + q * J < p.ntiles; ++q) stage_tile(j0 + q * J, q);
    __syncthreads();  // the first tiles' rstd and sequence starts

    constexpr int kPer = kScTileTokens / 8;  // tokens per warp and tile, their H rows in two halves
    constexpr int kHalf = kPer / 2;
    int it = 0;
    for (int j = j0; j < p.ntiles; j += J, ++it) {
        const int b = it % nbuf;
        const uint32_t phase = static_cast<uint32_t>((it / nbuf) & 1);
        const int jn = j + (nbuf - 1) * J;
        const int bn = (it + nbuf - 1) % nbuf;
        if (jn < p.ntiles) stage_tile(jn, bn);  // freed by the previous tile's closing barrier
        const int64_t t0 = static_cast<int64_t>(j) * kScTileTokens, t1 = tile_end(j), r0 = first_row(j);
        uint4 hv[kHalf];
        auto load_h = [&](int k0) {
#pragma unroll
            for (int k = 0; k < kHalf; ++k) {
                const int64_t t = t0 + warp + 8 * (k0 + k);
                hv[k] = (h4 && t < t1) ? __ldcs(h4 + static_cast<size_t>(t) * nvec) : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        load_h(0);
        const bool ok = mbar_wait(&bars[b], phase);
        if (__syncthreads_or(!ok)) {
            // a copy that never landed: report, and let thread 0 wait (bounded) for what is in flight
            if (threadIdx.x == 0) {
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                for (int q = 0; q < nbuf - 1 && j + q * J < p.ntiles; ++q)
                    mbar_wait(&bars[(it + q) % nbuf], static_cast<uint32_t>(((it + q) / nbuf) & 1));
            }
            return;
        }
        uint4(*rows)[32] = tile_rows(b);
        const float *rs = tile_rs(b);
        const int64_t *ss = tile_ss(b);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if (k == kHalf) load_h(kHalf);
            const int lt = warp + 8 * k;
            const int64_t t = t0 + lt;
            if (t >= t1) break;
            const int64_t s0 = ss[lt];
            float c[N], x0[N];
#pragma unroll
            for (int e = 0; e < N; ++e) c[e] = bv[e];
#pragma unroll
            for (int a = 0; a < kScAges; ++a) {
                const int64_t ta = t - static_cast<int64_t>(a) * dil;
                if (a < width && ta >= s0) {
                    const int ri = static_cast<int>(ta - r0);
                    float x[N];
                    V::unpack(rows[ri][lane], x);
                    const float ra = rs[ri];
#pragma unroll
                    for (int e = 0; e < N; ++e) c[e] = fmaf(KW[a][e], x[e] * ra, c[e]);
                    if (a == 0) {
#pragma unroll
                        for (int e = 0; e < N; ++e) x0[e] = x[e];
                    }
                }
            }
            float y[N];
            V::unpack(hv[k % kHalf], y);
            float o[N];
#pragma unroll
            for (int e = 0; e < N; ++e) o[e] = fmaf(c[e], sc_sigmoid_fast(c[e]), x0[e] + y[e]);
            if (active) __stcs(o4 + static_cast<size_t>(t) * nvec, V::pack(o));
        }
        __syncthreads();  // buffer b is free; the next tile's rstd and sequence starts are visible
    }
}

// ------------------------------------------------------------------------------- the stencil sweep

// Per-token scalars of the warp's sweep (indexed by the sweep position q), 64 at a time: lane l
// holds positions w0 + l and w0 + 32 + l of the current window and the next window's two.
struct ScWindow {
    float lo, hi, nlo, nhi;
};

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
    int64_t n_sw = 0, t_a = t_first;
    int s = 0;
    if (t_first < t_hi) {
        s = sc_seq_of(p.offs, p.num_seqs, t_first);
        const int64_t hist = t_first - static_cast<int64_t>(kScAges - 1) * dil;
        const int64_t s0 = __ldg(p.offs + s);
        t_a = first_class(hist > s0 ? hist : s0);
        int64_t t_b = t_hi + static_cast<int64_t>(kScAges - 1) * dil;
        if (t_b > p.T) t_b = p.T;
        n_sw = (t_b - t_a + dil - 1) / dil;
    }

    // lane 0 streams the sweep's rows: a lead-in token (before the chunk) needs V~ only.  A stage
    // stays resident for three tokens after its own, which read it back as their taps' inputs.
    const uint64_t pol = l2_evict_first_policy();
    constexpr bool two = true;
    const size_t col_off = static_cast<size_t>(c0) * sizeof(E);
    const size_t step_bytes = static_cast<size_t>(dil) * row_bytes;
    const uint8_t *src_v = p.v + static_cast<size_t>(t_a) * row_bytes + col_off;
    const uint8_t *src_2 = two ? p.x2 + static_cast<size_t>(t_a) * row_bytes + col_off : nullptr;
    int64_t issued = 0, t_issue = t_a;
    int ist = 0;
    auto issue = [&]() {
        const bool second = two && t_issue >= t_lo;
        uint8_t *dst = ring + static_cast<size_t>(ist) * 2 * seg_max;
        mbar_arrive_expect_tx(&full[ist], second ? 2 * seg : seg);
        bulk_load(dst, src_v, seg, &full[ist], pol);
        if (second) bulk_load(dst + seg_max, src_2, seg, &full[ist], pol);
        src_v += step_bytes;
        if (two) src_2 += step_bytes;
        t_issue += dil;
        ++issued;
        if (++ist == S) ist = 0;
    };
    if (lane == 0) {
        for (int q = 0; q < S; ++q) mbar_init(&full[q], 1);
        mbar_init_fence();
        while (issued < S && issued < n_sw) issue();
    }
    __syncwarp();

    // positions q of the sweep (token t_a + q dil): the chunk's tokens are [q_lo, q_hi)
    const int64_t n_sw_l = n_sw;
    const int nq = static_cast<int>(n_sw_l);
    const int q_lo = static_cast<int>((t_first - t_a) / dil);
    const int q_hi = static_cast<int>((t_hi - t_a + dil - 1) / dil);
    const int nb = p.nb;
    const float inv_d = 1.0f / static_cast<float>(p.d);
    const int num_seqs = p.num_seqs;
    const int64_t *offs = p.offs;
    const float *rstd_p = p.rstd;
    const float *tdot = p.token_dot;
    float *tdot_out = p.token_dot_out;
    auto pos_of = [&](int64_t tt) {  // first position whose token is >= tt
        return tt <= t_a ? 0 : static_cast<int>((tt - t_a + dil - 1) / dil);
    };

    // scalar windows: rstd, and the backward's row-dot totals (column 0 of token_dot) in the final sweep
    auto scalar_at = [&](int q, bool dot) -> float {
        if (q >= nq) return 0.f;
        const int64_t t = t_a + static_cast<int64_t>(q) * dil;
        return dot ? __ldg(tdot + static_cast<size_t>(t) * nb) : __ldg(rstd_p + t);
    };
    ScWindow wr{0.f, 0.f, scalar_at(lane, false), scalar_at(32 + lane, false)};
    ScWindow ws{0.f, 0.f, 0.f, 0.f};
    if (MODE == kScBwdFinal) ws.nlo = scalar_at(lane, true), ws.nhi = scalar_at(32 + lane, true);
    int w0 = -64;

    // histories by age (1..3): the RMSNorm output u and the scalars of those tokens, and (backward)
    // the du still collecting contributions and whether its token is the chunk's.  The raw rows of
    // those tokens stay in their stages.
    float u1[kScEV] = {}, u2[kScEV] = {}, u3[kScEV] = {};
    float P1[kScEV] = {}, P2[kScEV] = {}, P3[kScEV] = {};
    float r1 = 0.f, r2 = 0.f, r3 = 0.f, sd1 = 0.f, sd2 = 0.f, sd3 = 0.f;
    bool pend1 = false, pend2 = false, pend3 = false;
    int q_seq_end = nq > 0 ? pos_of(__ldg(offs + s + 1)) : 0;
    float dK[kScAges][kScEV], db[kScEV], dnw[kScEV];
#pragma unroll
    for (int e = 0; e < kScEV; ++e) {
        db[e] = dnw[e] = 0.f;
#pragma unroll
        for (int a = 0; a < kScAges; ++a) dK[a][e] = 0.f;
    }
    int st = 0;          // stage of position q
    uint32_t ph = 0;     // its phase
    auto stage_back = [&](int a) { return st - a < 0 ? st - a + S : st - a; };
    // this lane's output row segment of position q, and the row-dot entry
    uint8_t *out_q = p.out ? p.out + static_cast<size_t>(t_a) * row_bytes + col_off + lane * EV::kBytes : nullptr;
    float *dot_q = tdot_out ? tdot_out + static_cast<size_t>(t_a) * nb + cb : nullptr;
    const size_t dot_step = static_cast<size_t>(dil) * nb;

    // backward: a token's du is complete -> its row-dot partial, or its dv and dnorm_w share.  Its
    // V~ and dout are read back from its stage, `age` positions behind the current one.
    auto emit = [&](int age, const float (&du)[kScEV], float rt, float sd) {
        float x[kScEV] = {}, g[kScEV] = {};
        const uint8_t *stg = ring + static_cast<size_t>(stage_back(age)) * 2 * seg_max;
        if (active) {
            EV::load_smem(stg + lane * EV::kBytes, x);
            if (MODE == kScBwdFinal) EV::load_smem(stg + seg_max + lane * EV::kBytes, g);
        }
        if (MODE == kScBwdDot) {
            float acc = 0.f;
#pragma unroll
            for (int e = 0; e < kScEV; ++e) acc = fmaf(nw[e] * du[e], x[e], acc);
            acc = warp_sum(acc);
            if (lane == 0) dot_q[-static_cast<ptrdiff_t>(age * dot_step)] = acc;
        } else if (MODE == kScBwdFinal) {
            const float k3 = rt * rt * rt * sd * inv_d;
            float o[kScEV];
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                o[e] = g[e] + rt * nw[e] * du[e] - k3 * x[e];
                dnw[e] = fmaf(du[e] * x[e], rt, dnw[e]);
            }
            if (active) EV::store(out_q - static_cast<ptrdiff_t>(age * step_bytes), o);
        }
    };
    // the pending du have no more contributions (a sequence ended, or the sweep did); called
    // before position q is processed, so the pending tokens sit 1..3 positions back
    auto flush = [&]() {
        if (pend3) emit(3, P3, r3, sd3);
        if (pend2) emit(2, P2, r2, sd2);
        if (pend1) emit(1, P1, r1, sd1);
        pend1 = pend2 = pend3 = false;
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            u1[e] = u2[e] = u3[e] = 0.f;
            P1[e] = P2[e] = P3[e] = 0.f;
        }
    };

    bool failed = false;
    int q = 0;
    for (; q < nq; ++q) {
        // a new sequence: the taps reach back no further, and the pending du are complete
        if (q >= q_seq_end) {
            flush();
            if (q >= q_hi) break;  // the backward's look-ahead stays in the chunk's last sequence
            const int64_t t = t_a + static_cast<int64_t>(q) * dil;
            while (s + 1 < num_seqs && t >= __ldg(offs + s + 1)) ++s;
            q_seq_end = pos_of(__ldg(offs + s + 1));
            if (q_seq_end <= q) q_seq_end = q + 1;  // malformed offsets: treat the token as its own sequence
        }
        // scalars of position q
        if (q - w0 >= 64) {
            w0 += 64;
            wr.lo = wr.nlo, wr.hi = wr.nhi;
            wr.nlo = scalar_at(w0 + 64 + lane, false), wr.nhi = scalar_at(w0 + 96 + lane, false);
            if (MODE == kScBwdFinal) {
                ws.lo = ws.nlo, ws.hi = ws.nhi;
                ws.nlo = scalar_at(w0 + 64 + lane, true), ws.nhi = scalar_at(w0 + 96 + lane, true);
            }
        }
        const int wq = q - w0;
        const float rt = __shfl_sync(0xffffffffu, wq < 32 ? wr.lo : wr.hi, wq & 31);
        const float sdt = MODE == kScBwdFinal ? __shfl_sync(0xffffffffu, wq < 32 ? ws.lo : ws.hi, wq & 31) : 0.f;

        // the row segments of position q
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&full[st], ph));
        if (!ok) {
            if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            failed = true;
            break;
        }
        const uint8_t *stage = ring + static_cast<size_t>(st) * 2 * seg_max;
        const bool in_chunk = q >= q_lo && q < q_hi;
        const bool led = q < q_lo;  // lead-in: the taps' inputs only
        float x0[kScEV] = {}, y0[kScEV] = {};
        if (active) {
            EV::load_smem(stage + lane * EV::kBytes, x0);
            if (two && !led) EV::load_smem(stage + seg_max + lane * EV::kBytes, y0);
        }

        float u0[kScEV], c[kScEV];
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            u0[e] = x0[e] * rt * nw[e];
            c[e] = fmaf(K[3][e], u3[e], fmaf(K[2][e], u2[e], fmaf(K[1][e], u1[e], fmaf(K[0][e], u0[e], bias[e]))));
        }
        {
            // dc = dout SiLU'(c) for the chunk's tokens and the look-ahead; 0 for the lead-in
            float dc[kScEV];
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                const float sg = sc_sigmoid_fast(c[e]);
                dc[e] = led ? 0.f : y0[e] * sg * fmaf(c[e], 1.0f - sg, 1.0f);
            }
            if (MODE == kScBwdDot && in_chunk) {  // the taps' and the bias's gradients, in the first sweep
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
            if (pend3) {
                float du[kScEV];
#pragma unroll
                for (int e = 0; e < kScEV; ++e) du[e] = fmaf(K[3][e], dc[e], P3[e]);
                emit(3, du, r3, sd3);
            }
#pragma unroll
            for (int e = 0; e < kScEV; ++e) {
                P3[e] = fmaf(K[2][e], dc[e], P2[e]);
                P2[e] = fmaf(K[1][e], dc[e], P1[e]);
                P1[e] = K[0][e] * dc[e];
            }
            pend3 = pend2, pend2 = pend1, pend1 = in_chunk;
        }
        // age the histories and move to the next position
#pragma unroll
        for (int e = 0; e < kScEV; ++e) u3[e] = u2[e], u2[e] = u1[e], u1[e] = u0[e];
        r3 = r2, r2 = r1, r1 = rt;
        sd3 = sd2, sd2 = sd1, sd1 = sdt;
        if (++st == S) {
            st = 0;
            ph ^= 1u;
        }
        if (out_q) out_q += step_bytes;
        if (dot_q) dot_q += dot_step;
        // positions q - 2 .. q stay resident; the stage of q - 3 takes the next row
        __syncwarp();
        if (lane == 0 && issued < n_sw_l && issued < q + S - 2) issue();
    }
    if (!failed) flush();

    if (!failed && active) {
        // this work item's weight-gradient partial row: the taps (by tap index) and the bias from the
        // first sweep, the norm weight from the second
        const int d = p.d, width = p.width;
        float *prow = p.partial + static_cast<size_t>(k * dil + r) * (width + 2) * d;
#pragma unroll
        for (int e = 0; e < kScEV; ++e) {
            const int c = c0 + lane * kScEV + e;
            if (MODE == kScBwdDot) {
                for (int i = 0; i < width; ++i) prow[static_cast<size_t>(i) * d + c] = dK[width - 1 - i][e];
                prow[static_cast<size_t>(width) * d + c] = db[e];
            } else {
                prow[static_cast<size_t>(width + 1) * d + c] = dnw[e];
            }
        }
    }
    // copies issued but never consumed (the backward stops its look-ahead at a sequence end)
    if (lane == 0)
        for (int64_t qq = q; qq < issued; ++qq)
            if (!mbar_wait(&full[qq % S], static_cast<uint32_t>((qq / S) & 1)))
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
}

// The row-dot total of each token, its nb channel-block partials in ascending order, written to
// the row's first entry (which the final sweep reads).
__global__ void __launch_bounds__(256) conv_dot_total_kernel(float *__restrict__ token_dot, int64_t T, int32_t nb) {
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; t < T;
         t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float *row = token_dot + static_cast<size_t>(t) * nb;
        float s = 0.f;
        for (int b = 0; b < nb; ++b) s += row[b];
        row[0] = s;
    }
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
    if (dilation > kScMaxDil) return fail(ENGRAM_ERR_SHAPE, "%s: dilation = %d exceeds %d", fn, dilation, kScMaxDil);
    if (out == v) return fail(ENGRAM_ERR_SHAPE, "%s: out may not alias V~ (later tokens read it as taps)", fn);
    const void *ptrs[] = {v, h, out, norm_w, conv_w, bias, seq_offsets, rstd};
    DeviceInfo dev;
    if ((st = sc_ptrs(fn, ptrs, 8, 6, &dev)) != ENGRAM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t rgrid = cap_grid(std::min<int64_t>((T + 7) / 8, static_cast<int64_t>(dev.num_sms) * 8));
    if (dtype == ENGRAM_F32)
        conv_rstd_kernel<float><<<static_cast<unsigned>(rgrid), 256, 0, s>>>(static_cast<const uint8_t *>(v), T, d,
                                                                            eps, rstd);
    else
        conv_rstd_kernel<__nv_bfloat16><<<static_cast<unsigned>(rgrid), 256, 0, s>>>(static_cast<const uint8_t *>(v),
                                                                                    T, d, eps, rstd);
    if ((st = check_launch(fn)) != ENGRAM_OK) return st;
    const int nvec = static_cast<int>(static_cast<int64_t>(d) * dtype_size(dtype) / 16);
    ScFwdParams fp{};
    fp.v = static_cast<const uint8_t *>(v);
    fp.h = static_cast<const uint8_t *>(h);
    fp.norm_w = norm_w;
    fp.conv_w = conv_w;
    fp.bias = bias;
    fp.rstd = rstd;
    fp.offs = seq_offsets;
    fp.out = static_cast<uint8_t *>(out);
    fp.status = dev.status_word;
    fp.T = T;
    fp.num_seqs = num_seqs;
    fp.d = d;
    fp.width = width;
    fp.dil = dilation;
    fp.nblk = (nvec + 31) / 32;
    const int64_t ntiles = (T + kScTileTokens - 1) / kScTileTokens;
    if (ntiles > 0x7fffffff) return fail(ENGRAM_ERR_SHAPE, "%s: too many tokens", fn);
    fp.ntiles = static_cast<int32_t>(ntiles);
    fp.nbuf = sc_fwd_nbuf(width, dilation);
    // two CTAs per SM, each on one channel block; J CTAs share a block's tiles
    const int64_t per_block = std::max<int64_t>(1, std::min<int64_t>(ntiles, (2 * dev.num_sms + fp.nblk - 1) / fp.nblk));
    const int64_t grid = cap_grid(per_block * fp.nblk) / fp.nblk * fp.nblk;
    if (grid < fp.nblk) return fail(ENGRAM_ERR_SHAPE, "%s: the CTA cap is below %d channel blocks", fn, fp.nblk);
    const int smem = sc_fwd_smem(width, dilation);
    if (dtype == ENGRAM_F32) {
        if ((st = set_smem(reinterpret_cast<const void *>(conv_fwd_kernel<float>), smem)) != ENGRAM_OK) return st;
        conv_fwd_kernel<float><<<static_cast<unsigned>(grid), 256, smem, s>>>(fp);
    } else {
        if ((st = set_smem(reinterpret_cast<const void *>(conv_fwd_kernel<__nv_bfloat16>), smem)) != ENGRAM_OK)
            return st;
        conv_fwd_kernel<__nv_bfloat16><<<static_cast<unsigned>(grid), 256, smem, s>>>(fp);
    }
    return check_launch(fn);
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
    prm.partial = dw_partial;
    if ((st = sc_dispatch<kScBwdDot>(fn, dtype, prm, s)) != ENGRAM_OK) return st;
    conv_dot_total_kernel<<<static_cast<unsigned>(std::min<int64_t>((T + 255) / 256, 4096)), 256, 0, s>>>(
        token_dot, T, prm.nb);
    if ((st = check_launch(fn)) != ENGRAM_OK) return st;
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
