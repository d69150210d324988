// The multi-branch gate of the TileKernels release (NEXT-1 of the hot path).
//
// TileLang tutorial, ch. 34 "TileKernels: Engram and mHC":
//   sec. 2.1  hidden_states x [T, hc, d] and kv [T, hc+1, d] (rows 0..hc-1 the branch keys,
//             row hc the value shared by the branches); per branch h
//             alpha = sigmoid(sign(z) * sqrt(max(|z|, clamp))), z = dot * rstd_x * rstd_k / sqrt(d),
//             dot = sum_i x_i (w_h (*) w_e)_i k_i, out = x + alpha * v;
//   sec. 3.2  the forward kernel (the saved dot, alpha, rstd_x, rstd_k; in-place writing excludes
//             saving for the backward);
//   sec. 4.2  the backward: dL/dalpha = sum_i dout_i v_i; zero gradient where |z| < clamp;
//             grad_x = dout + c (k w - x dot rstd_x^2 / d), grad_k = c (x w - k dot rstd_k^2 / d),
//             and the per-block partials of dL/dw_fused = c x k.
// The shared value's gradient is dv = sum_h alpha_h dout_h.
//
// Design: one stage holds a whole token -- x [hc, d] and kv [hc+1, d] (plus dout [hc, d] in the
// backward), two or three 1-D bulk async copies -- so the shared value crosses HBM once per token
// and its gradient sums the branches inside one thread: consumer thread c owns the 16-byte
// vectors jj = c, c + 32*NCW, ... of every branch row.  The weight-gradient partials are laid out
// [P, hc * d], so the plain weight fold and the ordered reduction serve this variant unchanged.
#include <algorithm>
#include <atomic>

#include "gate_pipeline.cuh"

namespace engram {

// Vectors per branch row a thread may own: HC * kVpb <= 4 keeps the fp32 weights and gradient
// accumulators in registers.
template <int HC>
struct HcShape {
    static constexpr int kVpb = 4 / HC;
};

// Token layouts: token t's HC rows of x (and out) start at t * x_stride bytes; its kv block at
// t * kv_stride, with its HC key rows at k_off and its value row at v_off within it; its statistics
// at t * st_stride.  The natural [T, HC, d] / [T, HC + 1, d] / [T, HC] layouts are x_stride =
// HC rows, kv_stride = HC + 1 rows, k_off = 0, v_off = HC rows, st_stride = HC; one branch of a
// wider tensor is a view with the same strides and offset bases.
struct GateHcFwdParams {
    const uint8_t *x, *kv;
    const float *w;  // [hc, d]
    uint8_t *out;
    float *gate, *rstd_x, *rstd_k, *dot;  // [T, hc]
    uint32_t *status;
    int64_t T;
    int64_t x_stride, kv_stride;
    uint32_t k_off, v_off;
    int32_t st_stride;
    int32_t d;
    uint32_t row_bytes;
    int32_t stages;
    float eps, clamp, scale;
};

// The same layouts as the forward (dout and dx like x, dkv like kv); the weight-gradient partial
// rows are part_stride floats apart.  write_dv = 0 leaves the value row's gradient to
// hc_dv_kernel (a branch view sees one term of its sum).
struct GateHcBwdParams {
    const uint8_t *g, *x, *kv;
    const float *w, *gate, *rstd_x, *rstd_k, *dot;
    uint8_t *dx, *dkv;
    float *dw_partial;  // [P, hc * d]
    uint32_t *status;
    int64_t T;
    int64_t x_stride, kv_stride, part_stride;
    uint32_t k_off, v_off;
    int32_t st_stride;
    int32_t write_dv;
    int64_t chunk;
    int32_t P;
    int32_t d;
    uint32_t row_bytes;
    int32_t stages;
    float clamp, scale;
};

inline int hc_smem_bytes(int stages, int stage_bytes, int ncw, int hc) {
    return stages * stage_bytes + 2 * stages * 8 + 2 * ncw * 4 * hc * 4;
}

__device__ __forceinline__ float hc_activation(float z, float clamp) {
    const float r = sqrtf(fmaxf(fabsf(z), clamp));
    return 1.0f / (1.0f + expf(-copysignf(r, z)));
}

// Both kernels below have no separate producer warp: a 17-warp CTA would put five warps on one
// SM sub-partition and cap a thread at ~100 registers, too few for the per-branch weights and
// gradient accumulators.  Thread 0 issues a token's bulk copies instead, refilling a stage as soon
// as a CTA barrier shows every thread is done with it.

// Issue the copies of one token into a stage and arm its barrier (thread 0 only).
__device__ __forceinline__ void hc_issue(uint8_t *dst, uint64_t *bar, uint32_t bytes, uint64_t pol,
                                         const uint8_t *a, uint32_t na, const uint8_t *b, uint32_t nb,
                                         const uint8_t *c, uint32_t nc, const uint8_t *e = nullptr,
                                         uint32_t ne = 0) {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load(dst, a, na, bar, pol);
    bulk_load(dst + na, b, nb, bar, pol);
    if (c) bulk_load(dst + na + nb, c, nc, bar, pol);
    if (e) bulk_load(dst + na + nb + nc, e, ne, bar, pol);
}

// A token's key rows and value row into the stage at dst (after `before` bytes already issued):
// one copy when they are adjacent, else two.
struct HcKv {
    const uint8_t *k, *v;
    bool adjacent;
};
__device__ __forceinline__ HcKv hc_kv(const uint8_t *kv, int64_t t, int64_t kv_stride, uint32_t k_off,
                                      uint32_t v_off, uint32_t hc_rows) {
    const uint8_t *blk = kv + t * kv_stride;
    return {blk + k_off, blk + v_off, v_off == k_off + hc_rows};
}

// Forward: G groups of NCW warps share one CTA and a ring of S token stages; group g works on
// the CTA's tokens g, g + G, ...  While one group reduces and writes a token, the other's data is
// landing and being read, so the CTA's one-token-at-a-time latency is hidden inside the SM.
// Thread index gc within a group owns vectors jj = gc, gc + 32*NCW, ... (VPB of them) of every
// branch row.  Groups synchronise on their own named barriers (ids 1..G).
//
// SPLIT = 2 or 4 (rows too large for a whole token in one CTA's shared memory): a cluster of SPLIT
// CTAs shares each token, CTA `rank` holding bytes [rank * rb / SPLIT, (rank + 1) * rb / SPLIT) of
// every row.  Each group sums its part of the token's 3 HC sums, sends the totals to the same group
// of every other CTA (4-byte stores into their shared memory that complete on their mbarriers, one
// slot per sender and token parity), and adds all parts in rank order; every CTA of the cluster then
// holds the same statistics.  With SPLIT = 4 two CTAs share an SM (MINB), so one's wait for the
// others' parts overlaps the other's work.
template <typename T, int HC, int NCW, int G, int VPB, bool STRIDED, int SPLIT, int MINB = (SPLIT >= 4 ? 2 : 1)>
__global__ void __launch_bounds__(G * NCW * 32, MINB) gate_hc_fwd_kernel(const __grid_constant__ GateHcFwdParams p) {
    static_assert(SPLIT == 1 || ((SPLIT == 2 || SPLIT == 4) && !STRIDED), "the row split takes the natural layouts");
    using V = Vec<T>;
    constexpr int EV = V::N;
    constexpr int NC = NCW * 32;
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rb = p.row_bytes;
    const uint32_t hb = rb / SPLIT;  // bytes of each row this CTA holds
    const uint32_t rank = SPLIT > 1 ? cluster_ctarank() : 0u;
    const uint32_t coff = rank * hb;
    const int wcol = static_cast<int>(rank) * (p.d / SPLIT);
    // the token layout: the natural one at compile time, or the view's strides (STRIDED)
    const int64_t x_stride = STRIDED ? p.x_stride : static_cast<int64_t>(HC) * rb;
    const int64_t kv_stride = STRIDED ? p.kv_stride : static_cast<int64_t>(HC + 1) * rb;
    const uint32_t k_off = STRIDED ? p.k_off : 0u, v_off = STRIDED ? p.v_off : HC * rb;
    const int st_stride = STRIDED ? p.st_stride : HC;
    const uint32_t stage = (2 * HC + 1) * hb;  // x [HC rows] then kv [HC + 1 rows]
    const int S = p.stages;
    const int nvec = static_cast<int>(hb / 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * stage);
    uint32_t *issued_cnt = reinterpret_cast<uint32_t *>(full + S);  // per stage, for the final drain
    float *red = reinterpret_cast<float *>(full + 2 * S);           // [G][2][NCW][4 * HC]
    float *xbuf = red + G * 2 * NCW * 4 * HC;             // [G][2][SPLIT][4 * HC] the other parts' totals
    uint64_t *xbar = reinterpret_cast<uint64_t *>(xbuf + G * 2 * SPLIT * 4 * HC);  // [G][2]

    const int group = threadIdx.x / NC;
    const int gc = threadIdx.x - group * NC;
    const int gwarp = gc >> 5;
    const int lane = gc & 31;
    const int64_t first = SPLIT > 1 ? cluster_index() : blockIdx.x;
    const int64_t stride = SPLIT > 1 ? cluster_count() : gridDim.x;
    const int64_t n_my = first < p.T ? (p.T - 1 - first) / stride + 1 : 0;
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int64_t it) {
        const int64_t tok = first + it * stride;
        const int st = static_cast<int>(it % S);
        issued_cnt[st] += 1;
        const HcKv kv = hc_kv(p.kv, tok, kv_stride, k_off, v_off, HC * rb);
        if (SPLIT > 1) {  // this CTA's half of each of the token's 2 HC + 1 rows
            uint8_t *dst = smem + static_cast<size_t>(st) * stage;
            mbar_arrive_expect_tx(&full[st], stage);
            for (int r = 0; r < HC; ++r)
                bulk_load(dst + r * hb, p.x + tok * x_stride + r * rb + coff, hb, &full[st], pol);
            for (int r = 0; r < HC; ++r)
                bulk_load(dst + (HC + r) * hb, kv.k + r * rb + coff, hb, &full[st], pol);
            bulk_load(dst + 2 * HC * hb, kv.v + coff, hb, &full[st], pol);
        } else if (!STRIDED || kv.adjacent) {
            hc_issue(smem + static_cast<size_t>(st) * stage, &full[st], stage, pol, p.x + tok * x_stride, HC * rb,
                     kv.k, (HC + 1) * rb, nullptr, 0);
        } else {
            hc_issue(smem + static_cast<size_t>(st) * stage, &full[st], stage, pol, p.x + tok * x_stride, HC * rb,
                     kv.k, HC * rb, kv.v, rb);
        }
    };
    if (threadIdx.x == 0) {
        for (int q = 0; q < S; ++q) {
            mbar_init(&full[q], 1);
            issued_cnt[q] = 0;
        }
        if (SPLIT > 1)
            for (int q = 0; q < 2 * G; ++q) mbar_init(&xbar[q], 1);
        mbar_init_fence();
        for (int64_t q = 0; q < S && q < n_my; ++q) issue(q);
    }

    float w[HC][VPB][EV];
#pragma unroll
    for (int h = 0; h < HC; ++h)
#pragma unroll
        for (int m = 0; m < VPB; ++m) {
            const int jj = gc + m * NC;
#pragma unroll
            for (int e = 0; e < EV; ++e) w[h][m][e] = 0.f;
            if (jj < nvec) {
#pragma unroll
                for (int e = 0; e < EV; e += 4) {
                    const float4 q = __ldg(reinterpret_cast<const float4 *>(p.w + static_cast<size_t>(h) * p.d + wcol +
                                                                         jj * EV + e));
                    w[h][m][e] = q.x;
                    w[h][m][e + 1] = q.y;
                    w[h][m][e + 2] = q.z;
                    w[h][m][e + 3] = q.w;
                }
            }
        }
    const float inv_d = 1.0f / static_cast<float>(p.d);
    if (SPLIT > 1)
        cluster_barrier();  // both CTAs' barriers initialised before any store into the other's memory
    else
        __syncthreads();  // barriers initialised

    float *gred = red + static_cast<size_t>(group) * 2 * NCW * 4 * HC;
    int64_t li = 0;  // this group's iteration count
    for (int64_t it = group; it < n_my; it += G, ++li) {
        const int s = static_cast<int>(it % S);
        const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1));
        const uint8_t *st = smem + static_cast<size_t>(s) * stage;
        const uint8_t *kst = st + HC * hb;  // stage rows are hb apart

        float acc[HC][3];
#pragma unroll
        for (int h = 0; h < HC; ++h) acc[h][0] = acc[h][1] = acc[h][2] = 0.f;
        if (ok) {
#pragma unroll
            for (int h = 0; h < HC; ++h)
#pragma unroll
                for (int m = 0; m < VPB; ++m) {
                    const int jj = gc + m * NC;
                    if (jj < nvec) {
                        float xv[EV], kx[EV];
                        V::unpack(*reinterpret_cast<const uint4 *>(st + h * hb + jj * 16), xv);
                        V::unpack(*reinterpret_cast<const uint4 *>(kst + h * hb + jj * 16), kx);
#pragma unroll
                        for (int e = 0; e < EV; ++e) {
                            acc[h][0] = fmaf(xv[e], xv[e], acc[h][0]);
                            acc[h][1] = fmaf(kx[e], kx[e], acc[h][1]);
                            acc[h][2] = fmaf(xv[e] * w[h][m][e], kx[e], acc[h][2]);
                        }
                    }
                }
        }
        float *rbuf = gred + (li & 1) * NCW * 4 * HC;
#pragma unroll
        for (int h = 0; h < HC; ++h)
#pragma unroll
            for (int q = 0; q < 3; ++q) {
                const float v = warp_sum(acc[h][q]);
                if (lane == 0) rbuf[(gwarp * HC + h) * 4 + q] = v;
            }
        if (named_sync_or(1 + group, NC, !ok)) {
            if (gc == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
            break;
        }
        // Cross-warp totals: lane l of every warp sums quantity l (l < 4 HC, slot 3 of each branch
        // unused) over the group's warps in a fixed order, then the totals are broadcast by shuffles.
        float tot = 0.f;
        if (lane < 4 * HC) {
#pragma unroll
            for (int q = 0; q < NCW; ++q) tot += rbuf[q * HC * 4 + lane];
        }
        bool xfail = false;
        if (SPLIT > 1) {  // this part's totals to the other CTAs, then the parts' sum in rank order
            float *xs = xbuf + (group * 2 + (li & 1)) * SPLIT * 4 * HC;
            uint64_t *xb = xbar + group * 2 + (li & 1);
            if (gc == 0) mbar_arrive_expect_tx(xb, (SPLIT - 1) * 4 * HC * 4);
            if (gwarp == 0 && lane < 4 * HC)
                for (uint32_t q = 1; q < SPLIT; ++q) {
                    const uint32_t peer = (rank + q) % SPLIT;
                    cluster_store_tx(cluster_map(smem_addr(xs + rank * 4 * HC + lane), peer), tot,
                                     cluster_map(smem_addr(xb), peer));
                }
            xfail = !mbar_wait(xb, static_cast<uint32_t>((li >> 1) & 1));
            if (lane < 4 * HC) {
                float sum = 0.f;
#pragma unroll
                for (int r = 0; r < SPLIT; ++r) sum += r == static_cast<int>(rank) ? tot : xs[r * 4 * HC + lane];
                tot = sum;
            }
        }
        float gate[HC], rx[HC], rk[HC], dt[HC];
#pragma unroll
        for (int h = 0; h < HC; ++h) {
            const float a = __shfl_sync(0xffffffffu, tot, h * 4 + 0);
            const float b = __shfl_sync(0xffffffffu, tot, h * 4 + 1);
            const float dd = __shfl_sync(0xffffffffu, tot, h * 4 + 2);
            rx[h] = 1.0f / sqrtf(a * inv_d + p.eps);
            rk[h] = 1.0f / sqrtf(b * inv_d + p.eps);
            dt[h] = dd;
            gate[h] = hc_activation(dd * rx[h] * rk[h] * p.scale, p.clamp);
        }

        // out = x + gate * v (the value row is kv row HC)
        const int64_t tok = first + it * stride;
        uint8_t *orow = p.out + tok * x_stride + coff;
#pragma unroll
        for (int m = 0; m < VPB; ++m) {
            const int jj = gc + m * NC;
            if (jj < nvec) {
                float vv[EV];
                V::unpack(*reinterpret_cast<const uint4 *>(kst + HC * hb + jj * 16), vv);
#pragma unroll
                for (int h = 0; h < HC; ++h) {
                    float xv[EV];
                    V::unpack(*reinterpret_cast<const uint4 *>(st + h * hb + jj * 16), xv);
#pragma unroll
                    for (int e = 0; e < EV; ++e) xv[e] = fmaf(gate[h], vv[e], xv[e]);
                    st_global_v4(orow + h * rb + jj * 16, V::pack(xv));
                }
            }
        }
        if (gc < HC && rank == 0) {
            const size_t o = static_cast<size_t>(tok) * st_stride + gc;
            if (p.gate) p.gate[o] = gate[gc];
            if (p.rstd_x) p.rstd_x[o] = rx[gc];
            if (p.rstd_k) p.rstd_k[o] = rk[gc];
            if (p.dot) p.dot[o] = dt[gc];
        }
        // the whole group is done with stage s (refill it) and, split, agrees on whether the other half came
        if (SPLIT > 1) {
            if (named_sync_or(1 + group, NC, xfail)) {
                if (gc == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                break;
            }
        } else {
            named_sync(1 + group, NC);
        }
        if (gc == 0 && it + S < n_my) issue(it + S);
    }
    // Never leave while a copy into this CTA's shared memory may be in flight: wait for the last
    // copy issued into every stage (a completed phase returns at once).
    __syncthreads();
    if (threadIdx.x == 0)
        for (int q = 0; q < S; ++q)
            if (issued_cnt[q] > 0 && !mbar_wait(&full[q], (issued_cnt[q] - 1) & 1u))
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
    if (SPLIT > 1) cluster_barrier();  // no CTA leaves while the other may still store into it
}

// SPLIT = 2 or 4: a cluster of SPLIT CTAs shares each token as in the forward; the parts' dgate sums
// are exchanged the same way.  dv, dx, dk and the weight-gradient partials are per column, so each
// CTA writes its own part of them.
template <typename T, int HC, int NCW, bool STRIDED, int SPLIT, int MINB = (SPLIT >= 4 ? 2 : 1)>
__global__ void __launch_bounds__(NCW * 32, MINB) gate_hc_bwd_kernel(const __grid_constant__ GateHcBwdParams p) {
    static_assert(SPLIT == 1 || ((SPLIT == 2 || SPLIT == 4) && !STRIDED), "the row split takes the natural layouts");
    using V = Vec<T>;
    constexpr int EV = V::N;
    constexpr int NC = NCW * 32;
    constexpr int VPB = HcShape<HC>::kVpb;
    extern __shared__ __align__(128) uint8_t smem[];

    const uint32_t rb = p.row_bytes;
    const uint32_t hb = rb / SPLIT;  // bytes of each row this CTA holds
    const uint32_t rank = SPLIT > 1 ? cluster_ctarank() : 0u;
    const uint32_t coff = rank * hb;
    const int wcol = static_cast<int>(rank) * (p.d / SPLIT);
    // the token layout: the natural one at compile time, or the view's strides (STRIDED)
    const int64_t x_stride = STRIDED ? p.x_stride : static_cast<int64_t>(HC) * rb;
    const int64_t kv_stride = STRIDED ? p.kv_stride : static_cast<int64_t>(HC + 1) * rb;
    const int64_t part_stride = STRIDED ? p.part_stride : static_cast<int64_t>(HC) * p.d;
    const uint32_t k_off = STRIDED ? p.k_off : 0u, v_off = STRIDED ? p.v_off : HC * rb;
    const int st_stride = STRIDED ? p.st_stride : HC;
    const bool write_dv = !STRIDED || p.write_dv;
    const uint32_t stage = (3 * HC + 1) * hb;  // dout [HC], x [HC], kv [HC + 1]
    const int S = p.stages;
    const int nvec = static_cast<int>(hb / 16);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * stage);
    float *red = reinterpret_cast<float *>(full + 2 * S);  // [2][NCW][4 * HC]
    float *xbuf = red + 2 * NCW * 4 * HC;                    // [2][SPLIT][4 * HC] the other parts' dgate sums
    uint64_t *xbar = reinterpret_cast<uint64_t *>(xbuf + 2 * SPLIT * 4 * HC);  // [2]

    const int c = threadIdx.x;
    const int warp = c >> 5;
    const int lane = c & 31;
    // The CTA's (cluster's) tokens, in order: its partials b, b + G, ... each a chunk of C tokens (only
    // the last partial of the whole pass can be shorter, and it is the last of its CTA).
    const int64_t G = SPLIT > 1 ? cluster_count() : gridDim.x, C = p.chunk;
    const int64_t b0 = SPLIT > 1 ? cluster_index() : blockIdx.x;
    int64_t n_my = 0;
    for (int64_t pp = b0; pp < p.P; pp += G) {
        const int64_t t0 = pp * C;
        n_my += t0 >= p.T ? 0 : (t0 + C < p.T ? C : p.T - t0);
    }
    const uint64_t pol = l2_evict_first_policy();
    auto token_of = [&](int64_t j) { return (b0 + (j / C) * G) * C + j % C; };
    auto issue = [&](int64_t j) {
        const int64_t t = token_of(j);
        const HcKv kv = hc_kv(p.kv, t, kv_stride, k_off, v_off, HC * rb);
        if (SPLIT > 1) {  // this CTA's half of each of the token's 3 HC + 1 rows
            uint8_t *dst = smem + static_cast<size_t>(j % S) * stage;
            uint64_t *bar = &full[j % S];
            mbar_arrive_expect_tx(bar, stage);
            for (int r = 0; r < HC; ++r) bulk_load(dst + r * hb, p.g + t * x_stride + r * rb + coff, hb, bar, pol);
            for (int r = 0; r < HC; ++r)
                bulk_load(dst + (HC + r) * hb, p.x + t * x_stride + r * rb + coff, hb, bar, pol);
            for (int r = 0; r < HC; ++r) bulk_load(dst + (2 * HC + r) * hb, kv.k + r * rb + coff, hb, bar, pol);
            bulk_load(dst + 3 * HC * hb, kv.v + coff, hb, bar, pol);
        } else if (!STRIDED || kv.adjacent)
            hc_issue(smem + static_cast<size_t>(j % S) * stage, &full[j % S], stage, pol, p.g + t * x_stride,
                     HC * rb, p.x + t * x_stride, HC * rb, kv.k, (HC + 1) * rb);
        else
            hc_issue(smem + static_cast<size_t>(j % S) * stage, &full[j % S], stage, pol, p.g + t * x_stride,
                     HC * rb, p.x + t * x_stride, HC * rb, kv.k, HC * rb, kv.v, rb);
    };
    int64_t issued = 0;
    if (c == 0) {
        for (int q = 0; q < S; ++q) mbar_init(&full[q], 1);
        if (SPLIT > 1) mbar_init(&xbar[0], 1), mbar_init(&xbar[1], 1);
        mbar_init_fence();
        for (; issued < S && issued < n_my; ++issued) issue(issued);
    }

    float w[HC][VPB][EV];
#pragma unroll
    for (int h = 0; h < HC; ++h)
#pragma unroll
        for (int m = 0; m < VPB; ++m) {
            const int jj = c + m * NC;
#pragma unroll
            for (int e = 0; e < EV; ++e) w[h][m][e] = 0.f;
            if (jj < nvec) {
#pragma unroll
                for (int e = 0; e < EV; e += 4) {
                    const float4 q = __ldg(reinterpret_cast<const float4 *>(p.w + static_cast<size_t>(h) * p.d + wcol +
                                                                         jj * EV + e));
                    w[h][m][e] = q.x;
                    w[h][m][e + 1] = q.y;
                    w[h][m][e + 2] = q.z;
                    w[h][m][e + 3] = q.w;
                }
            }
        }
    const float inv_d = 1.0f / static_cast<float>(p.d);
    if (SPLIT > 1)
        cluster_barrier();  // both CTAs' barriers initialised before any store into the other's memory
    else
        __syncthreads();  // barriers initialised

    int64_t it = 0;
    bool failed = false;
    bool xfail = false;  // the last token's exchange gave up (agreed at the next barrier)
    for (int64_t pp = b0; pp < p.P && !failed; pp += G) {
        const int64_t t0 = pp * C;
        const int64_t t1 = t0 + C < p.T ? t0 + C : p.T;
        float acc[HC][VPB][EV];
#pragma unroll
        for (int h = 0; h < HC; ++h)
#pragma unroll
            for (int m = 0; m < VPB; ++m)
#pragma unroll
                for (int e = 0; e < EV; ++e) acc[h][m][e] = 0.f;

        for (int64_t t = t0; t < t1; ++t, ++it) {
            const int s = static_cast<int>(it % S);
            float gt[HC], rx[HC], rk[HC], dt[HC];
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                const size_t o = static_cast<size_t>(t) * st_stride + h;
                gt[h] = __ldg(p.gate + o);
                rx[h] = __ldg(p.rstd_x + o);
                rk[h] = __ldg(p.rstd_k + o);
                dt[h] = __ldg(p.dot + o);
            }
            const bool ok = mbar_wait(&full[s], static_cast<uint32_t>((it / S) & 1));
            const uint8_t *gst = smem + static_cast<size_t>(s) * stage;
            const uint8_t *xst = gst + HC * hb;  // stage rows are hb apart
            const uint8_t *kst = gst + 2 * HC * hb;

            // pass 1: dgate_h partials, and dv = sum_h gate_h dout_h
            float dg[HC];
#pragma unroll
            for (int h = 0; h < HC; ++h) dg[h] = 0.f;
            if (ok) {
#pragma unroll
                for (int m = 0; m < VPB; ++m) {
                    const int jj = c + m * NC;
                    if (jj < nvec) {
                        float vv[EV], dv[EV];
                        V::unpack(*reinterpret_cast<const uint4 *>(kst + HC * hb + jj * 16), vv);
#pragma unroll
                        for (int e = 0; e < EV; ++e) dv[e] = 0.f;
#pragma unroll
                        for (int h = 0; h < HC; ++h) {
                            float gv[EV];
                            V::unpack(*reinterpret_cast<const uint4 *>(gst + h * hb + jj * 16), gv);
#pragma unroll
                            for (int e = 0; e < EV; ++e) {
                                dg[h] = fmaf(gv[e], vv[e], dg[h]);
                                dv[e] = fmaf(gt[h], gv[e], dv[e]);
                            }
                        }
                        if (write_dv) st_global_v4(p.dkv + t * kv_stride + v_off + coff + jj * 16, V::pack(dv));
                    }
                }
            }
            float *rbuf = red + (it & 1) * NCW * 4 * HC;
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                const float v = warp_sum(dg[h]);
                if (lane == 0) rbuf[(warp * HC + h) * 4] = v;
            }
            // Split rows: one barrier per token.  The warps' dgate sums are in, every thread is done
            // with the previous token (so its stage is refilled here), and all agree on a failed
            // wait, this token's stage or the previous token's exchange.  Whole rows keep a second
            // barrier at the token's end and refill there, which measured faster for them.
            if (__syncthreads_or(!ok || xfail)) {
                if (c == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
                break;
            }
            if (SPLIT > 1 && c == 0 && it > 0 && issued < n_my) issue(issued++);
            // cross-warp totals of dgate: lane h sums branch h over the warps, then a broadcast
            float tot = 0.f;
            if (lane < HC) {
#pragma unroll
                for (int q = 0; q < NCW; ++q) tot += rbuf[(q * HC + lane) * 4];
            }
            if (SPLIT > 1) {  // this part's sums to the other CTAs, then the parts' sum in rank order
                float *xs = xbuf + (it & 1) * SPLIT * 4 * HC;
                uint64_t *xb = xbar + (it & 1);
                if (c == 0) mbar_arrive_expect_tx(xb, (SPLIT - 1) * HC * 4);
                if (warp == 0 && lane < HC)
                    for (uint32_t q = 1; q < SPLIT; ++q) {
                        const uint32_t peer = (rank + q) % SPLIT;
                        cluster_store_tx(cluster_map(smem_addr(xs + rank * 4 * HC + lane), peer), tot,
                                         cluster_map(smem_addr(xb), peer));
                    }
                xfail = !mbar_wait(xb, static_cast<uint32_t>((it >> 1) & 1));
                if (lane < HC) {
                    float sum = 0.f;
#pragma unroll
                    for (int r = 0; r < SPLIT; ++r) sum += r == static_cast<int>(rank) ? tot : xs[r * 4 * HC + lane];
                    tot = sum;
                }
            }
            float cc[HC], cx[HC], ck[HC];
#pragma unroll
            for (int h = 0; h < HC; ++h) {
                const float D = __shfl_sync(0xffffffffu, tot, h);
                // dL/d dot through the sigmoid, the signed square root and the scaling; the clamp
                // holds the activation constant where |z| < clamp, so no gradient flows there.
                const float sc = p.scale * rx[h] * rk[h];
                const float z = dt[h] * sc;
                const float a = gt[h];
                cc[h] = fabsf(z) < p.clamp ? 0.f : D * a * (1.0f - a) / (2.0f * sqrtf(fabsf(z))) * sc;
                cx[h] = cc[h] * dt[h] * rx[h] * rx[h] * inv_d;
                ck[h] = cc[h] * dt[h] * rk[h] * rk[h] * inv_d;
            }

            // pass 2: dx = dout + c (w k - dot rstd_x^2 x / d), dk = c (w x - dot rstd_k^2 k / d), dw partials
#pragma unroll
            for (int h = 0; h < HC; ++h)
#pragma unroll
                for (int m = 0; m < VPB; ++m) {
                    const int jj = c + m * NC;
                    if (jj < nvec) {
                        float xv[EV], kx[EV], gv[EV], ox[EV], okk[EV];
                        V::unpack(*reinterpret_cast<const uint4 *>(xst + h * hb + jj * 16), xv);
                        V::unpack(*reinterpret_cast<const uint4 *>(kst + h * hb + jj * 16), kx);
                        V::unpack(*reinterpret_cast<const uint4 *>(gst + h * hb + jj * 16), gv);
#pragma unroll
                        for (int e = 0; e < EV; ++e) {
                            const float cw = cc[h] * w[h][m][e];
                            ox[e] = gv[e] + fmaf(cw, kx[e], -cx[h] * xv[e]);
                            okk[e] = fmaf(cw, xv[e], -ck[h] * kx[e]);
                            acc[h][m][e] = fmaf(cc[h] * xv[e], kx[e], acc[h][m][e]);
                        }
                        st_global_v4(p.dx + t * x_stride + h * rb + coff + jj * 16, V::pack(ox));
                        st_global_v4(p.dkv + t * kv_stride + k_off + h * rb + coff + jj * 16, V::pack(okk));
                    }
                }
            if (SPLIT == 1) {  // every thread is done with stage s: refill it
                __syncthreads();
                if (c == 0 && issued < n_my) issue(issued++);
            }
        }
        if (failed) break;

        float *prow = p.dw_partial + pp * part_stride + wcol;
#pragma unroll
        for (int h = 0; h < HC; ++h)
#pragma unroll
            for (int m = 0; m < VPB; ++m) {
                const int jj = c + m * NC;
                if (jj < nvec) {
#pragma unroll
                    for (int e = 0; e < EV; e += 4)
                        *reinterpret_cast<float4 *>(prow + static_cast<size_t>(h) * p.d + jj * EV + e) =
                            make_float4(acc[h][m][e], acc[h][m][e + 1], acc[h][m][e + 2], acc[h][m][e + 3]);
                }
            }
    }
    // the last token's exchange, agreed here (a failed run has agreed already)
    if (__syncthreads_or(xfail) && !failed && c == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
    if (c == 0)
        for (int64_t q = it; q < issued; ++q)
            if (!mbar_wait(&full[q % S], static_cast<uint32_t>((q / S) & 1)))
                report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
    if (SPLIT > 1) cluster_barrier();  // no CTA leaves while the other may still store into it
}

// dv_t = sum_h gate[t, h] dout_t,h for the per-branch form of the backward: the same fused
// multiply-add chain over the branches in order that gate_hc_bwd_kernel runs, rounded once.
template <typename E>
__global__ void __launch_bounds__(256) hc_dv_kernel(const uint8_t *__restrict__ g, const float *__restrict__ gate,
                                                    uint8_t *__restrict__ dkv, int64_t T, int32_t hc, uint32_t rb) {
    using V = Vec<E>;
    constexpr int EV = V::N;
    const int64_t nvec = rb / 16;
    const int64_t total = T * nvec;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = i / nvec, jj = i - t * nvec;
        float dv[EV];
#pragma unroll
        for (int e = 0; e < EV; ++e) dv[e] = 0.f;
        for (int h = 0; h < hc; ++h) {
            const float a = __ldg(gate + t * hc + h);
            float gv[EV];
            V::unpack(__ldg(reinterpret_cast<const uint4 *>(g + (t * hc + h) * rb) + jj), gv);
#pragma unroll
            for (int e = 0; e < EV; ++e) dv[e] = fmaf(a, gv[e], dv[e]);
        }
        st_global_v4(dkv + (t * (hc + 1) + hc) * rb + jj * 16, V::pack(dv));
    }
}

namespace {

// Smallest NCW in {2, 4, 8, 16} whose threads cover a branch row with at most HcShape<HC>::kVpb
// vectors each; 0 when none does.
template <int HC>
int hc_consumer_warps(int nvec) {
    for (int ncw = 2; ncw <= 16; ncw *= 2)
        if (ncw * 32 * HcShape<HC>::kVpb >= nvec) return ncw;
    return 0;
}

constexpr int kHcDevices = 64;

// Shared memory of a CTA of either kernel: the ring, its mbarriers and cross-warp buffers, and with
// the row split the other parts' totals ([groups][2][split][4 HC] floats) and their mbarriers
// ([groups][2]).
inline int hc_kernel_smem(int stages, int stage_bytes, int ncw, int hc, int groups, int split) {
    return hc_smem_bytes(stages, stage_bytes, ncw, hc) + (split > 1 ? groups * 2 * (split * 4 * hc * 4 + 8) : 0);
}

// A kernel of the row split: launched in clusters of `split` CTAs (no dependent-launch attribute, like
// the other multi-branch launches).
template <typename Kern, typename Prm>
cudaError_t hc_cluster_launch(Kern kern, int split, int64_t grid, int threads, int smem, cudaStream_t stream,
                              const Prm &q) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, q);
}

// Forward launch: two groups of NCW warps, VPB = 2 * HcShape<HC>::kVpb vectors per branch row
// (the forward keeps no gradient accumulators, so it can afford twice the weights per thread).
// With the row split the persistent grid is as many clusters as are resident at once.
template <typename T, int HC, int NCW, bool STRIDED, int SPLIT>
engram_status launch_hc_fwd(const GateHcFwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    constexpr int G = 2;
    constexpr int NCWG = NCW / 2 > 0 ? NCW / 2 : 1;
    const auto kern = gate_hc_fwd_kernel<T, HC, NCWG, G, 2 * HcShape<HC>::kVpb, STRIDED, SPLIT>;
    // As many stages as fit (2..4): one stage is a whole token (or its part of every row), and with a
    // single CTA per SM the refill of a stage is issued only once the CTA is done with it, so depth
    // must come from stages.  With SPLIT = 4 two CTAs share an SM.
    const int stage = (2 * HC + 1) * static_cast<int>(p.row_bytes / SPLIT);
    const int per_cta = SPLIT >= 4 ? 113 * 1024 : 220 * 1024;
    int S = 4;
    while (S > 2 && hc_kernel_smem(S, stage, NCW, HC, G, SPLIT) > per_cta) --S;
    const int smem = hc_kernel_smem(S, stage, NCW, HC, G, SPLIT);
    if (smem > dev.smem_optin)
        return fail(ENGRAM_ERR_SHAPE, "engram_gate_hc_fwd: a token of %d bytes does not fit twice in shared memory",
                    stage);
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), smem);
    if (st != ENGRAM_OK) return st;
    GateHcFwdParams q = p;
    q.stages = S;
    if (SPLIT == 1) {
        int b = 227 * 1024 / smem;
        b = b < 1 ? 1 : (b > 4 ? 4 : b);
        int64_t grid = static_cast<int64_t>(dev.num_sms) * b;
        if (grid > p.T) grid = p.T;
        grid = cap_grid(grid);
        kern<<<static_cast<unsigned>(grid), G * NCWG * 32, smem, stream>>>(q);
        return check_launch("engram_gate_hc_fwd");
    }
    static std::atomic<int> resident[kHcDevices];  // clusters resident at once, per device
    std::atomic<int> &slot = resident[dev.device % kHcDevices];
    int maxcl = slot.load(std::memory_order_relaxed);
    if (maxcl <= 0) {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = SPLIT;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(SPLIT);
        cfg.blockDim = dim3(G * NCWG * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaOccupancyMaxActiveClusters(&maxcl, kern, &cfg);
        if (e != cudaSuccess || maxcl < 1) {
            cudaGetLastError();
            return fail(ENGRAM_ERR_CUDA, "engram_gate_hc_fwd: no cluster of %d CTAs with %d bytes fits (%s)", SPLIT,
                        smem, cudaGetErrorString(e));
        }
        slot.store(maxcl, std::memory_order_relaxed);
    }
    int64_t ncl = std::min<int64_t>(maxcl, p.T);
    ncl = std::max<int64_t>(1, cap_grid(SPLIT * ncl) / SPLIT);
    const cudaError_t e = hc_cluster_launch(kern, SPLIT, SPLIT * ncl, G * NCWG * 32, smem, stream, q);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_gate_hc_fwd launch: %s", cudaGetErrorString(e));
    return check_launch("engram_gate_hc_fwd");
}

// Backward launch: one CTA (one cluster, split) per partial, as in the single-branch backward.
template <typename T, int HC, int NCW, bool STRIDED, int SPLIT>
engram_status launch_hc_bwd(const GateHcBwdParams &p, const DeviceInfo &dev, cudaStream_t stream) {
    const auto kern = gate_hc_bwd_kernel<T, HC, NCW, STRIDED, SPLIT>;
    const int stage = (3 * HC + 1) * static_cast<int>(p.row_bytes / SPLIT);
    const int per_cta = SPLIT >= 4 ? 113 * 1024 : dev.smem_optin;  // two CTAs per SM with SPLIT = 4
    int S = 3;
    while (S >= 2 && hc_kernel_smem(S, stage, NCW, HC, 1, SPLIT) > per_cta) --S;
    if (S < 2)
        return fail(ENGRAM_ERR_SHAPE, "engram_gate_hc_bwd: a token of %d bytes does not fit twice in shared memory",
                    stage);
    const int smem = hc_kernel_smem(S, stage, NCW, HC, 1, SPLIT);
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), smem);
    if (st != ENGRAM_OK) return st;
    GateHcBwdParams q = p;
    q.stages = S;
    if (SPLIT == 1) {
        const int64_t grid = cap_grid(p.P);
        kern<<<static_cast<unsigned>(grid), NCW * 32, smem, stream>>>(q);
        return check_launch("engram_gate_hc_bwd");
    }
    const int64_t ncl = std::max<int64_t>(1, cap_grid(SPLIT * static_cast<int64_t>(p.P)) / SPLIT);
    const cudaError_t e = hc_cluster_launch(kern, SPLIT, SPLIT * ncl, NCW * 32, smem, stream, q);
    if (e != cudaSuccess) return fail(ENGRAM_ERR_CUDA, "engram_gate_hc_bwd launch: %s", cudaGetErrorString(e));
    return check_launch("engram_gate_hc_bwd");
}

template <typename T, int HC, bool STRIDED = false, int SPLIT = 1>
engram_status dispatch_hc_fwd(const GateHcFwdParams &p, const DeviceInfo &dev, cudaStream_t s) {
    switch (hc_consumer_warps<HC>(static_cast<int>(p.row_bytes / SPLIT / 16))) {
        case 2: return launch_hc_fwd<T, HC, 2, STRIDED, SPLIT>(p, dev, s);
        case 4: return launch_hc_fwd<T, HC, 4, STRIDED, SPLIT>(p, dev, s);
        case 8: return launch_hc_fwd<T, HC, 8, STRIDED, SPLIT>(p, dev, s);
        case 16: return launch_hc_fwd<T, HC, 16, STRIDED, SPLIT>(p, dev, s);
        default: return fail(ENGRAM_ERR_SHAPE, "engram_gate_hc_fwd: d = %d too large for %d branches", p.d, HC);
    }
}

template <typename T, int HC, bool STRIDED = false, int SPLIT = 1>
engram_status dispatch_hc_bwd(const GateHcBwdParams &p, const DeviceInfo &dev, cudaStream_t s) {
    switch (hc_consumer_warps<HC>(static_cast<int>(p.row_bytes / SPLIT / 16))) {
        case 2: return launch_hc_bwd<T, HC, 2, STRIDED, SPLIT>(p, dev, s);
        case 4: return launch_hc_bwd<T, HC, 4, STRIDED, SPLIT>(p, dev, s);
        case 8: return launch_hc_bwd<T, HC, 8, STRIDED, SPLIT>(p, dev, s);
        case 16: return launch_hc_bwd<T, HC, 16, STRIDED, SPLIT>(p, dev, s);
        default: return fail(ENGRAM_ERR_SHAPE, "engram_gate_hc_bwd: d = %d too large for %d branches", p.d, HC);
    }
}

// Whether a token of HC branches (split = 1) or each CTA's part of every row (split = 2, 4) fits the
// fused kernels: the consumer threads cover the row part and two stages fit in shared memory (in half
// of it with split = 4, two CTAs per SM).
template <int HC>
bool hc_fwd_fits(int rb, int smem_optin, int split) {
    if (rb % (16 * split) != 0) return false;
    const int ncw = hc_consumer_warps<HC>(rb / split / 16);
    const int cap = split >= 4 ? 113 * 1024 : smem_optin;
    return ncw > 0 && hc_kernel_smem(2, (2 * HC + 1) * rb / split, ncw, HC, 2, split) <= cap;
}
template <int HC>
bool hc_bwd_fits(int rb, int smem_optin, int split) {
    if (rb % (16 * split) != 0) return false;
    const int ncw = hc_consumer_warps<HC>(rb / split / 16);
    const int cap = split >= 4 ? 113 * 1024 : smem_optin;
    return ncw > 0 && hc_kernel_smem(2, (3 * HC + 1) * rb / split, ncw, HC, 1, split) <= cap;
}
bool hc_fits(int hc, bool fwd, int rb, int smem_optin, int split) {
    switch (hc) {
        case 1: return fwd ? hc_fwd_fits<1>(rb, smem_optin, split) : hc_bwd_fits<1>(rb, smem_optin, split);
        case 2: return fwd ? hc_fwd_fits<2>(rb, smem_optin, split) : hc_bwd_fits<2>(rb, smem_optin, split);
        default: return fwd ? hc_fwd_fits<4>(rb, smem_optin, split) : hc_bwd_fits<4>(rb, smem_optin, split);
    }
}

// 0: each call picks its form; 1: branch by branch; 2 or 4: the row split over clusters of 2 or 4 CTAs
// (where it fits).
std::atomic<int> g_hc_split{0};

enum HcForm { kHcWhole = 0, kHcBranches = 1, kHcSplit2 = 2, kHcSplit4 = 4 };

// The form a call runs in: a whole token per CTA when it fits, else each token shared by a cluster of
// CTAs when the parts fit (the value row and dout then still cross HBM once per token), else branch
// by branch; engram_set_hc_split forces one of them.  Measured at T = 4096, hc = 4, d = 7168 bf16:
// the forward 137 us on clusters of two against 139-141 on four; the backward, which has one group
// of warps per CTA and so waits for the other parts with nothing else to do, 248 us on four (two
// CTAs per SM) against 256 on two.
HcForm hc_form(int hc, bool fwd, int rb, int smem_optin) {
    const int force = g_hc_split.load(std::memory_order_relaxed);
    if (force == 1) return kHcBranches;
    if (force == 2 || force == 4)
        return hc_fits(hc, fwd, rb, smem_optin, force) ? static_cast<HcForm>(force) : kHcBranches;
    if (hc_fits(hc, fwd, rb, smem_optin, 1)) return kHcWhole;
    const int first = fwd ? 2 : 4, second = fwd ? 4 : 2;
    if (hc_fits(hc, fwd, rb, smem_optin, first)) return static_cast<HcForm>(first);
    return hc_fits(hc, fwd, rb, smem_optin, second) ? static_cast<HcForm>(second) : kHcBranches;
}

// Per-branch form, for rows too large for a whole token of hc branches (or when forced): branch h
// is a one-branch problem on strided views of x, kv, out and the statistics, with its row of the
// fused weight; in the backward the value row's gradient sum_h gate_h dout_h is one more kernel.
template <typename T>
engram_status dispatch_hc_fwd_t(int hc, const GateHcFwdParams &p, const DeviceInfo &dev, cudaStream_t s) {
    const HcForm form = hc_form(hc, true, p.row_bytes, dev.smem_optin);
    if (form == kHcWhole) {
        switch (hc) {
            case 1: return dispatch_hc_fwd<T, 1>(p, dev, s);
            case 2: return dispatch_hc_fwd<T, 2>(p, dev, s);
            default: return dispatch_hc_fwd<T, 4>(p, dev, s);
        }
    }
    if (form == kHcSplit2 || form == kHcSplit4) {
        const bool four = form == kHcSplit4;
        switch (hc) {
            case 1: return four ? dispatch_hc_fwd<T, 1, false, 4>(p, dev, s) : dispatch_hc_fwd<T, 1, false, 2>(p, dev, s);
            case 2: return four ? dispatch_hc_fwd<T, 2, false, 4>(p, dev, s) : dispatch_hc_fwd<T, 2, false, 2>(p, dev, s);
            default: return four ? dispatch_hc_fwd<T, 4, false, 4>(p, dev, s) : dispatch_hc_fwd<T, 4, false, 2>(p, dev, s);
        }
    }
    for (int h = 0; h < hc; ++h) {
        GateHcFwdParams q = p;
        q.x += static_cast<size_t>(h) * p.row_bytes;
        q.out += static_cast<size_t>(h) * p.row_bytes;
        q.k_off = p.k_off + h * p.row_bytes;
        q.w += static_cast<size_t>(h) * p.d;
        if (q.gate) q.gate += h;
        if (q.rstd_x) q.rstd_x += h;
        if (q.rstd_k) q.rstd_k += h;
        if (q.dot) q.dot += h;
        engram_status st = dispatch_hc_fwd<T, 1, true>(q, dev, s);
        if (st != ENGRAM_OK) return st;
    }
    return ENGRAM_OK;
}

template <typename T>
engram_status dispatch_hc_bwd_t(int hc, const GateHcBwdParams &p, const DeviceInfo &dev, cudaStream_t s) {
    const HcForm form = hc_form(hc, false, p.row_bytes, dev.smem_optin);
    if (form == kHcWhole) {
        switch (hc) {
            case 1: return dispatch_hc_bwd<T, 1>(p, dev, s);
            case 2: return dispatch_hc_bwd<T, 2>(p, dev, s);
            default: return dispatch_hc_bwd<T, 4>(p, dev, s);
        }
    }
    if (form == kHcSplit2 || form == kHcSplit4) {
        const bool four = form == kHcSplit4;
        switch (hc) {
            case 1: return four ? dispatch_hc_bwd<T, 1, false, 4>(p, dev, s) : dispatch_hc_bwd<T, 1, false, 2>(p, dev, s);
            case 2: return four ? dispatch_hc_bwd<T, 2, false, 4>(p, dev, s) : dispatch_hc_bwd<T, 2, false, 2>(p, dev, s);
            default: return four ? dispatch_hc_bwd<T, 4, false, 4>(p, dev, s) : dispatch_hc_bwd<T, 4, false, 2>(p, dev, s);
        }
    }
    // The value row's gradient reads dout; the branch kernels read the value row of kv.  So with
    // dx written over dout it runs first, and otherwise last (which keeps dkv written over kv
    // correct); the host refuses the two together in this form.
    const int64_t work = p.T * (p.row_bytes / 16);
    const int64_t grid = cap_grid(std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, 8LL * dev.num_sms)));
    const bool dx_on_dout = p.dx == p.g;
    if (dx_on_dout) {
        hc_dv_kernel<T><<<static_cast<unsigned>(grid), 256, 0, s>>>(p.g, p.gate, p.dkv, p.T, hc, p.row_bytes);
        engram_status st = check_launch("engram_gate_hc_bwd");
        if (st != ENGRAM_OK) return st;
    }
    for (int h = 0; h < hc; ++h) {
        GateHcBwdParams q = p;
        q.g += static_cast<size_t>(h) * p.row_bytes;
        q.x += static_cast<size_t>(h) * p.row_bytes;
        q.dx += static_cast<size_t>(h) * p.row_bytes;
        q.k_off = p.k_off + h * p.row_bytes;
        q.w += static_cast<size_t>(h) * p.d;
        q.gate += h;
        q.rstd_x += h;
        q.rstd_k += h;
        q.dot += h;
        q.dw_partial += static_cast<size_t>(h) * p.d;
        q.write_dv = 0;
        engram_status st = dispatch_hc_bwd<T, 1, true>(q, dev, s);
        if (st != ENGRAM_OK) return st;
    }
    if (dx_on_dout) return ENGRAM_OK;
    hc_dv_kernel<T><<<static_cast<unsigned>(grid), 256, 0, s>>>(p.g, p.gate, p.dkv, p.T, hc, p.row_bytes);
    return check_launch("engram_gate_hc_bwd");
}

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

engram_status hc_common_checks(const char *fn, engram_dtype dtype, int64_t T, int32_t hc, int32_t d, int *es,
                               int64_t *row_bytes) {
    *es = dtype_size(dtype);
    if (*es == 0) return fail(ENGRAM_ERR_DTYPE, "%s: dtype %d", fn, (int)dtype);
    if (hc != 1 && hc != 2 && hc != 4) return fail(ENGRAM_ERR_SHAPE, "%s: hc = %d (1, 2 or 4)", fn, hc);
    if (T < 0 || d <= 0) return fail(ENGRAM_ERR_SHAPE, "%s: T = %lld, d = %d", fn, (long long)T, d);
    *row_bytes = static_cast<int64_t>(d) * *es;
    if (*row_bytes % 16 != 0) return fail(ENGRAM_ERR_ALIGN, "%s: row of %lld bytes", fn, (long long)*row_bytes);
    if (*row_bytes > ENGRAM_MAX_ROW_BYTES)
        return fail(ENGRAM_ERR_SHAPE, "%s: row of %lld bytes exceeds %d", fn, (long long)*row_bytes,
                    ENGRAM_MAX_ROW_BYTES);
    return ENGRAM_OK;
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" engram_status engram_gate_hc_fwd(const void *x, const void *kv, engram_dtype dtype, const float *w_fused,
                                            int64_t T, int32_t hc, int32_t d, float eps, float clamp_value,
                                            void *out, float *gate, float *rstd_x, float *rstd_k, float *dot,
                                            engram_stream_t stream) {
    const char *fn = "engram_gate_hc_fwd";
    if (!w_fused || (T > 0 && (!x || !kv || !out))) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    int es;
    int64_t row_bytes;
    engram_status st = hc_common_checks(fn, dtype, T, hc, d, &es, &row_bytes);
    if (st != ENGRAM_OK) return st;
    if (out == x && (gate || rstd_x || rstd_k || dot))
        return fail(ENGRAM_ERR_SHAPE, "%s: in-place output overwrites x, which a backward reads; save no statistic", fn);
    if (!(clamp_value >= 0.0f)) return fail(ENGRAM_ERR_SHAPE, "%s: clamp_value %g", fn, clamp_value);
    const void *al[] = {x, kv, w_fused, out};
    for (const void *q : al)
        if (!aligned16(q)) return fail(ENGRAM_ERR_ALIGN, "%s: tensor not 16-byte aligned", fn);
    DeviceInfo dev;
    if ((st = current_device(&dev)) != ENGRAM_OK) return st;
    const void *dp[] = {x, kv, w_fused, out, gate, rstd_x, rstd_k, dot};
    for (const void *q : dp)
        if ((st = check_device_ptr(q, dev.device, fn)) != ENGRAM_OK) return st;
    if (T == 0) return ENGRAM_OK;
    GateHcFwdParams p{};
    p.x = static_cast<const uint8_t *>(x);
    p.kv = static_cast<const uint8_t *>(kv);
    p.w = w_fused;
    p.out = static_cast<uint8_t *>(out);
    p.gate = gate;
    p.rstd_x = rstd_x;
    p.rstd_k = rstd_k;
    p.dot = dot;
    p.status = dev.status_word;
    p.T = T;
    p.x_stride = hc * row_bytes;
    p.kv_stride = (hc + 1) * row_bytes;
    p.k_off = 0;
    p.v_off = static_cast<uint32_t>(hc * row_bytes);
    p.st_stride = hc;
    p.d = d;
    p.row_bytes = static_cast<uint32_t>(row_bytes);
    p.eps = eps;
    p.clamp = clamp_value;
    p.scale = 1.0f / sqrtf(static_cast<float>(d));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dtype == ENGRAM_F32 ? dispatch_hc_fwd_t<float>(hc, p, dev, s) : dispatch_hc_fwd_t<__nv_bfloat16>(hc, p, dev, s);
}

extern "C" engram_status engram_gate_hc_bwd(const void *dout, const void *x, const void *kv, engram_dtype dtype,
                                            const float *w_fused, const float *gate, const float *rstd_x,
                                            const float *rstd_k, const float *dot, int64_t T, int32_t hc, int32_t d,
                                            float clamp_value, void *dx, void *dkv, float *dw_partial, int32_t P,
                                            engram_stream_t stream) {
    const char *fn = "engram_gate_hc_bwd";
    if (!w_fused || !dw_partial ||
        (T > 0 && (!dout || !x || !kv || !gate || !rstd_x || !rstd_k || !dot || !dx || !dkv)))
        return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    int es;
    int64_t row_bytes;
    engram_status st = hc_common_checks(fn, dtype, T, hc, d, &es, &row_bytes);
    if (st != ENGRAM_OK) return st;
    if (P < 1) return fail(ENGRAM_ERR_SHAPE, "%s: P = %d", fn, P);
    if (!(clamp_value >= 0.0f)) return fail(ENGRAM_ERR_SHAPE, "%s: clamp_value %g", fn, clamp_value);
    const void *al[] = {dout, x, kv, w_fused, dx, dkv, dw_partial};
    for (const void *q : al)
        if (!aligned16(q)) return fail(ENGRAM_ERR_ALIGN, "%s: tensor not 16-byte aligned", fn);
    // Outputs may be written over the input of the same layout (dx over dout or x, dkv over kv):
    // every kernel reads a token's rows before writing that token's.  Any other overlap is refused.
    const int64_t xb = T * hc * row_bytes, kvb = T * (hc + 1) * row_bytes;
    if ((dx != dout && overlaps(dx, xb, dout, xb)) || (dx != x && overlaps(dx, xb, x, xb)) ||
        overlaps(dx, xb, kv, kvb) || (dkv != kv && overlaps(dkv, kvb, kv, kvb)) || overlaps(dkv, kvb, dout, xb) ||
        overlaps(dkv, kvb, x, xb) || overlaps(dx, xb, dkv, kvb))
        return fail(ENGRAM_ERR_SHAPE, "%s: dx or dkv overlaps an input other than in place", fn);
    DeviceInfo dev;
    if ((st = current_device(&dev)) != ENGRAM_OK) return st;
    if (T > 0 && dx == dout && dkv == kv &&
        hc_form(hc, false, static_cast<int>(row_bytes), dev.smem_optin) == kHcBranches)
        return fail(ENGRAM_ERR_SHAPE, "%s: dx over dout together with dkv over kv: rows of %lld bytes at hc = %d run "
                    "branch by branch here, which serves only one of the two", fn, (long long)row_bytes, hc);
    const void *dp[] = {dout, x, kv, w_fused, gate, rstd_x, rstd_k, dot, dx, dkv, dw_partial};
    for (const void *q : dp)
        if ((st = check_device_ptr(q, dev.device, fn)) != ENGRAM_OK) return st;
    GateHcBwdParams p{};
    p.g = static_cast<const uint8_t *>(dout);
    p.x = static_cast<const uint8_t *>(x);
    p.kv = static_cast<const uint8_t *>(kv);
    p.w = w_fused;
    p.gate = gate;
    p.rstd_x = rstd_x;
    p.rstd_k = rstd_k;
    p.dot = dot;
    p.dx = static_cast<uint8_t *>(dx);
    p.dkv = static_cast<uint8_t *>(dkv);
    p.dw_partial = dw_partial;
    p.status = dev.status_word;
    p.T = T;
    p.x_stride = hc * row_bytes;
    p.kv_stride = (hc + 1) * row_bytes;
    p.part_stride = static_cast<int64_t>(hc) * d;
    p.k_off = 0;
    p.v_off = static_cast<uint32_t>(hc * row_bytes);
    p.st_stride = hc;
    p.write_dv = 1;
    p.P = P;
    p.chunk = (T + P - 1) / P;
    p.d = d;
    p.row_bytes = static_cast<uint32_t>(row_bytes);
    p.clamp = clamp_value;
    p.scale = 1.0f / sqrtf(static_cast<float>(d));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dtype == ENGRAM_F32 ? dispatch_hc_bwd_t<float>(hc, p, dev, s) : dispatch_hc_bwd_t<__nv_bfloat16>(hc, p, dev, s);
}

extern "C" int32_t engram_set_hc_split(int32_t on) {
    return g_hc_split.exchange(on == 1 || on == 2 || on == 4 ? on : 0);
}
