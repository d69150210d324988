// The short convolution after the gate (NEXT-2): Y = SiLU(Conv1D(RMSNorm(V~))) + V~, H <- H + Y,
// a depthwise causal convolution of `width` taps (at most 4) with a dilation, per sequence
// (TileLang tutorial, ch. 34 "TileKernels: Engram and mHC", sec. 1.2 item 4: kernel size 4,
// dilation the largest N-gram order).  Tap i multiplies the token (width - 1 - i) * dilation steps
// back, so tap width - 1 is the current token (torch's depthwise conv1d layout with left padding).
//
// GB300 design.  The convolution couples tokens only along time, one channel at a time, and the
// RMSNorm couples channels only within a token, through one scalar.  So:
//   * conv_rstd_kernel: a warp per token computes rstd = 1/sqrt(mean(V~^2) + eps);
//   * conv_fwd_sweep_kernel: CTAs on one 1024-channel block sweep residue classes t = r (mod
//     dilation) of short time chunks.  A producer warp streams each token's V~ and H row segments
//     and rstd into a ring of shared-memory stages with a record of the position; every thread
//     carries its eight channels' last three taps' inputs in registers, so each row is converted
//     once;
//   * conv_bwd_kernel (the backward, one pass): a thread-block cluster of ceil(d / 512) CTAs takes
//     a contiguous range of work items (time chunk, residue class t = r (mod dilation)) in class
//     order, each CTA 512 channels.  Every tap of a class token lies in the same class, so the CTA
//     sweeps its class tokens in time order, across the chunks of its range, a producer warp
//     streaming each token's V~ and dout row segments and rstd into a ring of shared-memory stages;
//     each consumer thread carries its four channels' last three taps' inputs and the du still
//     collecting contributions in registers.  The row dot s = sum_c norm_w du V~ that dV~ needs
//     couples all d channels of a token: each warp sums its part for a few tokens at a time and
//     sends it to every CTA of its cluster through distributed shared memory, then it writes
//     dV~ = dout + rstd norm_w du - rstd^3 V~ s / d and keeps the weight-gradient partials of each
//     (time chunk, residue) work item;
//   * conv_grad_reduce_kernel sums the partials in a fixed order.
// The time chunks depend on T only, the clusters on d only, and every sum has a fixed order, so all
// results are bitwise reproducible on any GPU.
#include <algorithm>
#include <atomic>

#include "colsum.cuh"

namespace engram {

constexpr int kScEV = 4;                // channels per thread
constexpr int kScAges = 4;              // taps: width <= 4

// ---- four channels per lane: 8 bytes of bf16 or 16 bytes of fp32

template <typename E>
struct Ev4;

template <>
struct Ev4<float> {
    static constexpr int kBytes = 16;
    // a plain shared-memory load (the waits before it order it; the compiler may schedule it freely)
    __device__ __forceinline__ static void load_smem(const uint8_t *p, float (&x)[4]) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = u.x, x[1] = u.y, x[2] = u.z, x[3] = u.w;
    }
    __device__ __forceinline__ static void load2(const uint8_t *p, float2 (&x)[2]) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        x[0] = make_float2(u.x, u.y), x[1] = make_float2(u.z, u.w);
    }
    __device__ __forceinline__ static void store2(uint8_t *p, const float2 (&x)[2]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
    }
    __device__ __forceinline__ static void store(uint8_t *p, const float (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    }
};

template <>
struct Ev4<__nv_bfloat16> {
    static constexpr int kBytes = 8;
    __device__ __forceinline__ static void load_smem(const uint8_t *p, float (&x)[4]) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = __uint_as_float(u.x << 16), x[1] = __uint_as_float(u.x & 0xffff0000u);
        x[2] = __uint_as_float(u.y << 16), x[3] = __uint_as_float(u.y & 0xffff0000u);
    }
    __device__ __forceinline__ static void load2(const uint8_t *p, float2 (&x)[2]) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        x[0] = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u));
        x[1] = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    __device__ __forceinline__ static void store2(uint8_t *p, const float2 (&x)[2]) {
        *reinterpret_cast<uint2 *>(p) =
            make_uint2(Vec<__nv_bfloat16>::pack2(x[0].x, x[0].y), Vec<__nv_bfloat16>::pack2(x[1].x, x[1].y));
    }
    __device__ __forceinline__ static void store(uint8_t *p, const float (&x)[4]) {
        *reinterpret_cast<uint2 *>(p) =
            make_uint2(Vec<__nv_bfloat16>::pack2(x[0], x[1]), Vec<__nv_bfloat16>::pack2(x[2], x[3]));
    }
};

// ---- eight channels per lane (the forward): 16 bytes of bf16 or 32 bytes of fp32, as four pairs

template <typename E>
struct Ev8;

template <>
struct Ev8<float> {
    static constexpr int kBytes = 32;
    __device__ __forceinline__ static void load4(const uint8_t *p, float2 (&x)[4]) {
        const float4 u = *reinterpret_cast<const float4 *>(p);
        const float4 v = *reinterpret_cast<const float4 *>(p + 16);
        x[0] = make_float2(u.x, u.y), x[1] = make_float2(u.z, u.w);
        x[2] = make_float2(v.x, v.y), x[3] = make_float2(v.z, v.w);
    }
    __device__ __forceinline__ static void store4(uint8_t *p, const float2 (&x)[4]) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0].x, x[0].y, x[1].x, x[1].y);
        *reinterpret_cast<float4 *>(p + 16) = make_float4(x[2].x, x[2].y, x[3].x, x[3].y);
    }
};

template <>
struct Ev8<__nv_bfloat16> {
    static constexpr int kBytes = 16;
    __device__ __forceinline__ static float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ __forceinline__ static void load4(const uint8_t *p, float2 (&x)[4]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        x[0] = unpack(u.x), x[1] = unpack(u.y), x[2] = unpack(u.z), x[3] = unpack(u.w);
    }
    __device__ __forceinline__ static void store4(uint8_t *p, const float2 (&x)[4]) {
        *reinterpret_cast<uint4 *>(p) =
            make_uint4(Vec<__nv_bfloat16>::pack2(x[0].x, x[0].y), Vec<__nv_bfloat16>::pack2(x[1].x, x[1].y),
                       Vec<__nv_bfloat16>::pack2(x[2].x, x[2].y), Vec<__nv_bfloat16>::pack2(x[3].x, x[3].y));
    }
};

// Two channels at once: sm_100's paired fp32 instructions, each half rounded as the scalar
// operation would be.
__device__ __forceinline__ float2 p2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 p2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 p2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 p2(float v) { return make_float2(v, v); }

// sigmoid(c) = 1 / (1 + e^-c) on a channel pair, with e^-c = 2^(-c log2 e) from the hardware's
// approximate base-2 exponential and the sum's approximate reciprocal (a few ulp each; flushed
// denormals give the limits 0 and 1).  The outputs are rounded far coarser, and the tolerances carry
// the bound.
__device__ __forceinline__ float2 p2sigmoid(float2 c) {
    const float2 z = p2mul(c, p2(-1.44269504088896340736f));
    float e0, e1, r0, r1;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(z.x));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(z.y));
    const float2 den = p2add(make_float2(e0, e1), p2(1.0f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(den.x));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r1) : "f"(den.y));
    return make_float2(r0, r1);
}


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

// ------------------------------------------------------------------------------- backward

constexpr int kBwWarps = 4;                       // consumer warps, four channels per thread
constexpr int kBwCons = kBwWarps * 32;
constexpr int kBwThreads = kBwCons + 32;          // + the copy producer's warp
constexpr int kBwCW = kBwCons * kScEV;            // channels per CTA
constexpr int kBwMaxCluster = 16;                 // CTAs per cluster: d <= 16 * 512
constexpr int kBwLag = kScAges - 1;               // taps behind a token and readers after it
constexpr int kBwBatch = 4;                       // tokens whose row dots are exchanged together
constexpr int kBwPrefetch = 13;                   // stages the copies may run ahead
constexpr int kBwStages = 2 * kBwBatch + kBwLag + kBwPrefetch;  // two batches in flight
static_assert(kBwStages % 4 == 0, "a steady group's four stages are consecutive in the ring");
enum ScKind { kScLead = 0, kScMain = 1, kScTail = 2 };

struct ScBwdParams {
    const uint8_t *v;          // V~ [T, d]
    const uint8_t *dout;       // [T, d]
    const float *norm_w;       // [d]
    const float *conv_w;       // [d, width]
    const float *bias;         // [d] nullable
    const float *rstd;         // [T]
    const int64_t *offs;       // [num_seqs + 1]
    uint8_t *dv;               // [T, d]
    float *partial;            // [nitems, width + 2, d]
    uint32_t *status;
    int64_t T;
    int64_t chunk;             // tokens per time chunk
    int64_t nchunks;           // time chunks
    int64_t nitems;            // chunks x dilation
    int32_t num_seqs;
    int32_t d;
    int32_t width;
    int32_t dil;
};

// Shared memory of one backward CTA: the stage ring; by batch parity the y rows [2][kBwBatch][kBwCons]
// float4 and each thread's row-dot parts [2][kBwCons][kBwBatch]; by batch mod 4 the cluster's warp
// sums of the row dots [4][kBwMaxCluster rank][kBwBatch token][kBwWarps warp]; the stages' position
// records (16 bytes each); the mbarriers (full and empty per stage, 4 exchange); then the copy
// producer's state.
__host__ __device__ inline int sc_bwd_smem(int stages, int stage_bytes) {
    return stages * stage_bytes + 2 * kBwBatch * kBwCons * 16 + 2 * kBwBatch * kBwCons * 4 +
           4 * kBwMaxCluster * kBwBatch * kBwWarps * 4 + stages * 16 + (2 * stages + 4) * 8 + 128;
}

// A stage: the V~ segment of 512 channels, then the dout segment.
template <typename E>
__host__ __device__ constexpr int sc_bwd_stage_bytes() {
    return 2 * kBwCW * static_cast<int>(sizeof(E));
}

template <int N>
struct ScIdx {
    static constexpr int v = N;
};

__device__ __forceinline__ uint32_t sc_cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t sc_cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t sc_cluster_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t sc_num_clusters() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster; release / acquire order shared memory across it.
__device__ __forceinline__ void sc_cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address of this CTA's shared address `a` in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t sc_mapa(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// A 4-byte store into another CTA's shared memory that completes 4 tx bytes on its mbarrier.
__device__ __forceinline__ void sc_st_async(uint32_t raddr, float v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
                 "r"(__float_as_uint(v)), "r"(rbar)
                 : "memory");
}
// Whether the current phases of four consecutive mbarriers, bar0 .. bar0 + 3, with the same parity
// have completed: the four tests are issued back to back, so their latencies overlap.  Like
// mbar_try_wait, each may suspend the thread for a while before it answers.
__device__ __forceinline__ bool sc_try_wait4(uint64_t *bar0, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p0, p1, p2, p3;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p0, [%1], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p1, [%1+8], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p2, [%1+16], %2;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p3, [%1+24], %2;\n\t"
        "and.pred p0, p0, p1;\n\t"
        "and.pred p2, p2, p3;\n\t"
        "and.pred p0, p0, p2;\n\t"
        "selp.u32 %0, 1, 0, p0;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar0)), "r"(parity)
        : "memory");
    return done != 0;
}
// A 4-byte asynchronous global -> shared copy, and an arrival on `bar` once this thread's
// earlier asynchronous copies have landed (the barrier's count includes it).
__device__ __forceinline__ void sc_cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void sc_cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One segment of a work item: the class tokens first, first + dil, ... (n_main of them) of one
// sequence inside the item's chunk, with the n_lead class tokens before them whose V~ the first
// taps read, and (backward) the n_tail class tokens after them whose dc completes the last du.
struct ScSeg {
    int64_t first;
    int n_lead, n_main, n_tail;
};

// The next segment of class r in [x, t_hi), with up to tail_max look-ahead tokens; x and the
// sequence index s advance.  Offsets that are not sorted still give progress and tokens inside [0, T).
template <typename Prm>
__device__ __forceinline__ bool sc_next_seg(const Prm &p, int r, int64_t t_hi, int64_t &x, int &s, ScSeg &g,
                                            int tail_max = kBwLag) {
    const int64_t dil = p.dil;
    while (x < t_hi) {
        while (s + 1 < p.num_seqs && __ldg(p.offs + s + 1) <= x) ++s;
        int64_t s0 = __ldg(p.offs + s), s1 = __ldg(p.offs + s + 1);
        if (s0 > x) s0 = x;
        if (s0 < 0) s0 = 0;
        if (s1 > p.T) s1 = p.T;
        if (s1 <= x) s1 = x + 1;
        const int64_t e = s1 < t_hi ? s1 : t_hi;
        const int64_t first = x + ((r - x % dil) % dil + dil) % dil;
        x = e;
        if (first >= e) continue;
        const int64_t last = first + (e - 1 - first) / dil * dil;
        g.first = first;
        g.n_main = static_cast<int>((last - first) / dil + 1);
        const int64_t lead = (first - s0) / dil, tail = (s1 - 1 - last) / dil;
        g.n_lead = static_cast<int>(lead < kBwLag ? lead : kBwLag);
        g.n_tail = static_cast<int>(tail < tail_max ? tail : tail_max);
        return true;
    }
    return false;
}

// What the producer tells the consumers about each sweep position, beside its stage: the byte
// offset of the token's row in a [T, d] tensor, its rstd (copied asynchronously) and flags.
struct ScMeta {
    int64_t row;
    float rstd;
    uint32_t flags;
};
constexpr uint32_t kFlKind = 3u;          // bits 0-1: kScLead, kScMain or kScTail
constexpr int kFlSlotShift = 2;           // bits 2-3: slot (the position's place in the stream mod 4)
constexpr uint32_t kFlSegStart = 1u << 4;
constexpr uint32_t kFlSegEnd = 1u << 5;
constexpr uint32_t kFlGroup = 1u << 6;    // this and the next three positions form a steady group
                                          // (backward: it starts at a stream position divisible by 4)
constexpr uint32_t kFlItemStart = 1u << 7;
constexpr uint32_t kFlDone = 1u << 8;     // no position: the cluster's items are done
constexpr int kFlItemShift = 12;          // bits 12-31: the work item's stream index, at an item start
constexpr int64_t kBwMaxItems = int64_t(1) << 20;

// The backward's work items in stream order: index k = r * nchunks + c is time chunk c of residue
// class r, so that consecutive indices of one class continue one sweep; its partial row is
// item c * dilation + r.  A cluster takes a contiguous range of indices.
__host__ __device__ inline int64_t sc_bwd_item(int64_t k, int64_t nchunks, int64_t dil) {
    return (k % nchunks) * dil + k / nchunks;
}
__host__ __device__ inline int64_t sc_bwd_range_lo(int64_t cluster, int64_t ncl, int64_t nitems) {
    return cluster * nitems / ncl;
}

// The producer's place in the stream of sweep positions of its cluster's range of work items (in
// shared memory; lane 0 of the producer warp moves it on from one segment to the next).
struct ScBwdProd {
    int64_t kend;      // end of the current class's share of the range (stream index)
    int64_t khi;       // end of the cluster's range
    int64_t t_hi;      // end of the current class's tokens in the range
    int64_t xs;        // where the class's next segment starts looking
    int64_t t;         // token of the next position
    int64_t last_k;    // stream index of the last chunk token issued
    uint32_t issued;   // positions issued so far (the sentinel included)
    uint32_t round;    // times the ring has wrapped
    int32_t st;        // stage of the next position
    int32_t s;         // sequence index of xs
    int32_t r;         // the current class
    int32_t q, n, n_lead, n_main;  // next position of the segment, its positions, lead-in, chunk tokens
    int32_t state;     // 0 positions to issue, 1 only the sentinel, 2 finished
};
// The forward producer's place in the stream of sweep positions of its CTA's work items (in shared
// memory; lane 0 of the producer warp moves it on from one segment to the next).
struct ScProd {
    int64_t item;      // current work item
    int64_t t_hi;      // its chunk's end
    int64_t xs;        // where its next segment starts looking
    int64_t t;         // token of the next position
    int32_t s;         // sequence index of xs
    int32_t q, n, n_lead;  // next position of the segment, its positions, lead-in
    int32_t state;     // 0 positions to issue, 1 only the sentinel, 2 finished
};
static_assert(sizeof(ScProd) <= 128, "the producer state fits its shared-memory slot");
static_assert(sizeof(ScBwdProd) <= 128, "the producer state fits its shared-memory slot");

// The backward in one pass.  A cluster of ceil(d / 512) CTAs takes a contiguous range of work
// items (time chunk, residue class t = r mod dilation) in class order, so that one class's
// consecutive chunks form one sweep; CTA `rank` holds channels [512 rank, 512 rank + 512).
// A producer warp walks the range's segments (a sequence's class tokens in the range) and streams,
// per sweep position (one per lane), the token's V~ and dout row segments (1-D bulk copies) and its
// rstd (a 4-byte asynchronous copy) into a ring of stages, as far ahead as the ring allows, with a
// record of the position (row offset, kind, slot, segment and item boundaries).  Each of the 128
// consumer threads owns four channels and sweeps the positions in order.  With the norm weight
// folded into the taps (w'_a = w_a norm_w, w_a: tap width - 1 - a) and u' = V~ rstd (the last
// three kept by age in registers):
//   conv = bias + sum_a w'_a u'[t - a dil],  dc = dout SiLU'(conv),
//   A_a += dc u'[t - a dil] and db += dc over the item's outputs, and the
//   dn = norm_w du = sum_a w'_a dc[t + a dil] still collecting contributions (three, by age).
// When a token's dn is complete its stage is read back for V~ and dout:
//   y = dout + rstd dn  (kept in shared memory),  and the thread's part of the row dot
//   s = sum_c norm_w du V~ = sum_c dn V~.
// Every four tokens each warp sums its threads' parts of each row dot (one butterfly) and sends the
// sums to every CTA of the cluster (distributed shared memory, completing on their mbarrier); a
// batch later, when all the cluster's warp sums have arrived, every warp adds them in a fixed order
// and writes dv = y - rstd^3 V~ s / d.  At a work item's end its partial rows are norm_w A_a
// (tap width - 1 - a), db, and, for the norm weight, sum_i conv_w[i] A_(width-1-i): over a
// sequence dL/dnorm_w = sum_t du u' = sum_a w_a sum_t dc[t] u'[t - a dil], so no per-token
// accumulator and no norm weight are needed in the sweep.  All waits are bounded.
// The chunks depend on T only and every sum has a fixed order, so results are bitwise reproducible.
template <typename E>
__global__ void __launch_bounds__(kBwThreads, 3) conv_bwd_kernel(const __grid_constant__ ScBwdParams p) {
    using EV = Ev4<E>;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int S = kBwStages;
    constexpr int SB = sc_bwd_stage_bytes<E>();
    constexpr int half = SB / 2;
    uint8_t *ring = smem;
    float4 *ybuf = reinterpret_cast<float4 *>(smem + static_cast<size_t>(S) * SB);
    float *pbuf = reinterpret_cast<float *>(ybuf + 2 * kBwBatch * kBwCons);
    float *box = pbuf + 2 * kBwBatch * kBwCons;
    ScMeta *meta = reinterpret_cast<ScMeta *>(box + 4 * kBwMaxCluster * kBwBatch * kBwWarps);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + S);
    uint64_t *empty = full + S;
    uint64_t *boxbar = empty + S;
    ScBwdProd *prod = reinterpret_cast<ScBwdProd *>(boxbar + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = sc_cluster_rank();
    const uint32_t C = sc_cluster_size();
    const int c0 = static_cast<int>(rank) * kBwCW;
    const int ncols = p.d - c0 < kBwCW ? p.d - c0 : kBwCW;
    const int64_t dil = p.dil;
    bool failed = false;

    // producer lane 0: the tokens of class k / nchunks in the range's chunks from stream index k on
    auto prod_start_class = [&](int64_t k) {
        ScBwdProd &P = *prod;
        const int64_t r = k / p.nchunks;
        P.r = static_cast<int32_t>(r);
        P.kend = P.khi < (r + 1) * p.nchunks ? P.khi : (r + 1) * p.nchunks;
        P.xs = (k - r * p.nchunks) * p.chunk;
        const int64_t e = (P.kend - r * p.nchunks) * p.chunk;
        P.t_hi = e < p.T ? e : p.T;
        P.s = sc_seq_of(p.offs, p.num_seqs, P.xs);
    };
    // producer lane 0: the next segment of the producer's stream (one sequence's class tokens in the
    // current class's chunks, which may span several work items), moving on through the classes
    auto prod_next_seg = [&]() {
        ScBwdProd &P = *prod;
        ScSeg g;
        for (;;) {
            int64_t xs = P.xs;
            int s = P.s;
            const bool found = sc_next_seg(p, P.r, P.t_hi, xs, s, g);
            P.xs = xs;
            P.s = s;
            if (found) {
                P.q = 0;
                P.n = g.n_lead + g.n_main + g.n_tail;
                P.n_lead = g.n_lead;
                P.n_main = g.n_main;
                P.t = g.first - g.n_lead * dil;
                return;
            }
            if (P.kend >= P.khi) {
                P.state = 1;
                return;
            }
            prod_start_class(P.kend);
        }
    };
    // the producer warp: every position of the cluster's items in order, one position per lane as
    // stages free up, then the sentinel.  The state is kept in registers (the copies' asm
    // statements order shared memory, so shared fields would be reloaded around each of them).
    auto produce_all = [&]() {
        ScBwdProd &P = *prod;
        const uint32_t seg = static_cast<uint32_t>(ncols) * sizeof(E);
        const size_t row_bytes = static_cast<size_t>(p.d) * sizeof(E);
        const uint8_t *src_v = p.v + static_cast<size_t>(c0) * sizeof(E);
        const uint8_t *src_g = p.dout + static_cast<size_t>(c0) * sizeof(E);
        const int64_t L = p.chunk;
        const bool small = p.T <= 0x7fffffff;  // chunk of a token by 32-bit division
        auto chunk_of = [&](int64_t tk) {
            return small ? static_cast<int64_t>(static_cast<uint32_t>(tk) / static_cast<uint32_t>(L)) : tk / L;
        };
        int st = P.st, state = P.state;
        uint32_t round = P.round, issued = P.issued;
        int q = P.q, n = P.n, nl = P.n_lead, nm = P.n_main;
        int64_t kcls = static_cast<int64_t>(P.r) * p.nchunks;  // stream index of the class's chunk 0
        int64_t last_k = P.last_k;
        int64_t t = P.t;
        while (state != 2) {
            // the free stages from st on: lane l tests the one of position issued + l
            const int stl = st + lane < S ? st + lane : st + lane - S;
            const uint32_t rl = round + (st + lane < S ? 0u : 1u);
            const bool free_l = lane < S && (rl == 0 || mbar_test_wait(&empty[stl], (rl + 1) & 1u));
            const uint32_t mask = __ballot_sync(0xffffffffu, free_l);
            int cnt = __ffs(~mask) - 1;
            if (cnt < 0) cnt = 32;
            if (cnt == 0) {  // the ring is full: wait (bounded) for its oldest stage
                bool ok = true;
                if (lane == 0) ok = mbar_wait_sleep(&empty[st], (round + 1) & 1u);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                    failed = true;
                    break;
                }
                continue;
            }
            if (state == 1) {  // the sentinel: no copies, both arrivals
                if (lane == 0) {
                    meta[st].row = 0;
                    meta[st].flags = kFlDone;
                    mbar_arrive(&full[st]);
                    mbar_arrive(&full[st]);
                }
                state = 2;
                cnt = 1;
            } else {
                if (cnt > n - q) cnt = n - q;
                if (lane < cnt) {
                    const int ql = q + lane;
                    const int64_t tl = t + lane * dil;
                    const uint32_t kind = ql < nl ? kScLead : (ql < nl + nm ? kScMain : kScTail);
                    // the chunk token's work item: it starts one where the previous chunk token of the
                    // stream lies in another chunk (or, for a segment's first, another item)
                    const int64_t c = chunk_of(tl);
                    const int64_t kl = kcls + c;
                    const bool istart = kind == kScMain && (ql > nl ? tl - c * L < dil : kl != last_k);
                    // slots and steady groups by the position's place in the stream: the ring has a
                    // multiple of 4 stages, so a group's four stages are consecutive in it; a group's
                    // four chunk tokens lie in one item
                    const uint32_t gp = issued + static_cast<uint32_t>(lane);
                    const bool group = (gp & 3u) == 0 && ql >= nl + kBwLag && ql + 4 <= nl + nm && ql + 4 < n &&
                                       tl - c * L + 3 * dil < L;
                    uint32_t fl = kind | ((gp & 3u) << kFlSlotShift);
                    if (ql == 0) fl |= kFlSegStart;
                    if (ql == n - 1) fl |= kFlSegEnd;
                    if (group) fl |= kFlGroup;
                    if (istart) fl |= kFlItemStart | (static_cast<uint32_t>(kl) << kFlItemShift);
                    meta[stl].row = tl * static_cast<int64_t>(row_bytes);
                    meta[stl].flags = fl;
                    uint8_t *dst = ring + static_cast<size_t>(stl) * SB;
                    sc_cp_async4(&meta[stl].rstd, p.rstd + tl);
                    sc_cp_async_arrive(&full[stl]);
                    mbar_arrive_expect_tx(&full[stl], kind == kScLead ? seg : 2 * seg);
                    bulk_load_plain(dst, src_v + static_cast<size_t>(tl) * row_bytes, seg, &full[stl]);
                    if (kind != kScLead)
                        bulk_load(dst + half, src_g + static_cast<size_t>(tl) * row_bytes, seg, &full[stl],
                                  l2_evict_first_policy());
                }
                // the last chunk token issued, for the next segment's first
                const int lm = (q + cnt < nl + nm ? q + cnt : nl + nm) - 1;
                if (lm >= q && lm >= nl) last_k = kcls + chunk_of(t + (lm - q) * dil);
                q += cnt;
                t += cnt * dil;
                if (q == n) {  // the segment ends: the next one (rare) through the shared state
                    __syncwarp();
                    if (lane == 0) prod_next_seg();
                    __syncwarp();
                    state = P.state, q = P.q, n = P.n, nl = P.n_lead, nm = P.n_main;
                    kcls = static_cast<int64_t>(P.r) * p.nchunks;
                    t = P.t;
                }
            }
            issued += cnt;
            st += cnt;
            if (st >= S) st -= S, ++round;
        }
        // after a failure, copies may still be landing: wait for them (bounded) before the CTA leaves
        if (failed && lane == 0)
            for (uint32_t q2 = issued > static_cast<uint32_t>(S) ? issued - S : 0; q2 < issued; ++q2)
                mbar_wait_sleep(&full[q2 % S], (q2 / S) & 1u, kWaitLimitNs / 16);
        __syncwarp();
    };

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);  // the producer's arrival and its rstd copy's
            mbar_init(&empty[i], kBwWarps);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&boxbar[i], 1);
        mbar_init_fence();
    }
    sc_cluster_sync();  // every CTA's barriers exist before any remote arrival
    pdl_wait();
    const int64_t ncl = sc_num_clusters();
    const int64_t klo = sc_bwd_range_lo(sc_cluster_id(), ncl, p.nitems);
    const int64_t khi = sc_bwd_range_lo(sc_cluster_id() + 1, ncl, p.nitems);
    if (warp == kBwWarps) {
        if (lane == 0) {
            ScBwdProd &P = *prod;
            P = ScBwdProd{};
            P.khi = khi;
            P.last_k = -1;
            if (klo >= khi) {
                P.state = 1;
            } else {
                prod_start_class(klo);
                prod_next_seg();
            }
        }
        __syncwarp();
        produce_all();
    } else {

        const bool active = tid * kScEV < ncols;
        const uint8_t *my_ring = ring + tid * EV::kBytes;  // this thread's channels in stage 0
        const int width = p.width, d = p.d;
        const int cth = c0 + tid * kScEV;                  // the thread's first channel
        // the thread's four channels as two pairs: [h] holds channels 2h and 2h + 1; the taps carry
        // the norm weight (w'_a = w_a norm_w, rounded once)
        float2 w[kScAges][2], bias[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v[2][1 + kScAges];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = cth + 2 * h + k;
                const bool ok = active && c < d;
                const float nwc = ok ? __ldg(p.norm_w + c) : 0.f;
                v[k][0] = ok && p.bias ? __ldg(p.bias + c) : 0.f;
#pragma unroll
                for (int a = 0; a < kScAges; ++a)
                    v[k][1 + a] = ok && a < width ? __fmul_rn(__ldg(p.conv_w + static_cast<size_t>(c) * width +
                                                                    (width - 1 - a)),
                                                              nwc)
                                                  : 0.f;
            }
            bias[h] = make_float2(v[0][0], v[1][0]);
#pragma unroll
            for (int a = 0; a < kScAges; ++a) w[a][h] = make_float2(v[0][1 + a], v[1][1 + a]);
        }
        const float inv_d = 1.0f / static_cast<float>(d);

        float2 U[4][2];                 // u' by slot: position q's in slot q & 3
        float2 P1[2], P2[2], P3[2];     // dn collecting contributions, by age 1..3
        float2 A[kScAges][2], db[2];
        bool pend1 = false, pend2 = false, pend3 = false;
        int st = 0;
        uint32_t ph = 0;
        int nfin = 0, nb = 0, prev_n = 0;  // tokens of the open batch, batches posted, tokens of the pending one
        uint32_t bst = 0, pst = 0;         // the stages of the open and the pending batch's tokens, a byte each

        // a wait of the whole warp: every lane takes the same view of a failure
        auto wait_warp = [&](uint64_t *bar, uint32_t parity) {
            if (failed) return;
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(bar, parity))) {
                if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
            }
        };
        // stages st + k0 .. st + k1 - 1 full: every lane tries them all back to back and the warp
        // agrees; only when one is still filling, every lane waits for it (bounded)
        auto wait_stages = [&](int k0, int k1) {
            if (failed) return;
            bool ok = true;
#pragma unroll 4
            for (int k = k0; k < k1; ++k) {
                const bool wrap = st + k >= S;
                ok &= mbar_try_wait(&full[wrap ? st + k - S : st + k], wrap ? ph ^ 1u : ph);
            }
            if (__all_sync(0xffffffffu, ok)) return;
            ok = true;
            for (int k = k0; k < k1; ++k) {
                const bool wrap = st + k >= S;
                ok = ok && mbar_wait_sleep(&full[wrap ? st + k - S : st + k], wrap ? ph ^ 1u : ph);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
            }
        };
        auto advance = [&]() {
            if (++st == S) st = 0, ph ^= 1u;
        };
        auto back = [&](int a) { return st - a < 0 ? st - a + S : st - a; };
        // after a failure a warp arrives on no barrier and sends nothing: no phase can be overrun
        auto release = [&](int stage) {
            __syncwarp();
            mbar_arrive_if(&empty[stage], lane == 0 && !failed);
        };
        // the token at stage sa has its dn: its y and row-dot part, token k of the open batch
        auto complete_at = [&](int sa, int k, const float2 (&dn)[2]) {
            const uint8_t *stg = my_ring + sa * SB;
            float2 x[2], g[2], y[2];
            EV::load2(stg, x);
            EV::load2(stg + half, g);
            const float2 ra = p2(meta[sa].rstd);
#pragma unroll
            for (int h = 0; h < 2; ++h) y[h] = p2fma(ra, dn[h], g[h]);
            // the thread's part of the row dot: (c0 + c2) + (c1 + c3) of the products
            const float2 pp = p2fma(dn[1], x[1], p2mul(dn[0], x[0]));
            const float part = pp.x + pp.y;
            pbuf[((nb & 1) * kBwCons + tid) * kBwBatch + k] = active ? part : 0.f;
            ybuf[((nb & 1) * kBwBatch + k) * kBwCons + tid] = make_float4(y[0].x, y[0].y, y[1].x, y[1].y);
            bst |= static_cast<uint32_t>(sa) << (8 * k);
        };
        // a token `a` positions back has its dn
        auto complete = [&](int a, const float2 (&dn)[2]) {
            complete_at(back(a), nfin, dn);
            ++nfin;
        };
        // batch bf's dv rows once the cluster's row dots have arrived; its stages (a byte each in `stg`)
        // go back to the producer.  Rank k's sum of token j is b_k = (w_0 + w_1) + (w_2 + w_3) over its
        // warps' sums; token j's row dot is the sum of b_0 .. b_(C-1): lane 4k + j takes b_k (plus
        // b_(k+8) for clusters above 8) and a butterfly over k adds them pairwise, so lane j holds
        // ((b_0 + b_1) + (b_2 + b_3)) + ((b_4 + b_5) + (b_6 + b_7)); lane j then forms token j's scale.
        // The tokens' rows are then independent of each other.  FULL: four tokens.
        // batch bf's dv rows once the cluster's row dots have arrived; its stages (a byte each in `stg`)
        // go back to the producer.  Rank k's sum of token j is b_k = (w_0 + w_1) + (w_2 + w_3) over its
        // warps' sums; token j's row dot is the sum of b_0 .. b_(C-1): lane 4k + j takes b_k (plus
        // b_(k+8) for clusters above 8) and a butterfly over k adds them pairwise, so lane j holds
        // ((b_0 + b_1) + (b_2 + b_3)) + ((b_4 + b_5) + (b_6 + b_7)); lane j then forms token j's scale.
        // The tokens' rows are then independent of each other.  FULL: four tokens.
        auto finalize = [&](auto Fc, int bf, int n, uint32_t stg) {
            constexpr bool FULL = decltype(Fc)::v != 0;
            wait_warp(&boxbar[bf & 3], (bf >> 2) & 1);
            const float4 *bx = reinterpret_cast<const float4 *>(box) + (bf & 3) * kBwMaxCluster * kBwBatch;
            static_assert(kBwBatch == 4 && kBwMaxCluster == 16 && kBwWarps == 4,
                          "32 lanes take 8 ranks x 4 tokens, twice; a rank's four warp sums are one float4");
            const int kr = lane >> 2;
            float s = 0.f;
            if (kr < static_cast<int>(C)) {
                const float4 u = bx[lane];
                s = (u.x + u.y) + (u.z + u.w);
            }
            if (kr + 8 < static_cast<int>(C)) {
                const float4 u = bx[lane + 8 * kBwBatch];
                s += (u.x + u.y) + (u.z + u.w);
            }
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            s += __shfl_xor_sync(0xffffffffu, s, 8);
            s += __shfl_xor_sync(0xffffffffu, s, 16);
            const int sj_l = static_cast<int>((stg >> (8 * (lane & 3))) & 0xffu);
            const float r = meta[sj_l].rstd;
            const float kk_l = r * r * r * s * inv_d;
            uint8_t *dv_col = p.dv + static_cast<size_t>(c0) * sizeof(E) + tid * EV::kBytes;
#pragma unroll
            for (int j = 0; j < kBwBatch; ++j) {
                const float kk = __shfl_sync(0xffffffffu, kk_l, j);
                const int sj = static_cast<int>((stg >> (8 * j)) & 0xffu);
                if (FULL || j < n) {
                    float2 x[2];
                    EV::load2(my_ring + sj * SB, x);
                    const float4 y = ybuf[((bf & 1) * kBwBatch + j) * kBwCons + tid];
                    const float2 o[2] = {p2fma(p2(-kk), x[0], make_float2(y.x, y.y)),
                                         p2fma(p2(-kk), x[1], make_float2(y.z, y.w))};
                    if (active) EV::store2(dv_col + meta[sj].row, o);
                }
            }
            __syncwarp();
            mbar_arrive_if(&empty[sj_l], lane < n && !failed);
        };
        auto finalize_any = [&](int bf, int n, uint32_t stg) {
            if (n == kBwBatch) finalize(ScIdx<1>{}, bf, n, stg);
            else finalize(ScIdx<0>{}, bf, n, stg);
        };
        // the open batch is complete: the warp sums its threads' parts of each token in one transposed
        // butterfly (pairing lanes 16, 8, 4, 2, 1 apart; each lane passes on the tokens it does not
        // keep, so that after two steps lanes 8t .. 8t + 7 carry token t) and sends the sums to every
        // CTA of the cluster, itself included, with stores that complete on their exchange barrier,
        // which warp 0 arms; then the previous batch, whose sums have had a batch's time to arrive, is
        // finished.  Nobody waits for the others here.
        const uint32_t box_lo = smem_addr(box), bar_lo = smem_addr(boxbar);
        auto post = [&]() {
            const int b = nb;
            static_assert(kBwBatch == 4, "a thread's four parts are one float4");
            const float4 pp = *reinterpret_cast<const float4 *>(pbuf + ((b & 1) * kBwCons + tid) * kBwBatch);
            const bool hi = (lane & 16) != 0, b3 = (lane & 8) != 0;
            float s0 = hi ? pp.z : pp.x, s1 = hi ? pp.w : pp.y;
            s0 += __shfl_xor_sync(0xffffffffu, hi ? pp.x : pp.z, 16);
            s1 += __shfl_xor_sync(0xffffffffu, hi ? pp.y : pp.w, 16);
            float sum = b3 ? s1 : s0;
            sum += __shfl_xor_sync(0xffffffffu, b3 ? s0 : s1, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 2);
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            // lane 8t + q sends token t's sum to ranks q and q + 8, into slot [rank][t][warp]
            const int tk = lane >> 3;
            if (!failed && tk < nfin) {
                const uint32_t slot =
                    ((static_cast<uint32_t>(b & 3) * kBwMaxCluster + rank) * kBwBatch + tk) * kBwWarps + warp;
                for (int r = lane & 7; r < static_cast<int>(C); r += 8)
                    sc_st_async(sc_mapa(box_lo + slot * 4, r), sum, sc_mapa(bar_lo + (b & 3) * 8, r));
            }
            if (warp == 0 && lane == 0 && !failed)
                mbar_arrive_expect_tx(&boxbar[b & 3], C * kBwWarps * static_cast<uint32_t>(nfin) * 4);
            if (prev_n > 0) finalize_any(b - 1, prev_n, pst);
            prev_n = nfin;
            pst = bst;
            bst = 0;
            nfin = 0;
            ++nb;
        };
        // one sweep position in slot J at stage sp, already waited for.  STEADY: position J of a steady
        // group (stages st0 + J of a group starting at st0 = st), a chunk token with three chunk tokens
        // pending before it, so the one three back (stage sa3) completes as token J of its batch; the
        // group moves st on.  Otherwise `kind` and the pending flags decide, and the step moves st on.
        auto step = [&](auto Jc, auto Sc, uint32_t kind, int sp, int sa3) {
            constexpr int J = decltype(Jc)::v;
            constexpr bool STEADY = decltype(Sc)::v != 0;
            const uint8_t *stg = my_ring + sp * SB;
            const float2 rt = p2(meta[sp].rstd);
            float2 x[2];
            EV::load2(stg, x);
#pragma unroll
            for (int h = 0; h < 2; ++h) U[J][h] = p2mul(x[h], rt);
            if (!STEADY && kind == kScLead) {
                release(sp);
                advance();
                return;
            }
            float2 g[2], dc[2];
            EV::load2(stg + half, g);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float2 c = p2fma(w[3][h], U[(J + 1) & 3][h],
                                       p2fma(w[2][h], U[(J + 2) & 3][h],
                                             p2fma(w[1][h], U[(J + 3) & 3][h], p2fma(w[0][h], U[J][h], bias[h]))));
                const float2 sg = p2sigmoid(c);
                // SiLU'(c) = sg (1 + c (1 - sg))
                dc[h] = p2mul(g[h], p2fma(sg, p2fma(make_float2(-c.x, -c.y), sg, c), sg));
            }
            if (STEADY || kind == kScMain) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    db[h] = p2add(db[h], dc[h]);
                    A[0][h] = p2fma(dc[h], U[J][h], A[0][h]);
                    A[1][h] = p2fma(dc[h], U[(J + 3) & 3][h], A[1][h]);
                    A[2][h] = p2fma(dc[h], U[(J + 2) & 3][h], A[2][h]);
                    A[3][h] = p2fma(dc[h], U[(J + 1) & 3][h], A[3][h]);
                }
            }
            if (STEADY || pend3) {
                float2 dn[2];
#pragma unroll
                for (int h = 0; h < 2; ++h) dn[h] = p2fma(w[3][h], dc[h], P3[h]);
                if (STEADY) complete_at(sa3, J, dn);
                else complete(3, dn);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                P3[h] = p2fma(w[2][h], dc[h], P2[h]);
                P2[h] = p2fma(w[1][h], dc[h], P1[h]);
                P1[h] = p2mul(w[0][h], dc[h]);
            }
            if (!STEADY) {
                pend3 = pend2, pend2 = pend1, pend1 = kind == kScMain;
                if (kind == kScTail) release(sp);
                advance();
            }
        };

        // a work item's weight-gradient partial rows: the taps (by tap index) norm_w A_a, the bias, and
        // the norm weight sum_i conv_w[i] A_(width-1-i) (ascending i); the unfolded weights are read
        // again here, once per item
        auto write_rows = [&](int64_t item, bool zero) {
            if (!active) return;
            float *prow = p.partial + static_cast<size_t>(item) * (width + 2) * d + cth;
            float tap[kScAges][kScEV], dnw[kScEV];
#pragma unroll
            for (int k = 0; k < kScEV; ++k) {
                const int c = cth + k;
                const float nwc = __ldg(p.norm_w + c);
                dnw[k] = 0.f;
#pragma unroll
                for (int a = kScAges - 1; a >= 0; --a) {
                    const float Aa = (k & 1) ? A[a][k >> 1].y : A[a][k >> 1].x;
                    tap[a][k] = __fmul_rn(nwc, Aa);
                    if (a < width)
                        dnw[k] = __fmaf_rn(__ldg(p.conv_w + static_cast<size_t>(c) * width + (width - 1 - a)), Aa,
                                           dnw[k]);
                }
            }
            const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int a = 0; a < kScAges; ++a)
                if (a < width)
                    *reinterpret_cast<float4 *>(prow + static_cast<size_t>(width - 1 - a) * d) =
                        zero ? z : make_float4(tap[a][0], tap[a][1], tap[a][2], tap[a][3]);
            *reinterpret_cast<float4 *>(prow + static_cast<size_t>(width) * d) =
                zero ? z : make_float4(db[0].x, db[0].y, db[1].x, db[1].y);
            *reinterpret_cast<float4 *>(prow + static_cast<size_t>(width + 1) * d) =
                zero ? z : make_float4(dnw[0], dnw[1], dnw[2], dnw[3]);
        };
        // rows of the item just finished (if any) and zeros for the range's items without tokens before
        // stream index `next`
        int64_t cur_k = -1;
        auto finish_items = [&](int64_t next) {
            int64_t k = klo;
            if (cur_k >= 0) {
                write_rows(sc_bwd_item(cur_k, p.nchunks, dil), false);
                k = cur_k + 1;
            }
            for (; k < next; ++k) write_rows(sc_bwd_item(k, p.nchunks, dil), true);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                db[h] = make_float2(0.f, 0.f);
#pragma unroll
                for (int a = 0; a < kScAges; ++a) A[a][h] = make_float2(0.f, 0.f);
            }
        };
        finish_items(-1);  // clears the accumulators

        for (;;) {
            // a steady group starts only at a stage divisible by 4: there, its four stages are tried at
            // once (they do not wrap); otherwise, or while one is still filling, the first alone
            bool four = false;
            if (!failed && (st & 3) == 0) four = __all_sync(0xffffffffu, sc_try_wait4(&full[st], ph));
            if (!four) wait_stages(0, 1);
            if (failed) break;
            const uint32_t fl = meta[st].flags;
            if (fl & kFlDone) break;
            if (fl & kFlItemStart) {
                const int64_t k = static_cast<int64_t>(fl >> kFlItemShift);
                finish_items(k);
                cur_k = k;
            }
            if (fl & kFlSegStart) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    U[0][h] = U[1][h] = U[2][h] = U[3][h] = make_float2(0.f, 0.f);
                    P1[h] = P2[h] = P3[h] = make_float2(0.f, 0.f);
                }
                pend1 = pend2 = pend3 = false;
            }
            if (fl & kFlGroup) {
                if (nfin > 0) post();  // a steady group fills one batch of its own
                // all four stages first, so that the four positions' loads and arithmetic may overlap.
                // The group starts at a stage divisible by 4, so its stages st0 .. st0 + 3 do not wrap;
                // the tokens three back are at st0 - 3 .. st0 - 1 (wrapping when st0 = 0), then st0.
                if (!four) wait_stages(1, 4);
                if (failed) break;
                const int st0 = st;
                const int bk = (st0 == 0 ? S : st0) - kBwLag;
                step(ScIdx<0>{}, ScIdx<1>{}, kScMain, st0, bk);
                step(ScIdx<1>{}, ScIdx<1>{}, kScMain, st0 + 1, bk + 1);
                step(ScIdx<2>{}, ScIdx<1>{}, kScMain, st0 + 2, bk + 2);
                step(ScIdx<3>{}, ScIdx<1>{}, kScMain, st0 + 3, st0);
                nfin = kBwBatch;
                st = st0 + 4;
                if (st == S) st = 0, ph ^= 1u;
                pend1 = pend2 = pend3 = true;
            } else {
                const uint32_t kind = fl & kFlKind;
                switch ((fl >> kFlSlotShift) & 3u) {
                    case 0: step(ScIdx<0>{}, ScIdx<0>{}, kind, st, 0); break;
                    case 1: step(ScIdx<1>{}, ScIdx<0>{}, kind, st, 0); break;
                    case 2: step(ScIdx<2>{}, ScIdx<0>{}, kind, st, 0); break;
                    default: step(ScIdx<3>{}, ScIdx<0>{}, kind, st, 0); break;
                }
            }
            if (nfin == kBwBatch) post();
            if (fl & kFlSegEnd) {
                // the sequence (or the look-ahead) ends: the pending du have all their terms
                if (pend3) {
                    complete(3, P3);
                    if (nfin == kBwBatch) post();
                }
                if (pend2) {
                    complete(2, P2);
                    if (nfin == kBwBatch) post();
                }
                if (pend1) complete(1, P1);
                if (nfin > 0) post();
                if (prev_n > 0) finalize_any(nb - 1, prev_n, pst);
                prev_n = 0;
                pst = 0;
                pend1 = pend2 = pend3 = false;
            }
        }
        if (!failed) finish_items(khi);
    }
    sc_cluster_sync();  // no CTA leaves while a peer may still write into its shared memory
}

// ------------------------------------------------------------------------------- forward, swept

constexpr int kFwWarps = 4;                       // consumer warps
constexpr int kFwEV = 8;                          // channels per consumer thread (four pairs)
constexpr int kFwPairs = kFwEV / 2;
constexpr int kFwCons = kFwWarps * 32;
constexpr int kFwThreads = kFwCons + 32;          // + the copy producer's warp
constexpr int kFwCW = kFwCons * kFwEV;            // channels per CTA (one channel block)
// ring stages: 16 of 4 KB (bf16), 8 of 8 KB (fp32)
template <typename E>
__host__ __device__ constexpr int sc_fwd_stages() { return sizeof(E) == 2 ? 16 : 8; }
constexpr int kFwChunk = 128;                     // tokens per work item's time chunk

struct ScFwdSweepParams {
    const uint8_t *v, *h;                         // V~, H (nullable) [T, d]
    const float *norm_w, *conv_w, *bias, *rstd;
    const int64_t *offs;
    uint8_t *out;
    uint32_t *status;
    int64_t T;
    int64_t chunk;
    int64_t items;                                // per channel block: chunks x dilation
    int32_t num_seqs, d, width, dil, nblk, per_blk;  // per_blk: CTAs per channel block
};

template <typename E>
__host__ __device__ constexpr int sc_fwd_stage_bytes() {
    return 2 * kFwCW * static_cast<int>(sizeof(E));  // the V~ segment, then the H segment
}
// the ring, the stages' position records, full and empty mbarriers, the producer's state
template <typename E>
__host__ __device__ constexpr int sc_fwd_sweep_smem() {
    return sc_fwd_stages<E>() * (sc_fwd_stage_bytes<E>() + 16 + 2 * 8) + 128;
}

// The forward as a sweep.  CTA (block cb, j) owns channels [1024 cb, 1024 cb + 1024) and the work items
// j, j + per_blk, ... of that block, each one residue class t = r mod dilation of one time chunk.
// Its producer warp walks the items' segments and streams, per sweep position, the token's V~ and
// H row segments (1-D bulk copies) and rstd (a 4-byte asynchronous copy) into a ring of stages,
// with a record of the position; a segment starts with up to three lead-in tokens whose V~ the
// first taps read.  Every consumer thread owns eight channels (four pairs) and carries the last three
// taps' inputs u = V~ rstd in registers (slot q mod 4 for position q), so each row is converted
// once:
//   conv = bias + sum_a (conv_w[width-1-a] norm_w) u[t - a dil]   (a = 0, 1, 2, 3 in order),
//   out  = H + SiLU(conv) + V~,
// the taps before a sequence's start being zero.  All waits are bounded.
template <typename E, bool HAS_H>
__global__ void __launch_bounds__(kFwThreads, 3) conv_fwd_sweep_kernel(const __grid_constant__ ScFwdSweepParams p) {
    using EV = Ev8<E>;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int S = sc_fwd_stages<E>();
    constexpr int SB = sc_fwd_stage_bytes<E>();
    constexpr int half = SB / 2;
    uint8_t *ring = smem;
    ScMeta *meta = reinterpret_cast<ScMeta *>(smem + static_cast<size_t>(S) * SB);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + S);
    uint64_t *empty = full + S;
    ScProd *prod = reinterpret_cast<ScProd *>(empty + S);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int cb = static_cast<int>(blockIdx.x % p.nblk);
    const int j0 = static_cast<int>(blockIdx.x / p.nblk);
    const int c0 = cb * kFwCW;
    const int ncols = p.d - c0 < kFwCW ? p.d - c0 : kFwCW;
    const int64_t dil = p.dil;
    bool failed = false;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 2);  // the producer's arrival and its rstd copy's
            mbar_init(&empty[i], kFwWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();

    if (warp == kFwWarps) {
        // ---- the producer warp: one position per lane as stages free up, then the sentinel
        ScProd &P = *prod;
        auto start_item = [&](int64_t item) {  // item: k * dil + r of this block
            const int64_t t_lo = item / dil * p.chunk;
            P.item = item;
            P.xs = t_lo;
            P.t_hi = t_lo + p.chunk < p.T ? t_lo + p.chunk : p.T;
            P.s = sc_seq_of(p.offs, p.num_seqs, t_lo);
        };
        auto next_seg = [&]() {  // lane 0
            ScSeg g;
            for (;;) {
                int64_t xs = P.xs;
                int s = P.s;
                const bool found = sc_next_seg(p, static_cast<int>(P.item % dil), P.t_hi, xs, s, g, 0);
                P.xs = xs;
                P.s = s;
                if (found) {
                    P.q = 0;
                    P.n = g.n_lead + g.n_main;
                    P.n_lead = g.n_lead;
                    P.t = g.first - g.n_lead * dil;
                    return;
                }
                const int64_t next = P.item + p.per_blk;
                if (next >= p.items) {
                    P.state = 1;
                    return;
                }
                start_item(next);
            }
        };
        if (lane == 0) {
            P = ScProd{};
            if (j0 >= p.items) {
                P.state = 1;
            } else {
                start_item(j0);
                next_seg();
            }
        }
        __syncwarp();
        const uint32_t seg = static_cast<uint32_t>(ncols) * sizeof(E);
        const size_t row_bytes = static_cast<size_t>(p.d) * sizeof(E);
        const uint8_t *src_v = p.v + static_cast<size_t>(c0) * sizeof(E);
        const uint8_t *src_h = p.h ? p.h + static_cast<size_t>(c0) * sizeof(E) : nullptr;
        int st = 0, state = P.state;
        uint32_t round = 0, issued = 0;
        int q = P.q, n = P.n, nl = P.n_lead;
        int64_t t = P.t;
        while (state != 2) {
            const int stl = st + lane < S ? st + lane : st + lane - S;
            const uint32_t rl = round + (st + lane < S ? 0u : 1u);
            const bool free_l = lane < S && (rl == 0 || mbar_test_wait(&empty[stl], (rl + 1) & 1u));
            const uint32_t mask = __ballot_sync(0xffffffffu, free_l);
            int cnt = __ffs(~mask) - 1;
            if (cnt < 0) cnt = 32;
            if (cnt == 0) {  // the ring is full: wait (bounded) for its oldest stage
                bool ok = true;
                if (lane == 0) ok = mbar_wait_sleep(&empty[st], (round + 1) & 1u);
                if (!__shfl_sync(0xffffffffu, ok, 0)) {
                    if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                    failed = true;
                    break;
                }
                continue;
            }
            if (state == 1) {  // the sentinel: no copies, both arrivals
                if (lane == 0) {
                    meta[st].row = 0;
                    meta[st].flags = kFlDone;
                    mbar_arrive(&full[st]);
                    mbar_arrive(&full[st]);
                }
                state = 2;
                cnt = 1;
            } else {
                if (cnt > n - q) cnt = n - q;
                if (lane < cnt) {
                    const int ql = q + lane;
                    const int64_t tl = t + lane * dil;
                    const bool lead = ql < nl;
                    const bool group = (ql & 3) == 0 && ql >= nl && ql + 4 <= n;
                    uint32_t fl = (lead ? kScLead : kScMain) | (static_cast<uint32_t>(ql & 3) << kFlSlotShift);
                    if (ql == 0) fl |= kFlSegStart;
                    if (group) fl |= kFlGroup;
                    meta[stl].row = tl * static_cast<int64_t>(row_bytes);
                    meta[stl].flags = fl;
                    uint8_t *dst = ring + static_cast<size_t>(stl) * SB;
                    const bool with_h = !lead && src_h;
                    sc_cp_async4(&meta[stl].rstd, p.rstd + tl);
                    sc_cp_async_arrive(&full[stl]);
                    mbar_arrive_expect_tx(&full[stl], with_h ? 2 * seg : seg);
                    bulk_load_plain(dst, src_v + static_cast<size_t>(tl) * row_bytes, seg, &full[stl]);
                    if (with_h)
                        bulk_load(dst + half, src_h + static_cast<size_t>(tl) * row_bytes, seg, &full[stl],
                                  l2_evict_first_policy());
                }
                q += cnt;
                t += cnt * dil;
                if (q == n) {
                    __syncwarp();
                    if (lane == 0) next_seg();
                    __syncwarp();
                    state = P.state, q = P.q, n = P.n, nl = P.n_lead, t = P.t;
                }
            }
            issued += cnt;
            st += cnt;
            if (st >= S) st -= S, ++round;
        }
        // after a failure, copies may still be landing: wait for them (bounded) before the CTA leaves
        if (failed && lane == 0)
            for (uint32_t q2 = issued > static_cast<uint32_t>(S) ? issued - S : 0; q2 < issued; ++q2)
                mbar_wait(&full[q2 % S], (q2 / S) & 1u, kWaitLimitNs / 16);
    } else {
        // ---- consumers
        const bool active = tid * kFwEV < ncols;
        const uint8_t *my_ring = ring + tid * EV::kBytes;  // this thread's channels in stage 0
        const int width = p.width, d = p.d;
        float2 K[kScAges][kFwPairs], bias[kFwPairs];  // taps by age folded with norm_w; [h]: channels 2h, 2h + 1
#pragma unroll
        for (int h = 0; h < kFwPairs; ++h) {
            float v[2][1 + kScAges];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = c0 + tid * kFwEV + 2 * h + k;
                const bool ok = active && c < d;
                const float nwc = ok ? __ldg(p.norm_w + c) : 0.f;
                v[k][0] = ok && p.bias ? __ldg(p.bias + c) : 0.f;
#pragma unroll
                for (int a = 0; a < kScAges; ++a)
                    v[k][1 + a] =
                        ok && a < width ? __ldg(p.conv_w + static_cast<size_t>(c) * width + (width - 1 - a)) * nwc : 0.f;
            }
            bias[h] = make_float2(v[0][0], v[1][0]);
#pragma unroll
            for (int a = 0; a < kScAges; ++a) K[a][h] = make_float2(v[0][1 + a], v[1][1 + a]);
        }
        uint8_t *out_col = p.out + static_cast<size_t>(c0) * sizeof(E) + tid * EV::kBytes;
        float2 U[4][kFwPairs];  // u = V~ rstd by slot
        static_assert((S & (S - 1)) == 0, "stage and phase from the position count by mask and shift");
        constexpr int kLogS = S == 16 ? 4 : (S == 32 ? 5 : 3);
        static_assert((1 << kLogS) == S, "the ring's size is 8, 16 or 32");
        uint32_t gq = 0;  // positions consumed: position gq + k sits in stage (gq + k) mod S
        auto stage_of = [&](uint32_t k) { return static_cast<int>((gq + k) & (S - 1)); };
        auto parity_of = [&](uint32_t k) { return ((gq + k) >> kLogS) & 1u; };

        // stages of positions gq + k0 .. gq + k1 - 1 full: every lane tries them all back to back and
        // the warp agrees; only when one is still filling, every lane waits for it (bounded)
        auto wait_stages = [&](int k0, int k1) {
            if (failed) return;
            bool ok = true;
#pragma unroll 4
            for (int k = k0; k < k1; ++k) ok &= mbar_try_wait(&full[stage_of(k)], parity_of(k));
            if (__all_sync(0xffffffffu, ok)) return;
            ok = true;
            for (int k = k0; k < k1; ++k) ok = ok && mbar_wait_sleep(&full[stage_of(k)], parity_of(k));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) report(p.status, nullptr, ENGRAM_DEVERR_TIMEOUT);
                failed = true;
            }
        };
        // position gq + K in slot J, its stage already waited for; GROUP: its stage is released with
        // the group's
        auto step = [&](auto Jc, auto Kc, auto Gc, bool lead) {
            constexpr bool GROUP = decltype(Gc)::v != 0;
            constexpr int J = decltype(Jc)::v;
            const int st = stage_of(decltype(Kc)::v);
            const uint8_t *stg = my_ring + st * SB;
            const float2 rt = p2(meta[st].rstd);
            float2 x[kFwPairs];
            EV::load4(stg, x);
#pragma unroll
            for (int h = 0; h < kFwPairs; ++h) U[J][h] = p2mul(x[h], rt);
            if (!lead) {
                float2 y[kFwPairs];
#pragma unroll
                for (int h = 0; h < kFwPairs; ++h) y[h] = make_float2(0.f, 0.f);
                if (HAS_H) EV::load4(stg + half, y);
                float2 o[kFwPairs];
#pragma unroll
                for (int h = 0; h < kFwPairs; ++h) {
                    const float2 c = p2fma(K[3][h], U[(J + 1) & 3][h],
                                           p2fma(K[2][h], U[(J + 2) & 3][h],
                                                 p2fma(K[1][h], U[(J + 3) & 3][h], p2fma(K[0][h], U[J][h], bias[h]))));
                    o[h] = p2fma(c, p2sigmoid(c), p2add(x[h], y[h]));
                }
                if (active) EV::store4(out_col + meta[st].row, o);
            }
            if (!GROUP) {
                __syncwarp();
                mbar_arrive_if(&empty[st], lane == 0 && !failed);
            }
        };

        for (;;) {
            wait_stages(0, 1);
            if (failed) break;
            const uint32_t fl = meta[stage_of(0)].flags;
            if (fl & (kFlDone | kFlSegStart)) {
                if (fl & kFlDone) break;
#pragma unroll
                for (int h = 0; h < kFwPairs; ++h) U[0][h] = U[1][h] = U[2][h] = U[3][h] = make_float2(0.f, 0.f);
            }
            if (fl & kFlGroup) {
                // all four stages first, so that the four positions' loads and arithmetic may overlap
                wait_stages(1, 4);
                if (failed) break;
                step(ScIdx<0>{}, ScIdx<0>{}, ScIdx<1>{}, false);
                step(ScIdx<1>{}, ScIdx<1>{}, ScIdx<1>{}, false);
                step(ScIdx<2>{}, ScIdx<2>{}, ScIdx<1>{}, false);
                step(ScIdx<3>{}, ScIdx<3>{}, ScIdx<1>{}, false);
                __syncwarp();  // the group's four stages at once, one lane each
                mbar_arrive_if(&empty[stage_of(lane & 3)], lane < 4 && !failed);
                gq += 4;
            } else {
                const bool lead = (fl & kFlKind) == kScLead;
                switch ((fl >> kFlSlotShift) & 3u) {
                    case 0: step(ScIdx<0>{}, ScIdx<0>{}, ScIdx<0>{}, lead); break;
                    case 1: step(ScIdx<1>{}, ScIdx<0>{}, ScIdx<0>{}, lead); break;
                    case 2: step(ScIdx<2>{}, ScIdx<0>{}, ScIdx<0>{}, lead); break;
                    default: step(ScIdx<3>{}, ScIdx<0>{}, ScIdx<0>{}, lead); break;
                }
                gq += 1;
            }
        }
    }
}

// ------------------------------------------------------------------------------- weight-gradient reduction

// S = sum_p partial[p] over the (width + 2) * d columns (column_sums: an order that depends on P
// only), then dconv_w[c, i] = S[i * d + c], dbias[c] = S[width * d + c], dnorm_w[c] = S[(width + 1) * d + c]
// (d is a multiple of 4, so the four columns of a float4 lie in one row of S).
__global__ void __launch_bounds__(kColThreads, 1)
    conv_grad_reduce_kernel(const float4 *__restrict__ part, int32_t P, int32_t width, int32_t d,
                            float *__restrict__ dconv_w, float *__restrict__ dbias, float *__restrict__ dnorm_w) {
    __shared__ ColSumSmem sm;
    const int d4 = (width + 2) * (d / 4);
    column_sums(part, P, d4, sm, [&](int col, const float4 &t) {
        const int row = (4 * col) / d, c = 4 * col - row * d;
        const float v[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (row < width) dconv_w[static_cast<size_t>(c + i) * width + row] = v[i];
            else if (row == width) {
                if (dbias) dbias[c + i] = v[i];
            } else dnorm_w[c + i] = v[i];
        }
    });
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
    if (d > kBwMaxCluster * kBwCW) return fail(ENGRAM_ERR_SHAPE, "%s: d = %d exceeds %d", fn, d, kBwMaxCluster * kBwCW);
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

// Clusters of ceil(d / 512) CTAs, as many as fit at once (at most one per work item), each
// walking the work items cluster_id, cluster_id + clusters, ...
constexpr int kScDevices = 64;

template <typename E>
engram_status sc_bwd_launch(const char *fn, ScBwdParams prm, const DeviceInfo &dev, cudaStream_t s) {
    const int C = (prm.d + kBwCW - 1) / kBwCW;
    const int smem = sc_bwd_smem(kBwStages, sc_bwd_stage_bytes<E>());
    void (*kern)(ScBwdParams) = conv_bwd_kernel<E>;
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), smem);
    if (st != ENGRAM_OK) return st;
    // three CTAs per SM: the largest shared-memory carveout; clusters above 8 CTAs (d > 4096) are
    // a non-portable size
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
            cudaSuccess ||
        (C > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess))
        return check_launch(fn);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(C);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(C));
    cfg.blockDim = dim3(kBwThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // clusters resident at once, per (device, element size, cluster size)
    static std::atomic<int> cached[kScDevices][2][kBwMaxCluster + 1];
    std::atomic<int> &slot = cached[dev.device % kScDevices][sizeof(E) == 4 ? 1 : 0][C];
    int maxcl = slot.load(std::memory_order_relaxed);
    if (maxcl <= 0) {
        cudaError_t e = cudaOccupancyMaxActiveClusters(&maxcl, kern, &cfg);
        if (e != cudaSuccess || maxcl < 1) {
            cudaGetLastError();
            return fail(ENGRAM_ERR_CUDA, "%s: no cluster of %d CTAs with %d bytes of shared memory fits (%s)", fn, C,
                        smem, cudaGetErrorString(e));
        }
        slot.store(maxcl, std::memory_order_relaxed);
    }
    int64_t ncl = std::min<int64_t>(prm.nitems, maxcl);
    ncl = std::max<int64_t>(1, cap_grid(ncl * C) / C);
    cfg.gridDim = dim3(static_cast<unsigned>(ncl * C));
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    cudaLaunchKernelEx(&cfg, kern, prm);
    return check_launch(fn);
}

// The swept forward: nblk channel blocks x per_blk CTAs, as many as fit at once, with per_blk
// chosen so that every CTA of a block takes the same number of work items.
template <typename E>
engram_status sc_fwd_launch(const char *fn, ScFwdSweepParams fp, const DeviceInfo &dev, cudaStream_t s) {
    void (*kern)(ScFwdSweepParams) = fp.h ? conv_fwd_sweep_kernel<E, true> : conv_fwd_sweep_kernel<E, false>;
    const int smem = sc_fwd_sweep_smem<E>();
    engram_status st = set_smem(reinterpret_cast<const void *>(kern), smem);
    if (st != ENGRAM_OK) return st;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
        cudaSuccess)
        return check_launch(fn);
    static std::atomic<int> cached[kScDevices][2][2];
    std::atomic<int> &slot = cached[dev.device % kScDevices][sizeof(E) == 4 ? 1 : 0][fp.h ? 1 : 0];
    int per_sm = slot.load(std::memory_order_relaxed);
    if (per_sm <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFwThreads, smem) != cudaSuccess ||
            per_sm < 1) {
            cudaGetLastError();
            return fail(ENGRAM_ERR_CUDA, "%s: no CTA of %d bytes of shared memory fits", fn, smem);
        }
        slot.store(per_sm, std::memory_order_relaxed);
    }
    const int64_t cap = std::max<int64_t>(1, cap_grid(static_cast<int64_t>(per_sm) * dev.num_sms) / fp.nblk);
    const int64_t rounds = (fp.items + cap - 1) / cap;
    const int64_t per_blk = std::max<int64_t>(1, (fp.items + rounds - 1) / rounds);
    fp.per_blk = static_cast<int32_t>(per_blk);
    const int64_t grid = per_blk * fp.nblk;
    if (grid > 0x7fffffff) return fail(ENGRAM_ERR_SHAPE, "%s: too many CTAs", fn);
    cudaError_t e = launch_kernel(kern, dim3(static_cast<unsigned>(grid)), dim3(kFwThreads), smem, s, fp);
    (void)e;
    return check_launch(fn);
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

namespace {

// The forward; with `own_rstd` the statistic pass first writes rstd, else rstd is the caller's.
engram_status sc_fwd(const char *fn, const void *v, const void *h, engram_dtype dtype, const float *norm_w,
                     const float *conv_w, const float *bias, const int64_t *seq_offsets, int32_t num_seqs, int64_t T,
                     int32_t d, int32_t width, int32_t dilation, float eps, void *out, float *rstd, bool own_rstd,
                     engram_stream_t stream) {
    engram_status st = sc_check(fn, dtype, T, d, width, dilation, num_seqs);
    if (st != ENGRAM_OK) return st;
    if (!norm_w || !conv_w || !seq_offsets) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (T == 0) return ENGRAM_OK;
    if (!v || !out || !rstd) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (out == v) return fail(ENGRAM_ERR_SHAPE, "%s: out may not alias V~ (later tokens read it as taps)", fn);
    const void *ptrs[] = {v, h, out, norm_w, conv_w, bias, seq_offsets, rstd};
    DeviceInfo dev;
    if ((st = sc_ptrs(fn, ptrs, 8, 6, &dev)) != ENGRAM_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (own_rstd) {
        const int64_t rgrid = cap_grid(std::min<int64_t>((T + 7) / 8, static_cast<int64_t>(dev.num_sms) * 8));
        if (dtype == ENGRAM_F32)
            conv_rstd_kernel<float><<<static_cast<unsigned>(rgrid), 256, 0, s>>>(static_cast<const uint8_t *>(v), T,
                                                                                d, eps, rstd);
        else
            conv_rstd_kernel<__nv_bfloat16><<<static_cast<unsigned>(rgrid), 256, 0, s>>>(
                static_cast<const uint8_t *>(v), T, d, eps, rstd);
        if ((st = check_launch(fn)) != ENGRAM_OK) return st;
    }
    ScFwdSweepParams fp{};
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
    fp.chunk = kFwChunk;
    fp.items = (T + kFwChunk - 1) / kFwChunk * dilation;
    fp.num_seqs = num_seqs;
    fp.d = d;
    fp.width = width;
    fp.dil = dilation;
    fp.nblk = (d + kFwCW - 1) / kFwCW;
    return dtype == ENGRAM_F32 ? sc_fwd_launch<float>(fn, fp, dev, s) : sc_fwd_launch<__nv_bfloat16>(fn, fp, dev, s);
}

}  // namespace

extern "C" engram_status engram_short_conv_fwd(const void *v, const void *h, engram_dtype dtype, const float *norm_w,
                                               const float *conv_w, const float *bias, const int64_t *seq_offsets,
                                               int32_t num_seqs, int64_t T, int32_t d, int32_t width,
                                               int32_t dilation, float eps, void *out, float *rstd,
                                               engram_stream_t stream) {
    return sc_fwd("engram_short_conv_fwd", v, h, dtype, norm_w, conv_w, bias, seq_offsets, num_seqs, T, d, width,
                  dilation, eps, out, rstd, true, stream);
}

extern "C" engram_status engram_short_conv_fwd_given_rstd(const void *v, const void *h, engram_dtype dtype,
                                                          const float *norm_w, const float *conv_w, const float *bias,
                                                          const int64_t *seq_offsets, int32_t num_seqs, int64_t T,
                                                          int32_t d, int32_t width, int32_t dilation,
                                                          const float *rstd, void *out, engram_stream_t stream) {
    return sc_fwd("engram_short_conv_fwd_given_rstd", v, h, dtype, norm_w, conv_w, bias, seq_offsets, num_seqs, T, d,
                  width, dilation, 0.f, out, const_cast<float *>(rstd), false, stream);
}

extern "C" engram_status engram_short_conv_bwd(const void *dout, const void *v, engram_dtype dtype,
                                               const float *norm_w, const float *conv_w, const float *bias,
                                               const float *rstd, const int64_t *seq_offsets, int32_t num_seqs,
                                               int64_t T, int32_t d, int32_t width, int32_t dilation, void *dv,
                                               float *dw_partial, int32_t P, engram_stream_t stream) {
    const char *fn = "engram_short_conv_bwd";
    engram_status st = sc_check(fn, dtype, T, d, width, dilation, num_seqs);
    if (st != ENGRAM_OK) return st;
    int32_t want = 0;
    if ((st = engram_short_conv_num_partials(T, dilation, &want)) != ENGRAM_OK) return st;
    if (P != want) return fail(ENGRAM_ERR_SHAPE, "%s: P = %d, engram_short_conv_num_partials gives %d", fn, P, want);
    if (!norm_w || !conv_w || !seq_offsets) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (T == 0) return ENGRAM_OK;
    if (!dout || !v || !rstd || !dv || !dw_partial) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (dv == v || dv == dout) return fail(ENGRAM_ERR_SHAPE, "%s: dv may not alias V~ or dout", fn);
    const void *ptrs[] = {dout, v, dv, dw_partial, norm_w, conv_w, bias, rstd, seq_offsets};
    DeviceInfo dev;
    if ((st = sc_ptrs(fn, ptrs, 9, 4, &dev)) != ENGRAM_OK) return st;
    ScBwdParams prm{};
    prm.v = static_cast<const uint8_t *>(v);
    prm.dout = static_cast<const uint8_t *>(dout);
    prm.norm_w = norm_w;
    prm.conv_w = conv_w;
    prm.bias = bias;
    prm.rstd = rstd;
    prm.offs = seq_offsets;
    prm.dv = static_cast<uint8_t *>(dv);
    prm.partial = dw_partial;
    prm.status = dev.status_word;
    prm.T = T;
    prm.chunk = sc_chunk(T);
    prm.nchunks = (T + prm.chunk - 1) / prm.chunk;
    prm.nitems = static_cast<int64_t>(P);
    if (prm.nitems > kBwMaxItems) return fail(ENGRAM_ERR_SHAPE, "%s: %d work items exceed %lld", fn, P, (long long)kBwMaxItems);
    prm.num_seqs = num_seqs;
    prm.d = d;
    prm.width = width;
    prm.dil = dilation;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    return dtype == ENGRAM_F32 ? sc_bwd_launch<float>(fn, prm, dev, s) : sc_bwd_launch<__nv_bfloat16>(fn, prm, dev, s);
}

extern "C" engram_status engram_short_conv_grad_reduce(const float *dw_partial, int32_t P, int32_t width, int32_t d,
                                                       float *dconv_w, float *dbias, float *dnorm_w,
                                                       engram_stream_t stream) {
    const char *fn = "engram_short_conv_grad_reduce";
    if (P < 0 || d <= 0 || width < 1 || width > kScAges)
        return fail(ENGRAM_ERR_SHAPE, "%s: P = %d, d = %d, width = %d", fn, P, d, width);
    if ((!dw_partial && P > 0) || !dconv_w || !dnorm_w) return fail(ENGRAM_ERR_NULL, "%s: NULL pointer", fn);
    if (d % 4 != 0) return fail(ENGRAM_ERR_ALIGN, "%s: d = %d is not a multiple of 4", fn, d);
    if ((static_cast<int64_t>(width) + 2) * (d / 4) > 0x7fffffff) return fail(ENGRAM_ERR_SHAPE, "%s: d = %d", fn, d);
    const void *ptrs[] = {dw_partial, dconv_w, dbias, dnorm_w};
    DeviceInfo dev;
    engram_status st = sc_ptrs(fn, ptrs, 4, 1, &dev);  // the partials are read as float4
    if (st != ENGRAM_OK) return st;
    const int d4 = (width + 2) * (d / 4);
    conv_grad_reduce_kernel<<<column_sum_grid(d4, dev.num_sms), kColThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4 *>(dw_partial), P, width, d, dconv_w, dbias, dnorm_w);
    return check_launch(fn);
}
