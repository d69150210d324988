// The row-streaming pipeline shared by the gate forward and backward kernels.
//
// A CTA has NCW consumer warps and one producer warp.  The producer's elected
// lane streams whole token rows (h, k, v, and dout for the backward) from HBM
// into a ring of S shared-memory stages with 1-D bulk async copies (TMA),
// signalling each stage's `full` mbarrier with the transferred byte count.  The
// consumers cooperate on one token per stage: every consumer thread owns the
// 16-byte vectors j = c, c + 32*NCW, c + 64*NCW, ... of the row, reduces its
// partial sums with warp shuffles and then across warps through shared memory,
// and releases the stage on its `empty` mbarrier (one arrival per warp).
//
// No row is kept on chip beyond its stage: the paper-form output alpha * v
// needs h and k only for three sums, so each tensor is read from HBM once.
#pragma once

#include "engram_internal.cuh"

namespace engram {

// Template instances: NCW in {1, 2, 4, 8} consumer warps, up to VPT vectors per thread.
constexpr int kVPT = 4;

// Host-side choice of consumer warps for a row of `row_bytes` bytes.
inline int pick_consumer_warps(int row_bytes) {
    const int nvec = row_bytes / 16;
    int ncw = 1;
    while (ncw < 8 && ncw * 32 * kVPT < nvec) ncw *= 2;
    return ncw;
}

struct PipelineShape {
    int stages;         // S
    int blocks_per_sm;  // resident CTAs per SM a persistent grid is sized for (0: one CTA per work unit)
    int smem_bytes;     // dynamic shared memory per CTA
};

// Stage ring + 2*S mbarriers + the [2][NCW][4] fp32 cross-warp reduction buffer.
inline int pipeline_smem_bytes(int stages, int stage_bytes, int ncw) {
    return stages * stage_bytes + 2 * stages * 8 + 2 * ncw * 4 * 4;
}

// Forward: two stages per CTA and as many resident CTAs per SM (1..6) as keep about
// 160 KB of rows in flight per SM.  Measured on GB300 (T = 8192..131072, d = 2048..7168):
// more CTAs with fewer stages beat fewer, deeper CTAs, because each CTA works on one token
// at a time and its reduction bubble is hidden by the other CTAs' copies.  At d = 2048 bf16
// (12 KB stages, two consumer warps) six CTAs measured 23.5 us against 24.0-24.3 us for four;
// eight CTAs, or three stages, no better.
inline PipelineShape pick_fwd_pipeline(int stage_bytes, int ncw, int smem_optin) {
    const int smem = pipeline_smem_bytes(2, stage_bytes, ncw);
    if (smem > smem_optin) return {0, 0, 0};
    int b = (160 * 1024 + stage_bytes) / (2 * stage_bytes);  // round(160 KB / (2 stages))
    b = b < 1 ? 1 : (b > 6 ? 6 : b);
    while (b > 1 && b * smem > 227 * 1024) --b;
    return {2, b, smem};
}

// Backward: three stages per CTA (two when three do not fit) and one CTA per weight-gradient
// partial, left to the hardware scheduler: CTAs start as others finish, which balances the
// P equal chunks over the SMs far better than a persistent grid (P is fixed by T alone, so
// it is rarely a multiple of the resident CTA count).
inline PipelineShape pick_bwd_pipeline(int stage_bytes, int ncw, int smem_optin) {
    for (int s = 3; s >= 2; --s) {
        const int smem = pipeline_smem_bytes(s, stage_bytes, ncw);
        if (smem <= smem_optin) return {s, 0, smem};
    }
    return {0, 0, 0};
}

// Sum over a named barrier's threads of a "failed" flag: every consumer thread
// learns whether any of them gave up waiting, so they leave the loop together.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

}  // namespace engram
