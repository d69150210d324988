// Internal helpers of the Engram GB300 library: host-side validation and error
// state, and the device-side building blocks (mbarrier, bulk async copies,
// bounded waits, bf16 packing) shared by the kernels.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "engram.h"

namespace engram {

// ---------------------------------------------------------------------------- host side

// Per-device facts the launchers need (cached on first use of each device).
struct DeviceInfo {
    int device;
    int num_sms;
    int smem_optin;          // max dynamic shared memory per block (opt-in)
    uint32_t *status_word;   // device address of the library's status word on this device
};

// Fills `info` for the current device.  ENGRAM_ERR_CUDA on failure.
engram_status current_device(DeviceInfo *info);

// Records `msg` as the calling thread's last error text and returns `st`.
engram_status fail(engram_status st, const char *fmt, ...);

// ENGRAM_ERR_DEVICE unless `p` is device (or managed) memory reachable from `device`
// (skipped at validation level 0).  NULL pointers are the caller's business.
engram_status check_device_ptr(const void *p, int device, const char *name);

// ENGRAM_ERR_CUDA with the runtime's text if the last launch failed.
engram_status check_launch(const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int dtype_size(engram_dtype dt) { return dt == ENGRAM_F32 ? 4 : (dt == ENGRAM_BF16 ? 2 : 0); }

// Applies the process-wide CTA cap (engram_set_max_ctas) to a grid size (>= 1 in, >= 1 out).
int64_t cap_grid(int64_t grid);

// Opts a kernel into `bytes` of dynamic shared memory (idempotent, cheap after the first call).
engram_status set_smem(const void *kernel, int bytes);

// Launches `kernel` on `stream`; when programmatic dependent launch is on (engram_set_pdl, on by
// default) the launch carries the programmatic-stream-serialization attribute, so it may be
// scheduled before the previous kernel on the stream has finished -- the kernel then calls
// pdl_wait() before it touches global memory.
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------- device side

// Programmatic dependent launch: pdl_wait() blocks until the previous kernel on the stream has
// completed and its writes are visible; a no-op in a kernel launched without the attribute.  The
// step's kernels call it first thing and never trigger early: an explicit trigger at kernel start let
// the next kernel's CTAs take SM space while they only waited, and measured 3 % slower per step.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Longest time a pipeline wait may take before the kernel gives up (ns).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy and the other threads.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// An arrival only where `on` holds, under a predicate rather than a branch.
__device__ __forceinline__ void mbar_arrive_if(uint64_t *bar, bool on) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_addr(bar)),
        "r"(static_cast<uint32_t>(on))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Whether phase `parity` of `bar` has completed, without suspending the thread (try_wait may wait a
// while for the phase before it answers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// try_wait that may suspend the thread until the phase completes or about `hint_ns` pass, so that a
// waiting warp takes no issue slots from the others.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// mbar_wait (below) whose polls sleep: false after limit_ns.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 1000000u)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// Waits for phase `parity` of `bar` to complete; false after limit_ns (kWaitLimitNs by default).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// An L2 policy that evicts first: for data streamed through exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk (TMA) copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global to this CTA's shared memory; completion is signalled on `bar` as tx bytes.
__device__ __forceinline__ void bulk_load(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// The same bulk copy with the default L2 policy.
__device__ __forceinline__ void bulk_load_plain(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst_smem)), "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
                 : "memory");
}

// Named barrier over `count` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---- thread-block clusters: rank and count, the cluster barrier, distributed shared memory

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_index() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// Every thread of every CTA of the cluster; release / acquire order shared memory across it.
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
// The shared::cluster address, in CTA `rank` of the cluster, of this CTA's shared address `a`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// A 4-byte store into another CTA's shared memory that completes 4 tx bytes on its mbarrier.
__device__ __forceinline__ void cluster_store_tx(uint32_t raddr, float v, uint32_t rbar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr),
                 "r"(__float_as_uint(v)), "r"(rbar)
                 : "memory");
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sets bits in an optional device error word and in the library's status word.
__device__ __forceinline__ void report(uint32_t *status_word, uint32_t *err_word, uint32_t bits) {
    if (status_word) atomicOr(status_word, bits);
    if (err_word) atomicOr(err_word, bits);
}

// ---- element packing: one 16-byte vector = 8 bf16 or 4 fp32 values

template <typename T>
struct Vec;

template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&x)[N]) {
        x[0] = __uint_as_float(u.x);
        x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z);
        x[3] = __uint_as_float(u.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&x)[N]) {
        return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                          __float_as_uint(x[3]));
    }
};

template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ __forceinline__ static void unpack(const uint4 &u, float (&x)[N]) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint32_t pack2(float lo, float hi) {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&b);
    }
    __device__ __forceinline__ static uint4 pack(const float (&x)[N]) {
        return make_uint4(pack2(x[0], x[1]), pack2(x[2], x[3]), pack2(x[4], x[5]), pack2(x[6], x[7]));
    }
};

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p))
                 : "memory");
    return r;
}

__device__ __forceinline__ void st_global_v4(void *p, const uint4 &v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

}  // namespace engram
