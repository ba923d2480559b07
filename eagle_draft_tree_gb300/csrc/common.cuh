// common.cuh -- small helpers shared by the EAGLE round kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "eagle.h"

namespace eagle {

// The first 256 bytes of every workspace hold the device status word (offset 0) and, for the
// verify, its per-call failure tag (offset 16).
constexpr size_t kWsHeader = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Record an error code in the workspace's sticky status word (largest code wins).
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) { atomicMax(status, code); }

// Map a float to an unsigned key whose integer order is the float order (finite inputs; -0 is
// folded onto +0 so that equal values compare equal).
__device__ __forceinline__ uint32_t float_order_key(float x) {
    uint32_t u = __float_as_uint(x + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float float_from_order_key(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// 64-bit selection key: larger value first, then lower token id first.  Never 0 for a finite x.
__device__ __forceinline__ uint64_t topk_key(float x, uint32_t token) {
    return (uint64_t(float_order_key(x)) << 32) | uint64_t(0xffffffffu - token);
}
__device__ __forceinline__ uint32_t topk_key_token(uint64_t key) { return 0xffffffffu - uint32_t(key); }
__device__ __forceinline__ float topk_key_value(uint64_t key) { return float_from_order_key(uint32_t(key >> 32)); }

__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
    uint32_t lo = __shfl_xor_sync(0xffffffffu, uint32_t(v), m);
    uint32_t hi = __shfl_xor_sync(0xffffffffu, uint32_t(v >> 32), m);
    return (uint64_t(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        uint64_t o = shfl_xor_u64(v, m);
        v = o > v ? o : v;
    }
    return v;
}

// Warp-wide sorted top-KMAX list: lane j < KMAX holds the j-th largest key seen (0 = empty).
// insert() offers one key per lane; only keys above the current KMAX-th key enter, one at a time
// (the list is shifted down by one lane at the insertion point).  Keys must be unique.
template <int KMAX>
struct WarpTopK {
    uint64_t key = 0;  // this lane's slot (lanes >= KMAX keep 0)
    uint64_t thr = 0;  // current KMAX-th key, identical on every lane

    __device__ __forceinline__ void insert(uint64_t cand) {
        const int lane = threadIdx.x & 31;
        unsigned pend = __ballot_sync(0xffffffffu, cand > thr);
        while (pend) {
            const int src = __ffs(pend) - 1;
            pend &= pend - 1;
            const uint64_t c = __shfl_sync(0xffffffffu, cand, src);  // (2 x 32-bit shuffles)
            if (c <= thr) continue;
            const unsigned above = __ballot_sync(0xffffffffu, lane < KMAX && key > c);
            const int pos = __popc(above);
            const uint64_t up = __shfl_up_sync(0xffffffffu, key, 1);
            if (lane < KMAX && lane >= pos) key = (lane == pos) ? c : up;
            thr = __shfl_sync(0xffffffffu, key, KMAX - 1);
        }
    }
};

// Merge two descending 16-key lists held by one warp: lanes 0..15 pass list A's key `lane`,
// lanes 16..31 pass list B's key `31 - lane` (B reversed, so the 32 lanes form a bitonic
// sequence).  Returns the merged descending sequence; lanes 0..15 hold the top 16.
__device__ __forceinline__ uint64_t warp_bitonic_merge32(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int stride = 16; stride > 0; stride >>= 1) {
        const uint64_t o = shfl_xor_u64(v, stride);
        const bool lower = (lane & stride) == 0;
        v = lower ? (o > v ? o : v) : (o < v ? o : v);
    }
    return v;
}

// Query rows of one 128-row M-tile of the tensor-core tree attention: whole nodes only, so a tile
// holds floor(128 / G) nodes of G query heads each (all 128 rows when G divides 128).
__host__ __device__ __forceinline__ int attn_tc_rows_per_mtile(int G) { return (128 / G) * G; }

// Orderable 64-bit image of a double (integer order = numeric order; -0 folded onto +0 by an
// integer test, which keeps the narrow FP64 pipe out of it).
__device__ __forceinline__ uint64_t double_order_key(double d) {
    uint64_t u = static_cast<uint64_t>(__double_as_longlong(d));
    if (u == 0x8000000000000000ull) u = 0;
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

// 2^x on the SFU (approximate, relative error about 2^-22; used inside softmax loops).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- fixed-point weight sums (integers in units of a power of two: sums are exact, so every
// thread and CTA that forms one gets the same value, whatever the order) ----
// Warp-wide exact sum of values below 2^54 (the result in every lane): two 32-bit reductions of
// the low 27 bits and of the rest.
__device__ __forceinline__ uint64_t warp_sum_fx(uint64_t v) {
    const uint32_t lo = __reduce_add_sync(0xffffffffu, uint32_t(v) & 0x7ffffffu);
    const uint32_t hi = __reduce_add_sync(0xffffffffu, uint32_t(v >> 27));
    return (uint64_t(hi) << 27) + lo;
}
// floor(u * total) for u in [0, 1) given as a float, exactly (u = mant 2^-sh).
__device__ __forceinline__ uint64_t scale_fx(uint64_t total, float u) {
    if (!(u > 0.f)) return 0;
    const uint32_t ub = __float_as_uint(u);
    const int ex = int((ub >> 23) & 0xffu);
    const uint64_t mant = (ub & 0x7fffffu) | (ex ? 0x800000u : 0u);
    const int sh = 150 - (ex ? ex : 1);  // >= 24 for u < 1
    const uint64_t lo = total * mant, hi = __umul64hi(total, mant);
    if (sh >= 128) return 0;
    if (sh >= 64) return hi >> (sh - 64);
    return (hi << (64 - sh)) | (lo >> sh);
}

// ln x for a positive finite double without the double-precision log (on GB300 the FP64 pipe is
// narrow and a double log costs microseconds of latency): x = f 2^e with f in [1, 2) taken from
// the bits, ln x = e ln 2 + ln f, with ln f in single precision plus the first-order correction
// for f's rounding to float (absolute error about 6e-8).  For arguments that are themselves sums
// of single-precision terms.
__device__ __forceinline__ double ln_pos(double x) {
    const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(x));
    const int e = int((bits >> 52) & 0x7ffull) - 1023;
    const double f = __longlong_as_double(static_cast<long long>((bits & 0xfffffffffffffull) | 0x3ff0000000000000ull));
    const float hi = float(f);
    return double(e) * 0.69314718055994530942 + double(logf(hi)) + (f - double(hi)) * double(1.f / hi);
}

// ---- mbarrier + bulk copy (global -> own shared memory), with bounded waits ----
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(count));
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(a), "r"(bytes) : "memory");
}
// One bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) into this CTA's shared
// memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
    const uint32_t b = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(d),
                 "l"(src), "r"(bytes), "r"(b)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}

// ---- bounded waits ----
// Every wait in the library gives up after kWaitNs of wall-clock time (%globaltimer).  A poll
// count alone would not bound it: try_wait may suspend the thread for a hardware-defined time
// on each poll.  The timer is read once every 256 polls, so a wait that completes early never
// touches it.
constexpr uint64_t kWaitNs = 1000ull * 1000ull * 1000ull;  // 1 s
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
struct Deadline {
    uint64_t start = 0;
    // true once kWaitNs have passed since the first check; `it` is the poll count
    __device__ __forceinline__ bool passed(uint32_t it) {
        if ((it & 255u) != 255u) return false;
        if (it >= (1u << 31)) return true;  // backstop, should the timer not advance
        const uint64_t t = global_ns();
        if (start == 0) {
            start = t;
            return false;
        }
        return t - start > kWaitNs;
    }
    // the same, agreed by the whole warp (`it` must be warp-uniform)
    __device__ __forceinline__ bool passed_warp(uint32_t it) {
        return (it & 255u) == 255u && __any_sync(0xffffffffu, passed(it));
    }
};
// Wait for phase `parity` of `bar`; false when the deadline passed first.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
    Deadline d;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (d.passed(it)) return false;
    }
}
// The same for a whole converged warp: every lane polls and the warp agrees by vote.
__device__ __forceinline__ bool mbar_warp_wait_bounded(uint64_t *bar, uint32_t parity) {
    Deadline d;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (d.passed_warp(it)) return false;
    }
}
// try_wait with acquire at cluster scope: for a phase completed by another CTA of the cluster
// (st.async bytes, whose complete-tx releases at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_warp_wait_cluster_bounded(uint64_t *bar, uint32_t parity) {
    Deadline d;
    for (uint32_t it = 0;; ++it) {
        if (__all_sync(0xffffffffu, mbar_try_wait_cluster(bar, parity))) return true;
        if (d.passed_warp(it)) return false;
    }
}

// Programmatic dependent launch.  Every kernel of the library is launched with programmatic stream
// serialisation, so it may start while the previous kernel in the stream is still running; it
// waits for that kernel's completion (and its memory) before touching global memory, then lets
// the next kernel launch early.  Both instructions are no-ops without a programmatic predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLn2 = 0.69314718055994530942;

}  // namespace eagle

// Launch accounting (per host thread) used by eagle_last_launch_count().
namespace eagle {
void note_launch();
void reset_launches();

// Streaming multiprocessors of the current device, queried once per device (152 on GB300, and
// 152 when no device can be queried, as in host-only use of the workspace-size functions).
int device_sm_count();

// Function attributes (dynamic shared memory size, cluster shape) belong to a device: `set` runs
// once for each device this process launches on, recorded in the caller's bit set `ready`
// (devices 64 and up run `set` on every call).
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t> &ready, F &&set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (ready.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = set();
    if (e == cudaSuccess && bit) ready.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Launch `kernel` with programmatic stream serialisation (and a cluster shape when cluster_x > 1).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    unsigned na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = cluster_x;
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
}  // namespace eagle
