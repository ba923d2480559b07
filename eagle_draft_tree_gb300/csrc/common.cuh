// common.cuh -- small helpers shared by the EAGLE round kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "eagle.h"

namespace eagle {

// The first 256 bytes of every workspace hold the device status word.
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

// 2^x on the SFU (approximate, relative error about 2^-22; used inside softmax loops).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr double kLn2 = 0.69314718055994530942;

}  // namespace eagle

// Launch accounting (per host thread) used by eagle_last_launch_count().
namespace eagle {
void note_launch();
void reset_launches();
}  // namespace eagle
