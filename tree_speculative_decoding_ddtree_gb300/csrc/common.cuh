// Shared device helpers for the DDTree verify-step kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "ddtree.h"

#define DDT_DEVINL __device__ __forceinline__

namespace ddt {

// OR a device error bit into the caller's status word (nullable).
DDT_DEVINL void report(int32_t* dev_status, int bits) {
    if (dev_status) atomicOr(reinterpret_cast<int*>(dev_status), bits);
}

// Orderable 32-bit key of a float for an argmax where NaN ranks below
// every number and -0.0 equals +0.0: larger key <=> larger value.
DDT_DEVINL uint32_t float_order_key(float v) {
    if (v != v) return 0u;                     // NaN: below -inf
    if (v == 0.0f) v = 0.0f;                   // fold -0 into +0
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value key, index) packed so that a plain unsigned max picks the largest
// value and, among equal values, the lowest index.
DDT_DEVINL unsigned long long argmax_pack(uint32_t key, uint32_t idx) {
    return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFu - idx);
}
DDT_DEVINL uint32_t argmax_unpack_idx(unsigned long long p) {
    return 0xFFFFFFFFu - static_cast<uint32_t>(p & 0xFFFFFFFFull);
}

DDT_DEVINL unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

DDT_DEVINL float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

DDT_DEVINL float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// v[i] for a runtime i in 0..3 without indexing a register array (selects only)
DDT_DEVINL uint32_t pick4(const uint32_t (&v)[4], int i) {
    return i == 0 ? v[0] : (i == 1 ? v[1] : (i == 2 ? v[2] : v[3]));
}

}  // namespace ddt
