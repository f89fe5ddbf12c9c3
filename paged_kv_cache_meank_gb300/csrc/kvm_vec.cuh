// 16-byte vector helpers: one thread moves 16 bytes of a row per access
// (8 bf16 or 4 float32), converting to float32 registers and back with
// round-to-nearest-even.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace kvm {

template <typename T>
struct VecTraits;

template <>
struct VecTraits<float> {
    static constexpr int N = 4;
    __device__ static inline void unpack(const uint4 &v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static inline uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static inline void unpack(const uint4 &v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    __device__ static inline uint32_t pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ static inline uint4 pack(const float (&f)[8]) {
        return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]),
                          pack2(f[6], f[7]));
    }
};

// Read-once and write-once traffic: streaming cache hints.
__device__ inline uint4 ld_stream(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ inline void st_stream(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

template <typename T>
__device__ inline T from_float(float x);
template <>
__device__ inline float from_float<float>(float x) { return x; }
template <>
__device__ inline __nv_bfloat16 from_float<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <typename T>
__device__ inline float to_float(T x);
template <>
__device__ inline float to_float<float>(float x) { return x; }
template <>
__device__ inline float to_float<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}

}  // namespace kvm
