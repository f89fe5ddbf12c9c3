// Vector helpers: one thread moves one vector of a row per access (16 bytes:
// 8 bf16 or 4 float32; 8 bytes: 8 e4m3), converting to float32 registers and
// back with round-to-nearest-even (e4m3: saturating to +-448).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace kvm {

// One 8-bit E4M3 element (sign, 4 exponent bits with bias 7, 3 mantissa bits),
// held as its bit pattern.
struct e4m3 {
    uint8_t bits;
};

template <typename T>
struct VecTraits;

template <>
struct VecTraits<float> {
    using V = uint4;
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
    using V = uint4;
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

template <>
struct VecTraits<e4m3> {
    using V = uint2;
    static constexpr int N = 8;
    __device__ static inline void unpack(const uint2 &v, float (&f)[8]) {
        const uint32_t w[2] = {v.x, v.y};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // two elements, the lower-addressed one in the low byte; e4m3 is
                // a subset of fp16, so both conversions are exact
                const __nv_fp8x2_storage_t p = (__nv_fp8x2_storage_t)(w[i] >> (16 * h));
                const __half2 hh = __half2(__nv_cvt_fp8x2_to_halfraw2(p, __NV_E4M3));
                const float2 f2 = __half22float2(hh);
                f[4 * i + 2 * h] = f2.x;
                f[4 * i + 2 * h + 1] = f2.y;
            }
        }
    }
    __device__ static inline uint32_t pack2(float a, float b) {
        return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    }
    __device__ static inline uint2 pack(const float (&f)[8]) {
        return make_uint2(pack2(f[0], f[1]) | (pack2(f[2], f[3]) << 16),
                          pack2(f[4], f[5]) | (pack2(f[6], f[7]) << 16));
    }
};

// Read-once and write-once traffic: streaming cache hints.
__device__ inline uint4 ld_stream(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ inline void st_stream(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}
__device__ inline void ld_stream_v(const void *p, uint4 &v) {
    v = __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ inline void ld_stream_v(const void *p, uint2 &v) {
    v = __ldcs(reinterpret_cast<const uint2 *>(p));
}
__device__ inline void st_stream_v(void *p, const uint4 &v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}
__device__ inline void st_stream_v(void *p, const uint2 &v) {
    __stcs(reinterpret_cast<uint2 *>(p), v);
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
