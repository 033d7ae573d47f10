// ct_types.cuh -- element-type conversions shared by the kernels.
// Inputs are widened to fp32 exactly; results are rounded once to the output
// type with round-to-nearest-even.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace ct {

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Packed fp32 FMA on two lanes at once: d = a * b + d element-wise, each
// element an IEEE fp32 fused multiply-add with round-to-nearest (the same
// result as fmaf), at half the instruction count.
__device__ __forceinline__ void fma2(float2& d, const float2 a, const float2 b) {
    unsigned long long ud = (unsigned long long)__float_as_uint(d.x) |
                            ((unsigned long long)__float_as_uint(d.y) << 32);
    const unsigned long long ua = (unsigned long long)__float_as_uint(a.x) |
                                  ((unsigned long long)__float_as_uint(a.y) << 32);
    const unsigned long long ub = (unsigned long long)__float_as_uint(b.x) |
                                  ((unsigned long long)__float_as_uint(b.y) << 32);
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(ud) : "l"(ua), "l"(ub));
    d.x = __uint_as_float((unsigned)(ud & 0xffffffffull));
    d.y = __uint_as_float((unsigned)(ud >> 32));
}

// Activation (ct_activation codes of include/ct.h) of an fp32 value after
// the bias: 1 relu, 2 leaky relu (alpha), 3 silu, 4 gelu (erf form),
// 5 tanh, 6 sigmoid; anything else leaves v unchanged.
// act_fixed<A> is the same function for a compile-time code A (for loops that
// dispatch once on the code and then run one function at every site).
template <int A>
__device__ __forceinline__ float act_fixed(float v, float alpha) {
    if constexpr (A == 1) return v > 0.f ? v : 0.f;
    else if constexpr (A == 2) return v >= 0.f ? v : alpha * v;
    else if constexpr (A == 3) return v / (1.f + expf(-v));
    else if constexpr (A == 4) return 0.5f * v * (1.f + erff(v * 0.70710678118654752f));
    else if constexpr (A == 5) return tanhf(v);
    else if constexpr (A == 6) return 1.f / (1.f + expf(-v));
    else return v;
}

__device__ __forceinline__ float act_f32(float v, int act, float alpha) {
    switch (act) {
        case 1: return act_fixed<1>(v, alpha);
        case 2: return act_fixed<2>(v, alpha);
        case 3: return act_fixed<3>(v, alpha);
        case 4: return act_fixed<4>(v, alpha);
        case 5: return act_fixed<5>(v, alpha);
        case 6: return act_fixed<6>(v, alpha);
        default: return v;
    }
}

}  // namespace ct
