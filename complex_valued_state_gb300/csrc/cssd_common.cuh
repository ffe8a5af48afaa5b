// Device helpers shared by the libcssd kernels: complex64 arithmetic on
// float2 (x = re, y = im) and the discretisation a = exp(softplus(dt) * A).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/cssd.h"

namespace cssd {

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// a * b + c
__device__ __forceinline__ float2 cfma(float2 a, float2 b, float2 c) {
    return make_float2(fmaf(a.x, b.x, fmaf(-a.y, b.y, c.x)), fmaf(a.x, b.y, fmaf(a.y, b.x, c.y)));
}
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 cscale(float s, float2 a) { return make_float2(s * a.x, s * a.y); }

// log(1 + e^v) without overflow for large |v|.
__device__ __forceinline__ float softplusf(float v) { return fmaxf(v, 0.f) + log1pf(expf(-fabsf(v))); }

// Complex exponential exp(z) = e^{re} (cos im + i sin im), CUDA's accurate
// expf / sincosf (full range reduction of the angle).
__device__ __forceinline__ float2 cexpf2(float2 z) {
    float s, c;
    sincosf(z.y, &s, &c);
    const float m = expf(z.x);
    return make_float2(m * c, m * s);
}

// Log of the per-step factor: softplus(dt) * A (complex).
__device__ __forceinline__ float2 alog_of(float dt, float2 A) {
    const float sp = softplusf(dt);
    return make_float2(sp * A.x, sp * A.y);
}

}  // namespace cssd
