// Backward of the QK RMSNorm + RoPE prologue for one head vector, fused into
// the epilogues of the backward kernels (thread = one token's head vector).
//
// Given the gradient g with respect to xhat = RoPE(x / r, p) (r =
// sqrt(mean(x^2) + eps)), the gradient with respect to the raw x is
//   u  = R(p)^T g                       (rotate every pair (i, i + D/2) by -angle)
//   dx = (u - y <u, y> / D) / r,        y = x / r.
#pragma once

#include "nc_common.cuh"

namespace nc {

// g = out_scale * (the D fp32 columns of this thread's TMEM lane at `tm`);
// x: the raw bf16 row; cs: its RoPE table row (cos, sin) x D/2; urow: D
// floats of this thread's shared-memory staging; dx (nullptr = no store).
template <int D>
__device__ __forceinline__ void norm_rope_bwd_row(uint32_t tm, float out_scale, const __nv_bfloat16* __restrict__ x,
                                                  const float2* __restrict__ cs, float eps, float* urow,
                                                  __nv_bfloat16* __restrict__ dx) {
    constexpr int HALF = D / 2;
    float ss = 0.f;
#pragma unroll
    for (int e8 = 0; e8 < D / 8; ++e8) {
        float y[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + e8 * 8), y);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(y[i], y[i], ss);
    }
    const float rsd = rsqrtf(ss / D + eps);
    const float4* cs4 = reinterpret_cast<const float4*>(cs);
    // u = R^T g, staged in shared memory; <u, y> on the way
    float dot = 0.f;
#pragma unroll 2
    for (int ch = 0; ch < HALF / 8; ++ch) {
        uint32_t glo[8], ghi[8];
        tmem_ld8(tm + ch * 8, glo);
        tmem_ld8(tm + HALF + ch * 8, ghi);
        float ylo[8], yhi[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + ch * 8), ylo);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + HALF + ch * 8), yhi);
        float4 c4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c4[i] = cs4[ch * 4 + i];
        tmem_wait_ld();
        float ulo[8], uhi[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float c = (e & 1) ? c4[e >> 1].z : c4[e >> 1].x;
            const float sn = (e & 1) ? c4[e >> 1].w : c4[e >> 1].y;
            const float a = __uint_as_float(glo[e]) * out_scale;
            const float bb = __uint_as_float(ghi[e]) * out_scale;
            // R^T: (a, b) -> (a c + b s, -a s + b c)
            ulo[e] = a * c + bb * sn;
            uhi[e] = -a * sn + bb * c;
            dot = fmaf(ulo[e], ylo[e] * rsd, fmaf(uhi[e], yhi[e] * rsd, dot));
        }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            reinterpret_cast<float4*>(urow + ch * 8)[g] =
                make_float4(ulo[4 * g], ulo[4 * g + 1], ulo[4 * g + 2], ulo[4 * g + 3]);
            reinterpret_cast<float4*>(urow + HALF + ch * 8)[g] =
                make_float4(uhi[4 * g], uhi[4 * g + 1], uhi[4 * g + 2], uhi[4 * g + 3]);
        }
    }
    if (dx == nullptr) return;
    const float m = dot / D;
#pragma unroll
    for (int e8 = 0; e8 < D / 8; ++e8) {
        float y[8], o[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + e8 * 8), y);
        const float4 u0 = reinterpret_cast<const float4*>(urow + e8 * 8)[0];
        const float4 u1 = reinterpret_cast<const float4*>(urow + e8 * 8)[1];
        const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = (u[i] - y[i] * rsd * m) * rsd;
        *reinterpret_cast<uint4*>(dx + e8 * 8) =
            make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                       pack_bf16x2(o[6], o[7]));
    }
}

// Largest power of two alpha with alpha * bound <= 2^14 (clamped to
// 2^[-120, 120]); 1 when the bound is zero or not finite.  A dS stored as
// alpha * dS in fp16 then never overflows and keeps fp16's full precision.
__device__ __forceinline__ float ds_scale_for(float bound) {
    if (!(bound > 0.f && bound < 3.0e38f)) return 1.f;
    int e = static_cast<int>(floorf(log2f(16384.f / bound)));
    e = max(-120, min(120, e));
    return ldexpf(1.f, e);
}

}  // namespace nc
