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

// dx for row `row` of a 128-row tile whose raw x rows (bf16, D/64 spans)
// and RoPE table rows (fp32 (cos, sin) pairs, D/32 spans) were staged in
// shared memory by TMA with 128-byte swizzling, g = out_scale * (the D fp32
// columns of this thread's TMEM lane at `tm`), read twice (once for <u, y>,
// once for the output).  dx == nullptr: no store (rows past the sequence end
// still take part, tcgen05.ld being warp-collective).
template <int D>
__device__ __forceinline__ void norm_rope_bwd_tile_row(uint32_t tm, float out_scale, const uint8_t* xt,
                                                       const uint8_t* ct, int row, float eps,
                                                       __nv_bfloat16* __restrict__ dx) {
    constexpr int HALF = D / 2;
    // 8 bf16 of x starting at element e (e % 8 == 0); 4 fp32 of the table at f (f % 4 == 0)
    auto xchunk = [&](int e) -> uint4 {
        return *reinterpret_cast<const uint4*>(xt + (e >> 6) * (128 * 128) + sw128_offset(row, (e & 63) >> 3));
    };
    auto cchunk = [&](int f) -> float4 {
        return *reinterpret_cast<const float4*>(ct + (f >> 5) * (128 * 128) + sw128_offset(row, (f & 31) >> 2));
    };
    float ss = 0.f;
#pragma unroll
    for (int g = 0; g < D / 8; ++g) {
        float y[8];
        bf16x8_to_f32(xchunk(g * 8), y);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(y[i], y[i], ss);
    }
    const float rsd = rsqrtf(ss / D + eps);
    float dot = 0.f;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const float m = dot / D;
#pragma unroll 2
        for (int ch = 0; ch < HALF / 8; ++ch) {
            uint32_t glo[8], ghi[8];
            tmem_ld8(tm + ch * 8, glo);
            tmem_ld8(tm + HALF + ch * 8, ghi);
            float ylo[8], yhi[8];
            bf16x8_to_f32(xchunk(ch * 8), ylo);
            bf16x8_to_f32(xchunk(HALF + ch * 8), yhi);
            float4 c4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) c4[i] = cchunk(16 * ch + 4 * i);
            tmem_wait_ld();
            float olo[8], ohi[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float c = (e & 1) ? c4[e >> 1].z : c4[e >> 1].x;
                const float sn = (e & 1) ? c4[e >> 1].w : c4[e >> 1].y;
                const float a = __uint_as_float(glo[e]) * out_scale;
                const float bb = __uint_as_float(ghi[e]) * out_scale;
                // R^T: (a, b) -> (a c + b s, -a s + b c)
                const float ulo = a * c + bb * sn;
                const float uhi = -a * sn + bb * c;
                const float yl = ylo[e] * rsd, yh = yhi[e] * rsd;
                if (pass == 0) {
                    dot = fmaf(ulo, yl, fmaf(uhi, yh, dot));
                } else {
                    olo[e] = (ulo - yl * m) * rsd;
                    ohi[e] = (uhi - yh * m) * rsd;
                }
            }
            if (pass == 1 && dx != nullptr) {
                *reinterpret_cast<uint4*>(dx + ch * 8) =
                    make_uint4(pack_bf16x2(olo[0], olo[1]), pack_bf16x2(olo[2], olo[3]), pack_bf16x2(olo[4], olo[5]),
                               pack_bf16x2(olo[6], olo[7]));
                *reinterpret_cast<uint4*>(dx + HALF + ch * 8) =
                    make_uint4(pack_bf16x2(ohi[0], ohi[1]), pack_bf16x2(ohi[2], ohi[3]), pack_bf16x2(ohi[4], ohi[5]),
                               pack_bf16x2(ohi[6], ohi[7]));
            }
        }
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
