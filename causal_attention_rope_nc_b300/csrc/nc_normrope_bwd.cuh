// Backward of the QK RMSNorm + RoPE prologue for one head vector, fused into
// the epilogues of the backward kernels (two threads per token's head vector).
//
// Given the gradient g with respect to xhat = RoPE(x / r, p) (r =
// sqrt(mean(x^2) + eps)), the gradient with respect to the raw x is
//   u  = R(p)^T g                       (rotate every pair (i, i + D/2) by -angle)
//   dx = (u - y <u, y> / D) / r,        y = x / r.
#pragma once

#include "nc_common.cuh"

namespace nc {

// dx for one 128-row tile, two threads per row: thread `half` takes the
// rotation pairs (f, f + D/2) for f in [half D/4, (half + 1) D/4).
//   g   = out_scale * (the D fp32 columns of TMEM lane `row` at `tm`)
//   u   = R(p)^T g
//   dx  = u rsd - x rsd^3 <u, x> / D,   rsd = 1 / sqrt(mean(x^2) + eps)
// (the same as (u - y <u, y> / D) rsd with y = x rsd).  The raw x rows (bf16,
// layout of tile16_off) and the RoPE table rows (fp32 (cos, sin) pairs as
// D/32 boxes of 32 values x 128 rows, 128-byte swizzled; boxes [0, D/64) at
// ct0, the rest at ct1) were staged by TMA.  The two halves of a row swap
// their partial sums of x^2 and <u, x> through xch (2 x 128 float2) across
// named barrier `bar_id` over `nthreads` threads, which every participating
// thread reaches exactly once whether or not it is `active`.  The bf16 dx
// goes into `stage` (layout of tile16_off).
// With GTAB the table is read from global memory (L2) instead: ct0 is then
// the row's own D floats of the [T][D/2] (cos, sin) table and ct1 is unused.
template <int D, bool GTAB = false>
__device__ __forceinline__ void norm_rope_bwd_stage(bool active, uint32_t tm, float out_scale, const uint8_t* xt,
                                                    const uint8_t* ct0, const uint8_t* ct1, int row, int half,
                                                    float eps, float2* xch, uint8_t* stage, int bar_id,
                                                    int nthreads) {
    constexpr int HALF = D / 2, NF = D / 4;
    const int f0 = half * NF;
    const uint8_t* ct = half ? ct1 : ct0;  // this half's table floats [2 f0, 2 f0 + 2 NF)
    const float* gt = reinterpret_cast<const float*>(ct0) + 2 * f0;
    uint32_t u[2][NF];                     // g, then u, for the lo and hi columns
    float ss = 0.f, dot = 0.f;
    if (active) {
        tmem_ld_cols<NF>(tm + f0, u[0]);
        tmem_ld_cols<NF>(tm + HALF + f0, u[1]);
        tmem_wait_ld();
#pragma unroll
        for (int ch = 0; ch < NF / 8; ++ch) {
            const int e0 = f0 + ch * 8;
            float xl[8], xh[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(xt + tile16_off(row, e0)), xl);
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(xt + tile16_off(row, HALF + e0)), xh);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int f = 16 * ch + 4 * i;  // table float index relative to this half
                const float4 cs =
                    GTAB ? __ldg(reinterpret_cast<const float4*>(gt + f))
                         : *reinterpret_cast<const float4*>(ct + (f >> 5) * (128 * 128) + sw128_offset(row, (f & 31) >> 2));
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = ch * 8 + 2 * i + k;
                    const float c = k ? cs.z : cs.x, sn = k ? cs.w : cs.y;
                    const float a = __uint_as_float(u[0][e]) * out_scale;
                    const float bb = __uint_as_float(u[1][e]) * out_scale;
                    // R^T: (a, b) -> (a c + b s, b c - a s)
                    const float ul = fmaf(a, c, bb * sn), uh = fmaf(bb, c, -a * sn);
                    u[0][e] = __float_as_uint(ul);
                    u[1][e] = __float_as_uint(uh);
                    const float x0 = xl[2 * i + k], x1 = xh[2 * i + k];
                    ss = fmaf(x0, x0, fmaf(x1, x1, ss));
                    dot = fmaf(ul, x0, fmaf(uh, x1, dot));
                }
            }
        }
        xch[half * 128 + row] = make_float2(ss, dot);
    }
    named_bar_sync(bar_id, nthreads);
    if (active) {
        const float2 o = xch[(half ^ 1) * 128 + row];
        ss += o.x;
        dot += o.y;
        const float rsd = rsqrtf(ss / D + eps);
        const float kx = rsd * rsd * rsd * dot / D;
#pragma unroll
        for (int ch = 0; ch < NF / 8; ++ch) {
            const int e0 = f0 + ch * 8;
#pragma unroll
            for (int side = 0; side < 2; ++side) {
                const uint32_t off = tile16_off(row, side * HALF + e0);
                float x[8], o8[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(xt + off), x);
#pragma unroll
                for (int e = 0; e < 8; ++e) o8[e] = fmaf(__uint_as_float(u[side][ch * 8 + e]), rsd, -x[e] * kx);
                *reinterpret_cast<uint4*>(stage + off) = f32x8_to_bf16(o8);
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

// The backward's one dS scale for the whole call, from the row-norm maxima
// the preprocess publishes (gmax[0] = max ||dout_i||, gmax[1] = max ||v_j||):
//   |dS_ij| = P_ij |<dout_i, v_j> - <dout_i, out_i>| <= 2 max ||dout|| max ||v||
// (out_i is a convex combination of the v_j, so ||out_i|| <= max ||v||), with
// a 1/16 margin for the rounding of the factors.  Both backward kernels use
// it: the key side stores alpha * dS, the query side sums those blocks.
__device__ __forceinline__ float ds_scale_global(const unsigned int* gmax) {
    return ds_scale_for(2.f * __uint_as_float(gmax[0]) * __uint_as_float(gmax[1]) * 1.0625f);
}

}  // namespace nc
