// Memory-bound per-row kernels of the attention path.
//
// Every kernel here treats a head vector of D bf16 values as one "row" and
// gives it D/8 consecutive lanes (16 bytes per lane), so a warp streams
// whole 256-byte rows with 16-byte loads and the per-row reductions are
// lane shuffles.  The rotate-half RoPE partner of element i (i + D/2) is
// held by the lane D/16 positions away, one xor-shuffle from it.
#pragma once

#include <cuda_fp8.h>

#include "nc_common.cuh"

namespace nc {

// Eight floats times `scale` -> one store of eight OutT values: 16 bytes
// for bf16 or IEEE fp16 (scale 1), 8 bytes for E4M3 (round to nearest even,
// saturating).
template <typename OutT>
__device__ __forceinline__ void store8(OutT* dst, const float (&o)[8], float scale) {
    if constexpr (std::is_same<OutT, __nv_fp8_e4m3>::value) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            w[i] = static_cast<uint32_t>(
                __nv_cvt_float2_to_fp8x2(make_float2(o[2 * i] * scale, o[2 * i + 1] * scale), __NV_SATFINITE, __NV_E4M3));
        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
    } else {
        *reinterpret_cast<uint4*>(dst) = f32x8_to<OutT>(o);
    }
}

template <int D>
struct RowLanes {
    static constexpr int LPR = D / 8;        // lanes per row
    static constexpr int HALF = LPR / 2;     // lane distance to the RoPE partner
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
};

// Sum over the LPR lanes of a row group (groups are aligned, so the xor
// partners never leave the group).
template <int LPR>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------------ RoPE table --
// tab[t][i] = (cos, sin) of angle pos[t] * theta_i, t < T, i < D/2, with
// theta_i = base^(-2i/D) formed on the host in double precision (the same
// values every kernel of the library uses).  pos == nullptr means pos[t] = t.
__global__ void rope_table_kernel(float2* __restrict__ tab, const int* __restrict__ pos, int T, int D,
                                  const __grid_constant__ Theta theta) {
    const int half = D / 2;
    const long long n = static_cast<long long>(T) * half;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < n;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(e / half), i = static_cast<int>(e % half);
        const int p = pos ? pos[t] : t;
        if (NC_IN_RANGE(tab + e, sizeof(float2), 0x401)) tab[e] = rope_cos_sin(p, theta.t[i]);
    }
}

// ------------------------------------------------- QK RMSNorm + RoPE (K1) --
// qhat = RoPE(q / sqrt(mean(q^2) + eps)), same for k (k may be null: one
// tensor only), stored as OutT: IEEE fp16 for the forward/backward operands
// (the norm bounds every element by sqrt(D) <= 11.4, well inside fp16's
// range, and fp16's 3 extra mantissa bits keep the score products within the
// forward's error bound), bf16 for a key cache.  rstd (optional) receives 1/r,
// laid out [2][B][T][H] (q then k).  (With fewer key/value heads than query
// heads the host runs one launch per tensor, each with its own head count
// and its own part of rstd.)
//
// One group of D/16 lanes owns one token (b, t) of one tensor: lane j holds
// the 8 rotation pairs (i, i + D/2) for i in [8j, 8j + 8), i.e. 16 bytes of
// each half of a head row, so the rotation needs no data from another lane
// and only the row's sum of squares crosses lanes.  The group reads the
// token's rotation row from the table once and walks the token's H heads,
// NORM_HC heads at a time with every load of a chunk issued before any
// math.  Tokens are enumerated q tokens first, then k tokens.  (B=32,
// T=2048, H=10, D=128: the earlier layout, 16 lanes per token with the
// partner half fetched by 8 shuffles per head, ran with its issue slots 57 %
// busy; HC = 4 there took 135 us, 8 took 140 us, 16 took 196 us.)
constexpr int NORM_HC = 2;

template <int D, typename OutT>
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const __nv_bfloat16* __restrict__ q,
                                                           const __nv_bfloat16* __restrict__ k,
                                                           const float2* __restrict__ tab,
                                                           OutT* __restrict__ qhat,
                                                           OutT* __restrict__ khat,
                                                           float* __restrict__ rstd, long long tokens_per_tensor,
                                                           int T, int H, float eps, float out_scale = 1.f) {
    static_assert(D == 64 || D == 128, "head dim must be 64 or 128");
    constexpr int LPR = D / 16;  // lanes per token
    constexpr int HALF = D / 2;
    const int sub = threadIdx.x % LPR;
    const long long groups = blockDim.x / LPR;
    const long long ntok = (k ? 2 : 1) * tokens_per_tensor;
    const long long first = blockIdx.x * groups + threadIdx.x / LPR;
    const long long stride = static_cast<long long>(gridDim.x) * groups;
    // every lane of a warp runs the same number of iterations (shuffles)
    const long long warp_first = blockIdx.x * groups + (threadIdx.x & ~31) / LPR;
    const int i0 = sub * 8;  // this lane's pairs: columns [i0, i0 + 8) and [HALF + i0, HALF + i0 + 8)
    for (long long base = warp_first, tok = first; base < ntok; base += stride, tok += stride) {
        const bool valid = tok < ntok;
        const bool is_k = valid && tok >= tokens_per_tensor;
        const long long r = valid ? (is_k ? tok - tokens_per_tensor : tok) : 0;  // b*T + t
        const int t = static_cast<int>(r % T);
        float c[8], sn[8];
        {
            const float4* cs4 = reinterpret_cast<const float4*>(tab + static_cast<long long>(t) * (D / 2) + i0);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                const float4 v = valid ? cs4[e2] : make_float4(1.f, 0.f, 1.f, 0.f);
                c[2 * e2] = v.x, sn[2 * e2] = v.y, c[2 * e2 + 1] = v.z, sn[2 * e2 + 1] = v.w;
            }
        }
        const __nv_bfloat16* src = (is_k ? k : q) + r * H * D + i0;
        OutT* dst = (is_k ? khat : qhat) + r * H * D + i0;
        for (int h0 = 0; h0 < H; h0 += NORM_HC) {
            uint4 ul[NORM_HC], uh[NORM_HC];
#pragma unroll
            for (int j = 0; j < NORM_HC; ++j) {
                const bool in = valid && h0 + j < H;
                ul[j] = in ? *reinterpret_cast<const uint4*>(src + (h0 + j) * D) : make_uint4(0, 0, 0, 0);
                uh[j] = in ? *reinterpret_cast<const uint4*>(src + (h0 + j) * D + HALF) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < NORM_HC; ++j) {
                if (h0 + j >= H) break;  // uniform: H is the same for every lane
                float a[8], b[8];
                bf16x8_to_f32(ul[j], a);
                bf16x8_to_f32(uh[j], b);
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(a[e], a[e], ss);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(b[e], b[e], ss);
                ss = group_sum<LPR>(ss);
                const float rs = rsqrtf(ss / D + eps);
                float lo[8], hi[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    a[e] *= rs;
                    b[e] *= rs;
                }
                // (a, b) = (x_i, x_{i + D/2}) rotated by the pair's angle
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    lo[e] = a[e] * c[e] - b[e] * sn[e];
                    hi[e] = a[e] * sn[e] + b[e] * c[e];
                }
                if (valid) {
                    OutT* d = dst + (h0 + j) * D;
                    if (NC_IN_RANGE(d, 8 * sizeof(OutT), 0x402)) store8<OutT>(d, lo, out_scale);
                    if (NC_IN_RANGE(d + HALF, 8 * sizeof(OutT), 0x4f1)) store8<OutT>(d + HALF, hi, out_scale);
                    float* rp = rstd + ((is_k ? tokens_per_tensor : 0) + r) * H + h0 + j;
                    if (rstd && sub == 0 && NC_IN_RANGE(rp, 4, 0x403)) *rp = rs;
                }
            }
        }
    }
}

// --------------------------------------------- chunk prefill prologue ----
// For the C new tokens of stream b (positions start[b] + t, t < C):
//   qhat[b][t][h] = RoPE(RMSNorm(q[b][t][h]), start[b] + t)    (bf16, workspace; h < H)
//   kcache[b][start[b] + t][g] = RoPE(RMSNorm(k[b][t][g]), start[b] + t)  (bf16; g < Hkv)
//   vcache[b][start[b] + t][g] = v[b][t][g]                     (bf16 copy)
// One group of D/8 lanes owns one token of one stream: it forms the token's
// rotation (cos, sin of its 8 pair indices) from the frequencies and walks
// the token's H query heads and Hkv key/value heads.  A stream whose chunk does not fit its cache
// (start < 0 or start + C > Tcap) is skipped and recorded (status 2).
template <int D>
__global__ void __launch_bounds__(256) prefill_norm_rope_kernel(const __nv_bfloat16* __restrict__ q,
                                                                const __nv_bfloat16* __restrict__ k,
                                                                const __nv_bfloat16* __restrict__ v,
                                                                const int* __restrict__ start,
                                                                __nv_bfloat16* __restrict__ qhat,
                                                                __nv_bfloat16* kcache,
                                                                __nv_bfloat16* vcache, int B, int C, int H, int Hkv,
                                                                int Tcap, float eps,
                                                                const __grid_constant__ Theta theta) {
    using L = RowLanes<D>;
    const int sub = threadIdx.x % L::LPR;
    const long long groups = blockDim.x / L::LPR;
    const long long ntok = static_cast<long long>(B) * C;
    const long long first = blockIdx.x * groups + threadIdx.x / L::LPR;
    const long long stride = static_cast<long long>(gridDim.x) * groups;
    const long long warp_first = blockIdx.x * groups + (threadIdx.x & ~31) / L::LPR;
    const int i0 = (sub % L::HALF) * 8;
    const bool lo = sub < L::HALF;
    // every lane of a warp runs the same number of iterations (shuffles)
    for (long long base = warp_first, tok = first; base < ntok; base += stride, tok += stride) {
        bool valid = tok < ntok;
        const int b = valid ? static_cast<int>(tok / C) : 0;
        const int t = valid ? static_cast<int>(tok % C) : 0;
        const int s0 = valid ? start[b] : 0;
        if (valid && (s0 < 0 || s0 + C > Tcap)) {
            if (t == 0 && sub == 0) flag_error(2, 0x601);
            valid = false;
        }
        const int p = s0 + t;
        float c[8], sn[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 r = valid ? rope_cos_sin(p, theta.t[i0 + e]) : make_float2(1.f, 0.f);
            c[e] = r.x;
            sn[e] = r.y;
        }
        const long long tok_q = (static_cast<long long>(b) * C + t) * H * D + sub * 8;
        const long long tok_kv = (static_cast<long long>(b) * C + t) * Hkv * D + sub * 8;
        const long long slot = (static_cast<long long>(b) * Tcap + p) * Hkv * D + sub * 8;
        for (int h = 0; h < H; ++h) {
#pragma unroll
            for (int which = 0; which < 2; ++which) {  // q, then k (key/value heads: the first Hkv)
                if (which && h >= Hkv) break;  // uniform
                float x[8];
                if (valid)
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(which ? k + tok_kv + h * D : q + tok_q + h * D), x);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = 0.f;
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
                ss = group_sum<L::LPR>(ss);
                const float rs = rsqrtf(ss / D + eps);
                float y[8], o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] *= rs;
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], L::HALF);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = lo ? x[e] * c[e] - y[e] * sn[e] : y[e] * sn[e] + x[e] * c[e];
                if (valid) {
                    __nv_bfloat16* dst = which ? kcache + slot + h * D : qhat + tok_q + h * D;
                    if (NC_IN_RANGE(dst, 16, 0x404)) *reinterpret_cast<uint4*>(dst) = f32x8_to_bf16(o);
                }
            }
            if (valid && h < Hkv && NC_IN_RANGE(vcache + slot + h * D, 16, 0x405))
                *reinterpret_cast<uint4*>(vcache + slot + h * D) =
                    *reinterpret_cast<const uint4*>(v + tok_kv + h * D);
        }
    }
}

// -------------------------------------------------- backward preprocess ----
// delta[b][h][t] = <dout_t, out_t> (fp32), lse2[b][h][t] = lse * log2(e),
// both padded to Tpad columns (delta 0, lse2 +inf beyond T so that padded
// query rows get probability 0).  gmax[0] and gmax[1] receive the largest row
// norms ||dout_t|| and ||v_t|| over the whole tensors (they must be zero on
// entry): the backward's dS scale (ds_scale_global) is formed from them.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ out,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const __nv_bfloat16* __restrict__ v,
                                                      const float* __restrict__ lse, float* __restrict__ delta,
                                                      float* __restrict__ lse2, unsigned int* __restrict__ gmax,
                                                      int B, int T, int H, int Hkv, int Tpad) {
    using L = RowLanes<D>;
    constexpr int RB = 4;  // consecutive positions of one (b, h) per group and iteration
    __shared__ float s_max[2][32];
    const int sub = threadIdx.x % L::LPR;
    const long long groups = blockDim.x / L::LPR;
    const int tb = (T + RB - 1) / RB;  // position blocks per (b, h)
    const long long nblk = static_cast<long long>(B) * H * tb;
    const long long stride = static_cast<long long>(gridDim.x) * groups;
    const long long warp_first = blockIdx.x * groups + (threadIdx.x & ~31) / L::LPR;
    const long long first = blockIdx.x * groups + threadIdx.x / L::LPR;
    float mx_do = 0.f, mx_v = 0.f;  // squared norms
    // every lane of a warp runs the same iterations (the group sums shuffle)
    for (long long base = warp_first, k = first; base < nblk; base += stride, k += stride) {
        const bool valid = k < nblk;
        const long long bh = valid ? k / tb : 0;
        const int t0 = valid ? static_cast<int>(k % tb) * RB : 0;
        const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
        // every load of the block first
        uint4 ua[RB], ug[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            if (valid && t0 + i < T) {
                const long long r = (static_cast<long long>(b) * T + t0 + i) * H + h;
                ua[i] = *reinterpret_cast<const uint4*>(out + r * D + sub * 8);
                ug[i] = *reinterpret_cast<const uint4*>(dout + r * D + sub * 8);
            } else {
                ua[i] = make_uint4(0u, 0u, 0u, 0u);
                ug[i] = ua[i];
            }
        }
        float acc[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            float a[8], g[8];
            bf16x8_to_f32(ua[i], a);
            bf16x8_to_f32(ug[i], g);
            float d = 0.f, sdo = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                d = fmaf(a[e], g[e], d);
                sdo = fmaf(g[e], g[e], sdo);
            }
            acc[i] = group_sum<L::LPR>(d);
            mx_do = fmaxf(mx_do, group_sum<L::LPR>(sdo));
        }
        if (valid && sub == 0) {
            // delta and lse2 live in the workspace: o = bh * Tpad + t0 is a
            // multiple of 4 (Tpad a multiple of 128), so 16-byte stores are
            // aligned; lse is the caller's (4-byte aligned only): scalar loads
            const long long o = bh * Tpad + t0;
            float l2[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i)
                l2[i] = t0 + i < T ? lse[bh * T + t0 + i] * 1.4426950408889634f : 0.f;
            if (t0 + RB <= T) {
                if (NC_IN_RANGE(delta + o, 16, 0x406))
                    *reinterpret_cast<float4*>(delta + o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                if (NC_IN_RANGE(lse2 + o, 16, 0x407))
                    *reinterpret_cast<float4*>(lse2 + o) = make_float4(l2[0], l2[1], l2[2], l2[3]);
            } else {
#pragma unroll
                for (int i = 0; i < RB; ++i) {
                    if (t0 + i < T && NC_IN_RANGE(delta + o + i, 4, 0x408) && NC_IN_RANGE(lse2 + o + i, 4, 0x409)) {
                        delta[o + i] = acc[i];
                        lse2[o + i] = l2[i];
                    }
                }
            }
        }
    }
    // v rows ([B][T][Hkv] of them), RB consecutive rows per group and iteration
    const long long nv = static_cast<long long>(B) * T * Hkv;
    const long long nvb = (nv + RB - 1) / RB;
    for (long long base = warp_first, k = first; base < nvb; base += stride, k += stride) {
        uint4 u[RB];
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            const long long r = k * RB + i;
            u[i] = (k < nvb && r < nv) ? *reinterpret_cast<const uint4*>(v + r * D + sub * 8)
                                       : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int i = 0; i < RB; ++i) {
            float a[8];
            bf16x8_to_f32(u[i], a);
            float sv = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) sv = fmaf(a[e], a[e], sv);
            mx_v = fmaxf(mx_v, group_sum<L::LPR>(sv));
        }
    }
    // block maxima of the row norms, one atomic each per block (non-negative
    // floats order like their bit patterns)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx_do = fmaxf(mx_do, __shfl_xor_sync(0xffffffffu, mx_do, o));
        mx_v = fmaxf(mx_v, __shfl_xor_sync(0xffffffffu, mx_v, o));
    }
    const int wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        s_max[0][wid] = mx_do;
        s_max[1][wid] = mx_v;
    }
    __syncthreads();
    if (threadIdx.x < 2) {
        float m = 0.f;
        for (int w = 0; w < nw; ++w) m = fmaxf(m, s_max[threadIdx.x][w]);
        if (NC_IN_RANGE(gmax + threadIdx.x, 4, 0x40a)) atomicMax(gmax + threadIdx.x, __float_as_uint(sqrtf(m)));
    }
    // padding columns t in [T, Tpad)
    const int padw = Tpad - T;
    const long long npad = static_cast<long long>(B) * H * padw;
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < npad;
         e += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long bh = e / padw;
        const long long o = bh * Tpad + T + (e % padw);
        if (!NC_IN_RANGE(delta + o, 4, 0x40b) || !NC_IN_RANGE(lse2 + o, 4, 0x40c)) continue;
        delta[o] = 0.f;
        lse2[o] = __int_as_float(0x7f800000);  // +inf
    }
}

// ------------------------------------------------ FP8 value quantisation --
// vmax[bg] = max |v[b][t][g][d]| over t, d for bg = b * Hkv + g, as float
// bits (zero on entry; non-negative floats order like their bits).  Grid
// (token chunks of 256, B * Hkv); one group of D/8 lanes per token.
template <int D>
__global__ void __launch_bounds__(256) v_absmax_kernel(const __nv_bfloat16* __restrict__ v,
                                                       unsigned int* __restrict__ vmax, int T, int Hkv) {
    using L = RowLanes<D>;
    __shared__ float s_max[8];
    const int sub = threadIdx.x % L::LPR;
    const int bg = blockIdx.y, b = bg / Hkv, g = bg % Hkv;
    const int t_end = min(T, static_cast<int>(blockIdx.x) * 256 + 256);
    float a = 0.f;
    for (int t = blockIdx.x * 256 + threadIdx.x / L::LPR; t < t_end; t += blockDim.x / L::LPR) {
        float x[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(v + ((static_cast<long long>(b) * T + t) * Hkv + g) * D + sub * 8),
                      x);
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(x[e]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        float m = 0.f;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, s_max[w]);
        if (NC_IN_RANGE(vmax + bg, 4, 0x40d)) atomicMax(vmax + bg, __float_as_uint(m));
    }
}

// The exponent tau of one head's value scale: the largest integer with
// max 2^tau <= 448 (E4M3's largest finite value), clamped to [-126, 126] so
// that 2^-tau is a normal fp32 number; 0 for an all-zero head.
__device__ __forceinline__ int v_scale_exp(float mxf) {
    const double mx = mxf;
    if (!(mx > 0.0)) return 0;
    int tau = static_cast<int>(floor(log2(448.0 / mx)));
    while (ldexp(mx, tau) > 448.0) --tau;
    while (ldexp(mx, tau + 1) <= 448.0) ++tau;
    return max(-126, min(126, tau));
}

// v8t[bg][d][t] = E4M3(v[b][t][g][d] 2^tau) for t < Tpad (0 past T): the
// values transposed, keys contiguous, so that the fp8 forward's PV product
// reads a K-major B operand.  vscale[bg] = 2^-tau.  Grid (Tpad / 128,
// B * Hkv), 256 threads; each block transposes 128 tokens through a bf16
// shared tile [128 tokens][D] whose 16-byte chunks are XOR-swizzled by bits
// 4-6 of the token (chunk c of token t sits at chunk c ^ ((t >> 4) & 7)):
// the row loads store whole chunks, and in the column pass the eight lanes
// that read the same element of tokens 16 k + j (k = 0..7) hit eight
// different chunks, so neither pass has bank conflicts.  Each column-pass
// thread quantises 16 consecutive tokens of one d into one 16-byte store; a
// warp stores four whole 128-byte rows.
template <int D>
__global__ void __launch_bounds__(256) v_quant_t_kernel(const __nv_bfloat16* __restrict__ v,
                                                        const unsigned int* __restrict__ vmax,
                                                        uint8_t* __restrict__ v8t, float* __restrict__ vscale, int T,
                                                        int Tpad, int Hkv) {
    using L = RowLanes<D>;
    constexpr int ROW = D * 2;  // bytes per token row of the tile
    __shared__ __align__(16) uint8_t tile[128 * ROW];
    __shared__ int s_tau;
    const int sub = threadIdx.x % L::LPR;
    const int bg = blockIdx.y, b = bg / Hkv, g = bg % Hkv;
    const int t0 = blockIdx.x * 128;
    if (threadIdx.x == 0) {
        s_tau = v_scale_exp(__uint_as_float(vmax[bg]));
        if (blockIdx.x == 0 && NC_IN_RANGE(vscale + bg, 4, 0x40e)) vscale[bg] = ldexpf(1.f, -s_tau);
    }
    // row pass: token rows in, 16 bytes a lane
    for (int tl = threadIdx.x / L::LPR; tl < 128; tl += blockDim.x / L::LPR) {
        const int t = t0 + tl;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (t < T) x = *reinterpret_cast<const uint4*>(v + ((static_cast<long long>(b) * T + t) * Hkv + g) * D + sub * 8);
        *reinterpret_cast<uint4*>(tile + tl * ROW + ((sub ^ ((tl >> 4) & 7)) << 4)) = x;
    }
    __syncthreads();
    const float sc = __int_as_float((s_tau + 127) << 23);  // 2^tau, tau in [-126, 126]
    // column pass: item = (d, k): tokens 16 k .. 16 k + 15 of element d
    uint8_t* dst = v8t + static_cast<long long>(bg) * D * Tpad + t0;
    for (int it = threadIdx.x; it < D * 8; it += blockDim.x) {
        const int k = it & 7, d = it >> 3;
        const int cpos = ((d >> 3) ^ k) << 4, w = (d & 7) * 2;
        uint32_t word[4];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
            float x[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                x[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(tile + (16 * k + j + i) * ROW + cpos + w)) * sc;
            word[j / 4] = static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x[0], x[1]), __NV_SATFINITE, __NV_E4M3)) |
                          (static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(x[2], x[3]), __NV_SATFINITE, __NV_E4M3)) << 16);
        }
        uint8_t* p = dst + static_cast<long long>(d) * Tpad + 16 * k;
        if (NC_IN_RANGE(p, 16, 0x40f)) *reinterpret_cast<uint4*>(p) = make_uint4(word[0], word[1], word[2], word[3]);
    }
}

}  // namespace nc
