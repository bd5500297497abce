// Single-token decode over a bf16 KV cache (memory bound, CUDA cores).
//
// Cache layout [B][Tcap][H][D]: one cache slot holds all H heads of one
// position contiguously (2*H*D bytes).  Keys are cached normalised and
// rotated, in IEEE fp16 (elements bounded by sqrt(D)); values raw, in bf16.  The grid is (chunks of CHUNK slots,
// B); a CTA reads its chunk of K and V for every head once, with 16-byte
// loads that sweep whole slots, so the traffic is the algorithmic
// sum_b lens[b] * H * D * 2 bytes for each of K and V.
//
// Thread (x, y): x < H*D/8 owns 8 head-dim values of head x / (D/8); the
// D/8 lanes of one head form an aligned shuffle group.  y splits the chunk's
// slots.  Each thread runs an online softmax (running max in log2 units, so
// nothing is assumed about what the cache holds), then the y-slices merge
// in shared memory.  A stream whose length fits one chunk writes its output
// directly; otherwise every CTA stores a partial (m, l, o) and the last CTA
// of the stream (per-stream arrival counter) merges them and resets the
// counter to zero for the next call.
#pragma once

#include "nc_common.cuh"
#include "nc_rowops.cuh"

namespace nc {
namespace dec {

constexpr int CHUNK = 64;  // cache slots per CTA
constexpr int MAX_THREADS = 512;     // per CTA: H*D/8 lanes (rounded to warps) x slot slices
constexpr int MAX_SMEM = 96 * 1024;  // dynamic shared memory opt-in

template <int D>
struct Shape {
    static constexpr int LPR = D / 8;
    static int xthreads(int H) { return ((H * LPR + 31) / 32) * 32; }
    // slot-parallel slices: 2 while they fit in MAX_THREADS, else 1 (0 = too many heads)
    static int slices(int H) { return 2 * xthreads(H) <= MAX_THREADS ? 2 : (xthreads(H) <= MAX_THREADS ? 1 : 0); }
};

// Partials: o [B][nch][H][D] fp32, ml [B][nch][H][2] fp32, counters [B] u32.
template <int D>
__global__ void __launch_bounds__(MAX_THREADS) attn_decode_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __half* kcache, __nv_bfloat16* vcache,
    const int* __restrict__ lens, __nv_bfloat16* __restrict__ out, float* __restrict__ part_o,
    float* __restrict__ part_ml, unsigned int* __restrict__ counters, int H, int Tcap, int nch, float eps,
    double log2_base, float scale_log2) {
    constexpr int LPR = D / 8, HALF = LPR / 2;
    extern __shared__ float dsm[];
    float* qh = dsm;                                         // [H][D] scaled qhat
    float2* cs = reinterpret_cast<float2*>(qh + H * D);      // [D/2] rotation at position p
    float* red = reinterpret_cast<float*>(cs + D / 2);       // [KS][XT][10] merge area
    __shared__ int s_last;

    const int b = blockIdx.y, ch = blockIdx.x;
    const int L = lens[b];
    if (L < 1 || L > Tcap) {  // host validates lens when it can; never read out of the cache
        if (threadIdx.x == 0 && threadIdx.y == 0 && ch == 0) flag_error(2, 0x501);
        return;
    }
    const int nchunks = (L + CHUNK - 1) / CHUNK;
    if (ch >= nchunks) return;
    const int p = L - 1;  // position of the new token
    const int j0 = ch * CHUNK, j1 = min(L, j0 + CHUNK);
    const int XT = blockDim.x, KS = blockDim.y;
    const int tid = threadIdx.y * XT + threadIdx.x;
    const int nthr = XT * blockDim.y;

    for (int i = tid; i < D / 2; i += nthr) cs[i] = rope_cos_sin(p, rope_theta(i, D, log2_base));
    __syncthreads();

    // qhat (and, for the chunk holding slot p, the new key) = RoPE(RMSNorm(x))
    const bool own_new = (k_new != nullptr) && (j0 <= p) && (p < j1);
    const int nrows = own_new ? 2 * H : H;
    const int warp = tid >> 5, nwarps = nthr >> 5, lane = tid & 31;
    const int groups_per_warp = 32 / LPR;
    for (int base = warp * groups_per_warp; base < nrows; base += nwarps * groups_per_warp) {
        const int row = base + lane / LPR;
        const int sub = lane % LPR;
        const bool valid = row < nrows;
        const bool is_k = row >= H;
        const int hh = valid ? (is_k ? row - H : row) : 0;
        float x[8];
        if (valid) {
            const __nv_bfloat16* src = (is_k ? k_new : q) + (static_cast<long long>(b) * H + hh) * D + sub * 8;
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(src), x);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = 0.f;
        }
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
        ss = group_sum<LPR>(ss);
        const float rs = rsqrtf(ss / D + eps);
        float y[8], o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] *= rs;
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], HALF);
        const bool lo = sub < HALF;
        const int i0 = (sub % HALF) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 c = cs[i0 + e];
            o[e] = lo ? x[e] * c.x - y[e] * c.y : y[e] * c.y + x[e] * c.x;
        }
        if (valid) {
            if (!is_k) {
#pragma unroll
                for (int e = 0; e < 8; ++e) qh[hh * D + sub * 8 + e] = o[e] * scale_log2;
            } else {
                const long long slot = ((static_cast<long long>(b) * Tcap + p) * H + hh) * D + sub * 8;
                *reinterpret_cast<uint4*>(kcache + slot) = f32x8_to_f16(o);
                *reinterpret_cast<uint4*>(vcache + slot) = *reinterpret_cast<const uint4*>(
                    v_new + (static_cast<long long>(b) * H + hh) * D + sub * 8);
            }
        }
    }
    __syncthreads();  // qhat in smem; the new slot's global writes visible to the block

    // ---- online softmax over this chunk's slots ----
    const int x = threadIdx.x, y = threadIdx.y;
    const bool active = x < H * LPR;
    const int h = active ? x / LPR : 0, ds = x % LPR;
    float qr[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) qr[e] = active ? qh[h * D + ds * 8 + e] : 0.f;
    float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const long long slot_stride = static_cast<long long>(H) * D;
    const __half* kp = kcache + (static_cast<long long>(b) * Tcap) * slot_stride + h * D + ds * 8;
    const __nv_bfloat16* vp = vcache + (static_cast<long long>(b) * Tcap) * slot_stride + h * D + ds * 8;
    constexpr int U = 4;  // slots in flight per thread
    for (int j = j0 + y; j < j1; j += KS * U) {
        uint4 kv[U], vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = j + u * KS;
            if (active && jj < j1) {
                kv[u] = *reinterpret_cast<const uint4*>(kp + jj * slot_stride);
                vv[u] = *reinterpret_cast<const uint4*>(vp + jj * slot_stride);
            } else {
                kv[u] = make_uint4(0, 0, 0, 0);
                vv[u] = make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jj = j + u * KS;
            float kf[8];
            f16x8_to_f32(kv[u], kf);
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) s = fmaf(qr[e], kf[e], s);
            s = group_sum<LPR>(s);  // score in log2 units
            if (jj < j1 && active) {
                const float mn = fmaxf(m, s);
                const float corr = ex2(m - mn);
                const float pe = ex2(s - mn);
                float vf[8];
                bf16x8_to_f32(vv[u], vf);
                l = fmaf(l, corr, pe);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(acc[e], corr, pe * vf[e]);
                m = mn;
            }
        }
    }

    // ---- merge the KS slices ----
    float* my = red + (static_cast<long long>(y) * XT + x) * 10;
    my[0] = m;
    my[1] = l;
#pragma unroll
    for (int e = 0; e < 8; ++e) my[2 + e] = acc[e];
    __syncthreads();
    if (y == 0 && active) {
        for (int yy = 1; yy < KS; ++yy) {
            const float* o2 = red + (static_cast<long long>(yy) * XT + x) * 10;
            const float m2 = o2[0];
            if (m2 == -INFINITY) continue;
            const float mn = fmaxf(m, m2);
            const float c1 = ex2(m - mn), c2 = ex2(m2 - mn);
            l = l * c1 + o2[1] * c2;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = acc[e] * c1 + o2[2 + e] * c2;
            m = mn;
        }
    }
    __nv_bfloat16* orow = out + (static_cast<long long>(b) * H + h) * D + ds * 8;
    if (nchunks == 1) {
        if (y == 0 && active) {
            float o[8];
            const float inv = 1.f / l;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = acc[e] * inv;
            *reinterpret_cast<uint4*>(orow) = f32x8_to_bf16(o);
        }
        return;
    }
    if (y == 0 && active) {
        float* po = part_o + ((static_cast<long long>(b) * nch + ch) * H + h) * D + ds * 8;
        reinterpret_cast<float4*>(po)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(po)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if (ds == 0) {
            float* pm = part_ml + ((static_cast<long long>(b) * nch + ch) * H + h) * 2;
            pm[0] = m;
            pm[1] = l;
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&counters[b], 1u) == static_cast<unsigned>(nchunks - 1));
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (y == 0 && active) {
        float M = -INFINITY;
        for (int c = 0; c < nchunks; ++c)
            M = fmaxf(M, __ldcg(part_ml + ((static_cast<long long>(b) * nch + c) * H + h) * 2));
        float Ls = 0.f, o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = 0.f;
        for (int c = 0; c < nchunks; ++c) {
            const float* pm = part_ml + ((static_cast<long long>(b) * nch + c) * H + h) * 2;
            const float w = ex2(__ldcg(pm) - M);
            Ls = fmaf(__ldcg(pm + 1), w, Ls);
            const float4* po =
                reinterpret_cast<const float4*>(part_o + ((static_cast<long long>(b) * nch + c) * H + h) * D + ds * 8);
            const float4 a0 = __ldcg(po), a1 = __ldcg(po + 1);
            o[0] = fmaf(a0.x, w, o[0]); o[1] = fmaf(a0.y, w, o[1]);
            o[2] = fmaf(a0.z, w, o[2]); o[3] = fmaf(a0.w, w, o[3]);
            o[4] = fmaf(a1.x, w, o[4]); o[5] = fmaf(a1.y, w, o[5]);
            o[6] = fmaf(a1.z, w, o[6]); o[7] = fmaf(a1.w, w, o[7]);
        }
        const float inv = 1.f / Ls;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= inv;
        *reinterpret_cast<uint4*>(orow) = f32x8_to_bf16(o);
    }
    if (tid == 0) counters[b] = 0u;  // ready for the next call
}

}  // namespace dec
}  // namespace nc
