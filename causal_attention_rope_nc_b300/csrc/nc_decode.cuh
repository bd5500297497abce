// Single-token decode over a KV cache (memory bound, CUDA cores + TMA).
//
// Cache layout [B][Tcap][Hkv][D]: one cache slot holds all Hkv key/value
// heads of one position contiguously (2*Hkv*D bytes).  Query head h reads
// key/value head h / G (grouped-query attention, G = H / Hkv; G = 1 is plain
// multi-head attention).  Keys are cached normalised and rotated, values raw,
// both in bf16.
//
// Split over the cache: one CTA per (chunk c of CH slots, stream b), grid
// ceil(Tcap / CH) x B; a CTA whose chunk starts at or past the stream's
// length lens[b] exits at once, so the hardware block scheduler hands the
// real chunks to SMs as they free up and every SM streams about the same
// number of bytes whatever the length mix.  The register kernel also splits
// the heads over gridDim.z CTAs (head groups of whole key/value heads) and
// takes its chunk length as an argument, so that a call has enough small
// CTAs (several resident per SM) to keep every SM's loads in flight to the
// end.
//
// Two kernels share this split and the merge below.
//
// attn_decode_kernel (launched for plain multi-head attention, G = 1; it is
// correct for any G, reading key/value head h / G with cached loads when
// G > 1 and writing the key/value heads of its head group into the new slot
// first): warp w of head group z takes heads z HPG + w, z HPG + w + NW, ...
// below (z + 1) HPG.  For one head it walks the chunk's slots BATCH
// at a time: a group of D/8 lanes reads one slot's key row and value
// row (bf16) as 16-byte pieces, 32/(D/8) slots per warp load (streaming
// loads, evict-first).  The batches are software-pipelined over three
// register buffers: every load of batches n+1 and n+2 is issued before the
// arithmetic of batch n, so the rows come straight from HBM into registers
// with two batches in flight per warp (measured on 32 streams, H=10, D=128,
// a 2048-slot cache with lengths uniform in [1, 2048]: 47.1 us
// against 49.2 us with two buffers, 28.7 against 30.7 us with a 512-slot
// window).
//
// attn_decode_tma_kernel (grouped-query attention, G > 1): one producer
// warp streams the chunk through a ring of NST shared-memory stages with
// TMA: stage n holds slots s0 + n*SB ..
// s0 + n*SB + SB - 1, all Hkv heads of each, as one [SB][Hkv][D] box of
// keys and one of values (one tensor-map copy each).  The ring, not the
// register file, holds the bytes in flight, so a CTA keeps NST * SB * Hkv *
// D * 4 bytes in flight (about 80 KB, two CTAs per SM) however few warps do
// the arithmetic, and each cache row leaves HBM once per CTA even when G
// query heads read it.  Compute warp w takes query heads w*HPW .. w*HPW +
// HPW - 1 and walks each stage BATCH slots at a time: a group of D/8 lanes
// reads one slot's key row and value row of the head's key/value head from
// shared memory as 16-byte pieces, 32/(D/8) slots per warp load.  Scores are
// formed in log2 units (qhat carries scale * log2 e); each lane group keeps
// its part of an online softmax state (m shared by the warp, l and o per
// group) that the groups add up at the end of the chunk.  After its last
// read of a stage every compute warp arrives on the stage's empty barrier;
// the producer refills the stage once all have.  (Measured on the decode of
// 32 streams, H=10, D=128, a 2048-slot cache: the ring is 18% faster than the register kernel for groups of 5,
// 4% slower for plain multi-head attention and 29% slower with a 512-slot
// window, hence the split.)
//
// A stream with one chunk writes its output directly.  Otherwise each chunk
// stores (m, l, o) per head in the workspace, and the last CTA of the stream
// to finish (per-stream arrival counter over every chunk and head group)
// merges the chunks of every head and resets the counter for the next call: per head, lanes read the chunks' (m, l) side by
// side, and the weighted partial outputs are added in chunk order
// (deterministic), their loads issued back to back.
//
// With a sliding window W only the last W slots are attended (slot j is
// visible when 0 <= p - j < W); chunks wholly before them exit at once and
// take no part in the merge.
//
// The new token (position p = lens[b] - 1): the CTA that owns the last chunk
// normalises and rotates k_new, writes it (bf16) and v_new into slot p (in
// the ring kernel for every key/value head, followed by a proxy fence so the
// TMA engine sees the writes) and then reads the slot like every other, so
// the score at p uses exactly the stored bf16 key.
#pragma once

#include "nc_common.cuh"
#include "nc_rowops.cuh"

namespace nc {
namespace dec {

constexpr int CH = 128;          // cache slots per CTA of the ring kernel (one partial result)
constexpr int PART_SLOTS = 32;   // the workspace holds ceil(Tcap / PART_SLOTS) >= ceil(Tcap / chunk) partials
constexpr int MAX_WARPS = 10;    // warps per CTA of the register kernel (heads beyond this many loop)
constexpr int MAX_CWARPS = 16;   // compute warps per CTA of the ring kernel
constexpr int BATCH = 8;         // slots per online-softmax step
constexpr int MAX_SB = 64;       // slots per stage, at most
constexpr int STAGE_TARGET = 40 * 1024;  // bytes (keys + values) per stage, about
constexpr int RING_BUDGET = 96 * 1024;   // bytes of the ring when a stage is small enough for two
static_assert(CH % MAX_SB == 0 && CH >= PART_SLOTS, "chunking");

// Slots per stage: a power of two in [BATCH, MAX_SB] near STAGE_TARGET bytes.
inline int stage_slots(int Hkv, int D) {
    int sb = MAX_SB;
    while (sb > BATCH && static_cast<long long>(sb) * Hkv * D * 4 > STAGE_TARGET) sb >>= 1;
    return sb;
}
// Stages in the ring: as many as fit RING_BUDGET, 1 to 4.
inline int ring_stages(int Hkv, int D, int sb) {
    const long long stage = static_cast<long long>(sb) * Hkv * D * 4;
    long long n = RING_BUDGET / stage;
    if (n > 4) n = 4;
    return n < 1 ? 1 : static_cast<int>(n);
}
inline size_t smem_bytes(int Hkv, int D, int sb, int nst) {
    return static_cast<size_t>(nst) * sb * Hkv * D * 4 + 2 * nst * 8;
}
// Launch shape of the register kernel: head groups of whole key/value heads
// of at most REG_WARPS warps, and REG_CH slots per chunk.  (Measured on the
// decode of 32 streams, H=10, D=128: groups of 5 warps, three CTAs per SM, and 64-slot chunks both
// ran within one event tick (2 us) of one 10-warp CTA per 128-slot chunk,
// or slower with a 512-slot window; so heads are split only past 10, the
// most warps whose registers fit one SM with three buffers per warp.)
constexpr int REG_WARPS = MAX_WARPS;
constexpr int REG_CH = 128;
struct RegSplit {
    int hpg;     // query heads per group (a multiple of G)
    int groups;  // head groups: gridDim.z
    int warps;   // warps per CTA
    int ch;      // slots per chunk
};
inline RegSplit reg_split(int H, int G) {
    RegSplit r;
    if (G == 1) {
        r.groups = (H + REG_WARPS - 1) / REG_WARPS;
        r.hpg = (H + r.groups - 1) / r.groups;
    } else {
        r.hpg = G * (REG_WARPS / G > 1 ? REG_WARPS / G : 1);
    }
    r.groups = (H + r.hpg - 1) / r.hpg;  // every group holds at least one head
    r.warps = r.hpg < MAX_WARPS ? r.hpg : MAX_WARPS;
    r.ch = REG_CH;
    return r;
}
static_assert(REG_CH % (2 * BATCH) == 0 && REG_CH >= PART_SLOTS, "register kernel chunking");

// Query heads per compute warp: enough that at most MAX_CWARPS warps cover H.
inline int heads_per_warp(int H) {
    int hpw = 1;
    while (hpw * MAX_CWARPS < H) hpw <<= 1;
    return hpw;
}

template <int D>
struct Lanes {
    static constexpr int LPS = D / 8;        // lanes per slot row (16 bytes each)
    static constexpr int SPW = 32 / LPS;     // slots per warp load
    static constexpr int NLD = BATCH / SPW;  // key (and value) reads per lane per batch
    static_assert(NLD >= 1 && BATCH % SPW == 0, "batch shape");
};

// Make this thread's generic-proxy global writes visible to later
// async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 16-byte streaming load (read once: evict first).  A regular coherent global
// load, so a slot written earlier by the same warp is seen after __syncwarp.
__device__ __forceinline__ uint4 ld_stream16(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }

// The last of the n_arrive CTAs of stream b to finish (per-stream arrival
// counter) merges the partial results of chunks c_lo .. nch - 1 of every head
// into out and resets the counter.  Called by every thread of a CTA that
// stored a partial.
template <int D, int MGRP>
__device__ __forceinline__ void merge_chunks(int b, int c_lo, int nch, int H, int max_parts,
                                             const float* __restrict__ part_o, const float* __restrict__ part_ml,
                                             __nv_bfloat16* __restrict__ out, unsigned int* __restrict__ counters,
                                             int n_arrive, int* s_last) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NW = static_cast<int>(blockDim.x >> 5);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        *s_last = NC_IN_RANGE(counters + b, 4, 0x503) &&
                  atomicAdd(&counters[b], 1u) == static_cast<unsigned>(n_arrive - 1);
    __syncthreads();
    if (!*s_last) return;  // uniform
    __threadfence();
    for (int h = warp; h < H; h += NW) {
        // lane: D/32 consecutive elements of the output.  The (m, l) pairs
        // of the first 32 chunks (one per lane) and the partial outputs of
        // the first MGRP chunks do not depend on one another, so they are
        // loaded together: one L2 round trip for a stream of up to MGRP
        // chunks, one more per further MGRP.  The outputs are added in chunk
        // order (deterministic).
        constexpr int EPL = D / 32;
        const long long pstride = static_cast<long long>(H) * 2;  // between one chunk's (m, l) and the next's
        const float* pmb = part_ml + (static_cast<long long>(b) * max_parts * H + h) * 2;
        const float* pob = part_o + (static_cast<long long>(b) * max_parts * H + h) * D + lane * EPL;
        const int n = nch - c_lo;
        float pre[MGRP][EPL];
        auto load_group = [&](int g0) {
#pragma unroll
            for (int i = 0; i < MGRP; ++i) {
                if (g0 + i < n) {
                    const float* po = pob + static_cast<long long>(c_lo + g0 + i) * H * D;
                    if constexpr (EPL == 4) {
                        const float4 a = __ldcg(reinterpret_cast<const float4*>(po));
                        pre[i][0] = a.x, pre[i][1] = a.y, pre[i][2] = a.z, pre[i][3] = a.w;
                    } else {
                        const float2 a = __ldcg(reinterpret_cast<const float2*>(po));
                        pre[i][0] = a.x, pre[i][1] = a.y;
                    }
                }
            }
        };
        float2 mlv = make_float2(-INFINITY, 0.f);
        if (lane < n) mlv = __ldcg(reinterpret_cast<const float2*>(pmb + (c_lo + lane) * pstride));
        load_group(0);
        float M = mlv.x;
        for (int cc = c_lo + 32 + lane; cc < nch; cc += 32) M = fmaxf(M, __ldcg(pmb + cc * pstride));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float w_own = lane < n ? ex2(mlv.x - M) : 0.f;  // weight of chunk c_lo + lane
        float Ls = lane < n ? mlv.y * w_own : 0.f;
        for (int cc = c_lo + 32 + lane; cc < nch; cc += 32) {
            const float2 a = __ldcg(reinterpret_cast<const float2*>(pmb + cc * pstride));
            Ls = fmaf(a.y, ex2(a.x - M), Ls);
        }
        float o[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = 0.f;
        for (int g0 = 0; g0 < n; g0 += MGRP) {
            if (g0 > 0) load_group(g0);
#pragma unroll
            for (int i = 0; i < MGRP; ++i) {
                const int ci = g0 + i;
                if (ci >= n) break;  // uniform over the warp
                float wi;
                if (ci < 32) {
                    wi = __shfl_sync(0xffffffffu, w_own, ci);
                } else {
                    const float2 a = __ldcg(reinterpret_cast<const float2*>(pmb + (c_lo + ci) * pstride));
                    wi = ex2(a.x - M);
                }
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[e] = fmaf(pre[i][e], wi, o[e]);
            }
        }
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, k);
        const float inv = 1.f / Ls;
        __nv_bfloat16* orow = out + (static_cast<long long>(b) * H + h) * D + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; e += 2)
            if (NC_IN_RANGE(orow + e, 4, 0x501))
                *reinterpret_cast<uint32_t*>(orow + e) = pack_bf16x2(o[e] * inv, o[e + 1] * inv);
    }
    if (threadIdx.x == 0 && NC_IN_RANGE(counters + b, 4, 0x502)) counters[b] = 0u;  // ready for the next call
}

// Partials: o [B][max_parts][H][D] fp32, ml [B][max_parts][H][2] fp32,
// counters [B] u32 (zero between calls).  Grid (ceil(Tcap / ch), B, groups):
// ch slots per chunk (a multiple of 2 BATCH, at least PART_SLOTS), hpg
// query heads per head group (a multiple of G; the last group may be
// smaller, none is empty), at most MAX_WARPS warps.
template <int D>
__global__ void __launch_bounds__(MAX_WARPS * 32, 1) attn_decode_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* kcache, __nv_bfloat16* vcache,
    const int* __restrict__ lens, __nv_bfloat16* __restrict__ out, float* __restrict__ part_o,
    float* __restrict__ part_ml, unsigned int* __restrict__ counters, int B, int H, int Tcap, int max_parts, float eps,
    const __grid_constant__ Theta theta, float scale_log2, int W, int G, int ch, int hpg) {
    using Ln = Lanes<D>;
    constexpr int LPS = Ln::LPS, SPW = Ln::SPW, NLD = Ln::NLD;
    __shared__ float2 s_cs[D / 2];  // rotation at the new token's position
    __shared__ int s_last;
    const int c = blockIdx.x, b = blockIdx.y;
    const int L = lens[b];
    if (L < 1 || L > Tcap) {  // never read outside the cache; the stream's output is left untouched
        if (c == 0 && threadIdx.x == 0) flag_error(2, 0x501);
        return;
    }
    const int nch = (L + ch - 1) / ch;
    const int s_vis = max(0, L - W);  // first visible slot (W >= 2^30: slot 0)
    const int c_lo = s_vis / ch;      // first chunk holding a visible slot
    if (c >= nch || c < c_lo) return;  // uniform over the CTA
    const int n_parts = nch - c_lo;    // chunks that produce a partial
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NW = static_cast<int>(blockDim.x >> 5);
    const int h_lo = static_cast<int>(blockIdx.z) * hpg, h_hi = min(H, h_lo + hpg);  // this CTA's heads
    const int p_new = L - 1;
    const bool own_new = (k_new != nullptr) && (c == nch - 1);
    const int s0 = max(c * ch, s_vis), s1 = min(L, c * ch + ch);
    const int g = lane / LPS;    // slot of this lane group within a warp load
    const int sub = lane % LPS;  // 16-byte piece of the row
    const int e0 = sub * 8;      // first head-dim element of this lane
    const int Hkv = H / G;
    const long long slot_elems = static_cast<long long>(Hkv) * D;
    auto head_base = [&](int h) -> long long {  // query head h -> its key/value head's row in slot 0
        return static_cast<long long>(b) * Tcap * slot_elems + static_cast<long long>(h / G) * D + e0;
    };

    // RoPE(RMSNorm(x)) of row x (D bf16) at the new token's position: the 8
    // elements [e0, e0 + 8) of this lane (every lane group computes the row).
    auto norm_rope8 = [&](const __nv_bfloat16* x, float (&o)[8]) {
        float xv[8], yv[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + e0), xv);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(xv[e], xv[e], ss);
        ss = group_sum<LPS>(ss);
        const float rs = rsqrtf(ss / D + eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] *= rs;
        // pair (i, i + D/2): the partner element sits LPS/2 lanes away
#pragma unroll
        for (int e = 0; e < 8; ++e) yv[e] = __shfl_xor_sync(0xffffffffu, xv[e], LPS / 2);
        const bool lo_half = sub < LPS / 2;
        const int i0 = (sub % (LPS / 2)) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 cs = s_cs[i0 + e];
            o[e] = lo_half ? xv[e] * cs.x - yv[e] * cs.y : yv[e] * cs.y + xv[e] * cs.x;
        }
    };

    auto load_batch = [&](long long base, int j, uint4 (&kr)[NLD], uint4 (&vr)[NLD]) {
#pragma unroll
        for (int u = 0; u < NLD; ++u) {
            const int s = j + g + SPW * u;
            if (s < s1) {
                const long long at = base + static_cast<long long>(s) * slot_elems;
                if (!NC_IN_RANGE_LOAD(kcache + at, 16, 0x504) || !NC_IN_RANGE_LOAD(vcache + at, 16, 0x505)) {
                    kr[u] = make_uint4(0u, 0u, 0u, 0u);
                    vr[u] = kr[u];
                } else if (G == 1) {
                    kr[u] = ld_stream16(kcache + at);
                    vr[u] = ld_stream16(vcache + at);
                } else {
                    kr[u] = __ldcg(reinterpret_cast<const uint4*>(kcache + at));
                    vr[u] = __ldcg(reinterpret_cast<const uint4*>(vcache + at));
                }
            } else {
                kr[u] = make_uint4(0u, 0u, 0u, 0u);
                vr[u] = kr[u];
            }
        }
    };
    // The first batch of this warp's first head goes out before anything
    // else: its loads do not depend on qhat.  (When k_new is given, the
    // chunk that holds the new slot waits for the slot's store below.)
    uint4 ka[NLD], va[NLD], kb[NLD], vb[NLD], kc[NLD], vc[NLD];
    if (!own_new && h_lo + warp < h_hi) {
        load_batch(head_base(h_lo + warp), s0, ka, va);
        if (s0 + BATCH < s1) load_batch(head_base(h_lo + warp), s0 + BATCH, kb, vb);
    }
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) s_cs[i] = rope_cos_sin(p_new, theta.t[i]);
    __syncthreads();
    // RoPE(RMSNorm(k_new)) (bf16) and v_new into slot p, key/value head hk
    auto store_new = [&](int hk) {
        const long long row = (static_cast<long long>(b) * Hkv + hk) * D;
        float kv[8];
        norm_rope8(k_new + row, kv);
        if (g == 0) {
            const long long at = (static_cast<long long>(b) * Tcap + p_new) * slot_elems + static_cast<long long>(hk) * D + e0;
            if (NC_IN_RANGE(kcache + at, 16, 0x506)) *reinterpret_cast<uint4*>(kcache + at) = f32x8_to_bf16(kv);
            if (NC_IN_RANGE(vcache + at, 16, 0x507))
                *reinterpret_cast<uint4*>(vcache + at) = *reinterpret_cast<const uint4*>(v_new + row + e0);
        }
    };
    if (own_new && G > 1) {  // uniform over the CTA
        // the group's key/value heads (no other group reads them)
        for (int hk = h_lo / G + warp; hk < h_hi / G; hk += NW) store_new(hk);
        __syncthreads();  // every head of the slot is stored before any warp reads it
    }

    for (int h = h_lo + warp; h < h_hi; h += NW) {
        const long long row_bh = (static_cast<long long>(b) * H + h) * D;
        float qv[8];
        norm_rope8(q + row_bh, qv);
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] *= scale_log2;
        const long long base = head_base(h);
        if (own_new && G == 1) {
            store_new(h);
            __syncwarp();  // orders the slot's stores before the warp's loads below
        }
        if (own_new || h != h_lo + warp) {
            load_batch(base, s0, ka, va);
            if (s0 + BATCH < s1) load_batch(base, s0 + BATCH, kb, vb);
        }
        float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        auto math_batch = [&](int j, const uint4 (&kr)[NLD], const uint4 (&vr)[NLD]) {
            float sc[NLD];
#pragma unroll
            for (int u = 0; u < NLD; ++u) {
                float kf[8];
                bf16x8_to_f32(kr[u], kf);
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    a0 = fmaf(qv[e], kf[e], a0);
                    a1 = fmaf(qv[e + 1], kf[e + 1], a1);
                }
                sc[u] = a0 + a1;
            }
#pragma unroll
            for (int u = 0; u < NLD; ++u) {
                sc[u] = group_sum<LPS>(sc[u]);
                if (j + g + SPW * u >= s1) sc[u] = -INFINITY;
            }
            // the batch maximum over every lane group: one running max per warp
            float mx = m;
#pragma unroll
            for (int u = 0; u < NLD; ++u) mx = fmaxf(mx, sc[u]);
#pragma unroll
            for (int o = LPS; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float corr = ex2(m - mx);  // slot j is valid: mx is finite
            l *= corr;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= corr;
            m = mx;
#pragma unroll
            for (int u = 0; u < NLD; ++u) {
                const float pe = ex2(sc[u] - mx);
                float vf[8];
                bf16x8_to_f32(vr[u], vf);
                l += pe;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(pe, vf[e], acc[e]);
            }
        };
        // software pipeline over three register buffers: the loads of the
        // next two batches are in flight while the current one is reduced
        for (int j = s0; j < s1; j += 3 * BATCH) {
            if (j + 2 * BATCH < s1) load_batch(base, j + 2 * BATCH, kc, vc);
            math_batch(j, ka, va);
            if (j + BATCH >= s1) break;
            if (j + 3 * BATCH < s1) load_batch(base, j + 3 * BATCH, ka, va);
            math_batch(j + BATCH, kb, vb);
            if (j + 2 * BATCH >= s1) break;
            if (j + 4 * BATCH < s1) load_batch(base, j + 4 * BATCH, kb, vb);
            math_batch(j + 2 * BATCH, kc, vc);
        }
        // add the lane groups' parts (same m)
#pragma unroll
        for (int o = LPS; o < 32; o <<= 1) {
            l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
        }
        if (g == 0) {
            if (n_parts == 1) {
                float o[8];
                const float inv = 1.f / l;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = acc[e] * inv;
                if (NC_IN_RANGE(out + row_bh + e0, 16, 0x50a))
                    *reinterpret_cast<uint4*>(out + row_bh + e0) = f32x8_to_bf16(o);
            } else {
                const long long pi = (static_cast<long long>(b) * max_parts + c) * H + h;
                float4* po = reinterpret_cast<float4*>(part_o + pi * D + e0);
                if (NC_IN_RANGE(po, 32, 0x50b)) {
                    po[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    po[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                }
                if (sub == 0 && NC_IN_RANGE(part_ml + pi * 2, 8, 0x50c))
                    *reinterpret_cast<float2*>(part_ml + pi * 2) = make_float2(m, l);
            }
        }
    }
    if (n_parts == 1) return;  // uniform
    merge_chunks<D, 16>(b, c_lo, nch, H, max_parts, part_o, part_ml, out, counters, n_parts * static_cast<int>(gridDim.z),
                    &s_last);
}

// Partials: o [B][max_parts][H][D] fp32, ml [B][max_parts][H][2] fp32,
// counters [B] u32 (zero between calls).  blockDim = (compute warps + 1) * 32,
// compute warps = ceil(H / HPW) <= MAX_CWARPS; dynamic shared memory
// smem_bytes(Hkv, D, SB, NST).
// Registers.  A block of MAX_CWARPS + 1 = 17 warps puts five on one of the
// four schedulers, whose 16K registers then allow 96 per thread (allocated
// in steps of 8), the cap with several query heads per warp.  One head per
// warp fits 80 without spilling, which lets two CTAs of up to 11 warps
// share an SM (2 x 352 x 80 registers; six warps x 32 x 80 on one
// scheduler) beside their two shared-memory rings.
template <int HPW>
constexpr int decode_tma_maxnreg() {
    return HPW == 1 ? 80 : 16384 / (((MAX_CWARPS + 1 + 3) / 4) * 32) / 8 * 8;
}

template <int D, int HPW>
__global__ void __maxnreg__(decode_tma_maxnreg<HPW>()) attn_decode_tma_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* kcache, __nv_bfloat16* vcache,
    const int* __restrict__ lens, __nv_bfloat16* __restrict__ out, float* __restrict__ part_o,
    float* __restrict__ part_ml, unsigned int* __restrict__ counters, int B, int H, int Hkv, int Tcap, int max_parts,
    float eps,
    const __grid_constant__ Theta theta, float scale_log2, int W, int SB, int NST) {
    using Ln = Lanes<D>;
    constexpr int LPS = Ln::LPS, SPW = Ln::SPW, NLD = Ln::NLD;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float2 s_cs[D / 2];  // rotation at the new token's position
    __shared__ int s_last;
    const int c = blockIdx.x, b = blockIdx.y;
    const int L = lens[b];
    if (L < 1 || L > Tcap) {  // never read outside the cache; the stream's output is left untouched
        if (c == 0 && threadIdx.x == 0) flag_error(2, 0x501);
        return;
    }
    const int nch = (L + CH - 1) / CH;
    const int s_vis = max(0, L - W);  // first visible slot (W >= 2^30: slot 0)
    const int c_lo = s_vis / CH;      // first chunk holding a visible slot
    if (c >= nch || c < c_lo) return;  // uniform over the CTA
    const int n_parts = nch - c_lo;    // chunks that produce a partial
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NW = static_cast<int>(blockDim.x >> 5);
    const int nwc = NW - 1;  // compute warps; the last warp is the producer
    const int G = H / Hkv;
    const int p_new = L - 1;
    const bool own_new = (k_new != nullptr) && (c == nch - 1);
    const int s0 = max(c * CH, s_vis), s1 = min(L, c * CH + CH);
    const int n_st = (s1 - s0 + SB - 1) / SB;  // stages this chunk streams
    const int g = lane / LPS;    // slot of this lane group within a warp load
    const int sub = lane % LPS;  // 16-byte piece of the row
    const int e0 = sub * 8;      // first head-dim element of this lane
    const long long slot_elems = static_cast<long long>(Hkv) * D;
    const uint32_t stage_bytes = static_cast<uint32_t>(SB) * Hkv * D * 2;  // keys (or values) of one stage
    uint8_t* kst = smem;
    uint8_t* vst = smem + static_cast<size_t>(NST) * stage_bytes;
    const uint32_t bar0 = smem_u32(smem + static_cast<size_t>(2) * NST * stage_bytes);
    auto full_bar = [&](int st) -> uint32_t { return bar0 + 8 * st; };
    auto empty_bar = [&](int st) -> uint32_t { return bar0 + 8 * (NST + st); };

    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(full_bar(i), 1);
            mbar_init(empty_bar(i), nwc);
        }
        fence_mbar_init();
    }
    for (int i = threadIdx.x; i < D / 2; i += blockDim.x) s_cs[i] = rope_cos_sin(p_new, theta.t[i]);
    __syncthreads();

    // RoPE(RMSNorm(x)) of row x (D bf16) at the new token's position: the 8
    // elements [e0, e0 + 8) of this lane (every lane group computes the row).
    auto norm_rope8 = [&](const __nv_bfloat16* x, float (&o)[8]) {
        float xv[8], yv[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + e0), xv);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(xv[e], xv[e], ss);
        ss = group_sum<LPS>(ss);
        const float rs = rsqrtf(ss / D + eps);
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] *= rs;
        // pair (i, i + D/2): the partner element sits LPS/2 lanes away
#pragma unroll
        for (int e = 0; e < 8; ++e) yv[e] = __shfl_xor_sync(0xffffffffu, xv[e], LPS / 2);
        const bool lo_half = sub < LPS / 2;
        const int i0 = (sub % (LPS / 2)) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float2 cs = s_cs[i0 + e];
            o[e] = lo_half ? xv[e] * cs.x - yv[e] * cs.y : yv[e] * cs.y + xv[e] * cs.x;
        }
    };
    // RoPE(RMSNorm(k_new)) (bf16) and v_new into slot p of every key/value
    // head, before the producer's first copy
    if (own_new) {  // uniform over the CTA
        for (int hk = warp; hk < Hkv; hk += NW) {
            const long long row = (static_cast<long long>(b) * Hkv + hk) * D;
            float kv[8];
            norm_rope8(k_new + row, kv);
            if (g == 0) {
                const long long at = (static_cast<long long>(b) * Tcap + p_new) * slot_elems +
                                     static_cast<long long>(hk) * D + e0;
                if (NC_IN_RANGE(kcache + at, 16, 0x508)) *reinterpret_cast<uint4*>(kcache + at) = f32x8_to_bf16(kv);
                if (NC_IN_RANGE(vcache + at, 16, 0x509))
                    *reinterpret_cast<uint4*>(vcache + at) = *reinterpret_cast<const uint4*>(v_new + row + e0);
            }
        }
        fence_proxy_async_global();
        __syncthreads();
    }

    if (warp == nwc) {
        // ------------------------------------------------------- producer --
        if (lane == 0) {
            fence_proxy_async_global();
            int issued = 0;
            for (int n = 0; n < n_st; ++n) {
                const int st = n % NST;
                if (n >= NST && !mbar_wait(empty_bar(st), ((n / NST) - 1) & 1, 0x511)) break;
                mbar_expect_tx(full_bar(st), 2 * stage_bytes);
                tma_load_4d(smem_u32(kst + static_cast<size_t>(st) * stage_bytes), &tm_k, 0, 0, s0 + n * SB, b,
                            full_bar(st));
                tma_load_4d(smem_u32(vst + static_cast<size_t>(st) * stage_bytes), &tm_v, 0, 0, s0 + n * SB, b,
                            full_bar(st));
                ++issued;
            }
            // never leave the CTA with a copy still in flight
            for (int n = max(0, issued - NST); n < issued; ++n) mbar_wait(full_bar(n % NST), (n / NST) & 1, 0x512);
        }
    } else {
        // --------------------------------------------------- compute warps --
        const int h0 = warp * HPW;  // first query head of this warp
        float qv[HPW][8], m[HPW], l[HPW], acc[HPW][8];
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
            m[i] = -INFINITY;
            l[i] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
            if (h0 + i < H) {  // uniform over the warp
                norm_rope8(q + (static_cast<long long>(b) * H + h0 + i) * D, qv[i]);
#pragma unroll
                for (int e = 0; e < 8; ++e) qv[i][e] *= scale_log2;
            }
        }
        for (int n = 0; n < n_st; ++n) {
            const int st = n % NST;
            if (!mbar_wait_warp(full_bar(st), (n / NST) & 1, 0x513)) break;
            const uint8_t* ks = kst + static_cast<size_t>(st) * stage_bytes;
            const uint8_t* vs = vst + static_cast<size_t>(st) * stage_bytes;
            const int sb0 = s0 + n * SB;  // cache slot of the stage's first row
            for (int j = 0; j < SB && sb0 + j < s1; j += BATCH) {
#pragma unroll
                for (int i = 0; i < HPW; ++i) {
                    if (h0 + i >= H) break;  // uniform over the warp
                    const int hk = (h0 + i) / G;
                    uint4 kr[NLD], vr[NLD];
#pragma unroll
                    for (int u = 0; u < NLD; ++u) {
                        const int r = j + g + SPW * u;  // row of the stage (< SB)
                        const size_t at = (static_cast<size_t>(r) * Hkv + hk) * (D * 2) + e0 * 2;
                        kr[u] = *reinterpret_cast<const uint4*>(ks + at);
                        vr[u] = *reinterpret_cast<const uint4*>(vs + at);
                        if (sb0 + r >= s1) {  // past the chunk: whatever the cache holds there, read zeros
                            kr[u] = make_uint4(0u, 0u, 0u, 0u);
                            vr[u] = kr[u];
                        }
                    }
                    float sc[NLD];
#pragma unroll
                    for (int u = 0; u < NLD; ++u) {
                        float kf[8];
                        bf16x8_to_f32(kr[u], kf);
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            a0 = fmaf(qv[i][e], kf[e], a0);
                            a1 = fmaf(qv[i][e + 1], kf[e + 1], a1);
                        }
                        sc[u] = a0 + a1;
                    }
#pragma unroll
                    for (int u = 0; u < NLD; ++u) {
                        sc[u] = group_sum<LPS>(sc[u]);
                        if (sb0 + j + g + SPW * u >= s1) sc[u] = -INFINITY;
                    }
                    // the batch maximum over every lane group: one running max per warp
                    float mx = m[i];
#pragma unroll
                    for (int u = 0; u < NLD; ++u) mx = fmaxf(mx, sc[u]);
#pragma unroll
                    for (int o = LPS; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                    const float corr = ex2(m[i] - mx);  // slot sb0 + j is valid: mx is finite
                    l[i] *= corr;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[i][e] *= corr;
                    m[i] = mx;
#pragma unroll
                    for (int u = 0; u < NLD; ++u) {
                        const float pe = ex2(sc[u] - mx);
                        float vf[8];
                        bf16x8_to_f32(vr[u], vf);
                        l[i] += pe;
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pe, vf[e], acc[i][e]);
                    }
                }
            }
            mbar_arrive_warp(empty_bar(st));  // this warp is done with the stage
        }
#pragma unroll
        for (int i = 0; i < HPW; ++i) {
            const int h = h0 + i;
            if (h >= H) break;  // uniform over the warp
            // add the lane groups' parts (same m)
#pragma unroll
            for (int o = LPS; o < 32; o <<= 1) {
                l[i] += __shfl_xor_sync(0xffffffffu, l[i], o);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][e] += __shfl_xor_sync(0xffffffffu, acc[i][e], o);
            }
            if (g == 0) {
                if (n_parts == 1) {
                    float o[8];
                    const float inv = 1.f / l[i];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = acc[i][e] * inv;
                    __nv_bfloat16* op = out + (static_cast<long long>(b) * H + h) * D + e0;
                    if (NC_IN_RANGE(op, 16, 0x50d)) *reinterpret_cast<uint4*>(op) = f32x8_to_bf16(o);
                } else {
                    const long long pi = (static_cast<long long>(b) * max_parts + c) * H + h;
                    float4* po = reinterpret_cast<float4*>(part_o + pi * D + e0);
                    if (NC_IN_RANGE(po, 32, 0x50e)) {
                        po[0] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
                        po[1] = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
                    }
                    if (sub == 0 && NC_IN_RANGE(part_ml + pi * 2, 8, 0x50f))
                        *reinterpret_cast<float2*>(part_ml + pi * 2) = make_float2(m[i], l[i]);
                }
            }
        }
    }
    if (n_parts == 1) return;  // uniform
    // (8 partial outputs at a time: the ring kernel runs at 96 registers)
    merge_chunks<D, 8>(b, c_lo, nch, H, max_parts, part_o, part_ml, out, counters, n_parts, &s_last);
}

}  // namespace dec
}  // namespace nc
