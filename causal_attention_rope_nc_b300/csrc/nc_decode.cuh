// Single-token decode over a KV cache (memory bound, CUDA cores).
//
// Cache layout [B][Tcap][H][D]: one cache slot holds all H heads of one
// position contiguously (2*H*D bytes).  Keys are cached normalised and
// rotated, in IEEE fp16 (elements bounded by sqrt(D)); values raw, in bf16.
//
// Work: stream b's valid slots 0..L_b-1 are cut into items of ITEM slots.  A
// persistent grid of one CTA per SM takes a contiguous, equal share of all
// items (the item index -> (stream, item) map comes from a block-wide scan of
// the lengths), so the HBM traffic is spread evenly whatever the length mix;
// each run of one stream's items inside a CTA yields one partial result
// (m, l, o) per head.
//
// Inside a CTA one producer thread streams each item's K and V rows with
// bulk asynchronous copies (cp.async.bulk: the slots of one item are
// contiguous) into a STAGES-deep shared-memory ring of `sps` slots per stage,
// running ahead of the consumers by up to STAGES stages.  Consumer thread
// (x, y): x < H*D/8 owns 8 head-dim values of head x / (D/8) (the D/8 lanes of
// one head form an aligned shuffle group); y splits a stage's slots.  Each
// runs an online softmax (running max in log2 units, so nothing is assumed
// about what the cache holds); the y-slices merge in shared memory at the end
// of a run.  A stream handled by a single CTA writes its output directly;
// otherwise each run's partial goes to the workspace and the last CTA to
// finish one of the stream's runs (per-stream arrival counter) merges them in
// one pass and resets the counter to zero for the next call.
#pragma once

#include "nc_common.cuh"
#include "nc_rowops.cuh"

namespace nc {
namespace dec {

constexpr int ITEM = 32;                // cache slots per partial result
constexpr int STAGES = 4;               // depth of the K/V ring
constexpr int STAGE_BYTES = 40 * 1024;  // K + V bytes per stage (at most)
constexpr int MAX_CONSUMERS = 512;      // H*D/8 lanes (rounded to warps) x slot slices
constexpr int MAX_SLICES = 4;
constexpr int MAX_SPT = 8;              // slots a consumer takes per stage, at most
constexpr int SCAN_CHUNK = 256;         // lengths scanned per round
constexpr int MAX_SMEM = 232448;        // dynamic shared memory opt-in (227 KB)

template <int D>
struct Shape {
    static constexpr int LPR = D / 8;
    __host__ __device__ static int xthreads(int H) { return ((H * LPR + 31) / 32) * 32; }
    // slot-parallel slices: 2 while they fit, else 1 (0 = too many heads)
    // slot-parallel slices: as many as fit in MAX_CONSUMERS threads, at most
    // MAX_SLICES (0 = too many heads for one CTA)
    __host__ __device__ static int slices(int H) {
        const int k = MAX_CONSUMERS / xthreads(H);
        return k > MAX_SLICES ? MAX_SLICES : k;
    }
    // cache slots per ring stage (K and V of one slot: H*D*4 bytes)
    __host__ __device__ static int sps(int H) {
        const int s = STAGE_BYTES / (H * D * 4);
        return s < 1 ? 1 : (s > ITEM ? ITEM : s);
    }
};

// Shared memory: ring | barriers | q̂ | new k̂ | RoPE row | slice merge | scan
struct Layout {
    int ring, bars, qh, kn, cs, red, scan, bytes;
};
__host__ __device__ inline Layout layout(int H, int D, int sps, int xt, int ks) {
    Layout L;
    const int stage = sps * H * D * 4;
    L.ring = 0;
    L.bars = L.ring + STAGES * stage;
    L.qh = L.bars + 2 * STAGES * 8 + 64;          // full/empty barriers, scan scalars
    L.kn = L.qh + H * D * 4;
    L.cs = L.kn + H * D * 4;
    L.red = L.cs + (D / 2) * 8;
    L.scan = L.red + ks * xt * 10 * 4;
    L.bytes = L.scan + (SCAN_CHUNK + 32) * 4;
    return L;
}

__device__ __forceinline__ int items_of(int L) { return (L + ITEM - 1) / ITEM; }

// Partials: o [B][max_items][H][D] fp32, ml [B][max_items][H][2] fp32,
// counters [B] u32 (zero between calls).
template <int D>
__global__ void __launch_bounds__(MAX_CONSUMERS + 32) attn_decode_kernel(
    const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_new,
    const __nv_bfloat16* __restrict__ v_new, __half* kcache, __nv_bfloat16* vcache, const int* __restrict__ lens,
    __nv_bfloat16* __restrict__ out, float* __restrict__ part_o, float* __restrict__ part_ml,
    unsigned int* __restrict__ counters, int B, int H, int Tcap, int max_items, int sps, float eps,
    double log2_base, float scale_log2) {
    constexpr int LPR = D / 8, HALF = LPR / 2;
    const int XT = Shape<D>::xthreads(H), KS = Shape<D>::slices(H);
    const int NCONS = XT * KS;  // consumer threads; thread NCONS is the producer
    const Layout LY = layout(H, D, sps, XT, KS);
    extern __shared__ __align__(128) uint8_t dsm[];
    const uint32_t sbase = smem_u32(dsm);
    const int tid = threadIdx.x;
    const int stage_bytes = sps * H * D * 4;
    const long long slot_elems = static_cast<long long>(H) * D;
    auto full_bar = [&](int s) -> uint32_t { return sbase + LY.bars + 8 * s; };
    auto empty_bar = [&](int s) -> uint32_t { return sbase + LY.bars + 8 * (STAGES + s); };
    int* scan = reinterpret_cast<int*>(dsm + LY.scan);
    int* scal = reinterpret_cast<int*>(dsm + LY.bars + 2 * STAGES * 8);  // [0] total, [1] b0, [2] i0

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), NCONS / 32);  // one arrival per consumer warp
        }
        fence_mbar_init();
    }
    // ---- this CTA's share of the items: a block-wide scan of the lengths ----
    // pass 1: total number of items
    {
        int local = 0;
        for (int b = tid; b < B; b += blockDim.x) {
            const int L = lens[b];
            if (L >= 1 && L <= Tcap) local += items_of(L);
            else if (blockIdx.x == 0) flag_error(2, 0x501);  // never read outside the cache
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) local += __shfl_xor_sync(0xffffffffu, local, o);
        if (tid == 0) {
            scal[0] = 0;
            scal[1] = -1;
            scal[2] = 0;
        }
        __syncthreads();
        if ((tid & 31) == 0) atomicAdd(&scal[0], local);
        __syncthreads();
    }
    const int total = scal[0];
    const int lo = static_cast<int>((static_cast<long long>(total) * blockIdx.x) / gridDim.x);
    const int hi = static_cast<int>((static_cast<long long>(total) * (blockIdx.x + 1)) / gridDim.x);
    if (lo >= hi) return;  // uniform: nothing for this CTA
    // pass 2: the stream holding item `lo`
    {
        int running = 0;
        for (int base = 0; base < B; base += SCAN_CHUNK) {
            const int cnt = min(SCAN_CHUNK, B - base);
            for (int t = tid; t < cnt; t += blockDim.x) {  // blocks may be smaller than a chunk
                const int L = lens[base + t];
                scan[t] = (L >= 1 && L <= Tcap) ? items_of(L) : 0;
            }
            __syncthreads();
            if (tid == 0) {  // serial scan of the chunk's valid entries
                int acc = running;
                for (int i = 0; i < cnt; ++i) {
                    const int n = scan[i];
                    if (acc <= lo && lo < acc + n) {
                        scal[1] = base + i;
                        scal[2] = lo - acc;
                    }
                    acc += n;
                }
                scan[SCAN_CHUNK] = acc;
            }
            __syncthreads();
            running = scan[SCAN_CHUNK];
            __syncthreads();
            if (running > lo) break;
        }
    }
    const int b_first = scal[1], i_first = scal[2];
    const int n_my = hi - lo;
    if (b_first < 0 || b_first >= B) {  // cannot happen when the scan found `lo`; never index past lens
        if (tid == 0) flag_error(2, 0x502);
        return;
    }

    if (tid == NCONS) {
        // ------------------------------------------------------ producer ----
        int b = b_first, i = i_first, L = lens[b];
        int issued = 0;
        bool ok = true;
        for (int w = 0; ok && w < n_my; ++w) {
            const int s0 = i * ITEM, s1 = min(L, s0 + ITEM);
            for (int j = s0; j < s1; j += sps) {
                const int n = min(sps, s1 - j);
                const int st = issued % STAGES;
                if (issued >= STAGES && !mbar_wait(empty_bar(st), ((issued / STAGES) - 1) & 1, 0x511)) {
                    ok = false;
                    break;
                }
                const uint32_t bytes = static_cast<uint32_t>(n * slot_elems * 2);
                const uint32_t dst = sbase + LY.ring + st * stage_bytes;
                const long long off = (static_cast<long long>(b) * Tcap + j) * slot_elems;
                mbar_expect_tx(full_bar(st), 2 * bytes);
                bulk_load(dst, kcache + off, bytes, full_bar(st));
                bulk_load(dst + stage_bytes / 2, vcache + off, bytes, full_bar(st));
                ++issued;
            }
            if (++i >= items_of(L) && w + 1 < n_my) {
                ++b;
                while (b < B && !(lens[b] >= 1 && lens[b] <= Tcap)) ++b;  // invalid streams hold no items
                i = 0;
                L = b < B ? lens[b] : 1;
            }
        }
        // never leave the CTA with a bulk copy still in flight
        for (int k = (issued > STAGES ? issued - STAGES : 0); k < issued; ++k)
            mbar_wait(full_bar(k % STAGES), (k / STAGES) & 1, 0x512);
        return;
    }
    if (tid > NCONS) return;

    // --------------------------------------------------------- consumers ----
    // A CTA's items form at most a few segments (runs of one stream's items);
    // the online softmax state carries across a segment, which yields one
    // partial result, stored at the stream-local index of the segment's first
    // item.  Item I starts a segment when it is its stream's first item or the
    // first item of the CTA that owns it (cta_of: the last CTA whose range
    // starts at or before I), so any CTA can enumerate a stream's segments.
    float* qh = reinterpret_cast<float*>(dsm + LY.qh);   // [H][D] scaled qhat
    float* kn = reinterpret_cast<float*>(dsm + LY.kn);   // [H][D] new khat (fp16-rounded)
    float2* cs = reinterpret_cast<float2*>(dsm + LY.cs); // [D/2] rotation at position p
    float* red = reinterpret_cast<float*>(dsm + LY.red); // [KS][XT][10] merge area
    const int x = tid % XT, y = tid / XT;
    const bool active = x < H * LPR;
    const int h = active ? x / LPR : 0, ds = x % LPR;
    const int cwarp = tid >> 5, clane = tid & 31, ncwarps = NCONS >> 5;
    const long long G = gridDim.x;
    auto cta_of = [&](int I) -> int { return static_cast<int>(((static_cast<long long>(I) + 1) * G - 1) / total); };
    auto range_lo = [&](int g) -> int { return static_cast<int>((static_cast<long long>(total) * g) / G); };
    auto starts = [&](int I, int first) -> bool { return I == first || range_lo(cta_of(I)) == I; };
    int b = b_first, i = i_first, L = lens[b];
    int pb = lo - i_first;  // global index of stream b's first item
    int consumed = 0;
    bool ok = true, seg_start = true, own_new = false;
    int i_seg = 0;  // stream-local index of the segment's first item
    float qr[8], m = -INFINITY, l = 0.f, acc[8];
    for (int w = 0; w < n_my; ++w) {
        const int n_items = items_of(L);
        const int p = L - 1;  // position of the new token
        if (seg_start) {
            // this segment holds the stream's last item (the new token's slot)?
            own_new = (k_new != nullptr) && (pb + n_items - 1 < hi);
            // qhat (and the new key) = RoPE(RMSNorm(x)) at position p
            for (int e = tid; e < D / 2; e += NCONS) cs[e] = rope_cos_sin(p, rope_theta(e, D, log2_base));
            named_bar_sync(1, NCONS);
            const int nrows = own_new ? 2 * H : H;
            const int groups_per_warp = 32 / LPR;
            for (int base = cwarp * groups_per_warp; base < nrows; base += ncwarps * groups_per_warp) {
                const int row = base + clane / LPR;
                const int sub = clane % LPR;
                const bool valid = row < nrows;
                const bool is_k = row >= H;
                const int hh = valid ? (is_k ? row - H : row) : 0;
                float xv[8];
                if (valid) {
                    const __nv_bfloat16* src = (is_k ? k_new : q) + (static_cast<long long>(b) * H + hh) * D + sub * 8;
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(src), xv);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) xv[e] = 0.f;
                }
                float ss = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = fmaf(xv[e], xv[e], ss);
                ss = group_sum<LPR>(ss);
                const float rs = rsqrtf(ss / D + eps);
                float yv[8], o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[e] *= rs;
#pragma unroll
                for (int e = 0; e < 8; ++e) yv[e] = __shfl_xor_sync(0xffffffffu, xv[e], HALF);
                const bool lo_half = sub < HALF;
                const int i0 = (sub % HALF) * 8;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float2 c = cs[i0 + e];
                    o[e] = lo_half ? xv[e] * c.x - yv[e] * c.y : yv[e] * c.y + xv[e] * c.x;
                }
                if (valid) {
                    if (!is_k) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) qh[hh * D + sub * 8 + e] = o[e] * scale_log2;
                    } else {
                        const uint4 packed = f32x8_to_f16(o);
                        float r[8];
                        f16x8_to_f32(packed, r);  // what the cache holds
#pragma unroll
                        for (int e = 0; e < 8; ++e) kn[hh * D + sub * 8 + e] = r[e];
                        const long long slot = ((static_cast<long long>(b) * Tcap + p) * H + hh) * D + sub * 8;
                        *reinterpret_cast<uint4*>(kcache + slot) = packed;
                        *reinterpret_cast<uint4*>(vcache + slot) = *reinterpret_cast<const uint4*>(
                            v_new + (static_cast<long long>(b) * H + hh) * D + sub * 8);
                    }
                }
            }
            named_bar_sync(1, NCONS);  // qhat, new khat in smem
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                qr[e] = active ? qh[h * D + ds * 8 + e] : 0.f;
                acc[e] = 0.f;
            }
            m = -INFINITY;
            l = 0.f;
            i_seg = i;
            seg_start = false;
        }

        // ---- online softmax over this item's slots ----
        const int s0 = i * ITEM, s1 = min(L, s0 + ITEM);
        for (int j = s0; j < s1; j += sps) {
            const int n = min(sps, s1 - j);
            const int st = consumed % STAGES;
            if (ok && !mbar_wait_warp(full_bar(st), (consumed / STAGES) & 1, 0x521)) ok = false;
            const uint8_t* kst = dsm + LY.ring + st * stage_bytes;
            const uint8_t* vst = kst + stage_bytes / 2;
            // scores of this thread's slots first (independent chains), then one
            // rescale of the running state with the stage maximum
            float sc[MAX_SPT];
            int cnt = 0;
#pragma unroll
            for (int u = 0; u < MAX_SPT; ++u) {
                const int s = y + u * KS;
                sc[u] = -INFINITY;
                if (!ok || s >= n) continue;
                cnt = u + 1;
                float kf[8];
                if (own_new && j + s == p) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) kf[e] = active ? kn[h * D + ds * 8 + e] : 0.f;
                } else {
                    const long long e0 = static_cast<long long>(s) * slot_elems + h * D + ds * 8;
                    f16x8_to_f32(*reinterpret_cast<const uint4*>(kst + e0 * 2), kf);
                }
                float a = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) a = fmaf(qr[e], kf[e], a);
                sc[u] = a;
            }
#pragma unroll
            for (int u = 0; u < MAX_SPT; ++u)
                if (u < cnt) sc[u] = group_sum<LPR>(sc[u]);  // scores in log2 units
            if (active && cnt > 0) {
                float mx = m;
#pragma unroll
                for (int u = 0; u < MAX_SPT; ++u)
                    if (u < cnt) mx = fmaxf(mx, sc[u]);
                const float corr = ex2(m - mx);
                l *= corr;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] *= corr;
                m = mx;
#pragma unroll
                for (int u = 0; u < MAX_SPT; ++u) {
                    if (u >= cnt) continue;
                    const int s = y + u * KS;
                    float vf[8];
                    if (own_new && j + s == p) {
                        bf16x8_to_f32(
                            *reinterpret_cast<const uint4*>(v_new + (static_cast<long long>(b) * H + h) * D + ds * 8),
                            vf);
                    } else {
                        const long long e0 = static_cast<long long>(s) * slot_elems + h * D + ds * 8;
                        bf16x8_to_f32(*reinterpret_cast<const uint4*>(vst + e0 * 2), vf);
                    }
                    const float pe = ex2(sc[u] - mx);
                    l += pe;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(pe, vf[e], acc[e]);
                }
            }
            mbar_arrive_warp(empty_bar(st));
            ++consumed;
        }

        const bool seg_end = (w == n_my - 1) || (i == n_items - 1);
        if (seg_end) {
            // ---- merge the KS slices ----
            float* my = red + (static_cast<long long>(y) * XT + x) * 10;
            my[0] = m;
            my[1] = l;
#pragma unroll
            for (int e = 0; e < 8; ++e) my[2 + e] = acc[e];
            named_bar_sync(1, NCONS);
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
            int n_seg = 0;  // segments of this stream, over all CTAs
            for (int c = 0; c < n_items; ++c) n_seg += starts(pb + c, pb) ? 1 : 0;
            const int k = i_seg;  // this segment's partial index
            __nv_bfloat16* orow = out + (static_cast<long long>(b) * H + h) * D + ds * 8;
            if (n_seg == 1) {
                if (y == 0 && active && ok) {
                    float o[8];
                    const float inv = 1.f / l;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = acc[e] * inv;
                    *reinterpret_cast<uint4*>(orow) = f32x8_to_bf16(o);
                }
            } else {
                if (y == 0 && active) {
                    float* po = part_o + ((static_cast<long long>(b) * max_items + k) * H + h) * D + ds * 8;
                    reinterpret_cast<float4*>(po)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    reinterpret_cast<float4*>(po)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                    if (ds == 0) {
                        float* pm = part_ml + ((static_cast<long long>(b) * max_items + k) * H + h) * 2;
                        pm[0] = m;
                        pm[1] = l;
                    }
                }
                __threadfence();
                named_bar_sync(1, NCONS);
                int* last = scal + 3;
                if (tid == 0) *last = (atomicAdd(&counters[b], 1u) == static_cast<unsigned>(n_seg - 1));
                named_bar_sync(1, NCONS);
                if (*last) {
                    __threadfence();
                    if (y == 0 && active) {
                        // one pass over the stream's partials with running rescaling
                        float M = -INFINITY, Ls = 0.f, o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = 0.f;
                        const float* pmb = part_ml + (static_cast<long long>(b) * max_items * H + h) * 2;
                        const float* pob = part_o + (static_cast<long long>(b) * max_items * H + h) * D + ds * 8;
#pragma unroll 4
                        for (int c = 0; c < n_items; ++c) {
                            if (!starts(pb + c, pb)) continue;
                            const float2 ml =
                                __ldcg(reinterpret_cast<const float2*>(pmb + static_cast<long long>(c) * H * 2));
                            const float4* po = reinterpret_cast<const float4*>(pob + static_cast<long long>(c) * H * D);
                            const float4 a0 = __ldcg(po), a1 = __ldcg(po + 1);
                            const float mn = fmaxf(M, ml.x);
                            const float c1 = ex2(M - mn), c2 = ex2(ml.x - mn);
                            Ls = Ls * c1 + ml.y * c2;
                            o[0] = o[0] * c1 + a0.x * c2; o[1] = o[1] * c1 + a0.y * c2;
                            o[2] = o[2] * c1 + a0.z * c2; o[3] = o[3] * c1 + a0.w * c2;
                            o[4] = o[4] * c1 + a1.x * c2; o[5] = o[5] * c1 + a1.y * c2;
                            o[6] = o[6] * c1 + a1.z * c2; o[7] = o[7] * c1 + a1.w * c2;
                            M = mn;
                        }
                        const float inv = 1.f / Ls;
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] *= inv;
                        *reinterpret_cast<uint4*>(orow) = f32x8_to_bf16(o);
                    }
                    if (tid == 0) counters[b] = 0u;  // ready for the next call
                }
            }
            named_bar_sync(1, NCONS);  // smem (qh, kn, cs, red) reused by the next segment
            seg_start = true;
        }
        // next item
        if (++i >= n_items && w + 1 < n_my) {
            pb += n_items;
            ++b;
            while (b < B && !(lens[b] >= 1 && lens[b] <= Tcap)) ++b;  // invalid streams hold no items
            i = 0;
            L = b < B ? lens[b] : 1;
        }
    }
}

}  // namespace dec
}  // namespace nc
