// FP8 causal attention forward on sm_103a tensor cores (tcgen05 kind::f8f6f4,
// E4M3 x E4M3 -> fp32 in TMEM).  Head dimension 128.
//
// The quantisation reading (the pages name an fp8 training path and give no
// attention scheme; the oracle's orc_attn_fwd_fp8 states the same steps):
//   q8 = E4M3(qhat 2^5), k8 = E4M3(khat 2^5)    (QK-norm: |xhat| <= sqrt(D),
//                                                 so 2^5 stays within 448)
//   v8 = E4M3(v 2^tau), one tau per (batch, key/value head)
//   s_raw = q8 . k8 (= 2^10 qhat8 . khat8), exact products, fp32 sums
//   m = max over the row's visible keys of s_raw
//   P8 = E4M3(exp((s_raw - m) / (2^10 sqrt(D))) 2^8)
//   out = (sum_j P8_j v8_j) / (sum_j P8_j) 2^-tau,
//   lse = m / (2^10 sqrt(D)) + ln(sum_j exp(...))   (the unquantised sum)
// E4M3 has far less range than bf16, so P is taken relative to the row's
// true maximum, not the bf16 forward's fixed offset sqrt(D) (which would
// push typical weights below E4M3's smallest subnormal).  The maximum comes
// from a first pass over the keys (scores only); the second pass recomputes
// the scores and forms P8 and the PV product, so no accumulator is ever
// rescaled.
//
// One CTA per pair of 128-row query tiles of one (batch, head), as in the
// bf16 forward:
//   warp 8      TMA producer: both Q8 tiles, then K8 tiles (twice: one stream
//               per pass) and V8^T tiles (second pass) in 2-stage rings
//   warp 9      MMA issuer (one thread)
//   warps 0-3   softmax of tile 0, warps 4-7 of tile 1 (thread = row = TMEM lane)
// Tensor memory: S_t (128 fp32 columns) and O_t (128) per tile.  The softmax
// warps load S_t into registers and release it at once (S_READ), so the next
// S_t product never waits for the exponentials; P8 goes to a double-buffered
// shared-memory tile per query tile (the A operand of the PV product), and
// V8 arrives transposed ([D][keys], keys contiguous) so that both operands
// of every product are K-major.
#pragma once

#include <cuda_fp8.h>

#include "nc_common.cuh"
#include <type_traits>

namespace nc {
namespace fwd8 {

constexpr int D = 128;
constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;

enum Bar {
    Q_FULL = 0,
    K_FULL = 1,    // +stage (2)
    K_EMPTY = 3,   // +stage (2)
    V_FULL = 5,    // +stage (2)
    V_EMPTY = 7,   // +stage (2)
    S_FULL = 9,    // +tile
    S_READ = 11,   // +tile: the softmax warps hold S_t in registers
    P_FULL = 13,   // +2 tile + buffer: P8 of a key tile in that smem buffer
    O_FULL = 17,   // +tile
    MMA_DONE = 19,
    NUM_BARS = 20
};
// One P_FULL barrier per (tile, buffer), not per tile: the softmax warps may
// finish P8 of step j + 1 before the MMA thread has waited for P8 of step j
// (S of step j + 1 is issued before the PV product of step j), and a single
// barrier would then complete two phases under one parity wait.  P8 of step
// j + 2 (the next arrival on the same buffer's barrier) needs S of step
// j + 2, which the MMA thread issues only after it has consumed step j.

struct Smem {
    static constexpr int TILE = 128 * 128;      // one 128 x 128 E4M3 tile (16 KB)
    static constexpr int OFF_Q = 0;             // 2 query tiles
    static constexpr int OFF_K = OFF_Q + 2 * TILE;  // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * TILE;  // 2 stages (V8^T: [D][keys])
    static constexpr int OFF_P = OFF_V + 2 * TILE;  // 2 tiles x 2 buffers
    static constexpr int OFF_BAR = OFF_P + 4 * TILE;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TSLOT + 16;
    static constexpr int ALLOC = BYTES + 1024;
    // the output staging tile (bf16 [128][D] = 32 KB) of query tile t goes
    // over its two P buffers once its last PV product is done
    static_assert(BM * D * 2 <= 2 * TILE, "output staging");
};

constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_s(int t) { return static_cast<uint32_t>(t) * 128u; }
__host__ __device__ constexpr uint32_t tm_o(int t) { return 256u + static_cast<uint32_t>(t) * D; }

// kind::f8f6f4 instruction descriptor: E4M3 A and B (format code 0), K-major
// both, fp32 accumulator; the field layout is the one of kind::f16.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) { return idesc_f16kind(M, N, 0, 0, 0); }

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Two floats -> two E4M3 bytes (round to nearest even, saturating), low byte first.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
// Two E4M3 bytes (the low 16 bits of w) -> their values, exactly.
__device__ __forceinline__ float2 e4m3x2_value(uint32_t w) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_out,
                        const float* __restrict__ vscale, float* __restrict__ lse, int T, int H, int B, int n_qt,
                        int group, float c_log2, float c_ln, int W, int G) {
    using S = Smem;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x7f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_pairs = (n_qt + 1) / 2;
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * H, n_pairs, group);
    const int qt0 = 2 * (n_pairs - 1 - tc.rank);
    const int b = tc.bh / H, h = tc.bh % H;
    const int hk = h / G;
    const bool has1 = qt0 + 1 < n_qt;
    // key tiles of each query tile (window W >= 2^30: none cut); the stream
    // runs over the union [lo0, hi1]
    auto first_kt = [&](int qt) { return max(0, qt * BM - W + 1) / BN; };
    auto last_kt = [&](int qt) { return min(T - 1, qt * BM + BM - 1) / BN; };
    const int lo0 = first_kt(qt0), lo1 = has1 ? first_kt(qt0 + 1) : lo0;
    const int hi0 = last_kt(qt0), hi1 = has1 ? last_kt(qt0 + 1) : hi0;
    const int n_kv = hi1 - lo0 + 1;
    auto covers = [&](int t, int j) {  // does stream step j hold a key tile of query tile t
        const int kt = lo0 + j;
        return t == 0 ? kt <= hi0 : (has1 && kt >= lo1 && kt <= hi1);
    };
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);

    if (threadIdx.x == 0) {
        mbar_init(bar(Q_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(K_FULL + s), 1);
            mbar_init(bar(K_EMPTY + s), 1);
            mbar_init(bar(V_FULL + s), 1);
            mbar_init(bar(V_EMPTY + s), 1);
            mbar_init(bar(S_FULL + s), 1);
            mbar_init(bar(S_READ + s), 4);  // one arrival per softmax warp of the tile
            mbar_init(bar(P_FULL + 2 * s), 4);
            mbar_init(bar(P_FULL + 2 * s + 1), 4);
            mbar_init(bar(O_FULL + s), 1);
        }
        mbar_init(bar(MMA_DONE), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == WARP_TMA) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int issued_k[2] = {0, 0}, issued_v[2] = {0, 0};
            bool ok = true;
            mbar_expect_tx(bar(Q_FULL), (has1 ? 2 : 1) * S::TILE);
            for (int t = 0; t < (has1 ? 2 : 1); ++t)
                tma_load_4d(sb + S::OFF_Q + t * S::TILE, &tm_q, 0, h, (qt0 + t) * BM, b, bar(Q_FULL));
            // K8 twice (pass 1, pass 2), V8^T once, interleaved in pass 2
            for (int x = 0; ok && x < 2 * n_kv; ++x) {
                const int st = x & 1, use = x >> 1;
                const int kt = lo0 + (x < n_kv ? x : x - n_kv);
                if (x >= 2 && !mbar_wait(bar(K_EMPTY + st), (use - 1) & 1, 0x701)) { ok = false; break; }
                mbar_expect_tx(bar(K_FULL + st), S::TILE);
                tma_load_4d(sb + S::OFF_K + st * S::TILE, &tm_k, 0, hk, kt * BN, b, bar(K_FULL + st));
                ++issued_k[st];
                if (x >= n_kv) {
                    const int y = x - n_kv, vs = y & 1;
                    if (y >= 2 && !mbar_wait(bar(V_EMPTY + vs), ((y >> 1) - 1) & 1, 0x702)) { ok = false; break; }
                    mbar_expect_tx(bar(V_FULL + vs), S::TILE);
                    tma_load_3d(sb + S::OFF_V + vs * S::TILE, &tm_vt, kt * BN, 0, b * (H / G) + hk, bar(V_FULL + vs));
                    ++issued_v[vs];
                }
            }
            // never leave the CTA with a bulk copy still in flight
            mbar_wait(bar(Q_FULL), 0, 0x703);
            for (int s = 0; s < 2; ++s) {
                if (issued_k[s]) mbar_wait(bar(K_FULL + s), (issued_k[s] - 1) & 1, 0x704);
                if (issued_v[s]) mbar_wait(bar(V_FULL + s), (issued_v[s] - 1) & 1, 0x705);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_e4m3(BM, BN);  // q8 (K-major) x k8 (K-major)
            constexpr uint32_t IDESC_O = idesc_e4m3(BM, D);   // P8 (K-major) x v8^T (K-major)
            int ns[2] = {0, 0};  // S products issued per tile (both passes)
            int np[2] = {0, 0};  // PV products issued per tile
            auto issue_s = [&](int t, int st) {
#pragma unroll
                for (int kk = 0; kk < D / 32; ++kk)
                    mma_f8(tmem + tm_s(t), sdesc_sw128(sb + S::OFF_Q + t * S::TILE + kk * 32, 16, 1024),
                           sdesc_sw128(sb + S::OFF_K + st * S::TILE + kk * 32, 16, 1024), IDESC_S, kk > 0);
                mma_commit(bar(S_FULL + t));
            };
            bool ok = mbar_wait(bar(Q_FULL), 0, 0x710);
            // PV of stream step j for tile t (second pass)
            auto issue_pv = [&](int t, int j) -> bool {
                const int vs = j & 1;
                if (!mbar_wait(bar(P_FULL + 2 * t + (np[t] & 1)), (np[t] >> 1) & 1, 0x711)) return false;
                tc_fence_after();
                const uint32_t p_s = sb + S::OFF_P + (2 * t + (np[t] & 1)) * S::TILE;
#pragma unroll
                for (int kk = 0; kk < BN / 32; ++kk)
                    mma_f8(tmem + tm_o(t), sdesc_sw128(p_s + kk * 32, 16, 1024),
                           sdesc_sw128(sb + S::OFF_V + vs * S::TILE + kk * 32, 16, 1024), IDESC_O,
                           np[t] > 0 || kk > 0);
                ++np[t];
                return true;
            };
            for (int x = 0; ok && x < 2 * n_kv; ++x) {
                const int st = x & 1;
                const int j = x < n_kv ? x : x - n_kv;
                if (!mbar_wait(bar(K_FULL + st), (x >> 1) & 1, 0x712)) { ok = false; break; }
                for (int t = 0; ok && t < 2; ++t) {
                    if (!covers(t, j)) continue;
                    // S_t is free once the softmax warps hold the previous one
                    if (ns[t] > 0 && !mbar_wait(bar(S_READ + t), (ns[t] - 1) & 1, 0x713)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(t, st);
                    ++ns[t];
                }
                if (!ok) break;
                mma_commit(bar(K_EMPTY + st));
                // second pass: the PV products of the previous step
                if (x > n_kv) {
                    const int jp = j - 1;
                    if (!mbar_wait(bar(V_FULL + (jp & 1)), (jp >> 1) & 1, 0x714)) { ok = false; break; }
                    for (int t = 0; ok && t < 2; ++t)
                        if (covers(t, jp)) ok = issue_pv(t, jp);
                    if (!ok) break;
                    mma_commit(bar(V_EMPTY + (jp & 1)));
                }
            }
            // the last step's PV products, then the outputs
            if (ok && n_kv > 0) {
                const int jp = n_kv - 1;
                ok = mbar_wait(bar(V_FULL + (jp & 1)), (jp >> 1) & 1, 0x715);
                for (int t = 0; ok && t < 2; ++t)
                    if (covers(t, jp)) ok = issue_pv(t, jp);
                if (ok) {
                    mma_commit(bar(V_EMPTY + (jp & 1)));
                    mma_commit(bar(O_FULL + 0));
                    mma_commit(bar(O_FULL + 1));
                }
            }
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x716);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- softmax + epilogue -----
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int qt = qt0 + t;
        const int q_idx = qt * BM + row;
        const bool active = t == 0 || has1;  // uniform over the warpgroup
        const int lo_t = t ? lo1 : lo0;
        const int n_t = active ? (t ? hi1 : hi0) - lo_t + 1 : 0;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ts = tmem + lane_base + tm_s(t);
        float m = -INFINITY;             // row maximum of the raw scores
        float l_q = 0.f, l_x = 0.f;      // sums of P8 and of the exact p (both times 2^8)
        bool ok = true;
        int phase = 0;                   // S_FULL_t phases consumed
        for (int pass = 0; ok && pass < 2; ++pass) {
            for (int jt = 0; jt < n_t; ++jt, ++phase) {
                if (!mbar_wait_warp(bar(S_FULL + t), phase & 1, 0x720)) { ok = false; break; }
                tc_fence_after();
                uint32_t r[128];
                tmem_ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(r));
                tmem_ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
                tmem_ld32(ts + 64, *reinterpret_cast<uint32_t(*)[32]>(r + 64));
                tmem_ld32(ts + 96, *reinterpret_cast<uint32_t(*)[32]>(r + 96));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive_warp(bar(S_READ + t));  // S_t may be overwritten
                const int kt = lo_t + jt;
                const int d0 = q_idx - kt * BN;  // query - key at column 0
                const bool full = kt * BN + BN - 1 <= qt * BM && qt * BM + BM - 1 - kt * BN < W;
                // column e visible: 0 <= query - key < W (only the diagonal and
                // band-edge tiles test it: the loops below come in a masked and
                // an unmasked copy)
                auto vis = [&](int e) { return d0 - e >= 0 && d0 - e < W; };
                if (pass == 0) {
                    // eight independent maxima, so the reduction is not one
                    // 128-long dependency chain
                    float mm[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) mm[i] = -INFINITY;
                    auto max_tile = [&](auto masked) {
#pragma unroll
                        for (int e = 0; e < 128; ++e) {
                            const float x = __uint_as_float(r[e]);
                            if (!decltype(masked)::value || vis(e)) mm[e & 7] = fmaxf(mm[e & 7], x);
                        }
                    };
                    if (full)
                        max_tile(std::false_type{});
                    else
                        max_tile(std::true_type{});
                    m = fmaxf(m, fmaxf(fmaxf(fmaxf(mm[0], mm[1]), fmaxf(mm[2], mm[3])),
                                       fmaxf(fmaxf(mm[4], mm[5]), fmaxf(mm[6], mm[7]))));
                    continue;
                }
                // second pass: P8 = E4M3(exp2((s - m) c_log2 + 8)) into buffer jt % 2;
                // the sums of p and of P8 in four independent partials each
                const float off = 8.f - m * c_log2;
                uint32_t pw[32];
                float lx[4] = {0.f, 0.f, 0.f, 0.f}, lq[4] = {0.f, 0.f, 0.f, 0.f};
                auto p_tile = [&](auto masked) {
#pragma unroll
                    for (int e = 0; e < 128; e += 4) {
                        float p[4];
#pragma unroll
                        for (int i = 0; i < 4; i += 2) {
                            const float2 x2 = ffma2(make_float2(__uint_as_float(r[e + i]), __uint_as_float(r[e + i + 1])),
                                                    make_float2(c_log2, c_log2), make_float2(off, off));
                            p[i] = ex2(x2.x);
                            p[i + 1] = ex2(x2.y);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (decltype(masked)::value && !vis(e + i)) p[i] = 0.f;
                        const int a = (e >> 2) & 3;
                        lx[a] += (p[0] + p[1]) + (p[2] + p[3]);
                        const uint32_t lo2 = e4m3x2(p[0], p[1]), hi2 = e4m3x2(p[2], p[3]);
                        const float2 va = e4m3x2_value(lo2), vb = e4m3x2_value(hi2);
                        lq[a] += (va.x + va.y) + (vb.x + vb.y);
                        pw[e / 4] = lo2 | (hi2 << 16);
                    }
                };
                if (full)
                    p_tile(std::false_type{});
                else
                    p_tile(std::true_type{});
                l_x += (lx[0] + lx[1]) + (lx[2] + lx[3]);
                l_q += (lq[0] + lq[1]) + (lq[2] + lq[3]);
                uint8_t* pb = smem + S::OFF_P + (2 * t + (jt & 1)) * S::TILE;
                // buffer jt % 2 was last read by the PV product of step jt - 2,
                // which the MMA thread issued before the S product of step jt
                // that this thread has just read
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(pb + sw128_offset(row, c)) =
                        make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                fence_proxy_async_smem();
                mbar_arrive_warp(bar(P_FULL + 2 * t + (jt & 1)));
            }
        }
        // ---- epilogue: O / (l_q 2^tau) through the tile's P buffers (free:
        // every product of the tile is done), then TMA stores
        const bool epi = named_bar_and(2 + t, 128, active && ok && mbar_wait_warp(bar(O_FULL + t), 0, 0x721));
        uint8_t* stage = smem + S::OFF_P + 2 * t * S::TILE;
        if (epi) {
            tc_fence_after();
            const float vs = vscale[b * (H / G) + hk];  // 2^-tau
            const float inv = vs / l_q;
            float* lp = lse + (static_cast<long long>(b) * H + h) * T + q_idx;
            if (lse != nullptr && q_idx < T && NC_IN_RANGE(lp, 4, 0x411)) *lp = m * c_ln + logf(l_x * (1.f / 256.f));
#pragma unroll
            for (int c = 0; c < D / 32; ++c) stage_acc_bf16<32>(tmem + lane_base + tm_o(t), inv, stage, row, c * 32);
            fence_proxy_async_smem();
        }
        named_bar_sync(2 + t, 128);
        if (epi && quarter == 0 && lane == 0) {
            for (int c = 0; c < D / 64; ++c) tma_store_4d(&tm_out, smem_u32(stage) + c * (BM * 128), c * 64, h, qt * BM, b);
            bulk_commit();
            bulk_wait_read_all();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace fwd8
}  // namespace nc
