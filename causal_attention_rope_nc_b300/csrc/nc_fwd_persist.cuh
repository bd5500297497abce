// Causal attention forward, persistent form (the training forward; chunk
// prefill keeps the one-CTA-per-pair kernel of nc_fwd.cuh, whose header
// describes the per-pair computation this kernel repeats).
//
// One CTA per SM takes pairs of 128-row query tiles (the grouped order, the
// longest rows first in a group) from a global counter until none are left.
// The per-pair work is that of nc_fwd.cuh -- S_t = qhat khat^T, P_t written
// over S_t in TMEM as bf16 (split into P_hi + P_lo on the first query tile of
// each (b, h)), O_t += P_t V from TMEM, a fixed softmax offset -- and what
// persistence adds is the overlap of one pair's start with the previous
// pair's end:
//   - the producer loads the next pair's q tiles as soon as the last score
//     product of the current pair has read the q buffers (Q_EMPTY), and
//     streams its K/V tiles on through the same 2-stage rings;
//   - the MMA thread issues the next pair's first score products while the
//     softmax warps still finish the current pair (S_t is free once the last
//     PV product has read P_t; the tensor pipe runs one thread's products in
//     issue order);
//   - the output leaves from registers (16-byte stores of each row), so the
//     q buffers are never used as a staging tile.
// O_t of the next pair is first written by its first PV product, which the
// MMA thread issues only after the tile's softmax warps have arrived on
// P_FULL for that pair -- after their epilogue of the previous pair has read
// O_t out of TMEM.
//
// Roles: warp 8 producer (it also takes the pairs from the counter and hands
// their indices to the other roles through a 4-slot queue in shared memory),
// warp 9 MMA issuer, warps 0-3 / 4-7 softmax and epilogue of tile 0 / 1.
// Every barrier phase counts on across pairs.
#pragma once

#include "nc_fwd.cuh"

namespace nc {
namespace fwdp {

using fwd::BM;
using fwd::BN;
using fwd::p_col;
using fwd::tm_o;
using fwd::tm_s;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;
constexpr int NQ = 4;  // pair-index queue slots

enum Bar {
    Q_FULL = 0,
    Q_EMPTY = 1,   // the pair's score products are done with the q buffers
    K_FULL = 2,    // +stage
    K_EMPTY = 4,   // +stage
    V_FULL = 6,    // +stage
    V_EMPTY = 8,   // +stage
    S_FULL = 10,   // +tile
    P_FULL = 12,   // +tile
    O_FULL = 14,   // +tile
    MMA_DONE = 16,
    TQ_FULL = 17,  // +slot
    TQ_EMPTY = 21, // +slot
    NUM_BARS = 25
};
constexpr int TQ_READERS = 9;  // the MMA thread and the 8 softmax warps

template <int D>
struct Smem {
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int KBYTES = BN * D * 2;
    static constexpr int OFF_Q = 0;                   // 2 tiles
    static constexpr int OFF_K = OFF_Q + 2 * QBYTES;  // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KBYTES;  // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * KBYTES;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TQ = OFF_TSLOT + 16;
    static constexpr int BYTES = OFF_TQ + NQ * 4;
    static constexpr int ALLOC = BYTES + 1024;
};

// The tile ranges of pair `idx` (the same geometry as the per-pair kernel's,
// every query at its own position, keys 0..T-1).
struct Pair {
    int b, h, hk, qt0;
    bool has1;
    int lo0, lo1, hi0, hi1, f1, n0, n1, n_kv;
};
__device__ __forceinline__ Pair pair_of(int idx, int B, int H, int G, int n_qt, int group, int T, int W) {
    const int n_pairs = (n_qt + 1) / 2;
    const TileCoord tc = grouped_tile(idx, B * H, n_pairs, group);
    Pair p;
    p.qt0 = 2 * (n_pairs - 1 - tc.rank);
    p.b = tc.bh / H;
    p.h = tc.bh % H;
    p.hk = p.h / G;
    p.has1 = p.qt0 + 1 < n_qt;
    auto first_kt = [&](int qt) { return max(0, qt * BM - W + 1) / BN; };
    auto last_kt = [&](int qt) { return min(T - 1, qt * BM + BM - 1) / BN; };
    p.lo0 = first_kt(p.qt0);
    p.lo1 = p.has1 ? first_kt(p.qt0 + 1) : p.lo0;
    p.hi0 = last_kt(p.qt0);
    p.hi1 = p.has1 ? last_kt(p.qt0 + 1) : p.hi0;
    p.f1 = p.lo1 - p.lo0;
    p.n0 = p.hi0 - p.lo0 + 1;
    p.n1 = p.has1 ? p.hi1 - p.lo1 + 1 : 0;
    p.n_kv = p.hi1 - p.lo0 + 1;
    return p;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                               float* __restrict__ lse, int T, int H, int B, int n_qt, int group, float scale_log2,
                               float mfix_log2, float mfix, int W, int G, unsigned int* __restrict__ pair_counter) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x6f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_items = ((n_qt + 1) / 2) * B * H;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    volatile int* tq = reinterpret_cast<volatile int*>(smem + S::OFF_TQ);
    // the n-th pair of this CTA from the queue; -1: no more, or a wait gave up
    auto next_pair = [&](int n, bool warp_wide) -> int {
        const int q = n % NQ;
        const bool ok = warp_wide ? mbar_wait_warp(bar(TQ_FULL + q), (n / NQ) & 1, 0x630)
                                  : mbar_wait(bar(TQ_FULL + q), (n / NQ) & 1, 0x630);
        const int idx = ok ? tq[q] : -1;
        if (warp_wide)
            mbar_arrive_warp(bar(TQ_EMPTY + q));
        else
            mbar_arrive(bar(TQ_EMPTY + q));
        return idx;
    };
    // rows that see fewer than BN keys: P in two bf16 parts
    auto split_tile = [&](int qt) { return W < BN || qt * BM < BN; };

    if (threadIdx.x == 0) {
        mbar_init(bar(Q_FULL), 1);
        mbar_init(bar(Q_EMPTY), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(K_FULL + s), 1);
            mbar_init(bar(K_EMPTY + s), 1);
            mbar_init(bar(V_FULL + s), 1);
            mbar_init(bar(V_EMPTY + s), 1);
            mbar_init(bar(S_FULL + s), 1);
            mbar_init(bar(P_FULL + s), 4);  // one arrival per softmax warp of the tile
            mbar_init(bar(O_FULL + s), 1);
        }
        mbar_init(bar(MMA_DONE), 1);
        for (int q = 0; q < NQ; ++q) {
            mbar_init(bar(TQ_FULL + q), 1);
            mbar_init(bar(TQ_EMPTY + q), TQ_READERS);
        }
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tslot), fwd::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == WARP_TMA) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int xs = 0;  // K/V ring steps issued, all pairs
            int issued_k[2] = {0, 0}, issued_v[2] = {0, 0}, nq = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int q = n % NQ;
                if (n >= NQ && !mbar_wait(bar(TQ_EMPTY + q), (n / NQ - 1) & 1, 0x631)) break;
                const unsigned int got = atomicAdd(pair_counter, 1u);
                const int idx = got < static_cast<unsigned int>(n_items) ? static_cast<int>(got) : -1;
                tq[q] = idx;
                mbar_arrive(bar(TQ_FULL + q));
                if (idx < 0) break;
                const Pair p = pair_of(idx, B, H, G, n_qt, group, T, W);
                // the previous pair's score products have read the q buffers
                if (n > 0 && !mbar_wait(bar(Q_EMPTY), (n - 1) & 1, 0x632)) break;
                mbar_expect_tx(bar(Q_FULL), (p.has1 ? 2 : 1) * S::QBYTES);
                for (int t = 0; t < (p.has1 ? 2 : 1); ++t)
                    for (int c = 0; c < NC; ++c)
                        tma_load_4d(sb + S::OFF_Q + t * S::QBYTES + c * (BM * 128), &tm_q, c * 64, p.h,
                                    (p.qt0 + t) * BM, p.b, bar(Q_FULL));
                ++nq;
                for (int j = 0; j < p.n_kv; ++j, ++xs) {
                    const int st = xs & 1, use = xs >> 1;
                    if (xs >= 2 && !mbar_wait(bar(K_EMPTY + st), (use - 1) & 1, 0x633)) { ok = false; break; }
                    mbar_expect_tx(bar(K_FULL + st), S::KBYTES);
                    for (int c = 0; c < NC; ++c)
                        tma_load_4d(sb + S::OFF_K + st * S::KBYTES + c * (BN * 128), &tm_k, c * 64, p.hk,
                                    (p.lo0 + j) * BN, p.b, bar(K_FULL + st));
                    ++issued_k[st];
                    if (xs >= 2 && !mbar_wait(bar(V_EMPTY + st), (use - 1) & 1, 0x634)) { ok = false; break; }
                    mbar_expect_tx(bar(V_FULL + st), S::KBYTES);
                    for (int c = 0; c < NC; ++c)
                        tma_load_4d(sb + S::OFF_V + st * S::KBYTES + c * (BN * 128), &tm_v, c * 64, p.hk,
                                    (p.lo0 + j) * BN, p.b, bar(V_FULL + st));
                    ++issued_v[st];
                }
            }
            // never leave the CTA with a bulk copy still in flight
            if (nq) mbar_wait(bar(Q_FULL), (nq - 1) & 1, 0x635);
            for (int s = 0; s < 2; ++s) {
                if (issued_k[s]) mbar_wait(bar(K_FULL + s), (issued_k[s] - 1) & 1, 0x636);
                if (issued_v[s]) mbar_wait(bar(V_FULL + s), (issued_v[s] - 1) & 1, 0x637);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16kind(BM, BN, 0, 0, false);  // qhat (K-major) x khat (K-major), fp16
            constexpr uint32_t IDESC_O = idesc_bf16(BM, D, 0, 1);             // P (TMEM) x V (MN-major)
            int xs = 0;                // ring steps consumed, all pairs
            int np[2] = {0, 0};        // P_FULL phases consumed per tile
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = next_pair(n, false);
                if (idx < 0) break;
                const Pair p = pair_of(idx, B, H, G, n_qt, group, T, W);
                const bool split[2] = {split_tile(p.qt0), split_tile(p.qt0 + 1)};
                int s_left = p.n0 + p.n1;  // score products of this pair still to issue
                auto issue_s = [&](int t, int st) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                        const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                        mma_bf16(tmem + tm_s(t), sdesc_sw128(sb + S::OFF_Q + t * S::QBYTES + qa, 16, 1024),
                                 sdesc_sw128(sb + S::OFF_K + st * S::KBYTES + ka, 16, 1024), IDESC_S, kk > 0);
                    }
                    mma_commit(bar(S_FULL + t));
                    // the last score product of the pair: the q buffers are free once it is done
                    if (--s_left == 0) mma_commit(bar(Q_EMPTY));
                };
                auto issue_pv = [&](int t, int st, bool first) {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + tm_o<D>(t), tmem + tm_s(t) + p_col(kk),
                               sdesc_sw128(sb + S::OFF_V + st * S::KBYTES + kk * (16 * 128), BN * 128, 1024),
                               IDESC_O, (!first || kk > 0) ? 1u : 0u);
                    if (split[t]) {  // O += P_lo V
#pragma unroll
                        for (int kk = 0; kk < BN / 16; ++kk)
                            mma_ts(tmem + tm_o<D>(t), tmem + tm_s(t) + p_col(kk) + 16,
                                   sdesc_sw128(sb + S::OFF_V + st * S::KBYTES + kk * (16 * 128), BN * 128, 1024),
                                   IDESC_O, 1u);
                    }
                };
                ok = mbar_wait(bar(Q_FULL), n & 1, 0x640) && mbar_wait(bar(K_FULL + (xs & 1)), (xs >> 1) & 1, 0x641);
                if (!ok) break;
                tc_fence_after();
                issue_s(0, xs & 1);
                if (p.has1 && p.f1 == 0) issue_s(1, xs & 1);
                mma_commit(bar(K_EMPTY + (xs & 1)));
                for (int j = 0; ok && j < p.n_kv; ++j) {
                    const int x = xs + j, st = x & 1;
                    const bool nxt = j + 1 < p.n_kv;
                    if (!mbar_wait(bar(V_FULL + st), (x >> 1) & 1, 0x642)) { ok = false; break; }
                    bool k_ready = false;  // K of step j+1 waited for
                    if (j < p.n0) {
                        if (!mbar_wait(bar(P_FULL + 0), np[0] & 1, 0x643)) { ok = false; break; }
                        ++np[0];
                        tc_fence_after();
                        issue_pv(0, st, j == 0);
                        if (j == p.n0 - 1) mma_commit(bar(O_FULL + 0));
                        if (j + 1 < p.n0) {
                            if (!mbar_wait(bar(K_FULL + (st ^ 1)), ((x + 1) >> 1) & 1, 0x644)) { ok = false; break; }
                            k_ready = true;
                            tc_fence_after();
                            issue_s(0, st ^ 1);
                        }
                    }
                    if (p.has1 && j >= p.f1) {
                        if (!mbar_wait(bar(P_FULL + 1), np[1] & 1, 0x645)) { ok = false; break; }
                        ++np[1];
                        tc_fence_after();
                        issue_pv(1, st, j == p.f1);
                        if (j == p.n_kv - 1) mma_commit(bar(O_FULL + 1));
                    }
                    mma_commit(bar(V_EMPTY + st));
                    if (p.has1 && nxt) {
                        if (!k_ready && !mbar_wait(bar(K_FULL + (st ^ 1)), ((x + 1) >> 1) & 1, 0x646)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(1, st ^ 1);
                    }
                    if (nxt) mma_commit(bar(K_EMPTY + (st ^ 1)));
                }
                xs += p.n_kv;
            }
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x647);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- softmax + epilogue -----
        const int t = warp >> 2;        // query tile of this warpgroup
        const int quarter = warp & 3;   // TMEM lane quarter
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ts = tmem + lane_base + tm_s(t);
        int sphase = 0, ophase = 0;  // S_FULL and O_FULL phases consumed by this tile's warps
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int idx = next_pair(n, true);
            if (idx < 0) break;  // uniform over each warp
            const Pair p = pair_of(idx, B, H, G, n_qt, group, T, W);
            if (t == 1 && !p.has1) continue;  // uniform over the warpgroup: no second tile in this pair
            const int qt = p.qt0 + t;
            const int q_idx = qt * BM + row;
            const int n_t = t ? p.n1 : p.n0;
            const int lo_t = t ? p.lo1 : p.lo0;
            float2 l2 = make_float2(0.f, 0.f);  // the row sum: even and odd columns
            for (int j = 0; j < n_t; ++j) {
                if (!mbar_wait_warp(bar(S_FULL + t), sphase & 1, 0x650)) { ok = false; break; }
                ++sphase;
                tc_fence_after();
                uint32_t r[2][32];
                tmem_ld32(ts, r[0]);
                tmem_wait_ld();
                const int kt = lo_t + j;
                const int d0 = qt * BM + row - kt * BN;  // query - key at column 0 of the tile
                auto exp_tile = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
                        if (c + 1 < BN / 32) tmem_ld32(ts + (c + 1) * 32, r[(c + 1) & 1]);
                        const uint32_t* rc = r[c & 1];
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x2 = ffma2(make_float2(__uint_as_float(rc[e]), __uint_as_float(rc[e + 1])),
                                                    make_float2(scale_log2, scale_log2),
                                                    make_float2(-mfix_log2, -mfix_log2));
                            float p0 = ex2(x2.x);
                            float p1 = ex2(x2.y);
                            if constexpr (decltype(masked)::value) {
                                const int dd = d0 - (c * 32 + e);  // visible: 0 <= query - key < W
                                if (dd < 0 || dd >= W) p0 = 0.f;
                                if (dd - 1 < 0 || dd - 1 >= W) p1 = 0.f;
                            }
                            w[e / 2] = pack_bf16x2(p0, p1);
                            l2 = fadd2(l2, make_float2(p0, p1));
                        }
                        tmem_st16(ts + c * 32, w);
                        if (c + 1 < BN / 32) tmem_wait_ld();
                    }
                };
                auto exp_split = [&]() {
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t rc[32];
                        tmem_ld32(ts + c * 32, rc);
                        tmem_wait_ld();
                        uint32_t w[16], wl[16];
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const float2 x2 = ffma2(make_float2(__uint_as_float(rc[e]), __uint_as_float(rc[e + 1])),
                                                    make_float2(scale_log2, scale_log2),
                                                    make_float2(-mfix_log2, -mfix_log2));
                            float p0 = ex2(x2.x);
                            float p1 = ex2(x2.y);
                            const int dd = d0 - (c * 32 + e);
                            if (dd < 0 || dd >= W) p0 = 0.f;
                            if (dd - 1 < 0 || dd - 1 >= W) p1 = 0.f;
                            const uint32_t wv = pack_bf16x2(p0, p1);
                            const float2 ph = unpack_bf16x2(wv);
                            w[e / 2] = wv;
                            wl[e / 2] = pack_bf16x2(p0 - ph.x, p1 - ph.y);
                            l2 = fadd2(l2, make_float2(p0, p1));
                        }
                        tmem_st16(ts + c * 32, w);
                        tmem_st16(ts + c * 32 + 16, wl);
                    }
                };
                const bool full = kt * BN + BN - 1 <= qt * BM && qt * BM + BM - 1 - kt * BN < W;
                if (split_tile(qt))
                    exp_split();
                else if (full)
                    exp_tile(std::false_type{});
                else
                    exp_tile(std::true_type{});
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_warp(bar(P_FULL + t));
            }
            if (!ok) break;
            // ---- epilogue: O / l straight from TMEM to the output rows (16-byte
            // stores of each row; rows past T are skipped) and the lse
            if (!mbar_wait_warp(bar(O_FULL + t), ophase & 1, 0x651)) { ok = false; break; }
            ++ophase;
            tc_fence_after();
            const float l_sum = l2.x + l2.y;
            const float inv_l = 1.f / l_sum;
            float* lp = lse + (static_cast<long long>(p.b) * H + p.h) * T + q_idx;
            if (lse != nullptr && q_idx < T && NC_IN_RANGE(lp, 4, 0x652)) *lp = mfix + logf(l_sum);
            __nv_bfloat16* orow = out + ((static_cast<long long>(p.b) * T + q_idx) * H + p.h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + tm_o<D>(t) + c * 32, v);
                tmem_wait_ld();
                if (q_idx < T) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint32_t* u = v + 8 * g;
                        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32 + 8 * g);
                        if (NC_IN_RANGE(dst, 16, 0x653))
                            *dst = make_uint4(pack_bf16x2(__uint_as_float(u[0]) * inv_l, __uint_as_float(u[1]) * inv_l),
                                              pack_bf16x2(__uint_as_float(u[2]) * inv_l, __uint_as_float(u[3]) * inv_l),
                                              pack_bf16x2(__uint_as_float(u[4]) * inv_l, __uint_as_float(u[5]) * inv_l),
                                              pack_bf16x2(__uint_as_float(u[6]) * inv_l, __uint_as_float(u[7]) * inv_l));
                    }
                }
            }
            tc_fence_before();  // O_t has been read: the next pair's first PV product may overwrite it
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, fwd::TMEM_COLS);
    }
}

}  // namespace fwdp
}  // namespace nc
