// Causal attention forward on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA computes two consecutive 128-row query tiles (2p and 2p+1) of one
// (batch, head); both share every K/V tile it streams (those of key/value
// head h / G: grouped-query attention shares one among G query heads).  Query row r of stream
// b sits at position qoff[b] + r (qoff == nullptr: position r) among Tk key
// positions: a chunk of new tokens attending over a KV cache, or (offset 0,
// Tk = T) the whole sequence.  With a sliding window
// W (query i sees key j when 0 <= i - j < W) the stream starts at the first
// key tile either query tile can see, and tile 2p+1 may start one K/V tile
// later than tile 2p:
//   warp 8      TMA producer: both Q tiles once, then K_j / V_j in 2-stage rings
//   warp 9      MMA issuer (one thread)
//   warps 0-3   softmax of tile 0, warps 4-7 softmax of tile 1: thread r owns
//               query row r (TMEM lane r) of its tile
// Tensor memory: S_t (128 fp32 columns) per tile, overwritten in place by the
// bf16 probabilities P_t that the PV product reads as its A operand (the 32
// keys of chunk c in columns [32c, 32c + 16)), and an output accumulator O_t
// (D columns) per tile: 2 x 128 + 2 x D <= 512.
//
// Rows that see few keys (the first 128 positions of a sequence, or every
// row under a window shorter than 128) put large weights on few values, and
// there rounding P to bf16 (relative 2^-8) would dominate the output's error.
// For such query tiles P is split into P_hi = bf16(P) and P_lo = bf16(P -
// P_hi), the latter in columns [32c + 16, 32c + 32), and the PV product runs
// twice (O += P_hi V + P_lo V): P then carries about 16 bits.  Causal
// attention over whole sequences pays this once per (batch, head).
//
// The normaliser is the fp32 sum of the unrounded probabilities, two columns
// per paired add; the bf16 weights the PV product consumes then sum to one
// within their unbiased rounding (about 2^-9 / sqrt(keys) relative), far
// inside the output's own bf16 rounding.  (Summing the rounded weights
// instead costs one more instruction per element, a sixth of the softmax.)
//
// Issue order (the tensor pipe executes one thread's MMAs in issue order):
//   S_0(0) S_1(0) | PV_0(j) S_0(j+1) PV_1(j) S_1(j+1) | ...
// so each softmax warpgroup has the other tile's two products (about 1000
// cycles) to turn S_t(j) into P_t(j), and the two groups alternate.
//
// Exponentials: all on the special-function unit (ex2.approx), which on
// sm_103a sustains about 28 per clock per SM; the diagonal tile, the only
// one with masked entries, runs its own copy of the loop.
//
// Operand types: P and V are bf16; qhat and khat are IEEE fp16 (QK_BF16 =
// false: the forward, whose prologue writes them in fp16 for the accuracy of
// the scores) or bf16 (QK_BF16 = true: chunk prefill, whose keys come from
// the bf16 key cache; tcgen05 wants A and B of one product in one type).
//
// Fixed softmax offset.  q and k are RMS-normalised before the product, so
// |qhat . khat| <= |qhat| |khat| <= D (both norms are at most sqrt(D), up to
// 16-bit rounding of the stored vectors, which adds < 2^-8 relative).  Hence
// every scaled score s = qhat.khat / sqrt(D) lies in [-m, m] with
// m = sqrt(D) * 1.0079, and exp(s - m) lies in [exp(-2m), 1]: no running
// maximum and no rescaling of O are needed, in any row, for any input.  The
// softmax is shift invariant, so this is the same function as the max-shifted
// form; lse = m + ln(sum_j exp(s_j - m)).
#pragma once

#include "nc_common.cuh"
#include <type_traits>

namespace nc {
namespace fwd {

constexpr int BM = 128;  // query rows per tile (one TMEM lane each)
constexpr int BN = 128;  // keys per tile
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;

enum Bar {
    Q_FULL = 0,
    K_FULL = 1,    // +stage
    K_EMPTY = 3,   // +stage
    V_FULL = 5,    // +stage
    V_EMPTY = 7,   // +stage
    S_FULL = 9,    // +tile
    P_FULL = 11,   // +tile
    O_FULL = 13,   // +tile
    MMA_DONE = 15,
    NUM_BARS = 16
};

template <int D>
struct Smem {
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int KBYTES = BN * D * 2;
    static constexpr int OFF_Q = 0;                       // 2 tiles
    static constexpr int OFF_K = OFF_Q + 2 * QBYTES;      // 2 stages
    static constexpr int OFF_V = OFF_K + 2 * KBYTES;      // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * KBYTES;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TSLOT + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
};

constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_s(int t) { return static_cast<uint32_t>(t) * 128u; }
// TMEM column (relative to S_t) of the packed P_hi pairs of K-step kk (keys
// 16 kk .. 16 kk + 15): chunk kk / 2 of 32 keys, 8 columns per step; P_lo
// sits 16 columns further
__host__ __device__ constexpr uint32_t p_col(int kk) { return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8); }
template <int D>
__host__ __device__ constexpr uint32_t tm_o(int t) {
    return 256u + static_cast<uint32_t>(t) * D;
}

template <int D, bool QK_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_out,
                    float* __restrict__ lse, int T, int H, int B, int n_qt, int group, float scale_log2,
                    float mfix_log2, float mfix, int W, const int* __restrict__ qoff, int Tk, int G) {
    using S = Smem<D>;
    constexpr int NC = D / 64;  // 64-column (128-byte) swizzle spans per row
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x0f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped (b, h) order, longest rows (the last pair of query tiles) first in a group
    const int n_pairs = (n_qt + 1) / 2;
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * H, n_pairs, group);
    const int qt0 = 2 * (n_pairs - 1 - tc.rank);
    const int b = tc.bh / H, h = tc.bh % H;
    const int hk = h / G;  // key/value head (grouped-query attention; G = 1: hk = h)
    const bool has1 = qt0 + 1 < n_qt;
    const int qpos0 = qoff ? qoff[b] : 0;  // position of query row 0
    if (qpos0 < 0 || qpos0 + T > Tk) {     // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(2, 0x0f1);
        return;
    }
    // key tiles a query tile sees: from the first key within W of its first
    // row (W >= 2^30 means no window) to the key at its last row's position
    auto first_kt = [&](int qt) { return max(0, qpos0 + qt * BM - W + 1) / BN; };
    auto last_kt = [&](int qt) { return (qpos0 + min(T - 1, qt * BM + BM - 1)) / BN; };
    const int lo0 = first_kt(qt0), lo1 = has1 ? first_kt(qt0 + 1) : lo0;
    const int hi0 = last_kt(qt0), hi1 = has1 ? last_kt(qt0 + 1) : hi0;
    const int f1 = lo1 - lo0;               // stream index of tile qt0+1's first key tile (0 or 1)
    const int n0 = hi0 - lo0 + 1;           // key tiles of query tile qt0
    const int n1 = has1 ? hi1 - lo1 + 1 : 0;  // key tiles of query tile qt0 + 1
    const int n_kv = hi1 - lo0 + 1;         // the stream: tile qt0's tiles then tile qt0+1's last
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    // query tiles whose rows see fewer than BN keys: P in two bf16 parts
    auto split_tile = [&](int t) { return W < BN || qpos0 + (qt0 + t) * BM < BN; };

    if (threadIdx.x == 0) {
        mbar_init(bar(Q_FULL), 1);
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
            mbar_expect_tx(bar(Q_FULL), (has1 ? 2 : 1) * S::QBYTES);
            for (int t = 0; t < (has1 ? 2 : 1); ++t)
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_Q + t * S::QBYTES + c * (BM * 128), &tm_q, c * 64, h, (qt0 + t) * BM, b,
                                bar(Q_FULL));
            for (int j = 0; j < n_kv; ++j) {
                const int st = j & 1, use = j >> 1;
                if (j >= 2 && !mbar_wait(bar(K_EMPTY + st), (use - 1) & 1, 0x101)) break;
                mbar_expect_tx(bar(K_FULL + st), S::KBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_K + st * S::KBYTES + c * (BN * 128), &tm_k, c * 64, hk, (lo0 + j) * BN, b,
                                bar(K_FULL + st));
                ++issued_k[st];
                if (j >= 2 && !mbar_wait(bar(V_EMPTY + st), (use - 1) & 1, 0x102)) break;
                mbar_expect_tx(bar(V_FULL + st), S::KBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_V + st * S::KBYTES + c * (BN * 128), &tm_v, c * 64, hk, (lo0 + j) * BN, b,
                                bar(V_FULL + st));
                ++issued_v[st];
            }
            // drain: never leave the CTA with a bulk copy still in flight
            mbar_wait(bar(Q_FULL), 0, 0x103);
            for (int s = 0; s < 2; ++s) {
                if (issued_k[s]) mbar_wait(bar(K_FULL + s), (issued_k[s] - 1) & 1, 0x104);
                if (issued_v[s]) mbar_wait(bar(V_FULL + s), (issued_v[s] - 1) & 1, 0x105);
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16kind(BM, BN, 0, 0, QK_BF16);  // qhat (K-major) x khat (K-major)
            constexpr uint32_t IDESC_O = idesc_bf16(BM, D, 0, 1);  // P (TMEM) x V (MN-major)
            auto issue_s = [&](int t, int st) {
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + tm_s(t), sdesc_sw128(sb + S::OFF_Q + t * S::QBYTES + qa, 16, 1024),
                             sdesc_sw128(sb + S::OFF_K + st * S::KBYTES + ka, 16, 1024), IDESC_S, kk > 0);
                }
                mma_commit(bar(S_FULL + t));
            };
            auto issue_pv = [&](int t, int st, bool first) {
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_ts(tmem + tm_o<D>(t), tmem + tm_s(t) + p_col(kk),
                           sdesc_sw128(sb + S::OFF_V + st * S::KBYTES + kk * (16 * 128), BN * 128, 1024), IDESC_O,
                           (!first || kk > 0) ? 1u : 0u);
                if (split_tile(t)) {  // O += P_lo V
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + tm_o<D>(t), tmem + tm_s(t) + p_col(kk) + 16,
                               sdesc_sw128(sb + S::OFF_V + st * S::KBYTES + kk * (16 * 128), BN * 128, 1024), IDESC_O,
                               1u);
                }
            };
            bool ok = mbar_wait(bar(Q_FULL), 0, 0x201) && mbar_wait(bar(K_FULL + 0), 0, 0x202);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (has1 && f1 == 0) issue_s(1, 0);
                mma_commit(bar(K_EMPTY + 0));
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int st = j & 1;
                const bool nxt = j + 1 < n_kv;
                if (!mbar_wait(bar(V_FULL + st), (j >> 1) & 1, 0x203)) { ok = false; break; }
                bool k_ready = false;  // K_{j+1} waited for
                if (j < n0) {
                    if (!mbar_wait(bar(P_FULL + 0), j & 1, 0x204)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(0, st, j == 0);
                    if (j == n0 - 1) mma_commit(bar(O_FULL + 0));
                    if (j + 1 < n0) {
                        if (!mbar_wait(bar(K_FULL + (st ^ 1)), ((j + 1) >> 1) & 1, 0x205)) { ok = false; break; }
                        k_ready = true;
                        tc_fence_after();
                        issue_s(0, st ^ 1);
                    }
                }
                if (has1 && j >= f1) {
                    if (!mbar_wait(bar(P_FULL + 1), (j - f1) & 1, 0x206)) { ok = false; break; }
                    tc_fence_after();
                    issue_pv(1, st, j == f1);
                    if (j == n_kv - 1) mma_commit(bar(O_FULL + 1));
                }
                mma_commit(bar(V_EMPTY + st));
                if (has1 && nxt) {
                    if (!k_ready && !mbar_wait(bar(K_FULL + (st ^ 1)), ((j + 1) >> 1) & 1, 0x207)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(1, st ^ 1);
                }
                if (nxt) mma_commit(bar(K_EMPTY + (st ^ 1)));
            }
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x208);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- softmax + epilogue -----
        const int t = warp >> 2;        // query tile of this warpgroup
        const int quarter = warp & 3;   // TMEM lane quarter
        const int row = quarter * 32 + lane;
        const int qt = qt0 + t;
        const int q_idx = qt * BM + row;
        const int n_t = t ? n1 : n0;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t ts = tmem + lane_base + tm_s(t);
        float2 l2 = make_float2(0.f, 0.f);  // the row sum: even and odd columns
        bool ok = true;
        for (int j = 0; j < n_t; ++j) {
            if (!mbar_wait_warp(bar(S_FULL + t), j & 1, 0x301)) { ok = false; break; }
            tc_fence_after();
            uint32_t r[2][32];
            tmem_ld32(ts, r[0]);
            tmem_wait_ld();
            const int kt = (t ? lo1 : lo0) + j;            // key tile
            const int d0 = qpos0 + qt * BM + row - kt * BN;  // query - key position at column 0 of the tile
            auto exp_tile = [&](auto masked) {
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    // the load of chunk c+1 overlaps the exponentials of chunk c
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
                            // visible: 0 <= query - key < W
                            const int dd = d0 - (c * 32 + e);
                            if (dd < 0 || dd >= W) p0 = 0.f;
                            if (dd - 1 < 0 || dd - 1 >= W) p1 = 0.f;
                        }
                        w[e / 2] = pack_bf16x2(p0, p1);
                        l2 = fadd2(l2, make_float2(p0, p1));
                    }
                    // chunk c lands in packed columns [32c, 32c+16): its own, already read
                    tmem_st16(ts + c * 32, w);
                    if (c + 1 < BN / 32) tmem_wait_ld();
                }
            };
            // The split form (P_hi in packed columns [32c, 32c+16), P_lo in
            // [32c+16, 32c+32)) runs on few tiles (the first query tile of
            // each (b, h)), so it is a compact loop, one chunk at a time and
            // always with the visibility test (B=32, T=2048, H=10, D=128: 373-376 us against 378 us
            // with two more fully unrolled copies of the loop above, 271
            // against 280 us with a 512-key window).
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
            // every (query, key) pair of the tile visible: the plain loop
            const bool full = kt * BN + BN - 1 <= qpos0 + qt * BM && qpos0 + qt * BM + BM - 1 - kt * BN < W;
            if (split_tile(t))
                exp_split();
            else if (full)
                exp_tile(std::false_type{});
            else
                exp_tile(std::true_type{});
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive_warp(bar(P_FULL + t));
        }
        // ---- epilogue: O / l into the tile's qhat buffer (free: every product
        // of the tile is done), then TMA stores (rows past T are clipped).
        // Both barriers are reached by the group's four warps whatever
        // happened; the AND keeps their branch uniform.
        const bool epi = named_bar_and(2 + t, 128, n_t > 0 && ok && mbar_wait_warp(bar(O_FULL + t), 0, 0x303));
        uint8_t* stage = smem + S::OFF_Q + t * S::QBYTES;
        if (epi) {
            tc_fence_after();
            const float l_sum = l2.x + l2.y;
            const float inv_l = 1.f / l_sum;
            float* lp = lse + (static_cast<long long>(b) * H + h) * T + q_idx;
            if (lse != nullptr && q_idx < T && NC_IN_RANGE(lp, 4, 0x410)) *lp = mfix + logf(l_sum);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) stage_acc_bf16<32>(tmem + lane_base + tm_o<D>(t), inv_l, stage, row, c * 32);
            fence_proxy_async_smem();
        }
        named_bar_sync(2 + t, 128);
        if (epi && quarter == 0 && lane == 0) {
            for (int c = 0; c < NC; ++c)
                tma_store_4d(&tm_out, smem_u32(stage) + c * (BM * 128), c * 64, h, qt * BM, b);
            bulk_commit();
            bulk_wait_read_all();  // the staged tile stays valid until the stores have read it
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace fwd
}  // namespace nc
