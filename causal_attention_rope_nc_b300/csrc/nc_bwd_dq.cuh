// Causal attention backward, query side: dQ on sm_103a tensor cores
// (tcgen05 + TMEM + TMA), with the RoPE transpose and the RMSNorm backward
// fused into the epilogue, so dq leaves the kernel finished (bf16).
//
// One CTA owns one 128-query tile i of one (batch, head) and walks the key
// tiles j <= i that it can see (all of them, or with a sliding window W --
// query q sees key k when 0 <= q - k < W -- those from the tile of the first
// query's oldest visible key), recomputing what it needs from the forward's
// lse:
//   S_j   = qhat_i khat_j^T                 (M=128 queries, N=128 keys, K=D)
//   P_j   = exp2(S_j * scale*log2e - lse2_i)
//   dP_j  = dout_i v_j^T                    (M=128 queries, N=128 keys, K=D)
//   dS_j  = P_j o (dP_j - delta_i)
//   dQ_i += dS_j khat_j                     (M=128 queries, N=D, K=128 keys)
// Every dQ element is produced by exactly one CTA: no atomics, no fp32
// accumulator in global memory, deterministic results.
//
// Tensor memory: two S buffers (S_j in buffer j%2; the fp16 dS_j is written
// over it in place and read from there as the A operand of the dQ product),
// dP (128 columns) and the dQ accumulator (D columns).
//
// Issue order (one thread's MMAs execute in issue order):
//   S_0, S_1, dP_0 | [dP_j in registers] dP_{j+1} | [dS_j in TMEM] dQ(j), S_{j+2} | ...
// dS_j is written over S_j, not over dP_j, so the next dP may start as soon
// as the softmax warps have loaded dP_j: it runs while they form dS_j, and
// dQ(j) and S_{j+2} run while they form P_{j+1}.  K tiles
// sit in a 3-stage ring (tile j is read by S_j and by dQ(j) two steps later),
// V tiles in a 2-stage ring.
//
// Roles: warps 0-7 P and dS (warp w: TMEM lane quarter w%4 = 32 query rows,
// key half w/4 = 64 columns), warp 8 TMA, warp 9 MMA.  At the end the same
// eight warps (two threads per query row) stage dq in shared memory and it
// leaves through TMA stores.  The raw q rows and RoPE table rows it needs
// are prefetched while the last key tiles are processed, into the v stage
// and the two k stages the last key tile does not use, as they free up.
//
// dS is stored as alpha * dS in fp16 with a per-CTA power of two alpha from
// the bound |dS_ij| <= P_ij |dP_ij - delta_i| <= ||dout_i|| max_j ||v_j|| +
// |delta_i| (max_j ||v_j|| over the whole tensor, published by the dK/dV
// kernel), so |alpha dS| <= 2^14.
#pragma once

#include "nc_common.cuh"
#include <type_traits>
#include "nc_normrope_bwd.cuh"

namespace nc {
namespace bwdq {

constexpr int BM = 128;  // queries per CTA
constexpr int BN = 128;  // keys per tile
constexpr int KSTAGES = 3;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;
constexpr int SMEM_LIMIT = 232448;  // 227 KB opt-in per block

enum Bar {
    QD_FULL = 0,   // qhat_i and dout_i landed
    K_FULL = 1,    // +stage (3)
    K_EMPTY = 4,   // +stage (3)
    V_FULL = 7,    // +stage (2)
    V_EMPTY = 9,   // +stage (2)
    S_FULL = 11,   // +buffer (2)
    DP_FULL = 13,
    DS_FULL = 14,  // softmax read dP_j and wrote dS_j
    DQ_FULL = 15,
    MMA_DONE = 16,
    EPI_FULL = 17,  // raw q tile and RoPE table tile staged for the dq epilogue
    DP_READ = 18,   // the softmax warps hold dP_j in registers: dP_{j+1} may start
    NUM_BARS = 19
};

template <int D>
struct Smem {
    static constexpr int TBYTES = BN * D * 2;  // one 128-row tile of D 16-bit values
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + TBYTES;
    static constexpr int OFF_K = OFF_DO + TBYTES;         // KSTAGES stages
    static constexpr int OFF_V = OFF_K + KSTAGES * TBYTES;  // 2 stages
    static constexpr int OFF_BAR = OFF_V + 2 * TBYTES;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_MISC = OFF_TSLOT + 16;  // 4 warp maxima of the dS bound
    static constexpr int BYTES = OFF_MISC + 32;
    static constexpr int ALLOC = (BYTES + 1024 < SMEM_LIMIT) ? BYTES + 1024 : SMEM_LIMIT;
    // epilogue: the raw q tile over a v stage, the RoPE table tile (fp32
    // [128][D]) over two k stages, dq staged over the qhat tile and the
    // row-half exchange over the dout tile
    static constexpr int CBYTES = BM * D * 4;
    static_assert(BYTES <= SMEM_LIMIT, "dQ tiles exceed shared memory");
    static_assert(CBYTES == 2 * TBYTES && 2 * BM * 8 <= TBYTES, "epilogue tiles exceed the rings");
};

constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_s(int buf) { return static_cast<uint32_t>(buf) * 128u; }
constexpr uint32_t TM_DP = 256;
constexpr uint32_t TM_DQ = 384;  // D columns

// TMEM column of the packed pair holding keys (2c, 2c+1) of K-step kk: key
// half kk/4 sits inside the S columns its own warps read.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8); }

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_qraw, const __grid_constant__ CUtensorMap tm_tab,
                       const __grid_constant__ CUtensorMap tm_dq, const float* __restrict__ lse2,
                       const float* __restrict__ delta, const unsigned int* __restrict__ gmax, int T, int H, int B,
                       int Tpad, int group, float scale, float scale_log2, float eps, int W, int G) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x2f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped (b, h) order, longest walks (the last query tile) first in a group
    const int n_qt = (T + BM - 1) / BM;
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * H, n_qt, group);
    const int qt = n_qt - 1 - tc.rank;
    const int b = tc.bh / H, h = tc.bh % H;
    const int hk = h / G;  // key/value head (grouped-query attention; G = 1: hk = h)
    const int kt_lo = max(0, qt * BM - W + 1) / BN;  // first visible key tile (W >= 2^30: none cut)
    const int n_kv = qt - kt_lo + 1;                  // BM == BN: key tiles kt_lo..qt
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    float* misc = reinterpret_cast<float*>(smem + S::OFF_MISC);
    const long long bh = static_cast<long long>(b) * H + h;
    // epilogue space: the v stage of key tile n_kv-2 and the k stages of
    // tiles n_kv-3 and n_kv-2 (never used when those tiles do not exist)
    const int vs_epi = n_kv & 1, ks_a = n_kv % KSTAGES, ks_b = (n_kv + 1) % KSTAGES;

    if (threadIdx.x == 0) {
        mbar_init(bar(QD_FULL), 1);
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(bar(K_FULL + s), 1);
            mbar_init(bar(K_EMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(V_FULL + s), 1);
            mbar_init(bar(V_EMPTY + s), 1);
            mbar_init(bar(S_FULL + s), 1);
        }
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DS_FULL), 8);   // one arrival per softmax warp
        mbar_init(bar(DP_READ), 8);
        mbar_init(bar(DQ_FULL), 1);
        mbar_init(bar(MMA_DONE), 1);
        mbar_init(bar(EPI_FULL), 1);
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
            int issued_k[KSTAGES] = {0, 0, 0}, issued_v[2] = {0, 0};
            mbar_expect_tx(bar(QD_FULL), 2 * S::TBYTES);
            for (int c = 0; c < NC; ++c) {
                tma_load_4d(sb + S::OFF_Q + c * (BM * 128), &tm_q, c * 64, h, qt * BM, b, bar(QD_FULL));
                tma_load_4d(sb + S::OFF_DO + c * (BM * 128), &tm_do, c * 64, h, qt * BM, b, bar(QD_FULL));
            }
            for (int j = 0; j < n_kv; ++j) {
                const int ks = j % KSTAGES, vs = j & 1;
                if (j >= KSTAGES && !mbar_wait(bar(K_EMPTY + ks), (j / KSTAGES - 1) & 1, 0x121)) break;
                mbar_expect_tx(bar(K_FULL + ks), S::TBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_K + ks * S::TBYTES + c * (BN * 128), &tm_k, c * 64, hk, (kt_lo + j) * BN, b,
                                bar(K_FULL + ks));
                ++issued_k[ks];
                if (j >= 2 && !mbar_wait(bar(V_EMPTY + vs), ((j >> 1) - 1) & 1, 0x122)) break;
                mbar_expect_tx(bar(V_FULL + vs), S::TBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_V + vs * S::TBYTES + c * (BN * 128), &tm_v, c * 64, hk, (kt_lo + j) * BN, b,
                                bar(V_FULL + vs));
                ++issued_v[vs];
            }
            // dq epilogue tiles, each as soon as its stage is released
            mbar_expect_tx(bar(EPI_FULL), S::TBYTES + S::CBYTES);
            bool epi = n_kv < 2 || mbar_wait(bar(V_EMPTY + vs_epi), ((n_kv - 2) >> 1) & 1, 0x128);
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_V + vs_epi * S::TBYTES + c * (BM * 128), &tm_qraw, c * 64, h, qt * BM,
                                b, bar(EPI_FULL));
            }
            epi = epi && (n_kv < 3 || mbar_wait(bar(K_EMPTY + ks_a), ((n_kv - 3) / KSTAGES) & 1, 0x129));
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_2d(sb + S::OFF_K + ks_a * S::TBYTES + c * (BM * 128), &tm_tab, c * 32, qt * BM,
                                bar(EPI_FULL));
            }
            epi = epi && (n_kv < 2 || mbar_wait(bar(K_EMPTY + ks_b), ((n_kv - 2) / KSTAGES) & 1, 0x12a));
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_2d(sb + S::OFF_K + ks_b * S::TBYTES + c * (BM * 128), &tm_tab, (NC + c) * 32,
                                qt * BM, bar(EPI_FULL));
            }
            // never leave the CTA with a bulk copy still in flight
            mbar_wait(bar(QD_FULL), 0, 0x123);
            for (int s = 0; s < KSTAGES; ++s)
                if (issued_k[s]) mbar_wait(bar(K_FULL + s), (issued_k[s] - 1) & 1, 0x124);
            for (int s = 0; s < 2; ++s)
                if (issued_v[s]) mbar_wait(bar(V_FULL + s), (issued_v[s] - 1) & 1, 0x125);
            if (epi) mbar_wait(bar(EPI_FULL), 0, 0x127);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BM, BN, 0, 0);   // qhat x khat^T
            constexpr uint32_t IDESC_DP = idesc_bf16(BM, BN, 0, 0);  // dout x v^T
            constexpr uint32_t IDESC_DQ = idesc_f16(BM, D, 0, 1);    // dS (TMEM) x khat (MN-major)
            auto issue_s = [&](int j) {
                const uint32_t k_s = sb + S::OFF_K + (j % KSTAGES) * S::TBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + tm_s(j & 1), sdesc_sw128(sb + S::OFF_Q + off, 16, 1024),
                             sdesc_sw128(k_s + off, 16, 1024), IDESC_S, kk > 0);
                }
                mma_commit(bar(S_FULL + (j & 1)));
            };
            auto issue_dp = [&](int j) {
                const uint32_t v_s = sb + S::OFF_V + (j & 1) * S::TBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + TM_DP, sdesc_sw128(sb + S::OFF_DO + off, 16, 1024),
                             sdesc_sw128(v_s + off, 16, 1024), IDESC_DP, kk > 0);
                }
                mma_commit(bar(DP_FULL));
                mma_commit(bar(V_EMPTY + (j & 1)));
            };
            auto wait_k = [&](int j) { return mbar_wait(bar(K_FULL + j % KSTAGES), (j / KSTAGES) & 1, 0x221); };
            auto wait_v = [&](int j) { return mbar_wait(bar(V_FULL + (j & 1)), (j >> 1) & 1, 0x222); };
            bool ok = mbar_wait(bar(QD_FULL), 0, 0x220) && wait_k(0);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            if (ok && n_kv > 1) {
                ok = wait_k(1);
                if (ok) {
                    tc_fence_after();
                    issue_s(1);
                }
            }
            if (ok) {
                ok = wait_v(0);
                if (ok) {
                    tc_fence_after();
                    issue_dp(0);
                }
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                // dP_{j+1} as soon as the softmax warps hold dP_j
                if (j + 1 < n_kv) {
                    if (!mbar_wait(bar(DP_READ), j & 1, 0x225) || !wait_v(j + 1)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp(j + 1);
                }
                // dQ += dS_j khat_j, dS_j from TMEM
                if (!mbar_wait(bar(DS_FULL), j & 1, 0x223)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t k_s = sb + S::OFF_K + (j % KSTAGES) * S::TBYTES;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        mma_ts(tmem + TM_DQ, tmem + tm_s(j & 1) + packed_col(kk),
                               sdesc_sw128(k_s + kk * (16 * 128), BN * 128, 1024), IDESC_DQ,
                               (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(K_EMPTY + j % KSTAGES));
                }
                if (j + 2 < n_kv) {
                    if (!wait_k(j + 2)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(j + 2);
                }
            }
            if (ok) mma_commit(bar(DQ_FULL));
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x224);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- P, dS ----
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // query row within the tile = TMEM lane
        const int q = qt * BM + row;
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int cbase = half * 64;  // this warp's key columns
        const float lse2_row = lse2[bh * Tpad + q];  // +inf on padded rows: P = 0
        const float delta_row = delta[bh * Tpad + q];
        bool ok = mbar_wait_warp(bar(QD_FULL), 0, 0x320);
        // dS scale: the largest per-row bound over the tile
        if (half == 0) {
            float dn = 0.f;
            if (ok) {
#pragma unroll 4
                for (int g = 0; g < D / 8; ++g) {
                    float f[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(smem + S::OFF_DO + (g >> 3) * (BM * 128) +
                                                                  sw128_offset(row, g & 7)),
                                  f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dn = fmaf(f[i], f[i], dn);
                }
            }
            float bound = sqrtf(dn) * __uint_as_float(gmax[2]) + fabsf(delta_row);
            if (!(bound < 3.0e38f)) bound = 3.0e38f;  // padded rows: delta 0, dout 0
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) bound = fmaxf(bound, __shfl_xor_sync(0xffffffffu, bound, o));
            if (lane == 0) misc[quarter] = bound;
        }
        named_bar_sync(1, 256);
        const float alpha = ds_scale_for(fmaxf(fmaxf(misc[0], misc[1]), fmaxf(misc[2], misc[3])) * 1.0625f);
        // P feeds only dS here (no product reads it), so it stays in fp32
        // registers, and alpha (a power of two) rides in the exponent:
        // alpha P = exp2(S scale log2e - (lse2 - log2 alpha)).
        const float lse2a = lse2_row - static_cast<float>(ilogbf(alpha));
        for (int j = 0; ok && j < n_kv; ++j) {
            if (!mbar_wait_warp(bar(S_FULL + (j & 1)), (j >> 1) & 1, 0x321)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ts = tmem + lane_base + tm_s(j & 1) + cbase;
            // alpha P over this half's 64 keys.  Tiles with masked entries (the
            // diagonal one: key > query; at the far end of a window: query - key
            // >= W) take their own copy of the loop, so the other tiles pay
            // nothing for the mask.
            float pa[64];
            {
                uint32_t r[2][32];
                tmem_ld32(ts, r[0]);
                tmem_ld32(ts + 32, r[1]);
                tmem_wait_ld();
                const int kt = kt_lo + j;                     // key tile
                const int d0 = (qt - kt) * BN + row - cbase;  // query - key at this thread's first column
                auto exp_tile = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            float p = ex2(fmaf(__uint_as_float(r[c][e]), scale_log2, -lse2a));
                            if constexpr (decltype(masked)::value) {
                                const int dd = d0 - (c * 32 + e);  // visible: 0 <= dd < W
                                if (dd < 0 || dd >= W) p = 0.f;
                            }
                            pa[c * 32 + e] = p;
                        }
                };
                if (kt < qt && (qt - kt) * BM + BM - 1 < W)
                    exp_tile(std::false_type{});
                else
                    exp_tile(std::true_type{});
            }
            if (!mbar_wait_warp(bar(DP_FULL), j & 1, 0x322)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t r[2][32];
                tmem_ld32(tmem + lane_base + TM_DP + cbase, r[0]);
                tmem_ld32(tmem + lane_base + TM_DP + cbase + 32, r[1]);
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive_warp(bar(DP_READ));  // dP_j is in registers: the next dP may overwrite it
                // alpha dS = (alpha P) o (dP - delta) as fp16 pairs
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        const float d0 = pa[c * 32 + e] * (__uint_as_float(r[c][e]) - delta_row);
                        const float d1 = pa[c * 32 + e + 1] * (__uint_as_float(r[c][e + 1]) - delta_row);
                        w[c * 16 + e / 2] = pack_f16x2(d0, d1);
                    }
                // dS over this half's own S columns (already read)
                tmem_st16(ts, w);
                tmem_st16(ts + 16, w + 16);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive_warp(bar(DS_FULL));
        }
        // ------------------------------------------------------ epilogue ----
        // Every barrier below is reached by all 256 threads; the AND-barriers
        // keep their branches uniform even if a wait timed out somewhere.
        bool epi = named_bar_and(1, 256, ok && mbar_wait_warp(bar(DQ_FULL), 0, 0x323));
        epi = named_bar_and(1, 256, epi && mbar_wait_warp(bar(EPI_FULL), 0, 0x324));
        if (epi) tc_fence_after();
        // dq = RMSNorm^T(RoPE^T(dQhat * scale / alpha))
        norm_rope_bwd_stage<D>(epi, tmem + lane_base + TM_DQ, scale / alpha, smem + S::OFF_V + vs_epi * S::TBYTES,
                               smem + S::OFF_K + ks_a * S::TBYTES, smem + S::OFF_K + ks_b * S::TBYTES, row, half,
                               eps, reinterpret_cast<float2*>(smem + S::OFF_DO), smem + S::OFF_Q, 1, 256);
        if (epi) fence_proxy_async_smem();
        named_bar_sync(1, 256);
        if (epi && threadIdx.x == 0) {
            for (int c = 0; c < NC; ++c) tma_store_4d(&tm_dq, sb + S::OFF_Q + c * (BM * 128), c * 64, h, qt * BM, b);
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

}  // namespace bwdq
}  // namespace nc
