// Causal attention backward, key side: dK and dV on sm_103a tensor cores
// (tcgen05 + TMEM + TMA).  The query side (dQ) is a separate kernel
// (nc_bwd_dq.cuh), so that no gradient is accumulated through global
// atomics: each output element is owned by exactly one CTA.
//
// One CTA owns one 128-key tile j of one (batch, key/value head) and walks,
// for each of the G query heads that share that key/value head (grouped-query
// attention; G = 1 without it), the 128-query blocks i >= j that can see it (all of them, or with a sliding
// window W -- query q sees key k when 0 <= q - k < W -- those up to the block
// of the last query within W of the tile's last key).  Everything is computed transposed (keys on the
// TMEM lanes):
//   S^T   = khat_j qhat_i^T                 (M=128 keys, N=128 queries, K=D)
//   P^T   = exp2(S^T * scale*log2e - lse2_i)  recomputed from the forward's
//                                             lse; no running maximum
//   dP^T  = v_j dout_i^T                     (M=128 keys, N=128 queries, K=D)
//   dS^T  = P^T o (dP^T - delta_i)
//   dV_j += P^T dout_i                       (M=128 keys, N=D, K=128 queries)
//   dK_j += dS^T qhat_i                      (same shape)
// and every dS^T block goes, in fp16, to a scratch buffer in HBM too, for
// the query-side kernel's dQ = dS khat (nc_bwd_dq.cuh): dS is formed once.
// Tensor memory (512 columns): S^T (128) is overwritten in place by the
// bf16 P^T and dP^T (128) by the fp16 dS^T; both are then read from TMEM as
// the A operands of the dV and dK products.  dV and dK take D columns each.
// Only tensor memory and registers hold the per-block intermediates: the
// shared-memory traffic per block is the operand tiles and the SS products'
// reads (about 260 KB against 2048 cycles of tensor work), close to what
// shared memory delivers, so nothing else goes through it.  (Measured: P^T
// through a shared-memory tile, which would let S^T(i+1) start before dV(i),
// made the kernel 11% slower.)
//
// Issue order of the MMA thread for block i (one thread's MMAs execute in
// issue order, so a product that overwrites TMEM another one reads may
// follow it directly):
//   [P^T(i) in TMEM]   dV(i), S^T(i+1)      while the softmax warps make dS(i)
//   [dS^T(i) in TMEM]  dK(i), dP^T(i+1)     while they make P(i+1)
// so each softmax phase overlaps two products.
//
// Roles: warps 0-7 P and dS (warp w: TMEM lane quarter w%4 = 32 key rows,
// query half w/4 = 64 columns), warp 8 TMA, warp 9 MMA.  At the end the same
// eight warps stage dv and then dk (through the RoPE transpose and the RMSNorm
// backward, two threads per key row) in shared memory, and both tiles leave
// through TMA stores.  The raw k rows and RoPE table rows that dk needs are
// prefetched during the last query block: the table over the query stage the
// last block does not use, the raw rows over the khat tile once the last
// product that reads khat and v is done.
//
// Operand types: the score side (qhat, khat, dS) is IEEE fp16, the value
// side (P, v, dout) bf16; tcgen05 wants A and B of one product in one type.
// dS is stored as alpha * dS in fp16, alpha the call's one power of two from
// the bound of ds_scale_global (|alpha dS| <= 2^14, while small gradients
// keep fp16's full precision); dK is multiplied by 1/alpha on the way out,
// and the query-side kernel undoes the same alpha on dQ.
#pragma once

#include "nc_common.cuh"
#include <type_traits>
#include "nc_bwd_dq.cuh"
#include "nc_normrope_bwd.cuh"

namespace nc {
namespace bwd {

constexpr int BN = 128;  // keys per CTA
constexpr int BM = 128;  // queries per block
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;
constexpr int SMEM_LIMIT = 232448;  // 227 KB opt-in per block

enum Bar {
    KV_FULL = 0,
    QF = 1,       // +stage: qhat_i, dout_i, lse2_i, delta_i landed
    QE = 3,       // +stage: stage free again
    S_FULL = 5,   // S^T in TMEM
    P_FULL = 6,   // softmax wrote P^T over S^T
    DP_FULL = 7,  // dP^T in TMEM
    DS_FULL = 8,  // softmax wrote dS^T over dP^T
    DKV_FULL = 9,
    MMA_DONE = 10,
    EPI_FULL = 11,  // raw k tile and RoPE table tile staged for the dk epilogue
    KV_FREE = 12,   // the last products reading khat and v are done
    NUM_BARS = 13
};

template <int D>
struct Smem {
    static constexpr int KBYTES = BN * D * 2;  // khat or v tile
    static constexpr int QBYTES = BM * D * 2;  // qhat or dout stage
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KBYTES;
    static constexpr int OFF_Q = OFF_V + KBYTES;        // 2 stages
    static constexpr int OFF_DO = OFF_Q + 2 * QBYTES;   // 2 stages
    static constexpr int OFF_L = OFF_DO + 2 * QBYTES;   // 2 stages x BM fp32 (lse * log2e)
    static constexpr int OFF_DL = OFF_L + 2 * BM * 4;   // 2 stages x BM fp32 (delta)
    static constexpr int OFF_BAR = OFF_DL + 2 * BM * 4;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TSLOT + 16;
    static constexpr int ALLOC = (BYTES + 1024 < SMEM_LIMIT) ? BYTES + 1024 : SMEM_LIMIT;
    // epilogue: the raw k tile over the khat tile, the RoPE table tile (fp32
    // [128][D]) over the qhat and dout halves of the stage the last block
    // does not use; dv staged over the v tile, dk over the last block's qhat
    // stage, the row-half exchange over its dout stage
    static constexpr int XBYTES = BN * D * 2;
    static constexpr int CBYTES = BN * D * 4;
    static_assert(BYTES <= SMEM_LIMIT, "backward tiles exceed shared memory");
    static_assert(XBYTES <= KBYTES && CBYTES == 2 * QBYTES && 2 * BN * 8 <= QBYTES, "epilogue tiles exceed the stages");
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;
// dP^T, then dS^T: the query half h of the packed fp16 pairs sits in columns
// [64h, 64h + 32), i.e. inside the dP^T columns its own warps read.
constexpr uint32_t TM_DP = 128;
constexpr uint32_t TM_DV = 256;  // D columns; dK follows at TM_DV + D

// TMEM column of the packed pair holding queries (2c, 2c+1) of K-step kk
// (16 queries): half kk/4, offset 8 columns per step inside the half.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8); }

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_kraw, const __grid_constant__ CUtensorMap tm_tab,
                         const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                         const float* __restrict__ lse2, const float* __restrict__ delta,
                         const unsigned int* __restrict__ gmax, __half* __restrict__ ds_out, int T, int H, int B,
                         int Tpad, int group, float scale, float scale_log2, float eps, int W, int G) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    constexpr uint32_t TM_DK = TM_DV + D;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x1f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped (b, key/value head) order, longest walks (key tile 0) first in a group
    const int nqb = (T + BM - 1) / BM;
    const int Hkv = H / G;
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * Hkv, nqb, group);
    const int kt = tc.rank;
    const int b = tc.bh / Hkv, hk = tc.bh % Hkv;
    const int qb0 = kt;  // BM == BN: the diagonal query block
    const int qb_last = min(nqb - 1, (kt * BN + BN - 1 + W - 1) / BM);  // W >= 2^30 means no window
    const int n_it = qb_last - qb0 + 1;  // query blocks per query head
    const int n_tot = G * n_it;          // blocks of the whole walk: head hk*G + itf / n_it, block itf % n_it
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    const int sp = n_tot & 1;             // query stage the last block does not use
    const int st_last = (n_tot - 1) & 1;  // the last block's query stage

    if (threadIdx.x == 0) {
        mbar_init(bar(KV_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(QF + s), 1);
            mbar_init(bar(QE + s), 1);
        }
        mbar_init(bar(S_FULL), 1);
        mbar_init(bar(P_FULL), 8);   // one arrival per softmax warp
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DS_FULL), 8);
        mbar_init(bar(DKV_FULL), 1);
        mbar_init(bar(MMA_DONE), 1);
        mbar_init(bar(EPI_FULL), 1);
        mbar_init(bar(KV_FREE), 1);
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
            int issued[2] = {0, 0};
            mbar_expect_tx(bar(KV_FULL), 2 * S::KBYTES);
            for (int c = 0; c < NC; ++c) {
                tma_load_4d(sb + S::OFF_K + c * (BN * 128), &tm_k, c * 64, hk, kt * BN, b, bar(KV_FULL));
                tma_load_4d(sb + S::OFF_V + c * (BN * 128), &tm_v, c * 64, hk, kt * BN, b, bar(KV_FULL));
            }
            for (int itf = 0; itf < n_tot; ++itf) {
                const int st = itf & 1, use = itf >> 1;
                if (itf >= 2 && !mbar_wait(bar(QE + st), (use - 1) & 1, 0x111)) break;
                const int h = hk * G + itf / n_it;  // query head of this block
                const long long bh = static_cast<long long>(b) * H + h;
                const int q0 = (qb0 + itf % n_it) * BM;
                mbar_expect_tx(bar(QF + st), 2 * S::QBYTES + 2 * BM * 4);
                for (int c = 0; c < NC; ++c) {
                    tma_load_4d(sb + S::OFF_Q + st * S::QBYTES + c * (BM * 128), &tm_q, c * 64, h, q0, b,
                                bar(QF + st));
                    tma_load_4d(sb + S::OFF_DO + st * S::QBYTES + c * (BM * 128), &tm_do, c * 64, h, q0, b,
                                bar(QF + st));
                }
                bulk_load(sb + S::OFF_L + st * BM * 4, lse2 + bh * Tpad + q0, BM * 4, bar(QF + st));
                bulk_load(sb + S::OFF_DL + st * BM * 4, delta + bh * Tpad + q0, BM * 4, bar(QF + st));
                ++issued[st];
            }
            // dk epilogue tiles, each as soon as its space is free: the RoPE
            // table rows over stage sp (free once block n_tot-2 is done), the
            // raw k rows over the khat tile
            mbar_expect_tx(bar(EPI_FULL), S::XBYTES + S::CBYTES);
            bool epi = n_tot < 2 || mbar_wait(bar(QE + sp), ((n_tot - 2) >> 1) & 1, 0x117);
            if (epi) {
                for (int c = 0; c < D / 32; ++c) {
                    const uint32_t dst = c < NC ? S::OFF_Q + sp * S::QBYTES + c * (BN * 128)
                                                : S::OFF_DO + sp * S::QBYTES + (c - NC) * (BN * 128);
                    tma_load_2d(sb + dst, &tm_tab, c * 32, kt * BN, bar(EPI_FULL));
                }
            }
            epi = epi && mbar_wait(bar(KV_FREE), 0, 0x118);
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_K + c * (BN * 128), &tm_kraw, c * 64, hk, kt * BN, b, bar(EPI_FULL));
            }
            // never leave the CTA with a bulk copy still in flight
            mbar_wait(bar(KV_FULL), 0, 0x112);
            for (int s = 0; s < 2; ++s)
                if (issued[s]) mbar_wait(bar(QF + s), (issued[s] - 1) & 1, 0x113);
            if (epi) mbar_wait(bar(EPI_FULL), 0, 0x115);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BN, BM, 0, 0);   // khat x qhat^T
            constexpr uint32_t IDESC_DP = idesc_bf16(BN, BM, 0, 0);  // v x dout^T
            constexpr uint32_t IDESC_DV = idesc_bf16(BN, D, 0, 1);   // P^T (TMEM) x dout (MN-major)
            constexpr uint32_t IDESC_DK = idesc_f16(BN, D, 0, 1);    // dS^T (TMEM) x qhat (MN-major)
            auto issue_s = [&](int st) {
                const uint32_t q_s = sb + S::OFF_Q + st * S::QBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                    const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + TM_S, sdesc_sw128(sb + S::OFF_K + ka, 16, 1024), sdesc_sw128(q_s + qa, 16, 1024),
                             IDESC_S, kk > 0);
                }
                mma_commit(bar(S_FULL));
            };
            auto issue_dp = [&](int st) {
                const uint32_t do_s = sb + S::OFF_DO + st * S::QBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                    const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + TM_DP, sdesc_sw128(sb + S::OFF_V + ka, 16, 1024),
                             sdesc_sw128(do_s + qa, 16, 1024), IDESC_DP, kk > 0);
                }
                mma_commit(bar(DP_FULL));
            };
            bool ok = mbar_wait(bar(KV_FULL), 0, 0x211) && mbar_wait(bar(QF + 0), 0, 0x212);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                issue_dp(0);
                if (n_tot == 1) mma_commit(bar(KV_FREE));
            }
            for (int it = 0; ok && it < n_tot; ++it) {
                const int st = it & 1;
                const bool more = it + 1 < n_tot;
                if (!mbar_wait(bar(P_FULL), it & 1, 0x213)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t do_s = sb + S::OFF_DO + st * S::QBYTES;
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts(tmem + TM_DV, tmem + TM_S + packed_col(kk),
                               sdesc_sw128(do_s + kk * (16 * 128), BM * 128, 1024), IDESC_DV,
                               (it > 0 || kk > 0) ? 1u : 0u);
                }
                if (more) {
                    if (!mbar_wait(bar(QF + (st ^ 1)), ((it + 1) >> 1) & 1, 0x214)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(st ^ 1);
                }
                // dK += dS^T qhat, then dP^T of the next block over dS^T
                if (!mbar_wait(bar(DS_FULL), it & 1, 0x215)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t q_s = sb + S::OFF_Q + st * S::QBYTES;
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts(tmem + TM_DK, tmem + TM_DP + packed_col(kk),
                               sdesc_sw128(q_s + kk * (16 * 128), BM * 128, 1024), IDESC_DK,
                               (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(QE + st));
                }
                if (more) {
                    issue_dp(st ^ 1);
                    if (it + 2 == n_tot) mma_commit(bar(KV_FREE));  // that was the last S^T and dP^T
                }
            }
            if (ok) mma_commit(bar(DKV_FULL));
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x216);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------- P, dS ----
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // key row within the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int cbase = half * 64;  // this warp's query columns
        bool ok = true;
        const float alpha = ds_scale_global(gmax);
        const uint32_t ts = tmem + lane_base + TM_S, tdp = tmem + lane_base + TM_DP;
        for (int it = 0; ok && it < n_tot; ++it) {
            const int st = it & 1, use = it >> 1;
            if (!mbar_wait_warp(bar(QF + st), use & 1, 0x311)) { ok = false; break; }
            if (!mbar_wait_warp(bar(S_FULL), it & 1, 0x312)) { ok = false; break; }
            tc_fence_after();
            const float4* l2 = reinterpret_cast<const float4*>(smem + S::OFF_L + st * BM * 4 + cbase * 4);
            const float4* dl = reinterpret_cast<const float4*>(smem + S::OFF_DL + st * BM * 4 + cbase * 4);
            // P^T = exp2(S^T scale log2e - lse2) as bf16 pairs over this half's S^T
            // columns.  Blocks with masked entries (the diagonal one: query <
            // key; at the far end of a window: query - key >= W) take their
            // own copy of the loop, so the other blocks pay nothing for the mask.
            const int qb = qb0 + it % n_it;  // query block of this step
            const int d0 = (qb - kt) * BM + cbase - row;  // query - key at this thread's first column
            uint32_t pk[32];
            {
                uint32_t r[2][32];
                tmem_ld32(ts + cbase, r[0]);
                tmem_ld32(ts + cbase + 32, r[1]);
                tmem_wait_ld();
                auto exp_block = [&](auto masked) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 l4 = l2[c * 8 + e4];
                            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                            float p[4];
#pragma unroll
                            for (int i = 0; i < 4; i += 2) {
                                const float2 x2 = ffma2(make_float2(__uint_as_float(r[c][e4 * 4 + i]),
                                                                    __uint_as_float(r[c][e4 * 4 + i + 1])),
                                                        make_float2(scale_log2, scale_log2),
                                                        make_float2(-lv[i], -lv[i + 1]));
                                p[i] = ex2(x2.x);
                                p[i + 1] = ex2(x2.y);
                            }
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                if constexpr (decltype(masked)::value) {
                                    const int dd = d0 + c * 32 + e4 * 4 + i;  // visible: 0 <= dd < W
                                    if (dd < 0 || dd >= W) p[i] = 0.f;
                                }
                            }
                            pk[c * 16 + e4 * 2] = pack_bf16x2(p[0], p[1]);
                            pk[c * 16 + e4 * 2 + 1] = pack_bf16x2(p[2], p[3]);
                        }
                    }
                };
                if (qb > kt && (qb - kt) * BM + BM - 1 < W)
                    exp_block(std::false_type{});
                else
                    exp_block(std::true_type{});
            }
            // P^T into the shared-memory tile (K-major, 128-byte swizzled: this
            // thread's 64 queries of key row `row`) once dV(it-1) has read it
            tmem_st16(ts + cbase, pk);
            tmem_st16(ts + cbase + 16, pk + 16);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive_warp(bar(P_FULL));
            // dS^T = P^T o (dP^T - delta) * alpha as fp16 pairs over this half's dP^T columns
            if (!mbar_wait_warp(bar(DP_FULL), it & 1, 0x313)) { ok = false; break; }
            tc_fence_after();
            {
                uint32_t r[2][32];
                tmem_ld32(tdp + cbase, r[0]);
                tmem_ld32(tdp + cbase + 32, r[1]);
                tmem_wait_ld();
                uint32_t w[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) {
                        const float4 d4 = dl[c * 8 + e4];
                        const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                        float ds[4];
#pragma unroll
                        for (int i = 0; i < 4; i += 2) {
                            // alpha p (dP - delta), two columns per paired instruction
                            const uint32_t pw = pk[c * 16 + e4 * 2 + (i >> 1)];
                            const float2 p2 = make_float2(__uint_as_float(pw << 16), __uint_as_float(pw & 0xffff0000u));
                            const float2 t2 = ffma2(make_float2(1.f, 1.f),
                                                    make_float2(__uint_as_float(r[c][e4 * 4 + i]),
                                                                __uint_as_float(r[c][e4 * 4 + i + 1])),
                                                    make_float2(-dv4[i], -dv4[i + 1]));
                            const float2 d2 = fmul2(fmul2(make_float2(alpha, alpha), p2), t2);
                            ds[i] = d2.x;
                            ds[i + 1] = d2.y;
                        }
                        w[c * 16 + e4 * 2] = pack_f16x2(ds[0], ds[1]);
                        w[c * 16 + e4 * 2 + 1] = pack_f16x2(ds[2], ds[3]);
                    }
                }
                tmem_st16(tdp + cbase, w);
                tmem_st16(tdp + cbase + 16, w + 16);
                // the same fp16 alpha dS^T row half into the scratch block
                // (query tile qb, key tile kt) of query head h: 8 chunks of 8
                // queries, each a 16-byte store; in the scratch layout
                // (bwdq::ds_offset) the 32 key rows of the warp are 32
                // consecutive 16-byte slots, so every warp store writes 512
                // contiguous bytes.  (The earlier [key][query] layout needed a
                // 4-lane shuffle transpose of the chunks to coalesce.)
                const int h = hk * G + it / n_it;
                __half* blk = ds_out + bwdq::ds_block(static_cast<long long>(b) * H + h, nqb, qb, kt) * (BN * BM);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    __half* p = blk + bwdq::ds_offset(row, cbase + 8 * g);
                    if (NC_IN_RANGE(p, 16, 0x412))
                        *reinterpret_cast<uint4*>(p) = make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive_warp(bar(DS_FULL));
        }
        // ------------------------------------------------------ epilogue ----
        // Every barrier below is reached by all 256 threads; the AND-barriers
        // keep their branches uniform even if a wait timed out somewhere.
        const bool epi = named_bar_and(1, 256, ok && mbar_wait_warp(bar(DKV_FULL), 0, 0x315));
        uint8_t* dv_stage = smem + S::OFF_V;
        uint8_t* dk_stage = smem + S::OFF_Q + st_last * S::QBYTES;
        float2* xch = reinterpret_cast<float2*>(smem + S::OFF_DO + st_last * S::QBYTES);
        if (epi) {
            tc_fence_after();
            stage_acc_bf16<D / 2>(tmem + lane_base + TM_DV, 1.f, dv_stage, row, half * (D / 2));
            fence_proxy_async_smem();
        }
        const bool epi_dk = named_bar_and(1, 256, epi && mbar_wait_warp(bar(EPI_FULL), 0, 0x316));
        if (epi && threadIdx.x == 0) {
            for (int c = 0; c < NC; ++c) tma_store_4d(&tm_dv, sb + S::OFF_V + c * (BN * 128), c * 64, hk, kt * BN, b);
            bulk_commit();
        }
        // dk = RMSNorm^T(RoPE^T(dKhat * scale / alpha))
        norm_rope_bwd_stage<D>(epi_dk, tmem + lane_base + TM_DK, scale / alpha, smem + S::OFF_K,
                               smem + S::OFF_Q + sp * S::QBYTES, smem + S::OFF_DO + sp * S::QBYTES, row, half, eps,
                               xch, dk_stage, 1, 256);
        if (epi_dk) fence_proxy_async_smem();
        named_bar_sync(1, 256);
        if (threadIdx.x == 0) {
            if (epi_dk) {
                for (int c = 0; c < NC; ++c)
                    tma_store_4d(&tm_dk, smem_u32(dk_stage) + c * (BN * 128), c * 64, hk, kt * BN, b);
                bulk_commit();
            }
            bulk_wait_read_all();  // the staged tiles stay valid until the stores have read them
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace bwd
}  // namespace nc
