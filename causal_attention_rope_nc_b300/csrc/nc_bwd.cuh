// Causal attention backward on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA owns one 128-key tile j of one (batch, head) and walks the
// 128-query blocks i >= j.  Everything is computed transposed (keys on the
// TMEM lanes):
//   S^T   = khat_j qhat_i^T                 (M=128 keys, N=128 queries, K=D)
//   P^T   = exp2(S^T * scale*log2e - lse2_i)  recomputed from the forward's
//                                             lse; no running maximum
//   dP^T  = v_j dout_i^T                     (M=128 keys, N=128 queries, K=D)
//   dS^T  = P^T o (dP^T - delta_i)
//   dV_j += P^T dout_i                       (M=128 keys, N=D, K=128; P^T
//                                             read from TMEM)
//   dK_j += dS^T qhat_i                      (same shape, dS^T from smem)
//   dQ_i^T = khat_j^T dS^T                   (M=D, N=128 queries, K=128 keys)
// dV and dK accumulate in TMEM for the whole walk.  dQ_i^T is drained from
// TMEM after every block and added (fp32 reductions, already scaled by
// 1/sqrt(D)) into a [B,T,H,D] accumulator that a later pass turns into dq.
// At the end the CTA writes dv and, through the RoPE transpose and the
// RMSNorm backward, dk.
//
// Tensor memory (512 columns): S^T (128) is overwritten in place by the
// bf16 P^T that the dV product reads as its A operand; dP^T (128) is
// overwritten by dQ^T once the softmax warps have read it; dV and dK take D
// columns each.
//
// Issue order of the MMA thread for block i (the tensor pipe runs in order):
//   [P^T(i) in TMEM]       dV(i)
//   [dV(i) done]           S^T(i+1)      while the softmax warps compute dS(i)
//   [dS^T(i) in smem]      dQ^T(i), dK(i)
//   [dQ^T(i) drained]      dP^T(i+1)
// so that S^T(i+1) is ready when the softmax warps finish dS(i), their P(i+1)
// overlaps dQ^T(i), dK(i) and dP^T(i+1), and the tensor pipe never waits on a
// tile load of a later block.
//
// Roles: warps 0-3 P and dS (thread = key row = TMEM lane, all 128 query
// columns; the row's packed P stays in registers between the two phases),
// warps 4-7 drain dQ^T (thread = head-dim lane) so that the fp32 reductions,
// the slowest traffic of the kernel, overlap everything else; warp 8 TMA,
// warp 9 MMA.  At the end warps 0-3 write dv and warps 4-7 dk.
//
// Operand types: the score side (qhat, khat, dS) is IEEE fp16, the value
// side (P, v, dout) bf16; tcgen05 wants A and B of one product in one type.
// dS is stored as alpha * dS in fp16 with a per-CTA power of two alpha chosen
// from a rigorous bound,
//   |dS_ij| = P_ij |<dout_i, v_j> - <dout_i, out_i>|
//          <= max_i ||dout_i|| * (max_{j in tile} ||v_j|| + max_i ||out_i||),
// so that |alpha dS| <= 2^14 (fp16 overflows at 65504) while small gradients
// keep fp16's full precision; dK and dQ are multiplied by 1/alpha on the
// way out.
#pragma once

#include "nc_common.cuh"

namespace nc {
namespace bwd {

constexpr int BN = 128;  // keys per CTA
constexpr int BM = 128;  // queries per block
constexpr int WARP_DRAIN = 4;  // 4..7
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;
constexpr int SMEM_LIMIT = 232448;  // 227 KB opt-in per block

enum Bar {
    KV_FULL = 0,
    QF = 1,        // +stage: qhat_i, dout_i, lse2_i, delta_i landed
    QE = 3,        // +stage: stage free again
    S_FULL = 5,    // S^T in TMEM
    P_FULL = 6,    // softmax wrote P^T over S^T
    TMS_FREE = 7,  // dV finished reading P^T
    DP_FULL = 8,   // dP^T in TMEM
    DS_FULL = 9,   // dS^T in smem, dP^T read
    DS_FREE = 10,  // dK and dQ^T finished reading dS^T
    DQ_FULL = 11,  // dQ^T in TMEM
    DQ_FREE = 12,  // dQ^T drained
    DKV_FULL = 13,
    MMA_DONE = 14,
    NUM_BARS = 15
};

template <int D>
struct Smem {
    static constexpr int KBYTES = BN * D * 2;   // khat or v tile
    static constexpr int QBYTES = BM * D * 2;   // qhat or dout stage
    static constexpr int DSBYTES = BN * BM * 2;  // dS^T
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KBYTES;
    static constexpr int OFF_Q = OFF_V + KBYTES;       // 2 stages
    static constexpr int OFF_DO = OFF_Q + 2 * QBYTES;  // 2 stages
    static constexpr int OFF_DS = OFF_DO + 2 * QBYTES;  // [128 keys][128 q] fp16, SW128, 2 spans of 64 q
    static constexpr int OFF_L = OFF_DS + DSBYTES;      // 2 stages x BM fp32 (lse * log2e)
    static constexpr int OFF_DL = OFF_L + 2 * BM * 4;   // 2 stages x BM fp32 (delta)
    static constexpr int OFF_BAR = OFF_DL + 2 * BM * 4;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_MISC = OFF_TSLOT + 16;  // 4 warp maxima of ||v_j||^2
    static constexpr int BYTES = OFF_MISC + 32;
    static constexpr int ALLOC = (BYTES + 1024 < SMEM_LIMIT) ? BYTES + 1024 : SMEM_LIMIT;
    // dk epilogue: u = RoPE^T(dKhat) rows staged over the (then idle) qhat and
    // dout stages, 16 bytes of padding per row against bank conflicts
    static constexpr int U_STRIDE = D * 4 + 16;
    static_assert(BYTES <= SMEM_LIMIT, "backward tiles exceed shared memory");
    static_assert(BN * U_STRIDE <= 4 * QBYTES, "dk staging exceeds the qhat/dout stages");
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // S^T, then P^T (bf16 pairs) in columns [0, 64)
constexpr uint32_t TM_DP = 128;  // dP^T, then dQ^T
constexpr uint32_t TM_DV = 256;  // D columns; dK follows at TM_DV + D

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float* __restrict__ lse2, const float* __restrict__ delta, float* __restrict__ dq_acc,
                    const unsigned int* __restrict__ gmax, const __nv_bfloat16* __restrict__ k_raw,
                    const float2* __restrict__ tab, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                    int T, int H, int B, int Tpad, int group, float scale, float scale_log2, float eps) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    constexpr uint32_t TM_DK = TM_DV + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x1f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped (b, h) order, longest walks (key tile 0) first in a group
    const int nqb = (T + BM - 1) / BM;
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * H, nqb, group);
    const int kt = tc.rank;
    const int b = tc.bh / H, h = tc.bh % H;
    const int qb0 = kt;  // BM == BN: the diagonal query block
    const int n_it = nqb - qb0;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    float* misc = reinterpret_cast<float*>(smem + S::OFF_MISC);
    const long long bh = static_cast<long long>(b) * H + h;

    if (threadIdx.x == 0) {
        mbar_init(bar(KV_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(QF + s), 1);
            mbar_init(bar(QE + s), 1);
        }
        mbar_init(bar(S_FULL), 1);
        mbar_init(bar(P_FULL), 128);
        mbar_init(bar(TMS_FREE), 1);
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DS_FULL), 128);
        mbar_init(bar(DS_FREE), 1);
        mbar_init(bar(DQ_FULL), 1);
        mbar_init(bar(DQ_FREE), 128);
        mbar_init(bar(DKV_FULL), 1);
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
            int issued[2] = {0, 0};
            mbar_expect_tx(bar(KV_FULL), 2 * S::KBYTES);
            for (int c = 0; c < NC; ++c) {
                tma_load_4d(sb + S::OFF_K + c * (BN * 128), &tm_k, c * 64, h, kt * BN, b, bar(KV_FULL));
                tma_load_4d(sb + S::OFF_V + c * (BN * 128), &tm_v, c * 64, h, kt * BN, b, bar(KV_FULL));
            }
            for (int it = 0; it < n_it; ++it) {
                const int st = it & 1, use = it >> 1;
                if (it >= 2 && !mbar_wait(bar(QE + st), (use - 1) & 1, 0x111)) break;
                const int q0 = (qb0 + it) * BM;
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
            // never leave the CTA with a bulk copy still in flight
            mbar_wait(bar(KV_FULL), 0, 0x112);
            for (int s = 0; s < 2; ++s)
                if (issued[s]) mbar_wait(bar(QF + s), (issued[s] - 1) & 1, 0x113);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BN, BM, 0, 0);    // khat x qhat^T
            constexpr uint32_t IDESC_DP = idesc_bf16(BN, BM, 0, 0);  // v x dout^T
            constexpr uint32_t IDESC_DV = idesc_bf16(BN, D, 0, 1);   // P^T (TMEM) x dout (MN-major)
            constexpr uint32_t IDESC_DK = idesc_f16(BN, D, 0, 1);    // dS^T (K-major) x qhat (MN-major)
            constexpr uint32_t IDESC_DQ = idesc_f16(128, BM, 1, 1);  // khat^T (MN-major) x dS^T (MN-major)
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
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it & 1;
                const bool more = it + 1 < n_it;
                // dV += P^T dout, P^T straight from TMEM (packed columns [0, 64))
                if (!mbar_wait(bar(P_FULL), it & 1, 0x213)) { ok = false; break; }
                tc_fence_after();
                {
                    const uint32_t do_s = sb + S::OFF_DO + st * S::QBYTES;
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_ts(tmem + TM_DV, tmem + TM_S + kk * 8, sdesc_sw128(do_s + kk * (16 * 128), BM * 128, 1024),
                               IDESC_DV, (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(TMS_FREE));
                }
                // S^T of the next block, once dV has read P^T
                if (more) {
                    if (!mbar_wait(bar(QF + (st ^ 1)), ((it + 1) >> 1) & 1, 0x214)) { ok = false; break; }
                    if (!mbar_wait(bar(TMS_FREE), it & 1, 0x215)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(st ^ 1);
                }
                // dQ^T = khat^T dS^T into the dP^T columns, then dK += dS^T qhat
                if (!mbar_wait(bar(DS_FULL), it & 1, 0x216)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16(tmem + TM_DP, sdesc_sw128(sb + S::OFF_K + kk * (16 * 128), BN * 128, 1024),
                             sdesc_sw128(sb + S::OFF_DS + kk * (16 * 128), BN * 128, 1024), IDESC_DQ, kk > 0);
                mma_commit(bar(DQ_FULL));
                {
                    const uint32_t q_s = sb + S::OFF_Q + st * S::QBYTES;
#pragma unroll
                    for (int kk = 0; kk < BM / 16; ++kk)
                        mma_bf16(tmem + TM_DK,
                                 sdesc_sw128(sb + S::OFF_DS + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16, 1024),
                                 sdesc_sw128(q_s + kk * (16 * 128), BM * 128, 1024), IDESC_DK,
                                 (it > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(DS_FREE));
                    mma_commit(bar(QE + st));
                }
                // dP^T of the next block, once dQ^T has been drained
                if (more) {
                    if (!mbar_wait(bar(DQ_FREE), it & 1, 0x217)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp(st ^ 1);
                }
            }
            if (ok) mma_commit(bar(DKV_FULL));
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x218);
        }
        __syncwarp();
    } else if (warp < WARP_DRAIN) {
        // ------------------------------------------------------- P, dS ----
        const int row = warp * 32 + lane;  // key row within the tile = TMEM lane
        const int key = kt * BN + row;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        bool ok = mbar_wait(bar(KV_FULL), 0, 0x310);
        // dS scale alpha (see the header comment): max ||v_j|| over this tile
        // from shared memory, the global row-norm maxima from the preprocess.
        float alpha = 1.f;
        {
            float vn = 0.f;
            if (ok) {
#pragma unroll 4
                for (int g = 0; g < D / 8; ++g) {
                    const uint4 u = *reinterpret_cast<const uint4*>(smem + S::OFF_V + (g >> 3) * (BN * 128) +
                                                                    sw128_offset(row, g & 7));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = unpack_bf16x2(w[i]);
                        vn = fmaf(f.x, f.x, fmaf(f.y, f.y, vn));
                    }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vn = fmaxf(vn, __shfl_xor_sync(0xffffffffu, vn, o));
            if (lane == 0) misc[warp] = vn;
            named_bar_sync(2, 128);  // the four softmax warps
            const float vmax = sqrtf(fmaxf(fmaxf(misc[0], misc[1]), fmaxf(misc[2], misc[3])));
            const float bound = __uint_as_float(gmax[0]) * (vmax + __uint_as_float(gmax[1])) * 1.0625f;
            if (bound > 0.f && bound < 3.0e38f) {
                int e = static_cast<int>(floorf(log2f(16384.f / bound)));
                e = max(-120, min(120, e));
                alpha = ldexpf(1.f, e);
            }
            if (threadIdx.x == 0) misc[4] = alpha;
            named_bar_sync(1, 256);  // hand alpha to the drain warps
        }
        for (int it = 0; ok && it < n_it; ++it) {
            const int st = it & 1, use = it >> 1;
            const int q0 = (qb0 + it) * BM;
            if (!mbar_wait(bar(QF + st), use & 1, 0x311)) { ok = false; break; }
            if (!mbar_wait(bar(S_FULL), it & 1, 0x312)) { ok = false; break; }
            tc_fence_after();
            const float4* l2 = reinterpret_cast<const float4*>(smem + S::OFF_L + st * BM * 4);
            const float4* dl = reinterpret_cast<const float4*>(smem + S::OFF_DL + st * BM * 4);
            const bool diag = (it == 0);  // only the diagonal block has masked entries
            // P^T = exp2(S^T scale log2e - lse2) as bf16 pairs, written over S^T
            // (chunk c writes packed columns [16c, 16c+16), already read)
            uint32_t pk[BM / 2];
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_S + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 l4 = l2[c * 8 + e4];
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                    float p[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int qi = c * 32 + e4 * 4 + i;
                        const float x = fmaf(__uint_as_float(r[e4 * 4 + i]), scale_log2, -lv[i]);
                        p[i] = (diag && q0 + qi < key) ? 0.f : ex2(x);
                    }
                    pk[c * 16 + e4 * 2] = pack_bf16x2(p[0], p[1]);
                    pk[c * 16 + e4 * 2 + 1] = pack_bf16x2(p[2], p[3]);
                }
                tmem_st16(tmem + lane_base + TM_S + c * 16, pk + c * 16);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(P_FULL));
            // dS^T = P^T o (dP^T - delta) * alpha, fp16 into shared memory
            if (!mbar_wait(bar(DP_FULL), it & 1, 0x313)) { ok = false; break; }
            if (it >= 1 && !mbar_wait(bar(DS_FREE), (it - 1) & 1, 0x314)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_DP + c * 32, r);
                tmem_wait_ld();
                uint32_t w[16];
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 d4 = dl[c * 8 + e4];
                    const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                    float ds[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t pw = pk[c * 16 + e4 * 2 + (i >> 1)];
                        const float p = __uint_as_float((i & 1) ? (pw & 0xffff0000u) : (pw << 16));
                        ds[i] = alpha * p * (__uint_as_float(r[e4 * 4 + i]) - dv4[i]);
                    }
                    w[e4 * 2] = pack_f16x2(ds[0], ds[1]);
                    w[e4 * 2 + 1] = pack_f16x2(ds[2], ds[3]);
                }
                // queries c*32 .. c*32+31 live in span c/2, 16-byte chunks (c%2)*4 ..
                const uint32_t ds_row = sb + S::OFF_DS + (c >> 1) * (BN * 128);
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    st_shared_v4(ds_row + sw128_offset(row, (c & 1) * 4 + g), w[4 * g], w[4 * g + 1], w[4 * g + 2],
                                 w[4 * g + 3]);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(bar(DS_FULL));
        }
        // dv: one key row per thread
        if (ok && mbar_wait(bar(DKV_FULL), 0, 0x315)) {
            tc_fence_after();
            const bool valid = key < T;
            __nv_bfloat16* vrow = dv + ((static_cast<long long>(b) * T + key) * H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_DV + c * 32, r);
                tmem_wait_ld();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(vrow + c * 32);
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        dst[g] = make_uint4(
                            pack_bf16x2(__uint_as_float(r[8 * g]), __uint_as_float(r[8 * g + 1])),
                            pack_bf16x2(__uint_as_float(r[8 * g + 2]), __uint_as_float(r[8 * g + 3])),
                            pack_bf16x2(__uint_as_float(r[8 * g + 4]), __uint_as_float(r[8 * g + 5])),
                            pack_bf16x2(__uint_as_float(r[8 * g + 6]), __uint_as_float(r[8 * g + 7])));
                }
            }
        }
    } else if (warp < WARP_TMA) {
        // --------------------------------------- dQ drain + dk epilogue -----
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int row = quarter * 32 + lane;  // dQ^T lane = head-dim index; dk: key row
        named_bar_sync(1, 256);               // alpha from the softmax warps
        // dS was stored times alpha: undo it together with the 1/sqrt(D) scale
        const float out_scale = scale / misc[4];
        const long long rstride = static_cast<long long>(H) * D;  // one token in [B,T,H,D]
        bool ok = true;
        for (int it = 0; it < n_it; ++it) {
            const int q0 = (qb0 + it) * BM;
            if (!mbar_wait(bar(DQ_FULL), it & 1, 0x411)) { ok = false; break; }
            tc_fence_after();
            uint32_t r[BM / 32][32];
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) tmem_ld32(tmem + lane_base + TM_DP + c * 32, r[c]);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(DQ_FREE));
            if (row < D) {
                float* base = dq_acc + ((static_cast<long long>(b) * T + q0) * H + h) * D + row;
#pragma unroll
                for (int c = 0; c < BM / 32; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (q0 + c * 32 + e < T)
                            red_add_f32(base + (c * 32 + e) * rstride, __uint_as_float(r[c][e]) * out_scale);
            }
        }
        // dk = RMSNorm^T(RoPE^T(dKhat * scale / alpha)), thread = key row
        if (ok && mbar_wait(bar(DKV_FULL), 0, 0x412)) {
            tc_fence_after();
            constexpr int HALF = D / 2;
            const int key = kt * BN + row;
            const bool valid = key < T;
            const int kr = valid ? key : T - 1;  // clamp reads of invalid rows
            const __nv_bfloat16* krow = k_raw + ((static_cast<long long>(b) * T + kr) * H + h) * D;
            const float4* cs4 = reinterpret_cast<const float4*>(tab + static_cast<long long>(kr) * HALF);
            float ss = 0.f;
#pragma unroll
            for (int e8 = 0; e8 < D / 8; ++e8) {
                float y[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(krow + e8 * 8), y);
#pragma unroll
                for (int i = 0; i < 8; ++i) ss = fmaf(y[i], y[i], ss);
            }
            const float rsd = rsqrtf(ss / D + eps);
            // u = RoPE^T(dKhat) staged in shared memory (the stages are idle
            // now: every MMA and every tile load has completed); <u, y> on the way
            float* urow = reinterpret_cast<float*>(smem + S::OFF_Q + row * S::U_STRIDE);
            float dot = 0.f;
#pragma unroll 2
            for (int ch = 0; ch < HALF / 8; ++ch) {
                uint32_t glo[8], ghi[8];
                tmem_ld8(tmem + lane_base + TM_DK + ch * 8, glo);
                tmem_ld8(tmem + lane_base + TM_DK + HALF + ch * 8, ghi);
                float ylo[8], yhi[8];
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(krow + ch * 8), ylo);
                bf16x8_to_f32(*reinterpret_cast<const uint4*>(krow + HALF + ch * 8), yhi);
                float4 c4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) c4[i] = cs4[ch * 4 + i];
                tmem_wait_ld();
                float ulo[8], uhi[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float c = (e & 1) ? c4[e >> 1].z : c4[e >> 1].x;
                    const float sn = (e & 1) ? c4[e >> 1].w : c4[e >> 1].y;
                    const float a = __uint_as_float(glo[e]) * out_scale;
                    const float bb = __uint_as_float(ghi[e]) * out_scale;
                    // R^T: (a, b) -> (a c + b s, -a s + b c)
                    ulo[e] = a * c + bb * sn;
                    uhi[e] = -a * sn + bb * c;
                    dot = fmaf(ulo[e], ylo[e] * rsd, fmaf(uhi[e], yhi[e] * rsd, dot));
                }
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    reinterpret_cast<float4*>(urow + ch * 8)[g] =
                        make_float4(ulo[4 * g], ulo[4 * g + 1], ulo[4 * g + 2], ulo[4 * g + 3]);
                    reinterpret_cast<float4*>(urow + HALF + ch * 8)[g] =
                        make_float4(uhi[4 * g], uhi[4 * g + 1], uhi[4 * g + 2], uhi[4 * g + 3]);
                }
            }
            // dk = (u - y <u, y> / D) / r, y = k / r
            if (valid) {
                __nv_bfloat16* out_row = dk + ((static_cast<long long>(b) * T + key) * H + h) * D;
                const float m = dot / D;
#pragma unroll
                for (int e8 = 0; e8 < D / 8; ++e8) {
                    float y[8], o[8];
                    bf16x8_to_f32(*reinterpret_cast<const uint4*>(krow + e8 * 8), y);
                    const float4 u0 = reinterpret_cast<const float4*>(urow + e8 * 8)[0];
                    const float4 u1 = reinterpret_cast<const float4*>(urow + e8 * 8)[1];
                    const float u[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = (u[i] - y[i] * rsd * m) * rsd;
                    *reinterpret_cast<uint4*>(out_row + e8 * 8) =
                        make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]), pack_bf16x2(o[4], o[5]),
                                   pack_bf16x2(o[6], o[7]));
                }
            }
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
