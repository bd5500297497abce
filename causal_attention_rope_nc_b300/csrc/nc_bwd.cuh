// Causal attention backward on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA owns one 128-key tile j of one (batch, head) and walks the
// 64-query blocks i >= j.  Everything is computed transposed (keys on the
// TMEM lanes), which lets every product read its operands straight from the
// TMA-loaded tiles:
//   S^T   = khat_j qhat_i^T            (M=128 keys, N=64 queries, K=D)
//   dP^T  = v_j dout_i^T               (same shape)
//   P^T   = exp2(S^T * scale*log2e - lse2_i)      (recomputed; no max needed,
//                                                  lse comes from the forward)
//   dS^T  = P^T o (dP^T - delta_i)
//   dV_j += P^T dout_i                  (M=128 keys, N=D, K=64)
//   dK_j += dS^T qhat_i                 (same)
//   dQ_i^T = khat_j^T dS^T              (M=D, N=64 queries, K=128 keys)
// dV and dK accumulate in TMEM for the whole walk.  dQ_i^T is drained from
// TMEM after every block and added (fp32 reductions, already scaled by
// 1/sqrt(D)) into a [B,T,H,D] accumulator that a later pass turns into dq.
// At the end the CTA writes dv and, through the RoPE transpose and the
// RMSNorm backward, dk.
//
// Roles: warps 0-3 P/dS (thread r = key row r), warp 4 TMA, warp 5 MMA,
// warps 6-9 dQ drain and the dk epilogue.
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
constexpr int BM = 64;   // queries per block
constexpr int NUM_THREADS = 320;

enum Bar {
    KV_FULL = 0,
    FULL = 1,     // +stage: qhat_i, dout_i, lse2_i, delta_i
    EMPTY = 3,    // +stage
    S_FULL = 5,   // +buffer
    S_FREE = 7,   // +buffer
    DP_FULL = 9,
    DP_FREE = 10,
    DS_FULL = 11,
    DS_FREE = 12,
    DQ_FULL = 13,
    DQ_FREE = 14,
    DKV_FULL = 15,
    MMA_DONE = 16,
    ALPHA_READY = 17,  // warps 0-3 have published the dS scale
    NUM_BARS = 18
};

template <int D>
struct Smem {
    static constexpr int KBYTES = BN * D * 2;
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KBYTES;
    static constexpr int OFF_Q = OFF_V + KBYTES;     // 2 stages
    static constexpr int OFF_DO = OFF_Q + 2 * QBYTES;  // 2 stages
    static constexpr int OFF_PT = OFF_DO + 2 * QBYTES;  // P^T  [128 keys][64 q] bf16, SW128
    static constexpr int OFF_DST = OFF_PT + BN * BM * 2;  // dS^T [128 keys][64 q] bf16, SW128
    static constexpr int OFF_L = OFF_DST + BN * BM * 2;   // 2 stages x 64 fp32 (lse * log2e)
    static constexpr int OFF_DL = OFF_L + 2 * BM * 4;     // 2 stages x 64 fp32 (delta)
    static constexpr int OFF_BAR = OFF_DL + 2 * BM * 4;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_MISC = OFF_TSLOT + 16;  // 4 warp maxima + alpha
    static constexpr int BYTES = OFF_MISC + 32;
    static constexpr int ALLOC = BYTES + 1024;
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_ST = 0;     // 2 x 64 columns
constexpr uint32_t TM_DP = 128;   // 64 columns
constexpr uint32_t TM_DQ = 192;   // 64 columns (lanes = head dim)
constexpr uint32_t TM_DV = 256;   // D columns
// dK follows dV: TM_DV + D

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float* __restrict__ lse2, const float* __restrict__ delta, float* __restrict__ dq_acc,
                    const unsigned int* __restrict__ gmax, const __nv_bfloat16* __restrict__ k_raw,
                    const float2* __restrict__ tab,
                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int T, int H, int Tpad,
                    float scale, float scale_log2, float eps) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    const uint32_t TM_DK = TM_DV + D;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int qb0 = (kt * BN) / BM;
    const int nqb = (T + BM - 1) / BM;
    const int n_it = nqb - qb0;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    const long long bh = static_cast<long long>(b) * H + h;

    if (threadIdx.x == 0) {
        mbar_init(bar(KV_FULL), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
            mbar_init(bar(S_FULL + s), 1);
            mbar_init(bar(S_FREE + s), 128);
        }
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DP_FREE), 128);
        mbar_init(bar(DS_FULL), 128);
        mbar_init(bar(DS_FREE), 1);
        mbar_init(bar(DQ_FULL), 1);
        mbar_init(bar(DQ_FREE), 128);
        mbar_init(bar(DKV_FULL), 1);
        mbar_init(bar(MMA_DONE), 1);
        mbar_init(bar(ALPHA_READY), 128);
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

    if (warp == 4) {
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
                if (it >= 2 && !mbar_wait(bar(EMPTY + st), (use - 1) & 1, 0x111)) break;
                const int q0 = (qb0 + it) * BM;
                mbar_expect_tx(bar(FULL + st), 2 * S::QBYTES + 2 * BM * 4);
                for (int c = 0; c < NC; ++c) {
                    tma_load_4d(sb + S::OFF_Q + st * S::QBYTES + c * (BM * 128), &tm_q, c * 64, h, q0, b,
                                bar(FULL + st));
                    tma_load_4d(sb + S::OFF_DO + st * S::QBYTES + c * (BM * 128), &tm_do, c * 64, h, q0, b,
                                bar(FULL + st));
                }
                bulk_load(sb + S::OFF_L + st * BM * 4, lse2 + bh * Tpad + q0, BM * 4, bar(FULL + st));
                bulk_load(sb + S::OFF_DL + st * BM * 4, delta + bh * Tpad + q0, BM * 4, bar(FULL + st));
                ++issued[st];
            }
            mbar_wait(bar(KV_FULL), 0, 0x112);
            for (int s = 0; s < 2; ++s)
                if (issued[s]) mbar_wait(bar(FULL + s), (issued[s] - 1) & 1, 0x113);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_ST = idesc_f16(BN, BM, 0, 0);   // khat x qhat^T, fp16, K-major both
            constexpr uint32_t IDESC_DP = idesc_bf16(BN, BM, 0, 0);  // v x dout^T, bf16, K-major both
            constexpr uint32_t IDESC_DV = idesc_bf16(BN, D, 0, 1);   // P^T (K-major) x dout (MN-major)
            constexpr uint32_t IDESC_DK = idesc_f16(BN, D, 0, 1);    // dS^T (K-major) x qhat (MN-major)
            constexpr uint32_t IDESC_DQ = idesc_f16(128, BM, 1, 1);  // khat^T (MN-major) x dS^T (MN-major)
            bool ok = mbar_wait(bar(KV_FULL), 0, 0x211);
            // S^T = khat qhat^T for block `it` into score buffer it % 2
            auto issue_s = [&](int it) {
                const uint32_t q_s = sb + S::OFF_Q + (it & 1) * S::QBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                    const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + TM_ST + (it & 1) * BM, sdesc_sw128(sb + S::OFF_K + ka, 16, 1024),
                             sdesc_sw128(q_s + qa, 16, 1024), IDESC_ST, kk > 0);
                }
                mma_commit(bar(S_FULL + (it & 1)));
            };
            // dP^T = v dout^T for block `it`
            auto issue_dp = [&](int it) {
                const uint32_t do_s = sb + S::OFF_DO + (it & 1) * S::QBYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t ka = (kk >> 2) * (BN * 128) + (kk & 3) * 32;
                    const uint32_t qa = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                    mma_bf16(tmem + TM_DP, sdesc_sw128(sb + S::OFF_V + ka, 16, 1024),
                             sdesc_sw128(do_s + qa, 16, 1024), IDESC_DP, kk > 0);
                }
                mma_commit(bar(DP_FULL));
            };
            if (ok && n_it > 0) {
                ok = mbar_wait(bar(FULL + 0), 0, 0x212);
                if (ok) {
                    tc_fence_after();
                    issue_s(0);
                    issue_dp(0);
                }
            }
            // Software pipeline: the scores of block it+1 are computed while
            // warps 0-3 turn block it into P and dS.
            for (int it = 0; ok && it < n_it; ++it) {
                const int st = it & 1;
                if (it + 1 < n_it) {
                    const int st1 = (it + 1) & 1, use1 = (it + 1) >> 1;
                    if (!mbar_wait(bar(FULL + st1), use1 & 1, 0x213)) { ok = false; break; }
                    if (it + 1 >= 2 && !mbar_wait(bar(S_FREE + st1), (use1 - 1) & 1, 0x214)) { ok = false; break; }
                    tc_fence_after();
                    issue_s(it + 1);
                }
                if (!mbar_wait(bar(DS_FULL), it & 1, 0x215)) { ok = false; break; }
                tc_fence_after();
                const uint32_t q_s = sb + S::OFF_Q + st * S::QBYTES;
                const uint32_t do_s = sb + S::OFF_DO + st * S::QBYTES;
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk) {  // dV += P^T dout ; dK += dS^T qhat
                    const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                    mma_bf16(tmem + TM_DV, sdesc_sw128(sb + S::OFF_PT + kk * 32, 16, 1024),
                             sdesc_sw128(do_s + kk * (16 * 128), BM * 128, 1024), IDESC_DV, acc);
                    mma_bf16(tmem + TM_DK, sdesc_sw128(sb + S::OFF_DST + kk * 32, 16, 1024),
                             sdesc_sw128(q_s + kk * (16 * 128), BM * 128, 1024), IDESC_DK, acc);
                }
                if (it >= 1 && !mbar_wait(bar(DQ_FREE), (it - 1) & 1, 0x216)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {  // dQ^T = khat^T dS^T
                    mma_bf16(tmem + TM_DQ, sdesc_sw128(sb + S::OFF_K + kk * (16 * 128), BN * 128, 1024),
                             sdesc_sw128(sb + S::OFF_DST + kk * (16 * 128), BN * 128, 1024), IDESC_DQ, kk > 0);
                }
                mma_commit(bar(DQ_FULL));
                mma_commit(bar(DS_FREE));
                mma_commit(bar(EMPTY + st));
                if (it + 1 < n_it) {
                    // warps 0-3 finished reading dP^T(it) before signalling DS_FULL(it)
                    if (!mbar_wait(bar(DP_FREE), it & 1, 0x217)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp(it + 1);
                }
            }
            if (ok) mma_commit(bar(DKV_FULL));
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x218);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------- P, dS ----
        const int row = warp * 32 + lane;  // key row within the tile
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
            float* misc = reinterpret_cast<float*>(smem + S::OFF_MISC);
            if (lane == 0) misc[warp] = vn;
            named_bar_sync(1, 128);
            const float vmax = sqrtf(fmaxf(fmaxf(misc[0], misc[1]), fmaxf(misc[2], misc[3])));
            const float bound = __uint_as_float(gmax[0]) * (vmax + __uint_as_float(gmax[1])) * 1.0625f;
            if (bound > 0.f && bound < 3.0e38f) {
                int e = static_cast<int>(floorf(log2f(16384.f / bound)));
                e = max(-120, min(120, e));
                alpha = ldexpf(1.f, e);
            }
            if (threadIdx.x == 0) misc[4] = alpha;
            mbar_arrive(bar(ALPHA_READY));
        }
        for (int it = 0; ok && it < n_it; ++it) {
            const int st = it & 1, use = it >> 1;
            const int q0 = (qb0 + it) * BM;
            if (!mbar_wait(bar(FULL + st), use & 1, 0x311)) { ok = false; break; }
            if (!mbar_wait(bar(S_FULL + st), use & 1, 0x312)) { ok = false; break; }
            tc_fence_after();
            const float* l2 = reinterpret_cast<const float*>(smem + S::OFF_L + st * BM * 4);
            const float* dl = reinterpret_cast<const float*>(smem + S::OFF_DL + st * BM * 4);
            float p[BM];
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_ST + st * BM + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int qi = c * 32 + e;
                    const float x = fmaf(__uint_as_float(r[e]), scale_log2, -l2[qi]);
                    p[qi] = (q0 + qi < key) ? 0.f : ex2(x);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(S_FREE + st));
            if (!mbar_wait(bar(DP_FULL), it & 1, 0x313)) { ok = false; break; }
            tc_fence_after();
            float ds[BM];
#pragma unroll
            for (int c = 0; c < BM / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_DP + c * 32, r);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int qi = c * 32 + e;
                    ds[qi] = alpha * p[qi] * (__uint_as_float(r[e]) - dl[qi]);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(DP_FREE));
            if (it >= 1 && !mbar_wait(bar(DS_FREE), (it - 1) & 1, 0x314)) { ok = false; break; }
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                const uint32_t off = sw128_offset(row, ch);
                st_shared_v4(sb + S::OFF_PT + off, pack_bf16x2(p[8 * ch], p[8 * ch + 1]),
                             pack_bf16x2(p[8 * ch + 2], p[8 * ch + 3]), pack_bf16x2(p[8 * ch + 4], p[8 * ch + 5]),
                             pack_bf16x2(p[8 * ch + 6], p[8 * ch + 7]));
                st_shared_v4(sb + S::OFF_DST + off, pack_f16x2(ds[8 * ch], ds[8 * ch + 1]),
                             pack_f16x2(ds[8 * ch + 2], ds[8 * ch + 3]), pack_f16x2(ds[8 * ch + 4], ds[8 * ch + 5]),
                             pack_f16x2(ds[8 * ch + 6], ds[8 * ch + 7]));
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(DS_FULL));
        }
        // dv epilogue
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
    } else {
        // ------------------------------------------ dQ drain + dk epilogue --
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int d = quarter * 32 + lane;  // dQ^T lane = head-dim index
        bool ok = mbar_wait(bar(ALPHA_READY), 0, 0x410);
        // dS was stored times alpha: undo it together with the 1/sqrt(D) scale
        const float out_scale = ok ? scale / reinterpret_cast<const float*>(smem + S::OFF_MISC)[4] : 0.f;
        for (int it = 0; ok && it < n_it; ++it) {
            const int q0 = (qb0 + it) * BM;
            if (!mbar_wait(bar(DQ_FULL), it & 1, 0x411)) { ok = false; break; }
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + lane_base + TM_DQ, r0);
            tmem_ld32(tmem + lane_base + TM_DQ + 32, r1);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(DQ_FREE));
            if (d < D) {
                float* base = dq_acc + ((static_cast<long long>(b) * T + q0) * H + h) * D + d;
                const long long rs = static_cast<long long>(H) * D;
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (q0 + e < T) red_add_f32(base + e * rs, __uint_as_float(r0[e]) * out_scale);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (q0 + 32 + e < T) red_add_f32(base + (32 + e) * rs, __uint_as_float(r1[e]) * out_scale);
            }
        }
        // dk = RMSNorm^T(RoPE^T(dKhat * scale / alpha)), thread = key row
        if (ok && mbar_wait(bar(DKV_FULL), 0, 0x412)) {
            tc_fence_after();
            constexpr int HALF = D / 2;
            const int row = quarter * 32 + lane;
            const int key = kt * BN + row;
            const bool valid = key < T;
            const int kr = valid ? key : T - 1;  // clamp reads of invalid rows
            const __nv_bfloat16* krow = k_raw + ((static_cast<long long>(b) * T + kr) * H + h) * D;
            const float2* cs = tab + static_cast<long long>(kr) * HALF;
            float ss = 0.f;
#pragma unroll 4
            for (int e8 = 0; e8 < D / 8; ++e8) {
                const uint4 u = *reinterpret_cast<const uint4*>(krow + e8 * 8);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = unpack_bf16x2(w[i]);
                    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
                }
            }
            const float rs = rsqrtf(ss / D + eps);
            // two passes over the 32-pair chunks: <u, y> first, then the output
            float dot = 0.f;
            for (int pass = 0; pass < 2; ++pass) {
#pragma unroll 1
                for (int ch = 0; ch < HALF / 32; ++ch) {
                    uint32_t glo[32], ghi[32];
                    tmem_ld32(tmem + lane_base + TM_DK + ch * 32, glo);
                    tmem_ld32(tmem + lane_base + TM_DK + HALF + ch * 32, ghi);
                    tmem_wait_ld();
                    float olo[32], ohi[32];
#pragma unroll
                    for (int e8 = 0; e8 < 4; ++e8) {
                        const int i0 = ch * 32 + e8 * 8;
                        const uint4 ul = *reinterpret_cast<const uint4*>(krow + i0);
                        const uint4 uh = *reinterpret_cast<const uint4*>(krow + HALF + i0);
                        const uint32_t wl[4] = {ul.x, ul.y, ul.z, ul.w}, wh[4] = {uh.x, uh.y, uh.z, uh.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 yl = unpack_bf16x2(wl[i]), yh = unpack_bf16x2(wh[i]);
#pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2) {
                                const int e = e8 * 8 + 2 * i + k2;
                                const float2 c_s = cs[ch * 32 + e];
                                const float a = __uint_as_float(glo[e]) * out_scale;
                                const float bb = __uint_as_float(ghi[e]) * out_scale;
                                const float ulo = a * c_s.x + bb * c_s.y;
                                const float uhi = -a * c_s.y + bb * c_s.x;
                                const float ylo = (k2 ? yl.y : yl.x) * rs;
                                const float yhi = (k2 ? yh.y : yh.x) * rs;
                                if (pass == 0) {
                                    dot = fmaf(ulo, ylo, fmaf(uhi, yhi, dot));
                                } else {
                                    olo[e] = (ulo - ylo * (dot / D)) * rs;
                                    ohi[e] = (uhi - yhi * (dot / D)) * rs;
                                }
                            }
                        }
                    }
                    if (pass == 1 && valid) {
                        __nv_bfloat16* krow_out = dk + ((static_cast<long long>(b) * T + key) * H + h) * D;
                        uint4* dlo = reinterpret_cast<uint4*>(krow_out + ch * 32);
                        uint4* dhi = reinterpret_cast<uint4*>(krow_out + HALF + ch * 32);
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            dlo[g] = make_uint4(pack_bf16x2(olo[8 * g], olo[8 * g + 1]),
                                                pack_bf16x2(olo[8 * g + 2], olo[8 * g + 3]),
                                                pack_bf16x2(olo[8 * g + 4], olo[8 * g + 5]),
                                                pack_bf16x2(olo[8 * g + 6], olo[8 * g + 7]));
                            dhi[g] = make_uint4(pack_bf16x2(ohi[8 * g], ohi[8 * g + 1]),
                                                pack_bf16x2(ohi[8 * g + 2], ohi[8 * g + 3]),
                                                pack_bf16x2(ohi[8 * g + 4], ohi[8 * g + 5]),
                                                pack_bf16x2(ohi[8 * g + 6], ohi[8 * g + 7]));
                        }
                    }
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
