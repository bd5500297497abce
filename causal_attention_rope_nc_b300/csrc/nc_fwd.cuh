// Causal attention forward on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// One CTA computes one 128-row query tile of one (batch, head):
//   warp 4      TMA producer: Q once, then K_j / V_j tiles into 2-stage rings
//   warp 5      MMA issuer (one thread): S_j = Q K_j^T into a TMEM ping-pong,
//               O += P_j V_j into a TMEM accumulator
//   warps 0-3   softmax: thread r owns query row r (TMEM lane r); reads S_j
//               from TMEM, writes P_j = exp(S_j - m) in bf16 to shared
//               memory; at the end scales O by 1/l and writes out and lse.
//
// Operand types: qhat and khat arrive in fp16 (their elements are bounded by
// sqrt(D), so fp16's range suffices and its finer mantissa keeps the scores
// accurate); P and V are bf16.
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

namespace nc {
namespace fwd {

constexpr int BM = 128;  // query rows per CTA (one TMEM lane each)
constexpr int BN = 128;  // keys per tile
constexpr int NUM_THREADS = 192;

enum Bar {
    Q_FULL = 0,
    K_FULL = 1,    // +stage
    K_EMPTY = 3,   // +stage
    V_FULL = 5,    // +stage
    V_EMPTY = 7,   // +stage
    S_FULL = 9,    // +buffer
    S_FREE = 11,   // +buffer
    P_FULL = 13,   // +buffer
    P_FREE = 15,   // +buffer
    O_FULL = 17,
    MMA_DONE = 18,
    NUM_BARS = 19
};

template <int D>
struct Smem {
    static constexpr int QBYTES = BM * D * 2;
    static constexpr int KBYTES = BN * D * 2;
    static constexpr int PBYTES = BM * BN * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + QBYTES;
    static constexpr int OFF_V = OFF_K + 2 * KBYTES;
    static constexpr int OFF_P = OFF_V + 2 * KBYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * PBYTES;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TSLOT + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
};

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;    // two 128-column score buffers
constexpr uint32_t TM_O = 256;  // D-column output accumulator

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, int T, int H, int B, int n_qt, int group, float scale_log2,
                    float mfix_log2, float mfix) {
    using S = Smem<D>;
    constexpr int NC = D / 64;  // 64-column (128-byte) swizzle spans per row
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // grouped (b, h) order, longest rows (the last query tile) first in a group
    const TileCoord tc = grouped_tile(static_cast<int>(blockIdx.x), B * H, n_qt, group);
    const int qt = n_qt - 1 - tc.rank;
    const int b = tc.bh / H, h = tc.bh % H;
    const int n_kv = qt + 1;  // key tiles 0..qt (BM == BN)
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
            mbar_init(bar(S_FREE + s), 128);
            mbar_init(bar(P_FULL + s), 128);
            mbar_init(bar(P_FREE + s), 1);
        }
        mbar_init(bar(O_FULL), 1);
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

    if (warp == 4) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int issued_k[2] = {0, 0}, issued_v[2] = {0, 0};
            mbar_expect_tx(bar(Q_FULL), S::QBYTES);
            for (int c = 0; c < NC; ++c)
                tma_load_4d(sb + S::OFF_Q + c * (BM * 128), &tm_q, c * 64, h, qt * BM, b, bar(Q_FULL));
            for (int j = 0; j < n_kv; ++j) {
                const int st = j & 1, use = j >> 1;
                if (j >= 2 && !mbar_wait(bar(K_EMPTY + st), (use - 1) & 1, 0x101)) break;
                mbar_expect_tx(bar(K_FULL + st), S::KBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_K + st * S::KBYTES + c * (BN * 128), &tm_k, c * 64, h, j * BN, b,
                                bar(K_FULL + st));
                ++issued_k[st];
                if (j >= 2 && !mbar_wait(bar(V_EMPTY + st), (use - 1) & 1, 0x102)) break;
                mbar_expect_tx(bar(V_FULL + st), S::KBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_V + st * S::KBYTES + c * (BN * 128), &tm_v, c * 64, h, j * BN, b,
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
    } else if (warp == 5) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_f16(BM, BN, 0, 0);   // qhat (K-major) x khat (K-major), fp16
            constexpr uint32_t IDESC_O = idesc_bf16(BM, D, 0, 1);   // P (K-major) x V (MN-major)
            bool ok = mbar_wait(bar(Q_FULL), 0, 0x201);
            for (int j = 0; ok && j <= n_kv; ++j) {
                if (j < n_kv) {
                    const int st = j & 1, use = j >> 1;
                    if (!mbar_wait(bar(K_FULL + st), use & 1, 0x202)) { ok = false; break; }
                    if (j >= 2 && !mbar_wait(bar(S_FREE + st), (use - 1) & 1, 0x203)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t koff = (kk >> 2) * (BM * 128) + (kk & 3) * 32;
                        const uint64_t a = sdesc_sw128(sb + S::OFF_Q + koff, 16, 1024);
                        const uint64_t bd =
                            sdesc_sw128(sb + S::OFF_K + st * S::KBYTES + (kk >> 2) * (BN * 128) + (kk & 3) * 32, 16,
                                        1024);
                        mma_bf16(tmem + TM_S + st * BN, a, bd, IDESC_S, kk > 0);
                    }
                    mma_commit(bar(S_FULL + st));
                    mma_commit(bar(K_EMPTY + st));
                }
                if (j >= 1) {
                    const int jj = j - 1, st = jj & 1, use = jj >> 1;
                    if (!mbar_wait(bar(P_FULL + st), use & 1, 0x204)) { ok = false; break; }
                    if (!mbar_wait(bar(V_FULL + st), use & 1, 0x205)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t a = sdesc_sw128(
                            sb + S::OFF_P + st * S::PBYTES + (kk >> 2) * (BM * 128) + (kk & 3) * 32, 16, 1024);
                        const uint64_t bd =
                            sdesc_sw128(sb + S::OFF_V + st * S::KBYTES + kk * (16 * 128), BN * 128, 1024);
                        mma_bf16(tmem + TM_O, a, bd, IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(P_FREE + st));
                    mma_commit(bar(V_EMPTY + st));
                }
            }
            if (ok) mma_commit(bar(O_FULL));
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x206);
        }
        __syncwarp();
    } else {
        // ----------------------------------------- softmax + epilogue -----
        const int row = warp * 32 + lane;
        const int q_idx = qt * BM + row;
        const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
        float l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int st = j & 1, use = j >> 1;
            if (!mbar_wait(bar(S_FULL + st), use & 1, 0x301)) { ok = false; break; }
            tc_fence_after();
            if (j >= 2 && !mbar_wait(bar(P_FREE + st), (use - 1) & 1, 0x302)) { ok = false; break; }
            const bool diag = (j == qt);
            const uint32_t pb = sb + S::OFF_P + st * S::PBYTES;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_S + st * BN + c * 32, r);
                tmem_wait_ld();
                float p[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float x = fmaf(__uint_as_float(r[e]), scale_log2, -mfix_log2);
                    p[e] = (diag && (c * 32 + e) > row) ? 0.f : ex2(x);
                }
                // The normaliser sums the bf16-ROUNDED probabilities that the
                // PV product consumes, so each row's weights sum to exactly 1.
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(p[2 * i], p[2 * i + 1]);
#pragma unroll
                for (int i = 0; i < 16; i += 2)
                    l_sum += (__uint_as_float(w[i] << 16) + __uint_as_float(w[i] & 0xffff0000u)) +
                             (__uint_as_float(w[i + 1] << 16) + __uint_as_float(w[i + 1] & 0xffff0000u));
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int chunk = c * 4 + g;  // 16-byte chunk 0..15 of the 256-byte P row
                    const uint32_t addr = pb + (chunk >> 3) * (BM * 128) + sw128_offset(row, chunk & 7);
                    st_shared_v4(addr, w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive(bar(S_FREE + st));
            fence_proxy_async_smem();
            mbar_arrive(bar(P_FULL + st));
        }
        if (ok && mbar_wait(bar(O_FULL), 0, 0x303)) {
            tc_fence_after();
            const float inv_l = 1.f / l_sum;
            const bool valid = q_idx < T;
            if (valid) lse[(static_cast<long long>(b) * H + h) * T + q_idx] = mfix + logf(l_sum);
            __nv_bfloat16* orow = out + ((static_cast<long long>(b) * T + q_idx) * H + h) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + TM_O + c * 32, r);
                tmem_wait_ld();
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const float* f = reinterpret_cast<const float*>(r) + 8 * g;
                        dst[g] = make_uint4(pack_bf16x2(f[0] * inv_l, f[1] * inv_l),
                                            pack_bf16x2(f[2] * inv_l, f[3] * inv_l),
                                            pack_bf16x2(f[4] * inv_l, f[5] * inv_l),
                                            pack_bf16x2(f[6] * inv_l, f[7] * inv_l));
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

}  // namespace fwd
}  // namespace nc
