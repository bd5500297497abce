// Causal attention backward, key side: dK and dV on sm_103a tensor cores
// (tcgen05 + TMEM + TMA).  The query side (dQ) is a separate kernel
// (nc_bwd_dq.cuh), so that no gradient is accumulated through global
// atomics: each output element is owned by exactly one CTA.
//
// The unit of work is one 128-key tile j of one (batch, key/value head): its
// walk covers, for each of the G query heads that share that key/value head
// (grouped-query attention; G = 1 without it), the 128-query blocks i >= j
// that can see it (all of them, or with a sliding window W -- query q sees
// key k when 0 <= q - k < W -- those up to the block of the last query within
// W of the tile's last key).  Everything is computed transposed (keys on the
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
// Roles: warps 0-7 P, dS and the epilogue (warp w: TMEM lane quarter w%4 =
// 32 key rows, query half w/4 = 64 columns), warp 8 TMA producer, warp 9 MMA
// issuer.  The epilogue takes dk through the RoPE transpose and the RMSNorm
// backward (two threads per key row), stages dv and dk in shared memory, and
// the producer stores both tiles with TMA.
//
// Persistence.  One CTA per SM takes the key tiles from a global counter in
// the grouped order (longest walks first in a group) and keeps its barriers,
// tensor memory and pipelines across them.
// Measured per key tile of a one-CTA-per-tile form (B=32, T=2048, H=10,
// D=128; SM cycles):
// about 1.1K between one CTA's exit and the next one's entry, 1.5K of
// barrier and TMEM setup, 3.7K waiting for the first K, V, qhat and dout
// tiles, and 4.7K of epilogue, against 3.1-3.5K per query block of the walk
// (16 blocks at most, 5 with a 512-key window).  Here the setup happens once,
// and the next tile's loads overlap the current tile's end:
//   - khat and v of the next tile load as soon as the current walk's last
//     S^T and dP^T products have read them (KV_FREE);
//   - its first qhat/dout block loads into the stage of the current walk's
//     last block once that block's dK product is done;
//   - the RoPE table rows of the dk epilogue are staged by TMA into the other
//     query stage during the walk's last block; once the first pass of the
//     norm backward has read them, the same stage takes the bf16 dv and dk
//     tiles, which the producer stores with TMA (OUT_FULL) before it loads
//     the next walk's second block there;
//   - the raw k rows come from global memory straight into registers, loaded
//     before the wait for the last dK product.
// (Measured: L2 prefetches of the next walk's tiles, issued when the producer
// takes the walk, made the windowed case 1% slower and left causal as it was.)
// (Measured: dv and dk as direct 16-byte stores from registers -- 4096
// row-scattered requests per tile -- made the epilogue twice as long and,
// through the load/store queue they share, every block of the walk slower.)
// The two query stages therefore do not simply alternate across tiles: the
// next walk's first block takes the current walk's last stage.  Every role
// counts the fills of each stage (its mbarrier phases, kept in registers)
// and the producer remembers which kind of use (a query block, or the table
// and output tiles) it must wait out before refilling a stage.
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
constexpr int SMEM_LIMIT = 232448;  // 227 KB opt-in per block

constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;
// dP^T, then dS^T: the query half h of the packed fp16 pairs sits in columns
// [64h, 64h + 32), i.e. inside the dP^T columns its own warps read.
constexpr uint32_t TM_DP = 128;
constexpr uint32_t TM_DV = 256;  // D columns; dK follows at TM_DV + D

// TMEM column of the packed pair holding queries (2c, 2c+1) of K-step kk
// (16 queries): half kk/4, offset 8 columns per step inside the half.
__device__ __forceinline__ uint32_t packed_col(int kk) { return static_cast<uint32_t>((kk >> 2) * 64 + (kk & 3) * 8); }

constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;
constexpr int NQ = 4;  // key-tile queue slots

enum Bar {
    KV_FULL = 0,
    KV_FREE = 1,  // the walk's last S^T and dP^T products have read khat and v
    QF = 2,       // +stage: qhat_i, dout_i, lse2_i, delta_i landed
    QE = 4,       // +stage: the block's dK product is done (its products have read the stage)
    S_FULL = 6,
    P_FULL = 7,
    DP_FULL = 8,
    DS_FULL = 9,
    DKV_FULL = 10,  // the walk's dV and dK are complete in TMEM
    MMA_DONE = 11,
    EPI_FULL = 12,  // the walk's RoPE table rows are staged
    OUT_FULL = 13,  // the walk's dv and dk tiles are staged (over the table)
    TQ_FULL = 14,   // +slot
    TQ_EMPTY = 18,  // +slot
    NUM_BARS = 22
};
constexpr int TQ_READERS = 9;  // the MMA thread and the 8 softmax warps

template <int D>
struct Smem {
    static constexpr int KBYTES = BN * D * 2;  // khat or v tile
    static constexpr int QBYTES = BM * D * 2;  // qhat or dout stage
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + KBYTES;
    static constexpr int OFF_Q = OFF_V + KBYTES;         // 2 stages
    static constexpr int OFF_DO = OFF_Q + 2 * QBYTES;    // 2 stages
    static constexpr int OFF_L = OFF_DO + 2 * QBYTES;    // 2 stages x BM fp32 (lse * log2e)
    static constexpr int OFF_DL = OFF_L + 2 * BM * 4;    // 2 stages x BM fp32 (delta)
    static constexpr int OFF_XCH = OFF_DL + 2 * BM * 4;  // 2 (tile parity) x 2 (half) x 128 float2
    static constexpr int OFF_BAR = OFF_XCH + 2 * 2 * BN * 8;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TQ = OFF_TSLOT + 16;
    static constexpr int BYTES = OFF_TQ + NQ * 4;
    static constexpr int ALLOC = (BYTES + 1024 < SMEM_LIMIT) ? BYTES + 1024 : SMEM_LIMIT;
    // the RoPE table rows (fp32 [128][D] as D/32 boxes of 32 values x 128
    // rows) fill the qhat and dout halves of one query stage
    static_assert(BN * D * 4 == 2 * QBYTES, "table tile != one query stage");
    static_assert(BYTES <= SMEM_LIMIT, "backward tiles exceed shared memory");
};

// A pair of per-stage counters in registers (a runtime-indexed array would
// live in local memory, whose loads queue behind the kernel's stores).
struct StagePair {
    int a0 = 0, a1 = 0;
    __device__ __forceinline__ int get(int s) const { return s ? a1 : a0; }
    __device__ __forceinline__ int next(int s) {  // the value, then increment
        const int v = s ? a1 : a0;
        if (s)
            ++a1;
        else
            ++a0;
        return v;
    }
    __device__ __forceinline__ void set(int s, int v) {
        if (s)
            a1 = v;
        else
            a0 = v;
    }
};

// The walk of key tile `idx`: (b, key/value head), key tile kt, the query
// blocks qb0 .. qb0 + n_it - 1 of each of the G query heads.
struct Walk {
    int b, hk, kt, qb0, n_it, n_tot;
};
__device__ __forceinline__ Walk walk_of(int idx, int B, int Hkv, int G, int nqb, int group, int W) {
    const TileCoord tc = grouped_tile(idx, B * Hkv, nqb, group);
    Walk w;
    w.kt = tc.rank;
    w.b = tc.bh / Hkv;
    w.hk = tc.bh % Hkv;
    w.qb0 = w.kt;  // BM == BN: the diagonal query block
    const int qb_last = min(nqb - 1, (w.kt * BN + BN - 1 + W - 1) / BM);  // W >= 2^30 means no window
    w.n_it = qb_last - w.qb0 + 1;
    w.n_tot = G * w.n_it;
    return w;
}

// 10 warps put three on two of the schedulers, whose 16K registers then
// allow 170 per thread
constexpr int MAX_REGS = 168;

template <int D>
__global__ void __maxnreg__(MAX_REGS)
    attn_bwd_dkdv_persistent_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                                    const __grid_constant__ CUtensorMap tm_tab, const __grid_constant__ CUtensorMap tm_dk,
                                    const __grid_constant__ CUtensorMap tm_dv, const __nv_bfloat16* __restrict__ kraw,
                                    const float* __restrict__ lse2, const float* __restrict__ delta,
                                    const unsigned int* __restrict__ gmax, __half* __restrict__ ds_out, int T, int H,
                                    int B, int Tpad, int group, float scale, float scale_log2, float eps, int W, int G,
                                    unsigned int* __restrict__ tile_counter) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    constexpr uint32_t TM_DK = TM_DV + D;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x5f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nqb = (T + BM - 1) / BM;
    const int Hkv = H / G;
    const int n_items = nqb * B * Hkv;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    volatile int* tq = reinterpret_cast<volatile int*>(smem + S::OFF_TQ);
    // the key tile of walk n from the queue (-1: none left, or a wait gave up)
    auto next_walk = [&](int n, bool warp_wide) -> int {
        const int q = n % NQ;
        const bool ok = warp_wide ? mbar_wait_warp(bar(TQ_FULL + q), (n / NQ) & 1, 0x530)
                                  : mbar_wait(bar(TQ_FULL + q), (n / NQ) & 1, 0x530);
        const int idx = ok ? tq[q] : -1;
        if (warp_wide)
            mbar_arrive_warp(bar(TQ_EMPTY + q));
        else
            mbar_arrive(bar(TQ_EMPTY + q));
        return idx;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(KV_FULL), 1);
        mbar_init(bar(KV_FREE), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(QF + s), 1);
            mbar_init(bar(QE + s), 1);
        }
        mbar_init(bar(S_FULL), 1);
        mbar_init(bar(P_FULL), 8);  // one arrival per softmax warp
        mbar_init(bar(DP_FULL), 1);
        mbar_init(bar(DS_FULL), 8);
        mbar_init(bar(DKV_FULL), 1);
        mbar_init(bar(MMA_DONE), 1);
        mbar_init(bar(EPI_FULL), 1);
        mbar_init(bar(OUT_FULL), 8);  // one arrival per softmax warp
        for (int q = 0; q < NQ; ++q) {
            mbar_init(bar(TQ_FULL + q), 1);
            mbar_init(bar(TQ_EMPTY + q), TQ_READERS);
        }
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
            int st0 = 0;          // query stage of the walk's first block
            StagePair fills;      // query-block fills of each stage (QF / QE phases)
            StagePair last_use;   // what a stage held last: 0 nothing, 1 a block, 2 table + output tiles
            int tabs = 0, nkv = 0;  // walks whose table was loaded, key/value tile fills
            int outs = 0;           // walks whose dv and dk tiles were stored
            int out_b = 0, out_hk = 0, out_kt = 0, out_sp = 0;  // the walk whose tiles are pending
            // store the pending walk's dv and dk tiles once the softmax warps
            // have staged them, and wait until the copies have read them
            auto store_out = [&]() -> bool {
                if (outs == tabs) return true;  // nothing pending
                if (!mbar_wait(bar(OUT_FULL), outs & 1, 0x538)) return false;
                for (int c = 0; c < NC; ++c) {
                    tma_store_4d(&tm_dv, sb + S::OFF_Q + out_sp * S::QBYTES + c * (BN * 128), c * 64, out_hk,
                                 out_kt * BN, out_b);
                    tma_store_4d(&tm_dk, sb + S::OFF_DO + out_sp * S::QBYTES + c * (BN * 128), c * 64, out_hk,
                                 out_kt * BN, out_b);
                }
                bulk_commit();
                bulk_wait_read_all();
                ++outs;
                return true;
            };
            // the stage's last user has released it
            auto stage_free = [&](int s) -> bool {
                if (last_use.get(s) == 1) return mbar_wait(bar(QE + s), (fills.get(s) - 1) & 1, 0x531);
                if (last_use.get(s) == 2) return store_out();
                return true;
            };
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int q = n % NQ;
                if (n >= NQ && !mbar_wait(bar(TQ_EMPTY + q), (n / NQ - 1) & 1, 0x533)) break;
                const unsigned int got = atomicAdd(tile_counter, 1u);
                const int idx = got < static_cast<unsigned int>(n_items) ? static_cast<int>(got) : -1;
                tq[q] = idx;
                mbar_arrive(bar(TQ_FULL + q));
                if (idx < 0) break;
                const Walk w = walk_of(idx, B, Hkv, G, nqb, group, W);
                // khat and v, once the previous walk's last S^T and dP^T have read theirs
                if (n > 0 && !mbar_wait(bar(KV_FREE), (n - 1) & 1, 0x534)) break;
                mbar_expect_tx(bar(KV_FULL), 2 * S::KBYTES);
                for (int c = 0; c < NC; ++c) {
                    tma_load_4d(sb + S::OFF_K + c * (BN * 128), &tm_k, c * 64, w.hk, w.kt * BN, w.b, bar(KV_FULL));
                    tma_load_4d(sb + S::OFF_V + c * (BN * 128), &tm_v, c * 64, w.hk, w.kt * BN, w.b, bar(KV_FULL));
                }
                ++nkv;
                for (int itf = 0; itf < w.n_tot; ++itf) {
                    const int st = (st0 + itf) & 1;
                    if (!stage_free(st)) { ok = false; break; }
                    const int h = w.hk * G + itf / w.n_it;  // query head of this block
                    const long long bh = static_cast<long long>(w.b) * H + h;
                    const int q0 = (w.qb0 + itf % w.n_it) * BM;
                    mbar_expect_tx(bar(QF + st), 2 * S::QBYTES + 2 * BM * 4);
                    for (int c = 0; c < NC; ++c) {
                        tma_load_4d(sb + S::OFF_Q + st * S::QBYTES + c * (BM * 128), &tm_q, c * 64, h, q0, w.b,
                                    bar(QF + st));
                        tma_load_4d(sb + S::OFF_DO + st * S::QBYTES + c * (BM * 128), &tm_do, c * 64, h, q0, w.b,
                                    bar(QF + st));
                    }
                    bulk_load(sb + S::OFF_L + st * BM * 4, lse2 + bh * Tpad + q0, BM * 4, bar(QF + st));
                    bulk_load(sb + S::OFF_DL + st * BM * 4, delta + bh * Tpad + q0, BM * 4, bar(QF + st));
                    fills.next(st);
                    last_use.set(st, 1);
                }
                if (!ok) break;
                // the table rows of the dk epilogue into the stage the last block does not use
                const int sp = (st0 + w.n_tot) & 1;
                if (!stage_free(sp)) break;
                mbar_expect_tx(bar(EPI_FULL), 2 * S::QBYTES);
                for (int c = 0; c < D / 32; ++c) {
                    const uint32_t dst = c < NC ? S::OFF_Q + sp * S::QBYTES + c * (BN * 128)
                                                : S::OFF_DO + sp * S::QBYTES + (c - NC) * (BN * 128);
                    tma_load_2d(sb + dst, &tm_tab, c * 32, w.kt * BN, bar(EPI_FULL));
                }
                ++tabs;
                last_use.set(sp, 2);
                out_b = w.b, out_hk = w.hk, out_kt = w.kt, out_sp = sp;
                st0 = (st0 + w.n_tot - 1) & 1;  // the next walk starts in this walk's last stage
            }
            // the last walk's tiles, then never leave the CTA with a bulk copy in flight
            store_out();
            if (nkv) mbar_wait(bar(KV_FULL), (nkv - 1) & 1, 0x535);
            for (int s = 0; s < 2; ++s)
                if (fills.get(s)) mbar_wait(bar(QF + s), (fills.get(s) - 1) & 1, 0x536);
            if (tabs) mbar_wait(bar(EPI_FULL), (tabs - 1) & 1, 0x537);
            bulk_wait_read_all();
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
            int st0 = 0;      // query stage of the walk's first block
            StagePair used;   // query-block fills of each stage waited for (QF phases)
            int nb = 0;       // blocks of all walks so far (P_FULL and DS_FULL phases)
            auto wait_q = [&](int st, unsigned site) -> bool { return mbar_wait(bar(QF + st), used.next(st) & 1, site); };
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = next_walk(n, false);
                if (idx < 0) break;
                const Walk w = walk_of(idx, B, Hkv, G, nqb, group, W);
                if (!mbar_wait(bar(KV_FULL), n & 1, 0x540) || !wait_q(st0, 0x541)) break;
                tc_fence_after();
                // S^T and dP^T of the first block: TM_S and TM_DP are free, as
                // the previous walk's last dV and dK products (which read them)
                // were issued before these and complete in order
                issue_s(st0);
                issue_dp(st0);
                if (w.n_tot == 1) mma_commit(bar(KV_FREE));
                for (int it = 0; it < w.n_tot; ++it, ++nb) {
                    const int st = (st0 + it) & 1;
                    const bool more = it + 1 < w.n_tot;
                    // dV (+)= P^T dout: the softmax warps arrive on P_FULL of
                    // the walk's first block only after their epilogue of the
                    // previous walk has read dV and dK out of TMEM
                    if (!mbar_wait(bar(P_FULL), nb & 1, 0x542)) { ok = false; break; }
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
                        if (!wait_q(st ^ 1, 0x543)) { ok = false; break; }
                        tc_fence_after();
                        issue_s(st ^ 1);
                    }
                    // dK (+)= dS^T qhat, then dP^T of the next block over dS^T
                    if (!mbar_wait(bar(DS_FULL), nb & 1, 0x544)) { ok = false; break; }
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
                        if (it + 2 == w.n_tot) mma_commit(bar(KV_FREE));  // that was the last S^T and dP^T
                    }
                }
                if (!ok) break;
                mma_commit(bar(DKV_FULL));
                st0 = (st0 + w.n_tot - 1) & 1;
            }
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x545);
        }
        __syncwarp();
    } else {
        // ------------------------------------------ P, dS and the epilogue ----
        constexpr int HALF = D / 2, NF = D / 4;  // epilogue: rotation pairs (f, f + D/2), f in [half NF, half NF + NF)
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // key row within the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        const int cbase = half * 64;  // this warp's query columns
        const int f0 = half * NF;
        const float alpha = ds_scale_global(gmax);
        const uint32_t ts = tmem + lane_base + TM_S, tdp = tmem + lane_base + TM_DP;
        int st0 = 0;     // query stage of the walk's first block
        StagePair used;  // query-block fills of each stage waited for (QF phases)
        int nb = 0;      // blocks of all walks so far
        bool ok = true;
        for (int n = 0; ok; ++n) {
            const int idx = next_walk(n, true);
            // uniform over the 256 threads (the epilogue's named barriers need
            // all of them), also if one warp's wait gave up
            if (!named_bar_and(1, 256, idx >= 0)) break;
            const Walk w = walk_of(idx, B, Hkv, G, nqb, group, W);
            for (int it = 0; it < w.n_tot; ++it, ++nb) {
                const int st = (st0 + it) & 1;
                if (!mbar_wait_warp(bar(QF + st), used.next(st) & 1, 0x550)) { ok = false; break; }
                if (!mbar_wait_warp(bar(S_FULL), nb & 1, 0x551)) { ok = false; break; }
                tc_fence_after();
                const float4* l2 = reinterpret_cast<const float4*>(smem + S::OFF_L + st * BM * 4 + cbase * 4);
                const float4* dl = reinterpret_cast<const float4*>(smem + S::OFF_DL + st * BM * 4 + cbase * 4);
                // P^T = exp2(S^T scale log2e - lse2) as bf16 pairs over this
                // half's S^T columns; blocks with masked entries (the diagonal
                // one, the far end of a window) take their own copy of the loop
                const int qb = w.qb0 + it % w.n_it;             // query block of this step
                const int d0 = (qb - w.kt) * BM + cbase - row;  // query - key at this thread's first column
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
                    if (qb > w.kt && (qb - w.kt) * BM + BM - 1 < W)
                        exp_block(std::false_type{});
                    else
                        exp_block(std::true_type{});
                }
                tmem_st16(ts + cbase, pk);
                tmem_st16(ts + cbase + 16, pk + 16);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_warp(bar(P_FULL));
                // dS^T = P^T o (dP^T - delta) * alpha as fp16 pairs over this half's dP^T columns
                if (!mbar_wait_warp(bar(DP_FULL), nb & 1, 0x552)) { ok = false; break; }
                tc_fence_after();
                {
                    uint32_t r[2][32];
                    tmem_ld32(tdp + cbase, r[0]);
                    tmem_ld32(tdp + cbase + 32, r[1]);
                    tmem_wait_ld();
                    uint32_t wv[32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
#pragma unroll
                        for (int e4 = 0; e4 < 8; ++e4) {
                            const float4 d4 = dl[c * 8 + e4];
                            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w};
                            float ds[4];
#pragma unroll
                            for (int i = 0; i < 4; i += 2) {
                                const uint32_t pw = pk[c * 16 + e4 * 2 + (i >> 1)];
                                const float2 p2 =
                                    make_float2(__uint_as_float(pw << 16), __uint_as_float(pw & 0xffff0000u));
                                const float2 t2 = ffma2(make_float2(1.f, 1.f),
                                                        make_float2(__uint_as_float(r[c][e4 * 4 + i]),
                                                                    __uint_as_float(r[c][e4 * 4 + i + 1])),
                                                        make_float2(-dv4[i], -dv4[i + 1]));
                                const float2 d2 = fmul2(fmul2(make_float2(alpha, alpha), p2), t2);
                                ds[i] = d2.x;
                                ds[i + 1] = d2.y;
                            }
                            wv[c * 16 + e4 * 2] = pack_f16x2(ds[0], ds[1]);
                            wv[c * 16 + e4 * 2 + 1] = pack_f16x2(ds[2], ds[3]);
                        }
                    }
                    tmem_st16(tdp + cbase, wv);
                    tmem_st16(tdp + cbase + 16, wv + 16);
                    // the same row half into the dS scratch block (query tile
                    // qb, key tile kt) of query head h: 512 contiguous bytes
                    // per warp store in the scratch layout (bwdq::ds_offset)
                    const int h = w.hk * G + it / w.n_it;
                    __half* blk =
                        ds_out + bwdq::ds_block(static_cast<long long>(w.b) * H + h, nqb, qb, w.kt) * (BN * BM);
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        __half* pd = blk + bwdq::ds_offset(row, cbase + 8 * g);
                        if (NC_IN_RANGE(pd, 16, 0x553))
                            *reinterpret_cast<uint4*>(pd) =
                                make_uint4(wv[4 * g], wv[4 * g + 1], wv[4 * g + 2], wv[4 * g + 3]);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive_warp(bar(DS_FULL));
            }
            // ---- epilogue: dv and dk of this key tile
            const int key_c = min(w.kt * BN + row, T - 1);  // rows past T: any valid row (not stored)
            const long long rowoff = ((static_cast<long long>(w.b) * T + key_c) * Hkv + w.hk) * D;
            // this thread's raw k values (columns [f0, f0 + NF) and D/2 past
            // them), loaded while the last dK product runs
            uint4 xr[2][NF / 8];
#pragma unroll
            for (int ch = 0; ch < NF / 8; ++ch) {
                xr[0][ch] = __ldg(reinterpret_cast<const uint4*>(kraw + rowoff + f0 + 8 * ch));
                xr[1][ch] = __ldg(reinterpret_cast<const uint4*>(kraw + rowoff + HALF + f0 + 8 * ch));
            }
            // the named barriers below are reached by all 256 threads; the
            // AND keeps the branch uniform even if a wait timed out
            const bool epi = named_bar_and(1, 256,
                                           ok && mbar_wait_warp(bar(DKV_FULL), n & 1, 0x554) &&
                                               mbar_wait_warp(bar(EPI_FULL), n & 1, 0x555));
            if (!epi) { ok = false; break; }
            tc_fence_after();
            // dk = RMSNorm^T(RoPE^T(dKhat * scale / alpha)):
            //   g = dKhat scale / alpha, u = R(p)^T g,
            //   dx = u rsd - x rsd^3 <u, x> / D,  rsd = 1 / sqrt(mean(x^2) + eps),
            // the two halves of a row swapping their partial sums of x^2 and
            // <u, x>.  The table rows (fp32 (cos, sin) pairs, D/32 boxes of 32
            // values x 128 rows, 128-byte swizzled) fill the query stage the
            // walk's last block did not use; dv and dk are staged over them
            // once every thread has read its table values.
            const float out_scale = scale / alpha;
            const int sp = (st0 + w.n_tot) & 1;
            uint8_t* const q_sp = smem + S::OFF_Q + sp * S::QBYTES;   // table boxes [0, D/64), then dv
            uint8_t* const do_sp = smem + S::OFF_DO + sp * S::QBYTES;  // table boxes [D/64, D/32), then dk
            const uint8_t* ct = half ? do_sp : q_sp;
            uint32_t u[2][NF];  // g, then u, for the lo and hi columns
            float ss = 0.f, dot = 0.f;
            tmem_ld_cols<NF>(tmem + lane_base + TM_DK + f0, u[0]);
            tmem_ld_cols<NF>(tmem + lane_base + TM_DK + HALF + f0, u[1]);
            tmem_wait_ld();
#pragma unroll
            for (int ch = 0; ch < NF / 8; ++ch) {
                float xl[8], xh[8];
                bf16x8_to_f32(xr[0][ch], xl);
                bf16x8_to_f32(xr[1][ch], xh);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int f = 16 * ch + 4 * i;  // table float index relative to this half
                    const float4 cs =
                        *reinterpret_cast<const float4*>(ct + (f >> 5) * (128 * 128) + sw128_offset(row, (f & 31) >> 2));
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int e = ch * 8 + 2 * i + k;
                        const float c = k ? cs.z : cs.x, sn = k ? cs.w : cs.y;
                        const float a = __uint_as_float(u[0][e]) * out_scale;
                        const float bb = __uint_as_float(u[1][e]) * out_scale;
                        // R^T: (a, b) -> (a c + b s, b c - a s)
                        const float ul = fmaf(a, c, bb * sn), uh = fmaf(bb, c, -a * sn);
                        u[0][e] = __float_as_uint(ul);
                        u[1][e] = __float_as_uint(uh);
                        const float x0 = xl[2 * i + k], x1 = xh[2 * i + k];
                        ss = fmaf(x0, x0, fmaf(x1, x1, ss));
                        dot = fmaf(ul, x0, fmaf(uh, x1, dot));
                    }
                }
            }
            float2* xch = reinterpret_cast<float2*>(smem + S::OFF_XCH) + (n & 1) * (2 * BN);
            xch[half * BN + row] = make_float2(ss, dot);
            named_bar_sync(1, 256);  // every table value has been read; the partial sums are posted
            {
                const float2 o = xch[(half ^ 1) * BN + row];
                ss += o.x;
                dot += o.y;
                const float rsd = rsqrtf(ss / D + eps);
                const float kx = rsd * rsd * rsd * dot / D;
#pragma unroll
                for (int ch = 0; ch < NF / 8; ++ch) {
#pragma unroll
                    for (int side = 0; side < 2; ++side) {
                        float x[8], o8[8];
                        bf16x8_to_f32(xr[side][ch], x);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o8[e] = fmaf(__uint_as_float(u[side][ch * 8 + e]), rsd, -x[e] * kx);
                        *reinterpret_cast<uint4*>(do_sp + tile16_off(row, side * HALF + f0 + 8 * ch)) = f32x8_to_bf16(o8);
                    }
                }
            }
            // dv: this thread's half of the row, fp32 TMEM -> bf16, over the table
#pragma unroll
            for (int j = 0; j < 2; ++j)
                stage_acc_bf16<D / 4>(tmem + lane_base + TM_DV, 1.f, q_sp, row, half * HALF + j * (D / 4));
            // the staged tiles, for the producer's TMA stores (and dV, dK have
            // been read: the next walk's first dV and dK products wait for
            // this warp's first P_FULL arrival)
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(OUT_FULL));
            tc_fence_before();
            st0 = (st0 + w.n_tot - 1) & 1;
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
