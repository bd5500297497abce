// Causal attention backward, query side: dQ on sm_103a tensor cores
// (tcgen05 + TMEM + TMA), with the RoPE transpose and the RMSNorm backward
// fused into the epilogue, so dq leaves the kernel finished (bf16).
//
// The key-side kernel (nc_bwd.cuh) forms every visible block of
//   dS = P o (dP - delta)
// anyway (for dK), and writes it once, transposed (keys on rows), to a
// scratch buffer in HBM: the dS^T block of (query tile i, key tile j) of one
// (batch, query head) is a [128 keys][128 queries] fp16 tile holding
// alpha * dS (alpha: the call's one power-of-two scale, ds_scale_global,
// undone in the epilogue).  This kernel
// is then a streaming GEMM per query tile,
//   dQhat_i = sum_j dS_ij khat_j          (M=128 queries, N=D, K=128 keys per tile),
// that reads each dS block once (32 KB per 128 x D x 128 product: it is HBM
// bound), recomputes nothing and uses no atomics: each dQ element is
// produced by exactly one CTA.
//
// One CTA per 128-query tile i of one (batch, head), walking the key tiles
// j it can see (j <= i; with a sliding window W -- query q sees key k when
// 0 <= q - k < W -- from the tile of the first query's oldest visible key):
//   warp 8      TMA producer: (dS^T block, khat tile) pairs into an NST-stage ring
//   warp 9      MMA issuer (one thread): A = alpha dS (the MN-major view of
//               the dS^T tile), B = khat (MN-major), both fp16, fp32
//               accumulator in TMEM
//   warps 0-7   epilogue: two threads per query row apply RoPE^T and the
//               RMSNorm backward to dQhat, stage dq, TMA store
// The raw q rows and the RoPE table rows that the epilogue needs are loaded
// into ring stages as the last tiles free them.
#pragma once

#include "nc_common.cuh"
#include "nc_normrope_bwd.cuh"

namespace nc {
namespace bwdq {

constexpr int BM = 128;  // queries per CTA
constexpr int BN = 128;  // keys per tile
constexpr int NST = 3;   // ring stages
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int NUM_THREADS = 10 * 32;

enum Bar {
    FULL = 0,      // +stage
    EMPTY = 3,     // +stage
    DQ_FULL = 6,
    EPI_FULL = 7,  // raw q tile and RoPE table tile staged for the epilogue
    MMA_DONE = 8,
    NUM_BARS = 9
};

// Index of the dS^T block (query tile i, key tile j <= i) of one (batch,
// query head) bh in the scratch: the causal triangle of each (b, h), in
// row-major order.  Both backward kernels address the scratch through it.
__host__ __device__ __forceinline__ long long ds_block(long long bh, int n_t, int i, int j) {
    return bh * (static_cast<long long>(n_t) * (n_t + 1) / 2) + static_cast<long long>(i) * (i + 1) / 2 + j;
}

// Element offset inside one 16384-element dS^T block of dS^T[key][query]:
// the block is two [128 keys][64 queries] row-major halves (queries
// 64 h .. 64 h + 63), so that a 128-byte TMA box row is one key's 64 queries.
__host__ __device__ __forceinline__ int ds_offset(int key, int query) {
    return (query >> 6) * 8192 + key * 64 + (query & 63);
}

template <int D>
struct Smem {
    static constexpr int DSBYTES = BN * BM * 2;  // one dS^T block
    static constexpr int KBYTES = BN * D * 2;    // one khat tile
    static constexpr int STAGE = DSBYTES + KBYTES;
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_BAR = OFF_RING + NST * STAGE;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int BYTES = OFF_TSLOT + 16;
    static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024
    // epilogue (over the ring once its stages are free): raw q [128][D] bf16
    // and the first half of the RoPE table [128][D] fp32 in stage s_a, the
    // second half of the table in stage s_b (the stages of tiles n_kv - 2 and
    // n_kv - 3), the dq staging tile and the row-half exchange in the last
    // tile's stage
    static constexpr int XBYTES = BM * D * 2;
    static constexpr int CBYTES = BM * D * 4;
    static_assert(XBYTES + CBYTES / 2 <= STAGE && XBYTES + 2 * BM * 8 <= STAGE, "epilogue tiles exceed the stages");
    static_assert(ALLOC <= 232448, "dQ ring exceeds shared memory");
};

constexpr uint32_t TMEM_COLS = 128;  // the dQ accumulator (D <= 128 columns)

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_ds, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_qraw, const __grid_constant__ CUtensorMap tm_tab,
                       const __grid_constant__ CUtensorMap tm_dq, const unsigned int* __restrict__ gmax, int T,
                       int H, int B, int group, float scale, float eps, int W, int G) {
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
    auto stage = [&](int s) -> uint32_t { return sb + S::OFF_RING + s * S::STAGE; };
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    const long long blk0 = ds_block(tc.bh, n_qt, qt, 0);  // dS^T block of key tile 0
    // epilogue space: the stages of tiles n_kv - 2 (s_a) and n_kv - 3 (s_b),
    // free from the start when those tiles do not exist, and the last tile's
    const int s_last = (n_kv - 1) % NST, s_a = (n_kv + 1) % NST, s_b = n_kv % NST;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        mbar_init(bar(DQ_FULL), 1);
        mbar_init(bar(EPI_FULL), 1);
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
            int issued[NST] = {0, 0, 0};
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NST;
                if (j >= NST && !mbar_wait(bar(EMPTY + s), (j / NST - 1) & 1, 0x121)) {
                    ok = false;
                    break;
                }
                const int kt = kt_lo + j;
                mbar_expect_tx(bar(FULL + s), S::STAGE);
                const int row = static_cast<int>((blk0 + kt) * 2 * BN);  // < 2^31 (checked by the host)
                for (int c = 0; c < 2; ++c)
                    tma_load_2d(stage(s) + c * (BN * 128), &tm_ds, 0, row + c * BN, bar(FULL + s));
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(stage(s) + S::DSBYTES + c * (BN * 128), &tm_k, c * 64, hk, kt * BN, b,
                                bar(FULL + s));
                ++issued[s];
            }
            // epilogue tiles, each as soon as its stage is released
            mbar_expect_tx(bar(EPI_FULL), S::XBYTES + S::CBYTES);
            bool epi = ok && (n_kv < 2 || mbar_wait(bar(EMPTY + s_a), ((n_kv - 2) / NST) & 1, 0x128));
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(stage(s_a) + c * (BM * 128), &tm_qraw, c * 64, h, qt * BM, b, bar(EPI_FULL));
                for (int c = 0; c < NC; ++c)
                    tma_load_2d(stage(s_a) + S::XBYTES + c * (BM * 128), &tm_tab, c * 32, qt * BM, bar(EPI_FULL));
            }
            epi = epi && (n_kv < 3 || mbar_wait(bar(EMPTY + s_b), ((n_kv - 3) / NST) & 1, 0x129));
            if (epi) {
                for (int c = 0; c < NC; ++c)
                    tma_load_2d(stage(s_b) + c * (BM * 128), &tm_tab, (NC + c) * 32, qt * BM, bar(EPI_FULL));
            }
            // never leave the CTA with a bulk copy still in flight
            for (int s = 0; s < NST; ++s)
                if (issued[s]) mbar_wait(bar(FULL + s), (issued[s] - 1) & 1, 0x124);
            if (epi) mbar_wait(bar(EPI_FULL), 0, 0x127);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f16(BM, D, 1, 1);  // alpha dS (MN-major) x khat (MN-major), fp16
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NST;
                if (!mbar_wait(bar(FULL + s), (j / NST) & 1, 0x221)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    mma_bf16(tmem, sdesc_sw128(stage(s) + kk * (16 * 128), BN * 128, 1024),
                             sdesc_sw128(stage(s) + S::DSBYTES + kk * (16 * 128), BN * 128, 1024), IDESC,
                             (j > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(EMPTY + s));
            }
            if (ok) mma_commit(bar(DQ_FULL));
            // all MMAs issued by this thread complete before teardown
            mma_commit(bar(MMA_DONE));
            mbar_wait(bar(MMA_DONE), 0, 0x224);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue ----
        // Every barrier below is reached by all 256 threads; the AND-barriers
        // keep their branches uniform even if a wait timed out somewhere.
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;  // query row within the tile = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
        bool epi = named_bar_and(1, 256, mbar_wait_warp(bar(DQ_FULL), 0, 0x323));
        epi = named_bar_and(1, 256, epi && mbar_wait_warp(bar(EPI_FULL), 0, 0x324));
        if (epi) tc_fence_after();
        uint8_t* last = smem + S::OFF_RING + s_last * S::STAGE;
        uint8_t* sa = smem + S::OFF_RING + s_a * S::STAGE;
        // dq = RMSNorm^T(RoPE^T(dQhat * scale / alpha))
        const float alpha = ds_scale_global(gmax);
        norm_rope_bwd_stage<D>(epi, tmem + lane_base, scale / alpha, sa, sa + S::XBYTES, smem + S::OFF_RING + s_b * S::STAGE,
                               row, half, eps, reinterpret_cast<float2*>(last + S::XBYTES), last, 1, 256);
        if (epi) fence_proxy_async_smem();
        named_bar_sync(1, 256);
        if (epi && threadIdx.x == 0) {
            for (int c = 0; c < NC; ++c) tma_store_4d(&tm_dq, smem_u32(last) + c * (BM * 128), c * 64, h, qt * BM, b);
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
