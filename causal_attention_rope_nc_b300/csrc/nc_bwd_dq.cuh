// Causal attention backward, query side: dQ on sm_103a tensor cores
// (tcgen05 + TMEM + TMA), with the RoPE transpose and the RMSNorm backward
// fused into the epilogue, so dq leaves the kernel finished (bf16).
//
// The key-side kernel (nc_bwd.cuh) forms every visible block of
//   dS = P o (dP - delta)
// anyway (for dK), and writes it once to a scratch buffer in HBM: the block
// of (query tile i, key tile j) of one (batch, query head) is 128 keys x 128
// queries of alpha * dS in fp16 (alpha: the call's one power-of-two scale,
// ds_scale_global, undone in the epilogue), laid out (ds_offset) so that
// the key side's stores coalesce without a transpose and each 64-key half
// is one contiguous 16 KB piece in the tensor core's no-swizzle operand
// layout.  This kernel is then a streaming GEMM per query
// tile,
//   dQhat_i = sum_j dS_ij khat_j          (M=128 queries, N=D, K=64 keys per stage),
// that reads each dS block once (32 KB per 128 x D x 128 product: it is HBM
// bound), recomputes nothing and uses no atomics: each dQ element is
// produced by exactly one CTA.
//
// Persistent: one CTA per SM takes query tiles until none are left, so that a
// tile's epilogue overlaps the next tile's loads and products:
//   warp 8      producer of the dS stream: one 16 KB bulk copy per half-block
//               of 64 keys into an NSD-stage ring, tile after tile (it also
//               takes the tiles from the global counter)
//   warp 11     TMA producer of the khat stream: the matching 64 khat rows
//               into an NSK-stage ring
//   warp 10     TMA producer of the epilogue tile: the tile's raw q rows,
//               once the previous tile's epilogue is done
//   warp 9      MMA issuer (one thread): A = alpha dS (MN-major, no swizzle:
//               the stage as it came from HBM), B = khat (MN-major,
//               128-byte swizzled by TMA), both fp16; the fp32
//               accumulator alternates between two TMEM buffers
//   warps 0-7   epilogue: two threads per query row apply RoPE^T and the
//               RMSNorm backward to dQhat, overwrite the raw q rows with dq
//               (each thread only the columns it read) and store them by TMA;
//               the RoPE table rows come from L2 (the table is T x D floats),
//               which leaves the shared memory to the rings.
// The dS blocks come from HBM, the khat rows mostly from L2 (a (b, h)'s
// tiles share them), so the two streams have rings of their own: nine 16 KB
// dS stages keep 144 KB of the HBM stream in flight per SM, three khat
// stages cover the shorter L2 latency.  (One ring of six 32 KB (dS, khat)
// pairs, 96 KB of dS in flight, measured the same 393 us at B=32, T=2048, H=10, D=128: the bytes
// in flight are not what holds the stream at 4.5 TB/s.)
// Tile order: the grouped order of the other kernels ((batch, head) pairs
// in groups of about one wave, the longest walks first inside a group, so
// that a group's khat tiles stay in L2), handed out dynamically: the ring
// producer takes the next tile from a global counter and passes its index
// to the other roles through a 4-slot queue in shared memory, so every CTA
// keeps streaming until the list runs out.  (A static deal of the tiles
// sorted by length balanced the CTAs but spread them over 148 heads at a
// time and doubled the HBM traffic.)  With a sliding window
// (query q sees key k when 0 <= q - k < W) a tile walks the key tiles from
// the one holding its first query's oldest visible key.
#pragma once

#include "nc_common.cuh"
#include "nc_normrope_bwd.cuh"

namespace nc {
namespace bwdq {

constexpr int BM = 128;    // queries per tile
constexpr int BN = 128;    // keys per dS block
constexpr int KS = 64;     // keys per ring stage (half a block)
constexpr int NSD = 9;     // dS ring stages
constexpr int NSK = 3;     // khat ring stages
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int WARP_EPI_TMA = 10;
constexpr int WARP_K_TMA = 11;
constexpr int NUM_THREADS = 12 * 32;

constexpr int NQ = 4;      // tile-index queue slots

enum Bar {
    FULL = 0,                  // +dS stage
    EMPTY = FULL + NSD,        // +dS stage
    KFULL = EMPTY + NSD,       // +khat stage
    KEMPTY = KFULL + NSK,      // +khat stage
    DQ_FULL = KEMPTY + NSK,    // +buffer: the tile's dQhat is in TMEM
    DQ_EMPTY = DQ_FULL + 2,    // +buffer: the epilogue has read it
    EPI_FULL = DQ_EMPTY + 2,   // raw q tile of the tile staged
    EPI_EMPTY = EPI_FULL + 1,  // the previous tile's epilogue is done with it
    MMA_DONE = EPI_EMPTY + 1,
    TQ_FULL = MMA_DONE + 1,    // +slot: a tile index (or -1: no more) in the queue
    TQ_EMPTY = TQ_FULL + NQ,   // +slot: every consumer has read it
    NUM_BARS = TQ_EMPTY + NQ
};
constexpr int TQ_READERS = 11;  // the MMA thread, the two other producers, 8 epilogue warps

// Index of the dS^T block (query tile i, key tile j <= i) of one (batch,
// query head) bh in the scratch: the causal triangle of each (b, h), in
// row-major order.  Both backward kernels address the scratch through it.
__host__ __device__ __forceinline__ long long ds_block(long long bh, int n_t, int i, int j) {
    return bh * (static_cast<long long>(n_t) * (n_t + 1) / 2) + static_cast<long long>(i) * (i + 1) / 2 + j;
}

// Element offset of (key, query) inside one 16384-element dS block:
// [key half (2)][query chunk of 8 (16)][key within the half (64)][query
// within the chunk (8)].  The key side's thread for one key row stores its
// 8-query chunks as 16-byte pieces, and the 32 keys of a warp fill 512
// contiguous bytes.  A 64-key half is 16 KB of 8-key x 8-query core
// matrices (128 contiguous bytes, keys along rows): the no-swizzle MN-major
// layout of the dQ product's A operand, with core matrices 128 bytes apart
// along K (keys) and 1024 bytes apart along M (query chunks).
__host__ __device__ __forceinline__ int ds_offset(int key, int query) {
    return (key >> 6) * 8192 + (query >> 3) * 512 + (key & 63) * 8 + (query & 7);
}
constexpr uint32_t DS_LBO = 128;   // core-matrix stride along K (keys)
constexpr uint32_t DS_SBO = 1024;  // core-matrix stride along M (query chunks)

template <int D>
struct Smem {
    static constexpr int DSBYTES = KS * BM * 2;  // 64 keys x 128 queries of dS^T (two 8 KB query halves)
    static constexpr int KBYTES = KS * D * 2;    // 64 keys of khat (D/64 halves of 8 KB)
    static constexpr int OFF_RING = 0;           // NSD dS stages
    static constexpr int OFF_KRING = OFF_RING + NSD * DSBYTES;  // NSK khat stages
    static constexpr int OFF_X = OFF_KRING + NSK * KBYTES;  // raw q [128][D] bf16 (TMA box layout), then dq
    static constexpr int XBYTES = BM * D * 2;
    static constexpr int OFF_XCH = OFF_X + XBYTES;  // row-half exchange, 2 x 128 float2
    static constexpr int OFF_BAR = OFF_XCH + 2 * BM * 8;
    static constexpr int OFF_TSLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_TQ = OFF_TSLOT + 16;  // NQ tile indices
    static constexpr int BYTES = OFF_TQ + NQ * 4;
    // the base is 1024-aligned (the declaration asks for it); whatever slack
    // is left below the opt-in limit stays for smem_align1024
    static constexpr int ALLOC = (BYTES + 1024 <= 232448) ? BYTES + 1024 : 232448;
    static_assert(BYTES <= 232448, "dQ buffers exceed shared memory");
};

constexpr uint32_t TMEM_COLS = 256;  // two dQ accumulators of D <= 128 columns

// Tile idx of the grouped order: (query tile, (b, h)).
struct DqTile {
    int qt;  // query tile
    int bh;  // b * H + h
};
__device__ __forceinline__ DqTile dq_tile(int idx, int n_qt, int nbh, int group) {
    const TileCoord c = grouped_tile(idx, nbh, n_qt, group);
    DqTile t;
    t.qt = n_qt - 1 - c.rank;
    t.bh = c.bh;
    return t;
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_dq_kernel(const __half* __restrict__ ds, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_qraw, const float2* __restrict__ tab,
                       const __grid_constant__ CUtensorMap tm_dq, const unsigned int* __restrict__ gmax,
                       unsigned int* __restrict__ tile_counter, int T, int H, int B, int group, float scale, float eps,
                       int W, int G) {
    using S = Smem<D>;
    constexpr int NC = D / 64;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_align1024(smem_raw, S::BYTES, S::ALLOC);
    if (smem == nullptr) {  // uniform over the CTA: nothing has started yet
        if (threadIdx.x == 0) flag_error(3, 0x2f0);
        return;
    }
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_qt = (T + BM - 1) / BM;
    const int nbh = B * H;
    const int n_tiles = n_qt * nbh;
    auto bar = [&](int i) -> uint32_t { return sb + S::OFF_BAR + 8 * i; };
    auto dstage = [&](int s) -> uint32_t { return sb + S::OFF_RING + s * S::DSBYTES; };
    auto kstage = [&](int s) -> uint32_t { return sb + S::OFF_KRING + s * S::KBYTES; };
    auto kt_lo_of = [&](int qt) { return max(0, qt * BM - W + 1) / BN; };  // W >= 2^30: none cut
    uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + S::OFF_TSLOT);
    volatile int* tq = reinterpret_cast<volatile int*>(smem + S::OFF_TQ);
    // the n-th tile of this CTA from the queue (every consumer reads every slot
    // once, in order); -1: no more tiles, or a wait gave up
    auto next_tile = [&](int n, bool warp_wide) -> int {
        const int q = n % NQ;
        const bool ok = warp_wide ? mbar_wait_warp(bar(TQ_FULL + q), (n / NQ) & 1, 0x230)
                                  : mbar_wait(bar(TQ_FULL + q), (n / NQ) & 1, 0x230);
        const int idx = ok ? tq[q] : -1;
        if (warp_wide)
            mbar_arrive_warp(bar(TQ_EMPTY + q));
        else
            mbar_arrive(bar(TQ_EMPTY + q));
        return idx;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < NSD; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(KFULL + s), 1);
            mbar_init(bar(KEMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(DQ_FULL + i), 1);
            mbar_init(bar(DQ_EMPTY + i), 8);  // one arrival per epilogue warp
        }
        mbar_init(bar(EPI_FULL), 1);
        mbar_init(bar(EPI_EMPTY), 1);
        mbar_init(bar(MMA_DONE), 1);
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
        // ------------------------------------------ dS ring producer ----
        if (lane == 0) {
            int x = 0;  // stages filled so far (all tiles)
            int issued[NSD];
            for (int s = 0; s < NSD; ++s) issued[s] = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                // take the next tile and publish it to the other roles
                const int q = n % NQ;
                if (n >= NQ && !mbar_wait(bar(TQ_EMPTY + q), (n / NQ - 1) & 1, 0x231)) break;
                const unsigned int got = atomicAdd(tile_counter, 1u);
                const int idx = got < static_cast<unsigned int>(n_tiles) ? static_cast<int>(got) : -1;
                tq[q] = idx;
                mbar_arrive(bar(TQ_FULL + q));
                if (idx < 0) break;
                const DqTile tl = dq_tile(idx, n_qt, nbh, group);
                const int kt_lo = kt_lo_of(tl.qt);
                const long long blk0 = ds_block(tl.bh, n_qt, tl.qt, 0);
                for (int kt = kt_lo; ok && kt <= tl.qt; ++kt) {
                    for (int half = 0; half < 2; ++half, ++x) {
                        const int s = x % NSD, use = x / NSD;
                        if (x >= NSD && !mbar_wait(bar(EMPTY + s), (use - 1) & 1, 0x121)) {
                            ok = false;
                            break;
                        }
                        // keys kt*128 + 64 half .. + 63 of the block: one contiguous 16 KB piece
                        const __half* src = ds + (blk0 + kt) * (BN * BM) + half * (KS * BM);
                        if (NC_IN_RANGE_LOAD(src, S::DSBYTES, 0x129)) {
                            mbar_expect_tx(bar(FULL + s), S::DSBYTES);
                            bulk_load(dstage(s), src, S::DSBYTES, bar(FULL + s));
                        } else {
                            mbar_arrive(bar(FULL + s));  // recorded; the stage keeps what it held
                        }
                        ++issued[s];
                    }
                }
            }
            // never leave the CTA with a bulk copy still in flight
            for (int s = 0; s < NSD; ++s)
                if (issued[s]) mbar_wait(bar(FULL + s), (issued[s] - 1) & 1, 0x124);
        }
        __syncwarp();
    } else if (warp == WARP_K_TMA) {
        // ---------------------------------------- khat ring producer ----
        if (lane == 0) {
            int x = 0;  // stages filled so far (all tiles), in step with the dS ring
            int issued[NSK];
            for (int s = 0; s < NSK; ++s) issued[s] = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = next_tile(n, false);
                if (idx < 0) break;
                const DqTile tl = dq_tile(idx, n_qt, nbh, group);
                const int b = tl.bh / H, hk = (tl.bh % H) / G;
                for (int kt = kt_lo_of(tl.qt); ok && kt <= tl.qt; ++kt) {
                    for (int half = 0; half < 2; ++half, ++x) {
                        const int s = x % NSK, use = x / NSK;
                        if (x >= NSK && !mbar_wait(bar(KEMPTY + s), (use - 1) & 1, 0x125)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(bar(KFULL + s), S::KBYTES);
                        for (int c = 0; c < NC; ++c)
                            tma_load_4d(kstage(s) + c * (KS * 128), &tm_k, c * 64, hk, kt * BN + half * KS, b,
                                        bar(KFULL + s));
                        ++issued[s];
                    }
                }
            }
            for (int s = 0; s < NSK; ++s)
                if (issued[s]) mbar_wait(bar(KFULL + s), (issued[s] - 1) & 1, 0x126);
        }
        __syncwarp();
    } else if (warp == WARP_EPI_TMA) {
        // ------------------------------- epilogue tile producer ----
        if (lane == 0) {
            int issued = 0;
            for (int n = 0;; ++n) {
                const int idx = next_tile(n, false);
                if (idx < 0) break;
                // the previous tile's epilogue has stored its dq (read the buffers)
                if (n > 0 && !mbar_wait(bar(EPI_EMPTY), (n - 1) & 1, 0x128)) break;
                const DqTile tl = dq_tile(idx, n_qt, nbh, group);
                const int b = tl.bh / H, h = tl.bh % H;
                mbar_expect_tx(bar(EPI_FULL), S::XBYTES);
                for (int c = 0; c < NC; ++c)
                    tma_load_4d(sb + S::OFF_X + c * (BM * 128), &tm_qraw, c * 64, h, tl.qt * BM, b, bar(EPI_FULL));
                ++issued;
            }
            if (issued) mbar_wait(bar(EPI_FULL), (issued - 1) & 1, 0x127);
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------- MMA issuer -----
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f16(BM, D, 1, 1);  // alpha dS (MN-major) x khat (MN-major), fp16
            int x = 0;
            bool ok = true;
            for (int n = 0; ok; ++n) {
                const int idx = next_tile(n, false);
                if (idx < 0) break;
                const DqTile tl = dq_tile(idx, n_qt, nbh, group);
                const int buf = n & 1;
                // the epilogue of tile n - 2 has read this accumulator
                if (n >= 2 && !mbar_wait(bar(DQ_EMPTY + buf), ((n - 2) >> 1) & 1, 0x225)) break;
                tc_fence_after();
                const uint32_t acc = tmem + buf * 128;
                const int steps = 2 * (tl.qt - kt_lo_of(tl.qt) + 1);
                for (int j = 0; j < steps; ++j, ++x) {
                    const int s = x % NSD, sk = x % NSK;
                    if (!mbar_wait(bar(FULL + s), (x / NSD) & 1, 0x221) ||
                        !mbar_wait(bar(KFULL + sk), (x / NSK) & 1, 0x226)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < KS / 16; ++kk)
                        mma_bf16(acc, sdesc_noswz(dstage(s) + kk * (2 * DS_LBO), DS_LBO, DS_SBO),
                                 sdesc_sw128(kstage(sk) + kk * (16 * 128), KS * 128, 1024), IDESC,
                                 (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(EMPTY + s));
                    mma_commit(bar(KEMPTY + sk));
                }
                if (ok) mma_commit(bar(DQ_FULL + buf));
            }
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
        const float alpha = ds_scale_global(gmax);
        uint8_t* xq = smem + S::OFF_X;
        for (int n = 0;; ++n) {
            const int idx = next_tile(n, true);
            if (idx < 0) break;  // uniform over each warp (it read the slot as one)
            const DqTile tl = dq_tile(idx, n_qt, nbh, group);
            const int buf = n & 1;
            bool epi = named_bar_and(1, 256, mbar_wait_warp(bar(DQ_FULL + buf), (n >> 1) & 1, 0x323));
            epi = named_bar_and(1, 256, epi && mbar_wait_warp(bar(EPI_FULL), n & 1, 0x324));
            if (!epi) break;  // uniform: a wait gave up (recorded)
            tc_fence_after();
            // dq = RMSNorm^T(RoPE^T(dQhat * scale / alpha)), written over the raw q rows
            // (rows past T read the last table row; the TMA store clips them)
            const int t_row = min(tl.qt * BM + row, T - 1);
            const uint8_t* trow = reinterpret_cast<const uint8_t*>(tab + static_cast<long long>(t_row) * (D / 2));
            (void)NC_IN_RANGE_LOAD(trow, D * 4, 0x2f1);  // recorded only: t_row is clamped into the table
            norm_rope_bwd_stage<D, true>(true, tmem + lane_base + buf * 128, scale / alpha, xq, trow, nullptr, row,
                                         half, eps, reinterpret_cast<float2*>(smem + S::OFF_XCH), xq, 1, 256);
            // the accumulator has been read (norm_rope_bwd_stage waits for its TMEM loads)
            tc_fence_before();
            mbar_arrive_warp(bar(DQ_EMPTY + buf));
            fence_proxy_async_smem();
            named_bar_sync(1, 256);
            if (threadIdx.x == 0) {
                const int b = tl.bh / H, h = tl.bh % H;
                for (int c = 0; c < NC; ++c)
                    tma_store_4d(&tm_dq, smem_u32(xq) + c * (BM * 128), c * 64, h, tl.qt * BM, b);
                bulk_commit();
                bulk_wait_read_all();  // the staged rows stay valid until the stores have read them
                mbar_arrive(bar(EPI_EMPTY));
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

}  // namespace bwdq
}  // namespace nc
