// Shared device helpers for the sm_103a attention kernels: bf16 packing,
// mbarrier / TMA / tcgen05 inline PTX, bounded waits with a device error
// flag, and the RoPE angle helper.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

namespace nc {

// ----------------------------------------------------------------- status ---
// Device-side error word: 0 while healthy; the first failure writes
// (code << 16) | site.  Read and cleared by nc_device_status().
__device__ unsigned int g_dev_status = 0;

enum : unsigned int {
    DEV_ERR_TIMEOUT = 1,  // a bounded mbarrier wait gave up
    DEV_ERR_BOUNDS = 4,   // (bounds-checked build) an access outside every registered tensor
};

// A wait that has not completed after this long is treated as a failure:
// the kernel records it and unwinds instead of spinning forever.
constexpr unsigned long long WAIT_TIMEOUT_NS = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void flag_error(unsigned int code, unsigned int site) {
    atomicCAS(&g_dev_status, 0u, (code << 16) | (site & 0xffffu));
}

// ------------------------------------------------------- bounds checking --
// The bounds-checked build (compiled with -DNC_CHECK) keeps, per device, the
// byte ranges of the tensors the current call may write (its outputs and
// workspace) and may read (all of its tensors), registered by the entry point
// on the launch stream before its kernels.  Every raw global store goes
// through NC_IN_RANGE and the decode kernels' raw cache loads through
// NC_IN_RANGE_LOAD: an access outside every registered range is skipped and
// recorded as DEV_ERR_BOUNDS with its site.  TMA copies need no check: the tensor maps
// clip them to their tensors.  In the normal build NC_IN_RANGE is `true` and
// the code is unchanged.
constexpr int CHECK_MAX_RANGES = 24;
struct CheckRanges {
    unsigned long long lo[CHECK_MAX_RANGES], hi[CHECK_MAX_RANGES];
    int n;
};
#ifdef NC_CHECK
__device__ CheckRanges g_check_write;  // outputs and workspace of the current call
__device__ CheckRanges g_check_read;   // every tensor of the current call
__device__ __forceinline__ bool in_range(const CheckRanges& r, const void* p, unsigned long long bytes,
                                         unsigned int site) {
    const unsigned long long a = reinterpret_cast<unsigned long long>(p), e = a + bytes;
    for (int i = 0; i < r.n; ++i)
        if (a >= r.lo[i] && e <= r.hi[i]) return true;
    atomicCAS(&g_dev_status, 0u, (DEV_ERR_BOUNDS << 16) | (site & 0xffffu));
    return false;
}
#define NC_IN_RANGE(p, bytes, site) ::nc::in_range(::nc::g_check_write, (p), (bytes), (site))
#define NC_IN_RANGE_LOAD(p, bytes, site) ::nc::in_range(::nc::g_check_read, (p), (bytes), (site))
#else
#define NC_IN_RANGE(p, bytes, site) true
#define NC_IN_RANGE_LOAD(p, bytes, site) true
#endif

// --------------------------------------------------------------- smem/bf16 --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low half)
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
}


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void red_add_f32(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Eight 16-bit values (one 16-byte load or store) <-> eight floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = unpack_bf16x2(w[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 f32x8_to_bf16(const float (&x)[8]) {
    return make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                      pack_bf16x2(x[6], x[7]));
}

__device__ __forceinline__ uint4 f32x8_to_f16(const float (&x)[8]) {
    return make_uint4(pack_f16x2(x[0], x[1]), pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                      pack_f16x2(x[6], x[7]));
}

// Eight floats -> one 16-byte store of the 16-bit type T (bf16 or IEEE fp16).
template <typename T>
__device__ __forceinline__ uint4 f32x8_to(const float (&x)[8]) {
    if constexpr (std::is_same<T, __half>::value)
        return f32x8_to_f16(x);
    else
        return f32x8_to_bf16(x);
}

__device__ __forceinline__ void f16x8_to_f32(const uint4& u, float (&x)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = unpack_f16x2(w[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
}


// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a
// 128-byte-swizzled tile whose rows are 128 bytes: the layout that a TMA
// load with CU_TENSOR_MAP_SWIZZLE_128B writes and that a SW128 UMMA
// descriptor reads (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ----------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One arrival for the whole warp: the lanes' prior writes are ordered before
// the leader's (releasing) arrive by the warp barrier.  Barriers that count
// warps instead of threads avoid one shared-memory atomic per thread.  Only
// the active lanes synchronise, so a warp that (on an error path) is not
// converged cannot deadlock here.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    const unsigned m = __activemask();
    __syncwarp(m);
    if ((threadIdx.x & 31) == __ffs(m) - 1) mbar_arrive(bar);
}

__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok;
}

// Wait for the phase with the given parity to complete.  Bounded: after
// WAIT_TIMEOUT_NS the error flag is set and false is returned, so no
// kernel can spin forever on a barrier that is never signalled.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > WAIT_TIMEOUT_NS) {
            flag_error(DEV_ERR_TIMEOUT, site);
            return false;
        }
    }
}

// mbar_wait for warp-collective code: every lane waits, then the lanes agree
// on the outcome, so a timeout near the deadline cannot split the warp
// between the success and the error path (the warp-synchronous tcgen05 and
// shuffle instructions that follow need the whole warp).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, unsigned int site) {
    const bool ok = mbar_wait(bar, parity, site);
    return __all_sync(__activemask(), ok);
}

// ---------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Tile store shared -> global through a 4D tensor map (bulk-group
// completion).  Elements outside the tensor's extent are not written.  All
// coordinates must be non-negative.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed bulk store of this thread has finished reading
// shared memory (the source may then be reused or the CTA may exit).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the
// async proxy (tensor-core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05 --
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor, kind::f16 with an fp32 accumulator.  A and B share
// one 16-bit format (bf16 when `bf16` is set, else IEEE fp16); a_mn / b_mn
// select the MN-major ("transposed") operand form.
__host__ __device__ constexpr uint32_t idesc_f16kind(int M, int N, int a_mn, int b_mn, int bf16) {
    return (1u << 4)                                     // D format: f32
           | (static_cast<uint32_t>(bf16 ? 1 : 0) << 7)   // A format: f16 = 0, bf16 = 1
           | (static_cast<uint32_t>(bf16 ? 1 : 0) << 10)  // B format
           | (static_cast<uint32_t>(a_mn) << 15)          // A major-ness
           | (static_cast<uint32_t>(b_mn) << 16)          // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, 1);
}
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn, int b_mn) {
    return idesc_f16kind(M, N, a_mn, b_mn, 0);
}

// Shared-memory matrix descriptor with 128-byte swizzling.
//  K-major operand: rows of 128 bytes, 8-row groups SBO apart (LBO unused).
//  MN-major operand: LBO = distance between 64-element MN atoms,
//                    SBO = distance between 8-row K groups.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    d |= 2ull << 61;  // SWIZZLE_128B
    return d;
}

// Paired fp32 arithmetic (one instruction for two lanes of work on sm_100+):
// each component is rounded exactly as the scalar operation would round it.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Shared-memory matrix descriptor without swizzling: the operand is made of
// 8 x 16-byte core matrices (128 contiguous bytes each); lbo and sbo are the
// byte strides between core matrices along the two dimensions (for an
// MN-major operand: lbo along K, sbo along M/N).
__device__ __forceinline__ uint64_t sdesc_noswz(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;  // descriptor version for tcgen05
    return d;         // layout type 0: no swizzle
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Same product with the A operand (M rows on TMEM lanes, two 16-bit K
// elements per 32-bit column, K-major) read from tensor memory at `a_tmem`.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns (thread i: lane base + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 lanes x 8 consecutive 32-bit columns (thread i: lane base + i).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

// Inverse of tmem_ld16: thread i writes lane (base lane + i), 16 columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Inverse of tmem_ld32: thread i writes lane (base lane + i), columns
// [col, col + 32).  Complete with tmem_wait_st() before signalling readers.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Byte offset of the 8 16-bit values at columns [col, col + 8) of row `row`
// in a [128][D] tile kept as D/64 boxes of 128 rows x 128 bytes with 128-byte
// swizzling: the shared-memory layout of a TMA box of 64 values x 128 rows.
__device__ __forceinline__ uint32_t tile16_off(int row, int col) {
    return static_cast<uint32_t>((col >> 6) * (128 * 128)) + sw128_offset(row, (col & 63) >> 3);
}

// N consecutive TMEM columns of this warp's 32 lanes (thread i: lane base + i).
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t tm, uint32_t (&r)[N]) {
    static_assert(N % 16 == 0, "column count");
    if constexpr (N % 32 == 0) {
#pragma unroll
        for (int i = 0; i < N / 32; ++i) tmem_ld32(tm + 32 * i, *reinterpret_cast<uint32_t(*)[32]>(r + 32 * i));
    } else {
#pragma unroll
        for (int i = 0; i < N / 16; ++i) tmem_ld16(tm + 16 * i, *reinterpret_cast<uint32_t(*)[16]>(r + 16 * i));
    }
}

// bf16(s * acc) for row `row`, columns [c0, c0 + NCOL) of a TMEM fp32
// accumulator (tm = the accumulator's first column, this warp's lanes), into
// a staging tile in the layout of tile16_off.
template <int NCOL>
__device__ __forceinline__ void stage_acc_bf16(uint32_t tm, float s, uint8_t* stage, int row, int c0) {
    uint32_t r[NCOL];
    tmem_ld_cols<NCOL>(tm + c0, r);
    tmem_wait_ld();
#pragma unroll
    for (int g = 0; g < NCOL / 8; ++g) {
        const uint32_t* v = r + 8 * g;
        *reinterpret_cast<uint4*>(stage + tile16_off(row, c0 + 8 * g)) = make_uint4(
            pack_bf16x2(__uint_as_float(v[0]) * s, __uint_as_float(v[1]) * s),
            pack_bf16x2(__uint_as_float(v[2]) * s, __uint_as_float(v[3]) * s),
            pack_bf16x2(__uint_as_float(v[4]) * s, __uint_as_float(v[5]) * s),
            pack_bf16x2(__uint_as_float(v[6]) * s, __uint_as_float(v[7]) * s));
    }
}

// Dynamic shared memory rounded up to a 1024-byte boundary (128-byte swizzled
// tiles need it).  Returns nullptr when the rounding would leave fewer than
// `need` of the `alloc` bytes the launch provided.
__device__ __forceinline__ uint8_t* smem_align1024(uint8_t* raw, int need, int alloc) {
    const uint32_t s = smem_u32(raw);
    const uint32_t pad = ((s + 1023u) & ~1023u) - s;
    return (static_cast<int>(pad) + need <= alloc) ? raw + pad : nullptr;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also returns the AND of `p` over the participating
// threads, so that they all take the same branch afterwards.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool p) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred a, b;\n\t"
        "setp.ne.u32 a, %1, 0;\n\t"
        "bar.red.and.pred b, %2, %3, a;\n\t"
        "selp.u32 %0, 1, 0, b;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------- tile order --
// Work order of a one-CTA-per-tile grid over nbh (batch, head) pairs with
// n_t tiles each.  Pairs are taken in groups of g (the last group may be
// smaller); inside a group the tiles of rank 0 (the longest causal walks) of
// every pair come first, then rank 1, ...  A group's operands stay resident
// in L2 while its CTAs run, and the longest walks start first.
struct TileCoord {
    int rank;  // 0 = longest walk
    int bh;    // b * H + h
};

__device__ __forceinline__ TileCoord grouped_tile(int id, int nbh, int n_t, int g) {
    const int nfull = nbh / g;
    const int span = g * n_t;
    const int grp = id / span;
    TileCoord c;
    if (grp < nfull) {
        const int w = id - grp * span;
        c.rank = w / g;
        c.bh = grp * g + w % g;
    } else {
        const int rem = nbh - nfull * g;
        const int w = id - nfull * span;
        c.rank = w / rem;
        c.bh = nfull * g + w % rem;
    }
    return c;
}


// --------------------------------------------------------------------- RoPE --
// Rotation (cos, sin) of pair i at position p: angle p * theta_i with
// theta_i = base^(-2i/D).  The angle is formed and reduced modulo 2*pi in
// double precision, so the fp32 sin/cos that follow see an argument in
// [-pi, pi] and the rotation is accurate to fp32 rounding for any position.

// RoPE frequencies theta_i = base^(-2i/D), i < D/2, formed on the host in
// double precision and passed by value.
struct Theta {
    double t[64];
};

__device__ __forceinline__ float2 rope_cos_sin(int p, double theta) {
    const double two_pi = 6.283185307179586476925286766559;
    const double a = static_cast<double>(p) * theta;
    const double n = rint(a * (1.0 / two_pi));
    const float r = static_cast<float>(fma(-n, two_pi, a));
    float s, c;
    sincosf(r, &s, &c);
    return make_float2(c, s);
}

}  // namespace nc
