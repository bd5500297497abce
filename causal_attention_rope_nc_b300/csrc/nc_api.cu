// C ABI of the attention library: argument checks, TMA descriptors and
// kernel launches.  See include/ncattn.h for the contract of each call.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "ncattn.h"
#include "nc_bwd.cuh"
#include "nc_bwd_dq.cuh"
#include "nc_common.cuh"
#include "nc_decode.cuh"
#include "nc_fwd.cuh"
#include "nc_fwd_persist.cuh"
#include "nc_fwd_fp8.cuh"
#include "nc_rowops.cuh"

namespace {

// Dynamic shared memory the decode kernels may use: the per-block opt-in
// maximum of sm_103 (227 KB) less 1 KB for their static shared arrays.
constexpr int kDecodeSmemMax = 232448 - 1024;

thread_local int t_last_cuda_error = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];  // multiprocessors per device (set by device_ready)

// Per-device one-time set-up: architecture check and shared-memory opt-in.
int device_ready() {
    static std::mutex mu;
    static int state[kMaxDevices];  // 0 unknown, 1 ready, <0 error code
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        t_last_cuda_error = static_cast<int>(e);
        return NC_EDEVICE;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (state[dev] != 0) return state[dev] == 1 ? NC_OK : state[dev];
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
        state[dev] = NC_EUNSUPPORTED;
        return NC_EUNSUPPORTED;
    }
    if (!encode_fn()) {
        state[dev] = NC_EDEVICE;
        return NC_EDEVICE;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    g_sm_count[dev] = sms > 0 ? sms : 148;
    cudaError_t r = cudaSuccess;
    auto optin = [&](const void* f, int bytes) {
        cudaError_t x = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (x != cudaSuccess) r = x;
    };
    optin(reinterpret_cast<const void*>(nc::fwdp::attn_fwd_persistent_kernel<64>), nc::fwdp::Smem<64>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::fwdp::attn_fwd_persistent_kernel<128>), nc::fwdp::Smem<128>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::fwd::attn_fwd_kernel<64, true>), nc::fwd::Smem<64>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::fwd8::attn_fwd_fp8_kernel), nc::fwd8::Smem::ALLOC);
    optin(reinterpret_cast<const void*>(nc::fwd::attn_fwd_kernel<128, true>), nc::fwd::Smem<128>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::bwd::attn_bwd_dkdv_persistent_kernel<64>), nc::bwd::Smem<64>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::bwd::attn_bwd_dkdv_persistent_kernel<128>), nc::bwd::Smem<128>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::bwdq::attn_bwd_dq_kernel<64>), nc::bwdq::Smem<64>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::bwdq::attn_bwd_dq_kernel<128>), nc::bwdq::Smem<128>::ALLOC);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<64, 1>), kDecodeSmemMax);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<64, 2>), kDecodeSmemMax);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<64, 4>), kDecodeSmemMax);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<128, 1>), kDecodeSmemMax);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<128, 2>), kDecodeSmemMax);
    optin(reinterpret_cast<const void*>(nc::dec::attn_decode_tma_kernel<128, 4>), kDecodeSmemMax);
    if (r != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(r);
        state[dev] = NC_ELAUNCH;
        return NC_ELAUNCH;
    }
    state[dev] = 1;
    return NC_OK;
}

// Bounds-checked build: the tensors of one call, registered on its stream
// before its kernels (see nc::CheckRanges).  A no-op in the normal build.
struct CallRanges {
    nc::CheckRanges w{}, r{};
    void add(const void* p, size_t bytes, bool writable) {
        if (!p || !bytes) return;
        const unsigned long long a = reinterpret_cast<unsigned long long>(p);
        if (r.n < nc::CHECK_MAX_RANGES) r.lo[r.n] = a, r.hi[r.n] = a + bytes, ++r.n;
        if (writable && w.n < nc::CHECK_MAX_RANGES) w.lo[w.n] = a, w.hi[w.n] = a + bytes, ++w.n;
    }
    void in(const void* p, size_t bytes) { add(p, bytes, false); }
    void out(const void* p, size_t bytes) { add(p, bytes, true); }
    int publish(cudaStream_t s) const {
#ifdef NC_CHECK
        if (cudaMemcpyToSymbolAsync(nc::g_check_write, &w, sizeof(w), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyToSymbolAsync(nc::g_check_read, &r, sizeof(r), 0, cudaMemcpyHostToDevice, s) != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(cudaGetLastError());
            return NC_ELAUNCH;
        }
#else
        (void)s;
#endif
        return NC_OK;
    }
};
#ifdef NC_CHECK
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

int launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return NC_ELAUNCH;
    }
    return NC_OK;
}

// ---- optional per-kernel timing: CUDA events around every launch ----
struct ProfRec {
    const char* name;
    cudaEvent_t a, b;
    int kernels;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
    if (!g_prof_pool.empty()) {
        cudaEvent_t e = g_prof_pool.back();
        g_prof_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}

// Brackets the `kernels` kernel launches of one library step on `s` when
// timing is enabled.
struct ProfScope {
    const char* name;
    cudaStream_t s;
    int kernels;
    cudaEvent_t a = nullptr;
    ProfScope(const char* n, cudaStream_t st, int k = 1) : name(n), s(st), kernels(k) {
        if (!g_prof_on) return;
        std::lock_guard<std::mutex> lock(g_prof_mu);
        a = prof_event();
        cudaEventRecord(a, s);
    }
    ~ProfScope() {
        if (!a) return;
        std::lock_guard<std::mutex> lock(g_prof_mu);
        cudaEvent_t b = prof_event();
        cudaEventRecord(b, s);
        g_prof_recs.push_back({name, a, b, kernels});
    }
};

constexpr CUtensorMapDataType kBF16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
constexpr CUtensorMapDataType kF16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

// [B][T][H][D] 16-bit tensor, boxes of 64 head-dim values x `rows` tokens of
// one (b, h), 128-byte swizzled.  Rows past T read as zero.
int make_tmap(CUtensorMap* tm, const void* ptr, int B, int T, int H, int D, int rows,
              CUtensorMapDataType dt = kBF16) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(H) * D * 2,
                                   static_cast<cuuint64_t>(T) * H * D * 2};
    const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode_fn()(tm, dt, 4, const_cast<void*>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NC_OK : NC_EINVAL;
}

// The RoPE table [T][D/2] (cos, sin) viewed as an fp32 [T][D] tensor: boxes
// of 32 values x 128 rows, 128-byte swizzled.  Rows past T read as zero.
int make_tab_tmap(CUtensorMap* tm, const float2* tab, int T, int D) {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 4};
    const cuuint32_t box[2] = {32, 128};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode_fn()(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float2*>(tab), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NC_OK : NC_EINVAL;
}

bool shape_ok(int B, int T, int H, int D) {
    return B >= 0 && T >= 0 && H >= 0 && (D == 64 || D == 128) && B <= 65535 && H <= 65535 &&
           T <= (1 << 24);
}

bool params_ok(float eps, float base) { return std::isfinite(eps) && eps >= 0.f && std::isfinite(base) && base > 0.f; }

size_t tab_bytes(int T, int D) { return up256(static_cast<size_t>(T) * (D / 2) * sizeof(float2)); }
int tpad_of(int T) { return ((T + 127) / 128) * 128; }  // query blocks of 128

// Rows of 128 fp16 values in the backward's dS scratch: one 128 x 128 block
// per (query tile, key tile <= query tile) of every (batch, query head).
long long ds_rows(int B, int T, int H) {
    const long long n_t = (T + 127) / 128;
    return static_cast<long long>(B) * H * (n_t * (n_t + 1) / 2) * 128;
}

// Backward workspace: RoPE table, delta, lse * log2(e), two norm maxima,
// dS^T scratch.
size_t bwd_ws_bytes(int B, int T, int H, int D) {
    const int Tpad = tpad_of(T);
    return tab_bytes(T, D) + 2 * up256(static_cast<size_t>(B) * H * Tpad * 4) + 256 +
           static_cast<size_t>(ds_rows(B, T, H)) * 128 * 2;
}

int rows_grid(long long rows, int D) {
    const long long groups = 256 / (D / 8);
    long long g = (rows + groups - 1) / groups;
    if (g > 148LL * 16) g = 148LL * 16;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

// Blocks of a 256-thread kernel without dynamic shared memory that one SM
// holds at once (the occupancy calculator's answer; 1 if it has none).
template <typename Kern>
int resident_256(Kern kernel) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, 256, 0) != cudaSuccess || n < 1) n = 1;
    return n;
}

// One token per group of `lanes` lanes, 256 threads per block: enough
// blocks for every token, at most the blocks the SMs hold at once (per_sm each), so
// that a grid-stride walk runs as one wave with an even share per block
// instead of a partial last wave.  (Measured for the QK norm prologue at
// B=32, T=2048, H=10, D=128, whose 80 registers leave room for 3 blocks per
// SM: a grid sized for 8 ran 2.7 waves.)
int tok_grid(long long toks, int lanes, int per_sm) {
    int dev = 0;
    cudaGetDevice(&dev);
    const long long cap = static_cast<long long>(g_sm_count[dev] > 0 ? g_sm_count[dev] : 148) * per_sm;
    const long long groups = 256 / lanes;
    long long g = (toks + groups - 1) / groups;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

// (b, h) pairs per group of the grouped tile order: about two waves of
// one-CTA-per-SM tiles.
int tile_group(int n_t, int nbh) {
    int g = (2 * 148 + n_t - 1) / n_t;
    if (g > nbh) g = nbh;
    return g < 1 ? 1 : g;
}

// RoPE frequencies theta_i = base^(-2i/D), i < D/2, in double precision:
// the one set of values the tables, the decode and the prefill all use.
nc::Theta rope_thetas(int D, float base) {
    nc::Theta th{};
    for (int i = 0; i < D / 2; ++i) th.t[i] = std::exp2(-(2.0 * i / D) * std::log2(double(base)));
    return th;
}

int launch_rope_table(float2* tab, const int32_t* pos, int T, int D, float base, cudaStream_t s) {
    const long long n = static_cast<long long>(T) * (D / 2);
    int grid = static_cast<int>((n + 255) / 256);
    if (grid > 148 * 8) grid = 148 * 8;
    const nc::Theta th = rope_thetas(D, base);
    ProfScope ps("rope_table", s);
    nc::rope_table_kernel<<<grid, 256, 0, s>>>(tab, pos, T, D, th);
    return launch_status();
}

// qhat (H heads) and, when k is given, khat (Hkv heads).  rstd (optional):
// the q rows' [B][T][H] followed by the k rows' [B][T][Hkv].  One launch
// covers both when the head counts agree, else one launch per tensor.
template <int D, typename OutT>
int launch_norm_rope(const nc_bf16* q, const nc_bf16* k, const float2* tab, void* qh, void* kh, float* rstd,
                     int B, int T, int H, int Hkv, float eps, cudaStream_t s, float out_scale = 1.f) {
    const long long toks = static_cast<long long>(B) * T;
    static const int per_sm = resident_256(nc::qk_norm_rope_kernel<D, OutT>);
    ProfScope ps("qk_norm_rope", s, (!k || Hkv == H) ? 1 : 2);
    if (!k || Hkv == H) {
        nc::qk_norm_rope_kernel<D, OutT><<<tok_grid(toks * (k ? 2 : 1), D / 16, per_sm), 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k), tab,
            reinterpret_cast<OutT*>(qh), reinterpret_cast<OutT*>(kh), rstd, toks, T, H, eps, out_scale);
        return launch_status();
    }
    nc::qk_norm_rope_kernel<D, OutT><<<tok_grid(toks, D / 16, per_sm), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(q), nullptr, tab, reinterpret_cast<OutT*>(qh), nullptr, rstd, toks,
        T, H, eps, out_scale);
    int rc = launch_status();
    if (rc) return rc;
    nc::qk_norm_rope_kernel<D, OutT><<<tok_grid(toks, D / 16, per_sm), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(k), nullptr, tab, reinterpret_cast<OutT*>(kh), nullptr,
        rstd ? rstd + toks * H : nullptr, toks, T, Hkv, eps, out_scale);
    return launch_status();
}

// Sliding window as the kernels take it: a value no distance reaches when
// there is none (window <= 0, or at least the sequence length).
int window_eff(int window, int T) { return (window <= 0 || window >= T) ? (1 << 30) : window; }

// Key/value heads as the kernels take them: kv_heads = 0 means H (plain
// multi-head attention); otherwise it must divide H.  0 on a bad value.
int kv_heads_of(int kv_heads, int H) {
    if (kv_heads == 0) return H;
    if (kv_heads < 0 || kv_heads > H || H % kv_heads != 0) return 0;
    return kv_heads;
}

// The forward kernel over all pairs of query tiles, one CTA per pair in the
// grouped order.  (Measured: launching the first pair of each (batch, head),
// whose first tile's rows need the split-P path, separately from the rest
// through an instantiation without that path, was 6% slower in total.)
template <int D, bool QK_BF16>
int launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to, float* lse,
               int T, int H, int B, int Hkv, int W, const int* qoff, int Tk, const char* name, cudaStream_t s) {
    const int n_qt = (T + nc::fwd::BM - 1) / nc::fwd::BM;
    const int n_pairs = (n_qt + 1) / 2;
    const double scale = 1.0 / std::sqrt(double(D));
    const double log2e = 1.4426950408889634;
    const double mfix = std::sqrt(double(D)) * 1.0079;
    const long long nblk = static_cast<long long>(n_pairs) * B * H;
    if (nblk > 0x7fffffffLL) return NC_EINVAL;
    ProfScope ps(name, s);
    nc::fwd::attn_fwd_kernel<D, QK_BF16><<<static_cast<unsigned>(nblk), nc::fwd::NUM_THREADS,
                                           nc::fwd::Smem<D>::ALLOC, s>>>(
        tq, tk, tv, to, lse, T, H, B, n_qt, tile_group(n_pairs, B * H), float(scale * log2e), float(mfix * log2e),
        float(mfix), W, qoff, Tk, H / Hkv);
    return launch_status();
}

template <int D>
int fwd_impl(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, nc_bf16* out, float* lse,
             nc_f16* qhat, nc_f16* khat, float* rstd, void* ws, int B, int T, int H, int Hkv, float eps, float base,
             int W, cudaStream_t s) {
    float2* tab = reinterpret_cast<float2*>(ws);
    int rc = launch_rope_table(tab, pos, T, D, base, s);
    if (rc) return rc;
    rc = launch_norm_rope<D, __half>(q, k, tab, qhat, khat, rstd, B, T, H, Hkv, eps, s);
    if (rc) return rc;
    CUtensorMap tq, tk, tv;
    if (make_tmap(&tq, qhat, B, T, H, D, nc::fwd::BM, kF16) ||
        make_tmap(&tk, khat, B, T, Hkv, D, nc::fwd::BN, kF16) || make_tmap(&tv, v, B, T, Hkv, D, nc::fwd::BN))
        return NC_EINVAL;
    // persistent: one CTA per SM takes pairs of query tiles from a counter
    unsigned int* counter = reinterpret_cast<unsigned int*>(reinterpret_cast<uint8_t*>(ws) + tab_bytes(T, D));
    if (cudaMemsetAsync(counter, 0, sizeof(unsigned int), s) != cudaSuccess) return launch_status();
    const int n_qt = (T + nc::fwd::BM - 1) / nc::fwd::BM;
    const int n_pairs = (n_qt + 1) / 2;
    const long long n_items = static_cast<long long>(n_pairs) * B * H;
    if (n_items > 0x7fffffffLL) return NC_EINVAL;
    const double scale = 1.0 / std::sqrt(double(D));
    const double log2e = 1.4426950408889634;
    const double mfix = std::sqrt(double(D)) * 1.0079;
    int dev = 0;
    cudaGetDevice(&dev);
    const int grid = static_cast<int>(n_items < g_sm_count[dev] ? n_items : g_sm_count[dev]);
    ProfScope ps("attn_fwd", s);
    nc::fwdp::attn_fwd_persistent_kernel<D><<<static_cast<unsigned>(grid), nc::fwdp::NUM_THREADS,
                                              nc::fwdp::Smem<D>::ALLOC, s>>>(
        tq, tk, tv, reinterpret_cast<__nv_bfloat16*>(out), lse, T, H, B, n_qt, tile_group(n_pairs, B * H),
        float(scale * log2e), float(mfix * log2e), float(mfix), W, H / Hkv, counter);
    return launch_status();
}

// Chunk prefill: the prologue writes qhat (workspace) and the chunk's keys
// and values into the caches, then the forward kernel runs with the chunk's
// queries at their cache positions and the caches as keys and values.
template <int D>
int prefill_impl(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* start, nc_bf16* kcache,
                 nc_bf16* vcache, nc_bf16* out, float* lse, void* ws, int B, int C, int H, int Hkv, int Tcap,
                 float eps, float base, int W, cudaStream_t s) {
    const nc::Theta th = rope_thetas(D, base);
    __nv_bfloat16* qhat = reinterpret_cast<__nv_bfloat16*>(ws);
    {
        ProfScope ps("prefill_norm_rope", s);
        static const int per_sm = resident_256(nc::prefill_norm_rope_kernel<D>);
        nc::prefill_norm_rope_kernel<D><<<tok_grid(static_cast<long long>(B) * C, D / 8, per_sm), 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k),
            reinterpret_cast<const __nv_bfloat16*>(v), start, qhat, reinterpret_cast<__nv_bfloat16*>(kcache),
            reinterpret_cast<__nv_bfloat16*>(vcache), B, C, H, Hkv, Tcap, eps, th);
    }
    int rc = launch_status();
    if (rc) return rc;
    CUtensorMap tq, tk, tv, to;
    if (make_tmap(&tq, qhat, B, C, H, D, nc::fwd::BM) ||
        make_tmap(&tk, kcache, B, Tcap, Hkv, D, nc::fwd::BN) ||
        make_tmap(&tv, vcache, B, Tcap, Hkv, D, nc::fwd::BN) || make_tmap(&to, out, B, C, H, D, nc::fwd::BM))
        return NC_EINVAL;
    return launch_fwd<D, true>(tq, tk, tv, to, lse, C, H, B, Hkv, W, start, Tcap, "attn_prefill", s);
}

template <int D>
int bwd_impl(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, const nc_bf16* out,
             const float* lse, const nc_f16* qhat, const nc_f16* khat, const nc_bf16* dout, nc_bf16* dq,
             nc_bf16* dk, nc_bf16* dv, void* ws, int B, int T, int H, int Hkv, float eps, float base, int W,
             cudaStream_t s) {
    const int Tpad = tpad_of(T);
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    float2* tab = reinterpret_cast<float2*>(w);
    w += tab_bytes(T, D);
    float* delta = reinterpret_cast<float*>(w);
    w += up256(static_cast<size_t>(B) * H * Tpad * 4);
    float* lse2 = reinterpret_cast<float*>(w);
    w += up256(static_cast<size_t>(B) * H * Tpad * 4);
    // max ||dout_t||, max ||v_t||, the query side's and the key side's tile counters
    unsigned int* gmax = reinterpret_cast<unsigned int*>(w);
    w += 256;
    nc_f16* ds = reinterpret_cast<nc_f16*>(w);
    int rc = launch_rope_table(tab, pos, T, D, base, s);
    if (rc) return rc;
    if (cudaMemsetAsync(gmax, 0, 4 * sizeof(unsigned int), s) != cudaSuccess) return launch_status();
    const long long rows = static_cast<long long>(B) * T * H;
    {
        ProfScope ps("attn_bwd_pre", s);
        nc::bwd_pre_kernel<D><<<rows_grid(rows / 4 + 1, D), 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(out), reinterpret_cast<const __nv_bfloat16*>(dout),
            reinterpret_cast<const __nv_bfloat16*>(v), lse, delta, lse2, gmax, B, T, H, Hkv, Tpad);
    }
    if ((rc = launch_status())) return rc;
    CUtensorMap tq, tk, tv, tdo, tqr, ttab, tdq, tdk, tdv, tk64;
    if (make_tmap(&tq, qhat, B, T, H, D, 128, kF16) || make_tmap(&tk, khat, B, T, Hkv, D, 128, kF16) ||
        make_tmap(&tv, v, B, T, Hkv, D, 128) || make_tmap(&tdo, dout, B, T, H, D, 128) ||
        make_tmap(&tqr, q, B, T, H, D, 128) || make_tab_tmap(&ttab, tab, T, D) ||
        make_tmap(&tdq, dq, B, T, H, D, 128) || make_tmap(&tdk, dk, B, T, Hkv, D, 128) ||
        make_tmap(&tdv, dv, B, T, Hkv, D, 128) || make_tmap(&tk64, khat, B, T, Hkv, D, nc::bwdq::KS, kF16))
        return NC_EINVAL;
    const long long n_t = (T + 127) / 128;
    const long long nblk = n_t * B * H;
    const long long nblk_kv = n_t * B * Hkv;
    if (nblk > 0x7fffffffLL) return NC_EINVAL;
    const double scale = 1.0 / std::sqrt(double(D));
    const int G = H / Hkv;
    const int group = tile_group(static_cast<int>(n_t), B * H);
    int dev = 0;
    cudaGetDevice(&dev);
    {
        // key side: dk, dv; one persistent CTA per SM takes the key tiles of
        // the key/value heads (longest walks first in a group) from a counter
        // and walks the query blocks of all G heads that share each
        const int grid = static_cast<int>(nblk_kv < g_sm_count[dev] ? nblk_kv : g_sm_count[dev]);
        ProfScope ps("attn_bwd_dkdv", s);
        nc::bwd::attn_bwd_dkdv_persistent_kernel<D><<<static_cast<unsigned>(grid), nc::bwd::NUM_THREADS,
                                                       nc::bwd::Smem<D>::ALLOC, s>>>(
            tq, tk, tv, tdo, ttab, tdk, tdv, reinterpret_cast<const __nv_bfloat16*>(k), lse2, delta, gmax,
            reinterpret_cast<__half*>(ds), T, H, B, Tpad,
            tile_group(static_cast<int>(n_t), B * Hkv), float(scale), float(scale * 1.4426950408889634), eps, W, G,
            gmax + 3);
    }
    if ((rc = launch_status())) return rc;
    {
        // query side: dq = dS khat from the key side's dS^T scratch, one
        // persistent CTA per SM over all query tiles
        const long long n_tiles = n_t * B * H;
        const int grid = static_cast<int>(n_tiles < g_sm_count[dev] ? n_tiles : g_sm_count[dev]);
        ProfScope ps("attn_bwd_dq", s);
        nc::bwdq::attn_bwd_dq_kernel<D><<<static_cast<unsigned>(grid), nc::bwdq::NUM_THREADS,
                                          nc::bwdq::Smem<D>::ALLOC, s>>>(reinterpret_cast<const __half*>(ds), tk64, tqr, tab, tdq,
                                                                         gmax, gmax + 2, T,
                                                                         H, B, group, float(scale), eps, W, G);
    }
    return launch_status();
}

// FP8 forward workspace: RoPE table, q8 [B][T][H][D], k8 [B][T][Hkv][D],
// v8^T [B][Hkv][D][Tpad] (E4M3 bytes), per-head max |v| and scale 2^-tau.
// Sized with Hkv = H (an upper bound).
struct Fp8Ws {
    float2* tab;
    uint8_t *q8, *k8, *v8t;
    unsigned int* vmax;
    float* vscale;
};

size_t fp8_ws_layout(int B, int T, int H, int D, Fp8Ws* out, void* base) {
    const size_t tok = static_cast<size_t>(B) * T * H * D;
    const size_t vt = static_cast<size_t>(B) * H * D * tpad_of(T);
    const size_t o_tab = 0, o_q = o_tab + tab_bytes(T, D), o_k = o_q + up256(tok), o_v = o_k + up256(tok);
    const size_t o_m = o_v + up256(vt), o_s = o_m + up256(static_cast<size_t>(B) * H * 4);
    const size_t total = o_s + up256(static_cast<size_t>(B) * H * 4);
    if (out) {
        uint8_t* w = reinterpret_cast<uint8_t*>(base);
        out->tab = reinterpret_cast<float2*>(w + o_tab);
        out->q8 = w + o_q;
        out->k8 = w + o_k;
        out->v8t = w + o_v;
        out->vmax = reinterpret_cast<unsigned int*>(w + o_m);
        out->vscale = reinterpret_cast<float*>(w + o_s);
    }
    return total;
}

// [B][T][H][128] E4M3 tensor: boxes of 128 bytes (a whole head row) x 128
// tokens of one (b, h), 128-byte swizzled.  Rows past T read as zero.
int make_tmap_e4m3(CUtensorMap* tm, const void* ptr, int B, int T, int H, int D) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H) * D,
                                   static_cast<cuuint64_t>(T) * H * D};
    const cuuint32_t box[4] = {128, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode_fn()(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NC_OK : NC_EINVAL;
}

// v8^T [B Hkv][D][Tpad] E4M3: boxes of 128 keys (bytes) x D rows of one head.
int make_tmap_vt(CUtensorMap* tm, const void* ptr, int BH, int D, int Tpad) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(Tpad), static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(Tpad), static_cast<cuuint64_t>(D) * Tpad};
    const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(D), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode_fn()(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NC_OK : NC_EINVAL;
}

int fwd_fp8_impl(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, nc_bf16* out, float* lse,
                 void* ws, int B, int T, int H, int Hkv, float eps, float base, int W, cudaStream_t s) {
    constexpr int D = nc::fwd8::D;
    Fp8Ws w;
    fp8_ws_layout(B, T, H, D, &w, ws);
    const int Tpad = tpad_of(T);
    int rc = launch_rope_table(w.tab, pos, T, D, base, s);
    if (rc) return rc;
    // q8 = E4M3(qhat 2^5), k8 likewise
    rc = launch_norm_rope<D, __nv_fp8_e4m3>(q, k, w.tab, w.q8, w.k8, nullptr, B, T, H, Hkv, eps, s, 32.f);
    if (rc) return rc;
    if (cudaMemsetAsync(w.vmax, 0, static_cast<size_t>(B) * Hkv * 4, s) != cudaSuccess) return launch_status();
    {
        ProfScope ps("v_quant", s, 2);
        nc::v_absmax_kernel<D><<<dim3((T + 255) / 256, B * Hkv), 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(v), w.vmax, T, Hkv);
        if ((rc = launch_status())) return rc;
        nc::v_quant_t_kernel<D><<<dim3(Tpad / 128, B * Hkv), 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(v), w.vmax, w.v8t, w.vscale, T, Tpad, Hkv);
        if ((rc = launch_status())) return rc;
    }
    CUtensorMap tq, tk, tvt, to;
    if (make_tmap_e4m3(&tq, w.q8, B, T, H, D) || make_tmap_e4m3(&tk, w.k8, B, T, Hkv, D) ||
        make_tmap_vt(&tvt, w.v8t, B * Hkv, D, Tpad) || make_tmap(&to, out, B, T, H, D, nc::fwd8::BM))
        return NC_EINVAL;
    const int n_qt = (T + nc::fwd8::BM - 1) / nc::fwd8::BM;
    const int n_pairs = (n_qt + 1) / 2;
    const long long nblk = static_cast<long long>(n_pairs) * B * H;
    if (nblk > 0x7fffffffLL) return NC_EINVAL;
    const double craw = 1.0 / (1024.0 * std::sqrt(double(D)));  // raw E4M3 score -> scaled score
    ProfScope ps("attn_fwd_fp8", s);
    nc::fwd8::attn_fwd_fp8_kernel<<<static_cast<unsigned>(nblk), nc::fwd8::NUM_THREADS, nc::fwd8::Smem::ALLOC, s>>>(
        tq, tk, tvt, to, w.vscale, lse, T, H, B, n_qt, tile_group(n_pairs, B * H), float(craw * 1.4426950408889634),
        float(craw), W, H / Hkv);
    return launch_status();
}

struct DecodeWs {
    float* part_o;
    float* part_ml;
    unsigned int* counters;
};

size_t decode_ws_layout(int B, int H, int D, int Tcap, DecodeWs* out, void* base) {
    const int nit = (Tcap + nc::dec::PART_SLOTS - 1) / nc::dec::PART_SLOTS;  // partial results per stream, at most
    const size_t o_bytes = up256(static_cast<size_t>(B) * nit * H * D * 4);
    const size_t ml_bytes = up256(static_cast<size_t>(B) * nit * H * 2 * 4);
    const size_t c_bytes = up256(static_cast<size_t>(B) * 4);
    if (out) {
        uint8_t* w = reinterpret_cast<uint8_t*>(base);
        out->counters = reinterpret_cast<unsigned int*>(w);
        out->part_ml = reinterpret_cast<float*>(w + c_bytes);
        out->part_o = reinterpret_cast<float*>(w + c_bytes + ml_bytes);
    }
    return c_bytes + ml_bytes + o_bytes;
}

// Keys or values (bf16) of a [B][Tcap][Hkv][D] cache as a 4D tensor
// map with [sb][Hkv][D] boxes (no swizzle): one copy brings sb whole slots.
int make_cache_tmap(CUtensorMap* tm, const void* ptr, int B, int Tcap, int Hkv, int D, int sb,
                    CUtensorMapDataType dt) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                                static_cast<cuuint64_t>(Tcap), static_cast<cuuint64_t>(B)};
    const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hkv) * D * 2,
                                   static_cast<cuuint64_t>(Tcap) * Hkv * D * 2};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(Hkv),
                               static_cast<cuuint32_t>(sb), 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = encode_fn()(tm, dt, 4, const_cast<void*>(ptr), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? NC_OK : NC_EINVAL;
}

template <int D, int HPW>
int launch_decode_tma(const CUtensorMap& tk, const CUtensorMap& tv, const nc_bf16* q, const nc_bf16* k_new,
                      const nc_bf16* v_new, nc_bf16* kcache, nc_bf16* vcache, const int32_t* lens, nc_bf16* out,
                      const DecodeWs& ws, int B, int H, int Hkv, int Tcap, float eps, const nc::Theta& th,
                      float scale_log2, int W, int sb, int nst, cudaStream_t s) {
    const int nparts = (Tcap + nc::dec::PART_SLOTS - 1) / nc::dec::PART_SLOTS;
    const int nch = (Tcap + nc::dec::CH - 1) / nc::dec::CH;
    const int nwc = (H + HPW - 1) / HPW;  // compute warps (<= MAX_CWARPS), plus one producer warp
    const size_t smem = nc::dec::smem_bytes(Hkv, D, sb, nst);
    ProfScope ps("attn_decode", s);
    nc::dec::attn_decode_tma_kernel<D, HPW><<<dim3(static_cast<unsigned>(nch), static_cast<unsigned>(B)),
                                              (nwc + 1) * 32, smem, s>>>(
        tk, tv, reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k_new),
        reinterpret_cast<const __nv_bfloat16*>(v_new), reinterpret_cast<__nv_bfloat16*>(kcache),
        reinterpret_cast<__nv_bfloat16*>(vcache), lens, reinterpret_cast<__nv_bfloat16*>(out), ws.part_o,
        ws.part_ml, ws.counters, B, H, Hkv, Tcap, nparts, eps, th, scale_log2, W, sb, nst);
    return launch_status();
}

template <int D>
int decode_impl(const nc_bf16* q, const nc_bf16* k_new, const nc_bf16* v_new, nc_bf16* kcache, nc_bf16* vcache,
                const int32_t* lens, nc_bf16* out, const DecodeWs& ws, int B, int H, int Hkv, int Tcap, float eps,
                float base, int W, cudaStream_t s) {
    const float scale_log2 = float(1.4426950408889634 / std::sqrt(double(D)));
    const nc::Theta th = rope_thetas(D, base);
    if (Hkv == H) {
        // multi-head attention: the register-pipelined kernel, one warp per
        // head, the heads split over head groups
        const int nparts = (Tcap + nc::dec::PART_SLOTS - 1) / nc::dec::PART_SLOTS;
        const int G = H / Hkv;
        const nc::dec::RegSplit rs = nc::dec::reg_split(H, G);
        const int nch = (Tcap + rs.ch - 1) / rs.ch;
        ProfScope ps("attn_decode", s);
        nc::dec::attn_decode_kernel<D><<<dim3(static_cast<unsigned>(nch), static_cast<unsigned>(B),
                                              static_cast<unsigned>(rs.groups)),
                                         rs.warps * 32, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16*>(q), reinterpret_cast<const __nv_bfloat16*>(k_new),
            reinterpret_cast<const __nv_bfloat16*>(v_new), reinterpret_cast<__nv_bfloat16*>(kcache),
            reinterpret_cast<__nv_bfloat16*>(vcache), lens, reinterpret_cast<__nv_bfloat16*>(out), ws.part_o,
            ws.part_ml, ws.counters, B, H, Tcap, nparts, eps, th, scale_log2, W, G, rs.ch, rs.hpg);
        return launch_status();
    }
    // grouped-query attention: the TMA ring kernel
    const int sb = nc::dec::stage_slots(Hkv, D);
    const int nst = nc::dec::ring_stages(Hkv, D, sb);
    if (nc::dec::smem_bytes(Hkv, D, sb, nst) > static_cast<size_t>(kDecodeSmemMax)) return NC_EINVAL;
    CUtensorMap tk, tv;
    if (make_cache_tmap(&tk, kcache, B, Tcap, Hkv, D, sb, kBF16) ||
        make_cache_tmap(&tv, vcache, B, Tcap, Hkv, D, sb, kBF16))
        return NC_EINVAL;
    switch (nc::dec::heads_per_warp(H)) {
        case 1: return launch_decode_tma<D, 1>(tk, tv, q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, Hkv, Tcap,
                                           eps, th, scale_log2, W, sb, nst, s);
        case 2: return launch_decode_tma<D, 2>(tk, tv, q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, Hkv, Tcap,
                                           eps, th, scale_log2, W, sb, nst, s);
        case 4: return launch_decode_tma<D, 4>(tk, tv, q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, Hkv, Tcap,
                                           eps, th, scale_log2, W, sb, nst, s);
        default: return NC_EINVAL;  // more than 4 * MAX_CWARPS heads: rejected by the callers
    }
}

}  // namespace

extern "C" {

int nc_version(void) { return (0 << 16) | 3; }

const char* nc_strerror(int code) {
    switch (code) {
        case NC_OK: return "ok";
        case NC_EINVAL: return "invalid argument";
        case NC_EUNSUPPORTED: return "unsupported device (needs sm_103)";
        case NC_ELAUNCH: return "CUDA launch failed";
        case NC_EDEVICE: return "CUDA device unavailable";
        case NC_ETOOLARGE: return "problem too large for the library's fixed decode scratch";
        default: return "unknown error";
    }
}

int nc_last_cuda_error(void) { return t_last_cuda_error; }

int nc_profile_enable(int on) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_on = on != 0;
    return NC_OK;
}

int nc_profile_read(nc_kernel_time* out, int max_entries, int* n_entries) {
    if (!n_entries || (max_entries > 0 && !out)) return NC_EINVAL;
    std::vector<ProfRec> recs;
    {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        recs.swap(g_prof_recs);
    }
    std::vector<nc_kernel_time> acc;
    int rc = NC_OK;
    for (const ProfRec& r : recs) {
        float ms = 0.f;
        cudaError_t e = cudaEventSynchronize(r.b);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.a, r.b);
        if (e != cudaSuccess) {
            t_last_cuda_error = static_cast<int>(e);
            rc = NC_ELAUNCH;
        }
        size_t i = 0;
        while (i < acc.size() && std::strcmp(acc[i].name, r.name) != 0) ++i;
        if (i == acc.size()) {
            nc_kernel_time z;
            std::memset(&z, 0, sizeof(z));
            std::strncpy(z.name, r.name, sizeof(z.name) - 1);
            acc.push_back(z);
        }
        acc[i].launches += 1;
        acc[i].kernels += r.kernels;
        acc[i].total_ms += ms;
    }
    {
        std::lock_guard<std::mutex> lock(g_prof_mu);
        for (const ProfRec& r : recs) {
            g_prof_pool.push_back(r.a);
            g_prof_pool.push_back(r.b);
        }
    }
    const int n = static_cast<int>(acc.size());
    for (int i = 0; i < n && i < max_entries; ++i) out[i] = acc[i];
    *n_entries = n;
    return rc;
}

int nc_device_status(nc_stream_t stream, unsigned int* status) {
    if (!status) return NC_EINVAL;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    unsigned int v = 0, zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, nc::g_dev_status, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(nc::g_dev_status, &zero, sizeof(zero));
    if (e != cudaSuccess) {
        t_last_cuda_error = static_cast<int>(e);
        return NC_ELAUNCH;
    }
    *status = v;
    return NC_OK;
}

size_t nc_attn_workspace_size(int op, int B, int T, int H, int D) {
    if (!shape_ok(B, T, H, D)) return 0;
    switch (op) {
        case NC_OP_NORM_ROPE:
        case NC_OP_FWD: return tab_bytes(T, D) + 256;  // RoPE table, pair counter
        case NC_OP_BWD: return bwd_ws_bytes(B, T, H, D);
        case NC_OP_DECODE: return decode_ws_layout(B, H, D, T, nullptr, nullptr);
        case NC_OP_PREFILL: return up256(static_cast<size_t>(B) * T * H * D * 2);  // qhat of the chunk
        case NC_OP_FWD_FP8: return D == nc::fwd8::D ? fp8_ws_layout(B, T, H, D, nullptr, nullptr) : 0;
        default: return 0;
    }
}

int nc_qk_norm_rope(const nc_bf16* x, const int32_t* pos, nc_bf16* xhat, float* rstd, void* workspace,
                    size_t workspace_bytes, int B, int T, int H, int D, float eps, float rope_base,
                    nc_stream_t stream) {
    if (!shape_ok(B, T, H, D) || !params_ok(eps, rope_base)) return NC_EINVAL;
    if (B == 0 || T == 0 || H == 0) return NC_OK;
    if (!x || !xhat || !workspace || !aligned16(x) || !aligned16(xhat) || !aligned256(workspace)) return NC_EINVAL;
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_NORM_ROPE, B, T, H, D)) return NC_EINVAL;
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const size_t n = static_cast<size_t>(B) * T * H * D * 2;
        CallRanges cr;
        cr.in(x, n), cr.in(pos, pos ? T * 4 : 0), cr.out(xhat, n), cr.out(rstd, rstd ? n / (2 * D) * 4 : 0);
        cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    float2* tab = reinterpret_cast<float2*>(workspace);
    if ((rc = launch_rope_table(tab, pos, T, D, rope_base, s))) return rc;
    return D == 64 ? launch_norm_rope<64, __nv_bfloat16>(x, nullptr, tab, xhat, nullptr, rstd, B, T, H, H, eps, s)
                   : launch_norm_rope<128, __nv_bfloat16>(x, nullptr, tab, xhat, nullptr, rstd, B, T, H, H, eps, s);
}

int nc_attn_fwd(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, nc_bf16* out,
                float* lse, nc_f16* qhat, nc_f16* khat, float* rstd, void* workspace, size_t workspace_bytes,
                int B, int T, int H, int D, float eps, float rope_base, nc_stream_t stream) {
    return nc_attn_fwd_ex(q, k, v, pos, out, lse, qhat, khat, rstd, workspace, workspace_bytes, B, T, H, D, eps,
                          rope_base, 0, 0, stream);
}

int nc_attn_fwd_ex(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, nc_bf16* out,
                   float* lse, nc_f16* qhat, nc_f16* khat, float* rstd, void* workspace, size_t workspace_bytes,
                   int B, int T, int H, int D, float eps, float rope_base, int window, int kv_heads,
                   nc_stream_t stream) {
    if (!shape_ok(B, T, H, D) || !params_ok(eps, rope_base) || window < 0) return NC_EINVAL;
    if (H > 0 && !kv_heads_of(kv_heads, H)) return NC_EINVAL;
    if (B == 0 || T == 0 || H == 0) return NC_OK;
    if (!q || !k || !v || !out || !lse || !qhat || !khat || !workspace) return NC_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(qhat) || !aligned16(khat) ||
        !aligned256(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return NC_EINVAL;
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_FWD, B, T, H, D)) return NC_EINVAL;
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const size_t tq = static_cast<size_t>(B) * T * H * D * 2, tk = tq / H * kv_heads_of(kv_heads, H);
        CallRanges cr;
        cr.in(q, tq), cr.in(k, tk), cr.in(v, tk), cr.in(pos, pos ? T * 4 : 0);
        cr.out(out, tq), cr.out(qhat, tq), cr.out(khat, tk), cr.out(lse, static_cast<size_t>(B) * H * T * 4);
        cr.out(rstd, rstd ? (tq + tk) / (2 * D) * 4 : 0), cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = window_eff(window, T);
    const int Hkv = kv_heads_of(kv_heads, H);
    return D == 64 ? fwd_impl<64>(q, k, v, pos, out, lse, qhat, khat, rstd, workspace, B, T, H, Hkv, eps, rope_base,
                                  W, s)
                   : fwd_impl<128>(q, k, v, pos, out, lse, qhat, khat, rstd, workspace, B, T, H, Hkv, eps, rope_base,
                                   W, s);
}

int nc_attn_fwd_fp8(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, nc_bf16* out,
                    float* lse, void* workspace, size_t workspace_bytes, int B, int T, int H, int D, float eps,
                    float rope_base, int window, int kv_heads, nc_stream_t stream) {
    if (!shape_ok(B, T, H, D) || D != nc::fwd8::D || !params_ok(eps, rope_base) || window < 0) return NC_EINVAL;
    if (H > 0 && !kv_heads_of(kv_heads, H)) return NC_EINVAL;
    if (B == 0 || T == 0 || H == 0) return NC_OK;
    if (!q || !k || !v || !out || !workspace) return NC_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned256(workspace) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return NC_EINVAL;
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_FWD_FP8, B, T, H, D)) return NC_EINVAL;
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const size_t tq = static_cast<size_t>(B) * T * H * D * 2, tk = tq / H * kv_heads_of(kv_heads, H);
        CallRanges cr;
        cr.in(q, tq), cr.in(k, tk), cr.in(v, tk), cr.in(pos, pos ? T * 4 : 0);
        cr.out(out, tq), cr.out(lse, lse ? static_cast<size_t>(B) * H * T * 4 : 0), cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    return fwd_fp8_impl(q, k, v, pos, out, lse, workspace, B, T, H, kv_heads_of(kv_heads, H), eps, rope_base,
                        window_eff(window, T), reinterpret_cast<cudaStream_t>(stream));
}

int nc_attn_bwd(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, const nc_bf16* out,
                const float* lse, const nc_f16* qhat, const nc_f16* khat, const nc_bf16* dout, nc_bf16* dq,
                nc_bf16* dk, nc_bf16* dv, void* workspace, size_t workspace_bytes, int B, int T, int H, int D,
                float eps, float rope_base, nc_stream_t stream) {
    return nc_attn_bwd_ex(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace, workspace_bytes, B, T, H,
                          D, eps, rope_base, 0, 0, stream);
}

int nc_attn_bwd_ex(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* pos, const nc_bf16* out,
                   const float* lse, const nc_f16* qhat, const nc_f16* khat, const nc_bf16* dout, nc_bf16* dq,
                   nc_bf16* dk, nc_bf16* dv, void* workspace, size_t workspace_bytes, int B, int T, int H, int D,
                   float eps, float rope_base, int window, int kv_heads, nc_stream_t stream) {
    if (!shape_ok(B, T, H, D) || !params_ok(eps, rope_base) || window < 0) return NC_EINVAL;
    if (H > 0 && !kv_heads_of(kv_heads, H)) return NC_EINVAL;
    if (B == 0 || T == 0 || H == 0) return NC_OK;
    if (!q || !k || !v || !out || !lse || !qhat || !khat || !dout || !dq || !dk || !dv || !workspace)
        return NC_EINVAL;
    const void* b16[] = {q, k, v, out, qhat, khat, dout, dq, dk, dv};
    for (const void* p : b16)
        if (!aligned16(p)) return NC_EINVAL;
    if (!aligned256(workspace) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return NC_EINVAL;
    if (2 * ds_rows(B, T, H) >= (1LL << 31)) return NC_EINVAL;  // 2^24 dS blocks: the limit the header states
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_BWD, B, T, H, D)) return NC_EINVAL;
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const size_t tq = static_cast<size_t>(B) * T * H * D * 2, tk = tq / H * kv_heads_of(kv_heads, H);
        CallRanges cr;
        cr.in(q, tq), cr.in(k, tk), cr.in(v, tk), cr.in(pos, pos ? T * 4 : 0), cr.in(out, tq);
        cr.in(lse, static_cast<size_t>(B) * H * T * 4), cr.in(qhat, tq), cr.in(khat, tk), cr.in(dout, tq);
        cr.out(dq, tq), cr.out(dk, tk), cr.out(dv, tk), cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = window_eff(window, T);
    const int Hkv = kv_heads_of(kv_heads, H);
    return D == 64 ? bwd_impl<64>(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace, B, T, H, Hkv, eps,
                                  rope_base, W, s)
                   : bwd_impl<128>(q, k, v, pos, out, lse, qhat, khat, dout, dq, dk, dv, workspace, B, T, H, Hkv, eps,
                                   rope_base, W, s);
}

int nc_attn_decode(const nc_bf16* q, const nc_bf16* k_new, const nc_bf16* v_new, nc_bf16* kcache, nc_bf16* vcache,
                   const int32_t* lens, nc_bf16* out, void* workspace, size_t workspace_bytes, int B, int H, int D,
                   int Tcap, float eps, float rope_base, nc_stream_t stream) {
    return nc_attn_decode_ex(q, k_new, v_new, kcache, vcache, lens, out, workspace, workspace_bytes, B, H, D, Tcap,
                             eps, rope_base, 0, 0, stream);
}

int nc_attn_decode_ex(const nc_bf16* q, const nc_bf16* k_new, const nc_bf16* v_new, nc_bf16* kcache,
                      nc_bf16* vcache, const int32_t* lens, nc_bf16* out, void* workspace, size_t workspace_bytes,
                      int B, int H, int D, int Tcap, float eps, float rope_base, int window, int kv_heads,
                      nc_stream_t stream) {
    if (!shape_ok(B, Tcap, H, D) || !params_ok(eps, rope_base) || window < 0) return NC_EINVAL;
    if (H > 0 && !kv_heads_of(kv_heads, H)) return NC_EINVAL;
    if (B == 0 || H == 0 || Tcap == 0) return NC_OK;
    if (!q || !kcache || !vcache || !lens || !out || !workspace) return NC_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return NC_EINVAL;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) || !aligned256(workspace) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))) || (reinterpret_cast<uintptr_t>(lens) & 3u))
        return NC_EINVAL;
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_DECODE, B, Tcap, H, D)) return NC_EINVAL;
    if (H * (D / 8) > 512) return NC_EINVAL;  // at most 512 / (D/8) heads
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const int Hkv = kv_heads_of(kv_heads, H);
        const size_t tq = static_cast<size_t>(B) * H * D * 2, tn = static_cast<size_t>(B) * Hkv * D * 2;
        const size_t tc = static_cast<size_t>(B) * Tcap * Hkv * D * 2;
        CallRanges cr;
        cr.in(q, tq), cr.in(k_new, k_new ? tn : 0), cr.in(v_new, v_new ? tn : 0), cr.in(lens, B * 4);
        cr.out(kcache, tc), cr.out(vcache, tc), cr.out(out, tq), cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    DecodeWs ws;
    decode_ws_layout(B, H, D, Tcap, &ws, workspace);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = window_eff(window, Tcap);
    const int Hkv = kv_heads_of(kv_heads, H);
    return D == 64 ? decode_impl<64>(q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, Hkv, Tcap, eps, rope_base,
                                     W, s)
                   : decode_impl<128>(q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, Hkv, Tcap, eps,
                                      rope_base, W, s);
}

int nc_attn_prefill(const nc_bf16* q, const nc_bf16* k, const nc_bf16* v, const int32_t* start, nc_bf16* kcache,
                    nc_bf16* vcache, nc_bf16* out, float* lse, void* workspace, size_t workspace_bytes, int B, int C,
                    int H, int D, int Tcap, float eps, float rope_base, int window, int kv_heads,
                    nc_stream_t stream) {
    if (!shape_ok(B, C, H, D) || !params_ok(eps, rope_base) || window < 0 || Tcap < C || Tcap > (1 << 24))
        return NC_EINVAL;
    if (H > 0 && !kv_heads_of(kv_heads, H)) return NC_EINVAL;
    if (B == 0 || C == 0 || H == 0) return NC_OK;
    if (!q || !k || !v || !start || !kcache || !vcache || !out || !workspace) return NC_EINVAL;
    const void* b16[] = {q, k, v, kcache, vcache, out};
    for (const void* p : b16)
        if (!aligned16(p)) return NC_EINVAL;
    if (!aligned256(workspace) || (reinterpret_cast<uintptr_t>(start) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
        return NC_EINVAL;
    if (workspace_bytes < nc_attn_workspace_size(NC_OP_PREFILL, B, C, H, D)) return NC_EINVAL;
    int rc = device_ready();
    if (rc) return rc;
    if (kChecked) {
        const int Hkv = kv_heads_of(kv_heads, H);
        const size_t tq = static_cast<size_t>(B) * C * H * D * 2, tk = static_cast<size_t>(B) * C * Hkv * D * 2;
        const size_t tc = static_cast<size_t>(B) * Tcap * Hkv * D * 2;
        CallRanges cr;
        cr.in(q, tq), cr.in(k, tk), cr.in(v, tk), cr.in(start, B * 4);
        cr.out(kcache, tc), cr.out(vcache, tc), cr.out(out, tq), cr.out(lse, lse ? static_cast<size_t>(B) * H * C * 4 : 0);
        cr.out(workspace, workspace_bytes);
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int W = window_eff(window, Tcap);
    const int Hkv = kv_heads_of(kv_heads, H);
    return D == 64 ? prefill_impl<64>(q, k, v, start, kcache, vcache, out, lse, workspace, B, C, H, Hkv, Tcap, eps,
                                      rope_base, W, s)
                   : prefill_impl<128>(q, k, v, start, kcache, vcache, out, lse, workspace, B, C, H, Hkv, Tcap, eps,
                                       rope_base, W, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode with no device allocation at all.
//
// Some callers cannot hand the library a workspace: a serving loop that must
// not call cudaMalloc between tokens (it synchronises the whole device and
// stalls every stream), or a host application that owns all device memory
// and lends none of it to plug-ins.  For them the decode keeps its scratch
// (per-chunk partial results and per-stream arrival counters) in the fixed
// array below, which exists once per device for as long as the library is
// loaded.
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[NC_DECODE_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices];  // device address of g_decode_scratch, per device

// Host code cannot use the array's name as a device address; look the
// address up once per device, with that device current.
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        t_last_cuda_error = static_cast<int>(e);
        return NC_EDEVICE;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            t_last_cuda_error = static_cast<int>(e);
            return NC_EDEVICE;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return NC_OK;
}

}  // namespace

extern "C" {

int nc_attn_decode_noalloc(const nc_bf16* q, const nc_bf16* k_new, const nc_bf16* v_new, nc_bf16* kcache,
                           nc_bf16* vcache, const int32_t* lens, nc_bf16* out, int B, int H, int D, int Tcap,
                           float eps, float rope_base, nc_stream_t stream) {
    if (!shape_ok(B, Tcap, H, D) || !params_ok(eps, rope_base)) return NC_EINVAL;
    if (B == 0 || H == 0 || Tcap == 0) return NC_OK;
    if (!q || !kcache || !vcache || !lens || !out) return NC_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return NC_EINVAL;
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(out) ||
        (k_new && (!aligned16(k_new) || !aligned16(v_new))) || (reinterpret_cast<uintptr_t>(lens) & 3u))
        return NC_EINVAL;
    if (nc_attn_workspace_size(NC_OP_DECODE, B, Tcap, H, D) > NC_DECODE_NOALLOC_SCRATCH_BYTES)
        return NC_ETOOLARGE;
    if (H * (D / 8) > 512) return NC_EINVAL;  // at most 512 / (D/8) heads
    int rc = device_ready();
    if (rc) return rc;
    void* scratch = nullptr;
    if ((rc = scratch_address(&scratch))) return rc;
    if (kChecked) {
        const size_t tq = static_cast<size_t>(B) * H * D * 2, tc = static_cast<size_t>(B) * Tcap * H * D * 2;
        CallRanges cr;
        cr.in(q, tq), cr.in(k_new, k_new ? tq : 0), cr.in(v_new, v_new ? tq : 0), cr.in(lens, B * 4);
        cr.out(kcache, tc), cr.out(vcache, tc), cr.out(out, tq);
        cr.out(scratch, nc_attn_workspace_size(NC_OP_DECODE, B, Tcap, H, D));
        if ((rc = cr.publish(reinterpret_cast<cudaStream_t>(stream)))) return rc;
    }
    DecodeWs ws;
    decode_ws_layout(B, H, D, Tcap, &ws, scratch);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the array keeps whatever the previous call left: the arrival counters
    // must start from zero
    if (cudaMemsetAsync(ws.counters, 0, static_cast<size_t>(B) * sizeof(unsigned int), s) != cudaSuccess)
        return launch_status();
    const int W = window_eff(0, Tcap);
    return D == 64 ? decode_impl<64>(q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, H, Tcap, eps, rope_base, W,
                                     s)
                   : decode_impl<128>(q, k_new, v_new, kcache, vcache, lens, out, ws, B, H, H, Tcap, eps, rope_base,
                                      W, s);
}

}  // extern "C"
