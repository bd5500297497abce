/*
 * ncattn.h -- C ABI of the B300 (sm_103a) causal attention library with
 * parameter-free QK RMSNorm and rotary position embeddings.
 *
 * The operation.  Per batch b, head h and head dimension D (64 or 128):
 *   qhat_t = RoPE(q_t / sqrt(mean(q_t^2) + eps), pos_t),  khat_t likewise
 *   out_i  = sum_{j <= i} softmax_j(qhat_i . khat_j / sqrt(D)) v_j
 *   lse_i  = ln sum_{j <= i} exp(qhat_i . khat_j / sqrt(D))
 * RoPE rotates the pair (x_i, x_{i+D/2}) by the angle pos * base^(-2i/D),
 * i < D/2 (rotate-half pairing).
 *
 * Where it comes from.  nanochat's GPT block replaces positional embeddings
 * with rotary embeddings and normalises queries and keys (QK-norm, RMSNorm
 * without trainable parameters) before the dot product: ai.flicky.cc,
 * "nanochat: свой ChatGPT от токенизатора до чата", section
 * "Модель: что изменилось со времён GPT-2"; adg.csdn.net,
 * "4小时100美元！...nanochat...", section "1. 极致精简的技术架构".  Attention
 * runs through FlashAttention-3 with an SDPA fallback and generation uses a
 * KV cache with prefill/decode (ai.flicky.cc, section "Карта репозитория";
 * 7minutos.es "Andrej Karpathy lanza nanochat ...", section
 * "Entrenamiento medio, SFT y uso de herramientas").  The pages give no
 * formula; the pairing, the angle, eps placement and the per-head norm axis
 * above are the plainest reading they support.
 *
 * Conventions for every entry point.
 *  - Pointers are DEVICE pointers owned by the caller; the library keeps no
 *    pointer after the call returns and allocates no memory.  Scratch space
 *    is the caller's `workspace` of at least nc_attn_workspace_size() bytes,
 *    256-byte aligned.
 *  - bf16 tensors are raw bfloat16 bits (nc_bf16), row-major and
 *    contiguous: token tensors [B][T][H][D], lse [B][H][T] (fp32, natural
 *    log), decode tensors [B][H][D], caches [B][Tcap][H][D].  (With
 *    grouped-query attention, through the *_ex calls and nc_attn_prefill,
 *    the key/value-side tensors and the caches have Hkv heads instead of H.)
 *    Every 16-bit tensor must be 16-byte aligned.
 *  - Every 16-bit tensor is bf16 (nc_bf16), the KV caches included (the key
 *    cache holds keys normalised and rotated at their slot position), except
 *    qhat and khat, the normalised, rotated q and k that nc_attn_fwd writes
 *    and nc_attn_bwd reads back: these are this library's own side outputs,
 *    kept in IEEE fp16 (nc_f16).  RMSNorm bounds each of their elements by
 *    sqrt(D), well inside fp16's range, and fp16 carries 3 more mantissa bits
 *    than bf16 into the score products: with bf16 side outputs the forward's
 *    largest error against the exact result measured 1.02e-2 on a seeded
 *    128-head-dim-64 case, past the 1e-2 bound this library is held to, and
 *    within it with fp16.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and the call returns without synchronising.
 *  - Return value: NC_OK, or a negative code.  NC_EINVAL: a null pointer
 *    where one is required, misalignment, D not 64/128, a negative size,
 *    eps < 0, rope_base <= 0, or a workspace that is too small; nothing is
 *    launched.  NC_EUNSUPPORTED: the current device is not sm_103.
 *    NC_ELAUNCH: a CUDA launch (or the library's one-time per-device setup)
 *    failed; nc_last_cuda_error() gives the cudaError_t.  A size of zero in B, T or H (Tcap for decode) is an empty
 *    problem: NC_OK, nothing launched.
 *  - Kernels never spin unboundedly: a pipeline wait that has not completed
 *    after 2 s records a device-side status word and the kernel unwinds.
 *    nc_device_status() reads and clears it.
 */
#ifndef NCATTN_H
#define NCATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* 16-bit element types.  Distinct struct types (one uint16_t of raw bits
 * each), so that a compiler rejects an fp16 tensor passed where a bf16 one is
 * expected and the reverse; pointers to them are plain data pointers. */
typedef struct nc_bf16 { uint16_t bits; } nc_bf16; /* raw bfloat16 bits */
typedef struct nc_f16 { uint16_t bits; } nc_f16;   /* raw IEEE binary16 bits */
typedef struct CUstream_st *nc_stream_t; /* == cudaStream_t */

#define NC_OK 0
#define NC_EINVAL (-1)
#define NC_EUNSUPPORTED (-2)
#define NC_ELAUNCH (-3)
#define NC_EDEVICE (-4)

#define NC_OP_FWD 0
#define NC_OP_BWD 1
#define NC_OP_DECODE 2
#define NC_OP_NORM_ROPE 3
#define NC_OP_PREFILL 4
#define NC_OP_FWD_FP8 5

/* Library version, (major << 16) | minor.  0.2: the sliding-window calls
 * became the *_ex calls with a kv_heads argument (grouped-query attention),
 * and nc_attn_prefill gained kv_heads.  0.3: the key cache (decode, prefill,
 * nc_qk_norm_rope) is bf16 (it was IEEE fp16); nc_bf16 and nc_f16 are
 * distinct types; the backward workspace holds the dS scratch. */
int nc_version(void);

/* Human-readable name of an NC_* code. */
const char *nc_strerror(int code);

/* cudaError_t of the last failed launch in this thread (0 if none). */
int nc_last_cuda_error(void);

/* Synchronises `stream`, then reads and clears the device status word of
 * the current device.  *status = 0 when no kernel has reported a failure,
 * else (code << 16) | site with code 1 = a bounded wait timed out,
 * 2 = a decode length outside [1, Tcap] or a prefill chunk outside its cache.  Returns NC_OK or NC_ELAUNCH. */
int nc_device_status(nc_stream_t stream, unsigned int *status);

/* Optional per-kernel timing.  While enabled (on != 0), every step of a
 * call (one kernel, or a few launched back to back under one name: the
 * forward's two launches, the prologue's q and k launches with grouped-query
 * attention) is bracketed by two CUDA events recorded on the launch stream.
 * nc_profile_read() waits for the recorded events, writes up to max_entries
 * per-name sums (steps timed, kernels launched, total milliseconds) to
 * `out`, sets *n_entries to the number of distinct names, and clears the
 * record.  Timing does not change what the kernels compute. */
typedef struct {
    char name[48];
    int launches; /* timed steps */
    int kernels;  /* kernel launches inside them */
    double total_ms;
} nc_kernel_time;

int nc_profile_enable(int on);
int nc_profile_read(nc_kernel_time *out, int max_entries, int *n_entries);

/* Workspace bytes needed by an operation (op = NC_OP_*).  For
 * NC_OP_DECODE pass T = Tcap.  The decode workspace holds per-stream
 * counters that must be zero before the first call; every successful
 * call leaves them at zero again. */
size_t nc_attn_workspace_size(int op, int B, int T, int H, int D);

/* QK RMSNorm + RoPE alone (prefill of a KV cache, or a check of the
 * prologue): xhat = RoPE(x / sqrt(mean(x^2) + eps), pos) for x [B][T][H][D].
 * xhat is bf16, the key cache's format.  pos: [T] int32 positions, or NULL for 0..T-1.  rstd:
 * optional [B][T][H] fp32 output of 1/sqrt(mean(x^2) + eps).
 * Workspace: NC_OP_NORM_ROPE. */
int nc_qk_norm_rope(const nc_bf16 *x, const int32_t *pos, nc_bf16 *xhat, float *rstd, void *workspace,
                    size_t workspace_bytes, int B, int T, int H, int D, float eps, float rope_base,
                    nc_stream_t stream);

/* Forward.  In: q, k, v [B][T][H][D]; pos [T] or NULL (0..T-1).
 * Out: out [B][T][H][D]; lse [B][H][T]; qhat, khat [B][T][H][D] (the
 * normalised, rotated q and k in fp16, kept for the backward); rstd
 * optional [2][B][T][H] (q then k).  Scale 1/sqrt(D).  Workspace: NC_OP_FWD (the RoPE
 * table and the counter the persistent kernel's CTAs take tile pairs from). */
int nc_attn_fwd(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *pos, nc_bf16 *out,
                float *lse, nc_f16 *qhat, nc_f16 *khat, float *rstd, void *workspace, size_t workspace_bytes,
                int B, int T, int H, int D, float eps, float rope_base, nc_stream_t stream);

/* Backward.  In: the forward's inputs q, k, v, pos, its outputs out, lse,
 * qhat, khat, and the upstream gradient dout [B][T][H][D].  Out: dq, dk, dv
 * [B][T][H][D] (gradients with respect to the RAW q, k, v: through the
 * softmax, the RoPE rotation and the RMSNorm).  Every output element is
 * computed by one CTA (a key-side kernel writes dk and dv, a query-side
 * kernel dq): no atomics, bit-identical results on repeated calls.
 * Workspace: NC_OP_BWD, overwritten by every call: the RoPE table, per-row
 * delta and lse, two maxima and the two counters that the persistent
 * kernels' CTAs take tiles from, and the dS scratch.  The key-side kernel
 * forms each
 * visible 128 x 128 block of dS = P o (dP - delta) once and writes it there
 * (fp16, times one power of two for the whole call) for the query side's
 * dq = dS khat, so the workspace grows with B * H * n(n+1)/2 blocks of
 * 32 KB, n = ceil(T / 128) (1.4 GB at B = 32, T = 2048, H = 10).  Problems
 * with B * H * n(n+1)/2 >= 2^24 blocks (512 GB of scratch) are NC_EINVAL. */
int nc_attn_bwd(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *pos, const nc_bf16 *out,
                const float *lse, const nc_f16 *qhat, const nc_f16 *khat, const nc_bf16 *dout, nc_bf16 *dq,
                nc_bf16 *dk, nc_bf16 *dv, void *workspace, size_t workspace_bytes, int B, int T, int H, int D,
                float eps, float rope_base, nc_stream_t stream);

/* Single-token decode over a KV cache.  Stream b holds lens[b] valid cache
 * slots (1 <= lens[b] <= Tcap) INCLUDING the new token, whose position is
 * lens[b]-1.  q [B][H][D] is the new token's raw query.  If k_new and v_new
 * ([B][H][D], raw) are given, the new key is normalised and rotated and
 * written with v_new into slot lens[b]-1 of kcache / vcache first;
 * otherwise that slot must already hold them.  kcache holds keys already
 * normalised and rotated at their slot position (as nc_qk_norm_rope writes
 * them); vcache holds raw values; both bf16.
 * out [B][H][D] bf16.  Up to 512 / (D/8) heads (32 at D = 128).
 * Workspace: NC_OP_DECODE with T = Tcap (zeroed once before first use). */
int nc_attn_decode(const nc_bf16 *q, const nc_bf16 *k_new, const nc_bf16 *v_new, nc_bf16 *kcache,
                   nc_bf16 *vcache, const int32_t *lens, nc_bf16 *out, void *workspace, size_t workspace_bytes,
                   int B, int H, int D, int Tcap, float eps, float rope_base, nc_stream_t stream);

/* Sliding-window and grouped-query variants of the three calls above (same
 * arguments, plus `window` and `kv_heads`; window = kv_heads = 0 gives
 * exactly the calls above).
 *
 * window: query i sees key j exactly when 0 <= i - j < window: the
 * window's most recent positions, its own included.  The pages run most
 * layers with a short window of a quarter of the context (ai.flicky.cc,
 * "nanochat: свой ChatGPT от токенизатора до чата", section "Модель: что
 * изменилось со времён GPT-2", window-pattern bullet: pattern SSSL, the last
 * layer always full); the boundary convention is this library's reading.
 * window == 0 (or >= the sequence length / cache capacity) is the plain
 * causal mask, exactly the calls above; window < 0 is NC_EINVAL.  Key tiles
 * that no query of a tile can see are skipped, so the work shrinks with the
 * window.  For decode, position p = lens[b] - 1 attends slots
 * max(0, p - window + 1) .. p.
 *
 * kv_heads: the number Hkv of key/value heads (grouped-query attention, an
 * option of the pages' model: ai.flicky.cc, "nanochat: свой ChatGPT от
 * токенизатора до чата", section "Модель: что изменилось со времён GPT-2",
 * GQA bullet).  0 means H (plain multi-head attention); otherwise it must
 * divide H, else NC_EINVAL.  Query head h uses key/value head h / (H / Hkv):
 * consecutive query heads share one.  Every key-side tensor then has Hkv
 * heads instead of H: k, v, khat, dk, dv [B][T][Hkv][D], k_new and v_new
 * [B][Hkv][D], kcache and vcache [B][Tcap][Hkv][D]; rstd is the q rows'
 * [B][T][H] followed by the k rows' [B][T][Hkv].  dk and dv sum the
 * gradients of the query heads of each group (the key-side kernel walks all
 * of them for its key tile, still without atomics).  Workspace sizes are
 * those of the plain calls with H query heads. */
int nc_attn_fwd_ex(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *pos, nc_bf16 *out,
                   float *lse, nc_f16 *qhat, nc_f16 *khat, float *rstd, void *workspace, size_t workspace_bytes,
                   int B, int T, int H, int D, float eps, float rope_base, int window, int kv_heads,
                   nc_stream_t stream);
int nc_attn_bwd_ex(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *pos, const nc_bf16 *out,
                   const float *lse, const nc_f16 *qhat, const nc_f16 *khat, const nc_bf16 *dout, nc_bf16 *dq,
                   nc_bf16 *dk, nc_bf16 *dv, void *workspace, size_t workspace_bytes, int B, int T, int H, int D,
                   float eps, float rope_base, int window, int kv_heads, nc_stream_t stream);
int nc_attn_decode_ex(const nc_bf16 *q, const nc_bf16 *k_new, const nc_bf16 *v_new, nc_bf16 *kcache,
                      nc_bf16 *vcache, const int32_t *lens, nc_bf16 *out, void *workspace, size_t workspace_bytes,
                      int B, int H, int D, int Tcap, float eps, float rope_base, int window, int kv_heads,
                      nc_stream_t stream);

/* FP8 forward (head dimension 128): the forward of nc_attn_fwd_ex with its
 * products in E4M3 on the tensor cores (fp32 accumulation).  The pages name
 * an fp8 training path (ai.flicky.cc, "nanochat: свой ChatGPT от
 * токенизатора до чата", section "Карта репозитория", fp8.py row; the
 * "+fp8" leaderboard row of pigsec.cn "karpathy/nanochat") and give no
 * scheme for attention; this library's reading:
 *   qhat and khat (normalised and rotated as in nc_attn_fwd) are rounded to
 *   E4M3 after scaling by 2^5 (QK-norm bounds their elements by sqrt(D), so
 *   they stay within E4M3's 448); v by 2^tau per (batch, key/value head),
 *   tau the largest integer keeping max |v| 2^tau <= 448 (clamped to
 *   [-126, 126]); the probabilities p = exp(s - row max) by 2^8.
 *   out = sum_j P8_j v8_j / sum_j P8_j (rows of quantised weights that sum
 *   to one), lse = row max + ln sum_j p (unquantised).
 * Same arguments as nc_attn_fwd_ex minus qhat, khat and rstd (nothing is
 * kept for a backward); lse may be NULL.  Workspace: NC_OP_FWD_FP8 (RoPE
 * table, the E4M3 operands, the value scales).  D != 128 is NC_EINVAL. */
int nc_attn_fwd_fp8(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *pos, nc_bf16 *out,
                    float *lse, void *workspace, size_t workspace_bytes, int B, int T, int H, int D, float eps,
                    float rope_base, int window, int kv_heads, nc_stream_t stream);

/* Chunk prefill into a KV cache.  Stream b appends C new tokens at
 * positions start[b] .. start[b] + C - 1 (start: [B] int32, device): their
 * raw q [B][C][H][D] and k, v [B][C][Hkv][D] are normalised and rotated
 * at those positions (Hkv = kv_heads, 0 meaning H, as in the *_ex calls);
 * the keys (normalised and rotated, as nc_qk_norm_rope writes them)
 * and the values go into slots start[b] .. start[b] + C - 1 of kcache /
 * vcache [B][Tcap][Hkv][D]; each new query attends causally over slots
 * 0 .. its own position (the last `window` of them when window > 0, as in
 * the *_ex calls).  out [B][C][H][D] bf16; lse [B][H][C] fp32, natural log,
 * or NULL.  The slots before start[b] must already hold the stream's keys
 * and values, the keys normalised and rotated (as this call, nc_attn_decode
 * or nc_qk_norm_rope write them).  The prefill's softmax relies on that: it
 * subtracts the fixed offset sqrt(D) * 1.0079, which bounds every score
 * only when both vectors have norm at most sqrt(D).  A slot holding anything
 * else is not detected: its scores may exceed the offset, the row's weights
 * are then no longer bounded by 1, and a key whose norm exceeds about
 * sqrt(D) * 1.0079 + 88 can overflow the rows that see it to inf or NaN.
 * (Decode keeps a running maximum and has no such precondition.)  With start[b] = 0 and C = T this is nc_attn_fwd_ex over the
 * chunk (plus the cache writes); a prompt may also be fed in several chunks,
 * each starting where the previous one ended.  The pages prefill the KV
 * cache before decoding (ai.flicky.cc, "nanochat: свой ChatGPT от
 * токенизатора до чата", section "Карта репозитория", engine.py row).
 * A stream with start[b] < 0 or start[b] + C > Tcap is skipped and recorded
 * in the device status word (2).  Workspace: NC_OP_PREFILL with T = C. */
int nc_attn_prefill(const nc_bf16 *q, const nc_bf16 *k, const nc_bf16 *v, const int32_t *start, nc_bf16 *kcache,
                    nc_bf16 *vcache, nc_bf16 *out, float *lse, void *workspace, size_t workspace_bytes, int B,
                    int C, int H, int D, int Tcap, float eps, float rope_base, int window, int kv_heads,
                    nc_stream_t stream);

/* Decode without any device allocation.  The pages have no counterpart to
 * this call; it exists for callers that cannot provide a workspace: a
 * token-by-token serving loop that must not call cudaMalloc (which
 * synchronises the whole device), or a host program that owns all device
 * memory and lends none to the library.  It computes exactly what
 * nc_attn_decode computes, with the same arguments minus the workspace.
 *  - Scratch lives in one fixed array of NC_DECODE_NOALLOC_SCRATCH_BYTES
 *    (16 MiB) inside the library, present on every device that loads the
 *    library until the process exits.  Problems whose decode workspace
 *    (nc_attn_workspace_size(NC_OP_DECODE, B, Tcap, H, D)) exceeds it are
 *    rejected with NC_ETOOLARGE; nothing is launched.  (The 32-stream,
 *    10-head, D = 128, capacity 2048 case needs about 10.6 MB.)
 *  - The first call on a device looks up the array's device address; make
 *    that first call before any stream capture.
 *  - Every call on a device shares the one array.  Calls that may overlap on
 *    the GPU (different streams without ordering between them) race on it and
 *    give wrong results; order them, or use nc_attn_decode with separate
 *    workspaces.  Each call clears the counters it needs at its start.
 *  - No cudaMalloc, cudaFree or allocating library routine is called. */
#define NC_ETOOLARGE (-5)
#define NC_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

int nc_attn_decode_noalloc(const nc_bf16 *q, const nc_bf16 *k_new, const nc_bf16 *v_new, nc_bf16 *kcache,
                           nc_bf16 *vcache, const int32_t *lens, nc_bf16 *out, int B, int H, int D, int Tcap,
                           float eps, float rope_base, nc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* NCATTN_H */
