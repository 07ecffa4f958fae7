/*
 * nea_attn.h -- C ABI of the causal grouped-query FlashAttention library
 * (forward and backward) for GB300 / sm_103a.
 *
 * What it computes.  Softmax attention with a causal mask and grouped-query
 * heads, and its gradient:
 *   "NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", section "Tiled
 *   FlashAttention" -- attention computed tile by tile with an online
 *   softmax, so that no N x N matrix reaches global memory;
 *   same post, "Architecture Deep Dive" -- a GPT-2 style decoder, so row i
 *   attends keys j <= i;
 *   same post, "Build and Run" (config file: num_heads 12, num_kv_heads 4)
 *   -- grouped-query attention; query head h reads KV head h / (H / Hkv);
 *   same post, "Hand-written Backpropagation" -- a hand-derived backward.
 *
 *   S_ij = scale * Q_i . K_j          P = softmax_j(S) (j <= i when causal)
 *   O_i  = sum_j P_ij V_j             LSE_i = ln sum_j exp(S_ij)
 *   dP_ij = dO_i . V_j   D_i = dO_i . O_i   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i = scale sum_j dS_ij K_j
 *   dK_j = scale sum_{h in group} sum_i dS_ij Q_i
 *   dV_j =       sum_{h in group} sum_i P_ij dO_i
 *
 * Conventions shared by every entry point.
 *   Pointers are DEVICE pointers (from cudaMalloc or any allocator of the
 *   current device), 16-byte aligned, to contiguous row-major arrays:
 *     Q, O, dO, dQ : [B][H][N][d]        K, V, dK, dV : [B][Hkv][N][d]
 *     LSE          : [B][H][N] float32, natural log of the scaled logits
 *   Element type of Q/K/V/O/dO/dQ/dK/dV is `dtype` (bf16 or fp32); all
 *   accumulation is fp32; bf16 path: P and dS enter the tensor cores as
 *   bf16; fp32 path: operands enter as TF32.
 *   Supported: d in {64, 128} for bf16, d = 64 for fp32; H % Hkv == 0;
 *   any N >= 1 (a last, partial 128-row tile is masked inside the kernels);
 *   causal in {0, 1}; scale finite and > 0; B >= 1.
 *   `stream` is a cudaStream_t (NULL = legacy default stream).
 *   The caller owns every buffer.  No entry point allocates device memory.
 *   Calls validate their arguments on the host and return a status code
 *   synchronously; kernels then run asynchronously on `stream`.  Errors met
 *   while the kernels run are reported by nea_attn_check_status().  Outputs
 *   are unspecified when the status is not NEA_OK.
 *   Not thread-safe with respect to nea_attn_check_status() on the same
 *   device: the device status word is shared by all calls of the process.
 */
#ifndef NEA_ATTN_H_
#define NEA_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  NEA_OK = 0,
  NEA_ERR_INVALID = -1,     /* bad argument: null / misaligned pointer, bad size */
  NEA_ERR_UNSUPPORTED = -2, /* valid but not implemented (d, dtype, ragged N) */
  NEA_ERR_CUDA = -3,        /* a CUDA runtime / driver call failed */
  NEA_ERR_TIMEOUT = -4,     /* a kernel's bounded wait gave up (see check_status) */
  NEA_ERR_WORKSPACE = -5    /* workspace null, misaligned or too small */
} nea_status;

typedef enum { NEA_BF16 = 0, NEA_F32 = 1 } nea_dtype;

/*
 * Forward.  Writes O [B,H,N,d] (dtype) and LSE [B,H,N] (fp32, natural log).
 * Section "Tiled FlashAttention": the work is one item per 128-row query tile
 * of one (batch, head); K/V tiles of 128 rows stream through shared memory;
 * tiles entirely above the causal diagonal are skipped.  bf16 runs one wave
 * of persistent CTAs that each take several items; fp32 one CTA per item.
 * One launch on `stream`; no allocation; returns NEA_OK or the error code of
 * the first failed check or launch.
 */
int nea_attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H,
                 int Hkv, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Bytes of device workspace nea_attn_bwd() needs for these sizes (256-byte
 * aligned sub-buffers, with Npad = N rounded up to a multiple of 128:
 * D [B*H][Npad] fp32, -LSE*log2(e) [B*H][Npad] fp32, then for bf16 the fp32
 * dQ accumulator [B,H,N,d] and two 2 KB row-term tiles per 128-row query
 * tile [B*H][Npad/128][2][2048 B], for fp32 the transposed operands Q^T,
 * dO^T [B*H][d][Npad] and K^T [B*Hkv][d][Npad]).  Returns 0 for invalid or
 * unsupported sizes.
 */
size_t nea_attn_bwd_workspace_bytes(int B, int H, int Hkv, int N, int d, int dtype);

/*
 * Backward.  Given the forward's inputs, its O and LSE, and the upstream
 * gradient dO, writes dQ [B,H,N,d], dK and dV [B,Hkv,N,d] (dtype).
 * Section "Hand-written Backpropagation": the gradient is derived by hand
 * and P is recomputed from LSE instead of stored.  bf16: three kernels run
 * in order on `stream`: a preprocess D = rowsum(dO * O) (which also clears
 * the dQ accumulator), the main kernel (one CTA per 128-row KV tile of one
 * (batch, KV head); dK and dV are summed over the group's query heads in
 * tensor memory, without atomics; dQ partials are added into the fp32
 * accumulator by TMA reductions), and a cast of dQ.  fp32 (TF32 tensor
 * cores, whose operands must be K-major): the preprocess, tf32-rounded
 * transposes of Q, dO and K into the workspace, a dK/dV kernel per KV tile
 * and a dQ kernel per query tile (each dQ tile written once).
 * `workspace` is a device buffer of at least
 * nea_attn_bwd_workspace_bytes(...) bytes, 256-byte aligned, owned by the
 * caller and not used concurrently by another call; its contents on entry
 * do not matter.  The order of the dQ additions is not fixed, so dQ may
 * differ between runs in the last bits; dK and dV are deterministic (for a
 * bit-reproducible dQ see nea_attn_bwd_ex() with NEA_BWD_DETERMINISTIC).
 */
int nea_attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                 const float* LSE, void* dQ, void* dK, void* dV, void* workspace,
                 size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale,
                 int causal, int dtype, void* stream);

/*
 * The three stages nea_attn_bwd() runs, exposed so that a caller can place
 * events between them (profiling) or overlap them with its own work.  Called
 * in this order on one stream, with one workspace, they are exactly
 * nea_attn_bwd().  Arguments mean the same as there.
 *
 * Stage 1, preprocess (HBM-bound): writes scale * rowsum(dO * O) and
 * -LSE * log2(e) per row into the workspace and clears the fp32 dQ
 * accumulator (for fp32 dtype the accumulator is dQ itself).
 */
int nea_attn_bwd_preprocess(const void* O, const void* dO, const float* LSE, void* dQ,
                            void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                            int N, int d, float scale, int dtype, void* stream);

/*
 * Stage 2, main kernel(s): reads Q, K, V, dO and the stage-1 workspace;
 * writes dK, dV and (bf16) adds every dQ partial into the accumulator or
 * (fp32) writes dQ.
 */
int nea_attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                      void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H,
                      int Hkv, int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Stage 3, finalize: dQ = bf16(accumulator) for bf16; nothing to do (and
 * NEA_OK) for fp32.
 */
int nea_attn_bwd_finalize(void* dQ, void* workspace, size_t workspace_bytes, int B, int H,
                          int Hkv, int N, int d, int dtype, void* stream);

/*
 * Backward without a caller workspace.  The pages have no counterpart: this
 * entry point exists for callers that cannot allocate device memory -- a
 * host framework that hands a plugin only its input and output pointers, or
 * a path on which cudaMalloc (which can synchronise the whole device) is not
 * allowed.  Same arguments and results as nea_attn_bwd() minus the
 * workspace; the scratch it needs (the layout nea_attn_bwd_workspace_bytes()
 * describes: for bf16 D, -LSE*log2(e), the fp32 dQ accumulator and the
 * row-term tiles of the main kernel, about 4*d + 40 bytes per query row;
 * for fp32 D, -LSE*log2(e) and the transposed Q, dO and K, about
 * 4*(2d+2) bytes per query row plus 4*d per key row) lives in a fixed
 * array of nea_attn_bwd_noalloc_max_bytes() bytes (32 MiB) inside the
 * library.  So bf16 takes up to about 113,000 query rows (B*H*N) at
 * d = 64 (the GPT-2-small shape, 98,304 rows, fits) and 60,000 at d = 128;
 * fp32 at d = 64 about 43,000 (H = Hkv) to 55,000 (H = 3 Hkv).
 *   - Sizes whose nea_attn_bwd_workspace_bytes() exceeds that maximum return
 *     NEA_ERR_WORKSPACE and launch nothing.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  The first
 *     call on a device looks up the array's device address there
 *     (cudaGetSymbolAddress) and caches it.  With CUDA's lazy module loading
 *     (the default) that lookup is also when the runtime loads the part of
 *     the library that holds the array and reserves its 32 MiB on that
 *     device, which then stays reserved until the process exits.  Make the
 *     first call outside any latency-critical path and before any stream
 *     capture.
 *   - Every call uses the same array, and each call rewrites all of it that
 *     it reads (the dQ accumulator is cleared by the preprocess kernel), so
 *     sequential calls are independent.  Calls that overlap on the GPU (other
 *     streams, other host threads) race on the array: serialise them.
 */
int nea_attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                         int H, int Hkv, int N, int d, float scale, int causal, int dtype,
                         void* stream);

/* Size in bytes of the scratch array behind nea_attn_bwd_noalloc(). */
size_t nea_attn_bwd_noalloc_max_bytes(void);

/*
 * Rotary position embedding (RoPE).  The pages name RoPE among the model's
 * techniques ("NanoEuler: Hand-writing GPT-2 in Pure C/CUDA", FAQ on llm.c)
 * without a formula; these calls implement the original rotary embedding:
 * the pair (x_2i, x_2i+1) of the row at position n (n = row index within its
 * head, 0 .. N-1) turns by the angle n * theta_i, theta_i = base^(-2i/d):
 *   y_2i = x_2i cos - x_2i+1 sin,   y_2i+1 = x_2i sin + x_2i+1 cos.
 * Use: build the table once per (N, d, base); rotate Q and K into Qr, Kr;
 * run nea_attn_fwd() on (Qr, Kr, V); for the gradients call
 * nea_attn_bwd_rope(), which returns dQ and dK with respect to the
 * caller's unrotated Q and K.
 */

/*
 * Writes cos_sin [N][d/2][2] fp32 (cos, sin of n * theta_i, computed in
 * fp64).  cos_sin: device pointer, 8-byte aligned, N*d*4 bytes, owned by the
 * caller.  d even and >= 2, N >= 1, base finite and > 0, else
 * NEA_ERR_INVALID.  Asynchronous on `stream`.
 */
int nea_rope_table(float* cos_sin, int N, int d, double base, void* stream);

/*
 * Qr = R(Q), Kr = R(K) for Q [B,H,N,d], K [B,Hkv,N,d] (dtype), rotated in
 * fp32 and rounded once to the dtype.  Qr/Kr may alias Q/K (in place).  All
 * pointers 16-byte aligned device pointers; cos_sin from nea_rope_table()
 * for the same N and d.  Shape rules as for nea_attn_fwd().
 */
int nea_rope_qk(const void* Q, const void* K, void* Qr, void* Kr, const float* cos_sin, int B,
                int H, int Hkv, int N, int d, int dtype, void* stream);

/*
 * Forward with the rotation of Q done inside the kernel: Q is the caller's
 * unrotated Q, Kr the rotated K (e.g. from nea_rope_qk()), cos_sin the
 * table; O and LSE are those of nea_attn_fwd() on (R(Q), Kr, V).  Each
 * query tile is rotated in shared memory once it has landed, before its
 * first S = Q K^T (fp32 arithmetic, one rounding to bf16, as
 * nea_rope_qk()), so R(Q) is never written to memory.  bf16 only (fp32:
 * NEA_ERR_UNSUPPORTED); cos_sin 16-byte aligned, else NEA_ERR_INVALID;
 * other arguments as nea_attn_fwd().  The backward needs R(Q) itself
 * (nea_attn_bwd_rope() takes Qr, Kr).
 */
int nea_attn_fwd_rope_q(const void* Q, const void* Kr, const void* V, void* O, float* LSE,
                        const float* cos_sin, int B, int H, int Hkv, int N, int d, float scale,
                        int causal, int dtype, void* stream);

/*
 * Backward of attention on rotated inputs.  Arguments as nea_attn_bwd(),
 * with Qr, Kr the rotated Q and K the forward ran on, and cos_sin the table
 * they were rotated with.  dV is as nea_attn_bwd() gives it; dQ and dK are
 * the gradients with respect to the unrotated Q and K: the kernels apply
 * the transposed rotation to dQ (in the dQ cast, or the fp32 dQ kernel's
 * store) and to dK (in the main kernel's store), with no extra pass.
 */
int nea_attn_bwd_rope(const void* Qr, const void* Kr, const void* V, const void* O,
                      const void* dO, const float* LSE, const float* cos_sin, void* dQ, void* dK,
                      void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                      int N, int d, float scale, int causal, int dtype, void* stream);

/*
 * Backward with options.  Arguments as nea_attn_bwd(), plus:
 *   rope_cos_sin  null, or the RoPE table Q and K were rotated with (then Q
 *                 and K are the rotated inputs and dQ, dK come back with
 *                 respect to the unrotated ones, as nea_attn_bwd_rope());
 *   flags         0, or NEA_BWD_DETERMINISTIC: bit-reproducible gradients.
 *                 bf16: the main kernel computes dK and dV only and a second
 *                 kernel computes dQ with one CTA per 128-row query tile,
 *                 walking the key tiles in a fixed order (S and dP are
 *                 recomputed there: two more GEMMs per tile pair, no dQ
 *                 accumulator traffic).  fp32 is deterministic either way.
 *                 Other bits: NEA_ERR_INVALID.
 * The workspace is the one nea_attn_bwd_workspace_bytes() sizes.
 */
#define NEA_BWD_DETERMINISTIC 1
int nea_attn_bwd_ex(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                    const float* LSE, const float* rope_cos_sin, int flags, void* dQ, void* dK,
                    void* dV, void* workspace, size_t workspace_bytes, int B, int H, int Hkv, int N,
                    int d, float scale, int causal, int dtype, void* stream);

/*
 * Decode attention: the nq newest tokens of each sequence against its
 * key/value cache (the inference use the pages mention: "NanoEuler:
 * Hand-writing GPT-2 in Pure C/CUDA", FAQ on production inference).
 * Reading taken: batch element b's cache holds lens[b] valid rows, the new
 * tokens' own keys and values included, so new token t sits at position
 * lens[b] - nq + t and sees cache rows 0 .. lens[b] - nq + t.
 *   Q, O    [B][H][nq][d] dtype       Kc, Vc  [B][Hkv][Lmax][d] dtype
 *   LSE     [B][H][nq] fp32, natural log of the scaled logits
 *   lens    [B] int32, DEVICE memory, nq <= lens[b] <= Lmax; a length out
 *           of that range is clamped into it and reported by
 *           nea_attn_check_status() as NEA_ERR_INVALID.
 * Supported: d in {64, 128}; bf16 or fp32; (H / Hkv) * nq <= 32.
 * The cache is read once per KV head, split over the cache length in
 * 128-row chunks (one CTA per chunk and KV head) and combined by a second
 * kernel through `workspace` (nea_attn_decode_workspace_bytes() bytes,
 * 256-byte aligned, caller-owned, contents on entry irrelevant).
 */
size_t nea_attn_decode_workspace_bytes(int B, int H, int Hkv, int nq, int Lmax, int d);
int nea_attn_decode(const void* Q, const void* Kc, const void* Vc, const int* lens, void* O,
                    float* LSE, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                    int nq, int Lmax, int d, float scale, int dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word.  Returns NEA_ERR_INVALID if a decode call met a cache length outside
 * [nq, Lmax], NEA_ERR_TIMEOUT if a kernel's bounded wait gave up since the
 * last check, NEA_ERR_CUDA if the stream reports an error, else NEA_OK.
 */
int nea_attn_check_status(void* stream);

/* Static, human-readable text for a status code. */
const char* nea_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int nea_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NEA_ATTN_H_ */
