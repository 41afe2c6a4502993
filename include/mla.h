/*
 * libmla: DeepSeek-V3.2-Exp sparse latent attention (MLA) prefill on one B300 (sm_103a).
 *
 * The path, as the model atlas pages define it (DeepSeek-V3.2-Exp inference/model.py excerpts):
 *   1. kv_norm: RMSNorm(512) of the key-value latent c_kv, fp32 mean of squares, eps 1e-6,
 *      learned gain ("Key-value RMSNorm" page, RMSNorm class, model.py 281-293; MLA __init__,
 *      model.py 523-539, on the "Key-value down-projection" page).
 *   2. wkv_b: ColumnParallelLinear(512, H * (128 + 128)), weight [out, in]; output viewed
 *      [B, T, H, 256] and split into k_nope (first 128) and v (last 128) ("Keys" and "Split value
 *      heads" pages, MHA prefill, model.py 574-589).
 *   3. k = cat(k_nope, k_pe expanded over heads) (192 features per head); scores = q . k scaled
 *      by softmax_scale = 192^-0.5 * m^2, m = 1 + 0.1 ln 40 ("Scale scores" page; MLA __init__).
 *   4. index mask: -inf except at the indexer's top-k positions, plus the causal mask; softmax
 *      over keys; x = scores . v (MHA prefill, model.py 574-589).
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous row-major, 16-byte
 *     aligned (q and out: 32-byte aligned; lse: 4-byte). bf16 tensors are passed as mla_bf16 (the
 *     raw 16-bit pattern).
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default stream). No call
 *     synchronizes the device unless its comment says so.
 *   - Argument and shape errors are returned synchronously and nothing is enqueued.
 *   - Errors found on the device (a barrier wait that ran out, an index outside [0, T) when
 *     MLA_FLAG_VALIDATE_INDICES is set, a value outside the range the kernels carry exactly, a
 *     failed bounds check of the checked build) are OR-ed into a per-device status word that
 *     mla_get_status() reads after the caller synchronizes.
 *   - Index convention: key j is used by query t iff j occurs in topk_idx[b, t, :] and 0 <= j <= t.
 *     Duplicates count once; order does not matter; j < 0 or j > t (including j >= T) is ignored.
 *   - A query whose selected set is empty gets out = 0 and lse = -inf.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef uint16_t mla_bf16; /* bfloat16 bit pattern */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* null pointer, misalignment, non-positive or overflowing size */
  MLA_ERR_UNSUPPORTED = 2, /* shape outside what the kernels support (see mla_dims); device: a
                            * kernel found its shared memory less aligned than its tiles need */
  MLA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
  MLA_ERR_INDEX = 4,       /* device: an index outside [0, T) under MLA_FLAG_VALIDATE_INDICES */
  MLA_ERR_TIMEOUT = 5,     /* device: a barrier wait ran past its limit; the kernel unwound */
  MLA_ERR_WORKSPACE = 6,   /* workspace pointer misaligned or smaller than required */
  MLA_ERR_RANGE = 7,       /* device: a value left the range the kernels carry exactly: |q[..., 0:128]|
                            * above 65504 (fp16), |k_nope| at or above 512 (its e4m3 residual would
                            * saturate) or |v| above 65504 (fp16), NaN included; results are unusable */
  MLA_ERR_BOUNDS = 8       /* device, checked build only (compiled with MLA_CHECKS): an index or TMA
                            * coordinate fell outside its tensor; the access was skipped */
} mla_status;

/* Problem sizes. The feature widths are fixed by the model: latent 512, 128 non-rotary + 64
 * rotary query/key features, 128 value features. Supported: B >= 1, 1 <= T <= 65536,
 * 1 <= H <= 128, K >= 1, and B*T*H*K below 2^40. */
typedef struct {
  int32_t B; /* batch */
  int32_t T; /* positions (queries = keys, prefill from position 0) */
  int32_t H; /* heads */
  int32_t K; /* top-k width of topk_idx */
} mla_dims;

#define MLA_FLAG_VALIDATE_INDICES 1u /* report indices outside [0, T) as MLA_ERR_INDEX */
#define MLA_FLAG_FP8_LATENT 2u       /* FP8 round trip of the normalised latent before wkv_b (see
                                      * mla_prefill_options) */
#define MLA_FLAG_ROPE 4u             /* q[..., 128:192] and k_pe are unrotated: apply YaRN RoPE */

/* Bytes of device workspace mla_sparse_prefill needs for `d` (0 if `d` is invalid): the
 * up-projected keys/values kv [B, H, T, 256] fp16, the key residuals klo [B, H, T, 128] (1 byte
 * each), the canonical selection bitsets [B, T, ceil(T/128)*4] uint32 (see mla_kvnorm_wkvb and
 * mla_canon_select for their contents) and 1024 bytes holding the attention stage's tile counter,
 * each 1024-byte aligned. Calls that run at the same time need workspaces of their own. */
MLA_API size_t mla_sparse_prefill_workspace_size(mla_dims d);

/* The whole prefill path: kv_norm -> wkv_b -> sparse causal attention (steps 1-4 above: "Key-value
 * RMSNorm", "Keys", "Split value heads" and "Scale scores" pages; MHA prefill, model.py 574-589).
 *   q         [B, T, H, 192] bf16: features 0..127 pair with k_nope, 128..191 (rotary, already
 *             applied) with k_pe. Features 0..127 are used in fp16 (exact for magnitudes in
 *             [2^-14, 65504]; smaller ones lose low bits, larger ones overflow).
 *   c_kv      [B, T, 512] bf16: the key-value latent before kv_norm.
 *   k_pe      [B, T, 64] bf16: the rotary key (already rotated), shared by all heads.
 *   gamma     [512] fp32: kv_norm weight.
 *   wkv_b     [H*256, 512] bf16, [out, in]: rows h*256 + [0,128) give k_nope of head h,
 *             h*256 + [128,256) its v.
 *   topk_idx  [B, T, K] int32.
 *   out       [B, T, H, 128] bf16 (written): softmax(scale * q.k masked) . v, rounded to nearest.
 *   lse       [B, T, H] fp32 (written): natural log of sum_j exp(scale * q.k_j) over selected j.
 *   workspace device memory of at least mla_sparse_prefill_workspace_size(d) bytes, 1024-byte
 *             aligned, or NULL: the call then takes it with cudaMallocAsync on `stream` and
 *             returns it with cudaFreeAsync on the same stream.
 * Returns MLA_OK once the work is enqueued. */
MLA_API mla_status mla_sparse_prefill(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe, const float* gamma,
                              const mla_bf16* wkv_b, const int32_t* topk_idx, mla_bf16* out, float* lse,
                              mla_dims d, void* workspace, size_t workspace_bytes, void* stream);

/* Range of the values the kernels carry exactly (see MLA_ERR_RANGE), checked on every call:
 *   q[..., 0:128] is used in fp16: |q| <= 65504 (bf16 values of magnitude below 2^-14 lose low
 *     bits, an absolute error below 2^-25 per feature);
 *   k_nope is kept as fp16 k_hi plus an e4m3 residual (k_nope - k_hi) * 2^11: |k_nope| < 512;
 *   v is kept in fp16: |v| <= 65504. */
#define MLA_MAX_ABS_Q_NOPE 65504.0f
#define MLA_MAX_ABS_K_NOPE 512.0f
#define MLA_MAX_ABS_V 65504.0f

/* As mla_sparse_prefill, plus:
 *   n_keys  [B, T] int32 (written unless NULL): size of each query's selected key set.
 *   flags   MLA_FLAG_VALIDATE_INDICES or 0. */
MLA_API mla_status mla_sparse_prefill_ex(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe, const float* gamma,
                                 const mla_bf16* wkv_b, const int32_t* topk_idx, mla_bf16* out, float* lse,
                                 mla_dims d, void* workspace, size_t workspace_bytes, void* stream,
                                 int32_t* n_keys, unsigned flags);

/* Options of mla_sparse_prefill_opt: the steps of the model's prefill around the MHA excerpt that
 * the plain entry points leave to the caller. Zero-initialise and set what is wanted.
 *   flags        MLA_FLAG_VALIDATE_INDICES, and:
 *     MLA_FLAG_FP8_LATENT  the KV cache's FP8 round trip of the normalised latent before wkv_b
 *                  ("Keys" page, KV-cache excerpt, model.py 541-573: act_quant(kv, 128), then
 *                  fp8 * scale cast back to bf16). Per block of 128 latent features: scale =
 *                  max|y| / 448 (1 for an all-zero block), e4m3 = nearest(y / scale) in fp32,
 *                  y' = bf16(e4m3 * scale) (act_quant's format and scale rule are not on the
 *                  pages; this is the plain reading).
 *     MLA_FLAG_ROPE        q[..., 128:192] and k_pe arrive unrotated; YaRN RoPE is applied at
 *                  positions 0..T-1 ("Key-value down-projection" page, model.py 565-568;
 *                  ModelArgs: rope_theta 10000, rope_factor 40, beta_fast 32, beta_slow 1,
 *                  original_seq_len 4096). Pairs (2i, 2i+1) rotate by t * f_i, f_i YaRN's
 *                  frequencies; the rotation is done in fp32 from the fp64 angle and rounded to
 *                  bf16.
 *   n_keys       [B, T] int32 written unless NULL (as mla_sparse_prefill_ex).
 *   wkv_b_scale  NULL: wkv_b is bf16 [H*256, 512]. Otherwise wkv_b holds FP8 e4m3 bytes
 *                [H*256, 512] and this is fp32 [2H, 4], one scale per 128 x 128 block
 *                ("Key-value down-projection" page, Linear excerpt, model.py 15 and 179-193); the
 *                weight used is bf16(e4m3 * scale), dequantised on the device.
 *   kv_cache     NULL, or [B, cache_len, 512] bf16, 32-byte aligned: positions 0..T-1 receive the
 *                latent wkv_b consumed (after the FP8 round trip when it is on).
 *   pe_cache     NULL, or [B, cache_len, 64] bf16, 4-byte aligned: positions 0..T-1 receive k_pe
 *                as the attention used it (rotated under MLA_FLAG_ROPE).
 *   cache_len    positions per sequence in the caches; at least T when a cache is given. */
typedef struct {
  unsigned flags;
  int32_t* n_keys;
  const float* wkv_b_scale;
  mla_bf16* kv_cache;
  mla_bf16* pe_cache;
  int32_t cache_len;
} mla_prefill_options;

/* Workspace bytes of mla_sparse_prefill_opt (0 if `d` or `opt` is invalid; opt may be NULL):
 * mla_sparse_prefill_workspace_size(d) plus, with FP8 weights, the dequantised wkv_b (H*256*512
 * bf16) and, under MLA_FLAG_ROPE, the (cos, sin) table [T, 32] fp32 pairs and the rotated k_pe
 * [B, T, 64] bf16, each 1024-byte aligned. */
MLA_API size_t mla_sparse_prefill_opt_workspace_size(mla_dims d, const mla_prefill_options* opt);

/* mla_sparse_prefill with the options above (opt may be NULL: then it is mla_sparse_prefill).
 * wkv_b points at bf16 or, when opt->wkv_b_scale is set, at e4m3 bytes. The workspace rules are
 * mla_sparse_prefill's, with mla_sparse_prefill_opt_workspace_size. */
MLA_API mla_status mla_sparse_prefill_opt(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe,
                                          const float* gamma, const void* wkv_b, const int32_t* topk_idx,
                                          mla_bf16* out, float* lse, mla_dims d, void* workspace,
                                          size_t workspace_bytes, void* stream, const mla_prefill_options* opt);

/* Stage 1 alone: the index mask of the MHA prefill excerpt ("Keys" page, model.py 574-589: -inf
 * scattered to 0 at the top-k indices, plus the causal mask), written as canonical selection
 * bitsets instead of a [B, T, T] mask. Bit (j % 32) of word sel_bits[(b*T + t)*W + j/32], W =
 * ceil(T/128)*4, is set iff key j is selected for query t (0 <= j <= t). Words of row t at or
 * beyond (t/128 + 1)*4 are not written. n_keys [B, T] int32 may be NULL. */
MLA_API mla_status mla_canon_select(const int32_t* topk_idx, mla_dims d, uint32_t* sel_bits, int32_t* n_keys,
                            unsigned flags, void* stream);

/* Stages 2-3 alone: kv_norm (RMSNorm class, model.py 281-293, "Key-value RMSNorm" page) fused into
 * the wkv_b GEMM (ColumnParallelLinear, MLA __init__ and MHA prefill on the "Keys" and "Split value
 * heads" pages). For head h at position t, with k_nope and v the up-projected features (fp32
 * accumulation of bf16 products):
 *   kv  [B, H, T, 256] fp16 (IEEE binary16 bit patterns): kv[.., 0:128] = k_hi = fp16(k_nope),
 *       kv[.., 128:256] = fp16(v);
 *   klo [B, H, T, 128] fp8 e4m3 bytes: (k_nope - k_hi) * 2^11, the part of k_nope fp16 drops.
 * k_hi + klo * 2^-11 carries k_nope to about 2^-14 relative. |k_nope| >= MLA_MAX_ABS_K_NOPE or
 * |v| > MLA_MAX_ABS_V records MLA_ERR_RANGE. */
MLA_API mla_status mla_kvnorm_wkvb(const mla_bf16* c_kv, const float* gamma, const mla_bf16* wkv_b, mla_dims d,
                           uint16_t* kv, uint8_t* klo, void* stream);

/* Stage 4 alone: sparse causal attention ("Keys" and "Scale scores" pages; MHA prefill, model.py
 * 574-589) from the outputs of the two stages above. Its tile counter is one library-owned word
 * per device, zeroed on `stream` before the launch: calls of this entry point that can overlap on
 * one device (other streams, other threads) race on it. */
MLA_API mla_status mla_sparse_attention(const mla_bf16* q, const mla_bf16* k_pe, const uint16_t* kv,
                                const uint8_t* klo, const uint32_t* sel_bits, mla_bf16* out, float* lse,
                                mla_dims d, void* stream);

/* FP8 block-scaled wkv_b -> its bf16 weight ("Key-value down-projection" page, Linear excerpt,
 * model.py 15 and 179-193): w[n, c] = bf16(e4m3(w8[n, c]) * scale[n / 128, c / 128]), the product
 * in fp32, rounded to nearest.
 *   w8     [rows, 512] e4m3 bytes, 16-byte aligned; rows a multiple of 128 (H*256 for wkv_b).
 *   scale  [rows / 128, 4] fp32.
 *   w      [rows, 512] bf16 (written), 32-byte aligned. */
MLA_API mla_status mla_dequant_wkvb_fp8(const uint8_t* w8, const float* scale, int32_t rows, mla_bf16* w,
                                        void* stream);

/* Stages 2-3 with the options of mla_prefill_options: as mla_kvnorm_wkvb, plus
 *   flags     0 or MLA_FLAG_FP8_LATENT (the FP8 round trip of the normalised latent);
 *   kv_cache  NULL or [B, cache_len, 512] bf16, 32-byte aligned: receives the latent the GEMM
 *             consumed (positions 0..T-1). */
MLA_API mla_status mla_kvnorm_wkvb_opt(const mla_bf16* c_kv, const float* gamma, const mla_bf16* wkv_b, mla_dims d,
                                       uint16_t* kv, uint8_t* klo, unsigned flags, mla_bf16* kv_cache,
                                       int32_t cache_len, void* stream);

/* YaRN RoPE of k_pe at positions 0..T-1 (see MLA_FLAG_ROPE) and the table the attention stage
 * rotates q with.
 *   k_pe      [B, T, 64] bf16, unrotated, 4-byte aligned.
 *   k_pe_rot  [B, T, 64] bf16 (written), 4-byte aligned.
 *   rope_cs   [T, 32] pairs of fp32 (cos, sin) of the angle t * f_i (written), 32-byte aligned.
 *   pe_cache  NULL or [B, cache_len, 64] bf16: receives k_pe_rot. */
MLA_API mla_status mla_rope_k_pe(const mla_bf16* k_pe, mla_dims d, mla_bf16* k_pe_rot, float* rope_cs,
                                 mla_bf16* pe_cache, int32_t cache_len, void* stream);

/* The YaRN frequencies f_i (radians per position) of the 32 rotary pairs. Host-only. */
MLA_API void mla_yarn_frequencies(double* f32_out);

/* Stage 4 with RoPE on q: as mla_sparse_attention, plus rope_cs (NULL, or the table mla_rope_k_pe
 * wrote): q[..., 128:192] is then unrotated and is rotated at position t inside the stage. k_pe
 * must be the rotated one. */
MLA_API mla_status mla_sparse_attention_opt(const mla_bf16* q, const mla_bf16* k_pe, const uint16_t* kv,
                                            const uint8_t* klo, const uint32_t* sel_bits, mla_bf16* out, float* lse,
                                            mla_dims d, const float* rope_cs, void* stream);

/* Allocation-free form of mla_sparse_prefill, for callers that cannot allocate device memory
 * when they run the prefill (code inside an allocator or memory-pool callback, engines that fix
 * their device footprint ahead of time, hosts that forbid cudaMalloc during a step). The pages
 * have no counterpart to this: it is a property of this library's interface only.
 *
 * Same arguments and results as mla_sparse_prefill, without the workspace: the scratch is a
 * library-owned device array of MLA_NOALLOC_SCRATCH_BYTES that every GPU loading libmla holds
 * until the process exits. The call allocates nothing (no cudaMalloc / cudaMallocAsync / cudaFree).
 *   - Problems whose mla_sparse_prefill_workspace_size(d) exceeds MLA_NOALLOC_SCRATCH_BYTES are
 *     rejected with MLA_ERR_WORKSPACE before anything is enqueued (at H = 128 that is about 800
 *     positions in all; the small shapes fit).
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress) and
 *     caches it; make that first call before any stream capture on that device.
 *   - Every call on a device shares the one array and it keeps the last call's contents (no call
 *     depends on them). Calls that can overlap on the GPU (other streams, other threads) race on
 *     it: serialize them. */
#define MLA_NOALLOC_SCRATCH_BYTES (64u << 20)
MLA_API mla_status mla_sparse_prefill_noalloc(const mla_bf16* q, const mla_bf16* c_kv, const mla_bf16* k_pe,
                                              const float* gamma, const mla_bf16* wkv_b, const int32_t* topk_idx,
                                              mla_bf16* out, float* lse, mla_dims d, void* stream);

/* Device status word of the current device: MLA_OK, or the lowest error code recorded since
 * the last mla_clear_status(). Synchronizes the current device first. */
MLA_API mla_status mla_get_status(void);

/* Reset the current device's status word to MLA_OK (synchronous). */
MLA_API mla_status mla_clear_status(void);

/* The softmax scale the kernels use: 192^-0.5 * (1 + 0.1 ln 40)^2. Host-only. */
MLA_API double mla_softmax_scale(void);

/* Diagnostic of the device-side failure path; no part of the prefill. Enqueues on `stream` one
 * thread that waits, through the same bounded wait every kernel uses, on a barrier nothing
 * arrives on. After the wait limit (about 2 s) the wait gives up, MLA_ERR_TIMEOUT is recorded in
 * the status word and the kernel returns; the context stays usable. Read the status with
 * mla_get_status() and reset it with mla_clear_status() before further work: while the timeout
 * is recorded, waits in later kernels give up early (they take it for another CTA's timeout).
 *   result  [2] int32 device memory, 4-byte aligned (written): [0] = 1 if the wait completed
 *           (it must not), [1] = milliseconds waited.
 * Returns MLA_OK once the kernel is enqueued, MLA_ERR_INVALID_ARG for a null or misaligned
 * `result`. */
MLA_API mla_status mla_selftest_wait_timeout(int32_t* result, void* stream);

/* A static, human-readable name for a status code. Host-only. */
MLA_API const char* mla_status_string(mla_status s);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
