/*
 * libindexer_bwd -- backward pass of the DeepSeek-sparse-attention lightning
 * indexer on one GB300 (sm_103a).
 *
 * The forward being differentiated scores each selected key s of query row t
 * as  I[t,s] = sum_h w[t,h] * relu(q[t,h,:] . k[s,:])  with one shared key
 * head (cudnn-frontend #730 "optimize SM100 gradient kernels", benchmark
 * harness fixture: q [B,S_q,H,D], k [B,S_k,D], w [B,S_q,H], top-k ids
 * [B,S_q,topk]; #549 "restore range_constexpr in 8 kernel_gemm epilogue
 * loops" names the two kernels kernel_score_grad and kernel_gemm).
 *
 * Conventions shared by every entry point
 *  - Tensors are caller-owned, contiguous, row-major DEVICE memory on the
 *    current CUDA device.  bf16 tensors are passed as uint16_t bit patterns.
 *    Every pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All work is queued asynchronously on it; nothing blocks except
 *    indexer_bwd_last_device_status.
 *  - Every argument check (null pointers, alignment, device-resident memory,
 *    shape limits, workspace size, an sm_103 device) happens before anything
 *    is launched.  A failed check returns a nonzero ibwd_status and leaves all
 *    memory untouched.  No exception or abort crosses this interface.
 *  - A top-k id outside [0, S_k) is padding at every stage (-1 or any
 *    positive out-of-range id); padding slots contribute nothing even when
 *    index_score, attn_score or dI hold NaN there.  Ids are local to their
 *    batch (id s of batch b addresses k[b, s]).
 *  - Shape limits: B >= 1, S_q >= 1, S_k >= 1, topk >= 1, 1 <= H <= 64,
 *    8 <= D <= 128 with D % 8 == 0, B*S_q*topk < 2^31; the deterministic
 *    dK mode also needs S_k <= 40960 (its key sort keeps per-key state in
 *    shared memory).
 *  - q and k entries must lie in fp16 range (|x| <= 65504): the gemm stage
 *    feeds fp16 tensor-core operands converted from bf16, exactly for
 *    2^-14 <= |x| <= 65504 and to fp16 subnormals (absolute error at most
 *    2^-25) below that.  A larger or non-finite entry is reported as
 *    IBWD_ERR_RANGE by indexer_bwd_last_device_status.
 *  - The library allocates no memory on the compute path: every scratch
 *    buffer is in the caller's workspace.  Per device, one 4-byte status
 *    word, one internal stream and two events (the gemm stage builds its q
 *    copies on that stream, forked from and joined back to the caller's
 *    stream within each call) are created on first use and kept until
 *    process exit.
 */
#ifndef INDEXER_BWD_H
#define INDEXER_BWD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define IBWD_API __attribute__((visibility("default")))
#else
#define IBWD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IBWD_OK = 0,
  IBWD_ERR_INVALID_ARG = 1, /* null/misaligned/host pointer, bad shape */
  IBWD_ERR_UNSUPPORTED = 2, /* not an sm_103 device, or a shape beyond the limits */
  IBWD_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  IBWD_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  IBWD_ERR_TIMEOUT = 5,     /* a kernel's bounded wait gave up (device status) */
  IBWD_ERR_RANGE = 6        /* a q or k entry outside the fp16 operand range (device status) */
} ibwd_status;

typedef enum {
  IBWD_DK_ATOMIC = 0,       /* dK += with fp32 red.global.add (run-to-run jitter ~1e-7) */
  IBWD_DK_DETERMINISTIC = 1 /* dK = fixed-order segment sums by key (bitwise reproducible) */
} ibwd_dk_mode;

/*
 * Kernel 1, score-grad (#730 walkthrough: kernel 1 writes the gradient signal
 * over attn_score and leaves index_score intact; the dK zeroing is fused into
 * the same launch).  For each row t over its valid slots j:
 *   p_j = softmax_j(index_score[t,:]),  ahat_j = attn_score[t,j] / sum_valid attn_score,
 *   dI[t,j] = grad_scale * (p_j - ahat_j) / S_q,   dI = 0 on padding slots
 * (the gradient of grad_scale * mean_t KL(ahat_t || p_t); ahat = 0 if the row's
 * target sums to 0; a row without valid slots is all zero).
 *   index_score  fp32 [B,S_q,topk], read only
 *   attn_score   fp32 [B,S_q,topk], read, then overwritten with dI
 *   topk_idx     int32 [B,S_q,topk]
 *   dk_to_zero   optional fp32 [B,S_k,D] set to 0 by the same launch (NULL: skipped)
 */
IBWD_API int indexer_bwd_score_grad(const float* index_score, float* attn_score, const int32_t* topk_idx,
                           int B, int S_q, int S_k, int topk, float grad_scale, float* dk_to_zero,
                           int D, void* stream);

/* Bytes of device workspace indexer_bwd_gemm needs (always > 0).  The gemm
 * stage takes the query rows in blocks of four (nb = B * ceil(S_q / 4)
 * blocks) against the union of their keys; the workspace holds, each part
 * rounded up to 256 bytes: a 256-byte block of counters; an fp16 copy of k,
 * 256 bytes per key row plus one zero row per batch; per block a 64 KB fp16
 * copy of its q rows laid out as the tensor-core operand and 16 bytes of
 * block data; for the sparse variant per block 4 bytes of ordering and
 * ceil(min(S_k, 4*topk) / 128) tile records of 2560 bytes.  The
 * deterministic mode adds 512 bytes per record, per (block, key) entry
 * -- nb * min(S_k, 4*topk) of them, or for the dense variant one per
 * (block, causal key) -- a scaled fp16 dK row (2*D bytes rounded up to a
 * multiple of 32, then 32 bytes holding its factor), its key sort (4*S_k
 * bytes per two blocks, sparse variant only) with 4 bytes per block, and
 * 4*(B*S_k + 1) bytes of key offsets.  The workspace is
 * rewritten by every call: calls that may overlap on the GPU need separate
 * workspaces.  0 for unsupported arguments. */
IBWD_API size_t indexer_bwd_gemm_workspace_size(int B, int S_q, int S_k, int H, int D, int topk,
                                       int dk_mode);

/*
 * Kernel 2, gemm stage (#730 harness, ref_grads: the fp64 definition of the
 * gemm_only semantics), for each valid slot (t, j), s = topk_idx[t,j]:
 *   z[h] = q[t,h,:] . k[s,:];   dW[t,h] = sum_j dI[t,j] relu(z[h]);
 *   dz[h] = dI[t,j] w[t,h] [z[h] > 0];   dQ[t,h,:] = sum_j dz[h] k[s,:];
 *   dK[s,:] += sum_h dz[h] q[t,h,:]
 *   q      bf16 [B,S_q,H,D];  k bf16 [B,S_k,D];  w fp32 [B,S_q,H]
 *   dI     fp32 [B,S_q,topk]  (the attn_score buffer after kernel 1)
 *   dq     fp32 [B,S_q,H,D], fully written;  dw fp32 [B,S_q,H], fully written
 *   dk     fp32 [B,S_k,D]: IBWD_DK_ATOMIC accumulates into it (zero it first,
 *          e.g. through indexer_bwd_score_grad's dk_to_zero);
 *          IBWD_DK_DETERMINISTIC overwrites it: each (block, key) row of
 *          contributions is stored at its place in key order and every
 *          key's rows are summed in a fixed order.
 *   workspace  device memory of at least indexer_bwd_gemm_workspace_size bytes
 * dq and dw are bitwise reproducible run to run in both modes.
 */
IBWD_API int indexer_bwd_gemm(const uint16_t* q, const uint16_t* k, const float* w, const float* dI,
                     const int32_t* topk_idx, float* dq, float* dw, float* dk, int B, int S_q,
                     int S_k, int H, int D, int topk, int dk_mode, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Dense variant (#549 tests: test_DSA_dense_indexer_backward; #730 touches
 * dense_indexer_backward_sm100.py): every causal key s <= t is selected,
 * S_q = S_k = S, and the scores are [B,S,S] (entry [t,s] for key s).  The
 * formulas are those above with the valid set {s <= t}; dI above the
 * diagonal is written as 0.
 */
IBWD_API int indexer_bwd_dense_score_grad(const float* index_score, float* attn_score, int B, int S,
                                 float grad_scale, float* dk_to_zero, int D, void* stream);
IBWD_API size_t indexer_bwd_dense_gemm_workspace_size(int B, int S, int H, int D, int dk_mode);
IBWD_API int indexer_bwd_dense_gemm(const uint16_t* q, const uint16_t* k, const float* w, const float* dI,
                           float* dq, float* dw, float* dk, int B, int S, int H, int D,
                           int dk_mode, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Gemm stage without any allocation (the pages have no counterpart: this is a
 * service of this library).  Same computation, arguments and outputs as
 * indexer_bwd_gemm in IBWD_DK_ATOMIC mode (dk accumulates; zero it first),
 * but it takes no workspace and calls no allocating routine.  It is meant
 * for callers that cannot allocate device memory where they run the
 * backward: code running inside a memory allocator or pool callback (an
 * allocation there would re-enter the allocator), runtimes that hand out all
 * device memory up front, and launch paths that must not synchronize the
 * device (cudaMalloc and cudaFree may).
 *  - It runs a per-row form of the gemm kernel whose only scratch (a row
 *    counter and the fp16 copy of k) is a fixed 8 MiB array inside the
 *    library, held by every GPU that loads it until the process exits; hence
 *    B * (S_k + 1) <= 32768.  Larger shapes return IBWD_ERR_UNSUPPORTED before
 *    anything is launched.
 *  - The first use on a device (this call, indexer_bwd_gemm_noalloc_setup or
 *    indexer_bwd_gemm_noalloc_status) looks up the array's device address,
 *    which may load the library's device module (allocating the array) and
 *    synchronize, and sets the kernel's shared-memory attribute.  Make that
 *    first use from a context where allocating and synchronizing are allowed,
 *    and before any stream capture: indexer_bwd_gemm_noalloc_setup does it
 *    eagerly for the current device.
 *  - Every call shares the one array: calls that overlap on the GPU (two
 *    streams, or two host threads) race and corrupt each other's results.
 *    Each call rewrites the array before reading it.
 *  - A kernel wait that times out sets a bit in this entry point's own status
 *    word (not the one indexer_bwd_last_device_status reports); the word
 *    keeps its bits across calls until indexer_bwd_gemm_noalloc_status reads
 *    and clears it.
 */
IBWD_API int indexer_bwd_gemm_noalloc(const uint16_t* q, const uint16_t* k, const float* w, const float* dI,
                             const int32_t* topk_idx, float* dq, float* dw, float* dk, int B, int S_q,
                             int S_k, int H, int D, int topk, void* stream);

/* The one-time set-up of indexer_bwd_gemm_noalloc for the current device
 * (see above); IBWD_OK, IBWD_ERR_UNSUPPORTED (not an sm_103 device) or
 * IBWD_ERR_CUDA. */
IBWD_API int indexer_bwd_gemm_noalloc_setup(void);

/* Synchronizes `stream`, then reads and clears the status word of
 * indexer_bwd_gemm_noalloc on the current device: IBWD_ERR_TIMEOUT if a
 * kernel's bounded wait expired since the last read, IBWD_ERR_CUDA if the
 * stream reports an error, IBWD_OK otherwise.  Allocates nothing. */
IBWD_API int indexer_bwd_gemm_noalloc_status(void* stream);

/*
 * The whole backward in one call: kernel 1 then kernel 2 above, queued on the
 * same stream (the #730 harness runs them as a pair; the arguments keep the
 * meanings given above).
 *   index_score  fp32 [B,S_q,topk], read only
 *   attn_score   fp32 [B,S_q,topk]: read, then overwritten by dI
 *   dq, dw       written;  dk  written in both modes (zeroed first in
 *                IBWD_DK_ATOMIC mode by kernel 1, as through dk_to_zero)
 *   workspace    at least indexer_bwd_gemm_workspace_size bytes (same shapes
 *                and dk_mode)
 * The fp16 copy of k and the gemm kernel are launched with programmatic
 * stream serialization behind the score-grad kernel (#730 commit list: the
 * score-grad and the GEMM overlap through programmatic dependent launch):
 * they may start while it runs, and each waits for the kernels before it
 * before reading what they wrote.  Work queued on the stream after this call
 * still starts only when the whole call has completed.
 * The results are bitwise those of the two calls.  Every check of both calls
 * happens before either kernel is launched.
 */
IBWD_API int indexer_bwd(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                         float* attn_score, const int32_t* topk_idx, float* dq, float* dw, float* dk, int B,
                         int S_q, int S_k, int H, int D, int topk, float grad_scale, int dk_mode,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Dense variant of indexer_bwd: every key s <= t, S_q = S_k = S, scores
 * [B,S,S]; workspace of indexer_bwd_dense_gemm_workspace_size bytes. */
IBWD_API int indexer_bwd_dense(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                               float* attn_score, float* dq, float* dw, float* dk, int B, int S, int H, int D,
                               float grad_scale, int dk_mode, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * Options of indexer_bwd_ex / indexer_bwd_dense_ex (the #730 benchmark
 * harness builds its kernels with topk_indices_global=True, takes bf16 dq and
 * dw outputs, and its full-pipeline time includes a bf16 cast of dK).  A
 * zero-initialised struct (or NULL) gives the behaviour of indexer_bwd.
 *   ids_global  0: ids are local to their batch (id s of a row of batch b
 *               addresses k[b,s]); 1: ids index the flattened [B*S_k] keys,
 *               and a row of batch b reads id - b*S_k, valid iff that lies
 *               in [0, S_k) -- an id of another batch is padding, never an
 *               alias (needs B*S_k < 2^31; ignored by the dense variant)
 *   dq_bf16     1: dq is bf16 [B,S_q,H,D] (round to nearest even of the fp32
 *               result) instead of fp32
 *   dw_bf16     1: dw is bf16 [B,S_q,H] likewise
 *   dk_bf16     optional device bf16 [B,S_k,D], 16-byte aligned: written with
 *               the final fp32 dk rounded to nearest even (dk itself is still
 *               produced in fp32)
 *   sm_scale    logit scale s of the forward the gradients belong to,
 *               I[t,j] = sum_h w[t,h] relu(s q[t,h,:] . k[s_j,:]) (#730
 *               benchmark harness: sm_scale, 1.0 there, folded into the
 *               kernels at run time).  0 means 1.  For s > 0,
 *               relu(s x) = s relu(x), so dq, dw and dk are s times the
 *               unscaled results for the same dI; the factor is folded into
 *               the outputs' power-of-two scale (one fp32 multiply each, no
 *               extra rounding when s = 1).  index_score must be the scaled
 *               forward's (the score-grad reads it as given).  Negative, NaN
 *               or infinite values are IBWD_ERR_INVALID_ARG.
 * Any other value of the int fields is IBWD_ERR_INVALID_ARG.
 */
typedef struct {
  int ids_global;
  int dq_bf16;
  int dw_bf16;
  uint16_t* dk_bf16;
  float sm_scale;
} ibwd_options;

/* indexer_bwd with options; dq and dw are float* or (bf16) uint16_t* as the
 * options say.  Same workspace as indexer_bwd. */
IBWD_API int indexer_bwd_ex(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                            float* attn_score, const int32_t* topk_idx, void* dq, void* dw, float* dk, int B,
                            int S_q, int S_k, int H, int D, int topk, float grad_scale, int dk_mode,
                            const ibwd_options* options, void* workspace, size_t workspace_bytes, void* stream);

/* indexer_bwd_dense with options (ids_global does not apply). */
IBWD_API int indexer_bwd_dense_ex(const uint16_t* q, const uint16_t* k, const float* w, const float* index_score,
                                  float* attn_score, void* dq, void* dw, float* dk, int B, int S, int H, int D,
                                  float grad_scale, int dk_mode, const ibwd_options* options, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Forward of the indexer: the logits the backward differentiates (#730
 * benchmark harness: one shared key head scored against every indexer head
 * of the query, weighted and summed),
 *   index_score[t,j] = sum_h w[t,h] relu(q[t,h,:] . k[s,:]),  s = topk_idx[t,j],
 * written as 0 on padding slots (any id outside [0, S_k)).  The same shapes,
 * layouts and limits as indexer_bwd_gemm:
 *   q bf16 [B,S_q,H,D];  k bf16 [B,S_k,D];  w fp32 [B,S_q,H];
 *   topk_idx int32 [B,S_q,topk];  index_score fp32 [B,S_q,topk], fully written.
 * Products of the bf16 inputs are exact and summed in fp32 (tensor cores).
 * No workspace.
 */
IBWD_API int indexer_fwd(const uint16_t* q, const uint16_t* k, const float* w, const int32_t* topk_idx,
                         float* index_score, int B, int S_q, int S_k, int H, int D, int topk, void* stream);

/* Dense variant of the forward: every key s <= t; index_score fp32 [B,S,S]
 * (entry [t,s]), 0 above the diagonal. */
IBWD_API int indexer_fwd_dense(const uint16_t* q, const uint16_t* k, const float* w, float* index_score, int B,
                               int S, int H, int D, void* stream);

/* Synchronizes `stream`, then reads and clears this device's status word:
 * IBWD_ERR_TIMEOUT if a kernel's bounded wait expired, IBWD_ERR_RANGE if a
 * q or k entry of a gemm-stage call lay outside the fp16 operand range, IBWD_ERR_CUDA if the stream reports an error,
 * IBWD_OK otherwise.  A gemm-stage call that
 * reports IBWD_ERR_TIMEOUT or IBWD_ERR_RANGE has left dq, dw and dk undefined. */
IBWD_API int indexer_bwd_last_device_status(void* stream);

/* Static English description of a status code. */
IBWD_API const char* indexer_bwd_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* INDEXER_BWD_H */
