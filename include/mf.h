/*
 * mf.h -- C ABI of the packed native-resolution 2D-RoPE varlen attention library
 * (libmf.so, sm_103a / B300).
 *
 * The operation is the joint self-attention of Mage-Flow's native-resolution
 * MMDiT ("Mage-Flow: An Efficient Native-Resolution Foundation Model for Image
 * Generation and Editing", arXiv 2607.19064):
 *   - many samples, each a variable-length text sequence followed by a flattened
 *     image-latent grid of any H x W, are packed into one token stream without
 *     padding or resolution buckets (rcap.io post, training-step listing
 *     "native-resolution packed step": pack(text_tokens + tokens, budget=50_000);
 *     paperlayer.ai summary section 3.2.1 "Model Architecture and Native Packing");
 *   - per-sample 2D rotary embeddings are applied to Q and K from each image
 *     token's native (row, col) latent position (rcap.io post, same listing:
 *     per_sample_2d_rope; ai.thesatyajit.com explainer, "A backbone that doesn't
 *     crop");
 *   - non-causal multi-head attention runs within each sample only, realised with
 *     variable-length attention kernels (rcap.io post; paperlayer.ai section 3.2.1:
 *     joint self-attention over the concatenated text and image tokens);
 *   - packed classifier-free guidance is the same call with the conditional and
 *     unconditional branches as two samples (paperlayer.ai section 3.2.1).
 * The pages print no formula for the rotation; this library fixes it (and the
 * oracle used to test it follows the same reading):
 *   image token k of an H x W grid is at (r, c) = (k div W, k mod W), text tokens at
 *   (0, 0); dims [0, d/2) rotate by r and [d/2, d) by c; within a half, the pair
 *   (2j, 2j+1), j < d/4, rotates by theta = p * 10000^(-2j/(d/2)):
 *   (x, y) -> (x cos theta - y sin theta, x sin theta + y cos theta).
 *   Softmax scale defaults to 1/sqrt(d).  LSE is the natural-log logsumexp of the
 *   scaled logits.
 *
 * Conventions for every call:
 *   - Layout "THD": packed tensors are [T][heads][head_dim] bf16, row-major,
 *     contiguous; LSE and the like are [heads][T] fp32.  cu_seqlens is int32[n+1]
 *     with cu_seqlens[0] = 0, non-decreasing, cu_seqlens[n] = T.  pos is int32[T][2]
 *     = (r, c).
 *   - Pointers prefixed d_ and all tensor pointers are DEVICE pointers on the
 *     current CUDA device; `specs` is a HOST pointer.  The caller owns every buffer;
 *     the library allocates no device memory (workspaces are sized by
 *     mf_attn_workspace_bytes and passed in).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Argument errors are detected on the host before any launch and
 *     returned synchronously; launch failures return MF_ERR_CUDA.  Errors found on
 *     the device (malformed cu_seqlens, a wait that ran out) are recorded in the
 *     workspace and reported by mf_get_status.
 *   - Tensor pointers must be 16-byte aligned; head_dim must be 64 or 128; T and
 *     every index fit in int32 (T * heads * head_dim < 2^31 is not required, but
 *     T < 2^31 is).  Anything else: MF_ERR_UNSUPPORTED / MF_ERR_OVERFLOW.
 */
#ifndef MF_H_
#define MF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MF_OK = 0,
  MF_ERR_INVALID_ARG = 1,  /* bad argument (negative size, NULL pointer, ...) */
  MF_ERR_UNSUPPORTED = 2,  /* valid but not supported (head_dim, alignment, ...) */
  MF_ERR_OVERFLOW = 3,     /* a size does not fit in int32 */
  MF_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  MF_ERR_TIMEOUT = 5,      /* a device-side wait ran out (kernel gave up cleanly) */
  MF_ERR_BAD_SEQLENS = 6   /* device-side check: cu_seqlens malformed or a sample > max_len */
} mf_status;

typedef uint16_t mf_bf16; /* bfloat16 storage */
typedef void* mf_stream;  /* cudaStream_t */

/* Human-readable name of a status code (static string). */
const char* mf_status_string(mf_status s);

/* Library version, e.g. 10000 for 1.0.0. */
int32_t mf_version(void);

/*
 * Packing sizes (host only, no device work).
 * specs: HOST int32[n][3] = {text_len, H_lat, W_lat} per sample, in pack order.
 * Outputs: *total = T = sum_i (text_len_i + H_i * W_i); *max_len = max_i L_i
 * (0 when n = 0).  Either output pointer may be NULL.
 * Errors: MF_ERR_INVALID_ARG for n < 0, a NULL specs with n > 0, or a negative
 * entry; MF_ERR_OVERFLOW when T or an H*W product exceeds INT32_MAX.
 * Defined by: rcap.io post, training-step listing (pack(...)); paperlayer.ai 3.2.1.
 */
mf_status mf_pack_size(const int32_t* specs, int32_t n, int32_t* total, int32_t* max_len);

/*
 * Build the packed-stream tables on the device.
 * specs: HOST int32[n][3] as above (read before the call returns).
 * d_cu_seqlens: DEVICE int32[n+1] out: cu[0] = 0, cu[i+1] = cu[i] + L_i.
 * d_pos: DEVICE int32[T][2] out: token cu[i] + k is text at (0,0) for k < text_len_i,
 *   else image token m = k - text_len_i at (m div W_i, m mod W_i).  May be NULL.
 * Zero-length samples are allowed.  Same errors as mf_pack_size, plus
 * MF_ERR_INVALID_ARG for a NULL d_cu_seqlens and MF_ERR_UNSUPPORTED for a
 * misaligned d_pos (needs 8-byte alignment).
 * Defined by: rcap.io post, training-step listing; paperlayer.ai 3.2.1 (packing
 * under a token budget, native latent grid kept, no padding).
 */
mf_status mf_pack(const int32_t* specs, int32_t n, int32_t* d_cu_seqlens, int32_t* d_pos,
                  mf_stream stream);

/*
 * Standalone per-sample 2D RoPE on Q and K.
 * q, k: DEVICE bf16 [T][heads][head_dim] in; q_out, k_out: DEVICE bf16 out, same
 * layout (q_out == q and/or k_out == k is allowed: in place).  d_pos: DEVICE
 * int32[T][2].  Computes q_out = R(theta(pos)) q, k_out = R(theta(pos)) k with the
 * rotation defined at the top of this file, in fp32 with a correctly rounded
 * (nearest-even) bf16 result.  q (with q_out) or k (with k_out) may be NULL to
 * rotate only the other one.
 * Errors: MF_ERR_INVALID_ARG (T < 0, heads < 1, NULL d_pos with T > 0);
 * MF_ERR_UNSUPPORTED (head_dim not 64/128, misaligned pointer).
 * Defined by: rcap.io post (per_sample_2d_rope, native positions); explainer
 * "A backbone that doesn't crop".
 */
mf_status mf_rope2d_qk(const mf_bf16* q, const mf_bf16* k, mf_bf16* q_out, mf_bf16* k_out,
                       const int32_t* d_pos, int32_t T, int32_t heads, int32_t head_dim,
                       mf_stream stream);

/*
 * Workspace bytes needed by mf_varlen_attn_fwd (bwd = 0) or mf_varlen_attn_bwd
 * (bwd = 1) for these sizes.  The workspace is a DEVICE buffer of at least that
 * many bytes, 256-byte aligned, owned by the caller, not shared by concurrent
 * calls; its contents need no initialisation.  Returns 0 on invalid sizes.
 */
size_t mf_attn_workspace_bytes(int32_t T, int32_t n, int32_t heads, int32_t head_dim, int32_t bwd);

/*
 * Workspace bytes for the backward calls that selects their stored-dS form: the
 * dK / dV kernel also writes each (sample, head)'s scaled fp16 dS^T (its keys and
 * queries padded to multiples of 128) into the workspace, and dQ = scale R(-theta)
 * dS K' is then one streaming GEMM over it instead of a kernel that recomputes S
 * and dP.  Faster, at the cost of memory: 256 heads (ceil(T / 128) + n) max_len'
 * bytes (max_len' = max_len rounded up to 128) on top of
 * mf_attn_workspace_bytes(..., 1) (11.4 GB in all for 48k tokens, 24 heads,
 * max_len 4,291).  Any of the backward calls given a workspace of at least this
 * size, for the same T, n, heads and max_len, uses that form; its results equal
 * the other form's (the same fp16 dS values summed in the same order).  Returns 0
 * on invalid sizes.
 * No counterpart on the pages: a memory-for-time form of the backward.
 */
size_t mf_attn_workspace_bytes_ds(int32_t T, int32_t n, int32_t heads, int32_t head_dim,
                                  int32_t max_len);

/*
 * Varlen attention forward with per-sample 2D RoPE.
 * q, k, v: DEVICE bf16 [T][heads][head_dim], un-rotated.
 * d_cu_seqlens: DEVICE int32[n+1]; d_pos: DEVICE int32[T][2], or NULL for no
 * rotation.  max_len: an upper bound on every L_i (checked on the device).
 * softmax_scale <= 0 selects 1/sqrt(head_dim).
 * o: DEVICE bf16 [T][heads][head_dim] out.  lse: DEVICE fp32 [heads][T] out
 * (natural-log logsumexp of the scaled logits of each query row).
 * ws / ws_bytes: workspace from mf_attn_workspace_bytes(T, n, heads, head_dim, 0).
 * For each sample i and head a, and each query row j of sample i:
 *   O_j = sum_k softmax_k(scale * <q'_j, k'_k>) v_k over the keys of sample i only,
 * q' = R(theta) q, k' = R(theta) k.  Rows of zero-length samples do not exist; every
 * output row belongs to exactly one sample and is written exactly once.
 * Defined by: paperlayer.ai 3.2.1 (joint self-attention within the packed
 * sequence), rcap.io post (varlen attention, per-sample 2D RoPE).
 */
mf_status mf_varlen_attn_fwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                             const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t n,
                             int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                             float softmax_scale, mf_bf16* o, float* lse, void* ws,
                             size_t ws_bytes, mf_stream stream);

/*
 * The same forward with the 2D RoPE applied on the tile load (no rotation
 * pre-pass): the attention kernel's TMA warp stages the caller's bf16 Q, K and V
 * tiles in shared memory, two further warps rotate the Q and K tiles there (and
 * convert V to the kernel's fp16 operand type) in place, and the tensor core reads
 * the result.  The angles come from a small (cos, sin) table of v * omega_P for
 * v in [0, min(max_len, T)), built by one launch per call from the same
 * evaluation the pre-pass uses, so O and LSE are bit-identical to
 * mf_varlen_attn_fwd's for the same inputs.  Arguments, shapes, workspace
 * (mf_attn_workspace_bytes(..., 0)) and errors as mf_varlen_attn_fwd, plus: a
 * position outside [0, min(max_len, T)) is an error recorded in the workspace
 * (mf_get_status: MF_ERR_INVALID_ARG; such a coordinate is read as 0).  Positions
 * from mf_pack always lie in that range (r < H and c < W, each at most L_i).
 * It leaves no rotated operands in the workspace: a training step's backward
 * after it is mf_varlen_attn_bwd, not mf_varlen_attn_bwd_after_fwd.
 * Defined by: paperlayer.ai 3.3 "Training Infrastructure" (rotary embeddings
 * inside the fused Transformer chain) and 3.2.1 (the attention); rcap.io post
 * (per_sample_2d_rope applied within the packed step).
 */
mf_status mf_varlen_attn_fwd_fused_rope(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                        const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                        int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                        int32_t head_dim, float softmax_scale, mf_bf16* o,
                                        float* lse, void* ws, size_t ws_bytes, mf_stream stream);

/*
 * Varlen attention backward (gradients with respect to the UN-rotated q and k,
 * i.e. the rotation's transpose R(-theta) is folded in).
 * q, k, v, o, d_o: DEVICE bf16 [T][heads][head_dim]; lse: DEVICE fp32 [heads][T]
 * from the forward.  Other arguments as in the forward.
 * dq, dk, dv: DEVICE bf16 [T][heads][head_dim] out.
 * ws / ws_bytes: workspace from mf_attn_workspace_bytes(T, n, heads, head_dim, 1)
 * (holds the rotated Q/K and D = rowsum(dO * O)); a workspace of at least
 * mf_attn_workspace_bytes_ds(T, n, heads, head_dim, max_len) selects the faster
 * stored-dS form of the computation (same results).
 * Per sample and head: P = exp(S - LSE), dV = P^T dO, dP = dO V^T,
 * dS = P * (dP - D), dQ = R(-theta) scale dS K', dK = R(-theta) scale dS^T Q'.
 * Defined by: the training step of the rcap.io listing (loss.backward through the
 * attention); gradients are those of the forward above.
 */
mf_status mf_varlen_attn_bwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                             const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                             const int32_t* d_cu_seqlens, const int32_t* d_pos, int32_t n,
                             int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                             float softmax_scale, mf_bf16* dq, mf_bf16* dk, mf_bf16* dv,
                             void* ws, size_t ws_bytes, mf_stream stream);

/*
 * The backward of a training step whose forward ran on the SAME workspace.
 * mf_varlen_attn_fwd / _fwd_3d leave the rotated fp16 operands Q' = R q and
 * K' = R k in the workspace at the offsets the backward reads them from, so this
 * call skips the backward's own rotation pre-pass (one read of q and k and one
 * write of Q', K').  Arguments as mf_varlen_attn_bwd, plus pos_axes (2 for d_pos
 * [T][2], 3 for editing packs' [T][3]).  Preconditions, which the call cannot
 * check: ws (sized by mf_attn_workspace_bytes(..., bwd = 1), which also fits the
 * forward) was last used by the forward of these q, k, d_pos, n, T, heads and
 * head_dim on the same stream, and neither q nor k changed since.  The fp16 range
 * check of Q' and K' is then the forward's: read it with mf_get_status after the
 * forward.  Results equal mf_varlen_attn_bwd's.  No counterpart on the pages: a workspace-sharing form of the backward.
 */
mf_status mf_varlen_attn_bwd_after_fwd(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                       const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                       const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                       int32_t pos_axes, int32_t n, int32_t T, int32_t max_len,
                                       int32_t heads, int32_t head_dim, float softmax_scale,
                                       mf_bf16* dq, mf_bf16* dk, mf_bf16* dv, void* ws,
                                       size_t ws_bytes, mf_stream stream);

/*
 * Frame-aware 3D positions for editing packs.  The pages say that editing
 * extends the 2D rotary embedding with a frame dimension that tells source and
 * target visual tokens apart (hyper.ai summary "Method"; paperlayer.ai summary
 * 3.2.1), and that editing concatenates the text conditioning with the source
 * latents and the noisy target latents (paperlayer.ai summary 3.2.2).  They give
 * no layout or frequencies; this library's reading:
 *   - sample i is [text; source grid Hs x Ws; target grid Ht x Wt];
 *   - positions are (f, r, c): text (0, 0, 0), source token m at
 *     (0, m div Ws, m mod Ws), target token m at (1, m div Wt, m mod Wt);
 *   - head_dim splits into contiguous frame, row and column slices of d/4, 3d/8 and
 *     3d/8 dims (16, 24, 24 rotary pairs at d = 128); within a slice of width w the
 *     pair (2j, 2j+1) of the slice rotates by p * 10000^(-2j / w), p the token's
 *     coordinate on that axis, with the sign of the 2D rotation.
 * specs: HOST int32 [n][5] = {text_len, Hs, Ws, Ht, Wt}.
 */
mf_status mf_pack3d_size(const int32_t* specs, int32_t n, int32_t* total, int32_t* max_len);
/* d_cu_seqlens: DEVICE int32 [n+1]; d_pos3: DEVICE int32 [T][3] (may be NULL), 4-byte
 * aligned.  Errors as mf_pack. */
mf_status mf_pack3d(const int32_t* specs, int32_t n, int32_t* d_cu_seqlens, int32_t* d_pos3,
                    mf_stream stream);
/* Standalone 3D rotation of q and k (as mf_rope2d_qk, with d_pos3 [T][3]). */
mf_status mf_rope3d_qk(const mf_bf16* q, const mf_bf16* k, mf_bf16* q_out, mf_bf16* k_out,
                       const int32_t* d_pos3, int32_t T, int32_t heads, int32_t head_dim,
                       mf_stream stream);
/* The attention forward and backward of an editing pack: exactly mf_varlen_attn_fwd
 * and mf_varlen_attn_bwd with q' = R3 q, k' = R3 k (d_pos3 [T][3], not NULL) and the
 * gradients taken back through R3's transpose.  Same workspaces, shapes and errors. */
mf_status mf_varlen_attn_fwd_3d(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                const int32_t* d_cu_seqlens, const int32_t* d_pos3, int32_t n,
                                int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                                float softmax_scale, mf_bf16* o, float* lse, void* ws,
                                size_t ws_bytes, mf_stream stream);
mf_status mf_varlen_attn_bwd_3d(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                const int32_t* d_cu_seqlens, const int32_t* d_pos3, int32_t n,
                                int32_t T, int32_t max_len, int32_t heads, int32_t head_dim,
                                float softmax_scale, mf_bf16* dq, mf_bf16* dk, mf_bf16* dv,
                                void* ws, size_t ws_bytes, mf_stream stream);

/*
 * The 8-bit (E4M3) variant of the attention forward.  The pages give no
 * low-precision recipe; this is an engineering variant of mf_varlen_attn_fwd (same
 * operation, same arguments) that runs both GEMMs on 8-bit operands at twice the
 * tensor-core rate of 16-bit ones.  Its steps, each value rounded to the nearest
 * E4M3 value (OCP 8-bit floating point: 4 exponent bits with bias 7, 3 mantissa
 * bits, largest finite 448; ties to even, saturating):
 *   - every block below is divided by its scale s: the smallest power of two with
 *     (the block's largest magnitude A) / s <= 448, so the division is exact;
 *   - Q' = R q, one block per (token, head) row;
 *   - K' = R k, one block per head, with A the largest pair norm |(k_2P, k_2P+1)|
 *     of the un-rotated k over the head's tokens: the pair norm bounds every
 *     rotated component at any position;
 *   - V, one block per head;
 *   - S = Q'K'^T in fp32 from the E4M3 codes, then, per query row and tile of
 *     128 keys from the sample's first key, base-2 logits
 *     x = log2(e) * scale * sq * sk * S.  The running maximum m is set by the
 *     first tile and raised only when a tile's maximum exceeds it by more than 8
 *     (then l and the accumulator are rescaled), as in the 16-bit forward;
 *   - P = 2^(x - m) <= 256 rounded to E4M3 before it weights V; l sums the
 *     unrounded P;
 *   - O = sv * (sum_k P~_k V~_k) / l in bf16, LSE = ln 2 * (m + log2 l).
 * Accuracy: expect O errors of a few per cent of |O| against the exact attention
 * (3 mantissa bits on both operands and probabilities); LSE within the largest
 * logit change that the operand rounding permits.
 * d_pos: NULL (no rotation), [T][2] (pos_axes = 2) or [T][3] (pos_axes = 3, the
 * frame-aware 3D rotation).  Workspace: mf_attn_workspace_bytes(T, n, heads,
 * head_dim, 0), the forward's.  head_dim must be 128 (64 returns
 * MF_ERR_UNSUPPORTED before any launch); pos_axes other than 2 or 3 with a
 * non-NULL d_pos returns MF_ERR_INVALID_ARG.  Other arguments and errors as
 * mf_varlen_attn_fwd.
 */
mf_status mf_varlen_attn_fwd_fp8(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                 const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                 int32_t pos_axes, int32_t n, int32_t T, int32_t max_len,
                                 int32_t heads, int32_t head_dim, float softmax_scale, mf_bf16* o,
                                 float* lse, void* ws, size_t ws_bytes, mf_stream stream);

/*
 * The operands of the 8-bit forward on their own (its first two passes), for
 * callers that keep E4M3 copies: q8, k8, v8 DEVICE E4M3 [T][heads][128] bytes;
 * qscale DEVICE fp32 [T][heads], the Q row scales (powers of two; 0 for an
 * all-zero row); kv_max2 DEVICE fp32 [2][heads]: the squared largest pair norm of
 * k and the squared largest |v| of each head (the K and V scales are the powers of
 * two that mf_varlen_attn_fwd_fp8 describes, for A = sqrt(kv_max2)).
 * The call zeroes kv_max2 itself.  q, k, v, q8, k8, v8 16-byte aligned, qscale,
 * kv_max2 and d_pos 4-byte aligned.  head_dim must be 128 (else
 * MF_ERR_UNSUPPORTED); d_pos as in mf_varlen_attn_fwd_fp8.
 */
mf_status mf_quant_e4m3(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                        const int32_t* d_pos, int32_t pos_axes, int32_t T, int32_t heads,
                        int32_t head_dim, uint8_t* q8, uint8_t* k8, uint8_t* v8, float* qscale,
                        float* kv_max2, mf_stream stream);

/*
 * Varlen attention forward that allocates nothing and takes no workspace.
 * (The pages have no counterpart to this call: it is for callers of this library.)
 * Some callers cannot allocate device memory: a plugin inside a framework that
 * owns the device allocator and hands it only inputs and outputs, or a
 * latency-critical loop where cudaMalloc / cudaFree, which can synchronise the
 * device, are not allowed.  This entry point computes exactly what
 * mf_varlen_attn_fwd computes, with the same arguments minus ws / ws_bytes; its
 * scratch is one fixed device array inside the library, MF_NOALLOC_SCRATCH_BYTES
 * bytes, which every GPU that loads the library holds until the process exits.
 *  - Limits: n <= MF_NOALLOC_MAX_SAMPLES and T * heads * head_dim <=
 *    MF_NOALLOC_MAX_ELEMS; larger problems return MF_ERR_UNSUPPORTED before any
 *    launch (use mf_varlen_attn_fwd with a caller workspace for them).
 *  - The first call on each device looks up the array's device address once
 *    (cudaGetSymbolAddress, with that device current); make that first call before
 *    any stream capture.  Later calls only reuse the cached address.  The cache is
 *    keyed on the unique id of the current context, so after cudaDeviceReset (which
 *    loads the library's module again in a new context) the next call looks the
 *    address up afresh; make that call, too, before any stream capture.
 *  - Every call shares the one array, which keeps the previous call's contents;
 *    the forward rewrites everything it reads from it (status word, work list,
 *    fp16 operand copies), so no clearing is needed between calls.  Calls that
 *    overlap on the GPU (concurrent streams, other threads) race on the array:
 *    serialise them.
 *  - Device-side errors (a malformed cu_seqlens, a wait that ran out, a value
 *    outside the fp16 range of the internal operands) are recorded in the array's
 *    status word, as mf_varlen_attn_fwd records them in its workspace; read them
 *    with mf_noalloc_get_status.
 * No device memory is allocated by this call or by the library on its behalf.
 */
#define MF_NOALLOC_MAX_ELEMS 4194304LL   /* T * heads * head_dim */
#define MF_NOALLOC_MAX_SAMPLES 4096
#define MF_NOALLOC_SCRATCH_BYTES 25199616ULL
mf_status mf_varlen_attn_fwd_noalloc(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                     const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                     int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                     int32_t head_dim, float softmax_scale, mf_bf16* o,
                                     float* lse, mf_stream stream);

/*
 * Synchronise `stream` and report the device-side status that the last
 * mf_varlen_attn_fwd_noalloc call on the current device recorded in the
 * library's scratch array: MF_ERR_BAD_SEQLENS, MF_ERR_TIMEOUT, MF_ERR_OVERFLOW
 * (a value left the fp16 range of the internal operands), MF_ERR_CUDA if the
 * stream itself failed; MF_OK otherwise.  Allocates nothing.  Like the forward it
 * reports on, it shares the one array: a call that overlaps another no-alloc
 * forward on the GPU reads a status word that that call is rewriting.
 */
mf_status mf_noalloc_get_status(mf_stream stream);

/*
 * Packed classifier-free guidance followed by one rectified-flow Euler step.
 * The conditional and unconditional branches of each image are two samples of
 * one packed forward pass (paperlayer.ai summary 3.2.1 "Model Architecture and
 * Native Packing"; hyper.ai summary "Experiment": the denoising trajectory is
 * unchanged).  The pages give the flow-matching objective (hyper.ai "Method":
 * z_t = (1 - t) z + t eps, the network regresses z - eps), so a step from t to
 * t - dt is z <- z + dt v; they print no guidance formula, and the standard
 * v = v_u + g (v_c - v_u) is used.
 * v: DEVICE bf16 [T][C], the model's packed output for 2 * pairs samples laid out
 *    as mf_pack lays out `specs` (T = the pack's total).
 * specs: HOST int32 [2 * pairs][3] = {text_len, H, W}: pair p is samples 2p (cond)
 *    and 2p + 1 (uncond), which must have the same H and W.
 * z: DEVICE fp32 [N][C], N = sum_p H_p * W_p: each pair's image latent rows in pair
 *    order, updated in place: z[row] += dt * (v_u[row] + g (v_c[row] - v_u[row]))
 *    with v_c / v_u the pair's image-token rows of v (after each sample's text).
 * Arithmetic in fp32.  C must be a positive multiple of 8 and v, z 16-byte
 * aligned (else MF_ERR_UNSUPPORTED); negative entries, a pair whose grids differ
 * or a NULL pointer with work to do: MF_ERR_INVALID_ARG; totals beyond int32:
 * MF_ERR_OVERFLOW.
 */
mf_status mf_cfg_euler_step(const mf_bf16* v, const int32_t* specs, int32_t pairs, int32_t C,
                            float guidance, float dt, float* z, mf_stream stream);

/*
 * Adaptive LayerNorm modulation of a packed batch (the input side of the fused
 * Transformer chain of paperlayer.ai summary 3.3 "Training Infrastructure":
 * adaptive normalization, rotary embeddings and gated residual updates).  The
 * pages print no formula; the DiT-style block is used: for every token t of
 * sample s (by d_cu_seqlens),
 *   y_t = (x_t - mean_t) / sqrt(var_t + eps) * (1 + scale_s) + shift_s,
 * mean and biased variance over the Dm features, no affine parameters.
 * x, y: DEVICE bf16 [T][Dm] (y == x allowed); shift, scale: DEVICE bf16 [n][Dm];
 * d_cu_seqlens: DEVICE int32 [n+1] as for the attention.  fp32 arithmetic.
 * Dm must be a multiple of 8 and pointers 16-byte aligned (else
 * MF_ERR_UNSUPPORTED); n = 0 with T > 0, eps < 0 or NULL pointers:
 * MF_ERR_INVALID_ARG.  A malformed cu_seqlens gives wrong rows, never an
 * out-of-range access (every row maps to a sample index in [0, n)).
 */
mf_status mf_adaln_modulate(const mf_bf16* x, const int32_t* d_cu_seqlens, int32_t n, int32_t T,
                            int32_t Dm, const mf_bf16* shift, const mf_bf16* scale, float eps,
                            mf_bf16* y, mf_stream stream);

/*
 * Gated residual update of a packed batch (output side of the same fused chain):
 * out_t = x_t + gate_s * h_t for every token t of sample s.  x, h, out: DEVICE bf16
 * [T][Dm] (out may alias x or h); gate: DEVICE bf16 [n][Dm].  fp32 arithmetic.
 * Same shape rules and errors as mf_adaln_modulate.
 */
mf_status mf_gated_residual(const mf_bf16* x, const mf_bf16* h, const int32_t* d_cu_seqlens,
                            int32_t n, int32_t T, int32_t Dm, const mf_bf16* gate, mf_bf16* out,
                            mf_stream stream);

/*
 * Synchronise `stream` and report device-side errors recorded in `ws` by the last
 * mf_varlen_attn_* call that used it: MF_ERR_BAD_SEQLENS, MF_ERR_TIMEOUT, or
 * MF_ERR_CUDA if the stream itself failed; MF_OK otherwise.
 */
mf_status mf_get_status(void* ws, mf_stream stream);

/*
 * Test hook for failure detection (no counterpart on the pages; not for
 * production use).  Exactly mf_varlen_attn_fwd, except that in every CTA of the
 * attention kernel the thread that issues the tensor-core work first waits on a
 * barrier that nothing ever arrives on, for at most stall_us microseconds
 * (1 .. 1,000,000; else MF_ERR_INVALID_ARG).  That wait runs out, and the kernel
 * takes its time-out path: the CTA records MF_ERR_TIMEOUT in the workspace, lets
 * its copies in flight land, frees its tensor memory and exits, so the context
 * stays usable.  mf_get_status(ws) then returns MF_ERR_TIMEOUT; O and LSE are not
 * written.  A later call on the same or another workspace runs normally.
 */
mf_status mf_test_varlen_attn_fwd_stalled(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                          const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                          int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                          int32_t head_dim, float softmax_scale, mf_bf16* o,
                                          float* lse, void* ws, size_t ws_bytes,
                                          int32_t stall_us, mf_stream stream);
/* The same hook in the backward's attention kernel: exactly mf_varlen_attn_bwd,
 * except that its MMA-issuing thread first waits, at most stall_us microseconds,
 * on a barrier that nothing arrives on.  mf_get_status(ws) then returns
 * MF_ERR_TIMEOUT; dQ, dK and dV are not written.  A later call runs normally. */
mf_status mf_test_varlen_attn_bwd_stalled(const mf_bf16* q, const mf_bf16* k, const mf_bf16* v,
                                          const mf_bf16* o, const float* lse, const mf_bf16* d_o,
                                          const int32_t* d_cu_seqlens, const int32_t* d_pos,
                                          int32_t n, int32_t T, int32_t max_len, int32_t heads,
                                          int32_t head_dim, float softmax_scale, mf_bf16* dq,
                                          mf_bf16* dk, mf_bf16* dv, void* ws, size_t ws_bytes,
                                          int32_t stall_us, mf_stream stream);

/*
 * Optional per-kernel timing (instrumentation; no counterpart on the pages).
 * When enabled, every kernel launch made by the calls above is bracketed by two
 * CUDA events recorded on the call's stream (a few microseconds of host work per
 * launch; nothing changes on the device path).  mf_timing_read synchronises on
 * the recorded events and returns, for kernel `id`, the summed device time in
 * milliseconds and the number of launches since the last reset.  Ids:
 *   MF_K_PACK 0, MF_K_ROPE 1, MF_K_SCHEDULE 2, MF_K_ATTN_FWD 3, MF_K_BWD_PRE 4,
 *   MF_K_ATTN_BWD 5 (dK, dV), MF_K_ATTN_BWD_Q 6 (dQ), MF_K_CFG_EULER 7, MF_K_ADALN 8,
 *   MF_K_GATED_RESIDUAL 9, MF_K_F8_AMAX 10, MF_K_F8_QUANT 11, MF_K_ATTN_FWD_F8 12,
 *   MF_K_ROPE_TABLE 13, MF_K_ATTN_FWD_ROT 14 (the rotate-on-load forward's table and
 *   attention kernels), MF_K_ATTN_BWD_DQ 15 (dQ from the stored dS).
 * Process-wide state guarded by a mutex; not for use under stream capture.
 */
enum { MF_K_PACK = 0, MF_K_ROPE, MF_K_SCHEDULE, MF_K_ATTN_FWD, MF_K_BWD_PRE, MF_K_ATTN_BWD,
       MF_K_ATTN_BWD_Q, MF_K_CFG_EULER, MF_K_ADALN, MF_K_GATED_RESIDUAL, MF_K_F8_AMAX,
       MF_K_F8_QUANT, MF_K_ATTN_FWD_F8, MF_K_ROPE_TABLE, MF_K_ATTN_FWD_ROT, MF_K_ATTN_BWD_DQ,
       MF_K_COUNT };
mf_status mf_timing_enable(int32_t on);
mf_status mf_timing_reset(void);
mf_status mf_timing_read(int32_t id, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* MF_H_ */
