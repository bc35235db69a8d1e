/*
 * exattn.h -- C ABI of the fused exact-attention library for NVIDIA GB300
 * (sm_103a), libexattn.so.
 *
 * The operation is exact scaled-dot-product attention,
 *
 *     O = softmax(scale * Q K^T  [+ causal mask]) V,
 *
 * computed as one fused, tiled kernel with an online softmax so that the
 * score matrix S and the probability matrix P never reach device memory
 * ("Gemini 3 Flash的注意力内核重写：算子融合如何实现亚毫秒级推理",
 * §1 内核融合策略, §2 分块, §3 在线softmax算法), and its gradient, which
 * recomputes S and P tile by tile from the stored per-row statistic (same
 * page, §4 重计算).  The causal flag follows the flash_attn_func example of
 * "提示词再优也救不了的性能黑洞：Transformer注意力计算冗余分析（含
 * FlashAttention-3内核级优化验证数据）", 第一章: key j is visible to query i
 * iff j <= i (square, top-left aligned); key tiles wholly above the diagonal
 * are skipped.
 *
 * Conventions shared by every call
 *   - Q, K, V, O, dO, dQ, dK, dV are bf16 (2-byte __nv_bfloat16), device
 *     pointers, contiguous [B, H, N, d] with d fastest (the [B, H, T, D]
 *     layout of the "提示词再优…" page, §2.3), 16-byte aligned.
 *   - lse is fp32 [B, H, N], 4-byte aligned: lse[b,h,i] = m_i + ln(l_i), the
 *     natural-log logsumexp of row i of the scaled, masked logits (the row
 *     max m_i and normaliser l_i of the "Gemini 3 Flash…" page, §4, folded
 *     into one number).
 *   - 1 <= B, 1 <= H, 1 <= N, B*H*N < 2^31, d in {64, 128}; scale finite, > 0.
 *     N need not be a multiple of the tile size.
 *   - All pointers belong to the caller, who allocates and frees them; the
 *     library allocates no device memory and never synchronises.  Inputs are
 *     read only; outputs must not alias inputs or each other.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) on the current device.  The return value reports
 *     argument errors and launch errors; faults during execution surface at
 *     the caller's next synchronisation, and the kernels' own watchdog
 *     (every internal wait is bounded) is read with exattn_device_error().
 *   - Only sm_103 devices are supported (EXATTN_ERR_ARCH otherwise).
 */
#ifndef EXATTN_H
#define EXATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  EXATTN_OK = 0,
  EXATTN_ERR_NULL = 1,        /* a required pointer is NULL */
  EXATTN_ERR_SHAPE = 2,       /* B, H or N out of range */
  EXATTN_ERR_ALIGN = 3,       /* a pointer is not aligned as stated above */
  EXATTN_ERR_UNSUPPORTED = 4, /* d not in {64, 128} */
  EXATTN_ERR_ARCH = 5,        /* current device is not sm_103 */
  EXATTN_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required */
  EXATTN_ERR_CUDA = 7,        /* a CUDA runtime/driver call or a launch failed */
  EXATTN_ERR_TIMEOUT = 8,     /* a kernel's bounded internal wait gave up */
  EXATTN_ERR_VALUE = 9        /* scale not finite or not positive */
} exattn_status;

/*
 * attn_fwd -- forward pass.
 *   q, k, v : inputs, bf16 [B, H, N, d].
 *   o       : output, bf16 [B, H, N, d]; O_i = sum_j P_ij V_j, rounded to
 *             nearest-even bf16 from fp32.
 *   lse     : output, fp32 [B, H, N] (see above); it is the exact input that
 *             attn_bwd expects.
 *   causal  : 0 = full attention, nonzero = causal mask (j <= i).
 *   scale   : multiplies Q K^T before masking and softmax (1/sqrt(d) usual).
 *   stream  : cudaStream_t.
 * Arithmetic: bf16 products accumulated in fp32 on the tensor cores; the
 * softmax runs in fp32; P is rounded to f16 before the P V product, and V
 * is converted to f16 in shared memory for it (exact for 2^-14 <= |v| <=
 * 65504 and for 0; entries beyond +-65504 are not supported).
 * Returns an exattn_status.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
             int causal, float scale, void* stream);

/*
 * attn_bwd_workspace_size -- bytes of device workspace attn_bwd needs for
 * this shape (fp32 row terms D_i = sum_c dO_ic O_ic, one per query row).
 * Returns 0 for an invalid shape.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d, int causal);

/*
 * attn_bwd -- backward pass of attn_fwd for output gradient dO.
 *   q, k, v, o, lse : the forward's inputs and outputs (o and lse exactly as
 *                     attn_fwd wrote them).
 *   dO              : bf16 [B, H, N, d], gradient of the loss w.r.t. O.
 *   dq, dk, dv      : outputs, bf16 [B, H, N, d].
 *   workspace       : device memory of at least
 *                     attn_bwd_workspace_size(B, H, N, d, causal) bytes,
 *                     16-byte aligned, owned by the caller; its contents on
 *                     entry are ignored and on return are unspecified.
 * It computes D_i = sum_c dO_ic O_ic (inside the dQ kernel, which stores it
 * in the workspace for the dK/dV kernel that follows), and for every tile
 * pair recomputes
 * P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i.v_j, dS_ij = P_ij (dP_ij - D_i)
 * and accumulates dV_j += P_ij dO_i, dK_j += scale dS_ij q_i (one pass over
 * query tiles per key tile) and dQ_i += scale dS_ij k_j (one pass over key
 * tiles per query tile).  No atomics: every output element is summed by one
 * CTA in a fixed order, so results are bit-identical from run to run.
 * Returns an exattn_status.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
             void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* workspace,
             size_t workspace_bytes, void* stream);

/*
 * The stages of attn_bwd as separate calls, for callers that schedule them
 * themselves (e.g. dK/dV and dQ on two streams once D is ready, or timing
 * each kernel).  attn_bwd(...) equals attn_bwd_d_and_dq followed by
 * attn_bwd_dkdv on one stream, with D in the workspace; attn_bwd_preprocess
 * followed by attn_bwd_dkdv and attn_bwd_dq gives bit-identical results
 * with one more launch.
 *
 * attn_bwd_preprocess -- D[b,h,i] = sum_c dO[b,h,i,c] O[b,h,i,c], the
 *   per-row term of the softmax gradient (dS_ij = P_ij (dP_ij - D_i)).
 *   D: fp32 [B, H, N], 4-byte aligned, written.
 * attn_bwd_dkdv -- dK and dV (bf16 [B, H, N, d], written) from q, k, v, dO,
 *   lse (as written by attn_fwd) and D (from attn_bwd_preprocess).
 * attn_bwd_dq   -- dQ (bf16 [B, H, N, d], written) from the same inputs.
 * attn_bwd_d_and_dq -- both D (written, as attn_bwd_preprocess writes it,
 *   bit for bit) and dQ (as attn_bwd_dq computes it from that D) in one
 *   kernel, from q, k, v, o, dO and lse; D is complete when the call's work
 *   on the stream is.
 * Validation, alignment and error codes as for attn_bwd.
 */
int attn_bwd_preprocess(const void* o, const void* dO, float* D, int B, int H, int N, int d, void* stream);
int attn_bwd_dkdv(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* D,
                  void* dk, void* dv, int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_dq(const void* q, const void* k, const void* v, const void* dO, const float* lse, const float* D,
                void* dq, int B, int H, int N, int d, int causal, float scale, void* stream);
int attn_bwd_d_and_dq(const void* q, const void* k, const void* v, const void* o, const void* dO, const float* lse,
                      float* D, void* dq, int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * Element type and layout for the _ex calls below.  The flash_attn_func
 * example of "提示词再优也救不了的性能黑洞…", 第一章, passes fp16 tensors laid
 * out [batch, seqlen, heads, head_dim]; the _ex calls accept that layout (or
 * any other whose head_dim axis is contiguous) and either 16-bit type.
 *
 * exattn_dtype -- element type of every Q, K, V, O, dO, dQ, dK, dV of one
 *   call: EXATTN_DTYPE_BF16 (__nv_bfloat16) or EXATTN_DTYPE_F16 (__half).
 *   The tensor cores multiply that type and accumulate in fp32; P (and dS in
 *   the backward) are rounded to the same type; outputs are rounded to it.
 * exattn_strides -- element strides (not bytes) of a tensor seen as
 *   [B, H, N, d] with d contiguous: element (b, h, n, c) is at
 *   base[b*b_stride + h*h_stride + n*n_stride + c].  Every stride must be a
 *   multiple of 8 elements (16 bytes, the tensor-memory-accelerator rule),
 *   at least 0 and below 2^36, and nonzero along an axis of extent > 1
 *   (else EXATTN_ERR_ALIGN / EXATTN_ERR_SHAPE).  Contiguous [B, H, N, d] is
 *   {H*N*d, N*d, d}; contiguous [B, N, H, d] is {N*H*d, d, H*d}.  Rows of an
 *   output that overlap give undefined results.
 */
typedef enum { EXATTN_DTYPE_BF16 = 0, EXATTN_DTYPE_F16 = 1 } exattn_dtype;

typedef struct {
  long long b_stride;
  long long h_stride;
  long long n_stride;
} exattn_strides;

/*
 * window -- sliding-window (local) attention for the _ex calls.  The
 *   "Flash Attention V3：大模型加速的核心网络算子优化实践" page, §三.1, pairs
 *   local attention (LocalAttention(window_size=...)) with global attention
 *   without defining the window; here window = W >= 1 lets query i see key j
 *   only if i - j < W (the W keys ending at the diagonal under the causal
 *   mask) and, without the causal mask, also j - i < W.  window = 0 is no
 *   window; a negative window returns EXATTN_ERR_VALUE.  Key tiles wholly
 *   outside every row's window are skipped.
 *
 * attn_fwd_ex -- attn_fwd for any exattn_dtype, strided Q, K, V, O and an
 *   optional window (lse stays fp32 contiguous [B, H, N]).  Results and
 *   errors as attn_fwd; an unknown dtype returns EXATTN_ERR_UNSUPPORTED.
 */
int attn_fwd_ex(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                const void* v, exattn_strides v_strides, void* o, exattn_strides o_strides, float* lse, int B,
                int H, int N, int d, int causal, int window, float scale, void* stream);

/*
 * attn_bwd_ex -- attn_bwd for any exattn_dtype, strided Q, K, V, O, dO, dQ,
 *   dK, dV and the window the forward used (lse and the workspace as for
 *   attn_bwd).  Results and errors as attn_bwd.
 */
int attn_bwd_ex(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                const void* v, exattn_strides v_strides, const void* o, exattn_strides o_strides, const void* dO,
                exattn_strides do_strides, const float* lse, void* dq, exattn_strides dq_strides, void* dk,
                exattn_strides dk_strides, void* dv, exattn_strides dv_strides, int B, int H, int N, int d,
                int causal, int window, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The backward's row terms D_i = dO_i . O_i ("Gemini 3 Flash的注意力内核重写：
 * 算子融合如何实现亚毫秒级推理", §4 重计算: recompute from the stored row
 * statistics) taken from an fp32 copy of O instead of the O rounded to the
 * input type.  Where a row's softmax puts nearly all its weight on one key,
 * dS = P (dP - D) is a small difference and the 16-bit rounding of O
 * dominates it: on such rows the fp32 copy keeps the gradients within the
 * relative bound (a two-token sequence with weights 0.96 / 0.04: dQ relative
 * error 0.10 from the bf16 O, 1.5e-4 from the fp32 copy).  It costs a
 * d x 4-byte row per query in device memory and writes.
 *   attn_fwd_o32 -- attn_fwd_ex that also writes o32: fp32, contiguous
 *     [B, H, N, d], 16-byte aligned, owned by the caller; each row is the
 *     normalised O before its rounding to the output type.  Errors as
 *     attn_fwd_ex; a NULL o32 returns EXATTN_ERR_NULL.
 *   attn_bwd_o32 -- attn_bwd_ex with o32 (as attn_fwd_o32 wrote it) in place
 *     of O, which is not read.  Results and errors as attn_bwd_ex.
 */
int attn_fwd_o32(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                 const void* v, exattn_strides v_strides, void* o, exattn_strides o_strides, float* lse, float* o32,
                 int B, int H, int N, int d, int causal, int window, float scale, void* stream);
int attn_bwd_o32(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                 const void* v, exattn_strides v_strides, const float* o32, const void* dO, exattn_strides do_strides,
                 const float* lse, void* dq, exattn_strides dq_strides, void* dk, exattn_strides dk_strides, void* dv,
                 exattn_strides dv_strides, int B, int H, int N, int d, int causal, int window, float scale,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * Packed variable-length batches.  The masked_flash_attention sketch of
 * "Flash Attention V3：大模型加速的核心网络算子优化实践", §三.3, pads
 * variable-length sequences and masks the padding with a [batch, 1, seq,
 * seq] tensor; here the sequences are packed instead, so neither the padding
 * nor an N x N mask exists.
 *   cu_seqlens : device int32 [B + 1], 4-byte aligned, non-decreasing offsets
 *                with cu_seqlens[0] = 0 and cu_seqlens[B] = total: sequence b
 *                is rows [cu_seqlens[b], cu_seqlens[b+1]) of every tensor.
 *                Offsets are clamped to [0, total] and lengths to max_seqlen
 *                on the device, so a wrong table gives wrong results but
 *                never an out-of-bounds access.
 *   q, k, v, o, dO, dq, dk, dv : [total, H, d] (d contiguous) described by
 *                exattn_strides with b_stride unused (any multiple of 8),
 *                h_stride and n_stride (the token stride).
 *   lse        : fp32 [H, total] (head-major), as is the backward's D.
 *   max_seqlen : the longest sequence (sizes the grid; 1 <= max_seqlen).
 *   total      : rows of the packed tensors, H * total < 2^31.
 * Each sequence is its own attention problem (masks, window and causal
 * alignment apply within it).  Errors as the _ex calls; a null cu_seqlens
 * returns EXATTN_ERR_NULL.  attn_bwd_varlen needs a workspace of
 * attn_bwd_workspace_size(1, H, total, d, causal) bytes.
 */
int attn_fwd_varlen(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                    const void* v, exattn_strides v_strides, void* o, exattn_strides o_strides, float* lse,
                    const int* cu_seqlens, int B, int H, int max_seqlen, int total, int d, int causal, int window,
                    float scale, void* stream);
int attn_bwd_varlen(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                    const void* v, exattn_strides v_strides, const void* o, exattn_strides o_strides,
                    const void* dO, exattn_strides do_strides, const float* lse, void* dq,
                    exattn_strides dq_strides, void* dk, exattn_strides dk_strides, void* dv,
                    exattn_strides dv_strides, const int* cu_seqlens, int B, int H, int max_seqlen, int total,
                    int d, int causal, int window, float scale, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Decode-shaped forward: few queries against many keys (token-by-token
 * generation, the inference latency goal of "Gemini 3 Flash的注意力内核重写：
 * 算子融合如何实现亚毫秒级推理", §引言).  Q and O are [B, H, Nq, d], K and V
 * [B, H, Nk, d] (strided as for the _ex calls), lse fp32 [B, H, Nq].  The
 * queries are the last Nq positions of the key sequence (bottom-right
 * alignment): under the causal mask query i sees keys j <= i + Nk - Nq, and
 * a window counts from that position.  With Nq = Nk this is attn_fwd_ex.
 * The keys are split over several CTAs per (batch, head) when B*H alone
 * would leave SMs idle long enough for splits to finish sooner (few heads,
 * long key sequences); each split writes fp32 partial results to the
 * workspace and a second kernel merges them (the same logsumexp-weighted
 * combination the online softmax uses inside one CTA).  The split count
 * depends only on (B, H, Nq, Nk, d), so the workspace size does too.
 *   attn_fwd_decode_workspace_size -- bytes of workspace for this shape (0
 *     when no split is needed; then workspace may be NULL); 0 also for an
 *     invalid shape.
 *   Errors as attn_fwd_ex; Nq > Nk with the causal mask or a window
 *   returns EXATTN_ERR_SHAPE (a query would see no key).
 */
size_t attn_fwd_decode_workspace_size(int B, int H, int Nq, int Nk, int d);
int attn_fwd_decode(int dtype, const void* q, exattn_strides q_strides, const void* k, exattn_strides k_strides,
                    const void* v, exattn_strides v_strides, void* o, exattn_strides o_strides, float* lse, int B,
                    int H, int Nq, int Nk, int d, int causal, int window, float scale, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * attn_bwd_noalloc -- attn_bwd for callers that cannot allocate device
 * memory: a plugin given only its input and output buffers by a runtime that
 * owns all device memory, or code on a latency-critical path where an
 * allocation (which may synchronise the device) is not allowed.  The pages
 * this library follows have no counterpart of this call; it exists only for
 * such callers.
 *   Arguments, layout, results and errors are those of attn_bwd, without
 *   the workspace: the row terms D_i live in a 16 MiB array built into the
 *   library (fp32, one per query row), so B*H*N may be at most 4,194,304;
 *   larger shapes return EXATTN_ERR_WORKSPACE without launching anything.
 *   It calls no cudaMalloc, cudaFree or other allocating routine.
 *   The array occupies 16 MiB of device memory on every GPU that loads the
 *   library, until the library is unloaded.  The first call on each device
 *   looks up the array's device address (a runtime query, no allocation);
 *   make that first call before any stream capture.  The address stays
 *   valid for the life of the process's context on that device: after a
 *   cudaDeviceReset (or a primary-context teardown) this library must not
 *   be used again in that process.  Every call shares the
 *   array and it keeps the last call's contents (nothing in it needs to start
 *   at zero: each call writes every D_i before reading it), so calls whose
 *   executions overlap on the GPU (e.g. on two streams) race and must be
 *   ordered by the caller.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal,
                     float scale, void* stream);

/*
 * Forward and backward on host-resident tensors: attn_fwd followed by the
 * backward (the fused forward of "Gemini 3 Flash的注意力内核重写：算子融合如何
 * 实现亚毫秒级推理", §1 内核融合策略, and its recomputing backward, §4), with
 * the host <-> device copies inside the call.  The (batch, head) problems
 * run in `groups` groups: each group's Q, K, V then dO are copied in on
 * copy_in_stream while earlier groups compute; its O and lse are copied out
 * on copy_out_stream while its backward runs, dK and dV while its dQ is
 * computed, then dQ.  Odd-numbered groups compute on stream2 when it is
 * given (the kernels of small groups then share the GPU), the others on
 * `stream`.
 *   dtype : EXATTN_DTYPE_BF16 or EXATTN_DTYPE_F16.
 *   q, k, v, dO : HOST memory, contiguous [B, H, N, d] of dtype; o, dq, dk,
 *     dv likewise (outputs), lse fp32 [B, H, N] (output).  Use page-locked
 *     (pinned) memory: copies from pageable memory are not asynchronous and
 *     do not overlap the kernels.
 *   workspace : device memory of at least attn_fwd_bwd_host_workspace_size
 *     bytes, 16-byte aligned, owned by the caller; it holds the device copies
 *     of all nine tensors and the backward's row terms.
 *   groups : >= 1 (clamped to B*H).
 *   stream : the call's work is ordered after the work already queued on
 *     it, and everything queued on it afterwards runs after the call's work
 *     (the copies included): synchronise it before reading the outputs.
 *     copy_in_stream, copy_out_stream, stream2 : other streams of the same
 *     device, or NULL (that role then runs on `stream`, without overlap).
 * Asynchronous; allocates no device memory; creates and destroys a few CUDA
 * events per call (their last uses complete with the call's work).
 * Validation and errors as attn_bwd (workspace: EXATTN_ERR_WORKSPACE;
 * groups < 1: EXATTN_ERR_VALUE).  An error returned after the first copy
 * was queued leaves the outputs undefined.
 */
size_t attn_fwd_bwd_host_workspace_size(int B, int H, int N, int d, int causal);
int attn_fwd_bwd_host(int dtype, const void* q, const void* k, const void* v, const void* dO, void* o, float* lse,
                      void* dq, void* dk, void* dv, int B, int H, int N, int d, int causal, float scale,
                      void* workspace, size_t workspace_bytes, int groups, void* stream, void* copy_in_stream,
                      void* copy_out_stream, void* stream2);

/* Human-readable text of an exattn_status (static storage, never NULL). */
const char* exattn_status_string(int status);

/*
 * exattn_last_cuda_error -- the CUDA call behind the last EXATTN_ERR_CUDA
 * returned on the calling host thread: "<call>: <cudaError name> (<code>)",
 * or "<call>: CUresult <code>" for the driver's tensor-map encoder; "" if no
 * CUDA call of the library has failed on this thread.  Kept per thread, so
 * it is read on the thread that saw the status.  The text is owned by the
 * library and stays valid until the thread's next call of this function.
 */
const char* exattn_last_cuda_error(void);

/*
 * exattn_device_error -- synchronises the current device, reads and clears
 * the kernels' watchdog word.  Returns EXATTN_OK if no bounded wait gave up
 * since the last call, EXATTN_ERR_TIMEOUT if one did (the outputs of the
 * affected launches are then garbage), EXATTN_ERR_CUDA if the read failed.
 */
int exattn_device_error(void);

/*
 * exattn_device_error_poll -- the watchdog word without synchronising:
 * queues on `stream` a copy of the current device's word (0 = no wait gave
 * up; nonzero = exattn_device_error() would return EXATTN_ERR_TIMEOUT) into
 * *host_dst, after the work already queued there.  The value is valid once
 * that copy has completed (e.g. an event recorded after it has).  host_dst
 * should be page-locked, otherwise the copy is synchronous.  Does not clear
 * the word.  Returns EXATTN_ERR_NULL for a NULL host_dst.
 */
int exattn_device_error_poll(unsigned* host_dst, void* stream);

/*
 * exattn_watchdog_selftest -- exercises the failure path of the kernels'
 * bounded waits without any fault: launches one warp that waits on a
 * barrier nothing arrives on, giving up after timeout_us microseconds
 * (1..1,000,000).  The next exattn_device_error() then returns
 * EXATTN_ERR_TIMEOUT (and clears the word); the context stays usable.
 * While the word is set, waits in other launches that have to spin give up
 * early, so read it before launching real work.  Returns EXATTN_ERR_VALUE
 * for a timeout out of range.
 */
int exattn_watchdog_selftest(unsigned timeout_us, void* stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int exattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EXATTN_H */
