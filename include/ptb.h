/*
 * ptb.h - C ABI of libptb: the forward pass of MegaScale's parallel
 * transformer block (PTB) with causal sliding-window attention (SWA), as
 * hand-written CUDA kernels for GB300 (sm_103a).
 *
 * Definitions (MegaScale study notes, ai-yanyi-papers.pages.dev/papers/
 * 18-megascale.html, ch.2 §2.2 = paper §3.1, algorithm-change table):
 *   PTB row:  y = x + MLP(LN(x)) + Attention(LN(x))   -- one shared LN,
 *             attention and MLP branches computed side by side and summed.
 *   SWA row:  each token attends only to a fixed window of w positions,
 *             cost O(s*w) rather than O(s*s).
 * Readings fixed here: the window is causal and includes the token itself,
 * so query row i attends to keys max(0, i-w+1) .. i (exactly min(i+1, w)
 * keys); w >= s is plain causal attention.  Softmax scale 1/sqrt(d) unless
 * given; MLP(u) = gelu_tanh(u W_up^T) W_down^T; LayerNorm uses the biased
 * variance with eps = 1e-5; no biases, dropout or positional terms.
 *
 * Numerics: bf16 storage, fp32 accumulation in every contraction, fp32
 * LayerNorm statistics and softmax, one round-to-nearest-even bf16 rounding
 * per stored tensor.
 *
 * Common conventions
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the
 *     library never frees or retains caller memory.  bf16 values are passed
 *     as raw 16-bit patterns (ptb_bf16).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream) on the current CUDA device.  No entry
 *     point synchronises except ptb_last_device_error(stream), which waits
 *     for that one stream.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned as a ptb_status; nothing is written in that case.
 *   - Kernels never trap.  A device-side wait that does not complete within
 *     about two seconds makes the kernel give up, record PTB_ERR_TIMEOUT in
 *     the per-device status word and return; ptb_last_device_error(stream)
 *     reads and clears that word.
 */
#ifndef PTB_H_
#define PTB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t ptb_bf16; /* raw bfloat16 bits */
typedef void* ptb_stream;  /* cudaStream_t */

typedef enum {
  PTB_OK = 0,
  PTB_ERR_ARG = 1,         /* null pointer, non-positive size, bad window   */
  PTB_ERR_SHAPE = 2,       /* shape outside the supported set (see below)   */
  PTB_ERR_ALIGN = 3,       /* pointer or stride not 16-byte aligned         */
  PTB_ERR_WORKSPACE = 4,   /* caller workspace smaller than required        */
  PTB_ERR_LAUNCH = 5,      /* CUDA launch or runtime error                  */
  PTB_ERR_TIMEOUT = 6,     /* a device-side wait gave up (kernel unwound)   */
  PTB_ERR_UNSUPPORTED = 7, /* device is not sm_103 / sm_100 class           */
  PTB_ERR_DEVICE = 8       /* device query or allocation failed             */
} ptb_status;

/* Human-readable name of a status code (static string, never NULL). */
const char* ptb_status_string(ptb_status status);

/*
 * Bytes of scratch that ptb_forward needs for this shape on the current
 * device: the normalised activations xn [T, H] and the fused projection
 * output U [T, 3H + F] (T = batch * seq), each bf16 and 256-byte aligned,
 * followed by ptb_gemm_workspace_size(T, hidden, ffn) bytes for the GEMMs'
 * split last wave.  The last part depends on the device's SM count.
 */
size_t ptb_forward_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn);

/*
 * ptb_forward: y = x + Attn(LN(x)) + MLP(LN(x))  (PTB row, §2.2).
 *
 *   x        [batch, seq, hidden]   bf16, row-major (token-major)
 *   ln_gamma [hidden], ln_beta [hidden]  LayerNorm affine parameters
 *   w_qkv    [3*hidden, hidden]  nn.Linear layout [out, in]: rows hold all
 *            query heads, then all key heads, then all value heads; head h
 *            occupies rows h*d .. h*d+d-1 of each third (d = hidden/heads)
 *   w_o      [hidden, hidden]    input columns ordered by head
 *   w_up     [ffn, hidden], w_down [hidden, ffn]
 *   heads    number of attention heads; d = hidden / heads must be one of
 *            16, 32, 64, 96, 128
 *   window   SWA window w >= 1 (w >= seq means full causal attention)
 *   y        [batch, seq, hidden] bf16 output; must not alias any input
 *   workspace, workspace_bytes
 *            caller scratch of at least ptb_forward_workspace_size() bytes,
 *            256-byte aligned; or NULL/0, in which case the library uses
 *            an arena of its own per device, grown on demand with
 *            cudaMalloc and kept until ptb_release_workspace().
 *   stream   CUDA stream for every launch.
 *
 * Shapes: hidden and ffn multiples of 64, hidden <= 32768, batch*seq >= 1.
 * Pointers 16-byte aligned.  Four kernels run in order on `stream`:
 * LayerNorm, the [QKV | up] GEMM with the GELU epilogue, banded SWA, and the
 * K-concatenated [out | down] GEMM whose epilogue adds x.
 */
ptb_status ptb_forward(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                       const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                       const ptb_bf16* w_down, int64_t batch, int64_t seq, int64_t hidden,
                       int64_t ffn, int32_t heads, int32_t window, ptb_bf16* y,
                       void* workspace, size_t workspace_bytes, ptb_stream stream);

/*
 * Same as ptb_forward, and records `events[0..4]` (cudaEvent_t handles owned
 * by the caller; n_events must be 5) on `stream` before the LayerNorm, the
 * first GEMM, the attention, the second GEMM and after it, so a caller can
 * time each kernel.  Every handle must be a created event; a NULL handle or
 * a failed record returns PTB_ERR_ARG (kernels already enqueued stay queued).
 */
ptb_status ptb_forward_events(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                              const ptb_bf16* ln_beta, const ptb_bf16* w_qkv,
                              const ptb_bf16* w_o, const ptb_bf16* w_up, const ptb_bf16* w_down,
                              int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                              int32_t heads, int32_t window, ptb_bf16* y, void* workspace,
                              size_t workspace_bytes, ptb_stream stream, void* const* events,
                              int32_t n_events);

/*
 * ptb_forward_host: ptb_forward with x and y in host memory (the layer's
 * parameters stay in device memory).  Enqueues on `stream`: the copy of x
 * [batch, seq, hidden] to the device, the layer, and the copy of y back;
 * returns without waiting, so y_host is valid once the stream has reached
 * that point (cudaStreamSynchronize or an event).  x_host and y_host should
 * be page-locked (cudaHostAlloc / cudaHostRegister) for the copies to run
 * asynchronously and overlap with another stream's work; pageable memory
 * works but the copies then block the calling thread.  `workspace` is
 * caller-owned device memory of ptb_forward_host_workspace_size bytes
 * (256-byte aligned; not null), holding the device copies of x and y and
 * the layer's scratch; calls in flight at the same time need separate
 * workspaces.  For layers whose first GEMM exceeds 2^39 multiply-adds the
 * layer of each call runs after the layer of the previous such call on the
 * same device, whatever its stream (the kernels take every SM, so two large
 * layers at once only compete), while the copies of calls on different
 * streams overlap the other calls' layers; smaller layers of calls on
 * different streams may run side by side.  Errors as ptb_forward.
 */
size_t ptb_forward_host_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn);
ptb_status ptb_forward_host(const ptb_bf16* x_host, const ptb_bf16* ln_gamma,
                            const ptb_bf16* ln_beta, const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                            const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t batch,
                            int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                            int32_t window, ptb_bf16* y_host, void* workspace,
                            size_t workspace_bytes, ptb_stream stream);

/*
 * ptb_forward_noalloc: ptb_forward for callers that cannot allocate device
 * memory.  The paper has no counterpart; this is a deployment convenience.
 *
 * Programs that manage all device memory themselves (a framework's caching
 * allocator, a server that reserves memory at start-up and must not call
 * cudaMalloc later because it can stall the device or fail when memory is
 * fragmented, a plug-in whose host forbids raw allocations) can neither let
 * the library grow its arena nor always lend it a buffer.  This entry point
 * takes the same inputs and output as ptb_forward but uses, as scratch, one
 * fixed 64 MiB array compiled into the library, so it calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 *   - Size limit: ptb_forward_workspace_size(batch, seq, hidden, ffn) must
 *     be <= 64 MiB (67108864 bytes); larger layers return PTB_ERR_WORKSPACE
 *     without launching anything.
 *   - The array takes 64 MiB of device memory on every GPU where the
 *     library's code for this entry point is loaded, until the process exits.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps whatever the last call left
 *     in it; nothing in it has to start at zero.  Calls whose work overlaps on
 *     the GPU (other streams, other host threads) race on it: serialise them.
 * Other arguments, shape rules and errors are those of ptb_forward.
 */
ptb_status ptb_forward_noalloc(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                               const ptb_bf16* ln_beta, const ptb_bf16* w_qkv,
                               const ptb_bf16* w_o, const ptb_bf16* w_up, const ptb_bf16* w_down,
                               int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                               int32_t heads, int32_t window, ptb_bf16* y, ptb_stream stream);

/*
 * ptb_serial_forward: the serial block that the PTB replaces (MegaScale
 * notes, §2.2, PTB row, where it is printed without the attention residual;
 * read here as the standard pre-LN block):
 *   h = x + Attn(LN1(x)),   y = h + MLP(LN2(h)).
 * Same weights, layouts, shape rules and errors as ptb_forward, plus a
 * second LayerNorm (ln2_gamma, ln2_beta).  Seven kernels in order: LN1,
 * QKV GEMM, SWA, out-projection GEMM + x, LN2, up-projection GEMM + GELU,
 * down-projection GEMM + h.  workspace as for ptb_forward, sized by
 * ptb_serial_workspace_size().
 */
size_t ptb_serial_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn);
ptb_status ptb_serial_forward(const ptb_bf16* x, const ptb_bf16* ln1_gamma,
                              const ptb_bf16* ln1_beta, const ptb_bf16* ln2_gamma,
                              const ptb_bf16* ln2_beta, const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                              const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t batch,
                              int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                              int32_t window, ptb_bf16* y, void* workspace,
                              size_t workspace_bytes, ptb_stream stream);

/*
 * FP8 variant of ptb_forward.  The Megatron-LM page (mixed-precision
 * section) lists FP8 among the supported precisions, to be used with dynamic
 * scaling and with care for stability.  Both GEMMs take e4m3 operands with
 * one dynamic fp32 scale per row of each operand:
 *   xn8 = e4m3(LN(x) / sx), sx[t] = amax_t / 448   (per token)
 *   A8  = e4m3([ctx | G] / sa), sa[t] per token    (second GEMM's input)
 *   w1  = [W_qkv ; W_up] in e4m3 with s1[n] per output row   ([3H+F, H])
 *   w2  = [W_o | W_down] in e4m3 with s2[n] per output row    ([H, H+F])
 * and the accumulator is dequantized as sx[t] * s[n] * acc.  Attention, the
 * GELU, the residual and all stored activations other than the two e4m3
 * GEMM inputs stay bf16.  Accuracy is that of e4m3 (3 mantissa bits); the
 * tests bound it by an exact computation with the same e4m3 rounding points.
 *
 * ptb_prepare_fp8_weights quantizes the bf16 weights once (w1, s1, w2, s2 are
 * caller-owned device buffers of the sizes above).
 * ptb_forward_fp8 then runs LN+quantize, the e4m3 [QKV | up] GEMM + GELU,
 * SWA, a row quantization of [ctx | G], and the e4m3 [out | down] GEMM + x.
 * Same shape rules, workspace and error conventions as ptb_forward, except
 * that hidden and ffn must be multiples of 128 (one e4m3 k-block).
 */
size_t ptb_forward_fp8_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn);
ptb_status ptb_prepare_fp8_weights(const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                                   const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t hidden,
                                   int64_t ffn, uint8_t* w1, float* s1, uint8_t* w2, float* s2,
                                   ptb_stream stream);
ptb_status ptb_forward_fp8(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                           const uint8_t* w1, const float* s1, const uint8_t* w2, const float* s2,
                           int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                           int32_t window, ptb_bf16* y, void* workspace, size_t workspace_bytes,
                           ptb_stream stream);
/*
 * ptb_forward_fp8 that also records six caller-owned CUDA events (cudaEvent_t
 * passed as void*) on `stream`: before the LN + quantize kernel, the first
 * GEMM, SWA, the row quantization and the second GEMM, and after the second
 * GEMM.  n_events must be 6; a null event or a failed record returns
 * PTB_ERR_ARG (kernels already enqueued stay queued).
 */
ptb_status ptb_forward_fp8_events(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                                  const ptb_bf16* ln_beta, const uint8_t* w1, const float* s1,
                                  const uint8_t* w2, const float* s2, int64_t batch, int64_t seq,
                                  int64_t hidden, int64_t ffn, int32_t heads, int32_t window,
                                  ptb_bf16* y, void* workspace, size_t workspace_bytes,
                                  ptb_stream stream, void* const* events, int32_t n_events);

/*
 * Training: forward pass that keeps its activations, and the backward pass.
 *
 * The pages' workload is training: MegaScale counts 6N FLOPs per token, 2N
 * forward and 4N backward (MegaScale study notes, ch.2 §2.1, MFU
 * definition).  The backward pass is the chain rule of the PTB definition
 * (§2.2, PTB row):
 *   dW_o = dy^T ctx,   dW_down = dy^T G,   dctx = dy W_o,   dG = dy W_down,
 *   dZ = dG * gelu_tanh'(Z),   [dQ | dK | dV] = SWA backward of dctx,
 *   dxn = [dQ | dK | dV] W_qkv + dZ W_up,   [dW_qkv ; dW_up] = [dQ | dK | dV | dZ]^T xn,
 *   dx = dy + LN backward of dxn,   dgamma, dbeta = sums over tokens.
 *
 * ptb_forward_train computes y exactly as ptb_forward does and writes into
 * `saved` (caller-owned device memory of ptb_train_saved_size bytes, 256-byte
 * aligned) what the backward pass reads: xn = LN(x), the per-token LN mean
 * and 1/sqrt(var + eps) (fp32 pairs), U = [Q | K | V | G], the
 * pre-activation Z = xn W_up^T, ctx, and the attention's per-row
 * log-sum-exp (fp32, base 2).  `workspace` as in ptb_forward (null: the
 * library arena).
 *
 * ptb_backward takes the upstream gradient dy [batch, seq, H] (bf16), the
 * forward inputs x, ln_gamma and the four weights, and `saved` from
 * ptb_forward_train on the same inputs; it writes dx (bf16, [batch, seq, H])
 * and, in fp32, dln_gamma [H], dln_beta [H], dw_qkv [3H, H], dw_o [H, H],
 * dw_up [F, H], dw_down [H, F] (same layouts as the weights; overwritten, not
 * accumulated).  Scratch: `workspace` of ptb_backward_workspace_size bytes
 * (256-byte aligned), or null for the library arena.  Ten kernels on
 * `stream`: two GEMMs, the attention backward (three kernels), two GEMMs,
 * the LayerNorm backward (three kernels), plus a counter reset before each
 * GEMM whose last wave is split along K.  Sums run in a fixed order, so the
 * results are the same bits on every call.  Shape rules, alignment and errors as in
 * ptb_forward; PTB_ERR_WORKSPACE if `saved` is too small.
 */
size_t ptb_train_saved_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                            int32_t heads);
ptb_status ptb_forward_train(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                             const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                             const ptb_bf16* w_down, int64_t batch, int64_t seq, int64_t hidden,
                             int64_t ffn, int32_t heads, int32_t window, ptb_bf16* y, void* saved,
                             size_t saved_bytes, void* workspace, size_t workspace_bytes,
                             ptb_stream stream);
size_t ptb_backward_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                                   int32_t heads);
ptb_status ptb_backward(const ptb_bf16* dy, const ptb_bf16* x, const ptb_bf16* ln_gamma,
                        const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                        const ptb_bf16* w_down, const void* saved, size_t saved_bytes,
                        int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                        int32_t window, ptb_bf16* dx, float* dln_gamma, float* dln_beta,
                        float* dw_qkv, float* dw_o, float* dw_up, float* dw_down, void* workspace,
                        size_t workspace_bytes, ptb_stream stream);
/*
 * ptb_backward that also records seven caller-owned CUDA events (cudaEvent_t
 * passed as void*) on `stream`: before the [out | down] input-gradient GEMM,
 * the [out | down] weight-gradient GEMM, the attention backward, the
 * [QKV | up] input-gradient GEMM, the [QKV | up] weight-gradient GEMM and
 * the LayerNorm backward, and after it.  n_events must be 7; a null event or
 * a failed record returns PTB_ERR_ARG.
 */
ptb_status ptb_backward_events(const ptb_bf16* dy, const ptb_bf16* x, const ptb_bf16* ln_gamma,
                               const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                               const ptb_bf16* w_down, const void* saved, size_t saved_bytes,
                               int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                               int32_t heads, int32_t window, ptb_bf16* dx, float* dln_gamma,
                               float* dln_beta, float* dw_qkv, float* dw_o, float* dw_up,
                               float* dw_down, void* workspace, size_t workspace_bytes,
                               ptb_stream stream, void* const* events, int32_t n_events);

/*
 * ptb_set_gemm_pairs: tile shape of the bf16 GEMMs on the current device.
 * 1: 256 x 256 tiles on CTA pairs (a cluster of two CTAs on one TPC, tcgen05
 * cta_group::2) wherever the GEMM has 256-wide N tiles; 0: 128 x N tiles on
 * single CTAs; -1 (the default, or PTB_GEMM_PAIRS=0 / 1 in the environment
 * at first use): as 1, the faster shape on every layer measured (13B to
 * 530B class, bf16 and e4m3, forward and training).  The results agree within rounding
 * (the last wave's K split may differ).  *previous (if not null) receives
 * the old mode.  PTB_ERR_ARG for another mode.
 */
ptb_status ptb_set_gemm_pairs(int32_t mode, int32_t* previous);

/* Frees the library's own workspace arena on the current device (if any). */
ptb_status ptb_release_workspace(void);

/*
 * swa_attention: o = softmax_band(q k^T * scale) v  (SWA row, §2.2).
 *
 *   q, k, v, o  [batch, heads, seq, head_dim] bf16, contiguous
 *   head_dim    one of 16, 32, 64, 96, 128
 *   window      w >= 1; row i attends to keys max(0, i-w+1) .. i
 *   scale       softmax scale; 0 selects 1/sqrt(head_dim)
 * o must not alias q, k or v.
 */
ptb_status swa_attention(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v, int64_t batch,
                         int32_t heads, int64_t seq, int32_t head_dim, int32_t window,
                         float scale, ptb_bf16* o, ptb_stream stream);

/*
 * swa_attention_strided: the same operation on strided views.  Element
 * (b, h, i, c) of tensor t lives at t[b*sb + h*sh + i*ss + c]; strides are
 * in elements and must be multiples of 8 (16 bytes).  The PTB path uses it
 * on the column blocks of the fused projection output.  o may alias q
 * exactly (same pointer and strides): each query tile is read in full
 * before its output is written and no other tile reads it.
 */
ptb_status swa_attention_strided(const ptb_bf16* q, int64_t q_sb, int64_t q_sh, int64_t q_ss,
                                 const ptb_bf16* k, int64_t k_sb, int64_t k_sh, int64_t k_ss,
                                 const ptb_bf16* v, int64_t v_sb, int64_t v_sh, int64_t v_ss,
                                 ptb_bf16* o, int64_t o_sb, int64_t o_sh, int64_t o_ss,
                                 int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                 int32_t window, float scale, ptb_stream stream);

/*
 * swa_attention_lse: swa_attention that also writes, for every row
 * (b, h, i), lse[(b*heads + h)*seq + i] = log2(sum_j 2^(q_i.k_j * scale *
 * log2 e)) over the row's window (fp32, device memory): the softmax
 * denominator in base 2, which swa_attention_backward needs.
 *
 * swa_attention_backward: gradients of o = SWA(q, k, v) (contiguous
 * [batch, heads, seq, head_dim] bf16, as swa_attention) for the upstream
 * gradient dout, given o and lse from swa_attention_lse with the same scale:
 *   dv = P^T dout,  dP = dout v^T,  dS = P * (dP - rowsum(dout * o)),
 *   dq = scale * dS k,  dk = scale * dS^T q,
 * P recomputed from q, k and lse.  dq, dk, dv are bf16 of the same shape;
 * delta is fp32 scratch of batch*heads*seq elements.  Four launches
 * (rowsum, dK/dV over 128-key blocks, dQ over 128-query blocks), no atomics.
 * Shape and alignment rules as swa_attention.
 */
ptb_status swa_attention_lse(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                             int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                             int32_t window, float scale, ptb_bf16* o, float* lse,
                             ptb_stream stream);
ptb_status swa_attention_backward(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                                  const ptb_bf16* o, const ptb_bf16* dout, const float* lse,
                                  int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                  int32_t window, float scale, ptb_bf16* dq, ptb_bf16* dk,
                                  ptb_bf16* dv, float* delta, ptb_stream stream);

/*
 * swa_attention_counts: runs the attention kernel's own masking code and
 * writes, for every row (b, h, i), how many keys passed the band mask into
 * counts[(b*heads + h)*seq + i] (int32, device memory).  The expected value
 * is exactly min(i+1, window).  o receives the attention output as usual.
 */
ptb_status swa_attention_counts(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                                int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                int32_t window, float scale, ptb_bf16* o, int32_t* counts,
                                ptb_stream stream);

/*
 * ptb_layernorm: out[r, :] = (x[r, :] - mean) / sqrt(var + eps) * gamma + beta
 * for rows r < rows; x and out [rows, hidden] bf16 row-major; fp32
 * statistics, biased variance.  hidden a multiple of 8 and <= 32768.
 */
ptb_status ptb_layernorm(const ptb_bf16* x, const ptb_bf16* gamma, const ptb_bf16* beta,
                         int64_t rows, int64_t hidden, float eps, ptb_bf16* out,
                         ptb_stream stream);

/*
 * Scratch (bytes) with which either GEMM below can split the tiles of its
 * last, partial wave along K over the SMs that wave would leave idle: fp32
 * partial tiles plus arrival counters (the counters are cleared on the
 * stream before every launch).  Depends on the current device's SM count;
 * 0 when no split applies.
 */
size_t ptb_gemm_workspace_size(int64_t tokens, int64_t hidden, int64_t ffn);

/*
 * ptb_gemm_qkv_up: the fused first projection of the PTB,
 *   u[:, 0:3H]      = xn w_qkv^T
 *   u[:, 3H:3H+F]   = gelu_tanh(xn w_up^T)
 * xn [T, H], u [T, 3H+F] row-major bf16; H, F multiples of 64.
 * workspace: NULL, or >= ptb_gemm_workspace_size() bytes (256-byte aligned)
 * to let the last wave split along K; results are the same either way up to
 * fp32 summation order.
 */
ptb_status ptb_gemm_qkv_up(const ptb_bf16* xn, const ptb_bf16* w_qkv, const ptb_bf16* w_up,
                           int64_t tokens, int64_t hidden, int64_t ffn, ptb_bf16* u,
                           void* workspace, size_t workspace_bytes, ptb_stream stream);

/*
 * ptb_gemm_out_down: the fused output projection with the residual,
 *   y = x + ctx w_o^T + g w_down^T,
 * one GEMM over the concatenated inner dimension [ctx | g] (H + F).
 * ctx [T, H] with row stride ld_ctx, g [T, F] with row stride ld_g (strides
 * in elements, multiples of 8), x and y [T, H] contiguous.  workspace as
 * for ptb_gemm_qkv_up.
 */
ptb_status ptb_gemm_out_down(const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g, int64_t ld_g,
                             const ptb_bf16* w_o, const ptb_bf16* w_down, const ptb_bf16* x,
                             int64_t tokens, int64_t hidden, int64_t ffn, ptb_bf16* y,
                             void* workspace, size_t workspace_bytes, ptb_stream stream);

/*
 * ptb_last_device_error: waits for the work queued on `stream` so far
 * (cudaStreamSynchronize of that stream only; other streams keep running),
 * then returns the device status word written by the kernels and clears it
 * in the same atomic step: PTB_OK if no kernel gave up, PTB_ERR_TIMEOUT if a
 * bounded device-side wait expired, PTB_ERR_LAUNCH if the CUDA context
 * reports an error.  The word is per device, so it also holds a code that a
 * kernel on another stream recorded before the read.  NULL is the legacy
 * default stream, which waits for every blocking stream of the device.
 * Calls from several host threads are serialised inside the library.
 */
ptb_status ptb_last_device_error(ptb_stream stream);

/*
 * Test hook: the wait limit of the kernels' bounded waits.  ptb_wait_probe
 * launches one CTA that waits on an mbarrier nobody signals, with a limit
 * of `limit_ns`; it must come back with PTB_ERR_TIMEOUT recorded rather
 * than hang.  Returns the launch status.
 */
ptb_status ptb_wait_probe(uint64_t limit_ns, ptb_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PTB_H_ */
