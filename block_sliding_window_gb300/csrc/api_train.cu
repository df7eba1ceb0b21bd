// C ABI of libptb, the training step: the forward pass that keeps its
// activations and the backward pass of y = x + Attn(LN(x)) + MLP(LN(x))
// (MegaScale study notes, ch.2 §2.2, PTB row; §2.1 counts the backward as
// 4N of the 6N training FLOPs per token).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "api_internal.h"
#include "ptb_device.cuh"

using namespace ptb;
using namespace ptb::api;

namespace {

// Saved activations of ptb_forward_train, in this order, each region
// starting on a kAlign boundary.
struct SavedLayout {
  size_t xn, stats, u, z, ctx, lse, total;
};

SavedLayout saved_layout(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int64_t heads) {
  const size_t t = static_cast<size_t>(batch) * static_cast<size_t>(seq);
  SavedLayout l;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes, kAlign);
    return at;
  };
  l.xn = take(t * hidden * 2);
  l.stats = take(t * 8);
  l.u = take(t * (3 * hidden + ffn) * 2);
  l.z = take(t * ffn * 2);
  l.ctx = take(t * hidden * 2);
  l.lse = take(static_cast<size_t>(batch) * heads * seq * 4);
  l.total = off;
  return l;
}

// The four GEMMs of the backward pass (pointers left null: for sizing).
GemmCall call_dgrad_out(int64_t t, int64_t h, int64_t f) {  // [dctx | dG] = dy [W_o | W_down]
  GemmCall c;
  c.layout = kLayoutKN;
  c.epilogue = kEpiDgelu;
  c.M = t, c.N = h + f, c.K = h, c.n_split = h;
  c.lda0 = h, c.ldb0 = h, c.ldb1 = f;
  c.out_split_col = h, c.gelu_col = h;
  return c;
}
GemmCall call_wgrad_out(int64_t t, int64_t h, int64_t f, int64_t ldu) {  // dy^T [ctx | G]
  GemmCall c;
  c.layout = kLayoutNN;
  c.epilogue = kEpiF32;
  c.M = h, c.N = h + f, c.K = t, c.n_split = h;
  c.lda0 = h, c.ldb0 = h, c.ldb1 = ldu;
  c.out_split_col = h;
  return c;
}
GemmCall call_dgrad_in(int64_t t, int64_t h, int64_t f, int64_t ldu) {  // dU1 [W_qkv ; W_up]
  GemmCall c;
  c.layout = kLayoutKN;
  c.epilogue = kEpiF32;
  c.M = t, c.N = h, c.K = ldu, c.k_split = 3 * h;
  c.lda0 = ldu, c.lda1 = ldu, c.ldb0 = h, c.ldb1 = h;
  (void)f;
  return c;
}
GemmCall call_wgrad_in(int64_t t, int64_t h, int64_t f, int64_t ldu) {  // dU1^T xn
  GemmCall c;
  c.layout = kLayoutNN;
  c.epilogue = kEpiF32;
  c.M = ldu, c.N = h, c.K = t;
  c.lda0 = ldu, c.ldb0 = h;
  c.out_split_row = 3 * h;
  (void)f;
  return c;
}

struct BwdLayout {
  size_t dctx, du1, delta, dxn, ln_part, gemm, total;
};

BwdLayout bwd_layout(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int64_t heads,
                     int sms) {
  const int64_t t = batch * seq, ldu = 3 * hidden + ffn;
  BwdLayout l;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off += round_up(bytes, kAlign);
    return at;
  };
  l.dctx = take(static_cast<size_t>(t) * hidden * 2);
  l.du1 = take(static_cast<size_t>(t) * ldu * 2);
  l.delta = take(static_cast<size_t>(batch) * heads * seq * 4);
  l.dxn = take(static_cast<size_t>(t) * hidden * 4);
  l.ln_part = take(static_cast<size_t>(ln_backward_chunks(t)) * 2 * hidden * 4);
  size_t g = 0;
  for (const GemmCall& c : {call_dgrad_out(t, hidden, ffn), call_wgrad_out(t, hidden, ffn, ldu),
                            call_dgrad_in(t, hidden, ffn, ldu), call_wgrad_in(t, hidden, ffn, ldu)}) {
    const size_t b = call_scratch(c, sms);
    g = b > g ? b : g;
  }
  l.gemm = take(g);
  l.total = off;
  return l;
}

ptb_status check_saved(const void* saved, size_t saved_bytes, const SavedLayout& l) {
  if (!saved) return PTB_ERR_ARG;
  if (!aligned(saved, kAlign)) return PTB_ERR_ALIGN;
  if (saved_bytes < l.total) return PTB_ERR_WORKSPACE;
  return PTB_OK;
}

SwaBwdArgs swa_bwd_args(DeviceState* ds, const ptb_bf16* u, const ptb_bf16* ctx,
                        const ptb_bf16* dctx, ptb_bf16* du1, const float* lse, float* delta,
                        int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                        int32_t window) {
  const int64_t d = hidden / heads, ldu = 3 * hidden + ffn;
  SwaBwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = bf(u);
  a.k = bf(u) + hidden;
  a.v = bf(u) + 2 * hidden;
  a.o = bf(ctx);
  a.dout = bf(dctx);
  a.dq = bf(du1);
  a.dk = bf(du1) + hidden;
  a.dv = bf(du1) + 2 * hidden;
  a.q_sb = a.k_sb = a.v_sb = a.dq_sb = a.dk_sb = a.dv_sb = seq * ldu;
  a.q_sh = a.k_sh = a.v_sh = a.dq_sh = a.dk_sh = a.dv_sh = d;
  a.q_ss = a.k_ss = a.v_ss = a.dq_ss = a.dk_ss = a.dv_ss = ldu;
  a.o_sb = a.do_sb = seq * hidden;
  a.o_sh = a.do_sh = d;
  a.o_ss = a.do_ss = hidden;
  a.lse = lse;
  a.delta = delta;
  a.batch = static_cast<int>(batch);
  a.heads = heads;
  a.seq = static_cast<int>(seq);
  a.head_dim = static_cast<int>(d);
  a.window = window;
  a.scale = 1.0f / std::sqrt(static_cast<float>(d));
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.status = ds->status;
  a.sms = ds->sms;
  return a;
}

}  // namespace

extern "C" {

size_t ptb_train_saved_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                            int32_t heads) {
  if (batch < 1 || seq < 1 || hidden < 1 || ffn < 1 || heads < 1) return 0;
  return saved_layout(batch, seq, hidden, ffn, heads).total;
}

ptb_status ptb_forward_train(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                             const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                             const ptb_bf16* w_down, int64_t batch, int64_t seq, int64_t hidden,
                             int64_t ffn, int32_t heads, int32_t window, ptb_bf16* y, void* saved,
                             size_t saved_bytes, void* workspace, size_t workspace_bytes,
                             ptb_stream stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, y};
  ptb_status st = check_layer(ptrs, 8, batch, seq, hidden, ffn, heads, window);
  if (st != PTB_OK) return st;
  const SavedLayout l = saved_layout(batch, seq, hidden, ffn, heads);
  st = check_saved(saved, saved_bytes, l);
  if (st != PTB_OK) return st;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;
  const int64_t tokens = batch * seq, ldu = 3 * hidden + ffn;
  const size_t need = layer_gemm_scratch(tokens, hidden, ffn, ds->sms);
  st = acquire_workspace(ds, need, workspace, workspace_bytes, &workspace);
  if (st != PTB_OK) return st;
  char* sv = static_cast<char*>(saved);
  ptb_bf16* xn = reinterpret_cast<ptb_bf16*>(sv + l.xn);
  float2* stats = reinterpret_cast<float2*>(sv + l.stats);
  ptb_bf16* u = reinterpret_cast<ptb_bf16*>(sv + l.u);
  ptb_bf16* z = reinterpret_cast<ptb_bf16*>(sv + l.z);
  ptb_bf16* ctx = reinterpret_cast<ptb_bf16*>(sv + l.ctx);
  float* lse = reinterpret_cast<float*>(sv + l.lse);
  // 1. xn = LN(x), keeping (mean, rstd) per token
  if (launch_layernorm(bf(x), bf(ln_gamma), bf(ln_beta), tokens, static_cast<int>(hidden), 1e-5f,
                       bf(xn), stream, stats) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 2. U = [xn W_qkv^T | gelu(Z)], Z = xn W_up^T kept
  st = gemm_run(ds, spec_qkv_up(xn, w_qkv, w_up, hidden, ffn), tokens, u, ldu, nullptr, 0,
                3 * hidden, workspace, need, stream, z, ffn);
  if (st != PTB_OK) return st;
  // 3. ctx = SWA(Q, K, V) into its own buffer (Q is needed again), with the
  //    per-row log-sum-exp
  SwaArgs sa = swa_over_u(ds, u, ldu, batch, seq, hidden, heads, window);
  sa.o = bf(ctx);
  sa.o_sb = seq * hidden;
  sa.o_ss = hidden;
  sa.lse = lse;
  if (launch_swa(sa, stream) != cudaSuccess) return PTB_ERR_LAUNCH;
  // 4. y = x + [ctx | G] [W_o | W_down]^T
  return gemm_out_down(ds, ctx, hidden, u + 3 * hidden, ldu, w_o, w_down, x, tokens, hidden, ffn,
                       y, workspace, need, stream);
}

size_t ptb_backward_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                                   int32_t heads) {
  if (batch < 1 || seq < 1 || hidden < 64 || ffn < 64 || heads < 1) return 0;
  if (hidden % 64 || ffn % 64) return 0;
  return bwd_layout(batch, seq, hidden, ffn, heads, current_sms()).total;
}

ptb_status ptb_backward_events(const ptb_bf16* dy, const ptb_bf16* x, const ptb_bf16* ln_gamma,
                               const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                               const ptb_bf16* w_down, const void* saved, size_t saved_bytes,
                               int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                               int32_t heads, int32_t window, ptb_bf16* dx, float* dln_gamma,
                               float* dln_beta, float* dw_qkv, float* dw_o, float* dw_up,
                               float* dw_down, void* workspace, size_t workspace_bytes,
                               ptb_stream stream_, void* const* events, int32_t n_events) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, dx,
                        dln_gamma, dln_beta, dw_qkv, dw_o, dw_up, dw_down};
  ptb_status st = check_layer(ptrs, 14, batch, seq, hidden, ffn, heads, window);
  if (st != PTB_OK) return st;
  if (events && n_events != 7) return PTB_ERR_ARG;
  if (events)
    for (int i = 0; i < 7; ++i)
      if (!events[i]) return PTB_ERR_ARG;
  auto mark = [&](int i) -> bool {
    if (!events) return true;
    if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess) return true;
    cudaGetLastError();  // the failed record must not be reported by a later launch
    return false;
  };
  const SavedLayout l = saved_layout(batch, seq, hidden, ffn, heads);
  st = check_saved(saved, saved_bytes, l);
  if (st != PTB_OK) return st;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;
  const BwdLayout w = bwd_layout(batch, seq, hidden, ffn, heads, ds->sms);
  st = acquire_workspace(ds, w.total, workspace, workspace_bytes, &workspace);
  if (st != PTB_OK) return st;
  const int64_t t = batch * seq, ldu = 3 * hidden + ffn;
  const char* sv = static_cast<const char*>(saved);
  const ptb_bf16* xn = reinterpret_cast<const ptb_bf16*>(sv + l.xn);
  const float2* stats = reinterpret_cast<const float2*>(sv + l.stats);
  const ptb_bf16* u = reinterpret_cast<const ptb_bf16*>(sv + l.u);
  const ptb_bf16* z = reinterpret_cast<const ptb_bf16*>(sv + l.z);
  const ptb_bf16* ctx = reinterpret_cast<const ptb_bf16*>(sv + l.ctx);
  const float* lse = reinterpret_cast<const float*>(sv + l.lse);
  char* ws = static_cast<char*>(workspace);
  ptb_bf16* dctx = reinterpret_cast<ptb_bf16*>(ws + w.dctx);
  ptb_bf16* du1 = reinterpret_cast<ptb_bf16*>(ws + w.du1);
  float* delta = reinterpret_cast<float*>(ws + w.delta);
  float* dxn = reinterpret_cast<float*>(ws + w.dxn);
  float* ln_part = reinterpret_cast<float*>(ws + w.ln_part);
  void* scratch = ws + w.gemm;
  const size_t scratch_bytes = w.total - w.gemm;

  // 1. [dctx | dZ] = dy [W_o | W_down], dZ = dG * gelu'(Z) written into dU1
  if (!mark(0)) return PTB_ERR_ARG;
  GemmCall c = call_dgrad_out(t, hidden, ffn);
  c.a0 = dy, c.b0 = w_o, c.b1 = w_down;
  c.out = dctx, c.ld_out = hidden, c.out1 = du1 + 3 * hidden, c.ld_out1 = ldu;
  c.aux = const_cast<ptb_bf16*>(z), c.ld_aux = ffn;
  st = gemm_call(ds, c, scratch, scratch_bytes, stream);
  if (st != PTB_OK) return st;
  // 2. [dW_o | dW_down] = dy^T [ctx | G]
  if (!mark(1)) return PTB_ERR_ARG;
  c = call_wgrad_out(t, hidden, ffn, ldu);
  c.a0 = dy, c.b0 = ctx, c.b1 = u + 3 * hidden;
  c.out = dw_o, c.ld_out = hidden, c.out1 = dw_down, c.ld_out1 = ffn;
  st = gemm_call(ds, c, scratch, scratch_bytes, stream);
  if (st != PTB_OK) return st;
  // 3. [dQ | dK | dV] into dU1 from the banded attention backward
  if (!mark(2)) return PTB_ERR_ARG;
  if (launch_swa_backward(swa_bwd_args(ds, u, ctx, dctx, du1, lse, delta, batch, seq, hidden, ffn,
                                       heads, window),
                          stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 4. dxn = dU1 [W_qkv ; W_up]   (fp32)
  if (!mark(3)) return PTB_ERR_ARG;
  c = call_dgrad_in(t, hidden, ffn, ldu);
  c.a0 = du1, c.a1 = du1 + 3 * hidden, c.b0 = w_qkv, c.b1 = w_up;
  c.out = dxn, c.ld_out = hidden;
  st = gemm_call(ds, c, scratch, scratch_bytes, stream);
  if (st != PTB_OK) return st;
  // 5. [dW_qkv ; dW_up] = dU1^T xn
  if (!mark(4)) return PTB_ERR_ARG;
  c = call_wgrad_in(t, hidden, ffn, ldu);
  c.a0 = du1, c.b0 = xn;
  c.out = dw_qkv, c.ld_out = hidden, c.out1 = dw_up, c.ld_out1 = hidden;
  st = gemm_call(ds, c, scratch, scratch_bytes, stream);
  if (st != PTB_OK) return st;
  // 6. dx = dy + LN backward of dxn; dgamma, dbeta
  if (!mark(5)) return PTB_ERR_ARG;
  st = launch_status(launch_layernorm_backward(bf(x), bf(ln_gamma), stats, dxn, bf(dy), t,
                                               static_cast<int>(hidden), bf(dx), dln_gamma,
                                               dln_beta, ln_part, stream));
  if (st != PTB_OK) return st;
  if (!mark(6)) return PTB_ERR_ARG;
  return PTB_OK;
}

ptb_status ptb_backward(const ptb_bf16* dy, const ptb_bf16* x, const ptb_bf16* ln_gamma,
                        const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                        const ptb_bf16* w_down, const void* saved, size_t saved_bytes,
                        int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                        int32_t window, ptb_bf16* dx, float* dln_gamma, float* dln_beta,
                        float* dw_qkv, float* dw_o, float* dw_up, float* dw_down, void* workspace,
                        size_t workspace_bytes, ptb_stream stream) {
  return ptb_backward_events(dy, x, ln_gamma, w_qkv, w_o, w_up, w_down, saved, saved_bytes, batch,
                             seq, hidden, ffn, heads, window, dx, dln_gamma, dln_beta, dw_qkv,
                             dw_o, dw_up, dw_down, workspace, workspace_bytes, stream, nullptr, 0);
}

}  // extern "C"
