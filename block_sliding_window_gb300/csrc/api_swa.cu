// C ABI of libptb, the attention operator: causal sliding-window attention
// on contiguous or strided [batch, heads, seq, head_dim] views, its per-row
// attended-key counts, its log-sum-exp, and its backward pass (MegaScale
// study notes, ch.2 §2.2, SWA row).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "api_internal.h"
#include "ptb_device.cuh"

using namespace ptb;
using namespace ptb::api;

extern "C" {

ptb_status swa_attention_strided(const ptb_bf16* q, int64_t q_sb, int64_t q_sh, int64_t q_ss,
                                 const ptb_bf16* k, int64_t k_sb, int64_t k_sh, int64_t k_ss,
                                 const ptb_bf16* v, int64_t v_sb, int64_t v_sh, int64_t v_ss,
                                 ptb_bf16* o, int64_t o_sb, int64_t o_sh, int64_t o_ss,
                                 int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                 int32_t window, float scale, ptb_stream stream) {
  if (batch > 65535 || seq > (1ll << 30)) return PTB_ERR_SHAPE;
  SwaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = bf(q);
  a.k = bf(k);
  a.v = bf(v);
  a.o = bf(o);
  a.q_sb = q_sb; a.q_sh = q_sh; a.q_ss = q_ss;
  a.k_sb = k_sb; a.k_sh = k_sh; a.k_ss = k_ss;
  a.v_sb = v_sb; a.v_sh = v_sh; a.v_ss = v_ss;
  a.o_sb = o_sb; a.o_sh = o_sh; a.o_ss = o_ss;
  a.batch = static_cast<int>(batch);
  a.heads = heads;
  a.seq = static_cast<int>(seq);
  a.head_dim = head_dim;
  a.window = window;
  return swa_impl(a, scale, static_cast<cudaStream_t>(stream));
}

static ptb_status swa_contiguous(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                                 int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                 int32_t window, float scale, ptb_bf16* o, int32_t* counts,
                                 ptb_stream stream) {
  if (batch > 65535 || seq > (1ll << 30) || head_dim < 1) return batch < 1 ? PTB_ERR_ARG
                                                                           : PTB_ERR_SHAPE;
  if (o == q || o == k || o == v) return PTB_ERR_ARG;
  SwaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = bf(q);
  a.k = bf(k);
  a.v = bf(v);
  a.o = bf(o);
  const int64_t ss = head_dim, sh = seq * head_dim, sb = heads * seq * head_dim;
  a.q_sb = a.k_sb = a.v_sb = a.o_sb = sb;
  a.q_sh = a.k_sh = a.v_sh = a.o_sh = sh;
  a.q_ss = a.k_ss = a.v_ss = a.o_ss = ss;
  a.batch = static_cast<int>(batch);
  a.heads = heads;
  a.seq = static_cast<int>(seq);
  a.head_dim = head_dim;
  a.window = window;
  a.counts = counts;
  return swa_impl(a, scale, static_cast<cudaStream_t>(stream));
}

ptb_status swa_attention(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v, int64_t batch,
                         int32_t heads, int64_t seq, int32_t head_dim, int32_t window,
                         float scale, ptb_bf16* o, ptb_stream stream) {
  return swa_contiguous(q, k, v, batch, heads, seq, head_dim, window, scale, o, nullptr, stream);
}

ptb_status swa_attention_counts(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                                int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                int32_t window, float scale, ptb_bf16* o, int32_t* counts,
                                ptb_stream stream) {
  if (!counts || !aligned(counts, 4)) return PTB_ERR_ARG;
  return swa_contiguous(q, k, v, batch, heads, seq, head_dim, window, scale, o, counts, stream);
}

ptb_status swa_attention_lse(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                             int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                             int32_t window, float scale, ptb_bf16* o, float* lse,
                             ptb_stream stream) {
  if (!lse || !aligned(lse, 4)) return PTB_ERR_ARG;
  if (batch < 1 || seq < 1 || heads < 1) return PTB_ERR_ARG;
  if (batch > 65535 || seq > (1ll << 30)) return PTB_ERR_SHAPE;
  if (o == q || o == k || o == v) return PTB_ERR_ARG;
  SwaArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = bf(q), a.k = bf(k), a.v = bf(v), a.o = bf(o);
  const int64_t ss = head_dim, sh = seq * head_dim, sb = heads * seq * head_dim;
  a.q_sb = a.k_sb = a.v_sb = a.o_sb = sb;
  a.q_sh = a.k_sh = a.v_sh = a.o_sh = sh;
  a.q_ss = a.k_ss = a.v_ss = a.o_ss = ss;
  a.batch = static_cast<int>(batch);
  a.heads = heads;
  a.seq = static_cast<int>(seq);
  a.head_dim = head_dim;
  a.window = window;
  a.lse = lse;
  return swa_impl(a, scale, static_cast<cudaStream_t>(stream));
}

ptb_status swa_attention_backward(const ptb_bf16* q, const ptb_bf16* k, const ptb_bf16* v,
                                  const ptb_bf16* o, const ptb_bf16* dout, const float* lse,
                                  int64_t batch, int32_t heads, int64_t seq, int32_t head_dim,
                                  int32_t window, float scale, ptb_bf16* dq, ptb_bf16* dk,
                                  ptb_bf16* dv, float* delta, ptb_stream stream) {
  const void* ptrs[] = {q, k, v, o, dout, dq, dk, dv};
  for (const void* p : ptrs)
    if (!p) return PTB_ERR_ARG;
  if (!lse || !delta || batch < 1 || seq < 1 || heads < 1 || window < 1) return PTB_ERR_ARG;
  if (!head_dim_ok(head_dim)) return PTB_ERR_SHAPE;
  if (batch > 65535 || seq > (1ll << 30) || batch * static_cast<int64_t>(heads) > 65535)
    return PTB_ERR_SHAPE;
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return PTB_ERR_ALIGN;
  if (!aligned(lse, 4) || !aligned(delta, 4)) return PTB_ERR_ALIGN;
  if (scale < 0.f || !std::isfinite(scale)) return PTB_ERR_ARG;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  SwaBwdArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = bf(q), a.k = bf(k), a.v = bf(v), a.o = bf(o), a.dout = bf(dout);
  a.dq = bf(dq), a.dk = bf(dk), a.dv = bf(dv);
  const int64_t ss = head_dim, sh = seq * head_dim, sb = heads * seq * head_dim;
  a.q_sb = a.k_sb = a.v_sb = a.o_sb = a.do_sb = a.dq_sb = a.dk_sb = a.dv_sb = sb;
  a.q_sh = a.k_sh = a.v_sh = a.o_sh = a.do_sh = a.dq_sh = a.dk_sh = a.dv_sh = sh;
  a.q_ss = a.k_ss = a.v_ss = a.o_ss = a.do_ss = a.dq_ss = a.dk_ss = a.dv_ss = ss;
  a.lse = lse;
  a.delta = delta;
  a.batch = static_cast<int>(batch);
  a.heads = heads;
  a.seq = static_cast<int>(seq);
  a.head_dim = head_dim;
  a.window = window;
  a.scale = scale == 0.f ? 1.0f / std::sqrt(static_cast<float>(head_dim)) : scale;
  a.scale_log2 = a.scale * 1.4426950408889634f;
  a.status = ds->status;
  a.sms = ds->sms;
  return launch_status(launch_swa_backward(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
