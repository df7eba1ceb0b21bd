// C ABI of libptb, the FP8 variant of the layer: e4m3 GEMM operands with
// per-row dynamic scales (the Megatron-LM page lists FP8 among the
// supported precisions, with dynamic scaling).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>

#include "api_internal.h"
#include "ptb_device.cuh"

using namespace ptb;
using namespace ptb::api;

extern "C" {

size_t ptb_forward_fp8_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn) {
  if (batch < 1 || seq < 1 || hidden < 1 || ffn < 1) return 0;
  const size_t t = static_cast<size_t>(batch) * static_cast<size_t>(seq);
  size_t gemm = 0;
  if (hidden % 64 == 0 && ffn % 64 == 0)
    gemm = fp8_gemm_scratch(static_cast<int64_t>(t), hidden, ffn, current_sms());
  return round_up(t * hidden, kAlign) + round_up(t * 4, kAlign) +
         round_up(t * (3 * hidden + ffn) * 2, kAlign) + round_up(t * (hidden + ffn), kAlign) +
         round_up(t * 4, kAlign) + gemm;
}

ptb_status ptb_prepare_fp8_weights(const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                                   const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t hidden,
                                   int64_t ffn, uint8_t* w1, float* s1, uint8_t* w2, float* s2,
                                   ptb_stream stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {w_qkv, w_o, w_up, w_down, w1, s1, w2, s2};
  for (const void* p : ptrs)
    if (!p) return PTB_ERR_ARG;
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return PTB_ERR_ALIGN;
  if (hidden < 128 || ffn < 128) return PTB_ERR_ARG;
  if (hidden % 128 || ffn % 128) return PTB_ERR_SHAPE;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  const int h = static_cast<int>(hidden), f = static_cast<int>(ffn);
  // w1 = [W_qkv ; W_up] row by row, w2 = [W_o | W_down] (rows concatenated along K).
  if (launch_quantize_rows(bf(w_qkv), hidden, h, nullptr, 0, 0, 3 * hidden, 0, w1, s1, stream) !=
          cudaSuccess ||
      launch_quantize_rows(bf(w_up), hidden, h, nullptr, 0, 0, ffn, 3 * hidden, w1, s1, stream) !=
          cudaSuccess ||
      launch_quantize_rows(bf(w_o), hidden, h, bf(w_down), ffn, f, hidden, 0, w2, s2, stream) !=
          cudaSuccess)
    return PTB_ERR_LAUNCH;
  return PTB_OK;
}

ptb_status ptb_forward_fp8_events(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                                  const ptb_bf16* ln_beta, const uint8_t* w1, const float* s1,
                                  const uint8_t* w2, const float* s2, int64_t batch, int64_t seq,
                                  int64_t hidden, int64_t ffn, int32_t heads, int32_t window,
                                  ptb_bf16* y, void* workspace, size_t workspace_bytes,
                                  ptb_stream stream_, void* const* events, int32_t n_events) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {x, ln_gamma, ln_beta, w1, s1, w2, s2, y};
  ptb_status st = check_layer(ptrs, 8, batch, seq, hidden, ffn, heads, window);
  if (st != PTB_OK) return st;
  // e4m3 k-blocks are 128 elements.
  if (hidden % 128 || ffn % 128) return PTB_ERR_SHAPE;
  if (events && n_events != 6) return PTB_ERR_ARG;
  if (events)
    for (int i = 0; i < 6; ++i)
      if (!events[i]) return PTB_ERR_ARG;
  auto mark = [&](int i) -> bool {
    if (!events) return true;
    if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess) return true;
    cudaGetLastError();  // the failed record must not be reported by a later launch
    return false;
  };
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;
  const int64_t tokens = batch * seq;
  const size_t need = ptb_forward_fp8_workspace_size(batch, seq, hidden, ffn);
  st = acquire_workspace(ds, need, workspace, workspace_bytes, &workspace);
  if (st != PTB_OK) return st;
  char* p = static_cast<char*>(workspace);
  uint8_t* xn8 = reinterpret_cast<uint8_t*>(p);
  p += round_up(tokens * hidden, kAlign);
  float* sx = reinterpret_cast<float*>(p);
  p += round_up(tokens * 4, kAlign);
  ptb_bf16* u = reinterpret_cast<ptb_bf16*>(p);
  p += round_up(tokens * (3 * hidden + ffn) * 2, kAlign);
  uint8_t* a8 = reinterpret_cast<uint8_t*>(p);
  p += round_up(tokens * (hidden + ffn), kAlign);
  float* sa = reinterpret_cast<float*>(p);
  p += round_up(tokens * 4, kAlign);
  const size_t scratch_size = need - static_cast<size_t>(p - static_cast<char*>(workspace));
  const int64_t ldu = 3 * hidden + ffn;

  // 1. xn8, sx = quantize(LN(x)) per token
  if (!mark(0)) return PTB_ERR_ARG;
  if (launch_layernorm_fp8(bf(x), bf(ln_gamma), bf(ln_beta), tokens, static_cast<int>(hidden),
                           1e-5f, xn8, sx, stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 2. U = [xn W_qkv^T | gelu(xn W_up^T)] from e4m3 operands
  if (!mark(1)) return PTB_ERR_ARG;
  st = gemm_run(ds, spec_fp8(xn8, hidden, hidden, w1, ldu, sx, s1), tokens, u, ldu, nullptr, 0,
                3 * hidden, p, scratch_size, stream);
  if (st != PTB_OK) return st;
  // 3. ctx = SWA(Q, K, V) over Q (bf16, as in ptb_forward)
  if (!mark(2)) return PTB_ERR_ARG;
  if (launch_swa(swa_over_u(ds, u, ldu, batch, seq, hidden, heads, window), stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 4. a8, sa = quantize([ctx | G]) per token
  if (!mark(3)) return PTB_ERR_ARG;
  if (launch_quantize_rows(bf(u), ldu, static_cast<int>(hidden), bf(u) + 3 * hidden, ldu,
                           static_cast<int>(ffn), tokens, 0, a8, sa, stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 5. y = x + [ctx | G] [W_o | W_down]^T from e4m3 operands
  if (!mark(4)) return PTB_ERR_ARG;
  st = gemm_run(ds, spec_fp8(a8, hidden + ffn, hidden + ffn, w2, hidden, sa, s2), tokens, y,
                hidden, x, hidden, hidden, p, scratch_size, stream);
  if (st != PTB_OK) return st;
  if (!mark(5)) return PTB_ERR_ARG;
  return PTB_OK;
}

ptb_status ptb_forward_fp8(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                           const uint8_t* w1, const float* s1, const uint8_t* w2, const float* s2,
                           int64_t batch, int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                           int32_t window, ptb_bf16* y, void* workspace, size_t workspace_bytes,
                           ptb_stream stream) {
  return ptb_forward_fp8_events(x, ln_gamma, ln_beta, w1, s1, w2, s2, batch, seq, hidden, ffn,
                                heads, window, y, workspace, workspace_bytes, stream, nullptr, 0);
}

}  // extern "C"
