// Internal interface shared by the translation units of the C ABI
// (ptb_api.cu: common part and forward pass; api_swa.cu: the attention
// operator; api_fp8.cu: the FP8 variant; api_train.cu: the training step):
// device state, workspace handling, argument checks and the GEMM launch
// plumbing.  Not part of the public interface.
#pragma once

#include <cstdint>
#include <cstring>

#include "ptb_internal.h"

namespace ptb {
namespace api {

constexpr size_t kAlign = 256;  // alignment of every workspace region

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline const __nv_bfloat16* bf(const ptb_bf16* p) {
  return reinterpret_cast<const __nv_bfloat16*>(p);
}
inline __nv_bfloat16* bf(ptb_bf16* p) { return reinterpret_cast<__nv_bfloat16*>(p); }
inline bool head_dim_ok(int64_t d) { return d == 16 || d == 32 || d == 64 || d == 96 || d == 128; }

// Per-device state of the library.
struct DeviceState {
  bool ready = false;
  int sms = 0;
  // 256 x 256 CTA-pair GEMM tiles: -1 automatic, 0 never, 1 wherever they
  // apply (environment variable PTB_GEMM_PAIRS=0 / 1 overrides the default).
  int pairs = -1;
  unsigned* status = nullptr;
  // Device word that ptb_last_device_error swaps the status word into.
  unsigned* status_taken = nullptr;
  void* arena = nullptr;
  size_t arena_bytes = 0;
  // Recorded after the layer of the latest ptb_forward_host call, so that
  // the next call's layer (possibly on another stream) runs after it.
  cudaEvent_t host_layer_done = nullptr;
};

// Per-device set-up on first use (SM count, status word, architecture check,
// the driver's tensor-map encoder); PTB_OK and *out filled.
ptb_status device_state(DeviceState** out);
// SM count of the current device, or an upper bound when there is none.
int current_sms();
ptb_status launch_status(cudaError_t e);
int pick_block_n(int64_t a, int64_t b);

// One GEMM of the layer: C[M, N] = A[M, K] B[N, K]^T with
//   A = [a0 | a1] split along K at k0 (k1 == 0: a0 only), and
//   B = [b0 ; b1] split along N at n0 (n1 == 0: b0 only)
// -- at most one split at a time.  In a K split b0 is [N, k0] and b1 is
// [N, k1]; in an N split a0 is [M, K] and b0, b1 are [n0, K], [n1, K].
struct GemmSpec {
  const ptb_bf16 *a0, *a1, *b0, *b1;
  int64_t lda0, lda1, k0, k1, n0, n1;
  // e4m3 operands (a0, b0 then point at bytes): one scale per A row and per B row.
  bool fp8 = false;
  const float* a_scale = nullptr;
  const float* b_scale = nullptr;
  int64_t n() const { return n0 + n1; }
  int64_t k() const { return k0 + k1; }
  int64_t kb() const { return k() / (fp8 ? 128 : 64); }
  int block_n() const { return n1 ? pick_block_n(n0, n1) : pick_block_n(n0, n0); }
};

GemmSpec spec_fp8(const void* a, int64_t lda, int64_t k, const void* b, int64_t n,
                  const float* a_scale, const float* b_scale);
GemmSpec spec_plain(const ptb_bf16* a, int64_t lda, int64_t k, const ptb_bf16* b, int64_t n);
// [QKV | up] of the PTB: U = [xn W_qkv^T | gelu(xn W_up^T)].
GemmSpec spec_qkv_up(const ptb_bf16* xn, const ptb_bf16* w_qkv, const ptb_bf16* w_up,
                     int64_t hidden, int64_t ffn);
// [out | down] of the PTB: [ctx | G] [W_o | W_down]^T.
GemmSpec spec_out_down(const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g, int64_t ld_g,
                       const ptb_bf16* w_o, const ptb_bf16* w_down, int64_t hidden, int64_t ffn);

// One forward GEMM: out[tokens, N] from spec g, with the residual (resid not
// null) or the GELU epilogue from column gelu_col (optionally also storing
// the pre-activation to aux); `training` selects the training-step rule for
// CTA-pair tiles.
ptb_status gemm_run(DeviceState* ds, const GemmSpec& g, int64_t tokens, ptb_bf16* out, int64_t ldo,
                    const ptb_bf16* resid, int64_t ldr, int64_t gelu_col, void* scratch,
                    size_t scratch_bytes, cudaStream_t stream, ptb_bf16* aux = nullptr,
                    int64_t ld_aux = 0);
ptb_status gemm_qkv_up(DeviceState* ds, const ptb_bf16* xn, const ptb_bf16* w_qkv,
                       const ptb_bf16* w_up, int64_t tokens, int64_t hidden, int64_t ffn,
                       ptb_bf16* u, void* scratch, size_t scratch_bytes, cudaStream_t stream);
ptb_status gemm_out_down(DeviceState* ds, const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g,
                         int64_t ld_g, const ptb_bf16* w_o, const ptb_bf16* w_down,
                         const ptb_bf16* x, int64_t tokens, int64_t hidden, int64_t ffn,
                         ptb_bf16* y, void* scratch, size_t scratch_bytes, cudaStream_t stream);

// A GEMM of the backward pass, C[M, N] = A[M, K] B[N, K]^T, with operands
// read in place from row-major matrices:
//   A K-major:  a_i stored [M, K_i] (row stride lda_i);  A MN-major: [K_i, M].
//   B K-major:  b_i stored [N_i, K] or [N, K_i];  B MN-major: [K, N_i] or [K_i, N].
// A and B may be split in two along K at k_split (a0/b0 before, a1/b1
// after), or B along N at n_split; at most one split (0 = none).
struct GemmCall {
  int layout = kLayoutKK;
  int epilogue = kEpiF32;
  int64_t M = 0, N = 0, K = 0;
  const ptb_bf16 *a0 = nullptr, *a1 = nullptr, *b0 = nullptr, *b1 = nullptr;
  int64_t lda0 = 0, lda1 = 0, ldb0 = 0, ldb1 = 0;
  int64_t k_split = 0, n_split = 0;
  void* out = nullptr;
  int64_t ld_out = 0;
  void* out1 = nullptr;
  int64_t ld_out1 = 0;
  int64_t out_split_col = 0, out_split_row = 0;  // 0 = no split
  ptb_bf16* aux = nullptr;
  int64_t ld_aux = 0;
  int64_t gelu_col = 0;
  int block_n() const {
    return n_split ? pick_block_n(n_split, N - n_split) : pick_block_n(N, N);
  }
  int64_t kb() const { return (K + 63) / 64; }
};

// Split-wave scratch of a backward GEMM (either tile shape), and its launch.
size_t call_scratch(const GemmCall& c, int sms);
ptb_status gemm_call(DeviceState* ds, const GemmCall& c, void* scratch, size_t scratch_bytes,
                     cudaStream_t stream);

// Split-wave scratch of the layer's GEMMs (the largest of them).
size_t layer_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms);
size_t serial_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms);
size_t fp8_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms);

// Argument checks shared by the layer entry points (before any device use).
ptb_status check_layer(const void* const* ptrs, int nptrs, int64_t batch, int64_t seq,
                       int64_t hidden, int64_t ffn, int32_t heads, int32_t window);
// The caller's workspace if given (checked), else the library arena grown to `need`.
ptb_status acquire_workspace(DeviceState* ds, size_t need, void* workspace, size_t bytes,
                             void** out);
// The attention launch over the Q, K, V column blocks of U (ctx over Q).
SwaArgs swa_over_u(DeviceState* ds, ptb_bf16* u, int64_t ldu, int64_t batch, int64_t seq,
                   int64_t hidden, int32_t heads, int32_t window);
// Checked launch of the attention operator (scale 0: 1/sqrt(head_dim)).
ptb_status swa_impl(const SwaArgs& in, float scale, cudaStream_t stream);

}  // namespace api
}  // namespace ptb
