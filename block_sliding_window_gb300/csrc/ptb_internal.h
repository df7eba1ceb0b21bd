// Internal declarations shared by the translation units of libptb.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda_bf16.h>

#include "ptb.h"

namespace ptb {

// Epilogue of the tcgen05 GEMM.
enum GemmEpilogue : int {
  kEpiQkvGelu = 0,   // store bf16(acc); columns >= gelu_col store bf16(gelu_tanh(acc)) (and,
                     // with aux set, the pre-activation bf16(acc) at aux[row, col - gelu_col])
  kEpiResidual = 1,  // store bf16(acc + resid)
  kEpiDgelu = 2,     // columns >= gelu_col store bf16(acc * gelu_tanh'(aux[row, col - gelu_col])),
                     // the others bf16(acc)
  kEpiF32 = 3,       // store fp32 acc
};

// Operand layouts in shared memory (bit 0: A, bit 1: B).  K-major: the
// stored matrix is [M or N rows][K]; MN-major: it is [K rows][M or N], so the
// GEMM reads its transpose without a copy.
enum GemmLayout : int {
  kLayoutKK = 0,  // A K-major, B K-major
  kLayoutKN = 2,  // A K-major, B MN-major
  kLayoutNN = 3,  // A MN-major, B MN-major
};

// One GEMM launch: C[M, N] = A[M, K] * B[N, K]^T with A and B split into two
// tensor maps each.  Columns n < n_split read B from map b0 (index n), the
// rest from b1 (index n - n_split); inner indices k < k_split read A and B
// from a0/b0 (index k), the rest from a1/b1 (index k - k_split).  At most
// one of the two splits is active.  Maps of K-major operands are over
// [rows, K] (box 64 x 128 or 64 x block_n), maps of MN-major operands over
// [K, M or N] (box 64 x 64).
struct GemmArgs {
  CUtensorMap a0, a1, b0, b1;
  int M, N, K;
  int n_split, k_split;
  int block_n;  // 64, 128 or 256
  int layout;   // GemmLayout
  int n_fastest;  // tile order: 0 = M index fastest, 1 = N index fastest
  int a_keep, b_keep;  // L2 priority of the operand's loads: 1 evict_last, 0 evict_first
  int pair;  // 1: 256 x 256 tiles on CTA pairs (grid = 2 x pairs); bf16, K-major, block_n 256
  // Output: element (row, col) goes to out[row, col] (row stride ld_out),
  // except that columns >= out_split_col go to out1[row, col - out_split_col]
  // and rows >= out_split_row to out1[row - out_split_row, col] (row stride
  // ld_out1).  bf16 elements, fp32 for kEpiF32.
  void* out;
  int64_t ld_out;
  void* out1;
  int64_t ld_out1;
  int out_split_col, out_split_row;
  const __nv_bfloat16* resid;
  int64_t ld_resid;
  __nv_bfloat16* aux;  // kEpiQkvGelu: optional pre-activation out; kEpiDgelu: pre-activation in
  int64_t ld_aux;
  int gelu_col;
  int epilogue;
  int grid;  // persistent CTAs (<= number of SMs)
  unsigned* status;
  // K split of the last, partial wave (split_s < 2: no split).
  int split_r;          // remainder tiles that are split
  int split_s;          // pieces per remainder tile
  float* partials;      // [split_r * split_s][128][block_n] fp32
  unsigned* counters;   // [split_r][4] arrival counters, zeroed before each launch
  // e4m3 operands (fp8 != 0): K counted in e4m3 elements, 128 per k-block;
  // a_scale [M] and b_scale [N] dequantize the fp32 accumulator.
  int fp8;
  const float* a_scale;
  const float* b_scale;
};

// Each K piece of a split tile keeps at least this many 64-wide k-blocks.
constexpr int kMinSplitKBlocks = 8;

struct GemmPlan {
  int grid, split_r, split_s;
  size_t partial_bytes, counter_bytes;
};

// Grid and K split for `tiles` output tiles of `num_kb` k-blocks on `sms`
// SMs: whole waves of tiles, then the remainder tiles split along K over the
// SMs the last wave would leave idle.
// `workers` is the number of CTAs (or CTA pairs), `rows` the tile height
// (128, or 256 for pairs).
GemmPlan plan_gemm(int64_t tiles, int64_t num_kb, int workers, int block_n, int rows = 128);

struct SwaArgs {
  const __nv_bfloat16 *q, *k, *v;
  __nv_bfloat16* o;
  int64_t q_sb, q_sh, q_ss, k_sb, k_sh, k_ss, v_sb, v_sh, v_ss, o_sb, o_sh, o_ss;
  int batch, heads, seq, head_dim, window;
  float scale_log2;  // softmax scale * log2(e)
  int* counts;       // optional per-row attended-key counts
  float* lse;        // optional [batch][heads][seq]: log2 of row i's softmax denominator in
                     // base-2 units, log2(sum_j 2^(q_i.k_j * scale * log2 e))
  unsigned* status;  // device status word (bounded waits record timeouts here)
  int sms;           // SMs of the device (persistent grid size)
};

// Backward of causal SWA over strided [batch][heads][seq][head_dim] bf16 views
// (element (b, h, i, c) at base + b*sb + h*sh + i*ss + c).
struct SwaBwdArgs {
  const __nv_bfloat16 *q, *k, *v, *o, *dout;
  __nv_bfloat16 *dq, *dk, *dv;
  int64_t q_sb, q_sh, q_ss, k_sb, k_sh, k_ss, v_sb, v_sh, v_ss, o_sb, o_sh, o_ss;
  int64_t do_sb, do_sh, do_ss, dq_sb, dq_sh, dq_ss, dk_sb, dk_sh, dk_ss, dv_sb, dv_sh, dv_ss;
  const float* lse;  // [batch][heads][seq], as SwaArgs::lse of the forward pass
  float* delta;      // [batch][heads][seq] scratch: sum_c dO * o per row
  int batch, heads, seq, head_dim, window;
  float scale, scale_log2;  // softmax scale, and scale * log2(e)
  unsigned* status;
  int sms;
};

// Encodes a bf16 tiled tensor map with 128-byte swizzle (rank <= 5; dims and
// strides innermost first, strides in bytes for dims 1..rank-1).  Needs the
// driver entry point, which the per-device set-up of the C ABI loads.
bool make_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box);

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);
cudaError_t launch_layernorm(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                             const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                             __nv_bfloat16* out, cudaStream_t stream, float2* stats = nullptr);
// Backward of the LayerNorm plus the residual path of the block:
//   dx = dy + r * (g - mean(g) - xh * mean(g * xh)),  g = dxn * gamma,
//   xh = (x - mean) * r, with (mean, r) from the forward pass's stats;
//   dgamma = sum over rows of dxn * xh,  dbeta = sum over rows of dxn.
// `partials` holds 2 * hidden * ln_backward_chunks(rows) floats.
int64_t ln_backward_chunks(int64_t rows);
cudaError_t launch_layernorm_backward(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                      const float2* stats, const float* dxn,
                                      const __nv_bfloat16* dy, int64_t rows, int hidden,
                                      __nv_bfloat16* dx, float* dgamma, float* dbeta,
                                      float* partials, cudaStream_t stream);
cudaError_t launch_swa_backward(const SwaBwdArgs& a, cudaStream_t stream);
cudaError_t launch_swa(const SwaArgs& a, cudaStream_t stream);
cudaError_t launch_layernorm_fp8(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                 const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                                 uint8_t* out, float* scale, cudaStream_t stream);
cudaError_t launch_quantize_rows(const __nv_bfloat16* src0, int64_t ld0, int n0,
                                 const __nv_bfloat16* src1, int64_t ld1, int n1, int64_t rows,
                                 int64_t row0, uint8_t* out, float* scale, cudaStream_t stream);
cudaError_t launch_wait_probe(uint64_t limit_ns, unsigned* status, cudaStream_t stream);

}  // namespace ptb
