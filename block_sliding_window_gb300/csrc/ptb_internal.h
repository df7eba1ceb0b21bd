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
  kEpiQkvGelu = 0,   // store bf16(acc); columns >= gelu_col store bf16(gelu_tanh(acc))
  kEpiResidual = 1,  // store bf16(acc + resid)
};

// One GEMM launch: C[M, N] = A[M, K] * B[N, K]^T with A and B split into two
// tensor maps each.  Columns n < n_split read B rows from map b0 (row n),
// the rest from b1 (row n - n_split); inner indices k < k_split read A and B
// from a0/b0 (column k), the rest from a1/b1 (column k - k_split).  At most
// one of the two splits is active.
struct GemmArgs {
  CUtensorMap a0, a1, b0, b1;
  int M, N, K;
  int n_split, k_split;
  int block_n;  // 64, 128 or 256
  __nv_bfloat16* out;
  int64_t ld_out;
  const __nv_bfloat16* resid;
  int64_t ld_resid;
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
// Largest bf16 row (bytes) the e4m3 row quantizer stages in shared memory:
// the 227 KB opt-in block limit less room for its static reduction array.
constexpr int64_t kQuantizeRowMaxBytes = 226 * 1024;

struct GemmPlan {
  int grid, split_r, split_s;
  size_t partial_bytes, counter_bytes;
};

// Grid and K split for `tiles` output tiles of `num_kb` k-blocks on `sms`
// SMs: whole waves of tiles, then the remainder tiles split along K over the
// SMs the last wave would leave idle.
GemmPlan plan_gemm(int64_t tiles, int64_t num_kb, int sms, int block_n);

struct SwaArgs {
  const __nv_bfloat16 *q, *k, *v;
  __nv_bfloat16* o;
  int64_t q_sb, q_sh, q_ss, k_sb, k_sh, k_ss, v_sb, v_sh, v_ss, o_sb, o_sh, o_ss;
  int batch, heads, seq, head_dim, window;
  float scale_log2;  // softmax scale * log2(e)
  int* counts;       // optional per-row attended-key counts
  unsigned* status;  // device status word (bounded waits record timeouts here)
  int sms;           // SMs of the device (persistent grid size)
};

// Encodes a bf16 tiled tensor map with 128-byte swizzle (rank <= 5; dims and
// strides innermost first, strides in bytes for dims 1..rank-1).  Needs the
// driver entry point, which the per-device set-up of the C ABI loads.
bool make_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box);

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);
cudaError_t launch_layernorm(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                             const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                             __nv_bfloat16* out, cudaStream_t stream);
cudaError_t launch_swa(const SwaArgs& a, cudaStream_t stream);
cudaError_t launch_layernorm_fp8(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                 const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                                 uint8_t* out, float* scale, cudaStream_t stream);
cudaError_t launch_quantize_rows(const __nv_bfloat16* src0, int64_t ld0, int n0,
                                 const __nv_bfloat16* src1, int64_t ld1, int n1, int64_t rows,
                                 int64_t row0, uint8_t* out, float* scale, cudaStream_t stream);
cudaError_t launch_wait_probe(uint64_t limit_ns, unsigned* status, cudaStream_t stream);

}  // namespace ptb
