// LayerNorm of the parallel transformer block: the PTB applies one LN to x
// and feeds the result to both the attention and the MLP branch (MegaScale
// study notes, ch.2 §2.2, PTB row).
//
//   out[r, :] = (x[r, :] - mean_r) / sqrt(var_r + eps) * gamma + beta
//
// var is the biased (population) variance.  One CTA per row: the row is read
// once with 16-byte loads into registers, the mean and then the centred sum of
// squares are reduced in fp32 (warp shuffles, then across warps through shared
// memory), and the normalised row is written with 16-byte stores.  The kernel
// is a pure HBM stream: 2 * H bytes read and H * 2 bytes written per row.
// With `stats` set it also keeps (mean, 1/sqrt(var + eps)) of every row for
// the backward pass.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int kLnThreads = 256;
constexpr int kLnMaxVec = 16;  // 16-byte vectors per thread -> H <= 32768

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still be read from the previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kLnThreads / 32; ++w) t += red[w];
  return t;
}

// VPT: 16-byte vectors of the row per thread (the row cache is sized to the
// hidden size, so that more CTAs fit on an SM: at H = 12288, 6 instead of 16
// vectors per thread).
template <int VPT>
__global__ void __launch_bounds__(kLnThreads) layernorm_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, int hidden, float eps,
    __nv_bfloat16* __restrict__ out, float2* __restrict__ stats) {
  __shared__ float red[kLnThreads / 32];
  const int64_t row = blockIdx.x;
  const int nvec = hidden / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * hidden);

  uint4 cache[VPT];
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * kLnThreads;
    if (v < nvec) {
      cache[j] = __ldcs(src + v);
      const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += bf16_lo(w[e]) + bf16_hi(w[e]);
    }
  }
  const float mean = block_sum(sum, red) / static_cast<float>(hidden);

  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * kLnThreads;
    if (v < nvec) {
      const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16_lo(w[e]) - mean;
        const float b = bf16_hi(w[e]) - mean;
        sq += a * a + b * b;
      }
    }
  }
  const float var = block_sum(sq, red) / static_cast<float>(hidden);
  const float rstd = rsqrtf(var + eps);
  if (stats && threadIdx.x == 0) stats[row] = make_float2(mean, rstd);

  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(beta);
  uint4* dst = reinterpret_cast<uint4*>(out + row * hidden);
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int v = threadIdx.x + j * kLnThreads;
    if (v < nvec) {
      const uint4 gv = __ldg(g4 + v);
      const uint4 bv = __ldg(b4 + v);
      const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = (bf16_lo(w[e]) - mean) * rstd * bf16_lo(gw[e]) + bf16_lo(bw[e]);
        const float b = (bf16_hi(w[e]) - mean) * rstd * bf16_hi(gw[e]) + bf16_hi(bw[e]);
        o[e] = pack_bf16x2(a, b);
      }
      dst[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

cudaError_t launch_layernorm(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                             const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                             __nv_bfloat16* out, cudaStream_t stream, float2* stats) {
  if (hidden % 8 != 0 || hidden / 8 > kLnMaxVec * kLnThreads) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  if (rows > 0x7fffffff) return cudaErrorInvalidValue;
  const int vpt = (hidden / 8 + kLnThreads - 1) / kLnThreads;
  const unsigned grid = static_cast<unsigned>(rows);
#define PTB_LN_CASE(V)                                                                         \
  if (vpt <= V) {                                                                               \
    layernorm_kernel<V><<<grid, kLnThreads, 0, stream>>>(x, gamma, beta, hidden, eps, out,     \
                                                         stats);                               \
    return cudaGetLastError();                                                                  \
  }
  PTB_LN_CASE(1)
  PTB_LN_CASE(2)
  PTB_LN_CASE(3)
  PTB_LN_CASE(4)
  PTB_LN_CASE(6)
  PTB_LN_CASE(8)
  PTB_LN_CASE(10)
  PTB_LN_CASE(12)
  PTB_LN_CASE(16)
#undef PTB_LN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ptb
