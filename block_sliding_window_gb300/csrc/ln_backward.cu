// Backward pass of the PTB's LayerNorm, with the block's residual path.
//
// y = x + Attn(LN(x)) + MLP(LN(x)) (MegaScale study notes, ch.2 §2.2, PTB
// row), so dL/dx = dy + LN'(x)^T dxn, where dxn = dL/dLN(x) collects both
// branches.  For xh = (x - mean) * r, r = 1 / sqrt(var + eps) and
// g = dxn * gamma:
//   dx     = dy + r * (g - mean(g) - xh * mean(g * xh))
//   dgamma = sum over rows of dxn * xh,   dbeta = sum over rows of dxn.
// Three launches, all deterministic:
//   ln_bwd_rows_kernel     one CTA per row: dx (two block reductions).
//   ln_bwd_columns_kernel  one thread per column pair and chunk of 32 rows:
//                          partial sums of dxn * xh and dxn in row order.
//   ln_bwd_reduce_kernel   one lane per column, 8 warps over the chunks: the
//                          chunk partials summed in a fixed order.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int kThreads = 256;
constexpr int kChunkRows = 32;  // rows per column partial (more CTAs in flight)

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();  // red[] may still be read from the previous reduction
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += red[w];
  return t;
}

// 8 values of one 8-column vector v of a row: xh = (x - mean) * r and
// g = dxn * gamma.
__device__ __forceinline__ void load_vec(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                         const float* dxn, int64_t row, int hidden, int v,
                                         float mean, float r, float (&xh)[8], float (&g)[8]) {
  const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + row * hidden) + v);
  const uint4 gv = __ldg(reinterpret_cast<const uint4*>(gamma) + v);
  const float4 d0 = __ldg(reinterpret_cast<const float4*>(dxn + row * hidden) + 2 * v);
  const float4 d1 = __ldg(reinterpret_cast<const float4*>(dxn + row * hidden) + 2 * v + 1);
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
  const float dd[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    xh[2 * e] = (bf16_lo(xw[e]) - mean) * r;
    xh[2 * e + 1] = (bf16_hi(xw[e]) - mean) * r;
    g[2 * e] = dd[2 * e] * bf16_lo(gw[e]);
    g[2 * e + 1] = dd[2 * e + 1] * bf16_hi(gw[e]);
  }
}

// Two passes over the row: the sums of g and g * xh, then dx (the second
// pass re-reads the row, mostly from L1 / L2).
__global__ void __launch_bounds__(kThreads) ln_bwd_rows_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const float2* __restrict__ stats, const float* __restrict__ dxn,
    const __nv_bfloat16* __restrict__ dy, int hidden, __nv_bfloat16* __restrict__ dx) {
  __shared__ float red[kThreads / 32];
  const int64_t row = blockIdx.x;
  const int nvec = hidden / 8;
  const float2 st = stats[row];
  const float mean = st.x, r = st.y;
  float sg = 0.f, sgx = 0.f;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    float xh[8], g[8];
    load_vec(x, gamma, dxn, row, hidden, v, mean, r, xh, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sg += g[e];
      sgx += g[e] * xh[e];
    }
  }
  const float inv_h = 1.f / static_cast<float>(hidden);
  const float mg = block_sum(sg, red) * inv_h;
  const float mgx = block_sum(sgx, red) * inv_h;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    float xh[8], g[8];
    load_vec(x, gamma, dxn, row, hidden, v, mean, r, xh, g);
    const uint4 yv = __ldg(reinterpret_cast<const uint4*>(dy + row * hidden) + v);
    const uint32_t yw[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      o[e] = pack_bf16x2(bf16_lo(yw[e]) + r * (g[2 * e] - mg - xh[2 * e] * mgx),
                         bf16_hi(yw[e]) + r * (g[2 * e + 1] - mg - xh[2 * e + 1] * mgx));
    reinterpret_cast<uint4*>(dx + row * hidden)[v] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// partials[chunk][0][c] = sum over the chunk's rows of dxn * xh,
// partials[chunk][1][c] = sum of dxn, rows in increasing order.  A thread
// takes two adjacent columns (bf16x2 / float2 loads; hidden is a multiple of
// 8), and the rows are unrolled by 8 so that 16 loads are in flight.
__global__ void ln_bwd_columns_kernel(const __nv_bfloat16* __restrict__ x,
                                      const float2* __restrict__ stats,
                                      const float* __restrict__ dxn, int64_t rows, int hidden,
                                      float* __restrict__ partials) {
  const int c = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (c >= hidden) return;
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kChunkRows;
  const int64_t r1 = r0 + kChunkRows < rows ? r0 + kChunkRows : rows;
  float sgx0 = 0.f, sgx1 = 0.f, sd0 = 0.f, sd1 = 0.f;
#pragma unroll 8
  for (int64_t r = r0; r < r1; ++r) {
    const float2 st = __ldg(stats + r);
    const float2 d = __ldg(reinterpret_cast<const float2*>(dxn + r * hidden + c));
    const uint32_t xv = __ldg(reinterpret_cast<const unsigned int*>(x + r * hidden + c));
    sgx0 += d.x * ((bf16_lo(xv) - st.x) * st.y);
    sgx1 += d.y * ((bf16_hi(xv) - st.x) * st.y);
    sd0 += d.x;
    sd1 += d.y;
  }
  const int64_t base = static_cast<int64_t>(blockIdx.y) * 2 * hidden + c;
  *reinterpret_cast<float2*>(partials + base) = make_float2(sgx0, sgx1);
  *reinterpret_cast<float2*>(partials + base + hidden) = make_float2(sd0, sd1);
}

// dgamma / dbeta: the chunk partials of a column summed in a fixed order.
// A CTA takes 32 columns (lane = column); its 8 warps each sum every 8th
// chunk in increasing order, and warp 0 adds the 8 warp sums in warp order.
__global__ void __launch_bounds__(kThreads) ln_bwd_reduce_kernel(
    const float* __restrict__ partials, int64_t chunks, int hidden, float* __restrict__ dgamma,
    float* __restrict__ dbeta) {
  __shared__ float red[2][kThreads / 32][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float a = 0.f, b = 0.f;
  if (c < hidden) {
    for (int64_t k = warp; k < chunks; k += kThreads / 32) {
      a += __ldg(partials + (2 * k) * hidden + c);
      b += __ldg(partials + (2 * k + 1) * hidden + c);
    }
  }
  red[0][warp][lane] = a;
  red[1][warp][lane] = b;
  __syncthreads();
  if (warp == 0 && c < hidden) {
    float ta = 0.f, tb = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      ta += red[0][w][lane];
      tb += red[1][w][lane];
    }
    dgamma[c] = ta;
    dbeta[c] = tb;
  }
}

}  // namespace

int64_t ln_backward_chunks(int64_t rows) { return (rows + kChunkRows - 1) / kChunkRows; }

cudaError_t launch_layernorm_backward(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                      const float2* stats, const float* dxn,
                                      const __nv_bfloat16* dy, int64_t rows, int hidden,
                                      __nv_bfloat16* dx, float* dgamma, float* dbeta,
                                      float* partials, cudaStream_t stream) {
  if (hidden % 8 != 0 || hidden <= 0) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  const int64_t chunks = ln_backward_chunks(rows);
  if (rows > 0x7fffffff || chunks > 65535) return cudaErrorInvalidValue;
  ln_bwd_rows_kernel<<<static_cast<unsigned>(rows), kThreads, 0, stream>>>(x, gamma, stats, dxn,
                                                                          dy, hidden, dx);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const dim3 grid((hidden / 2 + kThreads - 1) / kThreads, static_cast<unsigned>(chunks));
  ln_bwd_columns_kernel<<<grid, kThreads, 0, stream>>>(x, stats, dxn, rows, hidden, partials);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ln_bwd_reduce_kernel<<<(hidden + 31) / 32, kThreads, 0, stream>>>(partials, chunks, hidden,
                                                                   dgamma, dbeta);
  return cudaGetLastError();
}

}  // namespace ptb
