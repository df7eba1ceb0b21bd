// e4m3 (FP8) operand preparation for the FP8 variant of the PTB forward pass.
//
// The Megatron-LM page (mixed-precision section) lists FP8 among the
// supported precisions, to be used with dynamic scaling and with care for
// numerical stability.  Here both GEMMs of the layer take e4m3 operands with
// one dynamic fp32 scale per row of each operand, so the scales factor out of
// every dot product: C[m, n] = a_scale[m] * b_scale[n] * sum_k A8[m, k] B8[n, k].
//   * layernorm_fp8_kernel: xn = LN(x) quantized per token row.
//   * quantize_rows_kernel: rows of [src0 | src1] (two column blocks of
//     bf16 matrices) quantized per row -- the second GEMM's A operand
//     [ctx | G] every layer, and the weights once.  Two passes, no staging.
// A row's scale is amax(|row|) / 448 (448 = largest finite e4m3), 1 for an
// all-zero row; values are rounded to nearest e4m3 with saturation.
#include <cuda_fp8.h>

#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr float kE4m3Max = 448.f;
constexpr int kQThreads = 256;

constexpr int kLnMaxVec = 16;  // 16-byte vectors of bf16 per thread -> H <= 32768

__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  return __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

template <int THREADS = kQThreads>
__device__ __forceinline__ float block_reduce(float v, float* red, bool is_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5;
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;  // both reductions here are of non-negative values or plain sums
  for (int w = 0; w < THREADS / 32; ++w) t = is_max ? fmaxf(t, red[w]) : t + red[w];
  return t;
}

// Stores 8 values (one 16-byte bf16 vector's worth) as 8 e4m3 bytes.
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float inv) {
  const uint32_t lo = static_cast<uint32_t>(e4m3x2(v[0] * inv, v[1] * inv)) |
                      (static_cast<uint32_t>(e4m3x2(v[2] * inv, v[3] * inv)) << 16);
  const uint32_t hi = static_cast<uint32_t>(e4m3x2(v[4] * inv, v[5] * inv)) |
                      (static_cast<uint32_t>(e4m3x2(v[6] * inv, v[7] * inv)) << 16);
  return make_uint2(lo, hi);
}

// VPT: 16-byte vectors of the row per thread (the row cache is sized to the
// hidden size so that more CTAs fit on an SM).
template <int VPT>
__global__ void __launch_bounds__(kQThreads) layernorm_fp8_kernel(
    const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
    const __nv_bfloat16* __restrict__ beta, int hidden, float eps, uint8_t* __restrict__ out,
    float* __restrict__ scale) {
  __shared__ float red[kQThreads / 32];
  const int64_t row = blockIdx.x;
  const int nvec = hidden / 8;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * hidden);
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const uint4* b4 = reinterpret_cast<const uint4*>(beta);
  uint4 cache[VPT];
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int i = threadIdx.x + j * kQThreads;
    if (i < nvec) {
      cache[j] = __ldcs(src + i);
      const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) sum += bf16_lo(w[e]) + bf16_hi(w[e]);
    }
  }
  const float mean = block_reduce(sum, red, false) / static_cast<float>(hidden);
  float sq = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    if (threadIdx.x + j * kQThreads < nvec) {
      const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16_lo(w[e]) - mean, b = bf16_hi(w[e]) - mean;
        sq += a * a + b * b;
      }
    }
  }
  const float rstd = rsqrtf(block_reduce(sq, red, false) / static_cast<float>(hidden) + eps);
  // The normalised row is recomputed from the cached input for the amax and
  // for the store (cheaper than keeping it in registers).
  auto normalised = [&](int j, int i, float (&f)[8]) {
    const uint4 gv = __ldg(g4 + i), bv = __ldg(b4 + i);
    const uint32_t w[4] = {cache[j].x, cache[j].y, cache[j].z, cache[j].w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, bw[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = (bf16_lo(w[e]) - mean) * rstd * bf16_lo(gw[e]) + bf16_lo(bw[e]);
      f[2 * e + 1] = (bf16_hi(w[e]) - mean) * rstd * bf16_hi(gw[e]) + bf16_hi(bw[e]);
    }
  };
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int i = threadIdx.x + j * kQThreads;
    if (i < nvec) {
      float f[8];
      normalised(j, i, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
    }
  }
  amax = block_reduce(amax, red, true);
  const float s = amax > 0.f ? amax / kE4m3Max : 1.f;
  const float inv = 1.f / s;
  uint2* dst = reinterpret_cast<uint2*>(out + row * hidden);
#pragma unroll
  for (int j = 0; j < VPT; ++j) {
    const int i = threadIdx.x + j * kQThreads;
    if (i < nvec) {
      float f[8];
      normalised(j, i, f);
      dst[i] = quant8(f, inv);
    }
  }
  if (threadIdx.x == 0) scale[row] = s;
}

// Row r of the output is [src0[r, 0:n0] | src1[r, 0:n1]] quantized with one
// scale; written to out[(row0 + r) * (n0 + n1) ...] and scale[row0 + r].
// Two passes over the row: the amax, then (re-reading the row, mostly from
// L2) the quantized store.  Nothing is staged in shared memory, so 2048
// threads per SM (eight CTAs of 256 or two of 1024) keep loads in flight.
// The rows in flight, one per CTA, must stay in L2 for the second pass, so
// rows over 64 KB take 1024-thread CTAs: with 256-thread ones the 123 KB
// rows of the 175B-shaped [ctx | G] (2048 x 61440) put ~150 MB in flight,
// more than L2 (quantize 94 -> 77 us; the 530B shape 153 -> 130 us), while
// the 51 KB rows of the 13B shape run faster on 256 (34 against 45 us).  (A
// version that staged the row in shared memory ran one CTA per SM and took
// 122 us for the 175B shape.)
__device__ __forceinline__ uint4 row_vec(const uint4* a, const uint4* b, int v0, int i) {
  return i < v0 ? __ldg(a + i) : __ldg(b + (i - v0));
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS) quantize_rows_kernel(
    const __nv_bfloat16* __restrict__ src0, int64_t ld0, int n0,
    const __nv_bfloat16* __restrict__ src1, int64_t ld1, int n1, int64_t row0,
    uint8_t* __restrict__ out, float* __restrict__ scale) {
  __shared__ float red[THREADS / 32];
  const int64_t r = blockIdx.x;
  const int v0 = n0 / 8, nv = (n0 + n1) / 8;
  const uint4* a = reinterpret_cast<const uint4*>(src0 + r * ld0);
  const uint4* b = src1 ? reinterpret_cast<const uint4*>(src1 + r * ld1) : a;
  float amax = 0.f;
  int i = threadIdx.x;
  for (; i + 3 * THREADS < nv; i += 4 * THREADS) {  // four 16-byte loads in flight
    uint4 c[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) c[u] = row_vec(a, b, v0, i + u * THREADS);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {c[u].x, c[u].y, c[u].z, c[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    }
  }
  for (; i < nv; i += THREADS) {
    const uint4 c = row_vec(a, b, v0, i);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
  }
  amax = block_reduce<THREADS>(amax, red, true);
  const float s = amax > 0.f ? amax / kE4m3Max : 1.f;
  const float inv = 1.f / s;
  uint2* dst = reinterpret_cast<uint2*>(out + (row0 + r) * static_cast<int64_t>(n0 + n1));
  for (int j = threadIdx.x; j < nv; j += THREADS) {
    const uint4 c = row_vec(a, b, v0, j);
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      f[2 * e] = bf16_lo(w[e]);
      f[2 * e + 1] = bf16_hi(w[e]);
    }
    dst[j] = quant8(f, inv);
  }
  if (threadIdx.x == 0) scale[row0 + r] = s;
}

}  // namespace

cudaError_t launch_layernorm_fp8(const __nv_bfloat16* x, const __nv_bfloat16* gamma,
                                 const __nv_bfloat16* beta, int64_t rows, int hidden, float eps,
                                 uint8_t* out, float* scale, cudaStream_t stream) {
  if (hidden % 8 != 0 || hidden / 8 > kLnMaxVec * kQThreads || rows > 0x7fffffff)
    return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  const int vpt = (hidden / 8 + kQThreads - 1) / kQThreads;
  const unsigned grid = static_cast<unsigned>(rows);
#define PTB_LNQ_CASE(V)                                                                        \
  if (vpt <= V) {                                                                               \
    layernorm_fp8_kernel<V><<<grid, kQThreads, 0, stream>>>(x, gamma, beta, hidden, eps, out,  \
                                                            scale);                            \
    return cudaGetLastError();                                                                  \
  }
  PTB_LNQ_CASE(1)
  PTB_LNQ_CASE(2)
  PTB_LNQ_CASE(3)
  PTB_LNQ_CASE(4)
  PTB_LNQ_CASE(6)
  PTB_LNQ_CASE(8)
  PTB_LNQ_CASE(10)
  PTB_LNQ_CASE(12)
  PTB_LNQ_CASE(16)
#undef PTB_LNQ_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_rows(const __nv_bfloat16* src0, int64_t ld0, int n0,
                                 const __nv_bfloat16* src1, int64_t ld1, int n1, int64_t rows,
                                 int64_t row0, uint8_t* out, float* scale, cudaStream_t stream) {
  if (n0 % 8 || n1 % 8 || n0 + n1 <= 0 || rows > 0x7fffffff) return cudaErrorInvalidValue;
  if (rows <= 0) return cudaSuccess;
  if (2 * static_cast<int64_t>(n0 + n1) > (int64_t{64} << 10))
    quantize_rows_kernel<1024><<<static_cast<unsigned>(rows), 1024, 0, stream>>>(
        src0, ld0, n0, src1, ld1, n1, row0, out, scale);
  else
    quantize_rows_kernel<256><<<static_cast<unsigned>(rows), 256, 0, stream>>>(
        src0, ld0, n0, src1, ld1, n1, row0, out, scale);
  return cudaGetLastError();
}

}  // namespace ptb
