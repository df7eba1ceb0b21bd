// Causal sliding-window attention (SWA), flash-style and banded.
//
// Every token attends to a fixed window of w positions, so the cost is
// O(s*w) rather than O(s*s) (MegaScale study notes, ch.2 §2.2, SWA row);
// FlashAttention-2 is the fused attention operator the notes list (§2.5,
// Table 3).  Row i attends to keys max(0, i-w+1) .. i (causal, self-inclusive).
//
// One CTA handles one (batch, head) and a tile of 64 query rows with four
// warps of 16 rows each.  It walks ONLY the 64-key K/V tiles that intersect
// the band [q0 - w + 1, q0 + 63], from the diagonal tile downwards, with the
// next tile's K and V streamed into shared memory (cp.async, double-buffered)
// while the current one is used.  Per tile and warp:
//   S = Q K^T        16 x 64, bf16 mma.sync, fp32 accumulate
//   mask             only on tiles that cross the band's edges
//   online softmax   running row max m and sum l in fp32 registers, in the
//                    log2 domain (the scale * log2(e) folded into S); row
//                    reductions with quad shuffles
//   O += P V         P re-packed to bf16 straight from the S registers
// At the end O / l is stored as bf16.  With counts enabled the kernel also
// reports, per row, how many keys passed its own mask.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int BQ = 64;
constexpr int BKV = 64;
constexpr int kSwaThreads = 128;

template <int D>
struct SwaSmem {
  static constexpr int LD = D + 8;  // padded row (elements): conflict-free ldmatrix
  static constexpr int kBytes = (BQ + 4 * BKV) * LD * 2;
};

// Copies rows row0 .. row0+nrows-1 of the [seq, D] matrix at `base` (row
// stride in elements) into shared memory; rows at or beyond seq are zero-filled
// without being read.
template <int D>
__device__ __forceinline__ void load_rows(__nv_bfloat16* dst, const __nv_bfloat16* base,
                                          int64_t row_stride, int row0, int nrows, int seq) {
  constexpr int LD = SwaSmem<D>::LD;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  for (int c = threadIdx.x; c < nrows * kChunks; c += kSwaThreads) {
    const int r = c / kChunks;
    const int ch = c % kChunks;
    const int gr = row0 + r;
    const bool valid = gr < seq;
    const __nv_bfloat16* g = base + static_cast<int64_t>(valid ? gr : 0) * row_stride + ch * 8;
    cp_async_16(smem_addr(dst + r * LD + ch * 8), g, valid);
  }
}

template <int D, bool COUNTS>
__global__ void __launch_bounds__(kSwaThreads) swa_kernel(const SwaArgs p) {
  constexpr int LD = SwaSmem<D>::LD;
  constexpr int KSTEPS = D / 16;  // k-steps of S = Q K^T
  constexpr int DTILES = D / 8;   // n-tiles of O
  extern __shared__ __align__(128) uint8_t swa_smem[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(swa_smem);
  __nv_bfloat16* sK = sQ + BQ * LD;        // [2][BKV][LD]
  __nv_bfloat16* sV = sK + 2 * BKV * LD;   // [2][BKV][LD]

  const int q0 = blockIdx.x * BQ;
  const int b = blockIdx.y / p.heads;
  const int h = blockIdx.y % p.heads;
  const int seq = p.seq;
  const int window = p.window;
  const __nv_bfloat16* Q = p.q + b * p.q_sb + h * p.q_sh;
  const __nv_bfloat16* K = p.k + b * p.k_sb + h * p.k_sh;
  const __nv_bfloat16* V = p.v + b * p.v_sb + h * p.v_sh;
  __nv_bfloat16* O = p.o + b * p.o_sb + h * p.o_sh;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;  // row inside the 8-row half of the fragment
  const int t = lane & 3;   // column pair inside the fragment

  // Key tiles that intersect the band of this query tile.
  const int k_first = max(0, q0 - window + 1);
  const int k_last = min(seq - 1, q0 + BQ - 1);
  const int kt_lo = k_first / BKV;
  const int kt_hi = k_last / BKV;
  const int n_tiles = kt_hi - kt_lo + 1;

  load_rows<D>(sQ, Q, p.q_ss, q0, BQ, seq);
  load_rows<D>(sK, K, p.k_ss, kt_hi * BKV, BKV, seq);
  load_rows<D>(sV, V, p.v_ss, kt_hi * BKV, BKV, seq);
  cp_async_commit();

  uint32_t qf[KSTEPS][4];
  float o[DTILES][4];
#pragma unroll
  for (int n = 0; n < DTILES; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  int cnt[2] = {0, 0};

  const int row_lo = q0 + warp * 16;  // first query row of this warp
  const int qi[2] = {row_lo + g, row_lo + g + 8};

  for (int it = 0; it < n_tiles; ++it) {
    const int kt = kt_hi - it;
    const int buf = it & 1;
    if (it + 1 < n_tiles) {
      const int nk = kt - 1;
      load_rows<D>(sK + (buf ^ 1) * BKV * LD, K, p.k_ss, nk * BKV, BKV, seq);
      load_rows<D>(sV + (buf ^ 1) * BKV * LD, V, p.v_ss, nk * BKV, BKV, seq);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    if (it == 0) {
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int r = warp * 16 + (lane & 15);
        const int c = kk * 16 + 8 * (lane >> 4);
        ldsm_x4(smem_addr(sQ + r * LD + c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }

    const __nv_bfloat16* k_s = sK + buf * BKV * LD;
    const __nv_bfloat16* v_s = sV + buf * BKV * LD;

    // S = Q K^T for this warp's 16 rows and the tile's 64 keys.
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int key = np * 16 + (lane & 7) + 8 * (lane >> 4);
        const int c = kk * 16 + 8 * ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_addr(k_s + key * LD + c), b0, b1, b2, b3);
        mma_bf16_16816(s[2 * np], qf[kk], b0, b1);
        mma_bf16_16816(s[2 * np + 1], qf[kk], b2, b3);
      }
    }

    // Scale into the log2 domain; mask only where the tile crosses the band.
    const int key0 = kt * BKV;
    const bool interior = (key0 + BKV - 1 <= row_lo) && (key0 >= row_lo + 15 - window + 1);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[j][e] * p.scale_log2;
        if (!interior) {
          const int kj = key0 + 8 * j + 2 * t + (e & 1);
          const int i = qi[e >> 1];
          const bool keep = (kj <= i) && (kj > i - window);
          x = keep ? x : -INFINITY;
          if (COUNTS) cnt[e >> 1] += keep ? 1 : 0;
        }
        s[j][e] = x;
      }
    }
    if (COUNTS && interior) {
      cnt[0] += 16;
      cnt[1] += 16;
    }

    // Online softmax update.
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) mx = fmaxf(mx, fmaxf(s[j][2 * r], s[j][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[r], mx);
      const float m_ref = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m_run[r] - m_ref);
      m_run[r] = m_new;
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float a = fast_exp2(s[j][2 * r] - m_ref);
        const float c = fast_exp2(s[j][2 * r + 1] - m_ref);
        s[j][2 * r] = a;
        s[j][2 * r + 1] = c;
        rs += a + c;
      }
      l_run[r] = l_run[r] * alpha + rs;
#pragma unroll
      for (int n = 0; n < DTILES; ++n) {
        o[n][2 * r] *= alpha;
        o[n][2 * r + 1] *= alpha;
      }
    }

    // O += P V.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int key = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = dp * 16 + 8 * (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_addr(v_s + key * LD + c), b0, b1, b2, b3);
        mma_bf16_16816(o[2 * dp], pa, b0, b1);
        mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();  // the buffer is refilled in the next iteration
  }

  // Normalise and store.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_run[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int i = qi[r];
    if (i < seq) {
      __nv_bfloat16* orow = O + static_cast<int64_t>(i) * p.o_ss;
#pragma unroll
      for (int n = 0; n < DTILES; ++n) {
        const uint32_t v = pack_bf16x2(o[n][2 * r] * inv, o[n][2 * r + 1] * inv);
        *reinterpret_cast<uint32_t*>(orow + 8 * n + 2 * t) = v;
      }
    }
    if (COUNTS) {
      int c = cnt[r];
      c += __shfl_xor_sync(0xffffffffu, c, 1);
      c += __shfl_xor_sync(0xffffffffu, c, 2);
      if (t == 0 && i < seq)
        p.counts[(static_cast<int64_t>(b) * p.heads + h) * seq + i] = c;
    }
  }
}

template <int D, bool COUNTS>
cudaError_t launch_typed(const SwaArgs& a, cudaStream_t stream) {
  constexpr int kBytes = SwaSmem<D>::kBytes;
  auto kern = swa_kernel<D, COUNTS>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const dim3 grid((a.seq + BQ - 1) / BQ, a.batch * a.heads);
  kern<<<grid, kSwaThreads, kBytes, stream>>>(a);
  return cudaGetLastError();
}

template <bool COUNTS>
cudaError_t dispatch(const SwaArgs& a, cudaStream_t stream) {
  switch (a.head_dim) {
    case 16: return launch_typed<16, COUNTS>(a, stream);
    case 32: return launch_typed<32, COUNTS>(a, stream);
    case 64: return launch_typed<64, COUNTS>(a, stream);
    case 96: return launch_typed<96, COUNTS>(a, stream);
    case 128: return launch_typed<128, COUNTS>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_swa(const SwaArgs& a, cudaStream_t stream) {
  if (a.seq <= 0 || a.batch <= 0 || a.heads <= 0) return cudaSuccess;
  return a.counts ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

}  // namespace ptb
