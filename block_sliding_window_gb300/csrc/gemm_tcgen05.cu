// The two GEMMs of the parallel transformer block on tcgen05 tensor cores.
//
//   [QKV | up]  : U = [xn W_qkv^T | gelu_tanh(xn W_up^T)]      (one GEMM, N = 3H + F)
//   [out | down]: y = x + [ctx | G] [W_o | W_down]^T            (one GEMM, K = H + F)
//
// The PTB computes the attention and MLP branches from the same LN(x) and
// sums both with the residual (MegaScale study notes, ch.2 §2.2, PTB row),
// so the two input projections share one GEMM and the two output
// projections share one GEMM whose epilogue adds x.  GeLU is fused into the
// first GEMM's epilogue (§2.5, Table 3, efficient-operators row).
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0      TMA producer: 128 x 64 A tile and BN x 64 B tile per stage
//               into a ring of shared-memory stages (128-byte swizzle).
//   warp 1      owns the TMEM allocation; one thread issues tcgen05.mma
//               (M = 128, N = BN, K = 16) into a double-buffered fp32
//               accumulator in TMEM and commits stage / tile completion to
//               mbarriers.  (Measured on GB300: with 128 x 256 tiles a
//               64-wide k-block takes ~790 cycles for 512 cycles of MMA work,
//               matching the shared-memory traffic per k-block -- 48 KB of
//               operand reads plus 48 KB of TMA writes at ~128 B/clk.)
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4) .. +31, i.e. one output row per thread),
//               GELU or residual add in fp32, bf16 stores.  The epilogue of
//               one work unit overlaps the main loop of the next.
//
// Work units.  The tiles that fill whole waves (a multiple of the grid) are
// processed whole, M-fastest, so the M tiles of one weight block run at the
// same time and share it through L2; odd waves walk K backwards, so each wave
// starts on the k-slabs the previous one left in L2.  The remaining R < grid tiles of the
// last, partial wave are each split along K into S pieces (R*S <= grid), one
// piece per otherwise idle CTA.  A piece writes its fp32 partial tile to the
// workspace and bumps an arrival counter per 32-row quarter of the tile; the
// epilogue warp that arrives last for a quarter sums the S partials of those
// rows in piece order (so the bits do not depend on who finished) and runs
// the epilogue for them.  Nothing ever waits on another CTA or another warp.
//
// Every mbarrier wait is bounded (see mbar_wait); on a timeout all roles
// unwind, wait for their own copies and MMAs, free TMEM and return.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int BM = 128;
// One k-block is one 128-byte swizzle row: 64 bf16 or 128 e4m3 elements,
// consumed by four MMAs (K = 16 bf16 or K = 32 e4m3 each, 32 bytes apart).
template <bool FP8>
struct Elem {
  static constexpr int kBK = FP8 ? 128 : 64;
};
constexpr int kMmasPerBlock = 4;
constexpr int kThreads = 192;

// The weight-gradient GEMMs (fp32 output, both operands MN-major) write
// their large outputs through shared memory: each epilogue warp stages its
// 32 rows x 32 columns (rows padded to 36 floats) and then writes whole
// 128-byte row segments, 4 rows per store instruction, instead of one
// 16-byte piece of 32 different rows.  Measured on GB300 (13B-class
// training step): the two weight-gradient GEMMs 7% and 9% faster; the same
// staging (and its 18 KB of shared memory) on every variant made the other
// GEMMs 3-15% slower, so only these variants use it.
constexpr int kF32Pad = 36;
constexpr int kF32StageBytes = 4 * 32 * kF32Pad * 4;

template <int EPI, int LAYOUT>
__host__ __device__ constexpr bool staged_f32() {
  return EPI == kEpiF32 && LAYOUT == kLayoutNN;
}

template <int BN, bool STAGE = false>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
  static constexpr int kABytes = BM * 128;  // 128-byte rows: 64 bf16 or 128 e4m3
  static constexpr int kBBytes = BN * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes =
      kStages * kStageBytes + kBarBytes + (STAGE ? kF32StageBytes : 0) + 1024;
};

__device__ __forceinline__ float gelu_tanh(float z) {
  const float k0 = 0.7978845608028654f;  // sqrt(2 / pi)
  const float k1 = 0.044715f;
  return 0.5f * z * (1.0f + tanhf(k0 * (z + k1 * z * z * z)));
}

// One unit of work: k-blocks [kb0, kb1) of one output tile.  slot >= 0 marks
// a K piece of a remainder tile (its index in the partial-tile buffer).
struct Unit {
  int tile, kb0, kb1, slot;
};

// The i-th unit of worker `self` of `count` (a CTA, or a CTA pair); false
// when the worker has no more work.
__device__ __forceinline__ bool unit_at(const GemmArgs& p, int num_tiles, int num_kb, int i,
                                        Unit& u, int self, int count) {
  if (p.split_s < 2) {
    const int tile = self + i * count;
    if (tile >= num_tiles) return false;
    u = {tile, 0, num_kb, -1};
    return true;
  }
  const int whole = num_tiles - p.split_r;  // a multiple of count
  const int n_whole = whole / count;
  if (i < n_whole) {
    u = {self + i * count, 0, num_kb, -1};
    return true;
  }
  if (i == n_whole && self < p.split_r * p.split_s) {
    const int r = self / p.split_s;
    const int s = self % p.split_s;
    u = {whole + r, s * num_kb / p.split_s, (s + 1) * num_kb / p.split_s, self};
    return true;
  }
  return false;
}

// The t-th k-block a unit processes.  Whole-tile units of odd waves (odd
// unit index i) walk K backwards: a wave's tiles read the shared operand
// k-slab by k-slab in step, and the operand of the long-K GEMMs is larger
// than L2, so a wave that starts where the previous one ended finds its
// first k-slabs still in L2 instead of re-reading them from DRAM.  K pieces
// of split tiles keep the forward order.
__device__ __forceinline__ int unit_kb(const Unit& u, int i, int t) {
  return ((i & 1) && u.slot < 0) ? u.kb1 - 1 - t : u.kb0 + t;
}

// e4m3 operands carry one scale per A row and one per B row (= output
// column): C[m, n] = a_scale[m] * b_scale[n] * sum_k A8[m, k] B8[n, k].
__device__ __forceinline__ void dequantize(const GemmArgs& p, int row, int col, float (&acc)[32]) {
  const float sa = row < p.M ? __ldg(p.a_scale + row) : 0.f;
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const float4 sb = __ldg(reinterpret_cast<const float4*>(p.b_scale + col) + v);
    acc[4 * v] *= sa * sb.x;
    acc[4 * v + 1] *= sa * sb.y;
    acc[4 * v + 2] *= sa * sb.z;
    acc[4 * v + 3] *= sa * sb.w;
  }
}

// d/dz gelu_tanh(z) = 0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3 a z^2),
// t = tanh(c (z + a z^3)), c = sqrt(2 / pi), a = 0.044715.
__device__ __forceinline__ float gelu_tanh_grad(float z) {
  const float k0 = 0.7978845608028654f;
  const float k1 = 0.044715f;
  const float t = tanhf(k0 * (z + k1 * z * z * z));
  return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * k0 * (1.0f + 3.0f * k1 * z * z);
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst_row, const uint32_t (&packed)[16]) {
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
#pragma unroll
  for (int v = 0; v < 4; ++v)
    dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
}

// Epilogue of one 32-column chunk of one output row: acc (fp32) -> out.
template <int EPI>
__device__ __forceinline__ void store_chunk(const GemmArgs& p, int row, int col,
                                            const float (&acc)[32]) {
  // Destination region (a 32-column chunk never straddles a split point).
  void* base = p.out;
  int64_t ld = p.ld_out;
  int64_t r = row, c = col;
  if (col >= p.out_split_col) {
    base = p.out1;
    ld = p.ld_out1;
    c -= p.out_split_col;
  } else if (row >= p.out_split_row) {
    base = p.out1;
    ld = p.ld_out1;
    r -= p.out_split_row;
  }
  if constexpr (EPI == kEpiF32) {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + r * ld + c);
#pragma unroll
    for (int v = 0; v < 8; ++v)
      dst[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
    return;
  }
  uint32_t packed[16];
  if constexpr (EPI == kEpiQkvGelu) {
    if (col >= p.gelu_col) {
      if (p.aux) {  // keep the pre-activation for the backward pass
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
        store_bf16x32(p.aux + row * p.ld_aux + (col - p.gelu_col), packed);
      }
#pragma unroll
      for (int j = 0; j < 16; ++j)
        packed[j] = pack_bf16x2(gelu_tanh(acc[2 * j]), gelu_tanh(acc[2 * j + 1]));
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
    }
  } else if constexpr (EPI == kEpiDgelu) {
    if (col >= p.gelu_col) {
      const uint4* src = reinterpret_cast<const uint4*>(p.aux + row * p.ld_aux + (col - p.gelu_col));
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 z = __ldg(src + v);
        const uint32_t zs[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = v * 8 + j * 2;
          packed[v * 4 + j] = pack_bf16x2(acc[e] * gelu_tanh_grad(bf16_lo(zs[j])),
                                          acc[e + 1] * gelu_tanh_grad(bf16_hi(zs[j])));
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) packed[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(p.resid + row * p.ld_resid + col);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const uint4 x = __ldg(src + v);
      const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = v * 8 + j * 2;
        packed[v * 4 + j] = pack_bf16x2(acc[e] + bf16_lo(xs[j]), acc[e + 1] + bf16_hi(xs[j]));
      }
    }
  }
  store_bf16x32(static_cast<__nv_bfloat16*>(base) + r * ld + c, packed);
}

// Output tile origin of tile index t (M index fastest, or N index fastest).
__device__ __forceinline__ void tile_origin(const GemmArgs& p, int t, int num_m, int num_n, int bm,
                                            int bn, int& m0, int& n0) {
  if (p.n_fastest) {
    m0 = (t / num_n) * bm;
    n0 = (t % num_n) * bn;
  } else {
    m0 = (t % num_m) * bm;
    n0 = (t / num_m) * bn;
  }
}

// fp32 epilogue of one 32-column chunk for the 32 consecutive rows of a warp
// (lane i holds row row0 + i): staged in `st` (32 x kF32Pad floats) and
// stored row segment by row segment.  Warp-collective.
__device__ __forceinline__ void store_chunk_f32_warp(const GemmArgs& p, int row, int col,
                                                     const float (&acc)[32], int lane,
                                                     float* st) {
  float* mine = st + lane * kF32Pad;
#pragma unroll
  for (int v = 0; v < 8; ++v)
    *reinterpret_cast<float4*>(mine + 4 * v) =
        make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
  __syncwarp();
  const int row0 = row - lane;
  const int c4 = lane & 7;
  const bool second_col = col >= p.out_split_col;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int r = 4 * k + (lane >> 3);
    const float4 v = *reinterpret_cast<const float4*>(st + r * kF32Pad + 4 * c4);
    const int grow = row0 + r;
    if (grow < p.M) {
      float* base = static_cast<float*>(p.out);
      int64_t ld = p.ld_out, rr = grow, cc = col + 4 * c4;
      if (second_col) {
        base = static_cast<float*>(p.out1);
        ld = p.ld_out1;
        cc -= p.out_split_col;
      } else if (grow >= p.out_split_row) {
        base = static_cast<float*>(p.out1);
        ld = p.ld_out1;
        rr -= p.out_split_row;
      }
      *reinterpret_cast<float4*>(base + rr * ld + cc) = v;
    }
  }
  __syncwarp();
}

// The epilogue of one unit for one thread's output row `row`: a whole tile
// goes straight from TMEM through store_chunk; a K piece of a split tile
// publishes its fp32 partial (row `prow` of the ROWS-row partial tile) and
// counts its warp's arrival on p.counters[counter], and the warp that
// arrives last for those 32 rows sums all pieces in piece order and stores.
template <int BN, int EPI, bool FP8, int ROWS, bool STAGE>
__device__ __forceinline__ void epilogue_unit(const GemmArgs& p, const Unit& u, int row, int prow,
                                              int counter, uint32_t t_row, int n0, int lane,
                                              float* f32_stage) {
  bool finish = true;
  if (u.slot >= 0) {
    // A K piece: publish the fp32 partial, then count the arrival.
    float* mine = p.partials + (static_cast<int64_t>(u.slot) * ROWS + prow) * BN;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c, r);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(mine + c);
#pragma unroll
      for (int v = 0; v < 8; ++v)
        __stcg(dst + v, make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                    __uint_as_float(r[4 * v + 2]),
                                    __uint_as_float(r[4 * v + 3])));
    }
    // Each warp owns its 32 rows: it counts its own arrival for that
    // quarter of the tile, and the last warp to arrive for the quarter
    // finishes those rows.  No warp waits for another.
    __threadfence();
    __syncwarp();
    unsigned prev = 0;
    if (lane == 0) prev = atomicAdd(p.counters + counter, 1u);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    finish = prev == static_cast<unsigned>(p.split_s - 1);
    if (finish) __threadfence();
  }
  if (finish && u.slot < 0) {
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c, r);
      tmem_ld_wait();
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = __uint_as_float(r[j]);
      if constexpr (FP8) dequantize(p, row, n0 + c, acc);
      if constexpr (STAGE)
        store_chunk_f32_warp(p, row, n0 + c, acc, lane, f32_stage);
      else if (row < p.M)
        store_chunk<EPI>(p, row, n0 + c, acc);
    }
  } else if (finish) {
    // Sum every piece's partial (this warp's own included) in piece order,
    // so the result does not depend on which warp happened to finish.
    const int group0 = (u.slot / p.split_s) * p.split_s;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float acc[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) acc[j] = 0.f;
      for (int s = 0; s < p.split_s; ++s) {
        const float4* src = reinterpret_cast<const float4*>(
            p.partials + (static_cast<int64_t>(group0 + s) * ROWS + prow) * BN + c);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 q = __ldcg(src + v);
          acc[4 * v] += q.x;
          acc[4 * v + 1] += q.y;
          acc[4 * v + 2] += q.z;
          acc[4 * v + 3] += q.w;
        }
      }
      if constexpr (FP8) dequantize(p, row, n0 + c, acc);
      if constexpr (STAGE)
        store_chunk_f32_warp(p, row, n0 + c, acc, lane, f32_stage);
      else if (row < p.M)
        store_chunk<EPI>(p, row, n0 + c, acc);
    }
  }
}

template <int BN, int EPI, bool FP8, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs p) {
  constexpr bool kStage = staged_f32<EPI, LAYOUT>();
  using C = Cfg<BN, kStage>;
  constexpr int BK = Elem<FP8>::kBK;
  // MN-major operands arrive as 64-wide MN blocks of 64 K rows (8 KB each).
  constexpr bool kAmn = (LAYOUT & 1) != 0;
  constexpr bool kBmn = (LAYOUT & 2) != 0;
  constexpr uint32_t kMnBlock = 64 * 128;
  static_assert(!(FP8 && LAYOUT != kLayoutKK), "e4m3 operands are K-major only");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* tfull_bar = empty_bar + C::kStages;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (p.M + BM - 1) / BM;
  const int num_n = p.N / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + BK - 1) / BK;  // a K tail is zero-filled by TMA

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.a0);
    tma_prefetch_desc(&p.a1);
    tma_prefetch_desc(&p.b0);
    tma_prefetch_desc(&p.b1);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * C::kStageBytes + C::kABytes; };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      // L2 priority of each operand's loads as the launcher chose it (the
      // layer's GEMMs keep both, evict_last).  Measured on this kernel with
      // the weights at normal priority instead of evict_first, the 175B
      // layer ran 11% slower; an L2 prefetch of the tiles 8 k-blocks ahead,
      // 48% slower.
      const uint64_t pol = p.a_keep ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_b = p.b_keep ? l2_policy_evict_last() : l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // bit s: stage s has had a load issued
      uint32_t armed_parity = 0;
      bool ok = true;
      Unit u;
      for (int i = 0; ok && unit_at(p, num_tiles, num_kb, i, u, blockIdx.x, gridDim.x); ++i) {
        int m0, n0;
        tile_origin(p, u.tile, num_m, num_n, BM, BN, m0, n0);
        const bool nlo = n0 < p.n_split;
        const int by = nlo ? n0 : n0 - p.n_split;
        for (int t = 0; t < u.kb1 - u.kb0; ++t) {
          const int kb = unit_kb(u, i, t);
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int k = kb * BK;
          const bool klo = k < p.k_split;
          const int kx = klo ? k : k - p.k_split;
          mbar_arrive_expect_tx(&full_bar[stage], C::kStageBytes);
          const CUtensorMap* amap = klo ? &p.a0 : &p.a1;
          const CUtensorMap* bmap = (nlo && klo) ? &p.b0 : &p.b1;
          if constexpr (kAmn) {
#pragma unroll
            for (int h = 0; h < BM / 64; ++h)
              tma_load_2d(stage_a(stage) + h * kMnBlock, amap, &full_bar[stage], m0 + 64 * h, kx,
                          pol);
          } else {
            tma_load_2d(stage_a(stage), amap, &full_bar[stage], kx, m0, pol);
          }
          if constexpr (kBmn) {
#pragma unroll
            for (int h = 0; h < BN / 64; ++h)
              tma_load_2d(stage_b(stage) + h * kMnBlock, bmap, &full_bar[stage], by + 64 * h, kx,
                          pol_b);
          } else {
            tma_load_2d(stage_b(stage), bmap, &full_bar[stage], kx, by, pol_b);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Unwinding: let every copy this thread issued land before the CTA
        // (and its shared memory) goes away.
        volatile int no_abort = 0;
        for (int s = 0; s < C::kStages; ++s)
          if (armed & (1u << s))
            mbar_wait(&full_bar[s], (armed_parity >> s) & 1u, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idesc = (FP8 ? umma_idesc_e4m3(BM, BN) : umma_idesc_bf16(BM, BN)) |
                                 (kAmn ? 1u << 15 : 0u) | (kBmn ? 1u << 16 : 0u);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit u;
      for (int i = 0; ok && unit_at(p, num_tiles, num_kb, i, u, blockIdx.x, gridDim.x); ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int t = 0; t < u.kb1 - u.kb0; ++t) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = kAmn ? sw128_mnmajor_desc(smem_addr(stage_a(stage)), kMnBlock)
                                      : sw128_kmajor_desc(smem_addr(stage_a(stage)));
          const uint64_t bdesc = kBmn ? sw128_mnmajor_desc(smem_addr(stage_b(stage)), kMnBlock)
                                      : sw128_kmajor_desc(smem_addr(stage_b(stage)));
          // One MMA step along K: +32 bytes inside a K-major swizzled row
          // (+2 in the descriptor's 16-byte units), or 16 rows of 128 bytes
          // of an MN-major block (+128).
          constexpr uint64_t kStepA = kAmn ? 128 : 2;
          constexpr uint64_t kStepB = kBmn ? 128 : 2;
#pragma unroll
          for (int kk = 0; kk < kMmasPerBlock; ++kk) {
            const uint32_t accum = (t != 0 || kk != 0) ? 1u : 0u;
            if constexpr (FP8)
              umma_e4m3_ss(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, idesc, accum);
            else
              umma_bf16_ss(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, idesc, accum);
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(&tfull_bar[acc]);
      }
      // Wait for every MMA this thread issued before TMEM is released.
      umma_commit(done_bar);
      volatile int no_abort = 0;
      mbar_wait(done_bar, 0, &no_abort, p.status);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int row_local = quarter * 32 + lane;
    float* f32_stage = reinterpret_cast<float*>(smem + C::kStages * C::kStageBytes + C::kBarBytes) +
                       quarter * 32 * kF32Pad;
    Unit u;
    for (int i = 0; unit_at(p, num_tiles, num_kb, i, u, blockIdx.x, gridDim.x); ++i) {
      const int acc_buf = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait_warp(&tfull_bar[acc_buf], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      int m0, n0;
      tile_origin(p, u.tile, num_m, num_n, BM, BN, m0, n0);
      const int row = m0 + row_local;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc_buf * BN);
      epilogue_unit<BN, EPI, FP8, BM, kStage>(p, u, row, row_local,
                                              (u.slot / p.split_s) * 4 + quarter, t_row, n0,
                                              lane, f32_stage);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc_buf]);
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------ CTA pairs --
// 256 x 256 output tiles on a CTA pair (a cluster of two CTAs on the two SMs
// of a TPC, tcgen05 cta_group::2).  Rank r loads rows m0 + 128 r of A and
// columns by + 128 r of B into its own shared memory; rank 0 issues M = 256,
// N = 256 MMAs that read both CTAs' tiles at the same offsets, and each CTA's
// TMEM receives its 128 rows of the accumulator.  Per SM and 64-wide k-block
// the stage is 32 KB instead of 48 KB, so the shared-memory traffic of TMA
// writes plus operand reads drops by a third.
//   warp 0      both ranks: TMA producer into their own ring of 5
//               stages (pair_stages).  The
//               copies of both ranks complete on rank 0's `full` barrier of
//               the stage (cta_group::2 TMA), which rank 0 arms with the
//               bytes of both.  (A first version relayed rank 1's stages with
//               a cluster-scope release arrive per stage and ran at 31%
//               tensor activity.)
//   warp 1      both ranks allocate TMEM together (cta_group::2).  Rank 0
//               issues the MMAs and commits stage and tile completion to the
//               barriers at the same offset in both CTAs.
//   warps 2..5  both ranks: epilogue of their 128 rows; each warp then
//               arrives on rank 0's `tempty` barrier (8 arrivals per tile).
// The remainder wave is split along K per pair as in the single-CTA kernel
// (256-row partial tiles, 8 arrival counters per tile).
constexpr int kPairBN = 256;
// Stages of the ring.  Fewer stages leave more of the SM's unified L1 /
// shared memory to L1.  With both operands loaded evict_last, 5 stages for
// every GEMM against 6 for [QKV | up] (5 for the others): 175B-class layer
// 4.41-4.47 vs 4.45-4.50 ms, 13B-class, e4m3 and training within noise; 6
// for all and 7 for [QKV | up] were slower everywhere (175B-class 4.54-4.57
// ms, training 14.3-14.7 vs 14.2-14.4 ms).  (Under the earlier evict_first
// weights, 6 had been 1.7% better for [QKV | up] at 13B.)
template <int EPI>
__host__ __device__ constexpr int pair_stages() { return 5; }
template <bool STAGE = false, int NSTAGES = 6>
struct PairCfg {
  static constexpr int kABytes = BM * 128;
  static constexpr int kBBytes = (kPairBN / 2) * 128;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kTmemCols = 2 * kPairBN;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes =
      NSTAGES * kStageBytes + kBarBytes + (STAGE ? kF32StageBytes : 0) + 1024;
};

template <int EPI, int LAYOUT, bool FP8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ GemmArgs p) {
  constexpr bool kStage = staged_f32<EPI, LAYOUT>();
  using C = PairCfg<kStage, pair_stages<EPI>()>;
  constexpr int BN = kPairBN;
  constexpr int BK = Elem<FP8>::kBK;
  static_assert(!(FP8 && LAYOUT != kLayoutKK), "e4m3 operands are K-major only");
  constexpr int NS = pair_stages<EPI>();
  // MN-major operands arrive as 64-wide MN blocks of 64 K rows (8 KB each).
  constexpr bool kAmn = (LAYOUT & 1) != 0;
  constexpr bool kBmn = (LAYOUT & 2) != 0;
  constexpr uint32_t kMnBlock = 64 * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + NS * C::kStageBytes);
  uint64_t* empty_bar = full_bar + NS;
  uint64_t* tfull_bar = empty_bar + NS;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t rank = cluster_ctarank();
  const int pair = static_cast<int>(blockIdx.x >> 1);
  const int npairs = static_cast<int>(gridDim.x >> 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_m = (p.M + 2 * BM - 1) / (2 * BM);
  const int num_n = p.N / BN;
  const int num_tiles = num_m * num_n;
  const int num_kb = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full_bar[s], 1);  // used in rank 0 only
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 8);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.a0);
    tma_prefetch_desc(&p.a1);
    tma_prefetch_desc(&p.b0);
    tma_prefetch_desc(&p.b1);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before anything crosses the pair
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto stage_a = [&](int s) { return smem + s * C::kStageBytes; };
  auto stage_b = [&](int s) { return smem + s * C::kStageBytes + C::kABytes; };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      const uint64_t pol = p.a_keep ? l2_policy_evict_last() : l2_policy_evict_first();
      const uint64_t pol_b = p.b_keep ? l2_policy_evict_last() : l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;
      bool ok = true;
      Unit u;
      for (int i = 0; ok && unit_at(p, num_tiles, num_kb, i, u, pair, npairs); ++i) {
        int m0, n0;
        tile_origin(p, u.tile, num_m, num_n, 2 * BM, BN, m0, n0);
        const bool nlo = n0 < p.n_split;
        const int by = (nlo ? n0 : n0 - p.n_split) + static_cast<int>(rank) * (BN / 2);
        const int my_m = m0 + static_cast<int>(rank) * BM;
        for (int t = 0; t < u.kb1 - u.kb0; ++t) {
          const int kb = unit_kb(u, i, t);
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          const int k = kb * BK;
          const bool klo = k < p.k_split;
          const int kx = klo ? k : k - p.k_split;
          const uint32_t leader_full = cluster_map(&full_bar[stage], 0);
          if (rank == 0) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::kStageBytes);
          const CUtensorMap* amap = klo ? &p.a0 : &p.a1;
          const CUtensorMap* bmap = (nlo && klo) ? &p.b0 : &p.b1;
          if constexpr (kAmn) {
#pragma unroll
            for (int h = 0; h < BM / 64; ++h)
              tma_load_2d_pair(stage_a(stage) + h * kMnBlock, amap, leader_full, my_m + 64 * h,
                               kx, pol);
          } else {
            tma_load_2d_pair(stage_a(stage), amap, leader_full, kx, my_m, pol);
          }
          if constexpr (kBmn) {
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d_pair(stage_b(stage) + h * kMnBlock, bmap, leader_full, by + 64 * h, kx,
                               pol_b);
          } else {
            tma_load_2d_pair(stage_b(stage), bmap, leader_full, kx, by, pol_b);
          }
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Unwinding: let every copy this thread issued land before the CTA
        // (and its shared memory) goes away.  Rank 0 waits for its stages;
        // rank 1's completions go to rank 0, so it gives them 100 us.
        volatile int no_abort = 0;
        if (rank == 0) {
          for (int s = 0; s < NS; ++s)
            if (armed & (1u << s))
              mbar_wait(&full_bar[s], (armed_parity >> s) & 1u, &no_abort, p.status);
        } else {
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 100000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ----------------------------------------------------- MMA issuer --
      constexpr uint32_t idesc =
          (FP8 ? umma_idesc_e4m3(2 * BM, BN) : umma_idesc_bf16(2 * BM, BN)) |
          (kAmn ? 1u << 15 : 0u) | (kBmn ? 1u << 16 : 0u);
      constexpr uint64_t kStepA = kAmn ? 128 : 2;
      constexpr uint64_t kStepB = kBmn ? 128 : 2;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      Unit u;
      for (int i = 0; ok && unit_at(p, num_tiles, num_kb, i, u, pair, npairs); ++i) {
        const int acc = i & 1;
        const uint32_t acc_phase = (i >> 1) & 1;
        if (!mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int t = 0; t < u.kb1 - u.kb0; ++t) {
          if (!mbar_wait_cluster(&full_bar[stage], phase, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = kAmn ? sw128_mnmajor_desc(smem_addr(stage_a(stage)), kMnBlock)
                                      : sw128_kmajor_desc(smem_addr(stage_a(stage)));
          const uint64_t bdesc = kBmn ? sw128_mnmajor_desc(smem_addr(stage_b(stage)), kMnBlock)
                                      : sw128_kmajor_desc(smem_addr(stage_b(stage)));
#pragma unroll
          for (int kk = 0; kk < kMmasPerBlock; ++kk) {
            const uint32_t accum = (t != 0 || kk != 0) ? 1u : 0u;
            if constexpr (FP8)
              umma_e4m3_pair(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, idesc, accum);
            else
              umma_bf16_pair(d_tmem, adesc + kStepA * kk, bdesc + kStepB * kk, idesc, accum);
          }
          umma_commit_pair(&empty_bar[stage], 0x3);
          if (++stage == NS) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(&tfull_bar[acc], 0x3);
      }
      // Every MMA this thread issued completes before TMEM is released in
      // either CTA.
      umma_commit_pair(done_bar, 0x3);
      volatile int no_abort = 0;
      mbar_wait(done_bar, 0, &no_abort, p.status);
    } else if (lane == 0) {
      // The pair's MMAs read this CTA's shared memory and write its TMEM:
      // wait for the last of them (rank 0 always commits this barrier).
      volatile int no_abort = 0;
      mbar_wait(done_bar, 0, &no_abort, p.status);
    }
  } else {
    // --------------------------------------------------------- epilogue --
    const int quarter = warp & 3;
    const int row_local = quarter * 32 + lane;
    float* f32_stage = reinterpret_cast<float*>(smem + NS * C::kStageBytes + C::kBarBytes) +
                       quarter * 32 * kF32Pad;
    Unit u;
    for (int i = 0; unit_at(p, num_tiles, num_kb, i, u, pair, npairs); ++i) {
      const int acc_buf = i & 1;
      const uint32_t acc_phase = (i >> 1) & 1;
      if (!mbar_wait_cluster_warp(&tfull_bar[acc_buf], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      int m0, n0;
      tile_origin(p, u.tile, num_m, num_n, 2 * BM, BN, m0, n0);
      const int prow = static_cast<int>(rank) * BM + row_local;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc_buf * BN);
      epilogue_unit<BN, EPI, FP8, 2 * BM, kStage>(
          p, u, m0 + prow, prow, (u.slot / p.split_s) * 8 + static_cast<int>(rank) * 4 + quarter,
          t_row, n0, lane, f32_stage);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_map(&tempty_bar[acc_buf], 0));
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // nothing of either CTA still signals the other
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <int EPI, int LAYOUT, bool FP8 = false>
cudaError_t launch_pair(const GemmArgs& a, cudaStream_t stream) {
  using C = PairCfg<staged_f32<EPI, LAYOUT>(), pair_stages<EPI>()>;
  auto kern = gemm_pair_kernel<EPI, LAYOUT, FP8>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  if (a.grid % 2) return cudaErrorInvalidValue;
  kern<<<a.grid, kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

template <int BN, int EPI, bool FP8, int LAYOUT>
cudaError_t launch_typed(const GemmArgs& a, cudaStream_t stream) {
  using C = Cfg<BN, staged_f32<EPI, LAYOUT>()>;
  auto kern = gemm_kernel<BN, EPI, FP8, LAYOUT>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kern<<<a.grid, kThreads, C::kSmemBytes, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

GemmPlan plan_gemm(int64_t tiles, int64_t num_kb, int sms, int block_n, int rows) {
  GemmPlan g;
  g.grid = static_cast<int>(tiles < sms ? tiles : sms);
  g.split_r = 0;
  g.split_s = 1;
  // Remainder tiles of the last, partial wave (all tiles if fewer than SMs).
  const int64_t r = tiles - (tiles / sms) * sms;
  if (r > 0) {
    int64_t s = sms / r;
    const int64_t s_k = num_kb / kMinSplitKBlocks;  // each piece keeps >= kMinSplitKBlocks
    if (s_k < s) s = s_k;
    if (s >= 2) {
      g.split_r = static_cast<int>(r);
      g.split_s = static_cast<int>(s);
      if (tiles < sms) g.grid = static_cast<int>(r * s);
    }
  }
  g.partial_bytes = static_cast<size_t>(g.split_r) * g.split_s * rows * block_n * sizeof(float);
  g.counter_bytes = static_cast<size_t>(g.split_r) * (rows / 32) * sizeof(unsigned);
  return g;
}

namespace {

template <int EPI, bool FP8, int LAYOUT>
cudaError_t launch_bn(const GemmArgs& a, cudaStream_t stream) {
  switch (a.block_n) {
    case 256: return launch_typed<256, EPI, FP8, LAYOUT>(a, stream);
    case 128: return launch_typed<128, EPI, FP8, LAYOUT>(a, stream);
    case 64: return launch_typed<64, EPI, FP8, LAYOUT>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream) {
  if (a.split_s >= 2 && a.split_r > 0) {
    cudaError_t e =
        cudaMemsetAsync(a.counters, 0, a.split_r * (a.pair ? 8 : 4) * sizeof(unsigned), stream);
    if (e != cudaSuccess) return e;
  }
  if (a.pair) {  // 256-wide N tiles on CTA pairs
    if (a.block_n != kPairBN) return cudaErrorInvalidValue;
    if (a.fp8) {
      if (a.layout != kLayoutKK) return cudaErrorInvalidValue;
      if (a.epilogue == kEpiQkvGelu) return launch_pair<kEpiQkvGelu, kLayoutKK, true>(a, stream);
      if (a.epilogue == kEpiResidual) return launch_pair<kEpiResidual, kLayoutKK, true>(a, stream);
      return cudaErrorInvalidValue;
    }
    if (a.layout == kLayoutKK && a.epilogue == kEpiQkvGelu)
      return launch_pair<kEpiQkvGelu, kLayoutKK>(a, stream);
    if (a.layout == kLayoutKK && a.epilogue == kEpiResidual)
      return launch_pair<kEpiResidual, kLayoutKK>(a, stream);
    if (a.layout == kLayoutKN && a.epilogue == kEpiDgelu)
      return launch_pair<kEpiDgelu, kLayoutKN>(a, stream);
    if (a.layout == kLayoutKN && a.epilogue == kEpiF32)
      return launch_pair<kEpiF32, kLayoutKN>(a, stream);
    if (a.layout == kLayoutNN && a.epilogue == kEpiF32)
      return launch_pair<kEpiF32, kLayoutNN>(a, stream);
    return cudaErrorInvalidValue;
  }
  // The instantiated (epilogue, operand type, layout) combinations: the
  // forward GEMMs (bf16 and e4m3, K-major) and the backward GEMMs (bf16).
  if (a.layout == kLayoutKK) {
    if (a.epilogue == kEpiQkvGelu)
      return a.fp8 ? launch_bn<kEpiQkvGelu, true, kLayoutKK>(a, stream)
                   : launch_bn<kEpiQkvGelu, false, kLayoutKK>(a, stream);
    if (a.epilogue == kEpiResidual)
      return a.fp8 ? launch_bn<kEpiResidual, true, kLayoutKK>(a, stream)
                   : launch_bn<kEpiResidual, false, kLayoutKK>(a, stream);
    return cudaErrorInvalidValue;
  }
  if (a.fp8) return cudaErrorInvalidValue;
  if (a.layout == kLayoutKN) {
    if (a.epilogue == kEpiDgelu) return launch_bn<kEpiDgelu, false, kLayoutKN>(a, stream);
    if (a.epilogue == kEpiF32) return launch_bn<kEpiF32, false, kLayoutKN>(a, stream);
    return cudaErrorInvalidValue;
  }
  if (a.layout == kLayoutNN && a.epilogue == kEpiF32)
    return launch_bn<kEpiF32, false, kLayoutNN>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ptb
