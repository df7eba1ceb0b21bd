// Causal sliding-window attention (SWA) on tcgen05 tensor cores, banded and
// flash-style.
//
// Every token attends to a fixed window of w positions, so the cost is
// O(s*w) rather than O(s*s) (MegaScale study notes, ch.2 §2.2, SWA row);
// FlashAttention-2 is the fused attention operator the notes list (§2.5,
// Table 3).  Row i attends to keys max(0, i-w+1) .. i (causal, self-inclusive).
//
// One CTA per (128-query tile, head, batch entry), 192 threads:
//   warp 0      TMA: the Q tile once, then the 64-key K and V tiles that
//               intersect the band [q0 - w + 1, q0 + 127] (diagonal tile
//               first) into a 3-stage ring.  d < 128 is read as 64-wide
//               boxes; columns past d are zero-filled by TMA.
//   warp 1      owns TMEM; one thread issues tcgen05.mma:
//                 S_j  = Q K_j^T       (M 128, N 64, K d)   -> TMEM, 2 buffers
//                 PV_j = P_j V_j       (M 128, N d, K 64)   -> TMEM, 2 buffers
//               in the order S_0, S_1, PV_0, S_2, PV_1, ... so the softmax of
//               one tile overlaps the tensor work of its neighbours.  V is
//               used in place as an MN-major operand.
//   warps 2..5  one query row per thread (TMEM lane = row): read the row of
//               S_j, mask only on tiles that cross the band's edges, online
//               softmax in the log2 domain (running max m and sum l in
//               registers; no cross-thread reductions), write the bf16 row of
//               P_j into shared memory in the 128-byte-swizzled layout the
//               MMA reads, then fold PV_j into the fp32 output row kept in
//               registers: O = O * alpha_j + PV_j.  Finally O / l -> bf16.
// Every mbarrier wait is bounded (see mbar_wait); on a timeout all roles
// unwind, wait for their own copies and MMAs, free TMEM and return.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int BQ = 128;  // query rows per CTA (= MMA M)
constexpr int BKV = 64;  // keys per K/V tile (= MMA N of S, K of PV)
constexpr int NS = 3;    // K/V stages
constexpr int kThreads = 192;

template <int D>
struct SwaCfg {
  static constexpr int kAtoms = (D + 63) / 64;     // 64-wide column blocks of d
  static constexpr int kQBytes = kAtoms * BQ * 128;
  static constexpr int kKVBytes = kAtoms * BKV * 128;  // one of K or V, one stage
  static constexpr int kPBytes = BQ * BKV * 2;        // one P buffer
  static constexpr int kSmemBytes = kQBytes + NS * 2 * kKVBytes + 2 * kPBytes + 256 + 1024;
  static constexpr int kTmemS = 0;                    // 2 x 64 columns
  static constexpr int kTmemPV = 2 * BKV;             // 2 x D columns
  static constexpr int kTmemCols = (2 * BKV + 2 * D) <= 256 ? 256 : 512;
};

struct SwaParams {
  CUtensorMap tq, tk, tv;  // 4-D maps {d, dim1, dim2, batch}; boxes {64, ., ., 1}
  SwaArgs a;
  int seq_dim;             // 1 or 2: which map dimension is the sequence
};

// Coordinates of (column block x, head h, row t, batch b) in a 4-D map whose
// dims 1 and 2 are (head, seq) or (seq, head).
__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                         int h, int t, int b, int seq_dim) {
  if (seq_dim == 2)
    tma_load_4d(dst, map, bar, x, h, t, b);
  else
    tma_load_4d(dst, map, bar, x, t, h, b);
}

template <int D, bool COUNTS>
__global__ void __launch_bounds__(kThreads, 1) swa_tc_kernel(const __grid_constant__ SwaParams P) {
  using C = SwaCfg<D>;
  const SwaArgs& a = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + C::kQBytes;                 // [NS][kKVBytes]
  uint8_t* sV = sK + NS * C::kKVBytes;           // [NS][kKVBytes]
  uint8_t* sP = sV + NS * C::kKVBytes;           // [2][kPBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * C::kPBytes);
  uint64_t* q_full = bars;
  uint64_t* kv_full = q_full + 1;       // [NS]
  uint64_t* kv_empty = kv_full + NS;    // [NS]
  uint64_t* s_full = kv_empty + NS;     // [2]
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* pv_full = p_full + 2;       // [2]
  uint64_t* pv_empty = pv_full + 2;     // [2]
  uint64_t* done_bar = pv_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = blockIdx.x * BQ;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int seq = a.seq;
  const int window = a.window;

  // Key tiles intersecting the band of this query tile, walked downwards.
  const int k_first = max(0, q0 - window + 1);
  const int k_last = min(seq - 1, q0 + BQ - 1);
  const int kt_hi = k_last / BKV;
  const int n_tiles = kt_hi - k_first / BKV + 1;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 4);
      mbar_init(&pv_full[i], 1);
      mbar_init(&pv_empty[i], 4);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&P.tq);
    tma_prefetch_desc(&P.tk);
    tma_prefetch_desc(&P.tv);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA --
    if (lane == 0) {
      bool ok = true;
      uint32_t armed = 0, armed_parity = 0;
      mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
      for (int at = 0; at < C::kAtoms; ++at)
        tma_rows(sQ + at * BQ * 128, &P.tq, q_full, at * 64, h, q0, b, P.seq_dim);
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const int key0 = (kt_hi - j) * BKV;
        mbar_arrive_expect_tx(&kv_full[st], 2 * C::kKVBytes);
#pragma unroll
        for (int at = 0; at < C::kAtoms; ++at) {
          tma_rows(sK + st * C::kKVBytes + at * BKV * 128, &P.tk, &kv_full[st], at * 64, h, key0,
                   b, P.seq_dim);
          tma_rows(sV + st * C::kKVBytes + at * BKV * 128, &P.tv, &kv_full[st], at * 64, h, key0,
                   b, P.seq_dim);
        }
        armed |= 1u << st;
        armed_parity = (armed_parity & ~(1u << st)) | (ph << st);
      }
      volatile int no_abort = 0;
      if (!ok) {
        for (int s = 0; s < NS; ++s)
          if (armed & (1u << s))
            mbar_wait(&kv_full[s], (armed_parity >> s) & 1u, &no_abort, a.status);
      }
      // The Q copy must have landed before the CTA can go away.
      mbar_wait(q_full, 0, &no_abort, a.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA --
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(BQ, BKV);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(BQ, D) | (1u << 16);  // B (V) MN-major
      bool ok = mbar_wait(q_full, 0, abort_flag, a.status);
      tc_fence_after();
      const uint32_t q_addr = smem_addr(sQ);
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int st = j % NS;
          if (!mbar_wait(&kv_full[st], (j / NS) & 1, abort_flag, a.status)) break;
          tc_fence_after();
          const uint32_t k_addr = smem_addr(sK + st * C::kKVBytes);
          const uint32_t d_tmem = tmem + C::kTmemS + (j & 1) * BKV;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t at = kk / 4, off = (kk % 4) * 32;
            umma_bf16_ss(d_tmem, sw128_kmajor_desc(q_addr + at * BQ * 128 + off),
                         sw128_kmajor_desc(k_addr + at * BKV * 128 + off), idesc_s, kk > 0);
          }
          umma_commit(&s_full[j & 1]);
        }
        if (j >= 1) {
          const int t = j - 1;
          const int pb = t & 1;
          const uint32_t ph = (t >> 1) & 1;
          if (!mbar_wait(&p_full[pb], ph, abort_flag, a.status) ||
              !mbar_wait(&pv_empty[pb], ph ^ 1u, abort_flag, a.status))
            break;
          tc_fence_after();
          const int st = t % NS;
          const uint32_t p_addr = smem_addr(sP + pb * C::kPBytes);
          const uint32_t v_addr = smem_addr(sV + st * C::kKVBytes);
          const uint32_t d_tmem = tmem + C::kTmemPV + pb * D;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            umma_bf16_ss(d_tmem, sw128_kmajor_desc(p_addr + kk * 32),
                         sw128_mnmajor_desc(v_addr + kk * 16 * 128, BKV * 128), idesc_pv, kk > 0);
          umma_commit(&pv_full[pb]);
          umma_commit(&kv_empty[st]);
        }
      }
      umma_commit(done_bar);
      volatile int no_abort = 0;
      mbar_wait(done_bar, 0, &no_abort, a.status);
    }
  } else {
    // --------------------------------------------------------- softmax --
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row in the tile = TMEM lane
    const int i = q0 + r;               // query position
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float o[D];
#pragma unroll
    for (int c = 0; c < D; ++c) o[c] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    float alpha_ring[2] = {0.f, 0.f};
    int cnt = 0;
    bool ok = true;

    auto fold_pv = [&](int t) -> bool {
      const int pb = t & 1;
      if (!mbar_wait(&pv_full[pb], (t >> 1) & 1, abort_flag, a.status)) return false;
      tc_fence_after();
      const float al = alpha_ring[pb];
      const uint32_t base = tmem + lane_base + C::kTmemPV + pb * D;
      if constexpr (D % 32 == 0) {
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(base + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[c + e] = o[c + e] * al + __uint_as_float(v[e]);
        }
      } else {
        uint32_t v[16];
        tmem_ld_32x32b_x16(base, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) o[e] = o[e] * al + __uint_as_float(v[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pv_empty[pb]);
      return true;
    };

    for (int j = 0; j < n_tiles; ++j) {
      const int sb = j & 1;
      if (!mbar_wait(&s_full[sb], (j >> 1) & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float x[BKV];
#pragma unroll
      for (int c = 0; c < BKV; c += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_base + C::kTmemS + sb * BKV + c, v);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c + e] = __uint_as_float(v[e]) * a.scale_log2;
      }
      const int key0 = (kt_hi - j) * BKV;
      const bool interior = (key0 + BKV - 1 <= i) && (key0 >= i - window + 1);
      if (!interior) {
#pragma unroll
        for (int e = 0; e < BKV; ++e) {
          const int kj = key0 + e;
          const bool keep = (kj <= i) && (kj > i - window);
          x[e] = keep ? x[e] : -INFINITY;
          if (COUNTS) cnt += keep ? 1 : 0;
        }
      } else if (COUNTS) {
        cnt += BKV;
      }
      float mx = -INFINITY;
#pragma unroll
      for (int e = 0; e < BKV; ++e) mx = fmaxf(mx, x[e]);
      const float m_new = fmaxf(m_run, mx);
      const float m_ref = m_new == -INFINITY ? 0.f : m_new;
      alpha_ring[sb] = fast_exp2(m_run - m_ref);
      m_run = m_new;
      float rs = 0.f;
      uint32_t pk[BKV / 2];
#pragma unroll
      for (int e = 0; e < BKV; e += 2) {
        const float p0 = fast_exp2(x[e] - m_ref);
        const float p1 = fast_exp2(x[e + 1] - m_ref);
        rs += p0 + p1;
        pk[e / 2] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha_ring[sb] + rs;
      // Row r of P_j, 64 keys = one 128-byte swizzled row: 16-byte chunk c
      // of the row sits at chunk position c ^ (r % 8).
      uint8_t* prow = sP + sb * C::kPBytes + r * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[sb]);
      if (j >= 1 && !fold_pv(j - 1)) {
        ok = false;
        break;
      }
    }
    if (ok && n_tiles > 0) ok = fold_pv(n_tiles - 1);

    if (ok && i < seq) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = a.o + b * a.o_sb + h * a.o_sh + static_cast<int64_t>(i) * a.o_ss;
#pragma unroll
      for (int c = 0; c < D; c += 8) {
        *reinterpret_cast<uint4*>(orow + c) =
            make_uint4(pack_bf16x2(o[c] * inv, o[c + 1] * inv),
                       pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv),
                       pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv),
                       pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv));
      }
      if (COUNTS) a.counts[(static_cast<int64_t>(b) * a.heads + h) * seq + i] = cnt;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool COUNTS>
cudaError_t launch_typed(const SwaParams& prm, cudaStream_t stream) {
  using C = SwaCfg<D>;
  auto kern = swa_tc_kernel<D, COUNTS>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  const dim3 grid((prm.a.seq + BQ - 1) / BQ, prm.a.heads, prm.a.batch);
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(prm);
  return cudaGetLastError();
}

template <bool COUNTS>
cudaError_t dispatch(const SwaParams& prm, cudaStream_t stream) {
  switch (prm.a.head_dim) {
    case 16: return launch_typed<16, COUNTS>(prm, stream);
    case 32: return launch_typed<32, COUNTS>(prm, stream);
    case 64: return launch_typed<64, COUNTS>(prm, stream);
    case 96: return launch_typed<96, COUNTS>(prm, stream);
    case 128: return launch_typed<128, COUNTS>(prm, stream);
  }
  return cudaErrorInvalidValue;
}

// 4-D map {d, heads, seq, batch} or {d, seq, heads, batch} (strides kept in
// increasing order) over one of q, k, v; boxes of 64 columns x `rows` rows.
bool swa_map(CUtensorMap* map, const __nv_bfloat16* base, int64_t sb, int64_t sh, int64_t ss,
             const SwaArgs& a, int rows, int* seq_dim) {
  const bool heads_first = sh <= ss;
  const uint64_t dims[4] = {static_cast<uint64_t>(a.head_dim),
                            static_cast<uint64_t>(heads_first ? a.heads : a.seq),
                            static_cast<uint64_t>(heads_first ? a.seq : a.heads),
                            static_cast<uint64_t>(a.batch)};
  const uint64_t strides[3] = {static_cast<uint64_t>(heads_first ? sh : ss) * 2,
                               static_cast<uint64_t>(heads_first ? ss : sh) * 2,
                               static_cast<uint64_t>(sb) * 2};
  const uint32_t box[4] = {64, heads_first ? 1u : static_cast<uint32_t>(rows),
                           heads_first ? static_cast<uint32_t>(rows) : 1u, 1};
  *seq_dim = heads_first ? 2 : 1;
  return make_tensor_map(map, base, 4, dims, strides, box);
}

}  // namespace

cudaError_t launch_swa(const SwaArgs& a, cudaStream_t stream) {
  if (a.seq <= 0 || a.batch <= 0 || a.heads <= 0) return cudaSuccess;
  if (a.batch > 65535 || a.heads > 65535) return cudaErrorInvalidValue;
  SwaParams prm;
  prm.a = a;
  int sd_q = 0, sd_k = 0, sd_v = 0;
  // With one batch entry the batch stride is never used; a non-positive one
  // is replaced by a harmless positive value for the tensor map.
  auto bstride = [&](int64_t sb, int64_t sh, int64_t ss) -> int64_t {
    if (sb > 0) return sb;
    return (sh > ss ? sh : ss) * (a.heads > a.seq ? a.heads : a.seq);
  };
  if (!swa_map(&prm.tq, a.q, bstride(a.q_sb, a.q_sh, a.q_ss), a.q_sh, a.q_ss, a, BQ, &sd_q) ||
      !swa_map(&prm.tk, a.k, bstride(a.k_sb, a.k_sh, a.k_ss), a.k_sh, a.k_ss, a, BKV, &sd_k) ||
      !swa_map(&prm.tv, a.v, bstride(a.v_sb, a.v_sh, a.v_ss), a.v_sh, a.v_ss, a, BKV, &sd_v))
    return cudaErrorInvalidValue;
  if (sd_q != sd_k || sd_q != sd_v) return cudaErrorInvalidValue;
  prm.seq_dim = sd_q;
  return a.counts ? dispatch<true>(prm, stream) : dispatch<false>(prm, stream);
}

}  // namespace ptb
