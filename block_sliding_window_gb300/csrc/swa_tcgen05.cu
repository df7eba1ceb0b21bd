// Causal sliding-window attention (SWA) on tcgen05 tensor cores, banded and
// flash-style.
//
// Every token attends to a fixed window of w positions, so the cost is
// O(s*w) rather than O(s*s) (MegaScale study notes, ch.2 §2.2, SWA row);
// FlashAttention-2 is the fused attention operator the notes list (§2.5,
// Table 3).  Row i attends to keys max(0, i-w+1) .. i (causal, self-inclusive).
//
// Persistent kernel: one CTA per SM walks work items = (256-query block,
// head, batch entry).  An item is two 128-row query tiles X = 0, 1 that share
// every K/V tile.  416 threads:
//   warp 0      TMA: the two Q tiles of an item, then the 64-key K and V
//               tiles intersecting the item's band [q0 - w + 1, q0 + 255]
//               (diagonal tile first) into a ring of 4 stages (d > 64; 6 for
//               d <= 64) that runs on across items.  d < 128 is read as
//               64-wide boxes; columns past d are zero-filled by TMA.  (An L2
//               prefetch of the tiles four positions ahead was measured
//               slightly slower.)
//   warps 1..4  four MMA-issuing threads, two per query tile X (warp 1 also
//               owns TMEM: 512 columns, per query tile two 64-column score
//               buffers and a d-column output accumulator):
//                 warps 1, 2   S_X = Q_X K_j^T   (M 128, N 64, K d)
//                 warps 3, 4   O_X += P_X V_j    (M 128, N d, K 64; P read
//                                               from TMEM, V read in place
//                                               as an MN-major operand)
//               skipping any tile that lies wholly outside the band of X.
//               Score tile n + 2 reuses the buffer of tile n, so it is issued
//               only once P V n has finished.  A single thread issues at most
//               one tcgen05 instruction (MMA or commit) every ~75 cycles,
//               whatever the MMA's N (measured), which is slower than the
//               tensor pipe runs these small MMAs; four instruction streams
//               keep it fed.
//   warps 5..12 two softmax warpgroups, one per query tile, one query row per
//               thread (TMEM lane = row).  Per tile: read the score row, mask
//               only on band-edge tiles, exponentiate in the log2 domain
//               against a reference max that is raised only when the row max
//               exceeds it by more than 8 (so P <= 2^8 in bf16); raising it
//               rescales the running sum and the output row in TMEM.  The
//               bf16 P row is written back into TMEM over the scores it came
//               from (row = lane, two keys per column), where the P V MMA
//               reads it as its A operand: P never passes through shared
//               memory, and a softmax warp waits for a P V only to rescale O.
//               At the end of an item O / l -> bf16, staged per warp in 4 KB
//               of shared memory (32 rows x 64 columns) and written with a TMA
//               store: 55.6 -> 52.5 us on the operator, against 16-byte
//               stores from registers (each warp store then touched 32 rows).
// Every mbarrier wait is bounded (see mbar_wait); on a timeout all roles
// unwind, wait for their own copies and MMAs, free TMEM and return.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int BQ = 128;       // rows per query tile (= MMA M)
constexpr int QT = 2;         // query tiles per work item
constexpr int BKV = 64;       // keys per K/V tile (= MMA N of S, K of PV)
constexpr int kThreads = 416;
constexpr float kRescaleLog2 = 8.0f;  // raise the reference max only past 2^8

template <int D>
struct SwaCfg {
  static constexpr int kAtoms = (D + 63) / 64;          // 64-wide column blocks of d
  static constexpr int kQTileBytes = kAtoms * BQ * 128;
  static constexpr int kKVBytes = kAtoms * BKV * 128;   // one of K or V, one stage
  // P never touches shared memory: it overwrites its own score buffer in TMEM.
  // Output staging: one 32-row x 64-column block (4 KB) per softmax warp.
  static constexpr int kOStageBytes = 32 * 128;
  static constexpr int kFixed = QT * kQTileBytes + 4 * QT * kOStageBytes + 512 + 1024;
  static constexpr int kNSFit = (227 * 1024 - kFixed) / (2 * kKVBytes);
  static constexpr int kNS = kNSFit < 6 ? kNSFit : 6;  // K/V stages
  static constexpr int kSmemBytes = kFixed + kNS * 2 * kKVBytes;
  static constexpr int kTmemCols = 512;
  __host__ __device__ static constexpr int s_col(int x, int buf) { return x * 256 + buf * BKV; }
  __host__ __device__ static constexpr int o_col(int x) { return x * 256 + 2 * BKV; }
};

struct SwaParams {
  CUtensorMap tq, tk, tv;  // 4-D maps {d, dim1, dim2, batch}; boxes {64, ., ., 1}
  CUtensorMap to;          // the output, boxes of 64 columns x 32 rows
  int o_seq_dim;           // which dimension of `to` is the sequence
  SwaArgs a;
  int seq_dim;             // 1 or 2: which map dimension is the sequence
  int num_items, q_blocks;
};

__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                         int h, int t, int b, int seq_dim) {
  if (seq_dim == 2)
    tma_load_4d(dst, map, bar, x, h, t, b);
  else
    tma_load_4d(dst, map, bar, x, t, h, b);
}

struct Item {
  int q0, h, b, kt_hi, n_tiles;
};

// Items are ordered by query block, last (most key tiles) first, and dealt
// to the CTAs in snake order (snake_item), which evens out the per-CTA work.
__device__ __forceinline__ Item decode_item(const SwaParams& P, int item) {
  Item it;
  const int per_block = P.a.heads * P.a.batch;
  const int qb = P.q_blocks - 1 - item / per_block;
  const int rest = item % per_block;
  it.h = rest % P.a.heads;
  it.b = rest / P.a.heads;
  it.q0 = qb * (QT * BQ);
  const int k_first = max(0, it.q0 - P.a.window + 1);
  const int k_last = min(P.a.seq - 1, it.q0 + QT * BQ - 1);
  it.kt_hi = k_last / BKV;
  it.n_tiles = it.kt_hi - k_first / BKV + 1;
  return it;
}

// Does key tile [key0, key0 + 63] meet the band of query tile x of the item?
__device__ __forceinline__ bool tile_relevant(const SwaParams& P, const Item& it, int x,
                                              int key0) {
  const int r0 = it.q0 + x * BQ;
  if (r0 >= P.a.seq) return false;
  const int r1 = min(r0 + BQ - 1, P.a.seq - 1);
  return key0 <= r1 && key0 + BKV - 1 >= r0 - P.a.window + 1;
}

template <int D, bool COUNTS>
__global__ void __launch_bounds__(kThreads, 1) swa_tc_kernel(const __grid_constant__ SwaParams P) {
  using C = SwaCfg<D>;
  constexpr int NS = C::kNS;
  const SwaArgs& a = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem;                               // [QT][kQTileBytes]
  uint8_t* sK = sQ + QT * C::kQTileBytes;           // [NS][kKVBytes]
  uint8_t* sV = sK + NS * C::kKVBytes;              // [NS][kKVBytes]
  uint8_t* sO = sV + NS * C::kKVBytes;              // [4 * QT][kOStageBytes]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sO + 4 * QT * C::kOStageBytes);
  uint64_t* q_full = bars;
  uint64_t* q_empty = q_full + 1;
  uint64_t* kv_full = q_empty + 1;      // [NS]
  uint64_t* kv_empty = kv_full + NS;    // [NS]
  uint64_t* s_full = kv_empty + NS;     // [QT][2]
  uint64_t* p_full = s_full + 2 * QT;   // [QT][2]: P in score buffer 0 / 1
  uint64_t* pv_done = p_full + 2 * QT;  // [QT][2]: P V of score buffer 0 / 1
  uint64_t* done_bar = pv_done + 2 * QT;  // [2 * QT]: one per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 2 * QT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, QT);  // both score threads release Q
    for (int s = 0; s < NS; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], QT);  // each query tile releases every K/V stage
    }
    for (int x = 0; x < QT; ++x) {
      mbar_init(&s_full[2 * x], 1);
      mbar_init(&s_full[2 * x + 1], 1);
      mbar_init(&p_full[2 * x], 4);
      mbar_init(&p_full[2 * x + 1], 4);
      mbar_init(&pv_done[2 * x], 1);
      mbar_init(&pv_done[2 * x + 1], 1);
    }
    for (int t = 0; t < 2 * QT; ++t) mbar_init(&done_bar[t], 1);
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
      uint32_t kv_count = 0, q_count = 0;
      uint32_t armed = 0, armed_parity = 0;
      for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
        const Item it = decode_item(P, item);
        if (!mbar_wait(q_empty, (q_count & 1) ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        const bool has_b = it.q0 + BQ < a.seq;
        mbar_arrive_expect_tx(q_full, (has_b ? 2 : 1) * C::kQTileBytes);
        for (int x = 0; x < (has_b ? 2 : 1); ++x)
#pragma unroll
          for (int at = 0; at < C::kAtoms; ++at)
            tma_rows(sQ + x * C::kQTileBytes + at * BQ * 128, &P.tq, q_full, at * 64, it.h,
                     it.q0 + x * BQ, it.b, P.seq_dim);
        ++q_count;
        for (int j = 0; j < it.n_tiles; ++j, ++kv_count) {
          const int st = kv_count % NS;
          const uint32_t ph = (kv_count / NS) & 1;
          if (!mbar_wait(&kv_empty[st], ph ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const int key0 = (it.kt_hi - j) * BKV;
          mbar_arrive_expect_tx(&kv_full[st], 2 * C::kKVBytes);
#pragma unroll
          for (int at = 0; at < C::kAtoms; ++at) {
            tma_rows(sK + st * C::kKVBytes + at * BKV * 128, &P.tk, &kv_full[st], at * 64, it.h,
                     key0, it.b, P.seq_dim);
            tma_rows(sV + st * C::kKVBytes + at * BKV * 128, &P.tv, &kv_full[st], at * 64, it.h,
                     key0, it.b, P.seq_dim);
          }
          armed |= 1u << st;
          armed_parity = (armed_parity & ~(1u << st)) | (ph << st);
        }
      }
      // Let every copy this thread issued land before the CTA goes away.
      volatile int no_abort = 0;
      for (int s = 0; s < NS; ++s)
        if (armed & (1u << s))
          mbar_wait(&kv_full[s], (armed_parity >> s) & 1u, &no_abort, a.status);
      if (q_count > 0) mbar_wait(q_full, (q_count - 1) & 1, &no_abort, a.status);
    }
  } else if (warp <= 2 * QT) {
    // ------------------------------------------------------------- MMA --
    // Four issuing threads: for each query tile X one issues its scores
    // (warps 1, 2) and one its P V products (warps 3, 4).  A single thread
    // issues at most one tcgen05 instruction (MMA or commit) every ~75
    // cycles whatever the MMA's N, slower than the tensor pipe runs these
    // small MMAs; split four ways the instruction streams keep it fed, and
    // each query tile's chain S -> softmax -> P V -> S overlaps across them.
    const bool pv_role = warp > QT;
    const int x = pv_role ? warp - 1 - QT : warp - 1;
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(BQ, BKV);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(BQ, D) | (1u << 16);  // B (V) MN-major
      bool ok = true;
      uint32_t kv_count = 0, q_count = 0, issued = 0;
      const uint32_t qx = smem_addr(sQ + x * C::kQTileBytes);
      for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
        const Item it = decode_item(P, item);
        if (!pv_role) {
          if (!mbar_wait(q_full, q_count & 1, abort_flag, a.status)) break;
          ++q_count;
          tc_fence_after();
        }
        bool first_pv = true;
        for (int j = 0; j < it.n_tiles; ++j) {
          // Stage arrivals are parity waits, exact only within one phase.  A
          // score thread observes every stage in order and releases the
          // tiles outside its band itself; the P V thread releases the
          // others after their P V and waits only on those, when score tile
          // n has already observed the arrival.  So no stage is refilled
          // before both threads of a query tile have seen its last fill.
          const uint32_t kc = kv_count + j;
          const int st = kc % NS;
          const bool relevant = tile_relevant(P, it, x, (it.kt_hi - j) * BKV);
          if (!pv_role || relevant) {
            if (!mbar_wait(&kv_full[st], (kc / NS) & 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t n = issued;
          if (!pv_role) {
            if (relevant) {
              // Score buffer n % 2 still holds P number n - 2 until its P V ends.
              if (n >= 2) {
                if (!mbar_wait(&pv_done[2 * x + (n & 1)], ((n - 2) >> 1) & 1, abort_flag,
                               a.status)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
              }
              const uint32_t d_tmem = tmem + C::s_col(x, n & 1);
              const uint32_t k_addr = smem_addr(sK + st * C::kKVBytes);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t at = kk / 4, off = (kk % 4) * 32;
                umma_bf16_ss(d_tmem, sw128_kmajor_desc(qx + at * BQ * 128 + off),
                             sw128_kmajor_desc(k_addr + at * BKV * 128 + off), idesc_s, kk > 0);
              }
              umma_commit(&s_full[2 * x + (n & 1)]);
              ++issued;
            } else {
              mbar_arrive(&kv_empty[st]);  // this query tile never reads the stage
            }
            if (j == it.n_tiles - 1) umma_commit(q_empty);  // Q_X is free once these finish
          } else {
            if (relevant) {
              // P number n sits in score buffer n % 2.  Score tile n was read
              // by then, so this P V also follows every score MMA of the stage
              // by this query tile.
              if (!mbar_wait(&p_full[2 * x + (n & 1)], (n >> 1) & 1, abort_flag, a.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t p_tmem = tmem + C::s_col(x, n & 1);
              const uint32_t d_tmem = tmem + C::o_col(x);
              const uint32_t v_addr = smem_addr(sV + st * C::kKVBytes);
#pragma unroll
              for (int kk = 0; kk < BKV / 16; ++kk)  // 16 keys = 8 packed P columns
                umma_bf16_ts(d_tmem, p_tmem + kk * 8,
                             sw128_mnmajor_desc(v_addr + kk * 16 * 128, BKV * 128), idesc_pv,
                             (!first_pv || kk > 0) ? 1u : 0u);
              umma_commit(&pv_done[2 * x + (n & 1)]);
              umma_commit(&kv_empty[st]);  // this query tile is done with the stage
              ++issued;
              first_pv = false;
            }
          }
        }
        kv_count += it.n_tiles;
      }
      const int me = pv_role ? QT + x : x;
      umma_commit(&done_bar[me]);
      volatile int no_abort = 0;
      mbar_wait(&done_bar[me], 0, &no_abort, a.status);
    }
  } else {
    // --------------------------------------------------------- softmax --
    const int x = (warp - 1 - 2 * QT) >> 2;  // query tile of this warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row in the query tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t o_tmem = tmem + lane_base + C::o_col(x);
    uint32_t seen = 0;  // relevant tiles of this query tile so far (all items)
    bool ok = true;

    // P V number n of this query tile completes phase n / 2 of
    // pv_done[x][n % 2].  A parity wait is exact only while its barrier is
    // at most one phase behind or ahead of the awaited one: here P V n - 2
    // has always finished (score tile n, already read, was issued after it)
    // and P V n + 2 cannot start (it needs P n + 2 from this warpgroup).
    // One barrier for both buffers would break this: waiting for the
    // item's last P V while the one before it was still running would
    // return at once.
    auto wait_pv = [&](uint32_t n) -> bool {
      if (!mbar_wait_warp(&pv_done[2 * x + (n & 1)], (n >> 1) & 1, abort_flag, a.status))
        return false;
      tc_fence_after();
      return true;
    };

    for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
      const Item it = decode_item(P, item);
      const int i = it.q0 + x * BQ + r;  // query position of this thread
      if (it.q0 + x * BQ >= a.seq) continue;
      float m_ref = -INFINITY, l_run = 0.f;
      int cnt = 0;
      bool any_pv = false;
      for (int j = 0; j < it.n_tiles; ++j) {
        const int key0 = (it.kt_hi - j) * BKV;
        if (!tile_relevant(P, it, x, key0)) continue;
        const int buf = seen & 1;
        if (!mbar_wait_warp(&s_full[2 * x + buf], (seen >> 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Raw scores q.k: both halves of the row are loaded before one wait,
        // and the scale goes into the exponent's FMA (the row max is taken on
        // raw scores; the scale is positive).
        static_assert(BKV == 64, "two 32-column TMEM loads per score row");
        uint32_t raw0[32], raw1[32];
        tmem_ld_32x32b_x32(tmem + lane_base + C::s_col(x, buf), raw0);
        tmem_ld_32x32b_x32(tmem + lane_base + C::s_col(x, buf) + 32, raw1);
        tmem_ld_wait();
        float v[BKV];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v[e] = __uint_as_float(raw0[e]);
          v[32 + e] = __uint_as_float(raw1[e]);
        }
        const bool interior = (key0 + BKV - 1 <= i) && (key0 >= i - a.window + 1);
        if (!interior) {
#pragma unroll
          for (int e = 0; e < BKV; ++e) {
            const int kj = key0 + e;
            const bool keep = (kj <= i) && (kj > i - a.window);
            v[e] = keep ? v[e] : -INFINITY;
            if (COUNTS) cnt += keep ? 1 : 0;
          }
        } else if (COUNTS) {
          cnt += BKV;
        }
        // Packed forms keep the per-score instruction count low: one
        // three-input max per two scores, one f32x2 FMA (scale, shift) and
        // one f32x2 add (row sum) per pair; the softmax warps are bound by
        // instruction issue, not by the exponent unit.
        // Row max as a tree of depth 4 (64 -> 22 -> 8 -> 3 -> 1) rather than
        // a chain: only two softmax warps share an SMSP to hide latency.
        static_assert(BKV == 64, "max tree sized for 64 scores");
        float m1[22], m2[8];
#pragma unroll
        for (int t = 0; t < 21; ++t) m1[t] = fmax3(v[3 * t], v[3 * t + 1], v[3 * t + 2]);
        m1[21] = v[63];
#pragma unroll
        for (int t = 0; t < 7; ++t) m2[t] = fmax3(m1[3 * t], m1[3 * t + 1], m1[3 * t + 2]);
        m2[7] = m1[21];
        float mx = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
        mx *= a.scale_log2;  // row max in the log2 domain
        // Raise the reference max only when the row max passes it by 2^8.
        float alpha = 1.f;
        const bool raise = mx > m_ref + kRescaleLog2;
        if (raise) {
          alpha = fast_exp2(m_ref - mx);  // 0 while m_ref is -inf
          l_run *= alpha;
          m_ref = mx;
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const uint64_t scale2 = f2(a.scale_log2, a.scale_log2), shift2 = f2(-m_use, -m_use);
        uint64_t sum2[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};
        uint32_t pk[BKV / 2];
#pragma unroll
        for (int e = 0; e < BKV; e += 2) {
          float t0, t1;
          f2_split(f2_fma(f2(v[e], v[e + 1]), scale2, shift2), t0, t1);
          const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
          sum2[(e >> 1) & 3] = f2_add(sum2[(e >> 1) & 3], f2(p0, p1));  // four chains
          pk[e / 2] = pack_bf16x2(p0, p1);
        }
        float s0, s1;
        f2_split(f2_add(f2_add(sum2[0], sum2[1]), f2_add(sum2[2], sum2[3])), s0, s1);
        l_run += s0 + s1;
        // P (bf16 pairs) over the first 32 columns of the scores just read.
        tmem_st_32x32b_x32(tmem + lane_base + C::s_col(x, buf), pk);
        if (any_pv && __any_sync(0xffffffffu, raise)) {
          // O must hold every earlier P V of this item before it is rescaled.
          if (!wait_pv(seen - 1)) {
            tmem_st_wait();
            ok = false;
            break;
          }
          if constexpr (D % 32 == 0) {
#pragma unroll
            for (int c = 0; c < D; c += 32) {
              uint32_t o[32];
              tmem_ld_32x32b_x32(o_tmem + c, o);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
              tmem_st_32x32b_x32(o_tmem + c, o);
            }
          } else {
            uint32_t o[16];
            tmem_ld_32x32b_x16(o_tmem, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x16(o_tmem, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[2 * x + buf]);
        any_pv = true;
        ++seen;
      }
      if (!ok) break;
      // The last P V of the item, then O / l.
      if (!wait_pv(seen - 1)) {
        ok = false;
        break;
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // O / l as bf16, one 64-column block at a time: each warp writes its 32
      // rows into its own 4 KB of shared memory in the 128-byte-swizzled
      // layout of the output tensor map (16-byte chunk c of row r at
      // r * 128 + ((c ^ (r % 8)) * 16)), and its lane 0 stores the block
      // with TMA (rows past the sequence and columns past d are not
      // written).  One 32-row TMA store replaces 256 scattered 16-byte stores
      // (32 rows x 8 chunks) per block and warp.
      uint8_t* stage = sO + (x * 4 + quarter) * C::kOStageBytes;
      constexpr int kCols = D < 32 ? D : 32;  // columns per TMEM load
#pragma unroll
      for (int at = 0; at < C::kAtoms; ++at) {
        // The previous block (of this item or the last one) has left shared memory.
        if (lane == 0) bulk_wait_read();
        __syncwarp();
#pragma unroll
        for (int c = at * 64; c < min(D, at * 64 + 64); c += kCols) {
          uint32_t o[32];
          if constexpr (kCols == 32)
            tmem_ld_32x32b_x32(o_tmem + c, o);
          else
            tmem_ld_32x32b_x16(o_tmem + c, *reinterpret_cast<uint32_t(*)[16]>(&o[0]));
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < kCols; e += 8) {
            const int chunk = ((c % 64) + e) / 8;
            *reinterpret_cast<uint4*>(stage + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                make_uint4(
                    pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv),
                    pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv),
                    pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv),
                    pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int row0 = it.q0 + x * BQ + quarter * 32;
          if (P.o_seq_dim == 2)
            tma_store_4d(&P.to, stage, at * 64, it.h, row0, it.b);
          else
            tma_store_4d(&P.to, stage, at * 64, row0, it.h, it.b);
          bulk_commit_group();
        }
      }
      tc_fence_before();
      if (COUNTS && i < a.seq)
        a.counts[(static_cast<int64_t>(it.b) * a.heads + it.h) * a.seq + i] = cnt;
      // Every row attends to itself, so l_run > 0 and m_ref is finite here.
      if (a.lse && i < a.seq)
        a.lse[(static_cast<int64_t>(it.b) * a.heads + it.h) * a.seq + i] = m_ref + log2f(l_run);
    }
    // The output stores this warp issued complete before the CTA ends.
    if (lane == 0) bulk_wait_all();
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
cudaError_t launch_typed(const SwaParams& prm, int grid, cudaStream_t stream) {
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
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(prm);
  return cudaGetLastError();
}

template <bool COUNTS>
cudaError_t dispatch(const SwaParams& prm, int grid, cudaStream_t stream) {
  switch (prm.a.head_dim) {
    case 16: return launch_typed<16, COUNTS>(prm, grid, stream);
    case 32: return launch_typed<32, COUNTS>(prm, grid, stream);
    case 64: return launch_typed<64, COUNTS>(prm, grid, stream);
    case 96: return launch_typed<96, COUNTS>(prm, grid, stream);
    case 128: return launch_typed<128, COUNTS>(prm, grid, stream);
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
  SwaParams prm;
  prm.a = a;
  // A window of s or more is plain causal attention; clamping it keeps every
  // index expression of the kernels (a row plus the window, ...) inside int.
  if (prm.a.window > prm.a.seq) prm.a.window = prm.a.seq;
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
  int sd_o = 0;
  if (!swa_map(&prm.to, a.o, bstride(a.o_sb, a.o_sh, a.o_ss), a.o_sh, a.o_ss, a, 32, &sd_o))
    return cudaErrorInvalidValue;
  prm.o_seq_dim = sd_o;
  prm.seq_dim = sd_q;
  prm.q_blocks = (a.seq + QT * BQ - 1) / (QT * BQ);
  const int64_t items = static_cast<int64_t>(prm.q_blocks) * a.heads * a.batch;
  if (items > 0x3fffffff) return cudaErrorInvalidValue;  // item numbers stay in int
  prm.num_items = static_cast<int>(items);
  const int grid = static_cast<int>(items < a.sms ? items : a.sms);
  return a.counts ? dispatch<true>(prm, grid, stream) : dispatch<false>(prm, grid, stream);
}

}  // namespace ptb
