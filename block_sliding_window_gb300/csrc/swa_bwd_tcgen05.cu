// Backward pass of causal sliding-window attention (SWA) on tcgen05 tensor
// cores.
//
// For o_i = sum_j P_ij v_j with P = softmax over the band of q_i.k_j * scale
// (row i sees keys max(0, i-w+1) .. i; MegaScale study notes, ch.2 §2.2, SWA
// row) and an upstream gradient dO, the chain rule gives, with
// delta_i = sum_c dO_ic o_ic = sum_j P_ij (dO_i . v_j):
//   dV = P^T dO,   dP = dO V^T,   dS = P * (dP - delta),
//   dQ = scale * dS K,   dK = scale * dS^T Q.
// P is recomputed from the scores and the forward pass's per-row log-sum-exp
// (base 2): P_ij = 2^(q_i.k_j * scale * log2 e - lse2_i).
//
// Two persistent kernels, so that no gradient is summed with atomics:
//   kKV  one item = 128 keys of one (batch entry, head): stationary K and V
//        tiles, moving 64-query tiles of Q and dO over the keys' band
//          S^T  = K Q^T,   dP^T = V dO^T      (M 128 keys, N 64, K d)
//          dV  += P^T dO,  dK  += dS^T Q      (M 128, N d, K 64 queries)
//   kQ   one item = 128 queries: stationary Q and dO, moving 64-key tiles
//          S = Q K^T,  dP = dO V^T            (M 128 queries, N 64, K d)
//          dQ += dS K                         (M 128, N d, K 64 keys)
// Roles (384 threads): warp 0 TMA; warps 1, 2, 3 issue the S, dP and
// accumulate MMAs (one thread each; warp 1 owns TMEM); warps 4..11 two
// warpgroups; warp w serves the stationary rows of TMEM lane
// quarter w % 4 (one row per thread) and the tile's columns 32 * g .. +31 of
// its warpgroup g: recompute P and dS for them in fp32 and write them as
// bf16 back into TMEM over the first half of those score columns (two
// positions per column), where the accumulate MMAs read them as their A
// operand: the stationary rows are the TMEM lanes in both kernels, so P^T and
// dS^T (kKV) or dS (kQ) are lane-major as they stand.  A score buffer takes
// tile n + 2 once the accumulate MMAs of tile n have finished.  At the end of
// an item the warps read the fp32 accumulators from TMEM and store bf16
// gradients.  (With one warpgroup doing all 64 columns the
// kernels ran at 14-19% tensor activity, ~6k / 3.5k cycles per tile.)  The
// moving tiles are read twice, once as K-major and once as MN-major operands
// of the same shared-memory copy.
// Every mbarrier wait is bounded (see mbar_wait); on a timeout all roles
// unwind, wait for their own copies and MMAs, free TMEM and return.
#include "ptb_device.cuh"

namespace ptb {
namespace {

constexpr int BR = 128;  // stationary rows per item (= MMA M)
constexpr int BC = 64;   // moving rows per tile (= N of the score MMAs)
constexpr int kThreads = 384;
constexpr int kGroupCols = BC / 2;  // moving columns per softmax warpgroup
constexpr int kKV = 0;   // dK, dV kernel
constexpr int kQ = 1;    // dQ kernel

template <int D, int MODE>
struct BwdCfg {
  static constexpr int kAtoms = (D + 63) / 64;
  static constexpr int kStatBytes = kAtoms * BR * 128;  // one stationary operand
  static constexpr int kMvBytes = kAtoms * BC * 128;    // one moving operand, one stage
  // P^T / dS^T (or dS) never touch shared memory: they overwrite their own
  // score columns in TMEM, so shared memory holds only the stationary tiles
  // and the ring of moving tiles.
  static constexpr int kStageLse = MODE == kKV ? 8 * 2 * kGroupCols * 4 : 0;  // lse / delta
  static constexpr int kFixed = 2 * kStatBytes + kStageLse + 512 + 1024;
  static constexpr int kNSFit = (227 * 1024 - kFixed) / (2 * kMvBytes);
  static constexpr int kNS = kNSFit < 6 ? kNSFit : 6;   // moving stages
  static constexpr int kSmemBytes = kFixed + kNS * 2 * kMvBytes;
  static constexpr int kTmemCols = 512;
  // Score buffers: S at buf * 128, dP at buf * 128 + 64; accumulators after.
  // Warpgroup g's 32 columns of a score buffer take its 16 packed bf16
  // columns of P (or dS) in their first half: p_col(g) from the buffer.
  __host__ __device__ static constexpr int s_col(int buf) { return buf * 128; }
  __host__ __device__ static constexpr int dp_col(int buf) { return buf * 128 + 64; }
  __host__ __device__ static constexpr int acc_col(int i) { return 256 + i * D; }
  __host__ __device__ static constexpr int p_col(int g) { return g * kGroupCols; }
};

struct BwdParams {
  CUtensorMap t_stat0, t_stat1, t_mv0, t_mv1;  // 4-D maps {d, dim1, dim2, batch}
  SwaBwdArgs a;
  int seq_dim;
  int num_items, blocks;
  int out32;  // every gradient row starts on a 32-byte boundary: 32-byte stores
};

__device__ __forceinline__ void tma_rows(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                         int h, int t, int b, int seq_dim) {
  if (seq_dim == 2)
    tma_load_4d(dst, map, bar, x, h, t, b);
  else
    tma_load_4d(dst, map, bar, x, t, h, b);
}

struct Item {
  int r0, h, b, t_lo, n_tiles;  // stationary rows r0 .. r0+127; moving tiles t_lo ..
};

// kKV: key blocks in increasing order (most query tiles first); kQ: query
// blocks in decreasing order (most key tiles first).  Either way the items
// run longest first and are dealt to the CTAs in snake order (snake_item).
template <int MODE>
__device__ __forceinline__ Item decode_item(const BwdParams& P, int item) {
  Item it;
  const int per_block = P.a.heads * P.a.batch;
  const int blk = MODE == kKV ? item / per_block : P.blocks - 1 - item / per_block;
  const int rest = item % per_block;
  it.h = rest % P.a.heads;
  it.b = rest / P.a.heads;
  it.r0 = blk * BR;
  int lo, hi;
  if (MODE == kKV) {  // queries that see any of keys r0 .. r0+127
    lo = it.r0;
    hi = min(P.a.seq - 1, it.r0 + BR - 1 + P.a.window - 1);
  } else {            // keys seen by any of queries r0 .. r0+127
    lo = max(0, it.r0 - P.a.window + 1);
    hi = min(P.a.seq - 1, it.r0 + BR - 1);
  }
  it.t_lo = lo / BC;
  it.n_tiles = hi / BC - it.t_lo + 1;
  return it;
}

template <int D>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16* dst, const float (&v)[D], float mul) {
#pragma unroll
  for (int e = 0; e < D; e += 8)
    *reinterpret_cast<uint4*>(dst + e) =
        make_uint4(pack_bf16x2(v[e] * mul, v[e + 1] * mul), pack_bf16x2(v[e + 2] * mul, v[e + 3] * mul),
                   pack_bf16x2(v[e + 4] * mul, v[e + 5] * mul),
                   pack_bf16x2(v[e + 6] * mul, v[e + 7] * mul));
}

// The same with 32-byte stores (dst 32-byte aligned): one sector per row and
// instruction instead of half of one, half the store instructions.  At the
// 13B-class shape the two kernels' stores of one item touch 128 rows x d of
// each gradient, one row per thread.
template <int D>
__device__ __forceinline__ void store_row_bf16_32(__nv_bfloat16* dst, const float (&v)[D],
                                                  float mul) {
  static_assert(D % 16 == 0, "whole 32-byte stores");
#pragma unroll
  for (int e = 0; e < D; e += 16) {
    uint32_t w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(v[e + 2 * u] * mul, v[e + 2 * u + 1] * mul);
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst + e),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
  }
}

template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) swa_bwd_kernel(const __grid_constant__ BwdParams P) {
  using C = BwdCfg<D, MODE>;
  constexpr int NS = C::kNS;
  const SwaBwdArgs& a = P.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sStat = smem;                               // [2][kStatBytes]
  uint8_t* sMv = sStat + 2 * C::kStatBytes;            // [NS][2][kMvBytes]
  float* sLse = reinterpret_cast<float*>(sMv + NS * 2 * C::kMvBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sLse) + C::kStageLse);
  uint64_t* stat_full = bars;
  uint64_t* stat_empty = stat_full + 1;
  uint64_t* mv_full = stat_empty + 1;   // [NS]
  uint64_t* mv_empty = mv_full + NS;    // [NS]
  uint64_t* s_full = mv_empty + NS;     // [2]
  uint64_t* p_full = s_full + 2;        // [2]
  uint64_t* acc_full = p_full + 2;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* done_bar = acc_empty + 1;   // [3]: one per issuing thread
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(stat_full, 1);
    mbar_init(stat_empty, 2);  // the S and dP threads release the stationary tiles
    for (int s = 0; s < NS; ++s) {
      mbar_init(&mv_full[s], 1);
      mbar_init(&mv_empty[s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 2);  // S and dP of one buffer, from two threads
      mbar_init(&p_full[k], 8);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    for (int k = 0; k < 3; ++k) mbar_init(&done_bar[k], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&P.t_stat0);
    tma_prefetch_desc(&P.t_stat1);
    tma_prefetch_desc(&P.t_mv0);
    tma_prefetch_desc(&P.t_mv1);
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
      uint32_t mv_count = 0, stat_count = 0;
      uint32_t armed = 0, armed_parity = 0;
      for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
        const Item it = decode_item<MODE>(P, item);
        if (!mbar_wait(stat_empty, (stat_count & 1) ^ 1u, abort_flag, a.status)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(stat_full, 2 * C::kStatBytes);
#pragma unroll
        for (int at = 0; at < C::kAtoms; ++at) {
          tma_rows(sStat + at * BR * 128, &P.t_stat0, stat_full, at * 64, it.h, it.r0, it.b,
                   P.seq_dim);
          tma_rows(sStat + C::kStatBytes + at * BR * 128, &P.t_stat1, stat_full, at * 64, it.h,
                   it.r0, it.b, P.seq_dim);
        }
        ++stat_count;
        for (int j = 0; j < it.n_tiles; ++j, ++mv_count) {
          const int st = mv_count % NS;
          const uint32_t ph = (mv_count / NS) & 1;
          if (!mbar_wait(&mv_empty[st], ph ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          const int row0 = (it.t_lo + j) * BC;
          uint8_t* dst = sMv + st * 2 * C::kMvBytes;
          mbar_arrive_expect_tx(&mv_full[st], 2 * C::kMvBytes);
#pragma unroll
          for (int at = 0; at < C::kAtoms; ++at) {
            tma_rows(dst + at * BC * 128, &P.t_mv0, &mv_full[st], at * 64, it.h, row0, it.b,
                     P.seq_dim);
            tma_rows(dst + C::kMvBytes + at * BC * 128, &P.t_mv1, &mv_full[st], at * 64, it.h,
                     row0, it.b, P.seq_dim);
          }
          armed |= 1u << st;
          armed_parity = (armed_parity & ~(1u << st)) | (ph << st);
        }
      }
      // Let every copy this thread issued land before the CTA goes away.
      volatile int no_abort = 0;
      for (int s = 0; s < NS; ++s)
        if (armed & (1u << s))
          mbar_wait(&mv_full[s], (armed_parity >> s) & 1u, &no_abort, a.status);
      if (stat_count > 0) mbar_wait(stat_full, (stat_count - 1) & 1, &no_abort, a.status);
    }
  } else if (warp <= 3) {
    // ------------------------------------------------------------- MMA --
    // Three issuing threads: warp 1 the S scores, warp 2 the dP scores,
    // warp 3 the accumulate MMAs.  One thread issues at most one tcgen05
    // instruction (MMA or commit) every ~75 cycles whatever the MMA's N,
    // slower than the tensor pipe runs these N = 64 MMAs; three streams keep
    // it fed.  All three observe every moving stage in order.  The stage is
    // released by the accumulate thread after the tile's accumulate MMAs,
    // which follow the tile's score MMAs (those were read before P / dS was
    // written), so no stage is refilled before all three have seen it.
    const int role = warp - 1;  // 0: S, 1: dP, 2: accumulate
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(BR, BC);
      constexpr uint32_t idesc_acc = umma_idesc_bf16(BR, D) | (1u << 16);  // B MN-major
      bool ok = true;
      uint32_t mv_count = 0, stat_count = 0, issued = 0, items_done = 0;
      const uint32_t stat = smem_addr(sStat) + (role == 1 ? C::kStatBytes : 0);
      for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
        const Item it = decode_item<MODE>(P, item);
        if (role < 2) {
          if (!mbar_wait(stat_full, stat_count & 1, abort_flag, a.status)) break;
          ++stat_count;
          tc_fence_after();
        }
        for (int j = 0; j < it.n_tiles; ++j) {
          const uint32_t mc = mv_count + j;
          const int st = mc % NS;
          if (!mbar_wait(&mv_full[st], (mc / NS) & 1, abort_flag, a.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t mv0 = smem_addr(sMv + st * 2 * C::kMvBytes), mv1 = mv0 + C::kMvBytes;
          const uint32_t n = issued;
          if (role < 2) {
            // Scores of the stationary rows against the moving tile:
            //   kKV: S^T = K Q^T, dP^T = V dO^T;  kQ: S = Q K^T, dP = dO V^T.
            // Buffer n % 2 holds P / dS of tile n - 2 until its accumulate
            // MMAs have finished, which is when the accumulate thread's
            // commit releases tile n - 2's moving stage.  (Every tile is
            // processed, so n is also the moving-tile number.)  That phase is
            // exact: the stage's next release needs score tile n - 2 + NS.
            if (n >= 2) {
              const uint32_t m2 = n - 2;
              if (!mbar_wait(&mv_empty[m2 % NS], (m2 / NS) & 1, abort_flag, a.status)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t mv = role == 0 ? mv0 : mv1;
            const uint32_t d_tmem = tmem + (role == 0 ? C::s_col(n & 1) : C::dp_col(n & 1));
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t at = kk / 4, off = (kk % 4) * 32;
              umma_bf16_ss(d_tmem, sw128_kmajor_desc(stat + at * BR * 128 + off),
                           sw128_kmajor_desc(mv + at * BC * 128 + off), idesc_s, kk > 0);
            }
            umma_commit(&s_full[n & 1]);
            if (j == it.n_tiles - 1) umma_commit(stat_empty);  // stationary tiles are free
          } else {
            if (!mbar_wait(&p_full[n & 1], (n >> 1) & 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            if (j == 0) {  // the accumulators of the previous item have been read out
              if (!mbar_wait(acc_empty, (items_done & 1) ^ 1u, abort_flag, a.status)) {
                ok = false;
                break;
              }
            }
            tc_fence_after();
            const bool first = j == 0;
            // A from TMEM: 16 moving positions = 8 packed columns, those of
            // warpgroup kk / 2 (positions 32 * (kk / 2) ..) in its half of the
            // score buffer.  B: the moving tile as the MN-major operand, rows
            // = its 64 positions (K), 64-column blocks of d (N) 64 * 128
            // bytes apart.
            auto a_col = [&](int base, int kk) {
              return tmem + base + C::p_col(kk >> 1) + (kk & 1) * 8;
            };
            if constexpr (MODE == kKV) {
              // dV += P^T dO, dK += dS^T Q
#pragma unroll
              for (int kk = 0; kk < BC / 16; ++kk)
                umma_bf16_ts(tmem + C::acc_col(0), a_col(C::s_col(n & 1), kk),
                             sw128_mnmajor_desc(mv1 + kk * 16 * 128, BC * 128), idesc_acc,
                             (!first || kk > 0) ? 1u : 0u);
#pragma unroll
              for (int kk = 0; kk < BC / 16; ++kk)
                umma_bf16_ts(tmem + C::acc_col(1), a_col(C::dp_col(n & 1), kk),
                             sw128_mnmajor_desc(mv0 + kk * 16 * 128, BC * 128), idesc_acc,
                             (!first || kk > 0) ? 1u : 0u);
            } else {
              // dQ += dS K
#pragma unroll
              for (int kk = 0; kk < BC / 16; ++kk)
                umma_bf16_ts(tmem + C::acc_col(0), a_col(C::dp_col(n & 1), kk),
                             sw128_mnmajor_desc(mv0 + kk * 16 * 128, BC * 128), idesc_acc,
                             (!first || kk > 0) ? 1u : 0u);
            }
            umma_commit(&mv_empty[st]);
          }
          ++issued;
        }
        if (!ok) break;
        if (role == 2) {
          umma_commit(acc_full);
          ++items_done;
        }
        mv_count += it.n_tiles;
      }
      umma_commit(&done_bar[role]);
      volatile int no_abort = 0;
      mbar_wait(&done_bar[role], 0, &no_abort, a.status);
    }
  } else {
    // ------------------------------------------------- P, dS and output --
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // stationary row = TMEM lane
    const int grp = (warp - 4) >> 2;    // this warpgroup's columns: 32 * grp .. +31
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    float* wl = sLse + (warp - 4) * 2 * kGroupCols;  // this warp's lse / delta staging (kKV)
    uint32_t seen = 0, items_done = 0;
    bool ok = true;
    for (int k = 0, item = snake_item(0); ok && item < P.num_items; item = snake_item(++k)) {
      const Item it = decode_item<MODE>(P, item);
      const int row = it.r0 + r;  // this thread's stationary position
      const int64_t bh = static_cast<int64_t>(it.b) * a.heads + it.h;
      float nlse_row = 0.f, delta_row = 0.f;  // -lse, so the exponent is one FMA
      if (MODE == kQ && row < a.seq) {
        nlse_row = -a.lse[bh * a.seq + row];
        delta_row = a.delta[bh * a.seq + row];
      }
      // kKV: lane j carries -lse and delta of query column j of the tile
      // (negated lse: one FMA below).  They are loaded one tile ahead, so
      // the global-load latency (~800 cycles measured) overlaps a tile's
      // work instead of stalling each tile's start.
      // (The loads are volatile asm, so the compiler keeps them here, ahead
      // of the tile's barrier wait, rather than next to their use.)
      auto col_stats = [&](int t, float& nl, float& dl) {
        const int q = (it.t_lo + t) * BC + grp * kGroupCols + lane;
        const bool in = t < it.n_tiles && q < a.seq;
        const int64_t off = in ? bh * a.seq + q : 0;  // row 0 always exists
        float l, d;
        asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(l) : "l"(a.lse + off));
        asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(d) : "l"(a.delta + off));
        nl = in ? -l : 0.f;
        dl = in ? d : 0.f;
      };
      float nl_next = 0.f, dl_next = 0.f;
      if (MODE == kKV) col_stats(0, nl_next, dl_next);
      for (int t = 0; t < it.n_tiles; ++t) {
        // First moving position of this warpgroup's 32 columns of the tile.
        const int c0 = (it.t_lo + t) * BC + grp * kGroupCols;
        const int buf = seen & 1;
        if (MODE == kKV) {  // staged per warp for broadcast reads
          __syncwarp();
          wl[lane] = nl_next;
          wl[kGroupCols + lane] = dl_next;
          __syncwarp();
          col_stats(t + 1, nl_next, dl_next);
        }
        if (!mbar_wait_warp(&s_full[buf], (seen >> 1) & 1, abort_flag, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t s_raw[kGroupCols], dp_raw[kGroupCols];
        tmem_ld_32x32b_x32(tmem + lane_base + C::s_col(buf) + grp * kGroupCols, s_raw);
        tmem_ld_32x32b_x32(tmem + lane_base + C::dp_col(buf) + grp * kGroupCols, dp_raw);
        tmem_ld_wait();
        float s[kGroupCols], dp[kGroupCols];
#pragma unroll
        for (int e = 0; e < kGroupCols; ++e) {
          s[e] = __uint_as_float(s_raw[e]);
          dp[e] = __uint_as_float(dp_raw[e]);
        }
        // Moving positions c0 + e with e in [lo, hi] are in the band of this
        // thread's row (kKV: queries row .. row + w - 1 that exist; kQ: keys
        // row - w + 1 .. row); a tile wholly inside it skips the mask.
        const int w = min(a.window, a.seq);  // no int overflow for any window
        const int lo = MODE == kKV ? row - c0 : row - w + 1 - c0;
        const int hi = row >= a.seq ? -1
                       : MODE == kKV ? min(row + w - 1, a.seq - 1) - c0 : row - c0;
        const bool interior = lo <= 0 && hi >= kGroupCols - 1;
        float nl2v[kGroupCols], dlv[kGroupCols];
        if constexpr (MODE == kKV) {  // per-query -lse and delta of the columns
#pragma unroll
          for (int e = 0; e < kGroupCols; e += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(wl + e);
            const float4 d4 = *reinterpret_cast<const float4*>(wl + kGroupCols + e);
            nl2v[e] = l4.x; nl2v[e + 1] = l4.y; nl2v[e + 2] = l4.z; nl2v[e + 3] = l4.w;
            dlv[e] = d4.x; dlv[e + 1] = d4.y; dlv[e + 2] = d4.z; dlv[e + 3] = d4.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < kGroupCols; ++e) {
            nl2v[e] = nlse_row;
            dlv[e] = delta_row;
          }
        }
        // Packed f32x2 arithmetic, two moving positions per instruction:
        // these warps are bound by instruction issue.
        const uint64_t scale2 = f2(a.scale_log2, a.scale_log2);
        float pv[kGroupCols];
#pragma unroll
        for (int e = 0; e < kGroupCols; e += 2) {
          float t0, t1;
          f2_split(f2_fma(f2(s[e], s[e + 1]), scale2, f2(nl2v[e], nl2v[e + 1])), t0, t1);
          pv[e] = fast_exp2(t0);
          pv[e + 1] = fast_exp2(t1);
        }
        if (!interior) {
#pragma unroll
          for (int e = 0; e < kGroupCols; ++e) pv[e] = (e >= lo && e <= hi) ? pv[e] : 0.f;
        }
        uint32_t pk_p[kGroupCols / 2], pk_ds[kGroupCols / 2];
#pragma unroll
        for (int e = 0; e < kGroupCols; e += 2) {
          float d0, d1;
          f2_split(f2_mul(f2(pv[e], pv[e + 1]),
                          f2_sub(f2(dp[e], dp[e + 1]), f2(dlv[e], dlv[e + 1]))), d0, d1);
          pk_p[e / 2] = pack_bf16x2(pv[e], pv[e + 1]);
          pk_ds[e / 2] = pack_bf16x2(d0, d1);
        }
        // P^T and dS^T (kKV) or dS (kQ) over the first half of this
        // warpgroup's score columns, which it has just read.
        if constexpr (MODE == kKV)
          tmem_st_32x32b_x16(tmem + lane_base + C::s_col(buf) + C::p_col(grp), pk_p);
        tmem_st_32x32b_x16(tmem + lane_base + C::dp_col(buf) + C::p_col(grp), pk_ds);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[buf]);
        ++seen;
      }
      if (!ok) break;
      // All accumulate MMAs of the item are done: gradients out.
      if (!mbar_wait_warp(acc_full, items_done & 1, abort_flag, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int prow = row < a.seq ? row : 0;
      // kKV: warpgroup 0 stores dV, warpgroup 1 dK; kQ: warpgroup 0 dQ.
      // Up to 64 columns are loaded per wait, and a warp releases the
      // accumulators right after its last TMEM load has landed: the next
      // item's accumulate MMAs do not wait for the stores.
      const bool active = MODE == kKV || grp == 0;
      __nv_bfloat16* dst =
          MODE == kQ ? a.dq + it.b * a.dq_sb + it.h * a.dq_sh + prow * a.dq_ss
          : grp == 0 ? a.dv + it.b * a.dv_sb + it.h * a.dv_sh + prow * a.dv_ss
                     : a.dk + it.b * a.dk_sb + it.h * a.dk_sh + prow * a.dk_ss;
      const float mul = MODE == kKV && grp == 0 ? 1.f : a.scale;
      const uint32_t tacc = tmem + lane_base + C::acc_col(active ? grp : 0);
      constexpr int kGrp = D % 64 == 0 ? 64 : D % 32 == 0 ? 32 : D;  // columns per wait
      static_assert(D % kGrp == 0 && kGrp % 8 == 0, "whole groups of whole 16-byte stores");
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += kGrp) {
        float g[kGrp];
        if (active) {
          if constexpr (kGrp % 32 == 0) {
            uint32_t r[kGrp / 32][32];
#pragma unroll
            for (int h = 0; h < kGrp / 32; ++h) tmem_ld_32x32b_x32(tacc + c0 + 32 * h, r[h]);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < kGrp / 32; ++h)
#pragma unroll
              for (int e = 0; e < 32; ++e) g[32 * h + e] = __uint_as_float(r[h][e]);
          } else {
            uint32_t r[16];
            tmem_ld_32x32b_x16(tacc + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) g[e] = __uint_as_float(r[e]);
          }
        }
        if (c0 + kGrp >= D) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty);
        }
        if (active && row < a.seq) {
          if constexpr (kGrp % 16 == 0) {
            if (P.out32)
              store_row_bf16_32<kGrp>(dst + c0, g, mul);
            else
              store_row_bf16<kGrp>(dst + c0, g, mul);
          } else {
            store_row_bf16<kGrp>(dst + c0, g, mul);
          }
        }
      }
      ++items_done;
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

// delta_i = sum_c dO_ic * o_ic for every (batch entry, head, row): eight
// lanes per row, lane j taking the 16-byte chunks j, j + 8, ... of the row
// (head_dim / 8 chunks), summed by shuffles within the eight lanes.
__global__ void swa_delta_kernel(const SwaBwdArgs a) {
  const int64_t rows = static_cast<int64_t>(a.batch) * a.heads * a.seq;
  // Every lane of a warp runs the same number of iterations (the bound is a
  // multiple of 4 and so is the stride), so the shuffles see all 32 lanes.
  const int64_t bound = (rows + 3) & ~static_cast<int64_t>(3);
  const int sub = threadIdx.x & 7;
  const int chunks = a.head_dim / 8;
  for (int64_t idx = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 3;
       idx < bound; idx += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 3) {
    float acc = 0.f;
    if (idx < rows) {
      const int i = static_cast<int>(idx % a.seq);
      const int64_t bh = idx / a.seq;
      const int h = static_cast<int>(bh % a.heads);
      const int b = static_cast<int>(bh / a.heads);
      const uint4* o = reinterpret_cast<const uint4*>(a.o + b * a.o_sb + h * a.o_sh + i * a.o_ss);
      const uint4* g = reinterpret_cast<const uint4*>(a.dout + b * a.do_sb + h * a.do_sh +
                                                      i * a.do_ss);
      for (int c = sub; c < chunks; c += 8) {
        const uint4 x = __ldg(o + c), y = __ldg(g + c);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          acc += bf16_lo(xs[e]) * bf16_lo(ys[e]) + bf16_hi(xs[e]) * bf16_hi(ys[e]);
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    if (idx < rows && sub == 0) a.delta[idx] = acc;
  }
}

template <int D, int MODE>
cudaError_t launch_typed(const BwdParams& prm, int grid, cudaStream_t stream) {
  using C = BwdCfg<D, MODE>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory");
  auto kern = swa_bwd_kernel<D, MODE>;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(prm);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t dispatch(const BwdParams& prm, int grid, cudaStream_t stream) {
  switch (prm.a.head_dim) {
    case 16: return launch_typed<16, MODE>(prm, grid, stream);
    case 32: return launch_typed<32, MODE>(prm, grid, stream);
    case 64: return launch_typed<64, MODE>(prm, grid, stream);
    case 96: return launch_typed<96, MODE>(prm, grid, stream);
    case 128: return launch_typed<128, MODE>(prm, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// 4-D map {d, heads, seq, batch} or {d, seq, heads, batch} over a strided
// [batch][heads][seq][d] view; boxes of 64 columns x `rows` positions.
bool bwd_map(CUtensorMap* map, const __nv_bfloat16* base, int64_t sb, int64_t sh, int64_t ss,
             const SwaBwdArgs& a, int rows, int* seq_dim) {
  const bool heads_first = sh <= ss;
  if (sb <= 0) sb = (sh > ss ? sh : ss) * (a.heads > a.seq ? a.heads : a.seq);  // unused stride
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

cudaError_t launch_swa_backward(const SwaBwdArgs& a, cudaStream_t stream) {
  if (a.seq <= 0 || a.batch <= 0 || a.heads <= 0) return cudaSuccess;
  const int64_t rows = static_cast<int64_t>(a.batch) * a.heads * a.seq;
  {
    const int64_t blocks = (rows * 8 + 255) / 256;
    const int grid = static_cast<int>(blocks < 16 * a.sms ? blocks : 16 * a.sms);
    swa_delta_kernel<<<grid, 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  BwdParams prm;
  prm.a = a;
  // A window of s or more is plain causal attention; clamping it keeps every
  // index expression of the kernels (a row plus the window, ...) inside int.
  if (prm.a.window > prm.a.seq) prm.a.window = prm.a.seq;
  prm.blocks = (a.seq + BR - 1) / BR;
  {
    auto a32 = [](const void* p, int64_t sb, int64_t sh, int64_t ss) {
      return (reinterpret_cast<uintptr_t>(p) % 32) == 0 && sb % 16 == 0 && sh % 16 == 0 &&
             ss % 16 == 0;
    };
    prm.out32 = a32(a.dq, a.dq_sb, a.dq_sh, a.dq_ss) && a32(a.dk, a.dk_sb, a.dk_sh, a.dk_ss) &&
                a32(a.dv, a.dv_sb, a.dv_sh, a.dv_ss);
  }
  const int64_t items = static_cast<int64_t>(prm.blocks) * a.heads * a.batch;
  if (items > 0x3fffffff) return cudaErrorInvalidValue;  // item numbers stay in int
  prm.num_items = static_cast<int>(items);
  const int grid = static_cast<int>(items < a.sms ? items : a.sms);
  int sd[4];
  // dK, dV: stationary K, V (128 rows); moving Q, dO (64 rows).
  if (!bwd_map(&prm.t_stat0, a.k, a.k_sb, a.k_sh, a.k_ss, a, BR, &sd[0]) ||
      !bwd_map(&prm.t_stat1, a.v, a.v_sb, a.v_sh, a.v_ss, a, BR, &sd[1]) ||
      !bwd_map(&prm.t_mv0, a.q, a.q_sb, a.q_sh, a.q_ss, a, BC, &sd[2]) ||
      !bwd_map(&prm.t_mv1, a.dout, a.do_sb, a.do_sh, a.do_ss, a, BC, &sd[3]))
    return cudaErrorInvalidValue;
  if (sd[0] != sd[1] || sd[0] != sd[2] || sd[0] != sd[3]) return cudaErrorInvalidValue;
  prm.seq_dim = sd[0];
  cudaError_t e = dispatch<kKV>(prm, grid, stream);
  if (e != cudaSuccess) return e;
  // dQ: stationary Q, dO (128 rows); moving K, V (64 rows).
  if (!bwd_map(&prm.t_stat0, a.q, a.q_sb, a.q_sh, a.q_ss, a, BR, &sd[0]) ||
      !bwd_map(&prm.t_stat1, a.dout, a.do_sb, a.do_sh, a.do_ss, a, BR, &sd[1]) ||
      !bwd_map(&prm.t_mv0, a.k, a.k_sb, a.k_sh, a.k_ss, a, BC, &sd[2]) ||
      !bwd_map(&prm.t_mv1, a.v, a.v_sb, a.v_sh, a.v_ss, a, BC, &sd[3]))
    return cudaErrorInvalidValue;
  return dispatch<kQ>(prm, grid, stream);
}

}  // namespace ptb
