// C ABI of libptb (declared in include/ptb.h), common part and forward pass:
// argument checks, tensor-map encoding, the GEMM launch plumbing, the
// per-device workspace arena and status word, and the launch sequence of the
// parallel transformer block forward pass
//   y = x + Attn(LN(x)) + MLP(LN(x))
// (MegaScale study notes, ch.2 §2.2, PTB row).  The attention operator, the
// FP8 variant and the training entry points are in api_swa.cu, api_fp8.cu
// and api_train.cu.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "api_internal.h"
#include "ptb_device.cuh"

namespace ptb {
namespace api {

constexpr int kMaxDevices = 64;

__device__ unsigned g_status_word;
// Where take_status_kernel leaves the word it swapped out, for the host to read.
__device__ unsigned g_status_taken;


std::mutex g_mutex;
// Serialises ptb_last_device_error calls: they share the device word that
// the status is swapped into.
std::mutex g_status_mutex;
// Serialises the layer launches of ptb_forward_host calls (see there).
std::mutex g_host_mutex;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up: SM count, device status word, architecture check and the
// driver's tensor-map encoder.  Returns PTB_OK and fills *out.
ptb_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PTB_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PTB_ERR_DEVICE;
    if (major != 10 || minor != 3) return PTB_ERR_UNSUPPORTED;
    const char* env = std::getenv("PTB_GEMM_PAIRS");
    s.pairs = (env && env[0] == '0') ? 0 : (env && env[0] == '1') ? 1 : -1;
    void* sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_status_word) != cudaSuccess) return PTB_ERR_DEVICE;
    s.status = static_cast<unsigned*>(sym);
    if (cudaGetSymbolAddress(&sym, g_status_taken) != cudaSuccess) return PTB_ERR_DEVICE;
    s.status_taken = static_cast<unsigned*>(sym);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return PTB_ERR_DEVICE;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    s.ready = true;
  }
  *out = &s;
  return PTB_OK;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix with row stride
// `ld` elements, read in boxes of 64 (inner) x box_outer with 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
              uint32_t box_outer, bool fp8 = false) {
  // One box row is 128 bytes: 64 bf16 or 128 e4m3 elements.
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {ld * (fp8 ? 1 : 2)};
  cuuint32_t box[2] = {fp8 ? 128u : 64u, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_block_n(int64_t a, int64_t b) {
  for (int bn : {256, 128, 64})
    if (a % bn == 0 && b % bn == 0) return bn;
  return 0;
}

ptb_status launch_status(cudaError_t e) { return e == cudaSuccess ? PTB_OK : PTB_ERR_LAUNCH; }

// SM count of the current device, or an upper bound when there is none.
int current_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
    return sms;
  cudaGetLastError();
  return 256;
}

size_t gemm_scratch_bytes(const GemmPlan& g) {
  return round_up(g.partial_bytes, kAlign) + round_up(g.counter_bytes, kAlign);
}

// Whether a GEMM that can run on CTA pairs does: always, unless pairs are
// switched off (ptb_set_gemm_pairs(0)).  Measured on GB300: pairs do a
// k-block in ~28% fewer cycles.  That made the 13B-class forward layer 9%
// faster at an unchanged 2070 MHz and the training step 6% faster at 13B and
// 175B.  Back-to-back 175B- and 530B-class forward layers run at the 1.4 kW
// power cap; there pairs first looked no faster (the clock fell from 1.92 to
// 1.5 GHz), but that was with the weights loaded evict_first, which left the
// pair kernel re-reading them from DRAM (6.1-6.5 GB per launch of the
// 175B-class [out | down] GEMM, 3.2 GB with evict_last).  With both operands
// evict_last, pairs for both GEMMs against single CTAs: 175B class 4.45 vs
// 4.58 ms, 530B class 12.13-12.18 vs 12.85-12.90 ms, e4m3 175B 2.48-2.53 vs
// 2.56-2.58 ms, e4m3 530B 6.42-6.47 vs 6.84-6.85 ms.
bool use_pairs(const DeviceState* ds, bool shape_ok, int64_t m) {
  return shape_ok && m > 128 && ds->sms >= 2 && ds->pairs != 0;
}

// Output tiles of a launch: 128-row tiles, or 256-row tiles on CTA pairs.
int64_t gemm_tiles(int64_t m, int64_t n, int block_n, bool pair) {
  const int64_t rows = pair ? 256 : 128;
  return (m + rows - 1) / rows * (n / block_n);
}

// Scratch for the split last wave of an M x N x (kb k-blocks) GEMM, either
// tile shape (whichever needs more).
size_t gemm_scratch_any(int64_t m, int64_t n, int64_t kb, int block_n, int sms) {
  const size_t a = gemm_scratch_bytes(plan_gemm(gemm_tiles(m, n, block_n, false), kb, sms, block_n));
  const size_t b = gemm_scratch_bytes(
      plan_gemm(gemm_tiles(m, n, block_n, true), kb, sms / 2, block_n, 256));
  return a > b ? a : b;
}

// Fills the grid / split fields of a launch (a.pair and a.block_n set).
// Without scratch (or with too little) the GEMM runs unsplit.
void apply_plan(GemmArgs& a, int64_t num_kb, int sms, void* scratch, size_t scratch_bytes) {
  const int64_t tiles = gemm_tiles(a.M, a.N, a.block_n, a.pair != 0);
  const int workers = a.pair ? sms / 2 : sms;
  GemmPlan g = plan_gemm(tiles, num_kb, workers, a.block_n, a.pair ? 256 : 128);
  const int per_worker = a.pair ? 2 : 1;
  if (g.split_s >= 2 && scratch && scratch_bytes >= gemm_scratch_bytes(g)) {
    a.grid = g.grid * per_worker;
    a.split_r = g.split_r;
    a.split_s = g.split_s;
    a.partials = static_cast<float*>(scratch);
    a.counters = reinterpret_cast<unsigned*>(static_cast<char*>(scratch) +
                                             round_up(g.partial_bytes, kAlign));
  } else {
    a.grid = static_cast<int>(tiles < workers ? tiles : workers) * per_worker;
    a.split_r = 0;
    a.split_s = 1;
    a.partials = nullptr;
    a.counters = nullptr;
  }
}


GemmSpec spec_fp8(const void* a, int64_t lda, int64_t k, const void* b, int64_t n,
                  const float* a_scale, const float* b_scale) {
  GemmSpec g{static_cast<const ptb_bf16*>(a), static_cast<const ptb_bf16*>(a),
             static_cast<const ptb_bf16*>(b), static_cast<const ptb_bf16*>(b), lda, lda, k, 0, n,
             0};
  g.fp8 = true;
  g.a_scale = a_scale;
  g.b_scale = b_scale;
  return g;
}

GemmSpec spec_plain(const ptb_bf16* a, int64_t lda, int64_t k, const ptb_bf16* b, int64_t n) {
  return GemmSpec{a, a, b, b, lda, lda, k, 0, n, 0};
}

size_t spec_scratch(const GemmSpec& g, int64_t tokens, int sms) {
  const int bn = g.block_n() ? g.block_n() : 64;
  return gemm_scratch_any(tokens, g.n(), g.kb(), bn, sms);
}

ptb_status gemm_run(DeviceState* ds, const GemmSpec& g, int64_t tokens, ptb_bf16* out, int64_t ldo,
                    const ptb_bf16* resid, int64_t ldr, int64_t gelu_col, void* scratch,
                    size_t scratch_bytes, cudaStream_t stream, ptb_bf16* aux,
                    int64_t ld_aux) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.block_n = g.block_n();
  if (!a.block_n) return PTB_ERR_SHAPE;
  const int64_t K = g.k(), N = g.n();
  // CTA pairs for bf16 GEMMs with 256-wide N tiles and more than one
  // 128-row tile of M; each CTA of a pair loads half of the B tile.
  a.pair = use_pairs(ds, a.block_n == 256, tokens) ? 1 : 0;
  const uint32_t box_b = a.pair ? a.block_n / 2 : a.block_n;
  bool ok;
  if (g.k1) {
    ok = make_map(&a.a0, g.a0, g.k0, tokens, g.lda0, 128) &&
         make_map(&a.a1, g.a1, g.k1, tokens, g.lda1, 128) &&
         make_map(&a.b0, g.b0, g.k0, N, g.k0, box_b) &&
         make_map(&a.b1, g.b1, g.k1, N, g.k1, box_b);
  } else {
    ok = make_map(&a.a0, g.a0, K, tokens, g.lda0, 128, g.fp8) &&
         make_map(&a.a1, g.a0, K, tokens, g.lda0, 128, g.fp8) &&
         make_map(&a.b0, g.b0, K, g.n0, K, box_b, g.fp8) &&
         make_map(&a.b1, g.n1 ? g.b1 : g.b0, K, g.n1 ? g.n1 : g.n0, K, box_b, g.fp8);
  }
  if (!ok) return PTB_ERR_ARG;
  a.M = static_cast<int>(tokens);
  a.N = static_cast<int>(N);
  a.K = static_cast<int>(K);
  a.n_split = static_cast<int>(g.n1 ? g.n0 : N);
  a.k_split = static_cast<int>(g.k1 ? g.k0 : K);
  a.layout = kLayoutKK;
  a.n_fastest = 0;
  // Both operands are loaded evict_last.  A is re-read by every wave of N
  // tiles (xn in the first GEMM, [ctx | G] in the second); a weight tile is
  // read by every M tile of its wave, and loaded evict_first its lines were
  // often gone before the wave's later tiles got to them: the 175B-class
  // [out | down] GEMM on CTA pairs read 6.1-6.5 GB from DRAM per launch
  // (3.2 GB with evict_last) and took 1.81-1.83 instead of 1.71-1.72 ms.
  // Layers: 175B class 4.71-4.72 -> 4.61-4.62 ms, 530B class 13.04-13.06 ->
  // 12.86-12.89, 13B class 0.827 -> 0.819-0.824, e4m3 175B class 2.64-2.65
  // -> 2.58-2.61.  (Keeping A alone, against streaming both, had made the
  // 530B-class layer 2.5% faster.)
  a.a_keep = 1;
  a.b_keep = 1;
  a.out = bf(out);
  a.ld_out = ldo;
  a.out1 = a.out;
  a.ld_out1 = ldo;
  a.out_split_col = static_cast<int>(N);
  a.out_split_row = static_cast<int>(tokens);
  a.aux = aux ? bf(aux) : nullptr;
  a.ld_aux = ld_aux;
  a.resid = resid ? bf(resid) : nullptr;
  a.ld_resid = ldr;
  a.gelu_col = static_cast<int>(gelu_col);
  a.epilogue = resid ? kEpiResidual : kEpiQkvGelu;
  a.fp8 = g.fp8 ? 1 : 0;
  a.a_scale = g.a_scale;
  a.b_scale = g.b_scale;
  apply_plan(a, g.kb(), ds->sms, scratch, scratch_bytes);
  a.status = ds->status;
  return launch_status(launch_gemm(a, stream));
}

// [QKV | up] of the PTB: U = [xn W_qkv^T | gelu(xn W_up^T)].
GemmSpec spec_qkv_up(const ptb_bf16* xn, const ptb_bf16* w_qkv, const ptb_bf16* w_up,
                     int64_t hidden, int64_t ffn) {
  return GemmSpec{xn, xn, w_qkv, w_up, hidden, hidden, hidden, 0, 3 * hidden, ffn};
}

// [out | down] of the PTB: [ctx | G] [W_o | W_down]^T.
GemmSpec spec_out_down(const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g, int64_t ld_g,
                       const ptb_bf16* w_o, const ptb_bf16* w_down, int64_t hidden,
                       int64_t ffn) {
  return GemmSpec{ctx, g, w_o, w_down, ld_ctx, ld_g, hidden, ffn, hidden, 0};
}

ptb_status gemm_qkv_up(DeviceState* ds, const ptb_bf16* xn, const ptb_bf16* w_qkv,
                       const ptb_bf16* w_up, int64_t tokens, int64_t hidden, int64_t ffn,
                       ptb_bf16* u, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return gemm_run(ds, spec_qkv_up(xn, w_qkv, w_up, hidden, ffn), tokens, u, 3 * hidden + ffn,
                  nullptr, 0, 3 * hidden, scratch, scratch_bytes, stream);
}

ptb_status gemm_out_down(DeviceState* ds, const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g,
                         int64_t ld_g, const ptb_bf16* w_o, const ptb_bf16* w_down,
                         const ptb_bf16* x, int64_t tokens, int64_t hidden, int64_t ffn,
                         ptb_bf16* y, void* scratch, size_t scratch_bytes, cudaStream_t stream) {
  return gemm_run(ds, spec_out_down(ctx, ld_ctx, g, ld_g, w_o, w_down, hidden, ffn), tokens, y,
                  hidden, x, hidden, hidden, scratch, scratch_bytes, stream);
}


// 2-D bf16 tensor map with boxes of 64 x 64 over a row-major [outer, inner]
// matrix (an MN-major operand: inner = M or N, outer = K).
bool make_map_mn(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld) {
  return make_map(map, base, inner, outer, ld, 64);
}

size_t call_scratch(const GemmCall& c, int sms) {
  const int bn = c.block_n() ? c.block_n() : 64;
  return gemm_scratch_any(c.M, c.N, c.kb(), bn, sms);
}

ptb_status gemm_call(DeviceState* ds, const GemmCall& c, void* scratch, size_t scratch_bytes,
                     cudaStream_t stream) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.block_n = c.block_n();
  if (!a.block_n || c.M < 1 || c.K < 1 || c.M > (1 << 30) || c.N > (1 << 30) || c.K > (1 << 30))
    return PTB_ERR_SHAPE;
  if ((c.k_split && c.n_split) || c.k_split % 64 || c.n_split % 64) return PTB_ERR_SHAPE;
  const bool amn = (c.layout & 1) != 0, bmn = (c.layout & 2) != 0;
  const int64_t k0 = c.k_split ? c.k_split : c.K, k1 = c.k_split ? c.K - c.k_split : 0;
  const int64_t n0 = c.n_split ? c.n_split : c.N, n1 = c.n_split ? c.N - c.n_split : 0;
  const ptb_bf16* a1 = c.k_split ? c.a1 : c.a0;
  const int64_t lda1 = c.k_split ? c.lda1 : c.lda0;
  const ptb_bf16* b1 = (c.k_split || c.n_split) ? c.b1 : c.b0;
  const int64_t ldb1 = (c.k_split || c.n_split) ? c.ldb1 : c.ldb0;
  const int64_t ka1 = k1 ? k1 : k0;
  a.pair = use_pairs(ds, a.block_n == 256, c.M) ? 1 : 0;
  const uint32_t box_b = a.pair ? a.block_n / 2 : a.block_n;
  bool ok;
  if (amn)
    ok = make_map_mn(&a.a0, c.a0, c.M, k0, c.lda0) && make_map_mn(&a.a1, a1, c.M, ka1, lda1);
  else
    ok = make_map(&a.a0, c.a0, k0, c.M, c.lda0, 128) && make_map(&a.a1, a1, ka1, c.M, lda1, 128);
  // B: the K extent of source i is its K part under a K split, else K; the
  // N extent is its N part under an N split, else N.
  const int64_t bk0 = c.k_split ? k0 : c.K, bk1 = c.k_split ? k1 : c.K;
  const int64_t bn0 = c.n_split ? n0 : c.N, bn1 = c.n_split ? n1 : c.N;
  if (bmn)
    ok = ok && make_map_mn(&a.b0, c.b0, bn0, bk0, c.ldb0) && make_map_mn(&a.b1, b1, bn1, bk1, ldb1);
  else
    ok = ok && make_map(&a.b0, c.b0, bk0, bn0, c.ldb0, box_b) &&
         make_map(&a.b1, b1, bk1, bn1, ldb1, box_b);
  if (!ok) return PTB_ERR_ARG;
  a.M = static_cast<int>(c.M);
  a.N = static_cast<int>(c.N);
  a.K = static_cast<int>(c.K);
  a.n_split = static_cast<int>(c.n_split ? c.n_split : c.N);
  a.k_split = static_cast<int>(c.k_split ? c.k_split : c.K);
  a.layout = c.layout;
  a.epilogue = c.epilogue;
  const int64_t num_m = (c.M + 127) / 128, num_n = c.N / a.block_n;
  a.n_fastest = num_m > num_n ? 1 : 0;
  // Both operands evict_last, as in gemm_run: with the operand read once
  // per wave evict_first (the former policy) the 175B-class training step
  // took 14.57-14.63 ms, with both kept 14.15-14.22 ms (13B class 2.56-2.59
  // -> 2.55-2.56 ms).
  a.a_keep = 1;
  a.b_keep = 1;
  a.out = c.out;
  a.ld_out = c.ld_out;
  a.out1 = c.out1 ? c.out1 : c.out;
  a.ld_out1 = c.out1 ? c.ld_out1 : c.ld_out;
  a.out_split_col = static_cast<int>(c.out_split_col ? c.out_split_col : c.N);
  a.out_split_row = static_cast<int>(c.out_split_row ? c.out_split_row : c.M);
  a.aux = c.aux ? bf(c.aux) : nullptr;
  a.ld_aux = c.ld_aux;
  a.gelu_col = static_cast<int>(c.gelu_col ? c.gelu_col : c.N);
  apply_plan(a, c.kb(), ds->sms, scratch, scratch_bytes);
  a.status = ds->status;
  return launch_status(launch_gemm(a, stream));
}

// Scratch for the split last waves of the PTB's two GEMMs (the larger one).
size_t layer_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms) {
  const ptb_bf16* z = nullptr;
  const size_t a = spec_scratch(spec_qkv_up(z, z, z, hidden, ffn), tokens, sms);
  const size_t b = spec_scratch(spec_out_down(z, hidden, z, ffn, z, z, hidden, ffn), tokens, sms);
  return a > b ? a : b;
}

// Scratch for the split last waves of the serial block's four GEMMs.
size_t serial_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms) {
  const ptb_bf16* z = nullptr;
  const GemmSpec specs[4] = {spec_plain(z, hidden, hidden, z, 3 * hidden),
                             spec_plain(z, hidden, hidden, z, hidden),
                             spec_plain(z, hidden, hidden, z, ffn),
                             spec_plain(z, ffn, ffn, z, hidden)};
  size_t m = 0;
  for (const GemmSpec& g : specs) {
    const size_t b = spec_scratch(g, tokens, sms);
    m = b > m ? b : m;
  }
  return m;
}

// Scratch for the split last waves of the FP8 layer's two GEMMs.
size_t fp8_gemm_scratch(int64_t tokens, int64_t hidden, int64_t ffn, int sms) {
  const GemmSpec g1 = spec_fp8(nullptr, hidden, hidden, nullptr, 3 * hidden + ffn, nullptr, nullptr);
  const GemmSpec g2 = spec_fp8(nullptr, hidden + ffn, hidden + ffn, nullptr, hidden, nullptr, nullptr);
  const size_t a = spec_scratch(g1, tokens, sms);
  const size_t b = spec_scratch(g2, tokens, sms);
  return a > b ? a : b;
}

ptb_status check_gemm_shape(int64_t tokens, int64_t hidden, int64_t ffn) {
  if (tokens < 1 || hidden < 64 || ffn < 64) return PTB_ERR_ARG;
  if (hidden % 64 || ffn % 64) return PTB_ERR_SHAPE;
  if (tokens > (1ll << 30) || 3 * hidden + ffn > (1ll << 30)) return PTB_ERR_SHAPE;
  return PTB_OK;
}

ptb_status swa_impl(const SwaArgs& in, float scale, cudaStream_t stream) {
  if (!in.q || !in.k || !in.v || !in.o) return PTB_ERR_ARG;
  if (in.batch < 1 || in.heads < 1 || in.seq < 1 || in.window < 1) return PTB_ERR_ARG;
  if (!head_dim_ok(in.head_dim)) return PTB_ERR_SHAPE;
  if (in.batch * static_cast<int64_t>(in.heads) > 65535) return PTB_ERR_SHAPE;
  const int64_t strides[12] = {in.q_sb, in.q_sh, in.q_ss, in.k_sb, in.k_sh, in.k_ss,
                               in.v_sb, in.v_sh, in.v_ss, in.o_sb, in.o_sh, in.o_ss};
  for (int64_t s : strides)
    if (s % 8) return PTB_ERR_ALIGN;
  if (!aligned(in.q, 16) || !aligned(in.k, 16) || !aligned(in.v, 16) || !aligned(in.o, 16))
    return PTB_ERR_ALIGN;
  if (scale < 0.f || !std::isfinite(scale)) return PTB_ERR_ARG;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  SwaArgs a = in;
  const float sc = scale == 0.f ? 1.0f / std::sqrt(static_cast<float>(in.head_dim)) : scale;
  a.scale_log2 = sc * 1.4426950408889634f;
  a.status = ds->status;
  a.sms = ds->sms;
  return launch_status(launch_swa(a, stream));
}

// ----------------------------------------------------------- wait probe --

__global__ void wait_probe_kernel(uint64_t limit_ns, unsigned* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Nobody arrives on `bar`: the wait must give up and record a timeout.
    mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  }
}

// Reads and clears the status word in one atomic step, so that a code
// recorded by a kernel on another stream between a read and a clear is
// never lost.
__global__ void take_status_kernel(unsigned* status, unsigned* taken) {
  *taken = atomicExch(status, 0u);
}

}  // namespace api

bool make_tensor_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box) {
  if (!api::g_encode || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return api::g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, b, e,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_wait_probe(uint64_t limit_ns, unsigned* status, cudaStream_t stream) {
  api::wait_probe_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace ptb

using namespace ptb;
using namespace ptb::api;

extern "C" {

const char* ptb_status_string(ptb_status s) {
  switch (s) {
    case PTB_OK: return "PTB_OK";
    case PTB_ERR_ARG: return "PTB_ERR_ARG: invalid argument";
    case PTB_ERR_SHAPE: return "PTB_ERR_SHAPE: unsupported shape";
    case PTB_ERR_ALIGN: return "PTB_ERR_ALIGN: pointer or stride not 16-byte aligned";
    case PTB_ERR_WORKSPACE: return "PTB_ERR_WORKSPACE: workspace too small";
    case PTB_ERR_LAUNCH: return "PTB_ERR_LAUNCH: CUDA launch or runtime error";
    case PTB_ERR_TIMEOUT: return "PTB_ERR_TIMEOUT: a device-side wait gave up";
    case PTB_ERR_UNSUPPORTED: return "PTB_ERR_UNSUPPORTED: device is not sm_103";
    case PTB_ERR_DEVICE: return "PTB_ERR_DEVICE: device query or allocation failed";
  }
  return "PTB_ERR_UNKNOWN";
}

size_t ptb_forward_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn) {
  if (batch < 1 || seq < 1 || hidden < 1 || ffn < 1) return 0;
  const size_t t = static_cast<size_t>(batch) * static_cast<size_t>(seq);
  size_t gemm = 0;
  if (hidden % 64 == 0 && ffn % 64 == 0)
    gemm = layer_gemm_scratch(static_cast<int64_t>(t), hidden, ffn, current_sms());
  return round_up(t * hidden * 2, kAlign) + round_up(t * (3 * hidden + ffn) * 2, kAlign) + gemm;
}

size_t ptb_gemm_workspace_size(int64_t tokens, int64_t hidden, int64_t ffn) {
  if (tokens < 1 || hidden < 64 || ffn < 64 || hidden % 64 || ffn % 64) return 0;
  return layer_gemm_scratch(tokens, hidden, ffn, current_sms());
}

}  // extern "C"

namespace ptb {
namespace api {

// Argument checks shared by the layer entry points (before any device use).
ptb_status check_layer(const void* const* ptrs, int nptrs, int64_t batch, int64_t seq,
                       int64_t hidden, int64_t ffn, int32_t heads, int32_t window) {
  for (int i = 0; i < nptrs; ++i)
    if (!ptrs[i]) return PTB_ERR_ARG;
  if (batch < 1 || seq < 1 || heads < 1 || window < 1) return PTB_ERR_ARG;
  ptb_status st = check_gemm_shape(batch * seq, hidden, ffn);
  if (st != PTB_OK) return st;
  if (hidden > 32768 || hidden % heads) return PTB_ERR_SHAPE;
  if (!head_dim_ok(hidden / heads)) return PTB_ERR_SHAPE;
  if (batch * static_cast<int64_t>(heads) > 65535) return PTB_ERR_SHAPE;
  for (int i = 0; i < nptrs; ++i)
    if (!aligned(ptrs[i], 16)) return PTB_ERR_ALIGN;
  return PTB_OK;
}

// The caller's workspace if given (checked), else the library arena grown to `need`.
ptb_status acquire_workspace(DeviceState* ds, size_t need, void* workspace, size_t bytes,
                             void** out) {
  if (workspace) {
    if (bytes < need) return PTB_ERR_WORKSPACE;
    if (!aligned(workspace, kAlign)) return PTB_ERR_ALIGN;
    *out = workspace;
    return PTB_OK;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (ds->arena_bytes < need) {
    if (ds->arena) {
      cudaDeviceSynchronize();
      cudaFree(ds->arena);
      ds->arena = nullptr;
      ds->arena_bytes = 0;
    }
    if (cudaMalloc(&ds->arena, need) != cudaSuccess) {
      ds->arena = nullptr;
      return PTB_ERR_DEVICE;
    }
    ds->arena_bytes = need;
  }
  *out = ds->arena;
  return PTB_OK;
}

// Attention over the Q, K, V column blocks of U ([T, ldu]), output over Q.
SwaArgs swa_over_u(DeviceState* ds, ptb_bf16* u, int64_t ldu, int64_t batch, int64_t seq,
                   int64_t hidden, int32_t heads, int32_t window) {
  const int64_t d = hidden / heads;
  SwaArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  sa.q = bf(u);
  sa.k = bf(u) + hidden;
  sa.v = bf(u) + 2 * hidden;
  sa.o = bf(u);
  sa.q_sb = sa.k_sb = sa.v_sb = sa.o_sb = seq * ldu;
  sa.q_sh = sa.k_sh = sa.v_sh = sa.o_sh = d;
  sa.q_ss = sa.k_ss = sa.v_ss = sa.o_ss = ldu;
  sa.batch = static_cast<int>(batch);
  sa.heads = heads;
  sa.seq = static_cast<int>(seq);
  sa.head_dim = static_cast<int>(d);
  sa.window = window;
  sa.scale_log2 = (1.0f / std::sqrt(static_cast<float>(d))) * 1.4426950408889634f;
  sa.status = ds->status;
  sa.sms = ds->sms;
  return sa;
}

}  // namespace api
}  // namespace ptb

extern "C" {

ptb_status ptb_forward_events(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                              const ptb_bf16* ln_beta, const ptb_bf16* w_qkv,
                              const ptb_bf16* w_o, const ptb_bf16* w_up, const ptb_bf16* w_down,
                              int64_t batch, int64_t seq, int64_t hidden, int64_t ffn,
                              int32_t heads, int32_t window, ptb_bf16* y, void* workspace,
                              size_t workspace_bytes, ptb_stream stream_, void* const* events,
                              int32_t n_events) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, y};
  ptb_status st = check_layer(ptrs, 8, batch, seq, hidden, ffn, heads, window);
  if (st != PTB_OK) return st;
  if (events && n_events != 5) return PTB_ERR_ARG;
  if (events)
    for (int i = 0; i < 5; ++i)
      if (!events[i]) return PTB_ERR_ARG;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;

  const int64_t tokens = batch * seq;
  const size_t need = ptb_forward_workspace_size(batch, seq, hidden, ffn);
  st = acquire_workspace(ds, need, workspace, workspace_bytes, &workspace);
  if (st != PTB_OK) return st;
  ptb_bf16* xn = static_cast<ptb_bf16*>(workspace);
  ptb_bf16* u = reinterpret_cast<ptb_bf16*>(static_cast<char*>(workspace) +
                                            round_up(tokens * hidden * 2, kAlign));
  char* gemm_scratch = reinterpret_cast<char*>(u) + round_up(tokens * (3 * hidden + ffn) * 2, kAlign);
  const size_t gemm_scratch_size =
      need - static_cast<size_t>(gemm_scratch - static_cast<char*>(workspace));
  const int64_t ldu = 3 * hidden + ffn;
  auto mark = [&](int i) -> bool {
    if (!events) return true;
    if (cudaEventRecord(static_cast<cudaEvent_t>(events[i]), stream) == cudaSuccess) return true;
    cudaGetLastError();  // the failed record must not be reported by a later launch
    return false;
  };

  // 1. xn = LN(x)
  if (!mark(0)) return PTB_ERR_ARG;
  if (launch_layernorm(bf(x), bf(ln_gamma), bf(ln_beta), tokens, static_cast<int>(hidden), 1e-5f,
                       bf(xn), stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 2. U = [xn W_qkv^T | gelu(xn W_up^T)]
  if (!mark(1)) return PTB_ERR_ARG;
  st = gemm_qkv_up(ds, xn, w_qkv, w_up, tokens, hidden, ffn, u, gemm_scratch, gemm_scratch_size,
                   stream);
  if (st != PTB_OK) return st;
  // 3. ctx = SWA(Q, K, V), written over Q inside U
  if (!mark(2)) return PTB_ERR_ARG;
  if (launch_swa(swa_over_u(ds, u, ldu, batch, seq, hidden, heads, window), stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // 4. y = x + [ctx | G] [W_o | W_down]^T
  if (!mark(3)) return PTB_ERR_ARG;
  st = gemm_out_down(ds, u, ldu, u + 3 * hidden, ldu, w_o, w_down, x, tokens, hidden, ffn, y,
                     gemm_scratch, gemm_scratch_size, stream);
  if (st != PTB_OK) return st;
  if (!mark(4)) return PTB_ERR_ARG;
  return PTB_OK;
}

size_t ptb_serial_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn) {
  if (batch < 1 || seq < 1 || hidden < 1 || ffn < 1) return 0;
  const size_t t = static_cast<size_t>(batch) * static_cast<size_t>(seq);
  size_t gemm = 0;
  if (hidden % 64 == 0 && ffn % 64 == 0)
    gemm = serial_gemm_scratch(static_cast<int64_t>(t), hidden, ffn, current_sms());
  return 2 * round_up(t * hidden * 2, kAlign) + round_up(t * (3 * hidden + ffn) * 2, kAlign) + gemm;
}

ptb_status ptb_serial_forward(const ptb_bf16* x, const ptb_bf16* ln1_gamma,
                              const ptb_bf16* ln1_beta, const ptb_bf16* ln2_gamma,
                              const ptb_bf16* ln2_beta, const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                              const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t batch,
                              int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                              int32_t window, ptb_bf16* y, void* workspace,
                              size_t workspace_bytes, ptb_stream stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const void* ptrs[] = {x, ln1_gamma, ln1_beta, ln2_gamma, ln2_beta, w_qkv, w_o, w_up, w_down, y};
  ptb_status st = check_layer(ptrs, 10, batch, seq, hidden, ffn, heads, window);
  if (st != PTB_OK) return st;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;

  const int64_t tokens = batch * seq;
  const size_t need = ptb_serial_workspace_size(batch, seq, hidden, ffn);
  st = acquire_workspace(ds, need, workspace, workspace_bytes, &workspace);
  if (st != PTB_OK) return st;
  char* base = static_cast<char*>(workspace);
  const size_t act = round_up(tokens * hidden * 2, kAlign);
  ptb_bf16* xn = reinterpret_cast<ptb_bf16*>(base);
  ptb_bf16* h = reinterpret_cast<ptb_bf16*>(base + act);
  ptb_bf16* u = reinterpret_cast<ptb_bf16*>(base + 2 * act);
  char* scratch = reinterpret_cast<char*>(u) + round_up(tokens * (3 * hidden + ffn) * 2, kAlign);
  const size_t scratch_size = need - static_cast<size_t>(scratch - base);
  const int64_t ldu = 3 * hidden + ffn;
  const int hid = static_cast<int>(hidden);

  // h = x + Attn(LN1(x))
  if (launch_layernorm(bf(x), bf(ln1_gamma), bf(ln1_beta), tokens, hid, 1e-5f, bf(xn), stream) !=
      cudaSuccess)
    return PTB_ERR_LAUNCH;
  st = gemm_run(ds, spec_plain(xn, hidden, hidden, w_qkv, 3 * hidden), tokens, u, ldu, nullptr, 0,
                3 * hidden, scratch, scratch_size, stream);
  if (st != PTB_OK) return st;
  if (launch_swa(swa_over_u(ds, u, ldu, batch, seq, hidden, heads, window), stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  st = gemm_run(ds, spec_plain(u, ldu, hidden, w_o, hidden), tokens, h, hidden, x, hidden, hidden,
                scratch, scratch_size, stream);
  if (st != PTB_OK) return st;
  // y = h + MLP(LN2(h))
  if (launch_layernorm(bf(h), bf(ln2_gamma), bf(ln2_beta), tokens, hid, 1e-5f, bf(xn), stream) !=
      cudaSuccess)
    return PTB_ERR_LAUNCH;
  st = gemm_run(ds, spec_plain(xn, hidden, hidden, w_up, ffn), tokens, u + 3 * hidden, ldu,
                nullptr, 0, 0, scratch, scratch_size, stream);
  if (st != PTB_OK) return st;
  return gemm_run(ds, spec_plain(u + 3 * hidden, ldu, ffn, w_down, hidden), tokens, y, hidden, h,
                  hidden, hidden, scratch, scratch_size, stream);
}

ptb_status ptb_forward(const ptb_bf16* x, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                       const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                       const ptb_bf16* w_down, int64_t batch, int64_t seq, int64_t hidden,
                       int64_t ffn, int32_t heads, int32_t window, ptb_bf16* y,
                       void* workspace, size_t workspace_bytes, ptb_stream stream) {
  return ptb_forward_events(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, batch, seq, hidden,
                            ffn, heads, window, y, workspace, workspace_bytes, stream, nullptr, 0);
}

size_t ptb_forward_host_workspace_size(int64_t batch, int64_t seq, int64_t hidden, int64_t ffn) {
  const size_t layer = ptb_forward_workspace_size(batch, seq, hidden, ffn);
  if (!layer) return 0;
  const size_t t = static_cast<size_t>(batch) * static_cast<size_t>(seq);
  return 2 * round_up(t * hidden * 2, kAlign) + layer;
}

namespace {
// The rest of ptb_forward_host for a layer that does not wait: the layer and
// the copy of y back, on `stream`.
ptb_status forward_host_tail(const ptb_bf16* x_dev, ptb_bf16* y_dev, ptb_bf16* y_host,
                             size_t bytes, const ptb_bf16* ln_gamma, const ptb_bf16* ln_beta,
                             const ptb_bf16* w_qkv, const ptb_bf16* w_o, const ptb_bf16* w_up,
                             const ptb_bf16* w_down, int64_t batch, int64_t seq, int64_t hidden,
                             int64_t ffn, int32_t heads, int32_t window, void* layer_ws,
                             size_t layer_bytes, cudaStream_t stream) {
  ptb_status st = ptb_forward(x_dev, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, batch, seq,
                              hidden, ffn, heads, window, y_dev, layer_ws, layer_bytes, stream);
  if (st != PTB_OK) return st;
  if (cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  return PTB_OK;
}
}  // namespace

ptb_status ptb_forward_host(const ptb_bf16* x_host, const ptb_bf16* ln_gamma,
                            const ptb_bf16* ln_beta, const ptb_bf16* w_qkv, const ptb_bf16* w_o,
                            const ptb_bf16* w_up, const ptb_bf16* w_down, int64_t batch,
                            int64_t seq, int64_t hidden, int64_t ffn, int32_t heads,
                            int32_t window, ptb_bf16* y_host, void* workspace,
                            size_t workspace_bytes, ptb_stream stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!x_host || !y_host || !workspace) return PTB_ERR_ARG;
  const size_t need = ptb_forward_host_workspace_size(batch, seq, hidden, ffn);
  if (!need) return PTB_ERR_ARG;
  if (workspace_bytes < need) return PTB_ERR_WORKSPACE;
  if (!aligned(workspace, kAlign)) return PTB_ERR_ALIGN;
  const size_t bytes = static_cast<size_t>(batch) * seq * hidden * 2;
  char* ws = static_cast<char*>(workspace);
  ptb_bf16* x_dev = reinterpret_cast<ptb_bf16*>(ws);
  ptb_bf16* y_dev = reinterpret_cast<ptb_bf16*>(ws + round_up(bytes, kAlign));
  void* layer_ws = ws + 2 * round_up(bytes, kAlign);
  const size_t layer_bytes = need - 2 * round_up(bytes, kAlign);
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  // The layer's kernels are persistent and take every SM.  For large layers
  // two layers in flight at once only fight over the SMs (175B-class: two
  // streams of layers 5.10 ms per layer, one stream 4.77-4.89 ms), so the
  // layer waits for the previous large call's layer, whatever its stream,
  // while the copies of one call still overlap the other call's layer.
  // Small layers gain from running side by side (13B-class: 2.50 M tokens/s
  // with two streams of calls, 2.32 M serialised), so they do not wait.  The
  // line lies between the two: a first GEMM of more than 2^39 multiply-adds.
  const bool serialise = static_cast<double>(batch) * seq * hidden * (3.0 * hidden + ffn) >
                         549755813888.0;
  if (!serialise)
    return forward_host_tail(x_dev, y_dev, y_host, bytes, ln_gamma, ln_beta, w_qkv, w_o, w_up,
                             w_down, batch, seq, hidden, ffn, heads, window, layer_ws,
                             layer_bytes, stream);
  {
    std::lock_guard<std::mutex> lock(g_host_mutex);
    if (!ds->host_layer_done &&
        cudaEventCreateWithFlags(&ds->host_layer_done, cudaEventDisableTiming) != cudaSuccess) {
      ds->host_layer_done = nullptr;
      return PTB_ERR_DEVICE;
    }
    if (cudaStreamWaitEvent(stream, ds->host_layer_done, 0) != cudaSuccess) return PTB_ERR_LAUNCH;
    st = ptb_forward(x_dev, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, batch, seq, hidden, ffn,
                     heads, window, y_dev, layer_ws, layer_bytes, stream);
    if (st != PTB_OK) return st;
    if (cudaEventRecord(ds->host_layer_done, stream) != cudaSuccess) return PTB_ERR_LAUNCH;
  }
  if (cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  return PTB_OK;
}

ptb_status ptb_release_workspace(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PTB_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState& s = g_dev[dev];
  if (s.arena) {
    cudaDeviceSynchronize();
    cudaFree(s.arena);
    s.arena = nullptr;
    s.arena_bytes = 0;
  }
  return PTB_OK;
}

ptb_status ptb_layernorm(const ptb_bf16* x, const ptb_bf16* gamma, const ptb_bf16* beta,
                         int64_t rows, int64_t hidden, float eps, ptb_bf16* out,
                         ptb_stream stream) {
  if (!x || !gamma || !beta || !out || rows < 1 || hidden < 8 || !(eps >= 0.f))
    return PTB_ERR_ARG;
  if (hidden % 8 || hidden > 32768 || rows > 0x7fffffff) return PTB_ERR_SHAPE;
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(beta, 16) || !aligned(out, 16))
    return PTB_ERR_ALIGN;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  return launch_status(launch_layernorm(bf(x), bf(gamma), bf(beta), rows, static_cast<int>(hidden),
                                        eps, bf(out), static_cast<cudaStream_t>(stream)));
}

ptb_status ptb_gemm_qkv_up(const ptb_bf16* xn, const ptb_bf16* w_qkv, const ptb_bf16* w_up,
                           int64_t tokens, int64_t hidden, int64_t ffn, ptb_bf16* u,
                           void* workspace, size_t workspace_bytes, ptb_stream stream) {
  if (!xn || !w_qkv || !w_up || !u) return PTB_ERR_ARG;
  ptb_status st = check_gemm_shape(tokens, hidden, ffn);
  if (st != PTB_OK) return st;
  if (!aligned(xn, 16) || !aligned(w_qkv, 16) || !aligned(w_up, 16) || !aligned(u, 16))
    return PTB_ERR_ALIGN;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;
  if (workspace && !aligned(workspace, kAlign)) return PTB_ERR_ALIGN;
  return gemm_qkv_up(ds, xn, w_qkv, w_up, tokens, hidden, ffn, u, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

ptb_status ptb_gemm_out_down(const ptb_bf16* ctx, int64_t ld_ctx, const ptb_bf16* g, int64_t ld_g,
                             const ptb_bf16* w_o, const ptb_bf16* w_down, const ptb_bf16* x,
                             int64_t tokens, int64_t hidden, int64_t ffn, ptb_bf16* y,
                             void* workspace, size_t workspace_bytes, ptb_stream stream) {
  if (!ctx || !g || !w_o || !w_down || !x || !y) return PTB_ERR_ARG;
  ptb_status st = check_gemm_shape(tokens, hidden, ffn);
  if (st != PTB_OK) return st;
  if (ld_ctx < hidden || ld_g < ffn) return PTB_ERR_ARG;
  if (ld_ctx % 8 || ld_g % 8) return PTB_ERR_ALIGN;
  const void* ptrs[] = {ctx, g, w_o, w_down, x, y};
  for (const void* p : ptrs)
    if (!aligned(p, 16)) return PTB_ERR_ALIGN;
  DeviceState* ds = nullptr;
  st = device_state(&ds);
  if (st != PTB_OK) return st;
  if (workspace && !aligned(workspace, kAlign)) return PTB_ERR_ALIGN;
  return gemm_out_down(ds, ctx, ld_ctx, g, ld_g, w_o, w_down, x, tokens, hidden, ffn, y, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream));
}

ptb_status ptb_last_device_error(ptb_stream stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  std::lock_guard<std::mutex> lock(g_status_mutex);
  take_status_kernel<<<1, 1, 0, stream>>>(ds->status, ds->status_taken);
  if (cudaGetLastError() != cudaSuccess) return PTB_ERR_LAUNCH;
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, ds->status_taken, sizeof(word), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return PTB_ERR_LAUNCH;
  return static_cast<ptb_status>(word);
}

ptb_status ptb_set_gemm_pairs(int32_t mode, int32_t* previous) {
  if (mode < -1 || mode > 1) return PTB_ERR_ARG;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (previous) *previous = ds->pairs;
  ds->pairs = mode;
  return PTB_OK;
}

ptb_status ptb_wait_probe(uint64_t limit_ns, ptb_stream stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return PTB_ERR_ARG;
  DeviceState* ds = nullptr;
  ptb_status st = device_state(&ds);
  if (st != PTB_OK) return st;
  return launch_status(launch_wait_probe(limit_ns, ds->status, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
