// ptb_forward_noalloc: the PTB forward pass for callers that cannot allocate
// device memory.
//
// Some programs own every byte of device memory themselves (a framework's
// caching allocator, a serving process that reserves its memory at start-up
// and treats any later cudaMalloc as a failure because it can stall the
// device or fail under fragmentation, a plug-in whose host forbids raw
// allocations).  They cannot let the library grow its own arena and may have
// no buffer of their own to lend it.  For them the scratch that ptb_forward
// needs (the normalised activations and the fused projection output) lives
// in one fixed array compiled into the library, so a call allocates nothing.
//
// The array is a file-scope __device__ variable.  Its name in host code is
// only a host-side stand-in, so the host asks the runtime for its device
// address (cudaGetSymbolAddress) once per device, on the first call made
// with that device current, and hands that address to the kernels.
#include <mutex>

#include "ptb_device.cuh"

namespace {

// 64 MiB: enough for any layer whose workspace,
// T*H*2 + T*(3H+F)*2 bytes (each part rounded up to 256), fits in it --
// e.g. 2048 tokens of a 1024-wide layer with a 4096-wide MLP (32 MiB).
constexpr size_t kScratchBytes = 64ull << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" ptb_status ptb_forward_noalloc(const ptb_bf16* x, const ptb_bf16* ln_gamma,
                                          const ptb_bf16* ln_beta, const ptb_bf16* w_qkv,
                                          const ptb_bf16* w_o, const ptb_bf16* w_up,
                                          const ptb_bf16* w_down, int64_t batch, int64_t seq,
                                          int64_t hidden, int64_t ffn, int32_t heads,
                                          int32_t window, ptb_bf16* y, ptb_stream stream) {
  const int64_t limit = 1ll << 30;
  if (batch < 1 || seq < 1 || hidden < 1 || ffn < 1 || batch > limit || seq > limit ||
      hidden > limit || ffn > limit)
    return PTB_ERR_ARG;
  if (ptb_forward_workspace_size(batch, seq, hidden, ffn) > kScratchBytes)
    return PTB_ERR_WORKSPACE;  // the layer needs more scratch than the fixed array holds

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PTB_ERR_DEVICE;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr) {
        cudaGetLastError();
        return PTB_ERR_DEVICE;
      }
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  // Nothing in the scratch has to start at zero: every byte the kernels read
  // is written earlier in the same call.
  return ptb_forward(x, ln_gamma, ln_beta, w_qkv, w_o, w_up, w_down, batch, seq, hidden, ffn,
                     heads, window, y, scratch, kScratchBytes, stream);
}
