// dcp_mla_decode_partial_noalloc: the decode entry point for callers that
// cannot allocate device memory.
//
// Some callers have no way to hand the library a scratch buffer: runtimes
// whose device memory is owned and fully reserved by a host framework,
// allocator-free embedded or real-time integrations, and plugins that are
// only given the input and output tensors.  The split-KV decode needs scratch
// for its per-split partial results, so this entry point takes it from a
// fixed array that lives in the library itself, instead of from a
// `workspace` argument.
//
// Rules for users:
//   - The array holds kNoAllocScratchBytes (24 MiB) on every device that
//     loads the library, for the life of the process.  That covers the split
//     plans of any call with H <= 128 heads on a GB300; a call whose plan
//     needs more returns DCP_ERR_WORKSPACE_TOO_SMALL without launching.
//   - The first call on a device looks up the array's device address (a
//     runtime query, no allocation); make that first call before capturing a
//     stream on that device.
//   - All calls share the one array and it keeps the last call's contents.
//     Nothing in it needs to start at zero (every split partial is written
//     before it is read), but two calls whose kernels overlap on the GPU race
//     on it: serialise them (one stream, or events).
// Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include "dcp_kernels.h"

#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device (nullptr on
// failure).  The host-side symbol is only a stand-in; the address must come
// from the runtime, per device.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_addr[dev] = p;
  }
  return g_addr[dev];
}

}  // namespace

extern "C" {

dcp_status_t dcp_mla_decode_partial_noalloc(
    const void* q, int64_t q_stride_tok, const void* kv_cache, int32_t num_blocks, int32_t block_size,
    const int32_t* block_table, int32_t bt_width, int64_t bt_stride, const int32_t* seq_lens,
    const int32_t* query_start_loc, int32_t B, int32_t T, int32_t H, int32_t max_seq_len, int32_t max_q_len,
    int32_t D, int32_t interleave, float scale, float* O_part, float* lse_part, int32_t* dev_error,
    void* stream) {
  const size_t need = dcp_decode_workspace_size(B, T, H, D, max_seq_len, max_q_len);
  if (need == static_cast<size_t>(-1)) return DCP_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return DCP_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (need > 0) {
    ws = scratch_address();
    if (!ws) return DCP_ERR_CUDA;
  }
  return dcp_mla_decode_partial(q, q_stride_tok, kv_cache, num_blocks, block_size, block_table, bt_width,
                                bt_stride, seq_lens, query_start_loc, B, T, H, max_seq_len, max_q_len, D, interleave,
                                scale, O_part, lse_part, ws, ws ? kNoAllocScratchBytes : 0, dev_error, stream);
}

}  // extern "C"
