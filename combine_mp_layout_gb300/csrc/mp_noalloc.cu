// mp_noalloc.cu -- mp_dispatch_noalloc: mp_dispatch without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// The receive-offset scan needs a little scratch memory of its own (a block of
// counters and one state word per (tile, destination)).  mp_dispatch takes it
// as a caller-allocated workspace.  Some callers cannot make that allocation:
// a host application that reserves (nearly) all device memory for its own pool
// at start-up, a plugin whose host framework owns every device allocation, or
// a latency-critical loop in which cudaMalloc / cudaFree would synchronise the
// device.  For them this file keeps the scratch in a fixed-size array in the
// library's own device memory and passes its address to the unchanged
// mp_dispatch.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/mp_layout.h"
#include "mp_common.cuh"

// The counters cleared before every call are the first two words of the
// workspace control block.
static_assert(offsetof(mp::Control, scan_tile_counter) == 0 &&
                  offsetof(mp::Control, scan_done) == 4 && offsetof(mp::Control, scan_epoch) == 8,
              "control block layout");

namespace {

// The scan's scratch.  Every GPU that loads this library holds these
// MP_NOALLOC_SCRATCH_BYTES until the process exits, and every call on that
// GPU shares them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Once per device, with that device current: find the device address of the
// array (in host code its name is only a host-side stand-in) and zero it.
int scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return MP_ERR_CUDA;
    if (cudaMemset(ptr, 0, MP_NOALLOC_SCRATCH_BYTES) != cudaSuccess) return MP_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return MP_OK;
}

}  // namespace

extern "C" int mp_dispatch_noalloc(int R, int N, int K, int E, int H, int dtype, const void* x,
                                   const float* x_scales, const int32_t* topk_idx,
                                   const float* topk_weights, const uint32_t* is_token_in_rank,
                                   const int32_t* num_tokens_per_rank,
                                   const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                                   void* recv_x, float* recv_scales, int32_t* recv_src_rank,
                                   int32_t* recv_src_idx, int32_t* recv_topk_idx,
                                   float* recv_topk_weights, int32_t* dest_offsets,
                                   int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                                   int32_t* send_row, int32_t* dev_err, mp_stream_t stream) {
  const size_t need = mp_workspace_size(R, N, E);
  if (need == 0 || need > size_t(MP_NOALLOC_SCRATCH_BYTES)) return MP_ERR_INVALID_ARG;
  unsigned char* scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != MP_OK) return st;
  // The scan's tile counter and finished-block counter (the first 8 bytes) must
  // start at zero; the array keeps whatever the previous call left, so clear
  // them.  The tile states need no clearing: each launch tags its own.
  if (cudaMemsetAsync(scratch, 0, 8, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MP_ERR_CUDA;
  return mp_dispatch(R, N, K, E, H, dtype, x, x_scales, topk_idx, topk_weights,
                     is_token_in_rank, num_tokens_per_rank, num_tokens_per_expert,
                     recv_capacity, recv_x, recv_scales, recv_src_rank, recv_src_idx,
                     recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                     num_recv_tokens_per_expert, send_row, dev_err, scratch, stream);
}
