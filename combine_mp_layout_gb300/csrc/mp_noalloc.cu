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

#include <cuda.h>  // driver types only; the two driver calls are looked up at run time
#include <cuda_runtime.h>

#include "../../include/mp_layout.h"
#include "mp_common.cuh"
#include "mp_internal.h"

// Every call clears the scan's tile counter and finished-block counter, the
// first two words of the workspace control block.  The third word, the scan
// epoch, is kept on purpose: the tile records are tagged with it, and every
// scan that runs to its end advances it, so records left by earlier calls
// never match.  (A scan block that finds no tile to do leaves early without
// touching the epoch; that only happens when the counters were not zero, and
// then MP_ERR_INVALID_ARG is raised.)
static_assert(offsetof(mp::Control, scan_tile_counter) == 0 &&
                  offsetof(mp::Control, scan_done) == 4,
              "the counters cleared before every call are the first 8 bytes");

namespace {

// The scan's scratch.  Every GPU that loads this library holds these
// MP_NOALLOC_SCRATCH_BYTES until the process exits, and every call on that
// GPU shares them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
// Per device: the id of the context whose copy of the array was zero-filled
// (0: none yet).  A device reset creates a new context with a new id, and the
// array is set up again in it.
unsigned long long g_ready_ctx[kMaxDevices] = {0};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (cuCtxGetId), through
// driver entry points looked up once, so the library needs no link to the
// driver library itself.
bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault,
                                         &q1) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f2);
    looked_up = true;
  }
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS && *id != 0;
}

// The array's device address on the current device.  In host code the
// array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress (which also makes the device's context current).  The
// first call in a context zero-fills the array on `stream` and waits for that
// fill to finish, so no call can use the array before it is complete,
// whatever stream it runs on.
int scratch_for_current_device(unsigned char** out, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MP_ERR_CUDA;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
    return MP_ERR_CUDA;
  unsigned long long ctx = 0;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!current_context_id(&ctx)) return MP_ERR_CUDA;
  if (g_ready_ctx[dev] != ctx) {
    if (cudaMemsetAsync(ptr, 0, MP_NOALLOC_SCRATCH_BYTES, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return MP_ERR_CUDA;
    g_ready_ctx[dev] = ctx;
  }
  *out = static_cast<unsigned char*>(ptr);
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
  // Every host-side check first: a refused call puts nothing on the stream.
  const size_t need = mp_workspace_size(R, N, E);
  if (need == 0 || need > size_t(MP_NOALLOC_SCRATCH_BYTES)) return MP_ERR_INVALID_ARG;
  int st = mp::check_offsets_buffers(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                     num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                     recv_src_rank, recv_src_idx, recv_topk_idx,
                                     recv_topk_weights, dest_offsets, rank_prefix,
                                     num_recv_tokens_per_expert, send_row, dev_err);
  if (st == MP_OK)
    st = mp::check_rows_args(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                             recv_scales);
  if (st != MP_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* scratch = nullptr;
  st = scratch_for_current_device(&scratch, cs);
  if (st != MP_OK) return st;
  // The scan's tile counter and finished-block counter (the first 8 bytes) must
  // start at zero; the array keeps whatever the previous call left, so clear
  // them.
  if (cudaMemsetAsync(scratch, 0, 8, cs) != cudaSuccess) return MP_ERR_CUDA;
  return mp_dispatch(R, N, K, E, H, dtype, x, x_scales, topk_idx, topk_weights,
                     is_token_in_rank, num_tokens_per_rank, num_tokens_per_expert,
                     recv_capacity, recv_x, recv_scales, recv_src_rank, recv_src_idx,
                     recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                     num_recv_tokens_per_expert, send_row, dev_err, scratch, stream);
}
