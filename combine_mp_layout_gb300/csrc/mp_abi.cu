// mp_abi.cu -- the C ABI declared in include/mp_layout.h: argument checks,
// workspace sizing and the launch sequence of each call.  No allocation,
// no synchronisation, no state kept between calls.
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mp_layout.h"
#include "mp_common.cuh"
#include "mp_internal.h"

namespace mp {

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 1;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static bool ep_shape_ok(int R, int N, int K, int E) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || K < 1 || K > MP_MAX_TOPK) return false;
  if (E < R || E > MP_MAX_EXPERTS || E % R != 0) return false;
  if (int64_t(R) * N * K >= (int64_t(1) << 31)) return false;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return false;
  return true;
}

static int check_layout_args(int R, int N, int K, int E, const int32_t* topk_idx,
                             const int32_t* num_tokens_per_rank,
                             const int32_t* num_tokens_per_expert,
                             const uint32_t* is_token_in_rank, const int32_t* dev_err,
                             const void* workspace) {
  if (!ep_shape_ok(R, N, K, E)) return MP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !dev_err || !workspace)
    return MP_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !is_token_in_rank)) return MP_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(num_tokens_per_rank) || !aligned4(num_tokens_per_expert) ||
      !aligned4(is_token_in_rank) || !aligned4(dev_err) || !aligned16(workspace))
    return MP_ERR_INVALID_ARG;
  return MP_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MP_OK : MP_ERR_CUDA; }

}  // namespace mp

using namespace mp;

extern "C" {

const char* mp_status_string(int status) {
  if (status == MP_OK) return "ok";
  if (status & MP_ERR_INVALID_ARG) return "invalid argument";
  if (status & MP_ERR_CUDA) return "CUDA launch failed";
  if (status & MP_ERR_CAPACITY) return "receive capacity exceeded";
  if (status & MP_ERR_BAD_EXPERT) return "expert id outside [-1, E)";
  if (status & MP_ERR_TIMEOUT) return "device-side wait timed out";
  return "unknown status";
}

size_t mp_workspace_size(int R, int N, int E) {
  if (!ep_shape_ok(R, N, 1, E)) return 0;
  return size_t(ws_total_bytes(R, N, E));
}

int mp_layout(int R, int N, int K, int E, const int32_t* topk_idx, int32_t* num_tokens_per_rank,
              int32_t* num_tokens_per_expert, uint32_t* is_token_in_rank, int32_t* dev_err,
              void* workspace, mp_stream_t stream) {
  const int st = check_layout_args(R, N, K, E, topk_idx, num_tokens_per_rank,
                                   num_tokens_per_expert, is_token_in_rank, dev_err, workspace);
  if (st != MP_OK) return st;
  return cuda_status(launch_layout(R, N, K, E, topk_idx, num_tokens_per_rank,
                                   num_tokens_per_expert, is_token_in_rank, dev_err,
                                   static_cast<unsigned char*>(workspace),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace mp {

// Checks shared by mp_dispatch, mp_dispatch_offsets and mp_dispatch_noalloc:
// every argument of the receive-offset scan except its workspace.
int check_offsets_buffers(int R, int N, int K, int E, const int32_t* topk_idx,
                          const float* topk_weights, const uint32_t* is_token_in_rank,
                          const int32_t* num_tokens_per_rank,
                          const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                          const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                          const int32_t* recv_topk_idx, const float* recv_topk_weights,
                          const int32_t* dest_offsets, const int32_t* rank_prefix,
                          const int32_t* num_recv_tokens_per_expert, const int32_t* send_row,
                          const int32_t* dev_err) {
  if (!ep_shape_ok(R, N, K, E) || recv_capacity < 0) return MP_ERR_INVALID_ARG;
  if (!num_tokens_per_rank || !num_tokens_per_expert || !dest_offsets || !rank_prefix ||
      !num_recv_tokens_per_expert || !dev_err)
    return MP_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !topk_weights || !is_token_in_rank || !send_row))
    return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 &&
      (!recv_src_rank || !recv_src_idx || !recv_topk_idx || !recv_topk_weights))
    return MP_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(topk_weights) ||
      !aligned4(is_token_in_rank) || !aligned4(send_row) || !aligned4(recv_src_rank) ||
      !aligned4(recv_src_idx) || !aligned4(recv_topk_idx) || !aligned4(recv_topk_weights) ||
      !aligned4(num_tokens_per_rank) || !aligned4(num_tokens_per_expert) ||
      !aligned4(dest_offsets) || !aligned4(rank_prefix) ||
      !aligned4(num_recv_tokens_per_expert) || !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  return MP_OK;
}

// The same with the caller's workspace (non-NULL, 16-byte aligned).
static int check_offsets_args(int R, int N, int K, int E, const int32_t* topk_idx,
                              const float* topk_weights, const uint32_t* is_token_in_rank,
                              const int32_t* num_tokens_per_rank,
                              const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                              const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                              const int32_t* recv_topk_idx, const float* recv_topk_weights,
                              const int32_t* dest_offsets, const int32_t* rank_prefix,
                              const int32_t* num_recv_tokens_per_expert, const int32_t* send_row,
                              const int32_t* dev_err, const void* workspace) {
  if (!workspace || !aligned16(workspace)) return MP_ERR_INVALID_ARG;
  return check_offsets_buffers(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                               num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                               recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                               dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                               dev_err);
}

// Checks shared by mp_dispatch, mp_dispatch_rows and mp_dispatch_noalloc.
int check_rows_args(int R, int N, int H, int dtype, const void* x, const float* x_scales,
                    const int32_t* send_row, int64_t recv_capacity, const void* recv_x,
                    const float* recv_scales) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || H <= 0 || recv_capacity < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (dtype != MP_BF16 && dtype != MP_E4M3) return MP_ERR_INVALID_ARG;
  const bool fp8 = dtype == MP_E4M3;
  if (fp8 ? (H % MP_SCALE_BLOCK != 0) : (H % 8 != 0)) return MP_ERR_INVALID_ARG;
  if (fp8 != (x_scales != nullptr) || fp8 != (recv_scales != nullptr)) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!x || !send_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && !recv_x) return MP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || !aligned4(x_scales) || !aligned4(recv_scales) ||
      !aligned4(send_row))
    return MP_ERR_INVALID_ARG;
  return MP_OK;
}

static cudaError_t launch_rows(int R, int N, int H, int dtype, const void* x,
                               const float* x_scales, const int32_t* send_row,
                               int64_t recv_capacity, void* recv_x, float* recv_scales,
                               cudaStream_t st) {
  const bool fp8 = dtype == MP_E4M3;
  const int64_t row_bytes = fp8 ? int64_t(H) : int64_t(H) * 2;
  return launch_dispatch_copy(R, int64_t(R) * N, row_bytes, x, recv_x, recv_capacity, send_row,
                              fp8 ? H / MP_SCALE_BLOCK : 0, x_scales, recv_scales, st);
}

}  // namespace mp

extern "C" {

int mp_dispatch_offsets(int R, int N, int K, int E, const int32_t* topk_idx,
                        const float* topk_weights, const uint32_t* is_token_in_rank,
                        const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                        int64_t recv_capacity, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* dest_offsets,
                        int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                        int32_t* send_row, int32_t* dev_err, void* workspace,
                        mp_stream_t stream) {
  const int st = check_offsets_args(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                    num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                    recv_src_rank, recv_src_idx, recv_topk_idx,
                                    recv_topk_weights, dest_offsets, rank_prefix,
                                    num_recv_tokens_per_expert, send_row, dev_err, workspace);
  if (st != MP_OK) return st;
  return cuda_status(launch_scan(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                 num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                 recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                                 dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                                 dev_err, static_cast<unsigned char*>(workspace),
                                 reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_offsets_global(int R, int N, int K, int E, const int32_t* topk_idx,
                               const float* topk_weights, const uint32_t* is_token_in_rank,
                               const int32_t* num_tokens_per_rank,
                               const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                               int32_t sentinel, int32_t* recv_src_rank, int32_t* recv_src_idx,
                               int32_t* recv_topk_idx, float* recv_topk_weights,
                               int32_t* dest_offsets, int32_t* rank_prefix,
                               int32_t* num_recv_tokens_per_expert, int32_t* send_row,
                               int32_t* dev_err, void* workspace, mp_stream_t stream) {
  const int st = check_offsets_args(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                    num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                    recv_src_rank, recv_src_idx, recv_topk_idx,
                                    recv_topk_weights, dest_offsets, rank_prefix,
                                    num_recv_tokens_per_expert, send_row, dev_err, workspace);
  if (st != MP_OK) return st;
  return cuda_status(launch_scan(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                 num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                 recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                                 dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                                 dev_err, static_cast<unsigned char*>(workspace),
                                 reinterpret_cast<cudaStream_t>(stream), 1, sentinel));
}

int mp_combine_weights(int R, int N, int K, const float* recv_topk_weights, int64_t recv_rows,
                       const int32_t* send_row, float* combined_topk_weights, int32_t* dev_err,
                       mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || K < 1 || K > MP_MAX_TOPK || recv_rows < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31) || int64_t(R) * N * K >= (int64_t(1) << 31))
    return MP_ERR_INVALID_ARG;
  if (!dev_err || (N > 0 && (!send_row || !combined_topk_weights)) ||
      (recv_rows > 0 && !recv_topk_weights))
    return MP_ERR_INVALID_ARG;
  if (!aligned4(recv_topk_weights) || !aligned4(send_row) || !aligned4(combined_topk_weights) ||
      !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_combine_weights(R, int64_t(R) * N, K, recv_topk_weights, recv_rows,
                                            send_row, combined_topk_weights, dev_err,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

int mp_layout_and_offsets(int R, int N, int K, int E, const int32_t* topk_idx,
                          const float* topk_weights, int64_t recv_capacity,
                          int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                          uint32_t* is_token_in_rank, int32_t* recv_src_rank,
                          int32_t* recv_src_idx, int32_t* recv_topk_idx,
                          float* recv_topk_weights, int32_t* dest_offsets, int32_t* rank_prefix,
                          int32_t* num_recv_tokens_per_expert, int32_t* send_row,
                          int32_t* dev_err, void* workspace, mp_stream_t stream) {
  int st = check_layout_args(R, N, K, E, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                             is_token_in_rank, dev_err, workspace);
  if (st == MP_OK)
    st = check_offsets_args(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                            num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                            recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                            dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                            dev_err, workspace);
  if (st != MP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  // small batches: one thread-block cluster; else one cooperative grid; else two launches
  cudaError_t e = launch_layout_cluster(
      R, N, K, E, topk_idx, topk_weights, recv_capacity, num_tokens_per_rank,
      num_tokens_per_expert, is_token_in_rank, recv_src_rank, recv_src_idx, recv_topk_idx,
      recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
      cs, /*meta=*/1);
  if (e == cudaSuccess) return MP_OK;
  if (e != cudaErrorNotSupported) return MP_ERR_CUDA;
  e = launch_layout_scan(
      R, N, K, E, topk_idx, topk_weights, recv_capacity, num_tokens_per_rank,
      num_tokens_per_expert, is_token_in_rank, recv_src_rank, recv_src_idx, recv_topk_idx,
      recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
      ws, cs);
  if (e == cudaSuccess) return MP_OK;
  if (e != cudaErrorNotSupported) return MP_ERR_CUDA;
  if (launch_layout(R, N, K, E, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                    is_token_in_rank, dev_err, ws, cs) != cudaSuccess)
    return MP_ERR_CUDA;
  return cuda_status(launch_scan(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                                 num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                                 recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                                 dest_offsets, rank_prefix, num_recv_tokens_per_expert,
                                 send_row, dev_err, ws, cs));
}

int mp_layout_dispatch(int R, int N, int K, int E, int H, int dtype, const void* x,
                       const float* x_scales, const int32_t* topk_idx,
                       const float* topk_weights, int64_t recv_capacity,
                       int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                       uint32_t* is_token_in_rank, void* recv_x, float* recv_scales,
                       int32_t* recv_src_rank, int32_t* recv_src_idx, int32_t* recv_topk_idx,
                       float* recv_topk_weights, int32_t* dest_offsets, int32_t* rank_prefix,
                       int32_t* num_recv_tokens_per_expert, int32_t* send_row, int32_t* dev_err,
                       void* workspace, mp_stream_t stream) {
  int st = check_layout_args(R, N, K, E, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                             is_token_in_rank, dev_err, workspace);
  if (st == MP_OK)
    st = check_offsets_args(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                            num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                            recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                            dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                            dev_err, workspace);
  if (st == MP_OK)
    st = check_rows_args(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                         recv_scales);
  if (st != MP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const bool fp8 = dtype == MP_E4M3;
  const int64_t row_bytes = fp8 ? int64_t(H) : int64_t(H) * 2;
  const int spr = fp8 ? H / MP_SCALE_BLOCK : 0;
  // small batches: one kernel whose blocks each count every token
  cudaError_t e = launch_layout_dispatch_fused(
      R, N, K, E, row_bytes, topk_idx, topk_weights, recv_capacity, num_tokens_per_rank,
      num_tokens_per_expert, is_token_in_rank, recv_src_rank, recv_src_idx, recv_topk_idx,
      recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, x, spr,
      x_scales, recv_x, recv_scales, dev_err, cs);
  if (e != cudaErrorNotSupported) return cuda_status(e);
  // else one launch for layout + offsets (receive metadata left out: a
  // thread-block cluster for small batches, else a cooperative grid), then the
  // row copy, which writes the metadata, as its programmatic dependent
  e = launch_layout_cluster(
      R, N, K, E, topk_idx, topk_weights, recv_capacity, num_tokens_per_rank,
      num_tokens_per_expert, is_token_in_rank, recv_src_rank, recv_src_idx, recv_topk_idx,
      recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row, dev_err,
      cs, /*meta=*/0);
  if (e == cudaErrorNotSupported)
    e = launch_layout_scan(
        R, N, K, E, topk_idx, topk_weights, recv_capacity, num_tokens_per_rank,
        num_tokens_per_expert, is_token_in_rank, recv_src_rank, recv_src_idx, recv_topk_idx,
        recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
        dev_err, ws, cs, /*meta=*/0);
  if (e == cudaSuccess)
    return cuda_status(launch_dispatch_after_offsets(
        R, N, K, E, row_bytes, x, recv_x, recv_capacity, send_row, spr, x_scales, recv_scales,
        topk_idx, topk_weights, recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
        cs));
  if (e != cudaErrorNotSupported) return MP_ERR_CUDA;
  // beyond one resident grid (or no tokens): layout, offsets and rows as three launches
  if (launch_layout(R, N, K, E, topk_idx, num_tokens_per_rank, num_tokens_per_expert,
                    is_token_in_rank, dev_err, ws, cs) != cudaSuccess ||
      launch_scan(R, N, K, E, topk_idx, topk_weights, is_token_in_rank, num_tokens_per_rank,
                  num_tokens_per_expert, recv_capacity, recv_src_rank, recv_src_idx,
                  recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                  num_recv_tokens_per_expert, send_row, dev_err, ws, cs) != cudaSuccess)
    return MP_ERR_CUDA;
  return cuda_status(launch_rows(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                                 recv_scales, cs));
}

int mp_dispatch_rows(int R, int N, int H, int dtype, const void* x, const float* x_scales,
                     const int32_t* send_row, int64_t recv_capacity, void* recv_x,
                     float* recv_scales, mp_stream_t stream) {
  const int st = check_rows_args(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                                 recv_scales);
  if (st != MP_OK) return st;
  return cuda_status(launch_rows(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                                 recv_scales, reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_rows_bulk(int R, int N, int H, int dtype, const void* x, const float* x_scales,
                          const int32_t* send_row, int64_t recv_capacity, void* recv_x,
                          float* recv_scales, int32_t* dev_err, mp_stream_t stream) {
  const int st = check_rows_args(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                                 recv_scales);
  if (st != MP_OK) return st;
  if (!dev_err || !aligned4(dev_err)) return MP_ERR_INVALID_ARG;
  const bool fp8 = dtype == MP_E4M3;
  return cuda_status(launch_dispatch_bulk(R, int64_t(R) * N, fp8 ? int64_t(H) : int64_t(H) * 2, x,
                                          recv_x, recv_capacity, send_row,
                                          fp8 ? H / MP_SCALE_BLOCK : 0, x_scales, recv_scales,
                                          dev_err, reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_rows_e4m3(int R, int N, int H, const void* x, const int32_t* send_row,
                          int64_t recv_capacity, void* recv_x, float* recv_scales,
                          mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || H <= 0 || H % MP_SCALE_BLOCK != 0 ||
      recv_capacity < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!x || !send_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && (!recv_x || !recv_scales)) return MP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || !aligned4(recv_scales) || !aligned4(send_row))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch_quant(R, int64_t(R) * N, H, x, recv_x, recv_scales, 0,
                                           recv_capacity, send_row,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_rows_mxfp8(int R, int N, int H, const void* x, const int32_t* send_row,
                           int64_t recv_capacity, void* recv_x, uint8_t* recv_scales,
                           mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || H <= 0 || H % 32 != 0 || recv_capacity < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!x || !send_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && (!recv_x || !recv_scales)) return MP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || !aligned4(send_row)) return MP_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch_quant(R, int64_t(R) * N, H, x, recv_x, recv_scales, 1,
                                           recv_capacity, send_row,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_rows_mxfp4(int R, int N, int H, const void* x, const int32_t* send_row,
                           int64_t recv_capacity, void* recv_x, uint8_t* recv_scales,
                           mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || H <= 0 || H % 32 != 0 || recv_capacity < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!x || !send_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && (!recv_x || !recv_scales)) return MP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || !aligned4(send_row)) return MP_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch_quant(R, int64_t(R) * N, H, x, recv_x, recv_scales, 2,
                                           recv_capacity, send_row,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch(int R, int N, int K, int E, int H, int dtype, const void* x, const float* x_scales,
                const int32_t* topk_idx, const float* topk_weights,
                const uint32_t* is_token_in_rank, const int32_t* num_tokens_per_rank,
                const int32_t* num_tokens_per_expert, int64_t recv_capacity, void* recv_x,
                float* recv_scales, int32_t* recv_src_rank, int32_t* recv_src_idx,
                int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* dest_offsets,
                int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert, int32_t* send_row,
                int32_t* dev_err, void* workspace, mp_stream_t stream) {
  int st = check_offsets_args(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                              num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                              recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                              dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                              dev_err, workspace);
  if (st == MP_OK)
    st = check_rows_args(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                         recv_scales);
  if (st != MP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch_scan(R, N, K, E, topk_idx, topk_weights, is_token_in_rank,
                              num_tokens_per_rank, num_tokens_per_expert, recv_capacity,
                              recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights,
                              dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
                              dev_err, static_cast<unsigned char*>(workspace), cs);
  if (e != cudaSuccess) return MP_ERR_CUDA;
  return cuda_status(launch_rows(R, N, H, dtype, x, x_scales, send_row, recv_capacity, recv_x,
                                 recv_scales, cs));
}

int mp_combine(int R, int N, int H, const void* y, int64_t y_rows, const int32_t* send_row,
               void* out, int32_t* dev_err, mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || H <= 0 || H % 8 != 0 || y_rows < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * R >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (!dev_err) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!send_row || !out || (y_rows > 0 && !y))) return MP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || !aligned4(send_row) || !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_combine(R, int64_t(R) * N, H, y, y_rows, send_row, out, dev_err,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int mp_reducescatterv(int R, int H, const int64_t* sizes, const void* in, void* out,
                      mp_stream_t stream) {
  if (R < 1 || H <= 0 || H % 8 != 0 || !sizes) return MP_ERR_INVALID_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return MP_ERR_INVALID_ARG;
    S += sizes[r];
  }
  if (S > 0 && (!in || !out || !aligned16(in) || !aligned16(out))) return MP_ERR_INVALID_ARG;
  return cuda_status(
      launch_reducescatterv(R, S, H, in, out, reinterpret_cast<cudaStream_t>(stream)));
}

int mp_allgatherv(int R, int64_t row_bytes, const int64_t* sizes, const void* in, void* out,
                  mp_stream_t stream) {
  if (R < 1 || row_bytes <= 0 || row_bytes % 16 != 0 || !sizes) return MP_ERR_INVALID_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return MP_ERR_INVALID_ARG;
    S += sizes[r];
  }
  if (S > 0 && (!in || !out || !aligned16(in) || !aligned16(out))) return MP_ERR_INVALID_ARG;
  return cuda_status(
      launch_allgatherv(R, S, row_bytes, in, out, reinterpret_cast<cudaStream_t>(stream)));
}

static int allgatherv_quant(int R, int H, int block, const int64_t* sizes, const void* in,
                            void* out, void* out_scales, int fmt, mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || H <= 0 || H % block != 0 || !sizes) return MP_ERR_INVALID_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return MP_ERR_INVALID_ARG;
    S += sizes[r];
  }
  if (S > 0 && (!in || !out || !out_scales || !aligned16(in) || !aligned16(out) ||
                (fmt == 0 && !aligned4(out_scales))))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_allgatherv_quant(R, S, H, in, out, out_scales, fmt,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int mp_allgatherv_e4m3(int R, int H, const int64_t* sizes, const void* in, void* out,
                       float* out_scales, mp_stream_t stream) {
  return allgatherv_quant(R, H, MP_SCALE_BLOCK, sizes, in, out, out_scales, 0, stream);
}

int mp_allgatherv_mxfp8(int R, int H, const int64_t* sizes, const void* in, void* out,
                        uint8_t* out_scales, mp_stream_t stream) {
  return allgatherv_quant(R, H, 32, sizes, in, out, out_scales, 1, stream);
}

int mp_allgatherv_mxfp4(int R, int H, const int64_t* sizes, const void* in, void* out,
                        uint8_t* out_scales, mp_stream_t stream) {
  return allgatherv_quant(R, H, 32, sizes, in, out, out_scales, 2, stream);
}

int mp_allgatherv_multi(int R, int ntensors, const int64_t* row_bytes, const int64_t* sizes,
                        const void* const* in, void* const* out, mp_stream_t stream) {
  if (R < 1 || ntensors < 1 || ntensors > MP_MAX_TENSORS || !row_bytes || !sizes || !in || !out)
    return MP_ERR_INVALID_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return MP_ERR_INVALID_ARG;
    S += sizes[r];
  }
  for (int j = 0; j < ntensors; ++j) {
    if (row_bytes[j] <= 0 || row_bytes[j] % 16 != 0) return MP_ERR_INVALID_ARG;
    if (S > 0 && (!in[j] || !out[j] || !aligned16(in[j]) || !aligned16(out[j])))
      return MP_ERR_INVALID_ARG;
  }
  return cuda_status(launch_allgatherv_multi(R, ntensors, row_bytes, S, in, out,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

static int ll_offsets_checked(int R, int N, int K, int E, int rank_major,
                              const int32_t* topk_idx, const int32_t* num_tokens_per_expert,
                              int64_t recv_capacity, int32_t* bin_offsets,
                              int32_t* bin_src_offsets, int32_t* recv_src_token,
                              int32_t* slot_row, int32_t* dev_err, mp_stream_t stream) {
  if (!ep_shape_ok(R, N, K, E) || recv_capacity < 0) return MP_ERR_INVALID_ARG;
  if (!bin_offsets || !bin_src_offsets || !dev_err) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !slot_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && !recv_src_token) return MP_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(num_tokens_per_expert) || !aligned4(bin_offsets) ||
      !aligned4(bin_src_offsets) || !aligned4(recv_src_token) || !aligned4(slot_row) ||
      !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_ll_offsets(R, N, K, E, rank_major, topk_idx, num_tokens_per_expert,
                                       recv_capacity, bin_offsets, bin_src_offsets,
                                       recv_src_token, slot_row, dev_err,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_ll_offsets(int R, int N, int K, int E, const int32_t* topk_idx,
                           const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                           int32_t* expert_offsets, int32_t* expert_src_offsets,
                           int32_t* recv_src_token, int32_t* slot_row, int32_t* dev_err,
                           mp_stream_t stream) {
  return ll_offsets_checked(R, N, K, E, 0, topk_idx, num_tokens_per_expert, recv_capacity,
                            expert_offsets, expert_src_offsets, recv_src_token, slot_row, dev_err,
                            stream);
}

int mp_dispatch_ll_offsets_rank_major(int R, int N, int K, int E, const int32_t* topk_idx,
                                      const int32_t* num_tokens_per_expert,
                                      int64_t recv_capacity, int32_t* dest_offsets,
                                      int32_t* dest_src_offsets, int32_t* recv_src_token,
                                      int32_t* slot_row, int32_t* dev_err, mp_stream_t stream) {
  return ll_offsets_checked(R, N, K, E, 1, topk_idx, num_tokens_per_expert, recv_capacity,
                            dest_offsets, dest_src_offsets, recv_src_token, slot_row, dev_err,
                            stream);
}

int mp_dispatch_ll_rows(int R, int N, int K, int H, int dtype, const void* x,
                        const float* x_scales, const int32_t* slot_row, int64_t recv_capacity,
                        void* recv_x, float* recv_scales, mp_stream_t stream) {
  if (K < 1 || K > MP_MAX_TOPK || R < 1 || R > MP_MAX_RANKS) return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * K >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  // the row copy with the K top-k slots of a token in place of its R destinations
  const int st = check_rows_args(1, N, H, dtype, x, x_scales, slot_row, recv_capacity, recv_x,
                                 recv_scales);
  if (st != MP_OK) return st;
  const bool fp8 = dtype == MP_E4M3;
  const int64_t row_bytes = fp8 ? int64_t(H) : int64_t(H) * 2;
  return cuda_status(launch_dispatch_copy(K, int64_t(R) * N, row_bytes, x, recv_x, recv_capacity,
                                          slot_row, fp8 ? H / MP_SCALE_BLOCK : 0, x_scales,
                                          recv_scales, reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_ll(int R, int N, int K, int E, int H, int dtype, int rank_major, const void* x,
                   const float* x_scales, const int32_t* topk_idx,
                   const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                   int32_t* bin_offsets, int32_t* bin_src_offsets, int32_t* recv_src_token,
                   int32_t* slot_row, void* recv_x, float* recv_scales, int32_t* dev_err,
                   mp_stream_t stream) {
  if (!ep_shape_ok(R, N, K, E) || recv_capacity < 0 || (rank_major != 0 && rank_major != 1))
    return MP_ERR_INVALID_ARG;
  if (!bin_offsets || !bin_src_offsets || !dev_err) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!topk_idx || !slot_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && !recv_src_token) return MP_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(num_tokens_per_expert) || !aligned4(bin_offsets) ||
      !aligned4(bin_src_offsets) || !aligned4(recv_src_token) || !aligned4(slot_row) ||
      !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  const int st = check_rows_args(1, N, H, dtype, x, x_scales, slot_row, recv_capacity, recv_x,
                                 recv_scales);
  if (st != MP_OK) return st;
  const bool fp8 = dtype == MP_E4M3;
  return cuda_status(launch_ll_dispatch(
      R, N, K, E, rank_major, fp8 ? int64_t(H) : int64_t(H) * 2, topk_idx, num_tokens_per_expert,
      recv_capacity, bin_offsets, bin_src_offsets, recv_src_token, slot_row, x,
      fp8 ? H / MP_SCALE_BLOCK : 0, x_scales, recv_x, recv_scales, dev_err,
      reinterpret_cast<cudaStream_t>(stream)));
}

static int ll_quant_rows_checked(int R, int N, int K, int H, int qformat, const void* x,
                                 const int32_t* slot_row, int64_t recv_capacity,
                                 const void* recv_x, const void* recv_scales) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || K < 1 || K > MP_MAX_TOPK || H <= 0 ||
      recv_capacity < 0)
    return MP_ERR_INVALID_ARG;
  if (qformat != MP_Q_E4M3 && qformat != MP_Q_MXFP8 && qformat != MP_Q_MXFP4)
    return MP_ERR_INVALID_ARG;
  if (H % (qformat == MP_Q_E4M3 ? MP_SCALE_BLOCK : 32) != 0) return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * K >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (N > 0 && (!x || !slot_row)) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && (!recv_x || !recv_scales)) return MP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(recv_x) || !aligned4(slot_row) ||
      (qformat == MP_Q_E4M3 && !aligned4(recv_scales)))
    return MP_ERR_INVALID_ARG;
  return MP_OK;
}

int mp_dispatch_ll_rows_quant(int R, int N, int K, int H, int qformat, const void* x,
                              const int32_t* slot_row, int64_t recv_capacity, void* recv_x,
                              void* recv_scales, mp_stream_t stream) {
  const int st = ll_quant_rows_checked(R, N, K, H, qformat, x, slot_row, recv_capacity, recv_x,
                                       recv_scales);
  if (st != MP_OK) return st;
  // the quantising copy with the K top-k slots of a token in place of its R destinations
  return cuda_status(launch_dispatch_quant(K, int64_t(R) * N, H, x, recv_x, recv_scales, qformat,
                                           recv_capacity, slot_row,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int mp_dispatch_ll_quant(int R, int N, int K, int E, int H, int qformat, int rank_major,
                         const void* x, const int32_t* topk_idx,
                         const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                         int32_t* bin_offsets, int32_t* bin_src_offsets, int32_t* recv_src_token,
                         int32_t* slot_row, void* recv_x, void* recv_scales, int32_t* dev_err,
                         mp_stream_t stream) {
  if (!ep_shape_ok(R, N, K, E) || recv_capacity < 0 || (rank_major != 0 && rank_major != 1))
    return MP_ERR_INVALID_ARG;
  if (!bin_offsets || !bin_src_offsets || !dev_err) return MP_ERR_INVALID_ARG;
  if (N > 0 && !topk_idx) return MP_ERR_INVALID_ARG;
  if (recv_capacity > 0 && !recv_src_token) return MP_ERR_INVALID_ARG;
  if (!aligned4(topk_idx) || !aligned4(num_tokens_per_expert) || !aligned4(bin_offsets) ||
      !aligned4(bin_src_offsets) || !aligned4(recv_src_token) || !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  const int st = ll_quant_rows_checked(R, N, K, H, qformat, x, slot_row, recv_capacity, recv_x,
                                       recv_scales);
  if (st != MP_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // small batches counting themselves: one kernel
  if (num_tokens_per_expert == nullptr) {
    const cudaError_t f = launch_ll_dispatch_quant_fused(
        R, N, K, E, rank_major, H, qformat, topk_idx, recv_capacity, bin_offsets,
        bin_src_offsets, recv_src_token, slot_row, x, recv_x, recv_scales, dev_err, cs);
    if (f != cudaErrorNotSupported) return cuda_status(f);
  }
  // else the sort, then the quantising row copy as its programmatic dependent
  const cudaError_t e = launch_ll_offsets(R, N, K, E, rank_major, topk_idx,
                                          num_tokens_per_expert, recv_capacity, bin_offsets,
                                          bin_src_offsets, recv_src_token, slot_row, dev_err, cs);
  if (e != cudaSuccess || N == 0) return cuda_status(e);
  return cuda_status(launch_dispatch_quant(K, int64_t(R) * N, H, x, recv_x, recv_scales, qformat,
                                           recv_capacity, slot_row, cs, /*dependent=*/true));
}

int mp_combine_ll(int R, int N, int K, int H, const void* y, int64_t y_rows,
                  const int32_t* slot_row, const float* topk_weights, void* out,
                  int32_t* dev_err, mp_stream_t stream) {
  if (R < 1 || R > MP_MAX_RANKS || N < 0 || K < 1 || K > MP_MAX_TOPK || H <= 0 || H % 8 != 0 ||
      y_rows < 0)
    return MP_ERR_INVALID_ARG;
  if (int64_t(R) * N * K >= (int64_t(1) << 31)) return MP_ERR_INVALID_ARG;
  if (!dev_err || (N > 0 && (!slot_row || !topk_weights || !out || (y_rows > 0 && !y))))
    return MP_ERR_INVALID_ARG;
  if (!aligned16(y) || !aligned16(out) || !aligned4(slot_row) || !aligned4(topk_weights) ||
      !aligned4(dev_err))
    return MP_ERR_INVALID_ARG;
  return cuda_status(launch_combine_weighted(K, int64_t(R) * N, H, y, y_rows, slot_row,
                                             topk_weights, out, dev_err,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
