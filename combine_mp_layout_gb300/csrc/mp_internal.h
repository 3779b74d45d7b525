// mp_internal.h -- launchers shared between the kernel files and the C ABI.
// Arguments are validated by the C ABI before any launcher is called.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mp {

// SM count of the current device (cached per device).
int sm_count();

// Host-side argument checks of mp_dispatch (MP_OK or MP_ERR_INVALID_ARG):
// the receive-offset scan's arguments without its workspace, and the row
// copy's.
int check_offsets_buffers(int R, int N, int K, int E, const int32_t* topk_idx,
                          const float* topk_weights, const uint32_t* is_token_in_rank,
                          const int32_t* num_tokens_per_rank,
                          const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                          const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                          const int32_t* recv_topk_idx, const float* recv_topk_weights,
                          const int32_t* dest_offsets, const int32_t* rank_prefix,
                          const int32_t* num_recv_tokens_per_expert, const int32_t* send_row,
                          const int32_t* dev_err);
int check_rows_args(int R, int N, int H, int dtype, const void* x, const float* x_scales,
                    const int32_t* send_row, int64_t recv_capacity, const void* recv_x,
                    const float* recv_scales);

cudaError_t launch_layout(int R, int N, int K, int E, const int32_t* topk_idx,
                          int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                          uint32_t* is_token_in_rank, int32_t* dev_err, unsigned char* ws,
                          cudaStream_t stream);

cudaError_t launch_scan(int R, int N, int K, int E, const int32_t* topk_idx,
                        const float* topk_weights, const uint32_t* is_token_in_rank,
                        const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                        int64_t recv_capacity, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* dest_offsets,
                        int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                        int32_t* send_row, int32_t* dev_err, unsigned char* ws,
                        cudaStream_t stream, int global_ids = 0, int32_t sentinel = -1);

// mp_k_layout + mp_k_scan as one cooperative launch; cudaErrorNotSupported
// (nothing launched) when the problem does not fit one resident grid.  With
// meta = 0 the receive metadata (recv_src_rank, recv_src_idx, recv_topk_idx,
// recv_topk_weights) is not written: launch_dispatch_after_offsets writes it.
cudaError_t launch_layout_scan(int R, int N, int K, int E, const int32_t* topk_idx,
                               const float* topk_weights, int64_t recv_capacity,
                               int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                               uint32_t* is_token_in_rank, int32_t* recv_src_rank,
                               int32_t* recv_src_idx, int32_t* recv_topk_idx,
                               float* recv_topk_weights, int32_t* dest_offsets,
                               int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                               int32_t* send_row, int32_t* dev_err, unsigned char* ws,
                               cudaStream_t stream, int meta = 1);

// Layout + offsets for small batches (R <= 16, N <= MP_CLUSTER_MAX_TOKENS) in
// one thread-block cluster, one CTA per source rank, exchanging counts through
// distributed shared memory (no workspace); cudaErrorNotSupported (nothing
// launched) when the shape or the device does not suit it.  meta as above.
cudaError_t launch_layout_cluster(int R, int N, int K, int E, const int32_t* topk_idx,
                                  const float* topk_weights, int64_t recv_capacity,
                                  int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                                  uint32_t* is_token_in_rank, int32_t* recv_src_rank,
                                  int32_t* recv_src_idx, int32_t* recv_topk_idx,
                                  float* recv_topk_weights, int32_t* dest_offsets,
                                  int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                                  int32_t* send_row, int32_t* dev_err, cudaStream_t stream,
                                  int meta);

// The row copy of mp_layout_dispatch, launched as the programmatic dependent of
// the fused layout + offsets kernel right before it on the stream: its first
// row loads (and the tokens' top-k ids and weights) overlap that kernel, its
// send_row reads wait for it.  Besides the rows (and e4m3 scales) it writes the
// receive metadata: recv_src_rank / recv_src_idx and the local top-k ids and
// weights of every receive row.
cudaError_t launch_dispatch_after_offsets(int R, int N, int K, int E, int64_t row_bytes,
                                          const void* x, void* recv_x, int64_t recv_capacity,
                                          const int32_t* send_row, int scales_per_row,
                                          const float* x_scales, float* recv_scales,
                                          const int32_t* topk_idx, const float* topk_weights,
                                          int32_t* recv_src_rank, int32_t* recv_src_idx,
                                          int32_t* recv_topk_idx, float* recv_topk_weights,
                                          cudaStream_t stream);

// Low-latency offsets, expert-major (rank_major = 0: bins are experts) or
// rank-major (1: bins are the ranks owning the experts); one block per source
// rank.
cudaError_t launch_ll_offsets(int R, int N, int K, int E, int rank_major,
                              const int32_t* topk_idx, const int32_t* num_tokens_per_expert,
                              int64_t recv_capacity, int32_t* bin_offsets,
                              int32_t* bin_src_offsets, int32_t* recv_src_token,
                              int32_t* slot_row, int32_t* dev_err, cudaStream_t stream);

// launch_ll_offsets followed by the row copy of each (token, top-k slot) to
// its slot row, launched as the sort's programmatic dependent.
cudaError_t launch_ll_dispatch(int R, int N, int K, int E, int rank_major, int64_t row_bytes,
                               const int32_t* topk_idx, const int32_t* num_tokens_per_expert,
                               int64_t recv_capacity, int32_t* bin_offsets,
                               int32_t* bin_src_offsets, int32_t* recv_src_token,
                               int32_t* slot_row, const void* x, int scales_per_row,
                               const float* x_scales, void* recv_x, float* recv_scales,
                               int32_t* dev_err, cudaStream_t stream);

// The low-latency dispatch as one kernel whose blocks each count all R*N*K
// ids (small batches with num_tokens_per_expert NULL): the same outputs as
// launch_ll_dispatch.  cudaErrorNotSupported, with nothing launched, when the
// problem is outside its limits.
cudaError_t launch_ll_dispatch_fused(int R, int N, int K, int E, int rank_major,
                                     int64_t row_bytes, const int32_t* topk_idx,
                                     int64_t recv_capacity, int32_t* bin_offsets,
                                     int32_t* bin_src_offsets, int32_t* recv_src_token,
                                     int32_t* slot_row, const void* x, int scales_per_row,
                                     const float* x_scales, void* recv_x, float* recv_scales,
                                     int32_t* dev_err, cudaStream_t stream);

// mp_dispatch_ll_quant as one kernel (blocks each count every id, then
// quantise their tokens' rows); fmt is MP_Q_E4M3 / MP_Q_MXFP8 / MP_Q_MXFP4.
// cudaErrorNotSupported, with nothing launched, outside its limits.
cudaError_t launch_ll_dispatch_quant_fused(int R, int N, int K, int E, int rank_major, int H,
                                           int fmt, const int32_t* topk_idx,
                                           int64_t recv_capacity, int32_t* bin_offsets,
                                           int32_t* bin_src_offsets, int32_t* recv_src_token,
                                           int32_t* slot_row, const void* x, void* recv_x,
                                           void* recv_scales, int32_t* dev_err,
                                           cudaStream_t stream);

// The whole high-throughput dispatch (mp_layout_dispatch's outputs) as one
// kernel whose blocks each count every token, for small batches.
// cudaErrorNotSupported, with nothing launched, outside its limits.
cudaError_t launch_layout_dispatch_fused(
    int R, int N, int K, int E, int64_t row_bytes, const int32_t* topk_idx,
    const float* topk_weights, int64_t recv_capacity, int32_t* num_tokens_per_rank,
    int32_t* num_tokens_per_expert, uint32_t* is_token_in_rank, int32_t* recv_src_rank,
    int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
    int32_t* dest_offsets, int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
    int32_t* send_row, const void* x, int scales_per_row, const float* x_scales, void* recv_x,
    float* recv_scales, int32_t* dev_err, cudaStream_t stream);

// The low-latency row copy launched as a programmatic dependent of the kernel
// before it on the stream (the LL sort): its row loads overlap that kernel,
// its slot_row reads wait for it.  Only for use right after the sort.
cudaError_t launch_ll_rows_after_sort(int K, int64_t tokens, int64_t row_bytes, const void* x,
                                      void* recv_x, int64_t recv_capacity,
                                      const int32_t* slot_row, int scales_per_row,
                                      const float* x_scales, float* recv_scales,
                                      cudaStream_t stream);

// out[t] = bf16( sum over k ascending of weights[t][k] * y[slot_row[t][k]] )
cudaError_t launch_combine_weighted(int K, int64_t tokens, int H, const void* y, int64_t y_rows,
                                    const int32_t* slot_row, const float* weights, void* out,
                                    int32_t* dev_err, cudaStream_t stream);

// combined[t][k] = sum over d ascending of recv_topk_weights[send_row[t][d]][k]
cudaError_t launch_combine_weights(int R, int64_t tokens, int K, const float* recv_topk_weights,
                                   int64_t recv_rows, const int32_t* send_row, float* combined,
                                   int32_t* dev_err, cudaStream_t stream);

// Copies token rows (row_bytes each, a multiple of 16) to every receive row
// listed in send_row; scales_per_row fp32 scales travel with each row.
cudaError_t launch_dispatch_copy(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                 void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                 int scales_per_row,
                                 const float* x_scales, float* recv_scales, cudaStream_t stream);

// The same copy as launch_dispatch_copy through the bulk-copy (TMA) engine:
// cp.async.bulk loads into a shared-memory ring and bulk stores per
// destination; its bounded mbarrier waits report MP_ERR_TIMEOUT in dev_err.
cudaError_t launch_dispatch_bulk(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                 void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                 int scales_per_row, const float* x_scales, float* recv_scales,
                                 int32_t* dev_err, cudaStream_t stream);

// Quantises bf16 token rows -- fmt 0: e4m3 with one fp32 scale per 128
// channels; 1: MXFP8 (e4m3, one UE8M0 byte per 32 channels); 2: MXFP4 (two
// e2m1 codes per byte, one UE8M0 byte per 32 channels) -- and copies them to
// every receive row listed in send_row (R entries per token; the K slot rows
// of the low-latency layout work the same way).  dependent: launched as the
// programmatic dependent of the kernel before it (the LL sort writing the
// destinations), its blocks waiting for that kernel before they read them.
cudaError_t launch_dispatch_quant(int R, int64_t tokens, int H, const void* x, void* recv_x,
                                  void* recv_scales, int fmt, int64_t recv_capacity,
                                  const int32_t* send_row, cudaStream_t stream,
                                  bool dependent = false);

cudaError_t launch_combine(int R, int64_t tokens, int H, const void* y, int64_t y_rows,
                           const int32_t* send_row, void* out, int32_t* dev_err,
                           cudaStream_t stream);

cudaError_t launch_reducescatterv(int R, int64_t S, int H, const void* in, void* out,
                                  cudaStream_t stream);

// Quantises each of the S bf16 rows of `in` once (scales as in
// launch_dispatch_quant) and writes codes and scales to all R logical ranks'
// copies: out[q][i] and out_scales[q][i] for q < R.
cudaError_t launch_allgatherv_quant(int R, int64_t S, int H, const void* in, void* out,
                                    void* out_scales, int fmt, cudaStream_t stream);
cudaError_t launch_allgatherv(int R, int64_t S, int64_t row_bytes, const void* in, void* out,
                              cudaStream_t stream);

// All-gatherv of n tensors (row_bytes[j] bytes per row, multiples of 16) with
// the same S gathered rows, in one launch.
cudaError_t launch_allgatherv_multi(int R, int n, const int64_t* row_bytes, int64_t S,
                                    const void* const* in, void* const* out, cudaStream_t stream);

}  // namespace mp
