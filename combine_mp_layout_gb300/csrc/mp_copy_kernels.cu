// mp_copy_kernels.cu -- the HBM-bound payload kernels: dispatch row copy,
// combine (gather + fp32 sum), reduce-scatterv (fp32 sum of R inputs) and
// all-gatherv (one read, R writes).
//
// All four are streaming kernels: nothing is reused, so they are bound by
// HBM bandwidth and the design goal is bytes in flight.  Each runs a
// persistent grid (SM count x resident blocks) and splits the work into
// small units handed out round-robin to warps:
//   dispatch / combine : (token, slab) with a slab of 32 lanes x U 16-byte
//                        vectors of the token's row, so consecutive warps
//                        stream consecutive slabs of the same row and the
//                        per-SM load evens out across rows of unequal fan-out;
//   reduce-scatterv / all-gatherv : 16-byte vectors of the flat arrays.
// Payload moves as 16-byte vectors with L1-bypassing streaming loads.
#include <cstdint>

#include "mp_common.cuh"
#include "mp_internal.h"

namespace mp {

constexpr int kCopyThreads = 256;

// ---------------------------------------------------------------------------
// Dispatch copy ("MSCCLPP EP implementation", microsoft/mscclpp PR #852:
// intranode_dispatch moves each token row, as 16-byte vectors, to every rank
// that owns one of its experts).  One read of x, one write per receive row.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_dispatch(int R, int64_t tokens, int64_t vpr, const int4* __restrict__ x,
              int4* __restrict__ recv_x, int64_t recv_capacity,
              const int32_t* __restrict__ send_row, int spr,
              const float* __restrict__ x_scales, float* __restrict__ recv_scales) {
  const int lane = threadIdx.x & 31;
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * (kCopyThreads / kWarp);
  for (int64_t unit = int64_t(blockIdx.x) * (kCopyThreads / kWarp) + (threadIdx.x >> 5);
       unit < units; unit += nw) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    const int my = lane < R ? __ldg(send_row + tok * R + lane) : -1;
    unsigned vm = __ballot_sync(kFull, my >= 0 && int64_t(my) < recv_capacity);
    if (vm == 0) continue;
    const int64_t i0 = slab * slab_vec + lane;
    int4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kWarp < vpr) v[u] = ld_stream(x + tok * vpr + i0 + u * kWarp);
    while (vm) {
      const int d = __ffs(vm) - 1;
      vm &= vm - 1;
      const int64_t row = __shfl_sync(kFull, my, d);
      int4* dst = recv_x + row * vpr;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kWarp < vpr) st_stream(dst + i0 + u * kWarp, v[u]);
      if (spr > 0 && slab == 0)
        for (int c = lane; c < spr; c += kWarp)
          recv_scales[row * spr + c] = __ldg(x_scales + tok * spr + c);
    }
  }
}

// ---------------------------------------------------------------------------
// Combine (same page: intranode_combine runs in the reverse direction of
// dispatch).  out[s][t] = bf16_rn( sum_{d ascending} float(y[send_row[s][t][d]]) )
// from +0.0f.  Up to 8 source rows are loaded at once (memory-level
// parallelism) and then added strictly in ascending d.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(kCopyThreads, 2)
mp_k_combine(int R, int64_t tokens, int64_t vpr, const int4* __restrict__ y, int64_t y_rows,
             const int32_t* __restrict__ send_row, int4* __restrict__ out,
             int32_t* __restrict__ dev_err) {
  const int lane = threadIdx.x & 31;
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * (kCopyThreads / kWarp);
  for (int64_t unit = int64_t(blockIdx.x) * (kCopyThreads / kWarp) + (threadIdx.x >> 5);
       unit < units; unit += nw) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    int my = lane < R ? __ldg(send_row + tok * R + lane) : -1;
    if (my >= 0 && int64_t(my) >= y_rows) {
      if (slab == 0) raise_error(dev_err, MP_ERR_CAPACITY);
      my = -1;
    }
    unsigned vm = __ballot_sync(kFull, my >= 0);
    const int64_t i0 = slab * slab_vec + lane;
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[u][j] = 0.0f;
    while (vm) {
      int64_t rows[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rows[j] = -1;
        if (vm) {
          const int d = __ffs(vm) - 1;
          vm &= vm - 1;
          rows[j] = __shfl_sync(kFull, my, d);
        }
      }
      int4 v[8][U];
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (rows[j] >= 0 && i0 + u * kWarp < vpr)
            v[j][u] = ld_stream(y + rows[j] * vpr + i0 + u * kWarp);
#pragma unroll
      for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (rows[j] >= 0 && i0 + u * kWarp < vpr) add_bf16x8(acc[u], v[j][u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kWarp < vpr) st_stream(out + tok * vpr + i0 + u * kWarp, pack_bf16x8(acc[u]));
  }
}

// ---------------------------------------------------------------------------
// Reduce-scatterv ("Add pynccl all-gatherv and reducescatterv",
// vllm-project/vllm PR #20154: one reduce per root over its slice of every
// rank's input).  With all R inputs in one memory the R reduces are one
// element-wise fp32 sum over q ascending, rounded once; rank r's shard is a
// row range of the output.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCopyThreads)
mp_k_rsv(int R, int64_t nvec, const int4* __restrict__ in, int4* __restrict__ out) {
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads;
  for (int64_t i = int64_t(blockIdx.x) * kCopyThreads + threadIdx.x; i < nvec; i += stride) {
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int q0 = 0; q0 < R; q0 += 8) {
      int4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (q0 + j < R) v[j] = ld_stream(in + int64_t(q0 + j) * nvec + i);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (q0 + j < R) add_bf16x8(acc, v[j]);
    }
    st_stream(out + i, pack_bf16x8(acc));
  }
}

// ---------------------------------------------------------------------------
// All-gatherv (same page: one broadcast per root of its rows into every
// rank's output).  Every logical rank's copy is the concatenated shards, so
// each 16-byte vector is read once and written R times.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kCopyThreads)
mp_k_agv(int R, int64_t nvec, const int4* __restrict__ in, int4* __restrict__ out) {
  constexpr int U = 4;
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads * U;
  for (int64_t i0 = int64_t(blockIdx.x) * kCopyThreads * U + threadIdx.x; i0 < nvec;
       i0 += stride) {
    int4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kCopyThreads < nvec) v[u] = ld_stream(in + i0 + u * kCopyThreads);
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kCopyThreads < nvec) st_stream(out + int64_t(q) * nvec + i0 + u * kCopyThreads, v[u]);
  }
}

// ---------------------------------------------------------------------------
// Launchers: a persistent grid of (SMs x resident blocks) blocks, trimmed to
// the work available.
// ---------------------------------------------------------------------------
template <typename Kernel>
static int resident_blocks(Kernel k) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kCopyThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

static unsigned grid_for(int per_sm, int64_t work_items_per_block_unit, int64_t items) {
  const int64_t full = int64_t(sm_count()) * per_sm;
  const int64_t need = (items + work_items_per_block_unit - 1) / work_items_per_block_unit;
  return unsigned(need < 1 ? 1 : (need < full ? need : full));
}

constexpr int kDispatchU = 4;
constexpr int kCombineU = 2;

cudaError_t launch_dispatch_copy(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                 void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                 int scales_per_row,
                                 const float* x_scales, float* recv_scales, cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  static int per_sm = resident_blocks(mp_k_dispatch<kDispatchU>);
  const int64_t vpr = row_bytes / 16;
  const int64_t slabs = (vpr + kWarp * kDispatchU - 1) / (kWarp * kDispatchU);
  const unsigned grid = grid_for(per_sm, kCopyThreads / kWarp, tokens * slabs);
  mp_k_dispatch<kDispatchU><<<grid, kCopyThreads, 0, stream>>>(
      R, tokens, vpr, static_cast<const int4*>(x), static_cast<int4*>(recv_x), recv_capacity,
      send_row,
      scales_per_row, x_scales, recv_scales);
  return cudaGetLastError();
}

cudaError_t launch_combine(int R, int64_t tokens, int H, const void* y, int64_t y_rows,
                           const int32_t* send_row, void* out, int32_t* dev_err,
                           cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  static int per_sm = resident_blocks(mp_k_combine<kCombineU>);
  const int64_t vpr = int64_t(H) / 8;
  const int64_t slabs = (vpr + kWarp * kCombineU - 1) / (kWarp * kCombineU);
  const unsigned grid = grid_for(per_sm, kCopyThreads / kWarp, tokens * slabs);
  mp_k_combine<kCombineU><<<grid, kCopyThreads, 0, stream>>>(
      R, tokens, vpr, static_cast<const int4*>(y), y_rows, send_row, static_cast<int4*>(out),
      dev_err);
  return cudaGetLastError();
}

cudaError_t launch_reducescatterv(int R, int64_t S, int H, const void* in, void* out,
                                  cudaStream_t stream) {
  const int64_t nvec = S * H / 8;
  if (nvec == 0) return cudaSuccess;
  static int per_sm = resident_blocks(mp_k_rsv);
  const unsigned grid = grid_for(per_sm, kCopyThreads, nvec);
  mp_k_rsv<<<grid, kCopyThreads, 0, stream>>>(R, nvec, static_cast<const int4*>(in),
                                               static_cast<int4*>(out));
  return cudaGetLastError();
}

cudaError_t launch_allgatherv(int R, int64_t S, int64_t row_bytes, const void* in, void* out,
                              cudaStream_t stream) {
  const int64_t nvec = S * row_bytes / 16;
  if (nvec == 0) return cudaSuccess;
  static int per_sm = resident_blocks(mp_k_agv);
  const unsigned grid = grid_for(per_sm, kCopyThreads * 4, nvec);
  mp_k_agv<<<grid, kCopyThreads, 0, stream>>>(R, nvec, static_cast<const int4*>(in),
                                               static_cast<int4*>(out));
  return cudaGetLastError();
}

}  // namespace mp
