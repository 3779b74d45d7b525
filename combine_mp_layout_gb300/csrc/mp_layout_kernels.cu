// mp_layout_kernels.cu -- the routing layout and the receive-offset scan.
//
// Layout ("MSCCLPP EP implementation", microsoft/mscclpp PR #852, port
// scope: get_dispatch_layout computes counts and token-in-rank).  One block
// per (source rank, 256-token slice); warp ballots build the per-rank
// counts, a shared-memory histogram the per-expert counts.  The last block
// of each source rank to finish adds the per-block partials in block order.
//
// Scan (the counterpart of the notify/prefix-matrix step of the same port,
// here a single-pass decoupled lookback).  The receive row of token (s,t)
// at destination d is
//     dest_base[d] + #{(s',t') < (s,t) in flattened order with bit d},
// dest_base[d] = rows of all destinations < d.  The flattened (s,t) axis is
// cut into 256-token tiles; each tile publishes its R-wide count vector,
// looks back over its predecessors for the exclusive prefix, publishes the
// inclusive prefix and writes the rows' metadata.  Tiles are handed out in
// launch order through an atomic counter, so every tile a block waits on
// belongs to a block that is already running.
#include <cstdint>

#include "mp_common.cuh"
#include "mp_internal.h"

namespace mp {

// ---------------------------------------------------------------------------
// Layout
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kLayoutTokens)
mp_k_layout(int R, int N, int K, int E, const int32_t* __restrict__ topk_idx,
            int32_t* __restrict__ num_tokens_per_rank, int32_t* __restrict__ num_tokens_per_expert,
            uint32_t* __restrict__ is_token_in_rank, int32_t* __restrict__ dev_err,
            unsigned char* __restrict__ ws) {
  extern __shared__ int32_t sm_layout[];
  int32_t* hist = sm_layout;            // [E]
  int32_t* rcount = sm_layout + E;      // [R]
  int32_t* idx_s = rcount + MP_MAX_RANKS;  // [kLayoutTokens * K]
  __shared__ int last_block;

  const int s = blockIdx.y;
  const int c = blockIdx.x;
  const int C = gridDim.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int El = E / R;
  const int t0 = c * kLayoutTokens;
  const int ntok = min(kLayoutTokens, N - t0);

  for (int i = tid; i < E; i += blockDim.x) hist[i] = 0;
  if (tid < MP_MAX_RANKS) rcount[tid] = 0;
  // stage this slice's topk_idx with coalesced loads
  const int32_t* src = topk_idx + (int64_t(s) * N + t0) * K;
  for (int i = tid; i < ntok * K; i += blockDim.x) idx_s[i] = src[i];
  __syncthreads();

  uint32_t mask = 0;
  int bad = 0;
  if (tid < ntok) {
    for (int k = 0; k < K; ++k) {
      const int e = idx_s[tid * K + k];
      if (e == -1) continue;
      if (e < -1 || e >= E) { bad = 1; continue; }
      atomicAdd(&hist[e], 1);
      mask |= 1u << (e / El);
    }
    is_token_in_rank[int64_t(s) * N + t0 + tid] = mask;
  }
  if (__any_sync(kFull, bad) && lane == 0) raise_error(dev_err, MP_ERR_BAD_EXPERT);
  for (int d = 0; d < R; ++d) {
    const unsigned b = __ballot_sync(kFull, (mask >> d) & 1u);
    if (lane == 0 && b) atomicAdd(&rcount[d], __popc(b));
  }
  __syncthreads();

  if (C == 1) {  // the only block of this source rank writes the result itself
    for (int i = tid; i < E; i += blockDim.x) num_tokens_per_expert[int64_t(s) * E + i] = hist[i];
    if (tid < R) num_tokens_per_rank[s * R + tid] = rcount[tid];
    return;
  }

  Control* ctl = reinterpret_cast<Control*>(ws);
  int32_t* part = reinterpret_cast<int32_t*>(ws + ws_partials_offset()) +
                  (int64_t(s) * C + c) * (E + R);
  for (int i = tid; i < E; i += blockDim.x) part[i] = hist[i];
  if (tid < R) part[E + tid] = rcount[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) last_block = (atomicAdd(&ctl->layout_done[s], 1u) == unsigned(C - 1));
  __syncthreads();
  if (!last_block) return;
  __threadfence();
  const int32_t* base = reinterpret_cast<const int32_t*>(ws + ws_partials_offset()) +
                        int64_t(s) * C * (E + R);
  for (int i = tid; i < E + R; i += blockDim.x) {
    int sum = 0;
    for (int b = 0; b < C; ++b) sum += ld_cg_i32(base + int64_t(b) * (E + R) + i);
    if (i < E) num_tokens_per_expert[int64_t(s) * E + i] = sum;
    else num_tokens_per_rank[s * R + (i - E)] = sum;
  }
  if (tid == 0) ctl->layout_done[s] = 0;  // leave the workspace zeroed for the next call
}

// ---------------------------------------------------------------------------
// Receive-offset scan (decoupled lookback) + row metadata
// ---------------------------------------------------------------------------
// Tile state word: [63:62] flag (1 = aggregate only, 2 = inclusive prefix),
// [61:32] launch epoch (30 bits), [31:0] count.
constexpr uint64_t kFlagAggregate = 1ull << 62;
constexpr uint64_t kFlagInclusive = 2ull << 62;
__device__ __forceinline__ uint64_t make_state(uint64_t flag, uint32_t epoch, uint32_t v) {
  return flag | (uint64_t(epoch & 0x3fffffffu) << 32) | v;
}

struct ScanArgs {
  int R, N, K, E;
  const int32_t* topk_idx;
  const float* topk_weights;
  const uint32_t* is_token_in_rank;
  const int32_t* num_tokens_per_rank;
  const int32_t* num_tokens_per_expert;
  int64_t recv_capacity;
  int32_t* recv_src_rank;
  int32_t* recv_src_idx;
  int32_t* recv_topk_idx;
  float* recv_topk_weights;
  int32_t* dest_offsets;
  int32_t* rank_prefix;
  int32_t* num_recv_tokens_per_expert;
  int32_t* send_row;
  int32_t* dev_err;
  unsigned char* ws;
};

constexpr int kScanWarps = kScanTokens / kWarp;

__global__ void __launch_bounds__(kScanTokens) mp_k_scan(ScanArgs a) {
  extern __shared__ int32_t sm_scan[];
  int32_t* idx_s = sm_scan;                               // [kScanTokens * K]
  float* w_s = reinterpret_cast<float*>(sm_scan + kScanTokens * a.K);  // [kScanTokens * K]
  __shared__ uint32_t wball[kScanWarps][MP_MAX_RANKS];    // per-warp ballots
  __shared__ int32_t woff[kScanWarps][MP_MAX_RANKS];      // per-warp exclusive offsets
  __shared__ int64_t row_base[MP_MAX_RANKS];              // dest_base[d] + tile prefix
  __shared__ int32_t tot[MP_MAX_RANKS];
  __shared__ uint32_t sh_tile, sh_epoch;
  __shared__ int sh_last;

  const int R = a.R, N = a.N, K = a.K, E = a.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  uint64_t* state = reinterpret_cast<uint64_t*>(a.ws + ws_status_offset(R, N, E));
  const int64_t T = int64_t(R) * N;

  if (tid == 0) {
    sh_epoch = ld_relaxed_u32(&ctl->scan_epoch);
    sh_tile = atomicAdd(&ctl->scan_tile_counter, 1u);
  }
  // totals per destination (independent of the tile)
  if (tid < R) {
    int sum = 0;
    for (int s = 0; s < R; ++s) sum += a.num_tokens_per_rank[s * R + tid];
    tot[tid] = sum;
  }
  __syncthreads();
  const uint32_t tile = sh_tile, epoch = sh_epoch;
  if (tile >= gridDim.x) {  // only possible if the workspace was not zero-filled
    if (tid == 0) raise_error(a.dev_err, MP_ERR_INVALID_ARG);
    return;
  }
  const int64_t g0 = int64_t(tile) * kScanTokens;
  const int ntok = int(T - g0 < kScanTokens ? T - g0 : kScanTokens);

  // stage this tile's topk rows (contiguous along the flattened axis)
  for (int i = tid; i < ntok * K; i += blockDim.x) {
    idx_s[i] = a.topk_idx[g0 * K + i];
    w_s[i] = a.topk_weights[g0 * K + i];
  }
  const uint32_t mask = tid < ntok ? a.is_token_in_rank[g0 + tid] : 0u;
  for (int d = 0; d < R; ++d) {
    const unsigned b = __ballot_sync(kFull, (mask >> d) & 1u);
    if (lane == 0) wball[warp][d] = b;
  }
  __syncthreads();

  if (warp == 0) {
    // lane d: the tile's count for destination d and per-warp offsets
    int cnt = 0;
    if (lane < R) {
      for (int w = 0; w < kScanWarps; ++w) {
        woff[w][lane] = cnt;
        cnt += __popc(wball[w][lane]);
      }
    }
    // destination bases: exclusive scan of the totals over d
    int incl = lane < R ? tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    const int dest_base = incl - (lane < R ? tot[lane] : 0);
    const int total_rows = __shfl_sync(kFull, incl, R - 1);

    int64_t excl = 0;
    if (lane < R) {
      uint64_t* my = state + int64_t(tile) * R + lane;
      if (tile == 0) {
        st_release_u64(my, make_state(kFlagInclusive, epoch, uint32_t(cnt)));
      } else {
        st_release_u64(my, make_state(kFlagAggregate, epoch, uint32_t(cnt)));
        // walk back until a predecessor with an inclusive prefix
        int64_t j = int64_t(tile) - 1;
        bool timed_out = false;
        while (j >= 0) {
          const uint64_t* p = state + j * R + lane;
          uint64_t v = ld_acquire_u64(p);
          uint32_t spins = 0, nap = 32;
          while (((v >> 32) & 0x3fffffffu) != (epoch & 0x3fffffffu) || (v >> 62) == 0) {
            if (++spins > kSpinLimit) { timed_out = true; break; }
            __nanosleep(nap);
            if (nap < 1024) nap <<= 1;
            v = ld_acquire_u64(p);
          }
          if (timed_out) break;
          excl += uint32_t(v);
          if ((v >> 62) == 2) break;
          --j;
        }
        if (timed_out) raise_error(a.dev_err, MP_ERR_TIMEOUT);
        st_release_u64(my, make_state(kFlagInclusive, epoch, uint32_t(excl + cnt)));
      }
      row_base[lane] = int64_t(dest_base) + excl;
    }
    // the first tile also writes the small per-destination tables
    if (tile == 0) {
      if (lane < R) a.dest_offsets[lane] = dest_base;
      if (lane == 0) a.dest_offsets[R] = total_rows;
    }
  }
  __syncthreads();

  // rows of this thread's token
  if (tid < ntok) {
    const int64_t g = g0 + tid;
    const int s = int(g / N), t = int(g - int64_t(s) * N);
    const int El = E / R;
    int32_t* sr = a.send_row + g * R;
    bool overflow = false;
    for (int d = 0; d < R; ++d) {
      int32_t out = -1;
      if ((mask >> d) & 1u) {
        const int64_t row = row_base[d] + woff[warp][d] + __popc(wball[warp][d] & lanemask_lt());
        if (row < a.recv_capacity) {
          out = int32_t(row);
          a.recv_src_rank[row] = s;
          a.recv_src_idx[row] = t;
          const int lo = d * El, hi = lo + El;
          for (int k = 0; k < K; ++k) {
            const int e = idx_s[tid * K + k];
            const bool local = e >= lo && e < hi;
            a.recv_topk_idx[row * K + k] = local ? e - lo : -1;
            a.recv_topk_weights[row * K + k] = local ? w_s[tid * K + k] : 0.0f;
          }
        } else {
          overflow = true;
        }
      }
      sr[d] = out;
    }
    if (overflow) raise_error(a.dev_err, MP_ERR_CAPACITY);
  }

  if (tile == 0) {
    // rank_prefix[s][d] = rows of d from sources < s; per-expert receive counts
    for (int i = tid; i < R * R; i += blockDim.x) {
      const int s = i / R, d = i - s * R;
      int sum = 0;
      for (int q = 0; q < s; ++q) sum += a.num_tokens_per_rank[q * R + d];
      a.rank_prefix[i] = sum;
    }
    for (int e = tid; e < E; e += blockDim.x) {
      int sum = 0;
      for (int s = 0; s < R; ++s) sum += a.num_tokens_per_expert[int64_t(s) * E + e];
      a.num_recv_tokens_per_expert[e] = sum;
    }
  }

  // the last block out resets the counters and moves to the next epoch
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    sh_last = (atomicAdd(&ctl->scan_done, 1u) == gridDim.x - 1);
  }
  __syncthreads();
  if (sh_last && tid == 0) {
    ctl->scan_tile_counter = 0;
    ctl->scan_done = 0;
    ctl->copy_unit_counter = 0;
    __threadfence();
    atomicAdd(&ctl->scan_epoch, 1u);
  }
}

}  // namespace mp

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
namespace mp {

cudaError_t launch_layout(int R, int N, int K, int E, const int32_t* topk_idx,
                          int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                          uint32_t* is_token_in_rank, int32_t* dev_err, unsigned char* ws,
                          cudaStream_t stream) {
  if (N == 0) {  // no tokens: all counts are zero
    cudaError_t e = cudaMemsetAsync(num_tokens_per_rank, 0, sizeof(int32_t) * R * R, stream);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(num_tokens_per_expert, 0, sizeof(int32_t) * size_t(R) * E, stream);
    return e;
  }
  const size_t smem = sizeof(int32_t) * (size_t(E) + MP_MAX_RANKS + size_t(kLayoutTokens) * K);
  static thread_local int configured_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < int(smem) && smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(mp_k_layout, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    configured_smem[dev] = int(smem);
  }
  dim3 grid(unsigned(layout_blocks_per_rank(N)), unsigned(R));
  mp_k_layout<<<grid, kLayoutTokens, smem, stream>>>(R, N, K, E, topk_idx, num_tokens_per_rank,
                                                      num_tokens_per_expert, is_token_in_rank,
                                                      dev_err, ws);
  return cudaGetLastError();
}

cudaError_t launch_scan(int R, int N, int K, int E, const int32_t* topk_idx,
                        const float* topk_weights, const uint32_t* is_token_in_rank,
                        const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                        int64_t recv_capacity, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* dest_offsets,
                        int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                        int32_t* send_row, int32_t* dev_err, unsigned char* ws,
                        cudaStream_t stream) {
  if (N == 0) {  // no tokens, no rows
    cudaError_t e = cudaMemsetAsync(dest_offsets, 0, sizeof(int32_t) * (R + 1), stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(rank_prefix, 0, sizeof(int32_t) * R * R, stream);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(num_recv_tokens_per_expert, 0, sizeof(int32_t) * size_t(E), stream);
    return e;
  }
  ScanArgs a{R, N, K, E, topk_idx, topk_weights, is_token_in_rank, num_tokens_per_rank,
             num_tokens_per_expert, recv_capacity, recv_src_rank, recv_src_idx, recv_topk_idx,
             recv_topk_weights, dest_offsets, rank_prefix, num_recv_tokens_per_expert, send_row,
             dev_err, ws};
  const size_t smem = 2 * sizeof(int32_t) * size_t(kScanTokens) * K;
  static thread_local int configured_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < int(smem) && smem > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(mp_k_scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    configured_smem[dev] = int(smem);
  }
  mp_k_scan<<<unsigned(scan_tiles(R, N)), kScanTokens, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mp
