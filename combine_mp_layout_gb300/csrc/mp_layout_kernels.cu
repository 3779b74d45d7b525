// mp_layout_kernels.cu -- the routing layout and the receive-offset scan.
//
// Layout ("MSCCLPP EP implementation", microsoft/mscclpp PR #852, port
// scope: get_dispatch_layout computes counts and token-in-rank).  One block
// per (source rank, 256-token slice); warp ballots build the per-rank
// counts, a shared-memory histogram the per-expert counts.  Blocks add their
// counts into a per-rank accumulator (integer adds: order-free, exact) and
// the last block of each rank copies the totals out.
//
// Scan (the counterpart of the notify/prefix-matrix step of the same port,
// here a single-pass decoupled lookback).  The receive row of token (s,t)
// at destination d is
//     dest_base[d] + rank_prefix[s][d] + #{t' < t : bit d of token (s,t')},
// dest_base[d] = rows of all destinations < d, rank_prefix[s][d] = rows of d
// from source ranks < s (both sums of num_tokens_per_rank).  Each source
// rank's tokens are cut into 128-token tiles; each tile publishes its R-wide
// count vector, looks back over the earlier tiles of its rank for the
// exclusive prefix, publishes the inclusive prefix and writes the rows'
// metadata.  Tiles are handed out in launch order through an atomic
// counter, so every tile a block waits on belongs to a block that is
// already running.
//
// Layout + scan fused (mp_k_layout_scan): the same tiles, in one cooperative
// launch with one grid barrier between the lookback and the rows.
//
// Low-latency offsets (mp_k_ll_offsets): one row per (token, top-k slot),
// grouped by expert or by the rank owning it, by a per-rank counting sort.
#include <cstddef>
#include <cstdint>

#include "mp_common.cuh"
#include "mp_internal.h"

// Longest back-off (ns) between polls of a predecessor tile's flag (the
// back-off starts at 32 ns and doubles up to this).  Measured on the fused
// layout + offsets (dsv3, 256 tiles): 1024 ns 24.4 us, 128 ns 22.9-23.3 us,
// 32 ns (no doubling) 22.5 us per call.
#ifndef MP_LOOKBACK_MAX_NAP
#define MP_LOOKBACK_MAX_NAP 32
#endif
// The fused layout + offsets kernel issues its first id loads before it
// publishes the epoch it read (1) or after (0): 24.5 -> 24.4 us (dsv3),
// 28.0/26.7 -> 26.7 us (skew), 23.5 -> 22.4 us (dsv3 at N = 128).
#ifndef MP_FUSED_EARLY_LOADS
#define MP_FUSED_EARLY_LOADS 1
#endif

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
  int32_t* hist = sm_layout;               // [E]
  int32_t* rcount = sm_layout + E;         // [MP_MAX_RANKS]
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
  {
    const int n = ntok * K;
#pragma unroll 4
    for (int i = tid; i < n; i += kLayoutTokens) idx_s[i] = __ldg(src + i);
  }
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

  // Several blocks per source rank: add this block's counts into the rank's
  // accumulator (integer adds, so the order of the blocks does not matter);
  // the last block to finish copies the totals out and zeroes the
  // accumulator for the next call.
  Control* ctl = reinterpret_cast<Control*>(ws);
  int32_t* acc = reinterpret_cast<int32_t*>(ws + ws_acc_offset()) + int64_t(s) * (E + R);
  for (int i = tid; i < E; i += blockDim.x)
    if (hist[i]) atomicAdd(&acc[i], hist[i]);
  if (tid < R && rcount[tid]) atomicAdd(&acc[E + tid], rcount[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) last_block = (atomicAdd(&ctl->layout_done[s], 1u) == unsigned(C - 1));
  __syncthreads();
  if (!last_block) return;
  __threadfence();
  for (int i = tid; i < E + R; i += blockDim.x) {
    const int v = __ldcg(acc + i);
    acc[i] = 0;
    if (i < E) num_tokens_per_expert[int64_t(s) * E + i] = v;
    else num_tokens_per_rank[s * R + (i - E)] = v;
  }
  if (tid == 0) ctl->layout_done[s] = 0;
}

// ---------------------------------------------------------------------------
// Receive-offset scan (decoupled lookback) + row metadata
// ---------------------------------------------------------------------------
// Tile record: flag word (epoch << 2 | status, status 1 = aggregate counts
// published, 2 = inclusive prefix published), then R aggregate counts and R
// inclusive prefixes.  A single thread writes a record's counts and then
// releases its flag, so a reader that acquires the flag sees the counts.
// The scan is segmented by source rank: the rows of source rank s start, at
// destination d, at dest_base[d] + rank_prefix[s][d] (both sums of
// num_tokens_per_rank), so a tile only looks back over the earlier tiles of
// its own rank and the first tile of each rank is inclusive at once.
constexpr uint32_t kStatusAggregate = 1u;
constexpr uint32_t kStatusInclusive = 2u;
__device__ __forceinline__ uint32_t make_flag(uint32_t epoch, uint32_t status) {
  return (epoch << 2) | status;
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
  int global_ids;    // recv_topk_idx: 0 = local ids / -1, 1 = global ids / sentinel
  int32_t sentinel;  // value for non-local entries when global_ids
};

constexpr int kScanThreads = 256;  // two threads per token of a tile
constexpr int kScanWarps = kScanThreads / kWarp;

// Warp-wide sum; every lane gets the total.
__device__ __forceinline__ uint32_t warp_sum(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Warp 0 of a scan tile: the tile's count per destination and per-warp
// offsets from the ballots, then its record (aggregate, or inclusive for a
// rank's first tile) and the decoupled lookback over the rank's earlier
// tiles.  Returns, in lane d, the rows of destination d in this rank's
// earlier tiles; tcount[d] ends as the inclusive prefix through this tile.
__device__ __forceinline__ uint32_t tile_publish_lookback(
    int R, int64_t tile, int c, int src_rank, int C, uint32_t epoch,
    const uint32_t (*wball)[MP_MAX_RANKS], int32_t (*woff)[MP_MAX_RANKS], uint32_t* tcount,
    uint32_t* tcnt, uint32_t* flags, uint32_t* agg, uint32_t* incl, int32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  // lane d: the tile's count for destination d and the per-warp offsets
  uint32_t cnt = 0;
  if (lane < R) {
    for (int w = 0; w < kScanWarps; ++w) {
      woff[w][lane] = int32_t(cnt);
      cnt += __popc(wball[w][lane]);
    }
    tcount[lane] = cnt;
    tcnt[lane] = cnt;
  }
  __syncwarp();
  const int64_t rec = int64_t(tile) * R;
  uint32_t excl = 0;  // lane d: rows of destination d in this rank's earlier tiles
  if (c == 0) {
    if (lane == 0) {
      for (int d = 0; d < R; ++d) incl[rec + d] = tcount[d];
      st_release_u32(&flags[tile], make_flag(epoch, kStatusInclusive));
    }
  } else {
    if (lane == 0) {
      for (int d = 0; d < R; ++d) agg[rec + d] = tcount[d];
      st_release_u32(&flags[tile], make_flag(epoch, kStatusAggregate));
    }
    // Look back over up to 32 earlier tiles of this rank at a time (lane j
    // looks at tile base - j), stopping at the nearest one whose inclusive
    // prefix is out.  Every wait is bounded (MP_ERR_TIMEOUT).
    const int64_t first = int64_t(src_rank) * C;
    bool timed_out = false;
    for (int64_t base = int64_t(tile) - 1; base >= first; base -= 32) {
      const int64_t p = base - lane;
      uint32_t status = 0;
      if (p >= first) {
        uint32_t f = ld_acquire_u32(&flags[p]);
        uint32_t spins = 0, nap = 32;
        while ((f >> 2) != epoch || (f & 3u) == 0) {
          if (++spins > kSpinLimit) { timed_out = true; break; }
          __nanosleep(nap);
          if (nap < MP_LOOKBACK_MAX_NAP) nap <<= 1;
          f = ld_acquire_u32(&flags[p]);
        }
        status = timed_out ? kStatusInclusive : (f & 3u);
      }
      const unsigned inclusive = __ballot_sync(kFull, p >= first && status == kStatusInclusive);
      const int stop = inclusive ? __ffs(inclusive) - 1 : 31;
      const bool use = p >= first && lane <= stop && !timed_out;
      const uint32_t* src = status == kStatusInclusive ? incl : agg;
      uint32_t v[MP_MAX_RANKS];
#pragma unroll
      for (int d = 0; d < MP_MAX_RANKS; ++d)
        v[d] = (use && d < R) ? __ldcg(src + p * R + d) : 0u;
#pragma unroll
      for (int d = 0; d < MP_MAX_RANKS; ++d) {
        if (d < R) {
          const uint32_t sum = warp_sum(v[d]);
          if (lane == d) excl += sum;
        }
      }
      if (__any_sync(kFull, timed_out) || inclusive) break;
    }
    if (__any_sync(kFull, timed_out) && lane == 0) raise_error(dev_err, MP_ERR_TIMEOUT);
    if (lane < R) tcount[lane] += excl;  // inclusive prefix through this tile
    __syncwarp();
    if (lane == 0) {
      for (int d = 0; d < R; ++d) incl[rec + d] = tcount[d];
      st_release_u32(&flags[tile], make_flag(epoch, kStatusInclusive));
    }
  }
  return excl;
}

// The rows of one scan tile.  A tile's rows for one destination are
// consecutive, so the tile's rows are numbered destination-major (j =
// dstart[d] + rank within d) and two shared-memory tables give each j its
// token and destination; the metadata stores then run over all of the tile's
// rows (and rows x top-k slots) at once, contiguous within each destination.
// Each token's row at each destination is staged in shared memory (send_row).
// Called by all threads of the block; needs the tile's masks (one per token
// thread), the per-warp ballots and offsets, the tile's first row and row
// count per destination, and its top-k ids and weights staged in shared memory.
// With META false only send_row is written (the receive metadata is then left
// to the row copy that follows, mp_k_dispatch_after_offsets).
struct TileRowsSmem {
  int32_t* sr_s;     // [kScanTokens][R]: send_row entries of the tile's tokens
  uint8_t* row_tok;  // [kScanTokens * MP_MAX_RANKS]: token of tile row j
  uint8_t* row_d;    // [kScanTokens * MP_MAX_RANKS]: destination of tile row j
  int32_t* dstart;   // [MP_MAX_RANKS + 1]: first tile row of destination d
  int32_t* nok;      // [MP_MAX_RANKS]: rows of d within the receive capacity
};

__device__ __forceinline__ void write_tile_rows(
    const ScanArgs& a, uint32_t mask, int ntok, int t0, int64_t g0, int src_rank,
    const uint32_t (*wball)[MP_MAX_RANKS], const int32_t (*woff)[MP_MAX_RANKS],
    const int64_t* row_base, const uint32_t* tcnt, const int32_t* idx_s, const float* w_s,
    const TileRowsSmem& sm, bool meta = true) {
  const int R = a.R, K = a.K, E = a.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (warp == 0) {  // destination-major numbering of the tile's rows; the capacity clamp
    const int c = lane < R ? int(tcnt[lane]) : 0;
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += v;
    }
    int ok = c;
    if (lane < R) {
      sm.dstart[lane] = inc - c;
      const int64_t room = a.recv_capacity - row_base[lane];
      ok = room <= 0 ? 0 : (room < c ? int(room) : c);
      sm.nok[lane] = ok;
    }
    if (lane == 31) sm.dstart[R] = inc;
    if (__any_sync(kFull, ok < c) && lane == 0) raise_error(a.dev_err, MP_ERR_CAPACITY);
  }
  if (tid < ntok)
    for (int d = 0; d < R; ++d) sm.sr_s[tid * R + d] = -1;
  __syncthreads();
  if (tid < ntok) {
    for (uint32_t m = mask; m; m &= m - 1u) {
      const int d = __ffs(m) - 1;
      const int rank = woff[warp][d] + __popc(wball[warp][d] & lanemask_lt());
      if (meta) {
        const int j = sm.dstart[d] + rank;
        sm.row_tok[j] = uint8_t(tid);
        sm.row_d[j] = uint8_t(d);
      }
      if (rank < sm.nok[d]) sm.sr_s[tid * R + d] = int32_t(row_base[d] + rank);
    }
  }
  __syncthreads();
#pragma unroll 4
  for (int i = tid; i < ntok * R; i += kScanThreads) a.send_row[g0 * R + i] = sm.sr_s[i];
  if (!meta) return;
  const int total = sm.dstart[R];
#pragma unroll 4
  for (int j = tid; j < total; j += kScanThreads) {
    const int d = sm.row_d[j], r = j - sm.dstart[d];
    if (r < sm.nok[d]) {
      const int64_t row = row_base[d] + r;
      a.recv_src_rank[row] = src_rank;
      a.recv_src_idx[row] = t0 + sm.row_tok[j];
    }
  }
  // element i = j*K + k of the tile's (row, slot) pairs; (j, k) advance by
  // (kScanThreads / K, kScanThreads % K) per step, avoiding a division
  const int El = E / R;
  const int step_j = kScanThreads / K, step_k = kScanThreads - step_j * K;
  int j = tid / K, k = tid - (tid / K) * K;
#pragma unroll 4
  for (int i = tid; i < total * K; i += kScanThreads) {
    const int d = sm.row_d[j], r = j - sm.dstart[d];
    if (r < sm.nok[d]) {
      const int tk = sm.row_tok[j];
      const int e = idx_s[tk * K + k];
      const int lo = d * El;
      const bool local = e >= lo && e < lo + El;
      const int64_t o = (row_base[d] + r) * K + k;
      a.recv_topk_idx[o] = a.global_ids ? (local ? e : a.sentinel) : (local ? e - lo : -1);
      a.recv_topk_weights[o] = local ? w_s[tk * K + k] : 0.0f;
    }
    j += step_j;
    k += step_k;
    if (k >= K) {
      k -= K;
      ++j;
    }
  }
}

__global__ void __launch_bounds__(kScanThreads) mp_k_scan(ScanArgs a) {
  extern __shared__ int32_t sm_scan[];
  int32_t* idx_s = sm_scan;                                             // [kScanTokens * K]
  float* w_s = reinterpret_cast<float*>(sm_scan + kScanTokens * a.K);  // [kScanTokens * K]
  int32_t* sr_s = sm_scan + 2 * kScanTokens * a.K;                      // [kScanTokens * R]
  __shared__ int32_t ntpr_s[MP_MAX_RANKS * MP_MAX_RANKS];  // num_tokens_per_rank
  __shared__ uint32_t wball[kScanWarps][MP_MAX_RANKS];     // per-warp ballots
  __shared__ int32_t woff[kScanWarps][MP_MAX_RANKS];       // per-warp exclusive offsets
  __shared__ uint32_t tcount[MP_MAX_RANKS];                // tile counts, then inclusive prefix
  __shared__ uint32_t tcnt[MP_MAX_RANKS];                  // tile counts
  __shared__ int64_t row_base[MP_MAX_RANKS];               // first receive row of the tile at d
  __shared__ uint8_t row_tok[kScanTokens * MP_MAX_RANKS], row_d[kScanTokens * MP_MAX_RANKS];
  __shared__ int32_t dstart[MP_MAX_RANKS + 1], nok[MP_MAX_RANKS];
  __shared__ uint32_t sh_tile, sh_epoch;
  __shared__ int sh_last;

  const int R = a.R, N = a.N, K = a.K, E = a.E;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.ws + ws_flags_offset(R, E));
  uint32_t* agg = reinterpret_cast<uint32_t*>(a.ws + ws_agg_offset(R, N, E));
  uint32_t* incl = reinterpret_cast<uint32_t*>(a.ws + ws_incl_offset(R, N, E));
  const int C = int(scan_tiles_per_rank(N));

  if (tid == 0) {
    sh_epoch = ld_relaxed_u32(&ctl->scan_epoch) & 0x3fffffffu;
    sh_tile = atomicAdd(&ctl->scan_tile_counter, 1u);
  }
  for (int i = tid; i < R * R; i += blockDim.x) ntpr_s[i] = __ldg(a.num_tokens_per_rank + i);
  __syncthreads();
  const uint32_t tile = sh_tile, epoch = sh_epoch;
  if (tile >= gridDim.x) {  // only possible if the workspace was not zero-filled
    if (tid == 0) raise_error(a.dev_err, MP_ERR_INVALID_ARG);
    return;
  }
  const int src_rank = int(tile / uint32_t(C));
  const int c = int(tile - uint32_t(src_rank) * uint32_t(C));  // tile index within the rank
  const int t0 = c * kScanTokens;
  const int ntok = min(kScanTokens, N - t0);
  const int64_t g0 = int64_t(src_rank) * N + t0;  // first token, flattened (s, t)

  // the mask first (the aggregate depends on it), the topk rows alongside
  const uint32_t mask = tid < ntok ? __ldg(a.is_token_in_rank + g0 + tid) : 0u;
  {
    const int n = ntok * K;
    const int32_t* gi = a.topk_idx + g0 * K;
    const float* gw = a.topk_weights + g0 * K;
#pragma unroll 4
    for (int i = tid; i < n; i += kScanThreads) {
      idx_s[i] = __ldg(gi + i);
      w_s[i] = __ldg(gw + i);
    }
  }
  for (int d = 0; d < R; ++d) {
    const unsigned b = __ballot_sync(kFull, (mask >> d) & 1u);
    if (lane == 0) wball[warp][d] = b;
  }
  __syncthreads();

  if (warp == 0) {
    const uint32_t excl = tile_publish_lookback(R, tile, c, src_rank, C, epoch, wball, woff,
                                                tcount, tcnt, flags, agg, incl, a.dev_err);
    // first row of this tile at d: rows of destinations < d (an exclusive
    // warp scan of the per-destination totals), rows of d from source ranks
    // < src_rank, rows of d from this rank's earlier tiles
    int64_t tot = 0, pre = 0;
    if (lane < R) {
      for (int s = 0; s < R; ++s) {
        const int v = ntpr_s[s * R + lane];
        tot += v;
        if (s < src_rank) pre += v;
      }
    }
    int64_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane < R) row_base[lane] = (inc - tot) + pre + excl;
  } else if (tile == 0) {
    // warps 1..: the small per-destination tables, while warp 0 publishes
    const int t = tid - kWarp, nt = kScanThreads - kWarp;
    for (int i = t; i < R * R; i += nt) {  // rank_prefix[s][d]
      const int s = i / R, d = i - s * R;
      int sum = 0;
      for (int q = 0; q < s; ++q) sum += ntpr_s[q * R + d];
      a.rank_prefix[i] = sum;
    }
    for (int d = t; d <= R; d += nt) {  // dest_offsets
      int sum = 0;
      for (int q = 0; q < R * R; ++q)
        if ((q - (q / R) * R) < d) sum += ntpr_s[q];
      a.dest_offsets[d] = sum;
    }
    for (int e = t; e < E; e += nt) {  // num_recv_tokens_per_expert[d][j], e = d*E/R + j
      int sum = 0;
#pragma unroll 8
      for (int s = 0; s < R; ++s) sum += __ldg(a.num_tokens_per_expert + int64_t(s) * E + e);
      a.num_recv_tokens_per_expert[e] = sum;
    }
  }
  __syncthreads();

  write_tile_rows(a, mask, ntok, t0, g0, src_rank, wball, woff, row_base, tcnt, idx_s, w_s,
                  TileRowsSmem{sr_s, row_tok, row_d, dstart, nok});

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
    __threadfence();
    atomicAdd(&ctl->scan_epoch, 1u);
  }
}

// ---------------------------------------------------------------------------
// Layout and receive offsets in one cooperative launch (the work of mp_k_layout
// followed by mp_k_scan, for callers of mp_layout_and_offsets and
// mp_layout_dispatch).  Every block is resident at once, so blocks own tiles
// statically (tile = blockIdx.x + i * gridDim.x, in increasing order, which
// keeps each lookback's predecessors running or done) and may meet at one
// grid barrier:
//  1. per tile: the top-k ids give each token's rank mask (is_token_in_rank)
//     and the tile's expert counts (added into the rank's accumulator); the
//     tile publishes its per-destination counts and looks back over its
//     rank's earlier tiles (the segmented decoupled lookback of mp_k_scan);
//  2. grid barrier (bounded);
//  3. each rank's last tile holds num_tokens_per_rank; from it every block
//     forms rank_prefix and the destination bases, the accumulators give
//     num_tokens_per_expert and num_recv_tokens_per_expert (and are zeroed),
//     and each tile writes its send_row entries and (with meta) the receive
//     metadata.
// The kernel lets its programmatic dependent (the row copy of
// mp_layout_dispatch) launch as soon as it starts.
// ---------------------------------------------------------------------------
constexpr int kFusedMaxTiles = 16;  // tiles one block may own (tiles <= 16 * grid)
// Up to this many tiles per source rank, the tiles publish plain aggregate
// counts before the barrier (and add them into their rank's totals), and after
// it each tile sums the aggregates of its rank's earlier tiles; beyond it (the
// C^2 / 2 reads per rank grow) the tiles run the decoupled lookback before the
// barrier.  Measured (globaltimer, dsv3 shape): with the lookback and its
// release fences the phase before the barrier took 3.5 us at N = 128 (one tile
// per rank) and 8-10 us at N = 4096; with aggregates 3.3 and 4.3 us.
#ifndef MP_FUSED_AGG_MAX_TILES
#define MP_FUSED_AGG_MAX_TILES 32
#endif
constexpr int kFusedAggMaxTiles = MP_FUSED_AGG_MAX_TILES;
// (the failure-detection test presets the barrier's base word at this offset)
static_assert(offsetof(Control, bar_count) == 144 && offsetof(Control, bar_base) == 148,
              "grid barrier words of the control block");

struct FusedArgs {
  ScanArgs a;                      // receive-side outputs (its layout inputs unused)
  uint32_t* is_token_in_rank;      // [R][N] out
  int32_t* num_tokens_per_rank;    // [R][R] out
  int32_t* num_tokens_per_expert;  // [R][E] out
};

// Grid barrier for a cooperative launch.  bar_count counts arrivals and is
// never reset; bar_base is its value when this launch began (every block reads
// it before arriving, and block 0 moves it on by the grid size once past the
// barrier, for the next launch).  Thread 0 of each block adds its arrival with
// acquire-release semantics -- which also publishes the block's earlier writes,
// ordered before it by the CTA barrier -- and polls (bounded) until every
// block's arrival is in: one atomic and one poll, with no reset on the way.
// Returns false when the wait gave up.
__device__ __forceinline__ bool grid_barrier(Control* ctl, uint32_t nblocks, uint32_t base,
                                             int* ok_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    uint32_t seen = atom_add_acq_rel_u32(&ctl->bar_count, 1u) + 1u;
    uint32_t spins = 0;
    while (int32_t(seen - base) < int32_t(nblocks)) {
      if (++spins > kSpinLimit) { ok = 0; break; }
      __nanosleep(32);
      seen = ld_acquire_u32(&ctl->bar_count);
    }
    *ok_s = ok;
  }
  __syncthreads();
  return *ok_s != 0;
}

// META: also write the receive metadata (else send_row only: the row copy of
// mp_layout_dispatch writes the metadata).  LOOKBACK: the decoupled lookback
// before the barrier (more than kFusedAggMaxTiles tiles per rank), else plain
// aggregates and rank totals.  Both are compile-time so that each launched
// instance holds only its own code: the kernel runs once per block, and its
// instructions are fetched cold.
template <bool META, bool LOOKBACK>
__global__ void __launch_bounds__(kScanThreads) mp_k_layout_scan(FusedArgs f) {
  const ScanArgs& a = f.a;
  extern __shared__ int32_t sm_scan[];
  int32_t* idx_s = sm_scan;                                             // [kScanTokens * K]
  float* w_s = reinterpret_cast<float*>(sm_scan + kScanTokens * a.K);  // [kScanTokens * K]
  int32_t* sr_s = sm_scan + 2 * kScanTokens * a.K;                      // [kScanTokens * R]
  int32_t* hist = sr_s + kScanTokens * a.R;                             // [E]
  __shared__ int32_t ntpr_s[MP_MAX_RANKS * MP_MAX_RANKS];  // num_tokens_per_rank
  __shared__ uint32_t wball[kScanWarps][MP_MAX_RANKS];
  __shared__ int32_t woff[kScanWarps][MP_MAX_RANKS];
  __shared__ uint32_t tcount[MP_MAX_RANKS];
  __shared__ uint32_t tcnt[MP_MAX_RANKS];
  __shared__ int64_t row_base[MP_MAX_RANKS];
  __shared__ int64_t dest_base[MP_MAX_RANKS];
  __shared__ uint8_t row_tok[kScanTokens * MP_MAX_RANKS], row_d[kScanTokens * MP_MAX_RANKS];
  __shared__ int32_t dstart[MP_MAX_RANKS + 1], nok[MP_MAX_RANKS];
  __shared__ uint32_t tile_excl[kFusedMaxTiles][MP_MAX_RANKS];
  __shared__ uint32_t sh_epoch, sh_gen, sh_fgen;
  __shared__ int sh_bad, sh_ok;

  const int R = a.R, N = a.N, K = a.K, E = a.E, El = E / R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Control* ctl = reinterpret_cast<Control*>(a.ws);
  uint32_t* flags = reinterpret_cast<uint32_t*>(a.ws + ws_flags_offset(R, E));
  uint32_t* agg = reinterpret_cast<uint32_t*>(a.ws + ws_agg_offset(R, N, E));
  uint32_t* incl = reinterpret_cast<uint32_t*>(a.ws + ws_incl_offset(R, N, E));
  int32_t* acc = reinterpret_cast<int32_t*>(a.ws + ws_acc_offset());  // [R][E + R]
  int32_t* tot = reinterpret_cast<int32_t*>(a.ws + ws_tot_offset(R, N, E));  // [2][32][32]
  const int C = int(scan_tiles_per_rank(N));
  const int T = R * C;
  pdl_launch_dependents();
  // The epoch and barrier base are read first; thread 0 keeps them in
  // registers until the first tile's id loads are issued, so those loads do
  // not wait for them (the first tile's barrier publishes them).
  uint32_t epoch0 = 0, gen0 = 0, fgen0 = 0;
  if (tid == 0) {
    epoch0 = ld_relaxed_u32(&ctl->scan_epoch) & 0x3fffffffu;
    gen0 = ld_relaxed_u32(&ctl->bar_base);
    fgen0 = ld_relaxed_u32(&ctl->fused_gen);
  }
#if !MP_FUSED_EARLY_LOADS
  if (tid == 0) {
    sh_epoch = epoch0;
    sh_gen = gen0;
    sh_fgen = fgen0;
    sh_bad = 0;
  }
  __syncthreads();
#endif
  // A block that owns a single tile keeps that tile's ids, weights, ballots,
  // offsets and masks across the barrier instead of reloading them.
  const bool single = T <= int(gridDim.x);
  if (!LOOKBACK)  // summed from the earlier tiles' aggregates after the barrier
    for (int i = tid; i < kFusedMaxTiles * MP_MAX_RANKS; i += kScanThreads)
      (&tile_excl[0][0])[i] = 0u;

  // 1. layout work, and per tile its per-destination counts: published as
  //    plain aggregates (the barrier publishes them), or with the decoupled
  //    lookback over the rank's earlier tiles
  int it = 0;
  uint32_t mask_kept = 0;
  for (int tile = blockIdx.x; tile < T; tile += gridDim.x, ++it) {
    const int s = tile / C, c = tile - s * C;
    const int t0 = c * kScanTokens, ntok = min(kScanTokens, N - t0);
    const int64_t g0 = int64_t(s) * N + t0;
    for (int i = tid; i < E; i += kScanThreads) hist[i] = 0;
    {
      const int n = ntok * K;
      const int32_t* gi = a.topk_idx + g0 * K;
      const float* gw = a.topk_weights + g0 * K;
#pragma unroll 4
      for (int i = tid; i < n; i += kScanThreads) {
        idx_s[i] = __ldg(gi + i);
        if (META && single) w_s[i] = __ldg(gw + i);
      }
    }
#if MP_FUSED_EARLY_LOADS
    if (it == 0 && tid == 0) {
      sh_epoch = epoch0;
      sh_gen = gen0;
      sh_fgen = fgen0;
      sh_bad = 0;
    }
#endif
    __syncthreads();
    uint32_t mask = 0;
    if (tid < ntok) {
      bool bad = false;
      for (int k = 0; k < K; ++k) {
        const int e = idx_s[tid * K + k];
        if (e == -1) continue;
        if (e < -1 || e >= E) { bad = true; continue; }
        atomicAdd(&hist[e], 1);
        mask |= 1u << (e / El);
      }
      f.is_token_in_rank[g0 + tid] = mask;
      if (bad) sh_bad = 1;
    }
    mask_kept = mask;
    for (int d = 0; d < R; ++d) {
      const unsigned b = __ballot_sync(kFull, (mask >> d) & 1u);
      if (lane == 0) wball[warp][d] = b;
    }
    __syncthreads();
    int32_t* acc_s = acc + int64_t(s) * (E + R);
    for (int i = tid; i < E; i += kScanThreads)
      if (hist[i]) atomicAdd(&acc_s[i], hist[i]);
    if (warp == 0) {
      if constexpr (LOOKBACK) {
        const uint32_t excl = tile_publish_lookback(R, tile, c, s, C, sh_epoch, wball, woff,
                                                    tcount, tcnt, flags, agg, incl, a.dev_err);
        if (lane < R) tile_excl[it][lane] = excl;
      } else if (lane < R) {  // the tile's count per destination and per-warp offsets
        uint32_t cnt = 0;
        for (int w = 0; w < kScanWarps; ++w) {
          woff[w][lane] = int32_t(cnt);
          cnt += __popc(wball[w][lane]);
        }
        tcnt[lane] = cnt;
        agg[int64_t(tile) * R + lane] = cnt;
        // the rank's totals (one tile per rank: the aggregate itself)
        if (C > 1 && cnt)
          atomicAdd(&tot[(sh_fgen & 1u) * kTotBufInts + s * MP_MAX_RANKS + lane], int32_t(cnt));
      }
    }
    __syncthreads();  // hist, idx_s and the ballots are reused by the next tile
  }
  const int nown = it;  // tiles this block owns
  if (tid == 0 && sh_bad) raise_error(a.dev_err, MP_ERR_BAD_EXPERT);

  // 2. every tile is published and every expert count added
  if (!grid_barrier(ctl, gridDim.x, sh_gen, &sh_ok)) {
    if (tid == 0) raise_error(a.dev_err, MP_ERR_TIMEOUT);
    return;
  }

  // 3. totals, tables, rows.  The lower half of the block gathers the
  //    per-destination counts, the upper half (in the last blocks of the grid,
  //    so that block 0's tables do not add up) the expert counts: both start
  //    their loads at once.
  constexpr int kHalf = kScanThreads / 2;
  if (tid < kHalf) {
    if constexpr (LOOKBACK) {
      for (int i = tid; i < R * R; i += kHalf) {  // rank s's last tile: its totals
        const int s = i / R, d = i - s * R;
        ntpr_s[i] = int32_t(__ldcg(incl + (int64_t(s) * C + C - 1) * R + d));
      }
    } else {
      // the rank totals (from this launch's totals buffer, or with one tile
      // per rank its aggregate), and for each of this block's tiles the
      // per-destination counts of its rank's earlier tiles, summed in shared
      // memory (integer adds: their order does not matter).  Items [0, R*R)
      // are the totals, then each own tile's c*R earlier counts; 16 loads are
      // in flight before they are added.
      int n_items = R * R;
      for (int q = 0; q < nown; ++q) n_items += ((int(blockIdx.x) + q * int(gridDim.x)) % C) * R;
      constexpr int kB = 16;
      for (int i0 = tid; i0 < n_items; i0 += kHalf * kB) {
        uint32_t v[kB];
        int dst[kB];  // < R*R: ntpr_s index; R*R + k: tile_excl entry k; -1: none
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          const int i = i0 + j * kHalf;
          v[j] = 0u;
          dst[j] = -1;
          if (i >= n_items) continue;
          if (i < R * R) {
            const int s = i / R, d = i - s * R;
            v[j] = C == 1 ? __ldcg(agg + i)
                          : uint32_t(__ldcg(tot + (sh_fgen & 1u) * kTotBufInts +
                                            s * MP_MAX_RANKS + d));
            dst[j] = i;
          } else {
            int r = i - R * R;
            for (int q = 0; q < nown; ++q) {  // the own tile this item belongs to
              const int own = int(blockIdx.x) + q * int(gridDim.x);
              const int span = (own % C) * R;
              if (r < span) {
                const int c = r / R, d = r - c * R;
                v[j] = __ldcg(agg + (int64_t(own - own % C) + c) * R + d);
                dst[j] = R * R + q * MP_MAX_RANKS + d;
                break;
              }
              r -= span;
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kB; ++j) {
          if (dst[j] < 0) continue;
          if (dst[j] < R * R) ntpr_s[dst[j]] = int32_t(v[j]);
          else if (v[j]) atomicAdd(&tile_excl[0][0] + (dst[j] - R * R), v[j]);
        }
      }
    }
  } else {
    for (int64_t e = int64_t(gridDim.x - 1 - blockIdx.x) * kHalf + (tid - kHalf); e < E;
         e += int64_t(gridDim.x) * kHalf) {
      int sum = 0;
      for (int s0 = 0; s0 < R; s0 += 8) {  // 8 loads in flight before their stores
        int v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = s0 + j < R ? __ldcg(acc + int64_t(s0 + j) * (E + R) + e) : 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (s0 + j < R) {
            acc[int64_t(s0 + j) * (E + R) + e] = 0;
            f.num_tokens_per_expert[int64_t(s0 + j) * E + e] = v[j];
            sum += v[j];
          }
        }
      }
      a.num_recv_tokens_per_expert[e] = sum;
    }
  }
  __syncthreads();
  if (warp == 0) {  // first receive row of each destination
    int64_t tot = 0;
    if (lane < R)
      for (int s = 0; s < R; ++s) tot += ntpr_s[s * R + lane];
    int64_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += v;
    }
    if (lane < R) dest_base[lane] = inc - tot;
    if (blockIdx.x == 0 && lane < R) {
      a.dest_offsets[lane] = int32_t(inc - tot);
      if (lane == R - 1) a.dest_offsets[R] = int32_t(inc);
    }
  }
  if (blockIdx.x == 0) {
    for (int i = tid; i < R * R; i += kScanThreads) {
      const int s = i / R, d = i - s * R;
      int pre = 0;
      for (int q = 0; q < s; ++q) pre += ntpr_s[q * R + d];
      f.num_tokens_per_rank[i] = ntpr_s[i];
      a.rank_prefix[i] = pre;
    }
    // the other totals buffer, zero for the next launch (nothing uses it in this one)
    int32_t* next = tot + ((sh_fgen + 1u) & 1u) * kTotBufInts;
    for (int i = tid; i < int(kTotBufInts); i += kScanThreads) next[i] = 0;
    if (tid == 0) {
      atomicAdd(&ctl->scan_epoch, 1u);  // every lookback of this launch is done
      ctl->bar_base = sh_gen + gridDim.x;  // every arrival of this launch is in
      ctl->fused_gen = sh_fgen + 1u;
    }
  }
  __syncthreads();
  it = 0;
  for (int tile = blockIdx.x; tile < T; tile += gridDim.x, ++it) {
    const int s = tile / C, c = tile - s * C;
    const int t0 = c * kScanTokens, ntok = min(kScanTokens, N - t0);
    const int64_t g0 = int64_t(s) * N + t0;
    const uint32_t mask =
        single ? mask_kept : (tid < ntok ? __ldcg(f.is_token_in_rank + g0 + tid) : 0u);
    if (!single) {  // ids, weights, ballots and offsets of this tile
      if constexpr (META) {
        const int n = ntok * K;
        const int32_t* gi = a.topk_idx + g0 * K;
        const float* gw = a.topk_weights + g0 * K;
#pragma unroll 4
        for (int i = tid; i < n; i += kScanThreads) {
          idx_s[i] = __ldg(gi + i);
          w_s[i] = __ldg(gw + i);
        }
      }
      for (int d = 0; d < R; ++d) {
        const unsigned b = __ballot_sync(kFull, (mask >> d) & 1u);
        if (lane == 0) wball[warp][d] = b;
      }
      __syncthreads();
      if (warp == 0 && lane < R) {
        uint32_t cnt = 0;
        for (int w = 0; w < kScanWarps; ++w) {
          woff[w][lane] = int32_t(cnt);
          cnt += __popc(wball[w][lane]);
        }
        tcnt[lane] = cnt;
      }
    }
    if (warp == 0 && lane < R) {
      int64_t pre = 0;
      for (int q = 0; q < s; ++q) pre += ntpr_s[q * R + lane];
      row_base[lane] = dest_base[lane] + pre + tile_excl[it][lane];
    }
    __syncthreads();
    if constexpr (META) {
      write_tile_rows(a, mask, ntok, t0, g0, s, wball, woff, row_base, tcnt, idx_s, w_s,
                      TileRowsSmem{sr_s, row_tok, row_d, dstart, nok});
    } else {
      // send_row only: each token's thread writes its R entries (the receive
      // metadata is written by the row copy)
      bool over = false;
      if (tid < ntok) {
        int32_t* dst = a.send_row + (g0 + tid) * R;
        for (int d = 0; d < R; ++d) {
          int32_t v = -1;
          if ((mask >> d) & 1u) {
            const int64_t row =
                row_base[d] + woff[warp][d] + __popc(wball[warp][d] & lanemask_lt());
            if (row < a.recv_capacity) v = int32_t(row);
            else over = true;
          }
          dst[d] = v;
        }
      }
      if (__any_sync(kFull, over) && lane == 0) raise_error(a.dev_err, MP_ERR_CAPACITY);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Low-latency expert-major offsets ("MSCCLPP EP implementation", the
// low-latency dispatch/combine: per-expert receive buffers).  One row per
// (token, top-k slot with a valid expert); expert e's rows are contiguous,
// blocks in ascending e, rows inside a block ordered by source rank, then
// token, then top-k slot.
//
// One block per source rank s, a stable counting sort of its N*K entries:
//  1. the rank's entries are cut into nseg contiguous segments (one per warp
//     in step 3); one pass of the whole block over the ids counts the
//     entries of each (segment, expert) in shared memory;
//  2. every expert's first row (a block-wide scan of the per-expert totals
//     over all source ranks, from the layout's num_tokens_per_expert, plus
//     the rows of e from ranks < s) and, per expert, the exclusive prefix of
//     the segment counts;
//  3. each warp walks its segment 32 entries at a time in order; lanes with
//     the same expert find each other with __match_any_sync and take
//     consecutive rows, so the order is deterministic.
// num_tokens_per_expert may be NULL: the pass of step 1 then reads every
// rank's ids (R*N*K reads from L2 per block) and counts the totals and
// lower-rank prefixes too, which saves the layout launch on the small batches
// this path is for.
// Shared memory: (nseg + 3) * E int32, nseg = min(32, 16384 / E) (>= 1).
// ---------------------------------------------------------------------------
constexpr int kLLThreads = 1024;
constexpr int kLLHistInts = 16384;
#ifndef MP_LL_BATCH
#define MP_LL_BATCH 8
#endif
constexpr int kLLBatch = MP_LL_BATCH;  // id loads in flight per lane in the in-order walk
#ifndef MP_LL_IDS
#define MP_LL_IDS 16
#endif
constexpr int kLLIds = MP_LL_IDS;  // ids per thread and batch while counting (a multiple of 4)
static_assert(kLLIds % 4 == 0, "counting batches are whole 16-byte loads");

// segments of a rank's entries (one warp each) for NT threads and a budget of
// hist_ints shared-memory counters
__host__ __device__ inline int ll_segments(int nbins, int nt = kLLThreads,
                                           int hist_ints = kLLHistInts) {
  const int n = hist_ints / (nbins > 0 ? nbins : 1);
  return n < 1 ? 1 : (n > nt / kWarp ? nt / kWarp : n);
}

// RANK_MAJOR (the same page's rank-major output for the LL path): the rows
// are grouped by the rank d = e / (E/R) that owns the expert instead of by
// expert; inside a group by source rank, token and top-k slot.  The kernel is
// the same counting sort over nbins = R bins instead of E.
//
// The counting sort of source rank s by one block of NT threads (the body of
// mp_k_ll_offsets); ll_smem holds (nseg + 3) * nbins int32,
// nseg = ll_segments(nbins, NT, HIST).
template <bool RANK_MAJOR, int NT, int HIST>
__device__ __forceinline__ void ll_offsets_block(
    int s, int R, int N, int K, int E, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ num_tokens_per_expert, int64_t recv_capacity,
    int32_t* __restrict__ bin_offsets, int32_t* __restrict__ bin_src_offsets,
    int32_t* __restrict__ recv_src_token, int32_t* __restrict__ slot_row,
    int32_t* __restrict__ dev_err, int32_t* ll_smem, int64_t* warp_sums) {
  const int nbins = RANK_MAJOR ? R : E;
  const int El = E / R;
  auto bin_of = [&](int e) { return RANK_MAJOR ? e / El : e; };
  const int nseg = ll_segments(nbins, NT, HIST);
  int32_t* hist = ll_smem;                    // [nseg][nbins]: counts, then running offsets
  int32_t* rowbase = ll_smem + nseg * nbins;  // [nbins]: first row of (bin, this rank)
  int32_t* tot = rowbase + nbins;             // [nbins]: rows of the bin over every rank
  int32_t* pre = tot + nbins;                 // [nbins]: rows of the bin from ranks < s
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nk = int64_t(N) * K;
  const int32_t* src = topk_idx + int64_t(s) * nk;
  int32_t* slots = slot_row + int64_t(s) * nk;
  const int64_t seg_len = (nk + nseg - 1) / nseg;
  const int64_t g0 = min(nk, int64_t(warp) * seg_len), g1 = min(nk, g0 + seg_len);
  // 1. one pass over the ids: per (segment, bin) counts of this rank's
  //    entries and, when num_tokens_per_expert is NULL, every rank's per-bin
  //    totals and the lower-rank prefixes (ids outside [-1, E) then flagged as
  //    the layout would); else the totals and prefixes from the layout's
  //    counts.  Each thread loads kLLIds ids per batch (16-byte loads where
  //    aligned) before its shared-memory adds, and the first batch's loads are
  //    issued before the counters are cleared.
  const bool self_count = num_tokens_per_expert == nullptr;
  const int64_t mine = int64_t(s) * nk;
  const int64_t lo = self_count ? 0 : mine, hi = self_count ? int64_t(R) * nk : mine + nk;
  const bool vec = (reinterpret_cast<uintptr_t>(topk_idx) & 15u) == 0 && lo % 4 == 0 &&
                   hi % 4 == 0;
  const int64_t per_batch = int64_t(kLLIds) * NT;
  int ids[kLLIds];
  auto id_index = [&](int64_t b0, int j) -> int64_t {
    return vec ? b0 + (int64_t(j / 4) * NT + tid) * 4 + (j & 3) : b0 + int64_t(j) * NT + tid;
  };
  auto load_batch = [&](int64_t b0) {
    if (vec) {
#pragma unroll
      for (int j = 0; j < kLLIds / 4; ++j) {
        const int64_t i = b0 + (int64_t(j) * NT + tid) * 4;
        const int4 q = i < hi ? __ldg(reinterpret_cast<const int4*>(topk_idx + i))
                              : make_int4(-1, -1, -1, -1);
        ids[4 * j] = q.x;
        ids[4 * j + 1] = q.y;
        ids[4 * j + 2] = q.z;
        ids[4 * j + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kLLIds; ++j) {
        const int64_t i = b0 + int64_t(j) * NT + tid;
        ids[j] = i < hi ? __ldg(topk_idx + i) : -1;
      }
    }
  };
  bool bad = false;
  auto count_batch = [&](int64_t b0) {
#pragma unroll
    for (int j = 0; j < kLLIds; ++j) {
      const int e = ids[j];
      if (e < 0 || e >= E) {
        bad |= e != -1;
        continue;
      }
      const int64_t i = id_index(b0, j);
      const int b = bin_of(e);
      if (i >= mine && i < mine + nk)
        atomicAdd(&hist[int(i - mine) / int(seg_len) * nbins + b], 1);
      if (self_count) {
        atomicAdd(&tot[b], 1);
        if (i < mine) atomicAdd(&pre[b], 1);
      }
    }
  };
  if (lo < hi) load_batch(lo);
  for (int i = tid; i < (nseg + 3) * nbins; i += NT) ll_smem[i] = 0;
  __syncthreads();
  if (lo < hi) count_batch(lo);
  for (int64_t b0 = lo + per_batch; b0 < hi; b0 += per_batch) {
    load_batch(b0);
    count_batch(b0);
  }
  if (!self_count) {
    for (int e = tid; e < E; e += NT) {
      int t = 0, p = 0;
      for (int q = 0; q < R; ++q) {
        const int c = __ldg(num_tokens_per_expert + int64_t(q) * E + e);
        t += c;
        if (q < s) p += c;
      }
      if (RANK_MAJOR) {
        atomicAdd(&tot[bin_of(e)], t);
        atomicAdd(&pre[bin_of(e)], p);
      } else {
        tot[e] = t;
        pre[e] = p;
      }
    }
  } else if (bad && s == 0) {
    raise_error(dev_err, MP_ERR_BAD_EXPERT);
  }
  __syncthreads();
  // 2a. this thread's bins [b0, b1) and their totals over every source rank
  const int cpt = (nbins + NT - 1) / NT;
  const int b0 = min(nbins, tid * cpt), b1 = min(nbins, b0 + cpt);
  int64_t chunk = 0;
  for (int b = b0; b < b1; ++b) chunk += tot[b];
  int64_t inc = chunk;  // block-wide exclusive scan of the chunk totals
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t v = __shfl_up_sync(kFull, inc, o);
    if (lane >= o) inc += v;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();  // also orders the segment counts before 2b
  if (warp == 0) {
    int64_t w = lane < NT / kWarp ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t v = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += v;
    }
    if (lane < NT / kWarp) warp_sums[lane] = w;
  }
  __syncthreads();
  int64_t base = (warp > 0 ? warp_sums[warp - 1] : 0) + inc - chunk;
  // 2b. per bin: outputs, first row of this rank, exclusive prefix over segments
  for (int b = b0; b < b1; ++b) {
    if (s == 0) bin_offsets[b] = int32_t(base);
    bin_src_offsets[int64_t(b) * R + s] = pre[b];
    rowbase[b] = int32_t(base + pre[b]);
    int run = 0;
    for (int g = 0; g < nseg; ++g) {
      const int c = hist[g * nbins + b];
      hist[g * nbins + b] = run;
      run += c;
    }
    base += tot[b];
  }
  if (s == 0 && b0 < nbins && b1 == nbins) bin_offsets[nbins] = int32_t(base);
  __syncthreads();
  // 3. rows, segment by segment in entry order
  bool overflow = false;
  if (warp < nseg) {
    for (int64_t i00 = g0; i00 < g1; i00 += int64_t(kLLBatch) * kWarp) {
      int v[kLLBatch];  // the batch's ids, loaded before the in-order walk
#pragma unroll
      for (int j = 0; j < kLLBatch; ++j) {
        const int64_t i = i00 + int64_t(j) * kWarp + lane;
        v[j] = i < g1 ? __ldg(src + i) : -1;
      }
#pragma unroll
      for (int j = 0; j < kLLBatch; ++j) {
        if (i00 + int64_t(j) * kWarp >= g1) break;  // (the same for the whole warp)
        const int64_t i = i00 + int64_t(j) * kWarp + lane;
        const int e = v[j];
        const bool ok = e >= 0 && e < E;
        const int b = ok ? bin_of(e) : -1;
        const unsigned peers = __match_any_sync(kFull, b);
        const int run = ok ? hist[warp * nbins + b] : 0;
        __syncwarp();
        if (ok) {
          const int64_t row = int64_t(rowbase[b]) + run + __popc(peers & lanemask_lt());
          if (row < recv_capacity) {
            slots[i] = int32_t(row);
            recv_src_token[row] = int32_t(int64_t(s) * N + i / K);
          } else {
            slots[i] = -1;
            overflow = true;
          }
          if ((peers >> lane) == 1u) hist[warp * nbins + b] = run + __popc(peers);  // highest peer
        } else if (i < g1) {
          slots[i] = -1;  // masked or invalid: no row
        }
        __syncwarp();
      }
    }
  }
  if (overflow) raise_error(dev_err, MP_ERR_CAPACITY);
}

template <bool RANK_MAJOR>
__global__ void __launch_bounds__(kLLThreads)
mp_k_ll_offsets(int R, int N, int K, int E, const int32_t* __restrict__ topk_idx,
                const int32_t* __restrict__ num_tokens_per_expert, int64_t recv_capacity,
                int32_t* __restrict__ bin_offsets, int32_t* __restrict__ bin_src_offsets,
                int32_t* __restrict__ recv_src_token, int32_t* __restrict__ slot_row,
                int32_t* __restrict__ dev_err) {
  // a row copy launched as this grid's programmatic dependent may start now:
  // it reads slot_row only after this grid has finished
  pdl_launch_dependents();
  // launched as a programmatic dependent of the kernel before it on the stream:
  // wait for it before any global memory access
  pdl_wait_prior_grid();
  extern __shared__ int32_t ll_smem[];
  __shared__ int64_t warp_sums[kLLThreads / kWarp];
  ll_offsets_block<RANK_MAJOR, kLLThreads, kLLHistInts>(
      blockIdx.x, R, N, K, E, topk_idx, num_tokens_per_expert, recv_capacity, bin_offsets,
      bin_src_offsets, recv_src_token, slot_row, dev_err, ll_smem, warp_sums);
}


// ---------------------------------------------------------------------------
// Layout and receive offsets for small batches in one thread-block cluster
// (mp_layout_and_offsets / mp_layout_dispatch when R <= 16 and N is at most
// MP_CLUSTER_MAX_TOKENS): CTA s of an R-CTA cluster takes source rank s whole.
//  1. in rounds of 1024 tokens: each token's rank mask (is_token_in_rank), the
//     rank's expert histogram in shared memory and, per (round, warp), a ballot
//     per destination; one warp per destination scans the ballots' counts,
//     which places every token among the rank's rows for that destination and
//     gives the rank's total per destination;
//  2. cluster barrier; each CTA reads the other ranks' totals, and for the
//     experts its rank owns their counts, from those CTAs' shared memory
//     (distributed shared memory): no global round trip, no workspace;
//  3. the tables, send_row (and with META the receive metadata);
//  4. a second cluster barrier keeps every CTA's shared memory alive until the
//     others have read it.
// Every thread reaches both cluster barriers (there is no early exit).
// ---------------------------------------------------------------------------
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / kWarp;
constexpr int kClMaxRounds = 4;  // tokens per rank <= 4096
constexpr int kClMaxRanks = 16;  // a cluster of at most 16 CTAs

struct ClusterArgs {
  int R, N, K, E;
  const int32_t* topk_idx;
  const float* topk_weights;
  int64_t recv_capacity;
  uint32_t* is_token_in_rank;
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  int32_t* recv_src_rank;
  int32_t* recv_src_idx;
  int32_t* recv_topk_idx;
  float* recv_topk_weights;
  int32_t* dest_offsets;
  int32_t* rank_prefix;
  int32_t* num_recv_tokens_per_expert;
  int32_t* send_row;
  int32_t* dev_err;
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: writes before it (shared and
// global) are visible to the cluster's threads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The 32-bit word at shared-memory address `p` of CTA `rank` of the cluster.
__device__ __forceinline__ int32_t ld_peer_smem(const void* p, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(p)), "r"(rank));
  int32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

template <bool META>
__global__ void __launch_bounds__(kClThreads, 1) mp_k_layout_cluster(ClusterArgs a) {
  extern __shared__ int32_t cl_hist[];  // [E]: this rank's expert counts (read by peers)
  __shared__ uint32_t ball[kClMaxRounds][kClWarps][kClMaxRanks];
  __shared__ int32_t woff[kClMaxRounds][kClWarps][kClMaxRanks];
  __shared__ int32_t tot[kClMaxRanks];  // this rank's rows per destination (read by peers)
  __shared__ int32_t ntpr[kClMaxRanks * kClMaxRanks];
  __shared__ int64_t row_base[kClMaxRanks];
  __shared__ int sh_bad;
  const int R = a.R, N = a.N, K = a.K, E = a.E, El = E / R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = int(cluster_ctarank());
  pdl_launch_dependents();
  // launched as a programmatic dependent of the kernel before it on the stream:
  // wait for it before any global memory access
  pdl_wait_prior_grid();
  const int rounds = (N + kClThreads - 1) / kClThreads;

  // 1. the ids of every round first (8 per token and round in flight), then
  //    the counting
  int ids[kClMaxRounds][8];
#pragma unroll
  for (int r = 0; r < kClMaxRounds; ++r) {
    const int t = r * kClThreads + tid;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      ids[r][j] = (r < rounds && t < N && j < K) ? __ldg(a.topk_idx + (int64_t(s) * N + t) * K + j)
                                                 : -1;
  }
  for (int e = tid; e < E; e += kClThreads) cl_hist[e] = 0;
  if (tid == 0) sh_bad = 0;
  __syncthreads();
  bool bad = false;
  uint32_t masks[kClMaxRounds];
#pragma unroll
  for (int r = 0; r < kClMaxRounds; ++r) {
    masks[r] = 0u;
    if (r >= rounds) continue;
    const int t = r * kClThreads + tid;
    if (t < N) {
      uint32_t m = 0u;
      for (int k0 = 0; k0 < K; k0 += 8) {
        int e8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          e8[j] = k0 == 0 ? ids[r][j]
                          : (k0 + j < K ? __ldg(a.topk_idx + (int64_t(s) * N + t) * K + k0 + j)
                                        : -1);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int e = e8[j];
          if (k0 + j >= K || e == -1) continue;
          if (e < -1 || e >= E) { bad = true; continue; }
          atomicAdd(&cl_hist[e], 1);
          m |= 1u << (e / El);
        }
      }
      masks[r] = m;
      a.is_token_in_rank[int64_t(s) * N + t] = m;
    }
    for (int d = 0; d < R; ++d) {
      const unsigned b = __ballot_sync(kFull, (masks[r] >> d) & 1u);
      if (lane == 0) ball[r][warp][d] = b;
    }
  }
  if (bad) sh_bad = 1;
  __syncthreads();
  if (warp < R) {  // destination d = warp: the counts of every (round, warp), in order
    const int d = warp, n = rounds * kClWarps;  // n <= 128: 4 entries per lane
    int v[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane * 4 + q;
      v[q] = j < n ? __popc(ball[j / kClWarps][j % kClWarps][d]) : 0;
      sum += v[q];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += x;
    }
    int run = inc - sum;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = lane * 4 + q;
      if (j < n) woff[j / kClWarps][j % kClWarps][d] = run;
      run += v[q];
    }
    if (lane == 31) tot[d] = inc;
  }
  for (int e = tid; e < E; e += kClThreads) a.num_tokens_per_expert[int64_t(s) * E + e] = cl_hist[e];
  if (tid == 0 && sh_bad) raise_error(a.dev_err, MP_ERR_BAD_EXPERT);

  // 2. every rank's totals and histogram are final
  cluster_sync_all();
  if (tid < R * R) {
    const int q = tid / R, d = tid - q * R;
    ntpr[tid] = q == s ? tot[d] : ld_peer_smem(&tot[d], uint32_t(q));
  }
  for (int j = tid; j < El; j += kClThreads) {  // the experts destination s owns
    const int e = s * El + j;
    int sum = 0;
    for (int q0 = 0; q0 < R; q0 += 8) {
      int c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        c[i] = q0 + i >= R ? 0 : (q0 + i == s ? cl_hist[e] : ld_peer_smem(&cl_hist[e], uint32_t(q0 + i)));
#pragma unroll
      for (int i = 0; i < 8; ++i) sum += c[i];
    }
    a.num_recv_tokens_per_expert[e] = sum;
  }
  __syncthreads();

  // 3. tables and rows
  if (warp == 0) {
    int64_t col = 0, pre = 0;
    if (lane < R)
      for (int q = 0; q < R; ++q) {
        const int v = ntpr[q * R + lane];
        col += v;
        if (q < s) pre += v;
      }
    int64_t inc = col;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t x = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += x;
    }
    if (lane < R) {
      row_base[lane] = inc - col + pre;
      a.num_tokens_per_rank[s * R + lane] = tot[lane];
      a.rank_prefix[s * R + lane] = int32_t(pre);
      if (s == 0) {
        a.dest_offsets[lane] = int32_t(inc - col);
        if (lane == R - 1) a.dest_offsets[R] = int32_t(inc);
      }
    }
  }
  __syncthreads();
  bool over = false;
#pragma unroll
  for (int r = 0; r < kClMaxRounds; ++r) {
    const int t = r * kClThreads + tid;
    if (r >= rounds || t >= N) continue;
    const int64_t tok = int64_t(s) * N + t;
    int32_t* dst = a.send_row + tok * R;
    for (int d = 0; d < R; ++d) {
      int32_t v = -1;
      if ((masks[r] >> d) & 1u) {
        const int64_t row = row_base[d] + woff[r][warp][d] + __popc(ball[r][warp][d] & lanemask_lt());
        if (row < a.recv_capacity) {
          v = int32_t(row);
          if constexpr (META) {
            a.recv_src_rank[row] = s;
            a.recv_src_idx[row] = t;
            const int lo = d * El;
            for (int k = 0; k < K; ++k) {
              const int e = __ldg(a.topk_idx + tok * K + k);
              const bool local = e >= lo && e < lo + El;
              a.recv_topk_idx[row * K + k] = local ? e - lo : -1;
              a.recv_topk_weights[row * K + k] = local ? __ldg(a.topk_weights + tok * K + k) : 0.0f;
            }
          }
        } else {
          over = true;
        }
      }
      dst[d] = v;
    }
  }
  if (__any_sync(kFull, over) && lane == 0) raise_error(a.dev_err, MP_ERR_CAPACITY);

  // 4. the peers have read this CTA's shared memory
  cluster_sync_all();
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
  return launch_kernel(mp_k_layout, dim3(grid), dim3(kLayoutTokens), smem, stream, R, N, K, E,
                       topk_idx, num_tokens_per_rank, num_tokens_per_expert, is_token_in_rank,
                       dev_err, ws);
}

cudaError_t launch_scan(int R, int N, int K, int E, const int32_t* topk_idx,
                        const float* topk_weights, const uint32_t* is_token_in_rank,
                        const int32_t* num_tokens_per_rank, const int32_t* num_tokens_per_expert,
                        int64_t recv_capacity, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int32_t* dest_offsets,
                        int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                        int32_t* send_row, int32_t* dev_err, unsigned char* ws,
                        cudaStream_t stream, int global_ids, int32_t sentinel) {
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
             dev_err, ws, global_ids, sentinel};
  const size_t smem = sizeof(int32_t) * size_t(kScanTokens) * (2 * size_t(K) + R);
  static thread_local int configured_smem[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && configured_smem[dev] < int(smem) && smem > 32 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(mp_k_scan, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    configured_smem[dev] = int(smem);
  }
  return launch_kernel(mp_k_scan, dim3(unsigned(scan_tiles(R, N))), dim3(kScanThreads), smem,
                       stream, a);
}



// Token count up to which layout + offsets run in one thread-block cluster.
// Measured (globaltimer, dsv3 shape R=8, one-call dispatch): the row copy's wait
// returned 1.3 us earlier than after the cooperative kernel at N=128, at the
// same time at N=512, and 3.5 us later at N=1024 (one CTA per rank then writes
// too many rows).
#ifndef MP_CLUSTER_MAX_TOKENS
#define MP_CLUSTER_MAX_TOKENS 256
#endif

// Layout + offsets in one thread-block cluster (one CTA per source rank);
// cudaErrorNotSupported (nothing launched) when the shape does not suit it.
cudaError_t launch_layout_cluster(int R, int N, int K, int E, const int32_t* topk_idx,
                                  const float* topk_weights, int64_t recv_capacity,
                                  int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                                  uint32_t* is_token_in_rank, int32_t* recv_src_rank,
                                  int32_t* recv_src_idx, int32_t* recv_topk_idx,
                                  float* recv_topk_weights, int32_t* dest_offsets,
                                  int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                                  int32_t* send_row, int32_t* dev_err, cudaStream_t stream,
                                  int meta) {
  if (N < 1 || N > MP_CLUSTER_MAX_TOKENS || N > kClMaxRounds * kClThreads || R > kClMaxRanks)
    return cudaErrorNotSupported;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorNotSupported;
  // per device and instance: 0 unknown, -1 unusable, else the largest cluster size that
  // could be scheduled when it was set up
  static thread_local int ready[64][2] = {};
  static thread_local int configured_smem[64][2] = {};
  void (*kernel)(ClusterArgs) = meta ? mp_k_layout_cluster<true> : mp_k_layout_cluster<false>;
  const int v = meta ? 1 : 0;
  const size_t smem = sizeof(int32_t) * size_t(E);
  if (ready[dev][v] == 0) {
    int ok = 0;
    if (cudaDeviceGetAttribute(&ok, cudaDevAttrClusterLaunch, dev) != cudaSuccess || !ok ||
        cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
      ready[dev][v] = -1;
      return cudaErrorNotSupported;
    }
    ready[dev][v] = 1;
  }
  if (ready[dev][v] < 0) return cudaErrorNotSupported;
  if (smem > 48 * 1024 && configured_smem[dev][v] < int(smem)) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
        cudaSuccess)
      return cudaErrorNotSupported;
    configured_smem[dev][v] = int(smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(R));
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(R);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // can a cluster of R such CTAs be scheduled at all (cached per size and memory)?
  static thread_local int checked[64][2][kClMaxRanks + 1] = {};
  if (checked[dev][v][R] != int(smem) + 1) {
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kernel, &cfg) != cudaSuccess ||
        nclusters < 1) {
      cudaGetLastError();  // clear a refused query
      return cudaErrorNotSupported;
    }
    checked[dev][v][R] = int(smem) + 1;
  }
  ClusterArgs args{R, N, K, E, topk_idx, topk_weights, recv_capacity, is_token_in_rank,
                   num_tokens_per_rank, num_tokens_per_expert, recv_src_rank, recv_src_idx,
                   recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                   num_recv_tokens_per_expert, send_row, dev_err};
  // launched as a programmatic dependent of the kernel before it (it waits first)
  cudaLaunchAttribute attr2[2] = {attr[0], {}};
  attr2[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr2[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr2;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, args);
}

// Returns cudaErrorNotSupported (nothing launched) when the problem does not
// fit one cooperative grid; the caller then runs mp_k_layout and mp_k_scan.
cudaError_t launch_layout_scan(int R, int N, int K, int E, const int32_t* topk_idx,
                               const float* topk_weights, int64_t recv_capacity,
                               int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert,
                               uint32_t* is_token_in_rank, int32_t* recv_src_rank,
                               int32_t* recv_src_idx, int32_t* recv_topk_idx,
                               float* recv_topk_weights, int32_t* dest_offsets,
                               int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
                               int32_t* send_row, int32_t* dev_err, unsigned char* ws,
                               cudaStream_t stream, int meta) {
  if (N == 0) return cudaErrorNotSupported;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorNotSupported;
  static thread_local int coop[64] = {0};  // 0 unknown, 1 supported, -1 not
  if (coop[dev] == 0) {
    int v = 0;
    coop[dev] = (cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess &&
                 v) ? 1 : -1;
  }
  if (coop[dev] < 0) return cudaErrorNotSupported;
  const size_t smem =
      sizeof(int32_t) * (size_t(kScanTokens) * (2 * size_t(K) + size_t(R)) + size_t(E));
  const int lookback = scan_tiles_per_rank(N) > kFusedAggMaxTiles ? 1 : 0;
  void (*kernel)(FusedArgs) =
      meta ? (lookback ? mp_k_layout_scan<true, true> : mp_k_layout_scan<true, false>)
           : (lookback ? mp_k_layout_scan<false, true> : mp_k_layout_scan<false, false>);
  const int variant = (meta ? 2 : 0) + lookback;
  static thread_local int configured[64][4] = {};
  if (smem > 48 * 1024 && configured[dev][variant] < int(smem)) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return cudaErrorNotSupported;
    configured[dev][variant] = int(smem);
  }
  // resident blocks per SM, cached per device, instance and shared-memory size
  static thread_local int occ_smem[64][4] = {}, occ_per_sm[64][4] = {};
  if (occ_per_sm[dev][variant] < 1 || occ_smem[dev][variant] != int(smem)) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kScanThreads, smem) !=
            cudaSuccess ||
        per_sm < 1)
      return cudaErrorNotSupported;
    occ_smem[dev][variant] = int(smem);
    occ_per_sm[dev][variant] = per_sm;
  }
  const int per_sm = occ_per_sm[dev][variant];
  const int64_t tiles = scan_tiles(R, N);
  const int64_t cap = int64_t(per_sm) * sm_count();
  const int64_t grid = tiles < cap ? tiles : cap;
  if (tiles > grid * kFusedMaxTiles) return cudaErrorNotSupported;
  FusedArgs f{ScanArgs{R, N, K, E, topk_idx, topk_weights, is_token_in_rank, num_tokens_per_rank,
                       num_tokens_per_expert, recv_capacity, recv_src_rank, recv_src_idx,
                       recv_topk_idx, recv_topk_weights, dest_offsets, rank_prefix,
                       num_recv_tokens_per_expert, send_row, dev_err, ws, 0, -1},
              is_token_in_rank, num_tokens_per_rank, num_tokens_per_expert};
  void* args[] = {&f};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kernel), dim3(unsigned(grid)),
                                     dim3(kScanThreads), args, smem, stream);
}
}  // namespace mp

namespace mp {

template <bool RANK_MAJOR>
static cudaError_t ll_offsets(int R, int N, int K, int E, const int32_t* topk_idx,
                              const int32_t* num_tokens_per_expert, int64_t recv_capacity,
                              int32_t* bin_offsets, int32_t* bin_src_offsets,
                              int32_t* recv_src_token, int32_t* slot_row, int32_t* dev_err,
                              cudaStream_t stream) {
  const int nbins = RANK_MAJOR ? R : E;
  const size_t smem = sizeof(int32_t) * size_t(ll_segments(nbins) + 3) * size_t(nbins);
  static thread_local int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > 48 * 1024 && configured[dev] < int(smem)) {
    cudaError_t e = cudaFuncSetAttribute(mp_k_ll_offsets<RANK_MAJOR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = int(smem);
  }
  // launched as a programmatic dependent of the kernel before it (it waits first)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(R));
  cfg.blockDim = dim3(kLLThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mp_k_ll_offsets<RANK_MAJOR>, R, N, K, E, topk_idx,
                            num_tokens_per_expert, recv_capacity, bin_offsets, bin_src_offsets,
                            recv_src_token, slot_row, dev_err);
}

// The low-latency dispatch: the sort, then the row copy launched as its
// programmatic dependent, whose row loads overlap the sort (measured against
// one kernel doing both, whose copy blocks waited for per-rank ready flags:
// 31.4 vs 34.8 us at R=8, N=128, top-8 of 256, H=7168; 96 vs 103 us at N=512).
cudaError_t launch_ll_dispatch(int R, int N, int K, int E, int rank_major, int64_t row_bytes,
                               const int32_t* topk_idx, const int32_t* num_tokens_per_expert,
                               int64_t recv_capacity, int32_t* bin_offsets,
                               int32_t* bin_src_offsets, int32_t* recv_src_token,
                               int32_t* slot_row, const void* x, int scales_per_row,
                               const float* x_scales, void* recv_x, float* recv_scales,
                               int32_t* dev_err, cudaStream_t stream) {
  if (num_tokens_per_expert == nullptr) {
    const cudaError_t f = launch_ll_dispatch_fused(
        R, N, K, E, rank_major, row_bytes, topk_idx, recv_capacity, bin_offsets, bin_src_offsets,
        recv_src_token, slot_row, x, scales_per_row, x_scales, recv_x, recv_scales, dev_err,
        stream);
    if (f != cudaErrorNotSupported) return f;
  }
  cudaError_t e = launch_ll_offsets(R, N, K, E, rank_major, topk_idx, num_tokens_per_expert,
                                    recv_capacity, bin_offsets, bin_src_offsets, recv_src_token,
                                    slot_row, dev_err, stream);
  if (e != cudaSuccess || N == 0) return e;
  return launch_ll_rows_after_sort(K, int64_t(R) * N, row_bytes, x, recv_x, recv_capacity,
                                   slot_row, scales_per_row, x_scales, recv_scales, stream);
}

cudaError_t launch_ll_offsets(int R, int N, int K, int E, int rank_major,
                              const int32_t* topk_idx, const int32_t* num_tokens_per_expert,
                              int64_t recv_capacity, int32_t* bin_offsets,
                              int32_t* bin_src_offsets, int32_t* recv_src_token,
                              int32_t* slot_row, int32_t* dev_err, cudaStream_t stream) {
  return rank_major
             ? ll_offsets<true>(R, N, K, E, topk_idx, num_tokens_per_expert, recv_capacity,
                                bin_offsets, bin_src_offsets, recv_src_token, slot_row, dev_err,
                                stream)
             : ll_offsets<false>(R, N, K, E, topk_idx, num_tokens_per_expert, recv_capacity,
                                 bin_offsets, bin_src_offsets, recv_src_token, slot_row, dev_err,
                                 stream);
}

}  // namespace mp
