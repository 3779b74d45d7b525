// mp_copy_kernels.cu -- the HBM-bound payload kernels: dispatch row copy
// (SM vectors, or the bulk-copy engine), quantising row copies (dispatch or
// gather destinations), combine (gather + fp32 sum, plain or top-k
// weighted), combined top-k weights, reduce-scatterv (fp32 sum of R inputs),
// all-gatherv (one read, R writes; one tensor or a list), and the
// low-latency row copy launched as a programmatic dependent of the LL sort.
//
// All are streaming kernels: nothing is reused, so they are bound by
// HBM bandwidth and the design goal is bytes in flight with few
// instructions.  The work is split into small units handed out to warps:
//   dispatch / combine : (token, slab) with a slab of 32 lanes x U vectors of
//                        the token's row, so consecutive warps stream
//                        consecutive slabs of the same row and the per-SM
//                        load evens out across rows of unequal fan-out;
//   reduce-scatterv / all-gatherv : vectors of the flat arrays.
// Payload moves as 32-byte vectors (the 256-bit global loads and stores of
// sm_100-class GPUs) when the row size and the pointers allow, else as
// 16-byte vectors; loads bypass L1 and are marked evict-first in L2.
// Read-dominated kernels (combine) run a persistent grid; write-dominated ones
// one short block per few units (see grid_full).
#include <cstdint>

#include "mp_common.cuh"
#include "mp_internal.h"

// Compile-time tuning (vector words: 8 = 32-byte, 4 = 16-byte accesses).
#ifndef MP_DISPATCH_NW
#define MP_DISPATCH_NW 8
#endif
#ifndef MP_DISPATCH_U
#define MP_DISPATCH_U 4
#endif
#ifndef MP_COMBINE_NW
#define MP_COMBINE_NW 8
#endif
#ifndef MP_COMBINE_U
#define MP_COMBINE_U 1
#endif
// Combine: rows read per batch and blocks per SM.  Measured on the dsv3
// combine (439 us with 4 rows and 3 blocks): 3 rows and 4 blocks 437 us,
// 3 rows and 3 blocks 440, 2 rows and 4 blocks 442, 2 and 5 484, 6 rows 466;
// 4 rows with 4 blocks spills (605 us).
#ifndef MP_COMBINE_RB
#define MP_COMBINE_RB 3
#endif
#ifndef MP_COMBINE_MINB
#define MP_COMBINE_MINB 4
#endif
// The weighted (low-latency) combine's shape; by default the unweighted one's.
// Measured at R=8, N=128, top-8 (8 rows per token): 16-byte vectors with all 8
// rows in flight (NW=4, U=1, RB=8) 29.8 us, 6 rows 30.0 us, against 28.5 us for
// the default; for the dsv3 combine 16-byte vectors cost 491-524 vs 440 us.
#ifndef MP_COMBINE_W_NW
#define MP_COMBINE_W_NW MP_COMBINE_NW
#endif
#ifndef MP_COMBINE_W_U
#define MP_COMBINE_W_U MP_COMBINE_U
#endif
#ifndef MP_COMBINE_W_RB
#define MP_COMBINE_W_RB MP_COMBINE_RB
#endif
// Small dispatches (fewer warp units at the default shape than the GPU holds
// warps, e.g. the low-latency batches of 128 tokens per rank) use 1 vector per
// lane and unit instead, for 4x the units: measured 29 -> 25 us for the rows
// of R=8, N=128, top-8, H=7168 (MP_SMALL_DISPATCH = 0 turns this off).
#ifndef MP_SMALL_DISPATCH
#define MP_SMALL_DISPATCH 1
#endif

// Shapes of the other copies.
// 1: the e4m3 quantiser divides by the block scale with a reciprocal and two
// FMA corrections instead of a division per element (see mp_k_quant_rows);
// 0: one correctly rounded division per element.
#ifndef MP_QUANT_FAST_DIV
#define MP_QUANT_FAST_DIV 1
#endif
// Quantising copies with 32 channels per lane (two 32-byte loads, one scale
// per lane for the 32-channel microscaling blocks, 32-byte FP8 code stores),
// per kind: bit FMT + (GATHER ? 3 : 0).  Measured against 16 channels per
// lane: e4m3 dispatch 256 vs 269 us, MXFP8 dispatch 255 vs 260, MXFP4
// dispatch 185 vs 184; gathers 270 vs 275 (e4m3), 269 vs 274 (MXFP8), 168 vs
// 174 (MXFP4).
#ifndef MP_QUANT_CPL32_MASK
#define MP_QUANT_CPL32_MASK 59
#endif
// Bulk-copy (TMA) dispatch: shared-memory stages per block, tokens per chunk,
// bytes per bulk copy, and one short block per chunk (1) or a persistent grid
// (0).  Measured on the dsv3 rows: a persistent grid stays near 500 us for
// every stage / chunk / piece shape tried (3-8 stages, 2-16 tokens, 4-16 KB);
// one block per chunk gives 444 us, and 3 stages of 8 KB with 2-token chunks
// 442 us.
#ifndef MP_TMA_STAGES
#define MP_TMA_STAGES 3
#endif
#ifndef MP_TMA_CHUNK
#define MP_TMA_CHUNK 2
#endif
#ifndef MP_TMA_PIECE
#define MP_TMA_PIECE 8192
#endif
#ifndef MP_TMA_GRID_FULL
#define MP_TMA_GRID_FULL 1
#endif

namespace mp {

constexpr int kCopyThreads = 256;
constexpr int kWarpsPerBlock = kCopyThreads / kWarp;

// ---------------------------------------------------------------------------
// Dispatch copy ("MSCCLPP EP implementation", microsoft/mscclpp PR #852:
// intranode_dispatch moves each token row, as vectors, to every rank that
// owns one of its experts).  One read of x, one write per receive row.
// ---------------------------------------------------------------------------
template <int NW, int U>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_dispatch(int R, int64_t tokens, int64_t vpr, const Words<NW>* __restrict__ x,
              Words<NW>* __restrict__ recv_x, int64_t recv_capacity,
              const int32_t* __restrict__ send_row, int spr, const float* __restrict__ x_scales,
              float* __restrict__ recv_scales) {
  pdl_launch_dependents();  // a combine launched as a dependent may stage its blocks
  const int lane = threadIdx.x & 31;
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * kWarpsPerBlock;
  for (int64_t unit = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); unit < units;
       unit += nw) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    const int my = lane < R ? __ldg(send_row + tok * R + lane) : -1;
    unsigned vm = __ballot_sync(kFull, my >= 0 && int64_t(my) < recv_capacity);
    if (vm == 0) continue;
    const int64_t i0 = slab * slab_vec + lane;
    Words<NW> v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kWarp < vpr) v[u] = ld_stream_w<NW>(x + tok * vpr + i0 + u * kWarp);
    while (vm) {
      const int d = __ffs(vm) - 1;
      vm &= vm - 1;
      const int64_t row = __shfl_sync(kFull, my, d);
      Words<NW>* dst = recv_x + row * vpr;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kWarp < vpr) st_stream_w<NW>(dst + i0 + u * kWarp, v[u]);
      if (spr > 0 && slab == 0)
        for (int c = lane; c < spr; c += kWarp)
          recv_scales[row * spr + c] = __ldg(x_scales + tok * spr + c);
    }
  }
}

// ---------------------------------------------------------------------------
// The row copy of mp_layout_dispatch: mp_k_dispatch launched as the
// programmatic dependent of the fused layout + offsets kernel, which also
// writes the receive metadata the fused kernel leaves out.  Its blocks may
// start while that kernel runs: each warp loads its first unit's row vectors
// (and, for a token's first slab, the token's top-k ids and weights) -- inputs
// of the call, complete before it began -- then waits for the offsets grid to
// finish (griddepcontrol.wait) and only then reads send_row.  For every
// receive row of a token the warp of its first slab writes recv_src_rank,
// recv_src_idx and the K local top-k ids and weights (e - d*E/R and the weight
// for an expert on the row's destination d, else -1 and 0).
// ---------------------------------------------------------------------------
template <int NW, int U>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_dispatch_after_offsets(int R, int N, int K, int El, int64_t tokens, int64_t vpr,
                            const Words<NW>* __restrict__ x, Words<NW>* __restrict__ recv_x,
                            int64_t recv_capacity, const int32_t* send_row, int spr,
                            const float* __restrict__ x_scales, float* __restrict__ recv_scales,
                            const int32_t* __restrict__ topk_idx,
                            const float* __restrict__ topk_weights,
                            int32_t* __restrict__ recv_src_rank, int32_t* __restrict__ recv_src_idx,
                            int32_t* __restrict__ recv_topk_idx,
                            float* __restrict__ recv_topk_weights) {
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * kWarpsPerBlock;
  int64_t unit = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  Words<NW> v[U];
  int my_e = -1;
  float my_w = 0.0f;
  auto load_unit = [&](int64_t u0) {
    const int64_t tok = u0 / slabs, i0 = (u0 - tok * slabs) * slab_vec + lane;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kWarp < vpr) v[u] = ld_stream_w<NW>(x + tok * vpr + i0 + u * kWarp);
    if (i0 < kWarp && lane < K) {  // the token's first slab: its top-k ids and weights
      my_e = __ldg(topk_idx + tok * K + lane);
      my_w = __ldg(topk_weights + tok * K + lane);
    }
  };
  if (unit < units) load_unit(unit);
  pdl_wait_prior_grid();
  for (bool first = true; unit < units; unit += nw, first = false) {
    if (!first) load_unit(unit);
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    const int64_t i0 = slab * slab_vec + lane;
    // send_row was written by the offsets grid: read through L2, not the read-only path
    const int my = lane < R ? __ldcg(send_row + tok * R + lane) : -1;
    unsigned vm = __ballot_sync(kFull, my >= 0 && int64_t(my) < recv_capacity);
    while (vm) {
      const int d = __ffs(vm) - 1;
      vm &= vm - 1;
      const int64_t row = __shfl_sync(kFull, my, d);
      Words<NW>* dst = recv_x + row * vpr;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kWarp < vpr) st_stream_w<NW>(dst + i0 + u * kWarp, v[u]);
      if (slab == 0) {
        if (spr > 0)
          for (int c = lane; c < spr; c += kWarp)
            recv_scales[row * spr + c] = __ldg(x_scales + tok * spr + c);
        const int src = int(tok / N);
        if (lane == 0) recv_src_rank[row] = src;
        if (lane == 1) recv_src_idx[row] = int(tok - int64_t(src) * N);
        if (lane < K) {
          const int lo = d * El;
          const bool local = my_e >= lo && my_e < lo + El;
          recv_topk_idx[row * K + lane] = local ? my_e - lo : -1;
          recv_topk_weights[row * K + lane] = local ? my_w : 0.0f;
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Dispatch copy with the bulk-copy (TMA) engine.  One warp per block; lane 0
// streams the block's token rows through a ring of NS shared-memory stages:
// a global->shared bulk load per row piece (completing on the stage's
// mbarrier), then one contiguous shared->global bulk store per destination.
// A stage is refilled once the stores issued LAG items earlier have finished
// reading it.  Blocks take chunks of kTmaChunk tokens round-robin (one chunk
// per block on the default short-block grid); the chunk's send_row entries are
// staged in shared memory by the whole warp.
// ---------------------------------------------------------------------------
constexpr int kTmaStages = MP_TMA_STAGES;
constexpr int kTmaLag = 2;
constexpr int kTmaChunk = MP_TMA_CHUNK;
constexpr uint32_t kTmaPiece = MP_TMA_PIECE;  // bytes per bulk copy (rows are cut into pieces)
static_assert(kTmaLag < kTmaStages, "lag below the stage count");

__host__ __device__ inline size_t tma_smem_bytes(uint32_t piece_bytes) {
  return size_t(kTmaStages) * piece_bytes + size_t(kTmaChunk) * MP_MAX_RANKS * 4 +
         size_t(kTmaStages) * 8;
}

__global__ void __launch_bounds__(kWarp)
mp_k_dispatch_tma(int R, int64_t tokens, int64_t row_bytes, uint32_t piece_bytes, int pieces,
                  const unsigned char* __restrict__ x, unsigned char* __restrict__ recv_x,
                  int64_t recv_capacity, const int32_t* __restrict__ send_row, int spr,
                  const float* __restrict__ x_scales, float* __restrict__ recv_scales,
                  int32_t* __restrict__ dev_err) {
  extern __shared__ __align__(128) unsigned char sm_tma[];
  unsigned char* stages = sm_tma;
  int32_t* table = reinterpret_cast<int32_t*>(sm_tma + size_t(kTmaStages) * piece_bytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(table + kTmaChunk * MP_MAX_RANKS);
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int i = 0; i < kTmaStages; ++i) mbar_init(&bars[i], 1);
    mbar_init_fence();
  }
  __syncwarp();

  const int64_t chunks = (tokens + kTmaChunk - 1) / kTmaChunk;
  uint32_t g = 0;  // items this block has processed before the current chunk
  bool failed = false;
  for (int64_t ch = blockIdx.x; ch < chunks; ch += gridDim.x) {
    const int64_t tok0 = ch * kTmaChunk;
    const int nt = int(tokens - tok0 < kTmaChunk ? tokens - tok0 : kTmaChunk);
    for (int i = lane; i < nt * R; i += kWarp) table[i] = __ldg(send_row + tok0 * R + i);
    __syncwarp();
    if (lane == 0 && !failed) {
      const int nitems = nt * pieces;
      auto issue_load = [&](int item) {
        const uint32_t st = (g + uint32_t(item)) % kTmaStages;
        const int t = item / pieces, pc = item - t * pieces;
        const int64_t off = int64_t(pc) * piece_bytes;
        const uint32_t bytes =
            uint32_t(row_bytes - off < piece_bytes ? row_bytes - off : piece_bytes);
        mbar_arrive_expect_tx(&bars[st], bytes);
        bulk_g2s(stages + size_t(st) * piece_bytes, x + (tok0 + t) * row_bytes + off, bytes,
                 &bars[st]);
      };
      const int pro = nitems < kTmaStages ? nitems : kTmaStages;
      for (int i = 0; i < pro; ++i) issue_load(i);
      int issued = pro;  // items whose load is in flight or done
      for (int i = 0; i < nitems; ++i) {
        const uint32_t gi = g + uint32_t(i);
        const uint32_t st = gi % kTmaStages, parity = (gi / kTmaStages) & 1u;
        uint32_t spins = 0;
        bool ok = true;
        while (!mbar_try_wait(&bars[st], parity)) {
          if (++spins > kSpinLimit) { ok = false; break; }
        }
        if (!ok) {
          // give up: report, then wait (bounded) for this block's loads in flight
          failed = true;
          raise_error(dev_err, MP_ERR_TIMEOUT);
          for (int k = i + 1; k < issued; ++k) {
            const uint32_t gk = g + uint32_t(k);
            uint32_t n = 0;
            while (!mbar_try_wait(&bars[gk % kTmaStages], (gk / kTmaStages) & 1u) &&
                   ++n < kSpinLimit) {
            }
          }
          break;
        }
        const int t = i / pieces, pc = i - t * pieces;
        const int64_t off = int64_t(pc) * piece_bytes;
        const uint32_t bytes =
            uint32_t(row_bytes - off < piece_bytes ? row_bytes - off : piece_bytes);
        const unsigned char* src = stages + size_t(st) * piece_bytes;
        for (int d = 0; d < R; ++d) {
          const int row = table[t * R + d];
          if (row >= 0 && int64_t(row) < recv_capacity)
            bulk_s2g(recv_x + int64_t(row) * row_bytes + off, src, bytes);
        }
        bulk_commit();
        const int j = i - kTmaLag;  // refill the stage of item j with item j + NS
        if (j >= 0 && j + kTmaStages < nitems) {
          bulk_wait_read<kTmaLag>();
          issue_load(j + kTmaStages);
          ++issued;
        }
      }
      bulk_wait_read<0>();  // every stage free again before the next chunk
      g += uint32_t(nitems);
    }
    __syncwarp();
    if (spr > 0) {  // e4m3 scales travel with the rows (plain copies by the warp)
      for (int t = 0; t < nt; ++t)
        for (int d = 0; d < R; ++d) {
          const int row = table[t * R + d];
          if (row >= 0 && int64_t(row) < recv_capacity)
            for (int c = lane; c < spr; c += kWarp)
              recv_scales[int64_t(row) * spr + c] = __ldg(x_scales + (tok0 + t) * spr + c);
        }
    }
    __syncwarp();
  }
  if (lane == 0) bulk_wait_all();
}

// ---------------------------------------------------------------------------
// Row copies with in-kernel quantisation.  Formats (FMT):
//  kQE4M3 -- [EP] (the FP8 commits of "MSCCLPP EP implementation"): E4M3
//    payloads with FP32 scales.  Each 128-channel block of a bf16 row gets
//    scale = amax / 448 (1 when the block is all zero) and codes
//    e4m3_rn_satfinite(x / scale).
//  kQMXFP8 -- the same page's later commits: E4M3 with one UE8M0 scale byte
//    per 32 channels, tiny non-zero blocks kept at code zero: code =
//    clamp(floor(log2 amax) - 8 + 127, 0, 254) (0 for an all-zero block),
//    X = 2^(code - 127), element codes e4m3(x / X).
//  kQMXFP4 -- [AGV] (the review note that gathering a list of tensors lets a
//    caller quantise to fp4 before the all-gather), in the same microscaling
//    form with E2M1 elements: code = clamp(floor(log2 amax) - 2 + 127, 0,
//    254), element codes e2m1_rn_satfinite(x / X) (magnitudes 0, 0.5, 1,
//    1.5, 2, 3, 4, 6; sign kept, also on a zero), two per byte with the
//    even channel in the low nibble.
// Dividing by a power of two and multiplying by its (exactly representable)
// reciprocal round the same real number once, so the microscaling formats
// multiply by 2^(127 - code).
//
// Destinations.  Dispatch (GATHER = false): token `tok`'s destinations are
// send_row[tok][d] for d < R, skipped when negative or >= `limit` (the receive
// capacity).  Gather (GATHER = true; [AGV] "Add pynccl all-gatherv and
// reducescatterv"): `limit` = S and logical rank q receives row tok at
// q * S + tok, so one launch quantises each row once and writes codes and
// scales R times.
//
// A lane holds CPL channels (CPL = 8: one 16-byte load; 16: one 32-byte load)
// and stores CPL (FP8) or CPL / 2 (FP4) code bytes per destination;
// kBlock / CPL lanes share a scale.  Each row is read once as bf16 and written
// as 1 (FP8) or 1/2 (FP4) byte per channel per destination.
// ---------------------------------------------------------------------------
enum QuantFormat { kQE4M3 = 0, kQMXFP8 = 1, kQMXFP4 = 2 };
static_assert(kQE4M3 == MP_Q_E4M3 && kQMXFP8 == MP_Q_MXFP8 && kQMXFP4 == MP_Q_MXFP4,
              "the C ABI's format codes are the kernels' format numbers");

__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Eight E2M1 codes in one 32-bit word, channel c[2b] in the low nibble and
// c[2b+1] in the high nibble of byte b: four pair conversions packed by one
// vector move.  A negative value that rounds to zero comes out +0 here;
// e2m1_signs puts the sign bits back.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float c0, float c1, float c2, float c3, float c4,
                                               float c5, float c6, float c7) {
  uint32_t r;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(r)
      : "f"(c0), "f"(c1), "f"(c2), "f"(c3), "f"(c4), "f"(c5), "f"(c6), "f"(c7));
  return r;
}

// The sign bits of eight E2M1 codes (one 32-bit word, channel 2b in the low
// nibble of byte b and channel 2b+1 in its high nibble) from the four bf16
// words of those channels (channel 2b in bits 0-15 of w[b], 2b+1 in bits
// 16-31): the bf16 sign bits 15 and 31 of w[b] become bits 3 and 7 of byte b.
// x / X has the sign of x for every finite x (X > 0), so every code, a zero
// included, keeps its input's sign.  Byte permutes gather the four words'
// high and low middle bytes, which hold those sign bits as their bit 7.
__device__ __forceinline__ uint32_t e2m1_signs(uint32_t w0, uint32_t w1, uint32_t w2,
                                               uint32_t w3) {
  const uint32_t hi = __byte_perm(__byte_perm(w0, w1, 0x0073), __byte_perm(w2, w3, 0x0073),
                                  0x5410);  // byte b = byte 3 of w[b]
  const uint32_t lo = __byte_perm(__byte_perm(w0, w1, 0x0051), __byte_perm(w2, w3, 0x0051),
                                  0x5410);  // byte b = byte 1 of w[b]
  return (hi & 0x80808080u) | ((lo >> 4) & 0x08080808u);
}

__device__ __forceinline__ int floor_log2_pos(float a) {  // a > 0, finite
  const uint32_t u = __float_as_uint(a);
  const int e = int((u >> 23) & 0xffu);
  if (e != 0) return e - 127;
  return (31 - __clz(u & 0x7fffffu)) - 149;  // binary32 subnormal: m * 2^-149
}

template <int NB>
__device__ __forceinline__ void st_codes(unsigned char* p, const uint32_t (&w)[NB]) {
  if constexpr (NB == 8) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]),
                 "r"(w[7])
                 : "memory");
  } else if constexpr (NB == 4) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3])
                 : "memory");
  } else if constexpr (NB == 2) {
    asm volatile("st.global.L1::no_allocate.v2.b32 [%0], {%1,%2};" ::"l"(p), "r"(w[0]), "r"(w[1])
                 : "memory");
  } else {
    static_assert(NB == 1, "4, 8, 16 or 32 code bytes per lane");
    asm volatile("st.global.L1::no_allocate.b32 [%0], %1;" ::"l"(p), "r"(w[0]) : "memory");
  }
}

// One lane vector of CPL bf16 channels (its NW = CPL/2 words in v) to its
// codes q[NB] and its scale (sbits: the fp32 scale's bits, or the UE8M0 code),
// the scale block's kBlock / CPL lanes combining their amax by shuffles: every
// lane of the warp calls it together (valid or not; whole scale blocks are
// valid or not).
template <int CPL, int FMT>
__device__ __forceinline__ void quant_vector(bool valid, const Words<CPL / 2>& v,
                                             uint32_t (&q)[FMT == kQMXFP4 ? CPL / 8 : CPL / 4],
                                             uint32_t& sbits) {
  constexpr bool MX = FMT != kQE4M3;
  constexpr bool FP4 = FMT == kQMXFP4;
  constexpr int kBlock = MX ? 32 : 128;      // channels per scale
  constexpr int kLanes = kBlock / CPL;       // lanes per scale block
  constexpr int kEmax = FP4 ? 2 : 8;         // exponent of the element format's largest normal
  constexpr int NW = CPL / 2;                // 32-bit words of bf16 per lane
  constexpr int NB = FP4 ? CPL / 8 : CPL / 4;  // 32-bit words of codes per lane
  static_assert(kLanes >= 1 && kLanes <= 32, "scale block spans whole lanes");
  float f[CPL];
  float amax = 0.0f;
  uint32_t sgn[FP4 ? NB : 1];  // FP4: the codes' sign bits, from the bf16 inputs
  if (valid) {
#pragma unroll
    for (int j = 0; j < NW; ++j) {
      f[2 * j] = __uint_as_float(v.w[j] << 16);
      f[2 * j + 1] = __uint_as_float(v.w[j] & 0xffff0000u);
    }
    if constexpr (FP4) {
#pragma unroll
      for (int j = 0; j < NB; ++j)
        sgn[j] = e2m1_signs(v.w[4 * j], v.w[4 * j + 1], v.w[4 * j + 2], v.w[4 * j + 3]);
    }
#pragma unroll
    for (int j = 0; j < CPL; ++j) amax = fmaxf(amax, fabsf(f[j]));
  }
#pragma unroll
  for (int o = kLanes / 2; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
  if constexpr (MX) {
    int c = 0;
    if (amax > 0.0f) c = min(254, max(0, floor_log2_pos(amax) - kEmax + 127));
    sbits = uint32_t(c);
    // 2^(127 - c): biased exponent 254 - c, or the subnormal 2^-127 at c = 254
    const float inv = c < 254 ? __uint_as_float(uint32_t(254 - c) << 23)
                              : __uint_as_float(0x00400000u);
    if (valid) {
#pragma unroll
      for (int j = 0; j < NB; ++j) {
        if constexpr (FP4) {  // 8 channels -> 4 bytes
          const float* c8 = f + 8 * j;
          q[j] = sgn[j] |
                 cvt_e2m1x8(__fmul_rn(c8[0], inv), __fmul_rn(c8[1], inv), __fmul_rn(c8[2], inv),
                            __fmul_rn(c8[3], inv), __fmul_rn(c8[4], inv), __fmul_rn(c8[5], inv),
                            __fmul_rn(c8[6], inv), __fmul_rn(c8[7], inv));
        } else {  // 4 channels -> 4 bytes
          const uint32_t lo = cvt_e4m3x2(__fmul_rn(f[4 * j + 1], inv), __fmul_rn(f[4 * j], inv));
          const uint32_t hi =
              cvt_e4m3x2(__fmul_rn(f[4 * j + 3], inv), __fmul_rn(f[4 * j + 2], inv));
          q[j] = lo | (hi << 16);
        }
      }
    }
  } else {
    const float sc = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    sbits = __float_as_uint(sc);
    if (valid) {
      if (MP_QUANT_FAST_DIV && sc >= 0x1p-60f) {
        // x / sc correctly rounded without a division per element (Markstein,
        // "IA-64 and Elementary Functions", the division theorem: with y the
        // correctly rounded 1/sc and q within one ulp of x / sc, the exact
        // remainder r = x - sc*q (one FMA) gives RN(q + r*y) = RN(x / sc)).
        // q0 = x*y is within 1.5 ulp; one correction brings it within one
        // ulp, the second rounds it correctly.  sc >= 2^-60 keeps every
        // remainder that matters for an e4m3 code exactly representable.
        // The corrections turn -0 into +0 (0 - 0 = +0), so the sign of x,
        // which x / sc always has, is put back.
        const float y = __frcp_rn(sc);
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const float a = f[j];
          float qv = __fmul_rn(a, y);
          qv = __fmaf_rn(__fmaf_rn(-sc, qv, a), y, qv);
          f[j] = copysignf(__fmaf_rn(__fmaf_rn(-sc, qv, a), y, qv), a);
        }
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const uint32_t lo = cvt_e4m3x2(f[4 * j + 1], f[4 * j]);
          const uint32_t hi = cvt_e4m3x2(f[4 * j + 3], f[4 * j + 2]);
          q[j] = lo | (hi << 16);
        }
      } else {
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          const uint32_t lo = cvt_e4m3x2(__fdiv_rn(f[4 * j + 1], sc), __fdiv_rn(f[4 * j], sc));
          const uint32_t hi = cvt_e4m3x2(__fdiv_rn(f[4 * j + 3], sc), __fdiv_rn(f[4 * j + 2], sc));
          q[j] = lo | (hi << 16);
        }
      }
    }
  }
}

template <int CPL, int U, int FMT, bool GATHER>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_quant_rows(int R, int64_t tokens, int H, const uint16_t* __restrict__ x,
                unsigned char* __restrict__ out, void* __restrict__ out_scales, int64_t limit,
                const int32_t* __restrict__ send_row) {
  constexpr bool MX = FMT != kQE4M3;
  constexpr bool FP4 = FMT == kQMXFP4;
  constexpr int kBlock = MX ? 32 : 128;      // channels per scale
  constexpr int kLanes = kBlock / CPL;       // lanes per scale block
  constexpr int NW = CPL / 2;                // 32-bit words of bf16 per lane
  constexpr int NB = FP4 ? CPL / 8 : CPL / 4;  // 32-bit words of codes per lane
  constexpr int kCodeBytes = NB * 4;
  static_assert(kLanes >= 1 && kLanes <= 32, "scale block spans whole lanes");
  // launched as the low-latency sort's programmatic dependent, the blocks start
  // while the sort runs and wait here for its slot rows (a no-op otherwise)
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t vpr = H / CPL;  // lane vectors per row
  const int64_t row_bytes = FP4 ? H / 2 : H;
  const int nb = H / kBlock;    // scales per row
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * kWarpsPerBlock;
  const Words<NW>* xv = reinterpret_cast<const Words<NW>*>(x);
  for (int64_t unit = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); unit < units;
       unit += nw) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    int64_t my;
    unsigned vm;
    if constexpr (GATHER) {
      my = int64_t(lane) * limit + tok;
      vm = R >= 32 ? kFull : ((1u << R) - 1u);
    } else {
      const int r = lane < R ? __ldg(send_row + tok * R + lane) : -1;
      my = r;
      vm = __ballot_sync(kFull, r >= 0 && int64_t(r) < limit);
      if (vm == 0) continue;
    }
    const int64_t i0 = slab * slab_vec + lane;
    uint32_t q[U][NB];
    uint32_t sbits[U];  // fp32 scale bits, or the UE8M0 code
    Words<NW> v[U];     // every unit's loads first, then the arithmetic
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = i0 + u * kWarp;
      if (i < vpr) {
        if constexpr (NW == 16) {  // 32 channels: two 32-byte loads
          const Words<8>* p8 = reinterpret_cast<const Words<8>*>(x) + 2 * (tok * vpr + i);
          const Words<8> a = ld_stream_w<8>(p8), b = ld_stream_w<8>(p8 + 1);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            v[u].w[j] = a.w[j];
            v[u].w[8 + j] = b.w[j];
          }
        } else {
          v[u] = ld_stream_w<NW>(xv + tok * vpr + i);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)  // (whole scale blocks are valid or not: H % kBlock == 0)
      quant_vector<CPL, FMT>(i0 + u * kWarp < vpr, v[u], q[u], sbits[u]);
    while (vm) {
      const int d = __ffs(vm) - 1;
      vm &= vm - 1;
      const int64_t row = GATHER ? int64_t(d) * limit + tok : __shfl_sync(kFull, my, d);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + u * kWarp;
        if (i < vpr) {
          st_codes<NB>(out + row * row_bytes + i * kCodeBytes, q[u]);
          if ((lane & (kLanes - 1)) == 0) {
            if constexpr (MX)
              static_cast<unsigned char*>(out_scales)[row * nb + i / kLanes] = uint8_t(sbits[u]);
            else
              static_cast<uint32_t*>(out_scales)[row * nb + i / kLanes] = sbits[u];
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Combine (same page: intranode_combine takes the dispatched rows back to
// their tokens).  out[s][t] = bf16_rn( sum_{d ascending} float(y[send_row[s][t][d]]) )
// from +0.0f.  Up to RB source rows are loaded at once (memory-level
// parallelism) and then added strictly in ascending d.
// ---------------------------------------------------------------------------
// With a weight array (the low-latency combine) the R "ranks" are the K top-k
// slots of the token and each row is scaled by its slot's weight first.
template <int NW, int U, int RB, bool WEIGHTED>
__global__ void __launch_bounds__(kCopyThreads, MP_COMBINE_MINB)
mp_k_combine(int R, int64_t tokens, int64_t vpr, const Words<NW>* __restrict__ y, int64_t y_rows,
             const int32_t* __restrict__ send_row, const float* __restrict__ weights,
             Words<NW>* __restrict__ out, int32_t* __restrict__ dev_err) {
  // launched with programmatic stream serialization: the blocks may be staged
  // while the kernel before it (e.g. the row copy producing y) finishes
  pdl_wait_prior_grid();
  const int lane = threadIdx.x & 31;
  const int64_t slab_vec = int64_t(kWarp) * U;
  const int64_t slabs = (vpr + slab_vec - 1) / slab_vec;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * kWarpsPerBlock;
  for (int64_t unit = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5); unit < units;
       unit += nw) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    int my = lane < R ? __ldg(send_row + tok * R + lane) : -1;
    if (my >= 0 && int64_t(my) >= y_rows) {
      if (slab == 0) raise_error(dev_err, MP_ERR_CAPACITY);
      my = -1;
    }
    float myw = 0.0f;
    if (WEIGHTED && lane < R) myw = __ldg(weights + tok * R + lane);
    unsigned vm = __ballot_sync(kFull, my >= 0);
    const int64_t i0 = slab * slab_vec + lane;
    float acc[U][2 * NW];
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int j = 0; j < 2 * NW; ++j) acc[u][j] = 0.0f;
    while (vm) {
      int64_t rows[RB];
      float wts[RB];
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        rows[j] = -1;
        wts[j] = 0.0f;
        if (vm) {
          const int d = __ffs(vm) - 1;
          vm &= vm - 1;
          rows[j] = __shfl_sync(kFull, my, d);
          if (WEIGHTED) wts[j] = __shfl_sync(kFull, myw, d);
        }
      }
      Words<NW> v[RB][U];
#pragma unroll
      for (int j = 0; j < RB; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (rows[j] >= 0 && i0 + u * kWarp < vpr)
            v[j][u] = ld_stream_w<NW>(y + rows[j] * vpr + i0 + u * kWarp);
#pragma unroll
      for (int j = 0; j < RB; ++j)
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (rows[j] >= 0 && i0 + u * kWarp < vpr) {
            if (WEIGHTED) add_bf16_weighted<NW>(acc[u], v[j][u], wts[j]);
            else add_bf16<NW>(acc[u], v[j][u]);
          }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kWarp < vpr)
        st_stream_w<NW>(out + tok * vpr + i0 + u * kWarp, pack_bf16<NW>(acc[u]));
  }
}

// ---------------------------------------------------------------------------
// Reduce-scatterv ("Add pynccl all-gatherv and reducescatterv",
// vllm-project/vllm PR #20154: one reduce per root over its slice of every
// rank's input).  With all R inputs in one memory the R reduces are one
// element-wise fp32 sum over q ascending, rounded once; rank r's shard is a
// row range of the output.
// ---------------------------------------------------------------------------
template <int NW>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_rsv(int R, int64_t nvec, const Words<NW>* __restrict__ in, Words<NW>* __restrict__ out) {
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads;
  for (int64_t i = int64_t(blockIdx.x) * kCopyThreads + threadIdx.x; i < nvec; i += stride) {
    float acc[2 * NW];
#pragma unroll
    for (int j = 0; j < 2 * NW; ++j) acc[j] = 0.0f;
    for (int q0 = 0; q0 < R; q0 += 8) {
      Words<NW> v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (q0 + j < R) v[j] = ld_stream_w<NW>(in + int64_t(q0 + j) * nvec + i);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (q0 + j < R) add_bf16<NW>(acc, v[j]);
    }
    st_stream_w<NW>(out + i, pack_bf16<NW>(acc));
  }
}

// ---------------------------------------------------------------------------
// All-gatherv (same page: one broadcast per root of its rows into every
// rank's output).  Every logical rank's copy is the concatenated shards, so
// each vector is read once and written R times.
// ---------------------------------------------------------------------------
template <int NW, int U>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_agv(int R, int64_t nvec, const Words<NW>* __restrict__ in, Words<NW>* __restrict__ out) {
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads * U;
  for (int64_t i0 = int64_t(blockIdx.x) * kCopyThreads * U + threadIdx.x; i0 < nvec;
       i0 += stride) {
    Words<NW> v[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (i0 + u * kCopyThreads < nvec) v[u] = ld_stream_w<NW>(in + i0 + u * kCopyThreads);
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kCopyThreads < nvec)
          st_stream_w<NW>(out + int64_t(q) * nvec + i0 + u * kCopyThreads, v[u]);
  }
}

// ---------------------------------------------------------------------------
// Multi-tensor all-gatherv (same page: all-gathering a list of tensors lets
// quantised data and its scales travel together).  Up to MP_MAX_TENSORS
// tensors share the per-rank row counts; one launch walks the concatenation
// of their 16-byte vectors, each read once and written R times.
// ---------------------------------------------------------------------------
struct AgvList {
  const void* in[MP_MAX_TENSORS];
  void* out[MP_MAX_TENSORS];
  int64_t nvec[MP_MAX_TENSORS];   // vectors of one gathered copy of tensor j
  int64_t first[MP_MAX_TENSORS];  // index of tensor j's first vector in the walk
  int n;
};

// Multi-tensor all-gatherv: the tensors' vectors are walked as one sequence;
// each thread reads U vectors once and stores each of them R times, like
// mp_k_agv (one short block per kCopyThreads * U vectors).
template <int NW, int U>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_agv_multi(int R, int64_t total, AgvList l) {
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads * U;
  for (int64_t i0 = int64_t(blockIdx.x) * kCopyThreads * U + threadIdx.x; i0 < total;
       i0 += stride) {
    Words<NW> v[U];
    int jj[U];
    int64_t ii[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t g = i0 + u * kCopyThreads;
      jj[u] = -1;
      ii[u] = 0;
      if (g < total) {
        int j = 0;
        while (j + 1 < l.n && g >= l.first[j + 1]) ++j;
        jj[u] = j;
        ii[u] = g - l.first[j];
        v[u] = ld_stream_w<NW>(static_cast<const Words<NW>*>(l.in[j]) + ii[u]);
      }
    }
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (jj[u] >= 0)
          st_stream_w<NW>(static_cast<Words<NW>*>(l.out[jj[u]]) + int64_t(q) * l.nvec[jj[u]] +
                              ii[u],
                          v[u]);
  }
}

// ---------------------------------------------------------------------------
// Launchers: a persistent grid of (SMs x resident blocks) blocks, trimmed to
// the work available; 32-byte vectors when sizes and pointers allow.
// ---------------------------------------------------------------------------
// Launch with programmatic stream serialization: the kernel's blocks may start
// before the kernel ahead of it on the stream has finished, once that kernel's
// blocks have all triggered (pdl_launch_dependents) or exited; the kernel
// itself must call pdl_wait_prior_grid before it touches that kernel's output.
template <typename... KArgs, typename... Args>
static cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, cudaStream_t stream,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kCopyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Any kernel launched with programmatic stream serialization (block size and
// shared memory given): it may start before the kernel ahead of it ends, so it
// must call pdl_wait_prior_grid() before touching memory that kernel writes.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename Kernel>
static int resident_blocks(Kernel k) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kCopyThreads, 0) != cudaSuccess || n < 1)
    n = 1;
  return n;
}

static unsigned grid_for(int per_sm, int64_t items_per_block, int64_t items) {
  const int64_t full = int64_t(sm_count()) * per_sm;
  const int64_t need = (items + items_per_block - 1) / items_per_block;
  return unsigned(need < 1 ? 1 : (need < full ? need : full));
}

// Write-dominated kernels (dispatch copy, reduce-scatterv, all-gatherv) launch
// one block per kWarpsPerBlock units instead of a persistent grid: measured on
// GB300, letting the block scheduler hand out short blocks balances the SMs
// better and reaches 6.8-7.1 TB/s where a persistent grid stayed at ~6 TB/s.
static unsigned grid_full(int64_t items_per_block, int64_t items) {
  const int64_t need = (items + items_per_block - 1) / items_per_block;
  return unsigned(need < 1 ? 1 : (need < 0x7fffffff ? need : 0x7fffffff));
}

static bool aligned(const void* p, int bytes) {
  return (reinterpret_cast<uintptr_t>(p) % uintptr_t(bytes)) == 0;
}

template <int NW, int U>
static cudaError_t dispatch_copy_nw(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                    void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                    int spr, const float* x_scales, float* recv_scales,
                                    cudaStream_t stream) {
  const int64_t vpr = row_bytes / (4 * NW);
  const int64_t slabs = (vpr + kWarp * U - 1) / (kWarp * U);
  const unsigned grid = grid_full(kWarpsPerBlock, tokens * slabs);
  return launch_kernel(mp_k_dispatch<NW, U>, dim3(grid), dim3(kCopyThreads), 0, stream, R, tokens,
                       vpr, static_cast<const Words<NW>*>(x), static_cast<Words<NW>*>(recv_x),
                       recv_capacity, send_row, spr, x_scales, recv_scales);
}

static cudaError_t dispatch_copy_tma(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                     void* recv_x, int64_t recv_capacity,
                                     const int32_t* send_row, int spr, const float* x_scales,
                                     float* recv_scales, int32_t* dev_err, cudaStream_t stream) {
  const uint32_t piece = uint32_t(row_bytes < kTmaPiece ? row_bytes : kTmaPiece);
  const int pieces = int((row_bytes + piece - 1) / piece);
  const size_t smem = tma_smem_bytes(piece);
  static thread_local int configured[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (configured[dev] < int(smem)) {
    cudaError_t e = cudaFuncSetAttribute(mp_k_dispatch_tma,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = int(smem);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mp_k_dispatch_tma, kWarp, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t chunks = (tokens + kTmaChunk - 1) / kTmaChunk;
  const unsigned grid = MP_TMA_GRID_FULL ? grid_full(1, chunks) : grid_for(per_sm, 1, chunks);
  return launch_kernel(mp_k_dispatch_tma, dim3(grid), dim3(kWarp), smem, stream, R, tokens,
                       row_bytes, piece, pieces, static_cast<const unsigned char*>(x),
                       static_cast<unsigned char*>(recv_x), recv_capacity, send_row, spr, x_scales,
                       recv_scales, dev_err);
}

cudaError_t launch_dispatch_copy(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                 void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                 int scales_per_row, const float* x_scales, float* recv_scales,
                                 cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  if (MP_SMALL_DISPATCH && MP_DISPATCH_NW == 8 && row_bytes % 32 == 0 && aligned(x, 32) &&
      aligned(recv_x, 32)) {
    const int64_t slabs = (row_bytes / 32 + kWarp * MP_DISPATCH_U - 1) / (kWarp * MP_DISPATCH_U);
    if (tokens * slabs < int64_t(sm_count()) * (2048 / kWarp))
      return dispatch_copy_nw<8, 1>(R, tokens, row_bytes, x, recv_x, recv_capacity, send_row,
                                    scales_per_row, x_scales, recv_scales, stream);
  }
  if (MP_DISPATCH_NW == 8 && row_bytes % 32 == 0 && aligned(x, 32) && aligned(recv_x, 32))
    return dispatch_copy_nw<MP_DISPATCH_NW, MP_DISPATCH_U>(R, tokens, row_bytes, x, recv_x,
                                                           recv_capacity, send_row,
                                                           scales_per_row, x_scales, recv_scales,
                                                           stream);
  return dispatch_copy_nw<4, 2 * MP_DISPATCH_U>(R, tokens, row_bytes, x, recv_x, recv_capacity,
                                                send_row, scales_per_row, x_scales, recv_scales,
                                                stream);
}

cudaError_t launch_dispatch_bulk(int R, int64_t tokens, int64_t row_bytes, const void* x,
                                 void* recv_x, int64_t recv_capacity, const int32_t* send_row,
                                 int scales_per_row, const float* x_scales, float* recv_scales,
                                 int32_t* dev_err, cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  return dispatch_copy_tma(R, tokens, row_bytes, x, recv_x, recv_capacity, send_row,
                           scales_per_row, x_scales, recv_scales, dev_err, stream);
}

template <int NW, int U>
static cudaError_t dispatch_after_offsets_nw(int R, int N, int K, int El, int64_t row_bytes,
                                             const void* x, void* recv_x, int64_t recv_capacity,
                                             const int32_t* send_row, int spr,
                                             const float* x_scales, float* recv_scales,
                                             const int32_t* topk_idx, const float* topk_weights,
                                             int32_t* recv_src_rank, int32_t* recv_src_idx,
                                             int32_t* recv_topk_idx, float* recv_topk_weights,
                                             cudaStream_t stream) {
  const int64_t tokens = int64_t(R) * N;
  const int64_t vpr = row_bytes / (4 * NW);
  const int64_t slabs = (vpr + kWarp * U - 1) / (kWarp * U);
  return launch_dependent(mp_k_dispatch_after_offsets<NW, U>,
                          dim3(grid_full(kWarpsPerBlock, tokens * slabs)), stream, R, N, K, El,
                          tokens, vpr, static_cast<const Words<NW>*>(x),
                          static_cast<Words<NW>*>(recv_x), recv_capacity, send_row, spr, x_scales,
                          recv_scales, topk_idx, topk_weights, recv_src_rank, recv_src_idx,
                          recv_topk_idx, recv_topk_weights);
}

cudaError_t launch_dispatch_after_offsets(int R, int N, int K, int E, int64_t row_bytes,
                                          const void* x, void* recv_x, int64_t recv_capacity,
                                          const int32_t* send_row, int scales_per_row,
                                          const float* x_scales, float* recv_scales,
                                          const int32_t* topk_idx, const float* topk_weights,
                                          int32_t* recv_src_rank, int32_t* recv_src_idx,
                                          int32_t* recv_topk_idx, float* recv_topk_weights,
                                          cudaStream_t stream) {
  const int64_t tokens = int64_t(R) * N;
  if (tokens == 0) return cudaSuccess;
  const int El = E / R;
  // the shapes of launch_dispatch_copy: 1 vector per lane and unit for small
  // problems (more units in flight), 4 otherwise; 16-byte vectors when the row
  // size or the pointers do not allow 32
  if (row_bytes % 32 == 0 && aligned(x, 32) && aligned(recv_x, 32)) {
    const int64_t slabs = (row_bytes / 32 + kWarp * MP_DISPATCH_U - 1) / (kWarp * MP_DISPATCH_U);
    if (MP_SMALL_DISPATCH && tokens * slabs < int64_t(sm_count()) * (2048 / kWarp))
      return dispatch_after_offsets_nw<8, 1>(R, N, K, El, row_bytes, x, recv_x, recv_capacity,
                                             send_row, scales_per_row, x_scales, recv_scales,
                                             topk_idx, topk_weights, recv_src_rank, recv_src_idx,
                                             recv_topk_idx, recv_topk_weights, stream);
    return dispatch_after_offsets_nw<8, MP_DISPATCH_U>(
        R, N, K, El, row_bytes, x, recv_x, recv_capacity, send_row, scales_per_row, x_scales,
        recv_scales, topk_idx, topk_weights, recv_src_rank, recv_src_idx, recv_topk_idx,
        recv_topk_weights, stream);
  }
  return dispatch_after_offsets_nw<4, 2 * MP_DISPATCH_U>(
      R, N, K, El, row_bytes, x, recv_x, recv_capacity, send_row, scales_per_row, x_scales,
      recv_scales, topk_idx, topk_weights, recv_src_rank, recv_src_idx, recv_topk_idx,
      recv_topk_weights, stream);
}

// Quantising copies.  Launch shapes measured on GB300 (dsv3 dispatch rows,
// R=8, N=4096, H=7168; rsv all-gatherv, R=8, S=44,383, H=4096):
//  - 16 channels per lane (32-byte loads, 16-byte code stores) beat 8 by
//    10-15%; a source that is not 32-byte aligned takes the 8-channel form;
//  - 2 vectors per lane and unit, except 1 for the e4m3 gather (276 vs
//    285 us);
//  - one short block per kWarpsPerBlock units (the write-heavy policy above)
//    for the FP8 dispatches (MXFP8 260 vs 296 us; e4m3 269 vs 290 us) and
//    every gather (MXFP4 173 vs 199 us, the FP8 ones 276-285 vs 321 us), but a
//    persistent grid for the MXFP4 dispatch, whose reads are a larger share of
//    its traffic (184 vs 191 us);
//  - the e4m3 quantiser's reciprocal-and-two-FMA division (MP_QUANT_FAST_DIV)
//    against a division per element: 269 vs 278 us for the dispatch (the best
//    launch shape of each);
//  - for MXFP4, 2 vectors per lane (190 us) beat 1 (211) and 4 (202).
// MP_QUANT_CPL = 8, MP_QUANT_U_FP4 and MP_QUANT_PERSISTENT_MASK (bit
// FMT + (GATHER ? 3 : 0) set = persistent grid) reproduce the other shapes.
#ifndef MP_QUANT_CPL
#define MP_QUANT_CPL 16
#endif
#ifndef MP_QUANT_PERSISTENT_MASK
#define MP_QUANT_PERSISTENT_MASK 4
#endif
#ifndef MP_QUANT_U_FP4
#define MP_QUANT_U_FP4 2
#endif


template <int CPL, int U, int FMT, bool GATHER>
static cudaError_t quant_rows(int R, int64_t tokens, int H, const void* x, void* out,
                              void* out_scales, int64_t limit, const int32_t* send_row,
                              bool dependent, cudaStream_t stream) {
  auto kernel = mp_k_quant_rows<CPL, U, FMT, GATHER>;
  static const int per_sm = resident_blocks(kernel);
  const int64_t vpr = H / CPL;
  const int64_t slabs = (vpr + kWarp * U - 1) / (kWarp * U);
  constexpr bool persistent = (MP_QUANT_PERSISTENT_MASK >> (FMT + (GATHER ? 3 : 0))) & 1;
  const unsigned grid = persistent ? grid_for(per_sm, kWarpsPerBlock, tokens * slabs)
                                   : grid_full(kWarpsPerBlock, tokens * slabs);
  if (dependent)
    return launch_dependent(kernel, dim3(grid), stream, R, tokens, H,
                            static_cast<const uint16_t*>(x), static_cast<unsigned char*>(out),
                            out_scales, limit, send_row);
  return launch_kernel(kernel, dim3(grid), dim3(kCopyThreads), 0, stream, R, tokens, H,
                       static_cast<const uint16_t*>(x), static_cast<unsigned char*>(out),
                       out_scales, limit, send_row);
}

template <int FMT, bool GATHER>
static cudaError_t quant_rows_any(int R, int64_t tokens, int H, const void* x, void* out,
                                  void* out_scales, int64_t limit, const int32_t* send_row,
                                  cudaStream_t stream, bool dependent = false) {
  if (tokens == 0) return cudaSuccess;
  constexpr int U = (GATHER && FMT == kQE4M3) ? 1 : (FMT == kQMXFP4 ? MP_QUANT_U_FP4 : 2);
  if constexpr ((MP_QUANT_CPL32_MASK >> (FMT + (GATHER ? 3 : 0))) & 1) {
    // 32 channels per lane: 32-byte FP8 code stores need a 32-byte aligned output
    if (aligned(x, 32) && (FMT == kQMXFP4 || aligned(out, 32)))
      return quant_rows<32, 1, FMT, GATHER>(R, tokens, H, x, out, out_scales, limit, send_row,
                                            dependent, stream);
  }
  if constexpr (MP_QUANT_CPL == 16) {
    if (aligned(x, 32))
      return quant_rows<16, U, FMT, GATHER>(R, tokens, H, x, out, out_scales, limit, send_row,
                                            dependent, stream);
  }
  return quant_rows<8, 2 * U, FMT, GATHER>(R, tokens, H, x, out, out_scales, limit, send_row,
                                           dependent, stream);
}

cudaError_t launch_dispatch_quant(int R, int64_t tokens, int H, const void* x, void* recv_x,
                                  void* recv_scales, int fmt, int64_t recv_capacity,
                                  const int32_t* send_row, cudaStream_t stream, bool dependent) {
  switch (fmt) {
    case kQE4M3:
      return quant_rows_any<kQE4M3, false>(R, tokens, H, x, recv_x, recv_scales, recv_capacity,
                                           send_row, stream, dependent);
    case kQMXFP8:
      return quant_rows_any<kQMXFP8, false>(R, tokens, H, x, recv_x, recv_scales, recv_capacity,
                                            send_row, stream, dependent);
    case kQMXFP4:
      return quant_rows_any<kQMXFP4, false>(R, tokens, H, x, recv_x, recv_scales, recv_capacity,
                                            send_row, stream, dependent);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_allgatherv_quant(int R, int64_t S, int H, const void* in, void* out,
                                    void* out_scales, int fmt, cudaStream_t stream) {
  switch (fmt) {
    case kQE4M3:
      return quant_rows_any<kQE4M3, true>(R, S, H, in, out, out_scales, S, nullptr, stream);
    case kQMXFP8:
      return quant_rows_any<kQMXFP8, true>(R, S, H, in, out, out_scales, S, nullptr, stream);
    case kQMXFP4:
      return quant_rows_any<kQMXFP4, true>(R, S, H, in, out, out_scales, S, nullptr, stream);
  }
  return cudaErrorInvalidValue;
}

template <int NW, int U, int RB, bool W>
static cudaError_t combine_nw(int R, int64_t tokens, int H, const void* y, int64_t y_rows,
                              const int32_t* send_row, const float* weights, void* out,
                              int32_t* dev_err, cudaStream_t stream) {
  static const int per_sm = resident_blocks(mp_k_combine<NW, U, RB, W>);
  const int64_t vpr = int64_t(H) * 2 / (4 * NW);
  const int64_t slabs = (vpr + kWarp * U - 1) / (kWarp * U);
  const unsigned grid = grid_for(per_sm, kWarpsPerBlock, tokens * slabs);
  return launch_dependent(mp_k_combine<NW, U, RB, W>, dim3(grid), stream, R, tokens, vpr,
                          static_cast<const Words<NW>*>(y), y_rows, send_row, weights,
                          static_cast<Words<NW>*>(out), dev_err);
}

template <bool W>
static cudaError_t combine_any(int R, int64_t tokens, int H, const void* y, int64_t y_rows,
                               const int32_t* send_row, const float* weights, void* out,
                               int32_t* dev_err, cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  constexpr int NW = W ? MP_COMBINE_W_NW : MP_COMBINE_NW;
  constexpr int U = W ? MP_COMBINE_W_U : MP_COMBINE_U;
  constexpr int RB = W ? MP_COMBINE_W_RB : MP_COMBINE_RB;
  if (NW == 8 && (int64_t(H) * 2) % 32 == 0 && aligned(y, 32) && aligned(out, 32))
    return combine_nw<8, U, RB, W>(R, tokens, H, y, y_rows, send_row, weights, out, dev_err,
                                   stream);
  return combine_nw<4, (NW == 8 ? 2 * U : U), RB, W>(R, tokens, H, y, y_rows, send_row, weights,
                                                     out, dev_err, stream);
}

cudaError_t launch_combine(int R, int64_t tokens, int H, const void* y, int64_t y_rows,
                           const int32_t* send_row, void* out, int32_t* dev_err,
                           cudaStream_t stream) {
  return combine_any<false>(R, tokens, H, y, y_rows, send_row, nullptr, out, dev_err, stream);
}

cudaError_t launch_combine_weighted(int K, int64_t tokens, int H, const void* y, int64_t y_rows,
                                    const int32_t* slot_row, const float* weights, void* out,
                                    int32_t* dev_err, cudaStream_t stream) {
  return combine_any<true>(K, tokens, H, y, y_rows, slot_row, weights, out, dev_err, stream);
}

template <int NW>
static cudaError_t rsv_nw(int R, int64_t bytes_per_rank, const void* in, void* out,
                          cudaStream_t stream) {
  const int64_t nvec = bytes_per_rank / (4 * NW);
  const unsigned grid = grid_full(kCopyThreads, nvec);
  return launch_kernel(mp_k_rsv<NW>, dim3(grid), dim3(kCopyThreads), 0, stream, R, nvec,
                       static_cast<const Words<NW>*>(in), static_cast<Words<NW>*>(out));
}

cudaError_t launch_reducescatterv(int R, int64_t S, int H, const void* in, void* out,
                                  cudaStream_t stream) {
  const int64_t bytes = S * H * 2;
  if (bytes == 0) return cudaSuccess;
  if (bytes % 32 == 0 && aligned(in, 32) && aligned(out, 32))
    return rsv_nw<8>(R, bytes, in, out, stream);
  return rsv_nw<4>(R, bytes, in, out, stream);
}

template <int NW, int U>
static cudaError_t agv_nw(int R, int64_t bytes, const void* in, void* out, cudaStream_t stream) {
  const int64_t nvec = bytes / (4 * NW);
  const unsigned grid = grid_full(int64_t(kCopyThreads) * U, nvec);
  return launch_kernel(mp_k_agv<NW, U>, dim3(grid), dim3(kCopyThreads), 0, stream, R, nvec,
                       static_cast<const Words<NW>*>(in), static_cast<Words<NW>*>(out));
}

cudaError_t launch_allgatherv(int R, int64_t S, int64_t row_bytes, const void* in, void* out,
                              cudaStream_t stream) {
  const int64_t bytes = S * row_bytes;
  if (bytes == 0) return cudaSuccess;
  if (bytes % 32 == 0 && aligned(in, 32) && aligned(out, 32))
    return agv_nw<8, 2>(R, bytes, in, out, stream);
  return agv_nw<4, 4>(R, bytes, in, out, stream);
}

}  // namespace mp

namespace mp {

template <int NW, int U>
static cudaError_t agv_multi_nw(int R, int n, const int64_t* row_bytes, int64_t S,
                                const void* const* in, void* const* out, cudaStream_t stream) {
  AgvList l{};
  l.n = n;
  int64_t total = 0;
  for (int j = 0; j < n; ++j) {
    l.in[j] = in[j];
    l.out[j] = out[j];
    l.nvec[j] = S * row_bytes[j] / (4 * NW);
    l.first[j] = total;
    total += l.nvec[j];
  }
  if (total == 0) return cudaSuccess;
  const unsigned grid = grid_full(int64_t(kCopyThreads) * U, total);
  return launch_kernel(mp_k_agv_multi<NW, U>, dim3(grid), dim3(kCopyThreads), 0, stream, R, total,
                       l);
}

cudaError_t launch_allgatherv_multi(int R, int n, const int64_t* row_bytes, int64_t S,
                                    const void* const* in, void* const* out,
                                    cudaStream_t stream) {
  bool wide = true;  // 32-byte vectors when every tensor allows them
  for (int j = 0; j < n; ++j)
    wide = wide && (S * row_bytes[j]) % 32 == 0 && aligned(in[j], 32) && aligned(out[j], 32);
  if (wide) return agv_multi_nw<8, 2>(R, n, row_bytes, S, in, out, stream);
  return agv_multi_nw<4, 4>(R, n, row_bytes, S, in, out, stream);
}

}  // namespace mp

namespace mp {

// Combined top-k weights ("MSCCLPP EP implementation": intranode_combine returns
// the combined weights with the rows): one thread per (token, slot), fp32 sum
// over the token's destinations in ascending order from +0.0f.
__global__ void __launch_bounds__(kCopyThreads)
mp_k_combine_weights(int R, int64_t tokens, int K, const float* __restrict__ w, int64_t rows,
                     const int32_t* __restrict__ send_row, float* __restrict__ out,
                     int32_t* __restrict__ dev_err) {
  const int64_t n = tokens * K;
  const int64_t stride = int64_t(gridDim.x) * kCopyThreads;
  for (int64_t i = int64_t(blockIdx.x) * kCopyThreads + threadIdx.x; i < n; i += stride) {
    const int64_t tok = i / K;
    const int k = int(i - tok * K);
    float acc = 0.0f;
    bool bad = false;
    for (int d = 0; d < R; ++d) {
      const int r = __ldg(send_row + tok * R + d);
      if (r < 0) continue;
      if (int64_t(r) >= rows) { bad = true; continue; }
      acc = __fadd_rn(acc, __ldg(w + int64_t(r) * K + k));
    }
    out[i] = acc;
    if (bad) raise_error(dev_err, MP_ERR_CAPACITY);
  }
}

cudaError_t launch_combine_weights(int R, int64_t tokens, int K, const float* recv_topk_weights,
                                   int64_t recv_rows, const int32_t* send_row, float* combined,
                                   int32_t* dev_err, cudaStream_t stream) {
  const int64_t n = tokens * K;
  if (n == 0) return cudaSuccess;
  static const int per_sm = resident_blocks(mp_k_combine_weights);
  const unsigned grid = grid_for(per_sm, kCopyThreads, n);
  return launch_kernel(mp_k_combine_weights, dim3(grid), dim3(kCopyThreads), 0, stream, R, tokens,
                       K, recv_topk_weights, recv_rows, send_row, combined, dev_err);
}

}  // namespace mp

namespace mp {

// ---------------------------------------------------------------------------
// Low-latency row copy as a programmatic dependent of the LL sort (the second
// kernel of mp_dispatch_ll).  It is launched with programmatic stream
// serialization, so its blocks may start while the sort still runs: each warp
// loads its first slab of a token row (x is an input of the sort's caller,
// complete before the sort started), then waits for the sort grid to finish
// and its writes to be visible (griddepcontrol.wait), then reads the token's
// slot rows and stores.  One 32-byte vector per lane and unit, one short
// block per kWarpsPerBlock units (the small-dispatch shape).
// ---------------------------------------------------------------------------
template <int NW>
__global__ void __launch_bounds__(kCopyThreads)
mp_k_ll_rows_after_sort(int K, int64_t tokens, int64_t vpr, const Words<NW>* __restrict__ x,
                        Words<NW>* __restrict__ recv_x, int64_t recv_capacity,
                        const int32_t* slot_row, int spr, const float* __restrict__ x_scales,
                        float* __restrict__ recv_scales) {
  const int lane = threadIdx.x & 31;
  const int64_t slabs = (vpr + kWarp - 1) / kWarp;
  const int64_t units = tokens * slabs;
  const int64_t nw = int64_t(gridDim.x) * kWarpsPerBlock;
  int64_t unit = int64_t(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
  pdl_launch_dependents();  // the weighted combine after it may stage its blocks
  Words<NW> v;
  if (unit < units) {  // the first unit's vector, before the wait
    const int64_t tok = unit / slabs, i = (unit - tok * slabs) * kWarp + lane;
    if (i < vpr) v = ld_stream_w<NW>(x + tok * vpr + i);
  }
  pdl_wait_prior_grid();
  for (bool first = true; unit < units; unit += nw, first = false) {
    const int64_t tok = unit / slabs;
    const int64_t slab = unit - tok * slabs;
    const int64_t i = slab * kWarp + lane;
    if (!first && i < vpr) v = ld_stream_w<NW>(x + tok * vpr + i);
    // slot_row was written by the sort grid: read through L2, not the read-only path
    const int my = lane < K ? __ldcg(slot_row + tok * K + lane) : -1;
    unsigned vm = __ballot_sync(kFull, my >= 0 && int64_t(my) < recv_capacity);
    while (vm) {
      const int d = __ffs(vm) - 1;
      vm &= vm - 1;
      const int64_t row = __shfl_sync(kFull, my, d);
      if (i < vpr) st_stream_w<NW>(recv_x + row * vpr + i, v);
      if (spr > 0 && slab == 0)
        for (int c = lane; c < spr; c += kWarp)
          recv_scales[row * spr + c] = __ldg(x_scales + tok * spr + c);
    }
  }
}

template <int NW>
static cudaError_t ll_rows_after_sort_nw(int K, int64_t tokens, int64_t row_bytes, const void* x,
                                         void* recv_x, int64_t recv_capacity,
                                         const int32_t* slot_row, int spr, const float* x_scales,
                                         float* recv_scales, cudaStream_t stream) {
  const int64_t vpr = row_bytes / (4 * NW);
  const int64_t slabs = (vpr + kWarp - 1) / kWarp;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_full(kWarpsPerBlock, tokens * slabs));
  cfg.blockDim = dim3(kCopyThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mp_k_ll_rows_after_sort<NW>, K, tokens, vpr,
                            static_cast<const Words<NW>*>(x), static_cast<Words<NW>*>(recv_x),
                            recv_capacity, slot_row, spr, x_scales, recv_scales);
}

cudaError_t launch_ll_rows_after_sort(int K, int64_t tokens, int64_t row_bytes, const void* x,
                                      void* recv_x, int64_t recv_capacity,
                                      const int32_t* slot_row, int scales_per_row,
                                      const float* x_scales, float* recv_scales,
                                      cudaStream_t stream) {
  if (tokens == 0) return cudaSuccess;
  if (row_bytes % 32 == 0 && aligned(x, 32) && aligned(recv_x, 32))
    return ll_rows_after_sort_nw<8>(K, tokens, row_bytes, x, recv_x, recv_capacity, slot_row,
                                    scales_per_row, x_scales, recv_scales, stream);
  return ll_rows_after_sort_nw<4>(K, tokens, row_bytes, x, recv_x, recv_capacity, slot_row,
                                  scales_per_row, x_scales, recv_scales, stream);
}

// ---------------------------------------------------------------------------
// The low-latency dispatch in one kernel for small batches, no block waiting
// for another.  The rows of a bin are ordered by source rank, token and top-k
// slot, which is the entries' flat index i = (s*N + n)*K + k, so entry i goes
// to the bin's first row plus the number of entries j < i in the same bin.
// Block b copies the units [V*b/G, V*(b+1)/G) of the token-major row space
// (V = R*N*vpr units of 16 or 32 bytes; in the quantising mode, QF >= 0, whole
// scale blocks, so that no block shares a scale block with another); for the
// tokens those units belong to it finds the rows itself:
//  1. one pass over all R*N*K ids (they are few: the path is for small
//     batches): per bin, the entries before the block's first entry (lower)
//     and the others (upper), counted in shared memory, and the block's own
//     ids kept;
//  2. the bins' first rows, an exclusive scan of lower + upper over the bins
//     (block 0 writes them out as bin_offsets);
//  3. one warp walks the block's entries in order (lanes of a bin find each
//     other with __match_any_sync) and continues the counts; for the
//     tokens whose first unit is the block's it writes slot_row and
//     recv_src_token, and, at the first entry of a rank s, the counts so far
//     as bin_src_offsets[., s];
//  4. the copy (quantising mode: each lane quantises 16 channels once, with
//     the same device function as the quantising copies, and stores the codes
//     to its token's rows, the scale block's first lane its scale), then the
//     owned tokens' scales.
// The kernel is launched as a programmatic dependent of the kernel before it
// on the stream and waits for that kernel before any memory access.
// The block's part of x is fetched while it counts.  With BULK (rows of at
// least kLLFBulkMinRow bytes) one thread loads it into shared memory with a
// bulk copy at the start, and in step 3 each lane of the walking warp stores
// its entry's piece of the token row with a shared -> global bulk copy (the
// quantising mode stages x the same way when it fits).  Else each
// thread loads its kLLFJ vectors into registers before the counting and
// stores them to the rows of their token (the register loads in flight slow
// the shared-memory adds of step 1, which the bulk load does not: measured
// 5.2 against 3.1 us for step 1 at R=8, N=128, top-8 of 256, H=7168).
// Every block reads all ids, so the launcher takes this path only up to
// kLLFMaxIds ids; the sort + dependent copy pair handles the rest.
// ---------------------------------------------------------------------------
// Launch shape: one block of 1,024 threads per SM (every block counts all ids,
// so fewer blocks count less in all; against two blocks of 512 per SM the step
// at R=8, top-8 of 256, H=7168 took 47.5 / 69.5 / 89.1 vs 47.9 / 71.2 / 91.3 us
// at N = 128 / 192 / 256).
#ifndef MP_LLF_THREADS
#define MP_LLF_THREADS 1024
#endif
#ifndef MP_LLF_BPS
#define MP_LLF_BPS 1
#endif
#ifndef MP_LLF_J
#define MP_LLF_J 3
#endif
#ifndef MP_LLF_MAX_IDS
#define MP_LLF_MAX_IDS 16384
#endif
#ifndef MP_LLF_BULK_MIN_ROW
#define MP_LLF_BULK_MIN_ROW 2048
#endif
constexpr int kLLFThreads = MP_LLF_THREADS;  // threads per block
constexpr int kLLFBlocksPerSM = MP_LLF_BPS;  // blocks per SM
constexpr int kLLFJ = MP_LLF_J;              // vectors per thread in flight (register copy)
constexpr int64_t kLLFMaxIds = MP_LLF_MAX_IDS;
constexpr int64_t kLLFBulkMinRow = MP_LLF_BULK_MIN_ROW;  // row bytes from which BULK is used
constexpr int kLLFMaxBins = 2048;
constexpr size_t kLLFMaxStage = (kLLFBlocksPerSM == 1 ? 192 : 96) * 1024;  // a block's part of x
constexpr size_t kLLFMaxTable = 32 * 1024;  // shared-memory bytes of counts and rows

// BULK staging of a block's units [vb0, vb1) of x: one bulk load into shared
// memory completing on one mbarrier (issued by one thread).  Loading each
// token's part on its own mbarrier, so that stores could start after the first
// part, measured slower (R=8, N=128, top-8 of 256, H=7168: low-latency step
// 48.6 vs 47.9 us, dsv3 step 41.2 vs 40.4 us).
template <int UB>
__device__ __forceinline__ void stage_units(unsigned char* stage, uint64_t* bar,
                                            const unsigned char* xb, int vb0, int vb1) {
  mbar_init(bar, 1);
  mbar_init_fence();
  if (vb1 > vb0) {
    const uint32_t bytes = uint32_t(vb1 - vb0) * UB;
    mbar_arrive_expect_tx(bar, bytes);
    bulk_g2s(stage, xb + int64_t(vb0) * UB, bytes, bar);
  }
}

// A bounded wait for the staged units: false (after raising MP_ERR_TIMEOUT) if
// it gave up.
__device__ __forceinline__ bool wait_staged(uint64_t* bar, int32_t* dev_err) {
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, 0)) {
    if (++spins > kSpinLimit) {
      raise_error(dev_err, MP_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Before the block exits (warp 0): the staged load has landed (a bounded wait,
// at once when it was waited for already), and every bulk store of this
// thread has been performed.
__device__ __forceinline__ void drain_stage(uint64_t* bar, bool staged_any, int lane) {
  if (lane == 0 && staged_any) {
    uint32_t n = 0;
    while (!mbar_try_wait(bar, 0) && ++n < kSpinLimit) {
    }
  }
  bulk_wait_all();
}

struct LLFusedArgs {
  int R, N, K, E, vpr, spr;
  uint32_t stage_bytes;  // BULK: bytes reserved for the block's part of x (multiple of 128)
  void* q_scales;        // quantising mode: the rows' scales (fp32 or UE8M0 bytes)
  const int32_t* topk_idx;
  int64_t recv_capacity;
  int32_t* bin_offsets;
  int32_t* bin_src_offsets;
  int32_t* recv_src_token;
  int32_t* slot_row;
  const void* x;
  void* recv_x;
  const float* x_scales;
  float* recv_scales;
  int32_t* dev_err;
};

template <int NW, bool RANK_MAJOR, bool BULK, int QF>
__global__ void __launch_bounds__(kLLFThreads, kLLFBlocksPerSM)
mp_k_ll_dispatch_fused(LLFusedArgs a) {
  pdl_launch_dependents();  // the weighted combine after it may stage its blocks
  // launched as a programmatic dependent of the kernel before it on the stream:
  // the blocks are placed while that kernel ends, and wait for it here, before
  // any global memory access (every input is then complete and visible)
  pdl_wait_prior_grid();
  extern __shared__ __align__(128) unsigned char llf_smem[];
  __shared__ int32_t warp_tot[kLLFThreads / kWarp];
  // bytes per unit: 16/32-byte vectors, or in the quantising mode a scale block of bf16
  constexpr int UB = QF >= 0 ? (QF == kQE4M3 ? 128 : 32) * 2 : 4 * NW;
  unsigned char* stage = llf_smem;           // BULK: the block's units of x
  uint64_t* bar = reinterpret_cast<uint64_t*>(llf_smem + a.stage_bytes);
  int32_t* lower = reinterpret_cast<int32_t*>(llf_smem + a.stage_bytes + 16);
  const int nbins = RANK_MAJOR ? a.R : a.E;
  const int El = a.E / a.R;
  const int K = a.K;
  int32_t* upper = lower + nbins;  // [nbins] the other entries, then the bins' first rows
  int32_t* rows = upper + nbins;   // [block's entries] their ids, then their rows (-1: none)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.R * a.N;
  const int V = T * a.vpr;  // < 2^30 (launcher)
  const int vb0 = int(int64_t(V) * blockIdx.x / gridDim.x);
  const int vb1 = int(int64_t(V) * (blockIdx.x + 1) / gridDim.x);
  const int tf = vb0 / a.vpr;                             // first token touched
  const int tl = vb1 > vb0 ? (vb1 - 1) / a.vpr + 1 : tf;  // one past the last
  const int town = (vb0 + a.vpr - 1) / a.vpr;             // first token whose first unit is here
  const int e0 = tf * K, e1 = tl * K;                     // the block's entries
  const unsigned char* xb = static_cast<const unsigned char*>(a.x);
  // the block's part of x into shared memory (BULK; and in the quantising mode
  // when it fits, stage_bytes > 0)
  const bool stage_x = BULK || (QF >= 0 && a.stage_bytes > 0);
  if (stage_x && tid == 0) stage_units<UB>(stage, bar, xb, vb0, vb1);
  // 1. per-bin counts below and from the block's first entry; the block's own
  //    ids kept in `rows` for the walk
  const int nall = T * K;
  const bool vec4 = (reinterpret_cast<uintptr_t>(a.topk_idx) & 15u) == 0;
  const int n4 = vec4 ? nall / 4 : 0;
  const int4* t4 = reinterpret_cast<const int4*>(a.topk_idx);
  constexpr int L = 4;  // 16-byte id loads in flight per thread
  int4 p[L];
  auto load_ids = [&](int q0) {
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const int q = q0 + l * kLLFThreads;
      p[l] = q < n4 ? __ldg(t4 + q) : make_int4(-1, -1, -1, -1);
    }
  };
  bool bad = false;
  auto count = [&](int i, int e) {
    if (i >= e0 && i < e1) rows[i - e0] = e;
    if (e < 0 || e >= a.E) {
      bad |= e != -1;
      return;
    }
    atomicAdd(i < e0 ? &lower[RANK_MAJOR ? e / El : e] : &upper[RANK_MAJOR ? e / El : e], 1);
  };
  auto count_ids = [&](int q0) {
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const int q = q0 + l * kLLFThreads;
      if (q < n4) {
        count(4 * q, p[l].x);
        count(4 * q + 1, p[l].y);
        count(4 * q + 2, p[l].z);
        count(4 * q + 3, p[l].w);
      }
    }
  };
  load_ids(tid);
  const Words<NW>* x = reinterpret_cast<const Words<NW>*>(xb);
  Words<NW> v[BULK ? 1 : kLLFJ];
  if (!BULK && QF < 0) {
#pragma unroll
    for (int j = 0; j < kLLFJ; ++j) {
      const int q = vb0 + tid + j * kLLFThreads;
      if (q < vb1) v[j] = ld_stream_w<NW>(x + q);
    }
  }
  for (int b = tid; b < 2 * nbins; b += kLLFThreads) lower[b] = 0;
  __syncthreads();  // (also publishes the mbarrier's initialisation)
  count_ids(tid);
  for (int q0 = tid + L * kLLFThreads; q0 < n4; q0 += L * kLLFThreads) {
    load_ids(q0);
    count_ids(q0);
  }
  for (int i = 4 * n4 + tid; i < nall; i += kLLFThreads) count(i, __ldg(a.topk_idx + i));
  if (bad && blockIdx.x == 0) raise_error(a.dev_err, MP_ERR_BAD_EXPERT);
  __syncthreads();
  // 2. the bins' first rows: each thread a run of consecutive bins, a warp
  //    scan of the runs' totals, then a scan of the warps' totals
  {
    const int cpt = (nbins + kLLFThreads - 1) / kLLFThreads;
    const int b0 = min(nbins, tid * cpt), b1 = min(nbins, b0 + cpt);
    int chunk = 0;
    for (int b = b0; b < b1; ++b) chunk += lower[b] + upper[b];
    int inc = chunk;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kLLFThreads / kWarp ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += t;
      }
      if (lane < kLLFThreads / kWarp) warp_tot[lane] = w;
    }
    __syncthreads();
    int base = (warp > 0 ? warp_tot[warp - 1] : 0) + inc - chunk;
    for (int b = b0; b < b1; ++b) {
      const int c = lower[b] + upper[b];
      if (blockIdx.x == 0) a.bin_offsets[b] = base;
      upper[b] = base;
      base += c;
    }
    if (blockIdx.x == 0 && b0 < nbins && b1 == nbins) a.bin_offsets[nbins] = base;
  }
  __syncthreads();
  if (warp == 0) {
    // with BULK each entry's piece is stored as the walk places it, once the
    // block's units are in shared memory (a bounded wait; a lane that gives up
    // stores nothing)
    bool staged = true;
    unsigned char* rxb = static_cast<unsigned char*>(a.recv_x);
    // 3. the block's entries in order; a batch never crosses the first entry
    //    of a rank
    bool overflow = false;
    const int NK = a.N * K;
    for (int i0 = e0; i0 < e1;) {
      const int i1 = min(min(i0 + kWarp, e1), (i0 / NK + 1) * NK);
      if (i0 % NK == 0 && i0 / K >= town) {  // rank s begins with a token of this block
        const int s = i0 / NK;
        for (int b = lane; b < nbins; b += kWarp) a.bin_src_offsets[int64_t(b) * a.R + s] = lower[b];
        __syncwarp();
      }
      const int i = i0 + lane;
      const int e = i < i1 ? rows[i - e0] : -1;  // the id, replaced by its row below
      const bool ok = e >= 0 && e < a.E;
      const int b = ok ? (RANK_MAJOR ? e / El : e) : -1;
      const unsigned peers = __match_any_sync(kFull, b);
      const int run = ok ? lower[b] : 0;
      __syncwarp();
      int row = -1;
      if (ok) {
        const int64_t r = int64_t(upper[b]) + run + __popc(peers & lanemask_lt());
        if (r < a.recv_capacity) row = int(r);
        else overflow = true;
        if ((peers >> lane) == 1u) lower[b] = run + __popc(peers);  // highest peer
      }
      if (i < i1) {
        rows[i - e0] = row;
        const int t = i / K;
        if (t >= town) {
          a.slot_row[i] = row;
          if (row >= 0) a.recv_src_token[row] = t;
        }
        if (BULK && row >= 0 && staged && (staged = wait_staged(bar, a.dev_err))) {
          const int p0 = max(vb0, t * a.vpr), p1 = min(vb1, (t + 1) * a.vpr);
          bulk_s2g(rxb + (int64_t(row) * a.vpr + (p0 - t * a.vpr)) * UB, stage + (p0 - vb0) * UB,
                   uint32_t(p1 - p0) * UB);
        }
      }
      __syncwarp();
      i0 = i1;
    }
    if (overflow) raise_error(a.dev_err, MP_ERR_CAPACITY);
    if (BULK) {
      bulk_commit();
      drain_stage(bar, vb1 > vb0, lane);  // the load landed, the pieces written
    }
  }
  __syncthreads();
  // 4. the register copy (BULK: stored in step 3), or the quantising one
  if constexpr (QF >= 0) {
    // units are scale blocks; each lane quantises CPL channels once (the scale
    // block's lanes combining their amax) and stores the codes to its token's
    // rows, the block's first lane its scale
    constexpr int CPL = 16;
    constexpr bool FP4 = QF == kQMXFP4;
    constexpr int kLanes = (QF == kQE4M3 ? 128 : 32) / CPL;  // lanes per scale block
    constexpr int NB = FP4 ? CPL / 8 : CPL / 4;             // 32-bit words of codes per lane
    const int lvpr = a.vpr * kLanes;                        // lane vectors per row
    const int lv0 = vb0 * kLanes, lv1 = vb1 * kLanes;
    const int64_t code_row = int64_t(lvpr) * NB * 4;        // code bytes per row
    const Words<8>* xw = reinterpret_cast<const Words<8>*>(xb);
    const Words<8>* sw = reinterpret_cast<const Words<8>*>(stage);  // lane vector lv0 first
    unsigned char* out = static_cast<unsigned char*>(a.recv_x);
    // the staged units (a bounded wait; on a timeout report it, wait once more so
    // the load is not left writing shared memory, and read x from memory instead)
    bool from_smem = stage_x && lv0 + warp * kWarp < lv1;
    if (from_smem && !wait_staged(bar, a.dev_err)) {
      uint32_t n = 0;
      while (!mbar_try_wait(bar, 0) && ++n < kSpinLimit) {
      }
      from_smem = false;
    }
    for (int base = lv0 + warp * kWarp; base < lv1; base += kLLFThreads) {
      const int qv = base + lane;
      const bool valid = qv < lv1;  // (whole scale blocks: lv1 is a multiple of kLanes)
      Words<8> w;
      if (valid) {
        if (from_smem) {
          const uint4* s4 = reinterpret_cast<const uint4*>(sw + (qv - lv0));
          const uint4 lo = s4[0], hi = s4[1];
          w.w[0] = lo.x, w.w[1] = lo.y, w.w[2] = lo.z, w.w[3] = lo.w;
          w.w[4] = hi.x, w.w[5] = hi.y, w.w[6] = hi.z, w.w[7] = hi.w;
        } else {
          w = ld_stream_w<8>(xw + qv);
        }
      }
      uint32_t q[NB], sbits;
      quant_vector<CPL, QF>(valid, w, q, sbits);
      if (valid) {
        const int t = qv / lvpr, off = qv - t * lvpr;
        const int32_t* tr = rows + (t - tf) * K;
        for (int k = 0; k < K; ++k) {
          const int r = tr[k];
          if (r < 0) continue;
          st_codes<NB>(out + int64_t(r) * code_row + off * (NB * 4), q);
          if ((lane & (kLanes - 1)) == 0) {
            if constexpr (QF == kQE4M3)
              static_cast<uint32_t*>(a.q_scales)[int64_t(r) * a.vpr + off / kLanes] = sbits;
            else
              static_cast<unsigned char*>(a.q_scales)[int64_t(r) * a.vpr + off / kLanes] =
                  uint8_t(sbits);
          }
        }
      }
    }
  } else if (!BULK) {
    Words<NW>* rx = static_cast<Words<NW>*>(a.recv_x);
    for (int q0 = vb0; q0 < vb1; q0 += kLLFJ * kLLFThreads) {
      if (q0 != vb0) {
#pragma unroll
        for (int j = 0; j < kLLFJ; ++j) {
          const int q = q0 + tid + j * kLLFThreads;
          if (q < vb1) v[j] = ld_stream_w<NW>(x + q);
        }
      }
#pragma unroll
      for (int j = 0; j < kLLFJ; ++j) {
        const int q = q0 + tid + j * kLLFThreads;
        if (q < vb1) {
          const int t = q / a.vpr;
          const int off = q - t * a.vpr;
          const int32_t* tr = rows + (t - tf) * K;
          for (int k = 0; k < K; ++k) {
            const int r = tr[k];
            if (r >= 0) st_stream_w<NW>(rx + int64_t(r) * a.vpr + off, v[j]);
          }
        }
      }
    }
  }
  if (a.spr > 0) {
    const int nown = (tl - town) * K;  // entries of the owned tokens (<= 0: none)
    for (int idx = tid; idx < nown * a.spr; idx += kLLFThreads) {
      const int ent = idx / a.spr, c = idx - ent * a.spr;
      const int i = town * K + ent;
      const int r = rows[i - e0];
      if (r >= 0)
        a.recv_scales[int64_t(r) * a.spr + c] = __ldg(a.x_scales + int64_t(i / K) * a.spr + c);
    }
  }
}

template <int NW, bool RANK_MAJOR, bool BULK, int QF = -1>
static cudaError_t ll_dispatch_fused_nw(LLFusedArgs a, cudaStream_t stream) {
  const int nbins = RANK_MAJOR ? a.R : a.E;
  const int64_t V = int64_t(a.R) * a.N * a.vpr;
  int64_t G = int64_t(sm_count()) * kLLFBlocksPerSM;
  if (G > V) G = V;
  const int64_t vmax = (V + G - 1) / G;                 // units of one block at most
  const int64_t tmax = (vmax + a.vpr - 1) / a.vpr + 1;  // tokens one block's units touch
  const size_t table = sizeof(int32_t) * size_t(2 * nbins + tmax * a.K);
  if (table > kLLFMaxTable) return cudaErrorNotSupported;
  size_t stage = 0;
  if (BULK) {
    stage = (size_t(vmax) * 4 * NW + 127) / 128 * 128;
    if (stage > kLLFMaxStage) return cudaErrorNotSupported;
  } else if (QF >= 0) {  // staged when it fits, else read from memory
    stage = (size_t(vmax) * (QF == kQE4M3 ? 128 : 32) * 2 + 127) / 128 * 128;
    if (stage > kLLFMaxStage) stage = 0;
  }
  a.stage_bytes = uint32_t(stage);
  const size_t smem = stage + 16 + table;
  auto kernel = mp_k_ll_dispatch_fused<NW, RANK_MAJOR, BULK, QF>;
  static thread_local int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > 48 * 1024 && configured[dev] < int(smem)) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = int(smem);
  }
  return launch_pdl(kernel, dim3(unsigned(G)), dim3(kLLFThreads), smem, stream, a);
}

template <int QF>
static cudaError_t ll_quant_fused_q(int rank_major, const LLFusedArgs& a, cudaStream_t stream) {
  return rank_major ? ll_dispatch_fused_nw<8, true, false, QF>(a, stream)
                    : ll_dispatch_fused_nw<8, false, false, QF>(a, stream);
}

cudaError_t launch_ll_dispatch_quant_fused(int R, int N, int K, int E, int rank_major, int H,
                                           int fmt, const int32_t* topk_idx,
                                           int64_t recv_capacity, int32_t* bin_offsets,
                                           int32_t* bin_src_offsets, int32_t* recv_src_token,
                                           int32_t* slot_row, const void* x, void* recv_x,
                                           void* recv_scales, int32_t* dev_err,
                                           cudaStream_t stream) {
  const int nbins = rank_major ? R : E;
  const int64_t ids = int64_t(R) * N * K;
  const int block = fmt == kQE4M3 ? 128 : 32;  // channels per scale (H is a multiple)
  if (N <= 0 || ids > kLLFMaxIds || nbins > kLLFMaxBins || H % block != 0 || !aligned(x, 32) ||
      !aligned(recv_x, 16) || int64_t(R) * N * (H / 16) >= (int64_t(1) << 30))
    return cudaErrorNotSupported;
  LLFusedArgs a{};
  a.R = R, a.N = N, a.K = K, a.E = E, a.vpr = H / block, a.spr = 0;
  a.topk_idx = topk_idx, a.recv_capacity = recv_capacity, a.bin_offsets = bin_offsets;
  a.bin_src_offsets = bin_src_offsets, a.recv_src_token = recv_src_token, a.slot_row = slot_row;
  a.x = x, a.recv_x = recv_x, a.q_scales = recv_scales, a.dev_err = dev_err;
  switch (fmt) {
    case kQE4M3: return ll_quant_fused_q<kQE4M3>(rank_major, a, stream);
    case kQMXFP8: return ll_quant_fused_q<kQMXFP8>(rank_major, a, stream);
    case kQMXFP4: return ll_quant_fused_q<kQMXFP4>(rank_major, a, stream);
  }
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// The whole high-throughput dispatch in one kernel for small batches (layout,
// receive offsets, receive metadata and row copy), no block waiting for
// another.  The rows of destination d are ordered by source rank and token,
// which is the flat token index t = s*N + n, so token t's row on d is
// dest_offsets[d] + P(t, d), P(t, d) = the number of tokens t' < t that go to
// d.  Block b copies the units [V*b/G, V*(b+1)/G) of the token-major row
// space, like the low-latency kernel above:
//  1. one pass over all tokens: each token's destination mask from its K ids;
//     per destination, the tokens before the block's first (lower = P(tf, .)),
//     the others (upper), and the tokens before the end of the last rank whose
//     first token the block owns (rend);
//  2. warp 0: dest_offsets (a scan of lower + upper; block 0 writes it), then
//     it walks the block's tokens in order, 32 at a time, placing each token
//     on each of its destinations with a ballot, and stores (BULK) each row's
//     piece as it is placed; for the tokens whose first unit is the block's it
//     writes is_token_in_rank and send_row, and keeps P(s*N, .) for each rank
//     s that begins with one of them;
//  3. all threads: rank_prefix[s] = P(s*N, .) and num_tokens_per_rank[s] (the
//     difference to the next rank's P) for those ranks, the receive metadata of
//     the owned tokens' rows, the register copy (without BULK) and the scales;
//  4. one job per block while the bulk copies run: job j < R counts source
//     rank j's ids per expert (num_tokens_per_expert[j]), job R every id
//     (num_recv_tokens_per_expert).
// The pass of step 1 keeps its counts in registers (four 8-bit fields per
// word; within the id limit a thread tallies at most 32 tokens) and reduces
// them over the warp once at the end; for K = 4 or 8 each thread loads whole
// tokens, else a token's 16-byte id vectors sit on neighbouring lanes; its
// first id loads go out before the block's x.  A warp reduction per
// destination and group of tokens, or the ids queued behind x, cost several
// microseconds at R=8, N=128 (every block reads every id).
// The kernel is launched as a programmatic dependent of the kernel before it
// on the stream and waits for that kernel before any memory access.
// ---------------------------------------------------------------------------
struct HTFusedArgs {
  int R, N, K, E, vpr, spr;
  uint32_t stage_bytes;  // BULK: bytes reserved for the block's part of x (multiple of 128)
  int tmax;              // tokens one block's units touch, at most
  const int32_t* topk_idx;
  const float* topk_weights;
  int64_t recv_capacity;
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  uint32_t* is_token_in_rank;
  int32_t* recv_src_rank;
  int32_t* recv_src_idx;
  int32_t* recv_topk_idx;
  float* recv_topk_weights;
  int32_t* dest_offsets;
  int32_t* rank_prefix;
  int32_t* num_recv_tokens_per_expert;
  int32_t* send_row;
  const void* x;
  void* recv_x;
  const float* x_scales;
  float* recv_scales;
  int32_t* dev_err;
};

// shared-memory int32 words of the fused dispatch's tables
__host__ __device__ inline int htf_table_words(int R, int E, int tmax) {
  return 3 * R + E + 2 * tmax * R + tmax;
}

// The one-kernel high-throughput dispatch's launch shape: one block per SM.
// Its counting pass costs every block the same whatever its share, so fewer,
// larger blocks count less in all (dsv3 N=256 step 70.2 -> 66.8 us against two
// blocks of 512 threads per SM); 512 threads up to kHTFSmallIds ids (N=128 step
// 37.9 us, against 39.3 with 1,024), 1,024 above.
#ifndef MP_HTF_SMALL_IDS
#define MP_HTF_SMALL_IDS 8192
#endif
constexpr int64_t kHTFSmallIds = MP_HTF_SMALL_IDS;
// a block's stage of x: what the SM's shared memory leaves beside the tables
constexpr size_t kHTFMaxStage = 192 * 1024;

template <int NW, bool BULK, int NT>
__global__ void __launch_bounds__(NT, 1)
mp_k_layout_dispatch_fused(HTFusedArgs a) {
  pdl_launch_dependents();  // the combine after it may stage its blocks
  // launched as a programmatic dependent of the kernel before it on the stream:
  // the blocks are placed while that kernel ends, and wait for it here, before
  // any global memory access (every input is then complete and visible)
  pdl_wait_prior_grid();
  extern __shared__ __align__(128) unsigned char htf_smem[];
  constexpr int UB = 4 * NW;  // bytes per unit
  constexpr int L = 4;        // 16-byte id loads in flight per thread
  const int R = a.R, N = a.N, K = a.K, E = a.E, El = E / R;
  unsigned char* stage = htf_smem;  // BULK: the block's units of x
  uint64_t* bar = reinterpret_cast<uint64_t*>(htf_smem + a.stage_bytes);
  int32_t* lower = reinterpret_cast<int32_t*>(htf_smem + a.stage_bytes + 16);  // [R]
  int32_t* upper = lower + R;                      // [R]
  int32_t* rend = upper + R;                       // [R]
  int32_t* hist = rend + R;                        // [E] expert counts (step 4)
  int32_t* rows = hist + E;                        // [tmax][R] the block's tokens' rows
  int32_t* pref = rows + a.tmax * R;               // [tmax][R] P(s*N, .) of its ranks
  uint32_t* masks = reinterpret_cast<uint32_t*>(pref + a.tmax * R);  // [tmax]
  __shared__ int sh_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = R * N;
  const int V = T * a.vpr;  // < 2^30 (launcher)
  const int vb0 = int(int64_t(V) * blockIdx.x / gridDim.x);
  const int vb1 = int(int64_t(V) * (blockIdx.x + 1) / gridDim.x);
  const int tf = vb0 / a.vpr;                             // first token touched
  const int tl = vb1 > vb0 ? (vb1 - 1) / a.vpr + 1 : tf;  // one past the last
  const int town = (vb0 + a.vpr - 1) / a.vpr;             // first token whose first unit is here
  // the ranks s whose first token s*N is owned: [s_lo, s_lo + nranks)
  const int s_lo = (town + N - 1) / N;
  const int nranks = max(0, (tl - 1) / N - s_lo + 1);
  const int split2 = nranks > 0 ? (s_lo + nranks) * N : -1;  // rend counts the tokens below
  const unsigned char* xb = static_cast<const unsigned char*>(a.x);
  const Words<NW>* x = reinterpret_cast<const Words<NW>*>(xb);
  // e / El as a multiply-high (exact for every e, El < 8192 above 1)
  const uint32_t el_magic = El > 1 ? 0xFFFFFFFFu / uint32_t(El) + 1u : 0u;
  auto dest_of = [&](int e) { return El > 1 ? int(__umulhi(uint32_t(e), el_magic)) : e; };
  bool bad = false;
  auto add_mask = [&](uint32_t& m, int e) {
    if (e == -1) return;
    if (e < -1 || e >= E) {
      bad = true;
      return;
    }
    m |= 1u << dest_of(e);
  };
  const int G4 = K / 4;  // 16-byte id vectors per token
  const bool vec = K % 4 == 0 && (kWarp % G4) == 0 &&
                   (reinterpret_cast<uintptr_t>(a.topk_idx) & 15u) == 0;
  const int4* t4 = reinterpret_cast<const int4*>(a.topk_idx);
  int4 p[L];
  auto load_ids = [&](int base, int q1) {
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const int q = base + l * NT + tid;
      p[l] = q < q1 ? __ldg(t4 + q) : make_int4(-1, -1, -1, -1);
    }
  };
  // K = 4 or 8: each thread loads whole tokens (L / G4 of them, tokens
  // base_t + j*NT + tid), so that every lane tallies and no shuffle is needed
  const bool whole = vec && G4 <= 2;
  const int gs = G4 - 1;  // (whole) log2 of the vectors per token
  auto load_tokens = [&](int base_t) {
#pragma unroll
    for (int l = 0; l < L; ++l) {
      const int t = base_t + (l >> gs) * NT + tid;
      p[l] = t < T ? __ldg(t4 + int64_t(t) * G4 + (l & gs)) : make_int4(-1, -1, -1, -1);
    }
  };
  // 1. every token's destinations.  The first id loads go out first, then the
  //    block's x with BULK (x and the ids are inputs of the call, complete at
  //    launch; without BULK the row vectors are loaded after this pass).
  if (whole) load_tokens(0);
  else if (vec) load_ids(0, T * G4);
  for (int i = tid; i < 3 * R; i += NT) lower[i] = 0;  // lower, upper, rend
  if (tid == 0) sh_bad = 0;
  __syncthreads();
  // (the stage's mbarrier is first waited on after the next block barrier)
  if (BULK && tid == 0) stage_units<UB>(stage, bar, xb, vb0, vb1);
  {
    const int nw = (R + 3) / 4;  // count words (4 destinations each)
    uint32_t ca[8], cb[8], cc[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) ca[w] = cb[w] = cc[w] = 0u;
    auto tally = [&](int t, uint32_t m) {
      if (t >= tf && t < tl) masks[t - tf] = m;
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < nw) {
          const uint32_t u = m >> (4 * w);  // bits 0..3 to the low bit of bytes 0..3
          const uint32_t sp = (u & 1u) | ((u & 2u) << 7) | ((u & 4u) << 14) | ((u & 8u) << 21);
          if (t < tf) ca[w] += sp;
          else cb[w] += sp;
          if (t < split2) cc[w] += sp;
        }
    };
    if (whole) {
      for (int base_t = 0; base_t < T; base_t += (L >> gs) * NT) {
        if (base_t != 0) load_tokens(base_t);
        uint32_t mprev = 0u;
#pragma unroll
        for (int l = 0; l < L; ++l) {
          uint32_t m = 0u;
          add_mask(m, p[l].x);
          add_mask(m, p[l].y);
          add_mask(m, p[l].z);
          add_mask(m, p[l].w);
          if (gs == 1) {  // a token's two vectors: l even, then l odd
            if ((l & 1) == 0) {
              mprev = m;
              continue;
            }
            m |= mprev;
          }
          const int t = base_t + (l >> gs) * NT + tid;
          if (t < T) tally(t, m);
        }
      }
    } else if (vec) {  // a token's K/4 vectors on neighbouring lanes, masks OR-ed by shuffles
      const int q1 = T * G4;
      for (int base = 0; base < q1; base += L * NT) {
        if (base != 0) load_ids(base, q1);
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const int q = base + l * NT + tid;
          uint32_t m = 0u;
          add_mask(m, p[l].x);
          add_mask(m, p[l].y);
          add_mask(m, p[l].z);
          add_mask(m, p[l].w);
          for (int o = 1; o < G4; o <<= 1) m |= __shfl_xor_sync(kFull, m, o);
          if (q < q1 && (lane & (G4 - 1)) == 0) tally(q / G4, m);
        }
      }
    } else {  // one token per thread
      for (int t = tid; t < T; t += NT) {
        uint32_t m = 0u;
        for (int k = 0; k < K; ++k) add_mask(m, __ldg(a.topk_idx + int64_t(t) * K + k));
        tally(t, m);
      }
    }
    // one warp reduction per destination and count, then one shared add
#pragma unroll
    for (int w = 0; w < 8; ++w)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int d = 4 * w + j;
        if (d < R) {
          const int sa = __reduce_add_sync(kFull, (ca[w] >> (8 * j)) & 0xffu);
          const int sb = __reduce_add_sync(kFull, (cb[w] >> (8 * j)) & 0xffu);
          const int sc = split2 >= 0 ? __reduce_add_sync(kFull, (cc[w] >> (8 * j)) & 0xffu) : 0;
          if (lane == 0) {
            if (sa) atomicAdd(&lower[d], sa);
            if (sb) atomicAdd(&upper[d], sb);
            if (sc) atomicAdd(&rend[d], sc);
          }
        }
      }
  }
  if (bad) sh_bad = 1;
  __syncthreads();
  if (sh_bad && blockIdx.x == 0 && tid == 0) raise_error(a.dev_err, MP_ERR_BAD_EXPERT);
  Words<NW> v[BULK ? 1 : kLLFJ];  // the register copy's first vectors, in flight during the walk
  if (!BULK) {
#pragma unroll
    for (int j = 0; j < kLLFJ; ++j) {
      const int q = vb0 + tid + j * NT;
      if (q < vb1) v[j] = ld_stream_w<NW>(x + q);
    }
  }
  // 2. (warp 0) dest_offsets, then the walk
  if (warp == 0) {
    const int col = lane < R ? lower[lane] + upper[lane] : 0;  // lane d: tokens to d
    int inc = col;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    const int base = inc - col;  // lane d: dest_offsets[d]
    if (blockIdx.x == 0 && lane < R) {
      a.dest_offsets[lane] = base;
      if (lane == R - 1) a.dest_offsets[R] = inc;
    }
    int low = lane < R ? lower[lane] : 0;  // lane d: P(next token of the walk, d)
    bool staged = true;  // BULK: the block's units arrived (a bounded wait)
    unsigned char* rxb = static_cast<unsigned char*>(a.recv_x);
    bool overflow = false;
    for (int t0 = tf; t0 < tl; t0 += kWarp) {
      const int t = t0 + lane;
      const bool valid = t < tl;
      const uint32_t m = valid ? masks[t - tf] : 0u;
      const bool rank_start = valid && t >= town && t % N == 0;
      int p0 = 0, p1 = 0;
      if (valid) p0 = max(vb0, t * a.vpr), p1 = min(vb1, (t + 1) * a.vpr);
      for (int d = 0; d < R; ++d) {
        const bool hit = (m >> d) & 1u;
        const unsigned b = __ballot_sync(kFull, hit);
        const int ld = __shfl_sync(kFull, low, d), bd = __shfl_sync(kFull, base, d);
        if (lane == d) low += __popc(b);
        const int before = ld + __popc(b & lanemask_lt());  // P(t, d)
        if (rank_start) pref[(t / N - s_lo) * R + d] = before;
        int row = -1;
        if (hit) {
          const int64_t r = int64_t(bd) + before;
          if (r < a.recv_capacity) row = int(r);
          else overflow = true;
        }
        if (valid) {
          rows[(t - tf) * R + d] = row;
          if (t >= town) a.send_row[int64_t(t) * R + d] = row;
          if (BULK && row >= 0 && staged && (staged = wait_staged(bar, a.dev_err)))
            bulk_s2g(rxb + (int64_t(row) * a.vpr + (p0 - t * a.vpr)) * UB,
                     stage + (p0 - vb0) * UB, uint32_t(p1 - p0) * UB);
        }
      }
      if (valid && t >= town) a.is_token_in_rank[t] = m;
    }
    if (overflow) raise_error(a.dev_err, MP_ERR_CAPACITY);
    if (BULK) bulk_commit();
  }
  __syncthreads();
  // 3. the tables of the ranks beginning here, the metadata of the owned
  //    tokens' rows, the register copy, the scales
  for (int idx = tid; idx < nranks * R; idx += NT) {
    const int i = idx / R, d = idx - i * R, s = s_lo + i;
    const int here = pref[i * R + d];
    const int next = i + 1 < nranks ? pref[(i + 1) * R + d] : rend[d];
    a.rank_prefix[s * R + d] = here;
    a.num_tokens_per_rank[s * R + d] = next - here;
  }
  const int nown = tl - town;  // (<= 0: none)
  for (int idx = tid; idx < nown * R * K; idx += NT) {
    const int j = idx / (R * K), rem = idx - j * R * K, d = rem / K, k = rem - d * K;
    const int t = town + j;
    const int r = rows[(t - tf) * R + d];
    if (r < 0) continue;
    const int e = __ldg(a.topk_idx + int64_t(t) * K + k);
    const int lo = d * El;
    const bool local = e >= lo && e < lo + El;
    a.recv_topk_idx[int64_t(r) * K + k] = local ? e - lo : -1;
    a.recv_topk_weights[int64_t(r) * K + k] = local ? __ldg(a.topk_weights + int64_t(t) * K + k) : 0.0f;
    if (k == 0) {
      a.recv_src_rank[r] = t / N;
      a.recv_src_idx[r] = t - (t / N) * N;
    }
  }
  if (!BULK) {
    Words<NW>* rx = static_cast<Words<NW>*>(a.recv_x);
    for (int q0 = vb0; q0 < vb1; q0 += kLLFJ * NT) {
      if (q0 != vb0) {
#pragma unroll
        for (int j = 0; j < kLLFJ; ++j) {
          const int q = q0 + tid + j * NT;
          if (q < vb1) v[j] = ld_stream_w<NW>(x + q);
        }
      }
#pragma unroll
      for (int j = 0; j < kLLFJ; ++j) {
        const int q = q0 + tid + j * NT;
        if (q < vb1) {
          const int t = q / a.vpr;
          const int off = q - t * a.vpr;
          const int32_t* tr = rows + (t - tf) * R;
          for (int d = 0; d < R; ++d) {
            const int r = tr[d];
            if (r >= 0) st_stream_w<NW>(rx + int64_t(r) * a.vpr + off, v[j]);
          }
        }
      }
    }
  }
  if (a.spr > 0) {
    for (int idx = tid; idx < nown * R * a.spr; idx += NT) {
      const int j = idx / (R * a.spr), rem = idx - j * R * a.spr, d = rem / a.spr,
                c = rem - d * a.spr;
      const int t = town + j;
      const int r = rows[(t - tf) * R + d];
      if (r >= 0)
        a.recv_scales[int64_t(r) * a.spr + c] = __ldg(a.x_scales + int64_t(t) * a.spr + c);
    }
  }
  // 4. job j < R: source rank j's expert counts; job R: every id's expert
  for (int job = blockIdx.x; job <= R; job += gridDim.x) {
    for (int i = tid; i < E; i += NT) hist[i] = 0;
    __syncthreads();
    const int i0 = job < R ? job * N * K : 0;
    const int i1 = job < R ? i0 + N * K : T * K;
    int i4 = i0;  // 16-byte loads, L in flight per thread, where the range allows
    if ((reinterpret_cast<uintptr_t>(a.topk_idx) & 15u) == 0 && i0 % 4 == 0) {
      const int q1 = i1 / 4;
      for (int q0 = i0 / 4; q0 < q1; q0 += L * NT) {
        load_ids(q0, q1);
#pragma unroll
        for (int l = 0; l < L; ++l) {
          const int e4[4] = {p[l].x, p[l].y, p[l].z, p[l].w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (e4[j] >= 0 && e4[j] < E) atomicAdd(&hist[e4[j]], 1);
        }
      }
      i4 = 4 * q1;
    }
    for (int i = i4 + tid; i < i1; i += NT) {
      const int e = __ldg(a.topk_idx + i);
      if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    int32_t* out = job < R ? a.num_tokens_per_expert + int64_t(job) * E : a.num_recv_tokens_per_expert;
    for (int e = tid; e < E; e += NT) out[e] = hist[e];
    __syncthreads();
  }
  if (BULK && warp == 0) drain_stage(bar, vb1 > vb0, lane);  // the load landed, pieces written
}

template <int NW, bool BULK, int NT>
static cudaError_t layout_dispatch_fused_nw(HTFusedArgs a, cudaStream_t stream) {
  const int64_t V = int64_t(a.R) * a.N * a.vpr;
  int64_t G = int64_t(sm_count());
  if (G > V) G = V;
  const int64_t vmax = (V + G - 1) / G;
  const int64_t tmax = (vmax + a.vpr - 1) / a.vpr + 1;
  const size_t table = sizeof(int32_t) * size_t(htf_table_words(a.R, a.E, int(tmax)));
  const size_t stage = BULK ? (size_t(vmax) * 4 * NW + 127) / 128 * 128 : 0;
  if (table > kLLFMaxTable || stage > kHTFMaxStage) return cudaErrorNotSupported;
  a.stage_bytes = uint32_t(stage);
  a.tmax = int(tmax);
  const size_t smem = stage + 16 + table;
  auto kernel = mp_k_layout_dispatch_fused<NW, BULK, NT>;
  static thread_local int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem > 48 * 1024 && configured[dev] < int(smem)) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured[dev] = int(smem);
  }
  return launch_pdl(kernel, dim3(unsigned(G)), dim3(NT), smem, stream, a);
}

cudaError_t launch_layout_dispatch_fused(
    int R, int N, int K, int E, int64_t row_bytes, const int32_t* topk_idx,
    const float* topk_weights, int64_t recv_capacity, int32_t* num_tokens_per_rank,
    int32_t* num_tokens_per_expert, uint32_t* is_token_in_rank, int32_t* recv_src_rank,
    int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
    int32_t* dest_offsets, int32_t* rank_prefix, int32_t* num_recv_tokens_per_expert,
    int32_t* send_row, const void* x, int scales_per_row, const float* x_scales, void* recv_x,
    float* recv_scales, int32_t* dev_err, cudaStream_t stream) {
  const int64_t ids = int64_t(R) * N * K;
  if (N <= 0 || ids > kLLFMaxIds || R > 32 || row_bytes % 16 != 0 || !aligned(x, 16) ||
      !aligned(recv_x, 16))
    return cudaErrorNotSupported;
  const bool bulk = row_bytes >= kLLFBulkMinRow;
  const bool wide = !bulk && row_bytes % 32 == 0 && aligned(x, 32) && aligned(recv_x, 32);
  const int64_t vpr = row_bytes / (wide ? 32 : 16);
  if (int64_t(R) * N * vpr >= (int64_t(1) << 30)) return cudaErrorNotSupported;
  HTFusedArgs a{};
  a.R = R, a.N = N, a.K = K, a.E = E, a.vpr = int(vpr), a.spr = scales_per_row;
  a.topk_idx = topk_idx, a.topk_weights = topk_weights, a.recv_capacity = recv_capacity;
  a.num_tokens_per_rank = num_tokens_per_rank, a.num_tokens_per_expert = num_tokens_per_expert;
  a.is_token_in_rank = is_token_in_rank, a.recv_src_rank = recv_src_rank;
  a.recv_src_idx = recv_src_idx, a.recv_topk_idx = recv_topk_idx;
  a.recv_topk_weights = recv_topk_weights, a.dest_offsets = dest_offsets;
  a.rank_prefix = rank_prefix, a.num_recv_tokens_per_expert = num_recv_tokens_per_expert;
  a.send_row = send_row, a.x = x, a.recv_x = recv_x, a.x_scales = x_scales;
  a.recv_scales = recv_scales, a.dev_err = dev_err;
  const bool small = ids <= kHTFSmallIds;
  if (bulk) {
    const cudaError_t e = small ? layout_dispatch_fused_nw<4, true, 512>(a, stream)
                                : layout_dispatch_fused_nw<4, true, 1024>(a, stream);
    if (e != cudaErrorNotSupported) return e;  // else the register copy (16-byte units)
  }
  if (wide)
    return small ? layout_dispatch_fused_nw<8, false, 512>(a, stream)
                 : layout_dispatch_fused_nw<8, false, 1024>(a, stream);
  return small ? layout_dispatch_fused_nw<4, false, 512>(a, stream)
               : layout_dispatch_fused_nw<4, false, 1024>(a, stream);
}

cudaError_t launch_ll_dispatch_fused(int R, int N, int K, int E, int rank_major,
                                     int64_t row_bytes, const int32_t* topk_idx,
                                     int64_t recv_capacity, int32_t* bin_offsets,
                                     int32_t* bin_src_offsets, int32_t* recv_src_token,
                                     int32_t* slot_row, const void* x, int scales_per_row,
                                     const float* x_scales, void* recv_x, float* recv_scales,
                                     int32_t* dev_err, cudaStream_t stream) {
  const int nbins = rank_major ? R : E;
  const int64_t ids = int64_t(R) * N * K;
  if (N <= 0 || ids > kLLFMaxIds || nbins > kLLFMaxBins || row_bytes % 16 != 0 ||
      !aligned(x, 16) || !aligned(recv_x, 16))
    return cudaErrorNotSupported;
  const bool bulk = row_bytes >= kLLFBulkMinRow;
  const bool wide = !bulk && row_bytes % 32 == 0 && aligned(x, 32) && aligned(recv_x, 32);
  const int64_t vpr = row_bytes / (wide ? 32 : 16);
  if (int64_t(R) * N * vpr >= (int64_t(1) << 30)) return cudaErrorNotSupported;
  LLFusedArgs a{};
  a.R = R, a.N = N, a.K = K, a.E = E, a.vpr = int(vpr), a.spr = scales_per_row;
  a.topk_idx = topk_idx, a.recv_capacity = recv_capacity, a.bin_offsets = bin_offsets;
  a.bin_src_offsets = bin_src_offsets, a.recv_src_token = recv_src_token, a.slot_row = slot_row;
  a.x = x, a.recv_x = recv_x, a.x_scales = x_scales, a.recv_scales = recv_scales;
  a.dev_err = dev_err;
  cudaError_t e;
  if (bulk) {
    e = rank_major ? ll_dispatch_fused_nw<4, true, true>(a, stream)
                   : ll_dispatch_fused_nw<4, false, true>(a, stream);
    if (e != cudaErrorNotSupported) return e;  // else the register copy (16-byte units)
  }
  if (wide)
    return rank_major ? ll_dispatch_fused_nw<8, true, false>(a, stream)
                      : ll_dispatch_fused_nw<8, false, false>(a, stream);
  return rank_major ? ll_dispatch_fused_nw<4, true, false>(a, stream)
                    : ll_dispatch_fused_nw<4, false, false>(a, stream);
}

}  // namespace mp
