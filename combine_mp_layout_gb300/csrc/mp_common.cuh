// mp_common.cuh -- device helpers shared by the sm_103a kernels of the
// MoE layout / dispatch / combine path.  Everything here is inline PTX or
// plain CUDA C++ written for this library.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

#include "../../include/mp_layout.h"

namespace mp {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Workspace layout (bytes).  A 512-byte control block of counters, then the
// layout kernel's per-rank count accumulators, then the scan's tile records
// (a flag word per tile, then the tiles' aggregate counts, then their
// inclusive prefixes, R words each), then the fused kernel's two rank-totals
// buffers.  Every region starts on a 256-byte boundary.
// ---------------------------------------------------------------------------
struct Control {
  uint32_t scan_tile_counter;  // next scan tile to hand out
  uint32_t scan_done;          // scan blocks finished
  uint32_t scan_epoch;         // tags tile records of the current scan launch
  uint32_t fused_gen;          // fused layout + scan launches: picks the rank-totals buffer
  uint32_t layout_done[MP_MAX_RANKS];  // layout blocks finished, per source rank
  uint32_t bar_count;          // grid barrier of the fused layout + scan: arrivals (never reset)
  uint32_t bar_base;           // ... and their count when the current launch began
};
static_assert(sizeof(Control) <= 512, "control block");

constexpr int kLayoutTokens = 256;  // tokens per layout block (= threads)
constexpr int kScanTokens = 128;    // tokens per scan tile (= threads)

inline __host__ __device__ int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }
inline __host__ __device__ int64_t layout_blocks_per_rank(int N) {
  return (int64_t(N) + kLayoutTokens - 1) / kLayoutTokens;
}
// Scan tiles never straddle two source ranks: rank s owns tiles
// [s * C, (s + 1) * C), C = ceil(N / kScanTokens).
inline __host__ __device__ int64_t scan_tiles_per_rank(int N) {
  return (int64_t(N) + kScanTokens - 1) / kScanTokens;
}
inline __host__ __device__ int64_t scan_tiles(int R, int N) {
  return int64_t(R) * scan_tiles_per_rank(N);
}
// layout accumulators: int32 [R][E + R]
inline __host__ __device__ int64_t ws_acc_offset() { return 512; }
inline __host__ __device__ int64_t ws_acc_bytes(int R, int E) {
  return align256(int64_t(R) * (E + R) * 4);
}
// scan tile records
inline __host__ __device__ int64_t ws_flags_offset(int R, int E) {
  return ws_acc_offset() + ws_acc_bytes(R, E);
}
inline __host__ __device__ int64_t ws_agg_offset(int R, int N, int E) {
  return ws_flags_offset(R, E) + align256(scan_tiles(R, N) * 4);
}
inline __host__ __device__ int64_t ws_incl_offset(int R, int N, int E) {
  return ws_agg_offset(R, N, E) + align256(scan_tiles(R, N) * R * 4);
}
// rank totals of the fused layout + scan: two buffers of int32
// [MP_MAX_RANKS][MP_MAX_RANKS], used by alternate launches (a launch adds into
// one and zeroes the other for the next)
constexpr int64_t kTotBufInts = int64_t(MP_MAX_RANKS) * MP_MAX_RANKS;
inline __host__ __device__ int64_t ws_tot_offset(int R, int N, int E) {
  return ws_incl_offset(R, N, E) + align256(scan_tiles(R, N) * R * 4);
}
inline __host__ __device__ int64_t ws_total_bytes(int R, int N, int E) {
  return ws_tot_offset(R, N, E) + 2 * kTotBufInts * 4;
}

// ---------------------------------------------------------------------------
// Memory-order helpers (PTX ISA memory consistency model, gpu scope).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Atomic add with acquire-release semantics at gpu scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Programmatic dependent launch (sm_90+): let the grid launched after this one
// on the stream (with programmatic stream serialization) start its blocks now,
// and, in such a dependent grid, wait until the grid before it has finished
// and its writes are visible.  Both are no-ops without such a neighbour.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Streaming vector accesses: payload rows are touched once, so they bypass
// L1 (and loads are marked evict-first in L2).  Vectors of NW 32-bit words
// (NW = 4: 16 bytes; NW = 8: 32 bytes, the 256-bit global accesses
// sm_100-class GPUs provide).
template <int NW>
struct alignas(NW * 4) Words {
  uint32_t w[NW];
};

template <int NW>
__device__ __forceinline__ Words<NW> ld_stream_w(const Words<NW>* p) {
  Words<NW> v;
  if constexpr (NW == 8) {
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
          "=r"(v.w[6]), "=r"(v.w[7])
        : "l"(p));
  } else {
    static_assert(NW == 4, "16- or 32-byte vectors");
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3])
                 : "l"(p));
  }
  return v;
}

template <int NW>
__device__ __forceinline__ void st_stream_w(Words<NW>* p, const Words<NW>& v) {
  if constexpr (NW == 8) {
    asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
                 "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
  } else {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.w[0]),
                 "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3])
                 : "memory");
  }
}

// acc[0 .. 2*NW) += the 2*NW bf16 of v, each a separate round-to-nearest add.
template <int NW>
__device__ __forceinline__ void add_bf16(float* acc, const Words<NW>& v) {
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __uint_as_float(v.w[i] << 16));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __uint_as_float(v.w[i] & 0xffff0000u));
  }
}

// acc += w * v for the 2*NW bf16 of v: a binary32 product, then a binary32
// add (two roundings, never fused).
template <int NW>
__device__ __forceinline__ void add_bf16_weighted(float* acc, const Words<NW>& v, float w) {
#pragma unroll
  for (int i = 0; i < NW; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, __uint_as_float(v.w[i] << 16)));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, __uint_as_float(v.w[i] & 0xffff0000u)));
  }
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void raise_error(int32_t* dev_err, int bits) {
  if (dev_err) atomicOr(dev_err, bits);
}

// ---------------------------------------------------------------------------
// bf16 <-> fp32.  Widening a bf16 is a 16-bit shift into the top half of a
// binary32; narrowing uses the hardware round-to-nearest-even conversion
// (cvt.rn.bf16x2.f32 packs a into the high half and b into the low half).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// acc[0..7] += the eight bf16 of v, each add a separate round-to-nearest
// binary32 add (no contraction: there is no multiply to fuse with).
__device__ __forceinline__ void add_bf16x8(float* acc, const int4& v) {
  const uint32_t w[4] = {uint32_t(v.x), uint32_t(v.y), uint32_t(v.z), uint32_t(v.w)};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], bf16_lo(w[i]));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16_hi(w[i]));
  }
}
template <int NW>
__device__ __forceinline__ Words<NW> pack_bf16(const float* acc) {
  Words<NW> r;
#pragma unroll
  for (int i = 0; i < NW; ++i) r.w[i] = pack_bf16x2_rn(acc[2 * i], acc[2 * i + 1]);
  return r;
}
__device__ __forceinline__ int4 pack_bf16x8(const float* acc) {
  int4 r;
  r.x = int(pack_bf16x2_rn(acc[0], acc[1]));
  r.y = int(pack_bf16x2_rn(acc[2], acc[3]));
  r.z = int(pack_bf16x2_rn(acc[4], acc[5]));
  r.w = int(pack_bf16x2_rn(acc[6], acc[7]));
  return r;
}

// Kernel launch used by every launcher (one place to change launch attributes).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                        size_t smem, cudaStream_t stream, Args&&... args) {
  kernel<<<grid, block, smem, stream>>>(std::forward<Args>(args)...);
  return cudaGetLastError();
}

// Bounded spin for the decoupled lookback: about a second at most (2^20
// polls, back-off capped at ~1 us), then the caller reports MP_ERR_TIMEOUT.
constexpr uint32_t kSpinLimit = 1u << 20;

}  // namespace mp

namespace mp {

// ---------------------------------------------------------------------------
// Bulk-copy (TMA) and mbarrier helpers, inline PTX for sm_90+ / sm_100-class.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// One bounded attempt: returns once the phase with the given parity has
// completed (true) or after at most ~1 us of suspension (false), so that
// callers can cap their total wait (kSpinLimit attempts ~ 1 s).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000u)
      : "memory");
  return ok != 0;
}
// global -> shared bulk copy completing on an mbarrier (bytes: multiple of 16,
// both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// shared -> global bulk copy in the current bulk async-group
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until at most N committed groups still read shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// wait until every committed group has completed (writes visible)
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace mp
