// mp_common.cuh -- device helpers shared by the sm_103a kernels of the
// MoE layout / dispatch / combine path.  Everything here is inline PTX or
// plain CUDA C++ written for this library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mp_layout.h"

namespace mp {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// Workspace layout (bytes).  A 512-byte control block of counters, then the
// layout kernel's per-block partial counts, then the scan's tile states.
// Every region starts on a 256-byte boundary.
// ---------------------------------------------------------------------------
struct Control {
  uint32_t scan_tile_counter;  // next scan tile to hand out
  uint32_t scan_done;          // scan blocks finished
  uint32_t scan_epoch;         // tags tile states of the current scan launch
  uint32_t copy_unit_counter;  // reserved for dynamically scheduled copies
  uint32_t layout_done[MP_MAX_RANKS];  // layout blocks finished, per source rank
};
static_assert(sizeof(Control) <= 512, "control block");

constexpr int kLayoutTokens = 256;  // tokens per layout block (= threads)
constexpr int kScanTokens = 256;    // tokens per scan tile (= threads)

inline __host__ __device__ int64_t align256(int64_t v) { return (v + 255) & ~int64_t(255); }
inline __host__ __device__ int64_t layout_blocks_per_rank(int N) {
  return (int64_t(N) + kLayoutTokens - 1) / kLayoutTokens;
}
inline __host__ __device__ int64_t scan_tiles(int R, int N) {
  return (int64_t(R) * N + kScanTokens - 1) / kScanTokens;
}
inline __host__ __device__ int64_t ws_partials_offset() { return 512; }
inline __host__ __device__ int64_t ws_partials_bytes(int R, int N, int E) {
  return align256(int64_t(R) * layout_blocks_per_rank(N) * (E + R) * 4);
}
inline __host__ __device__ int64_t ws_status_offset(int R, int N, int E) {
  return ws_partials_offset() + ws_partials_bytes(R, N, E);
}
inline __host__ __device__ int64_t ws_status_bytes(int R, int N) {
  return align256(scan_tiles(R, N) * R * 8);
}
inline __host__ __device__ int64_t ws_total_bytes(int R, int N, int E) {
  return ws_status_offset(R, N, E) + ws_status_bytes(R, N);
}

// ---------------------------------------------------------------------------
// Memory-order helpers (PTX ISA memory consistency model, gpu scope).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cg_i32(const int32_t* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Streaming 16-byte accesses: payload rows are touched once, so keep them
// out of L1.
__device__ __forceinline__ int4 ld_stream(const int4* p) {
  int4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void st_stream(int4* p, const int4& v) {
  asm volatile("st.global.L1::no_allocate.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
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
__device__ __forceinline__ int4 pack_bf16x8(const float* acc) {
  int4 r;
  r.x = int(pack_bf16x2_rn(acc[0], acc[1]));
  r.y = int(pack_bf16x2_rn(acc[2], acc[3]));
  r.z = int(pack_bf16x2_rn(acc[4], acc[5]));
  r.w = int(pack_bf16x2_rn(acc[6], acc[7]));
  return r;
}

// Bounded spin for the decoupled lookback: about a second at most (2^20
// polls, back-off capped at ~1 us), then the caller reports MP_ERR_TIMEOUT.
constexpr uint32_t kSpinLimit = 1u << 20;

}  // namespace mp
