/*
 * c_abi_smoke.c -- the C ABI used from plain C (no Python, no torch): one
 * layout -> dispatch -> combine pass on a small problem, with device memory
 * from the CUDA runtime, checked on the host against properties that hold by
 * definition:
 *   - sum of num_tokens_per_rank == dest_offsets[R] (every receive row is
 *     some token's row at some destination);
 *   - a token's send_row has one entry >= 0 per distinct rank owning one of
 *     its experts (expert e lives on rank e / (E/R));
 *   - combining the un-modified dispatch gives c * x, c = that rank count
 *     (exact here: x holds small integers, so every fp32 sum is exact);
 *   - the whole dispatch in one call (mp_layout_dispatch) gives the same send_row
 *     and the same combine;
 *   - the low-latency dispatch in one call gives every routed (token, slot) a row,
 *     and its weighted combine with unit weights gives K' * x, K' = the token's
 *     routed slots;
 *   - the low-latency dispatch with MXFP8 quantisation in the row copy gives the
 *     same slot rows, and every received row decodes back to x exactly (x holds
 *     small integers, so each 32-channel block's scale 2^(floor(log2 amax) - 8)
 *     makes every element an exact e4m3 value).
 * Prints "c abi smoke ok" and returns 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mp_layout.h"

#define R 4
#define N 300
#define K 3
#define E 16
#define H 64

static int fail(const char *what) {
  fprintf(stderr, "c abi smoke FAILED: %s\n", what);
  return 1;
}

#define CUDA(call)                                  \
  do {                                              \
    if ((call) != cudaSuccess) return fail(#call);  \
  } while (0)

#define MP(call)                                                  \
  do {                                                            \
    int st_ = (call);                                             \
    if (st_ != MP_OK) {                                           \
      fprintf(stderr, "%s: %s\n", #call, mp_status_string(st_));  \
      return 1;                                                   \
    }                                                             \
  } while (0)

static uint16_t bf16_of_small_int(int v) { /* exact: |v| < 256 */
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(u >> 16);
}

/* e4m3 ("fn") code -> value, from the format's definition (finite codes only) */
static float f32_of_e4m3(uint8_t c) {
  const int e = (c >> 3) & 15, m = c & 7;
  const float mag = e == 0 ? (float)m / 512.0f : (1.0f + (float)m / 8.0f) * (float)(1 << e) / 128.0f;
  return (c & 0x80) ? -mag : mag;
}

static float f32_of_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

int main(void) {
  const int El = E / R;
  const int64_t cap = (int64_t)R * N * (R < K ? R : K);
  static int32_t topk[R * N * K];
  static float w[R * N * K];
  static uint16_t x[R * N * H];
  static int32_t send_row[R * N * R];
  static uint16_t out[R * N * H];
  int32_t ntpr[R * R], dest_offsets[R + 1], err = 0;

  /* K distinct experts per token from a fixed LCG; every 11th token masked */
  uint32_t lcg = 12345u;
  for (int tok = 0; tok < R * N; ++tok) {
    for (int k = 0; k < K; ++k) {
      int e, dup;
      do {
        lcg = lcg * 1664525u + 1013904223u;
        e = (int)((lcg >> 8) % E);
        dup = 0;
        for (int j = 0; j < k; ++j) dup |= topk[tok * K + j] == e;
      } while (dup);
      topk[tok * K + k] = e;
      w[tok * K + k] = 1.0f / K;
    }
    if (tok % 11 == 0)
      for (int k = 0; k < K; ++k) topk[tok * K + k] = -1;
    for (int h = 0; h < H; ++h) x[tok * H + h] = bf16_of_small_int((tok + h) % 7 - 3);
  }

  void *d_topk, *d_w, *d_x, *d_ntpr, *d_ntpe, *d_mask, *d_err, *d_ws, *d_recv_x, *d_rsr, *d_rsi,
      *d_rti, *d_rtw, *d_doff, *d_rp, *d_nrtpe, *d_send, *d_out;
  const size_t ws = mp_workspace_size(R, N, E);
  if (ws == 0) return fail("mp_workspace_size");
  CUDA(cudaMalloc(&d_topk, sizeof topk));
  CUDA(cudaMalloc(&d_w, sizeof w));
  CUDA(cudaMalloc(&d_x, sizeof x));
  CUDA(cudaMalloc(&d_ntpr, sizeof(int32_t) * R * R));
  CUDA(cudaMalloc(&d_ntpe, sizeof(int32_t) * R * E));
  CUDA(cudaMalloc(&d_mask, sizeof(uint32_t) * R * N));
  CUDA(cudaMalloc(&d_err, sizeof(int32_t)));
  CUDA(cudaMalloc(&d_ws, ws));
  CUDA(cudaMalloc(&d_recv_x, sizeof(uint16_t) * (size_t)cap * H));
  CUDA(cudaMalloc(&d_rsr, sizeof(int32_t) * (size_t)cap));
  CUDA(cudaMalloc(&d_rsi, sizeof(int32_t) * (size_t)cap));
  CUDA(cudaMalloc(&d_rti, sizeof(int32_t) * (size_t)cap * K));
  CUDA(cudaMalloc(&d_rtw, sizeof(float) * (size_t)cap * K));
  CUDA(cudaMalloc(&d_doff, sizeof(int32_t) * (R + 1)));
  CUDA(cudaMalloc(&d_rp, sizeof(int32_t) * R * R));
  CUDA(cudaMalloc(&d_nrtpe, sizeof(int32_t) * E));
  CUDA(cudaMalloc(&d_send, sizeof send_row));
  CUDA(cudaMalloc(&d_out, sizeof out));
  CUDA(cudaMemset(d_ws, 0, ws));
  CUDA(cudaMemset(d_err, 0, sizeof(int32_t)));
  CUDA(cudaMemcpy(d_topk, topk, sizeof topk, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_w, w, sizeof w, cudaMemcpyHostToDevice));
  CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));

  MP(mp_layout(R, N, K, E, d_topk, d_ntpr, d_ntpe, d_mask, d_err, d_ws, NULL));
  MP(mp_dispatch(R, N, K, E, H, MP_BF16, d_x, NULL, d_topk, d_w, d_mask, d_ntpr, d_ntpe, cap,
                 d_recv_x, NULL, d_rsr, d_rsi, d_rti, d_rtw, d_doff, d_rp, d_nrtpe, d_send,
                 d_err, d_ws, NULL));
  MP(mp_combine(R, N, H, d_recv_x, cap, d_send, d_out, d_err, NULL));
  CUDA(cudaDeviceSynchronize());

  CUDA(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(ntpr, d_ntpr, sizeof ntpr, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(dest_offsets, d_doff, sizeof dest_offsets, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(send_row, d_send, sizeof send_row, cudaMemcpyDeviceToHost));
  CUDA(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
  if (err != 0) {
    fprintf(stderr, "device error: %s\n", mp_status_string(err));
    return 1;
  }

  int64_t total = 0;
  for (int i = 0; i < R * R; ++i) total += ntpr[i];
  if (total != dest_offsets[R]) return fail("sum of num_tokens_per_rank != dest_offsets[R]");
  for (int tok = 0; tok < R * N; ++tok) {
    int owners = 0, rows = 0;
    for (int d = 0; d < R; ++d) {
      int owns = 0;
      for (int k = 0; k < K; ++k) {
        const int e = topk[tok * K + k];
        owns |= e >= d * El && e < (d + 1) * El;
      }
      owners += owns;
      if (owns != (send_row[tok * R + d] >= 0)) return fail("send_row entry vs owning rank");
      rows += send_row[tok * R + d] >= 0;
    }
    if (rows != owners) return fail("destination count");
    for (int h = 0; h < H; ++h) {
      const float want = (float)owners * f32_of_bf16(x[tok * H + h]);
      if (f32_of_bf16(out[tok * H + h]) != want) return fail("combine != c * x");
    }
  }
  /* the whole dispatch in one call: layout, offsets and rows (the row copy a
   * programmatic dependent of the offsets kernel, writing the receive metadata) */
  {
    static int32_t send_row2[R * N * R];
    CUDA(cudaMemset(d_send, 0xff, sizeof send_row));
    CUDA(cudaMemset(d_recv_x, 0, sizeof(uint16_t) * (size_t)cap * H));
    CUDA(cudaMemset(d_out, 0, sizeof out));
    MP(mp_layout_dispatch(R, N, K, E, H, MP_BF16, d_x, NULL, d_topk, d_w, cap, d_ntpr, d_ntpe,
                          d_mask, d_recv_x, NULL, d_rsr, d_rsi, d_rti, d_rtw, d_doff, d_rp,
                          d_nrtpe, d_send, d_err, d_ws, NULL));
    MP(mp_combine(R, N, H, d_recv_x, cap, d_send, d_out, d_err, NULL));
    CUDA(cudaDeviceSynchronize());
    CUDA(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(send_row2, d_send, sizeof send_row2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(out, d_out, sizeof out, cudaMemcpyDeviceToHost));
    if (err != 0) {
      fprintf(stderr, "device error (one-call dispatch): %s\n", mp_status_string(err));
      return 1;
    }
    if (memcmp(send_row, send_row2, sizeof send_row) != 0) return fail("one-call send_row");
    for (int tok = 0; tok < R * N; ++tok) {
      int owners = 0;
      for (int d = 0; d < R; ++d) owners += send_row[tok * R + d] >= 0;
      for (int h = 0; h < H; ++h)
        if (f32_of_bf16(out[tok * H + h]) != (float)owners * f32_of_bf16(x[tok * H + h]))
          return fail("one-call combine != c * x");
    }
  }
  /* the low-latency path in one call: one row per valid (token, slot), then the
   * weighted combine with unit weights, which gives K * x for a routed token */
  {
    const int64_t lcap = (int64_t)R * N * K;
    static int32_t slot[R * N * K];
    static float ones[R * N * K];
    for (int i = 0; i < R * N * K; ++i) ones[i] = 1.0f;
    void *d_boff, *d_bsoff, *d_src, *d_slot, *d_lrx, *d_ones, *d_lout;
    CUDA(cudaMalloc(&d_boff, sizeof(int32_t) * (E + 1)));
    CUDA(cudaMalloc(&d_bsoff, sizeof(int32_t) * E * R));
    CUDA(cudaMalloc(&d_src, sizeof(int32_t) * (size_t)lcap));
    CUDA(cudaMalloc(&d_slot, sizeof slot));
    CUDA(cudaMalloc(&d_lrx, sizeof(uint16_t) * (size_t)lcap * H));
    CUDA(cudaMalloc(&d_ones, sizeof ones));
    CUDA(cudaMalloc(&d_lout, sizeof out));
    CUDA(cudaMemcpy(d_ones, ones, sizeof ones, cudaMemcpyHostToDevice));
    MP(mp_dispatch_ll(R, N, K, E, H, MP_BF16, 0, d_x, NULL, d_topk, NULL, lcap, d_boff, d_bsoff,
                      d_src, d_slot, d_lrx, NULL, d_err, NULL));
    MP(mp_combine_ll(R, N, K, H, d_lrx, lcap, d_slot, d_ones, d_lout, d_err, NULL));
    CUDA(cudaDeviceSynchronize());
    CUDA(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(slot, d_slot, sizeof slot, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(out, d_lout, sizeof out, cudaMemcpyDeviceToHost));
    if (err != 0) {
      fprintf(stderr, "device error (low-latency): %s\n", mp_status_string(err));
      return 1;
    }
    for (int tok = 0; tok < R * N; ++tok) {
      int valid = 0;
      for (int k = 0; k < K; ++k) {
        const int routed = topk[tok * K + k] >= 0;
        if (routed != (slot[tok * K + k] >= 0)) return fail("slot_row vs routed slot");
        valid += routed;
      }
      for (int h = 0; h < H; ++h) {
        const float want = (float)valid * f32_of_bf16(x[tok * H + h]);
        if (f32_of_bf16(out[tok * H + h]) != want) return fail("low-latency combine != c * x");
      }
    }
    /* the same dispatch with MXFP8 quantisation in the row copy */
    static int32_t slot2[R * N * K];
    static uint8_t codes[(size_t)R * N * K * H], scales[(size_t)R * N * K * (H / 32)];
    void *d_q, *d_qs;
    CUDA(cudaMalloc(&d_q, sizeof codes));
    CUDA(cudaMalloc(&d_qs, sizeof scales));
    MP(mp_dispatch_ll_quant(R, N, K, E, H, MP_Q_MXFP8, 0, d_x, d_topk, NULL, lcap, d_boff,
                            d_bsoff, d_src, d_slot, d_q, d_qs, d_err, NULL));
    CUDA(cudaDeviceSynchronize());
    CUDA(cudaMemcpy(&err, d_err, sizeof err, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(slot2, d_slot, sizeof slot2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(codes, d_q, sizeof codes, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(scales, d_qs, sizeof scales, cudaMemcpyDeviceToHost));
    if (err != 0) {
      fprintf(stderr, "device error (quantised low-latency): %s\n", mp_status_string(err));
      return 1;
    }
    if (memcmp(slot, slot2, sizeof slot) != 0) return fail("quantised slot_row");
    for (int tok = 0; tok < R * N; ++tok)
      for (int k = 0; k < K; ++k) {
        const int32_t row = slot2[tok * K + k];
        if (row < 0) continue;
        for (int h = 0; h < H; ++h) {
          const int code = scales[(size_t)row * (H / 32) + h / 32];
          const float X = code == 0 ? 0.0f : (float)(code >= 127 ? (1u << (code - 127)) : 1u) /
                                                 (float)(code < 127 ? (1u << (127 - code)) : 1u);
          if (f32_of_e4m3(codes[(size_t)row * H + h]) * X != f32_of_bf16(x[tok * H + h]))
            return fail("MXFP8 row does not decode to x");
        }
      }
  }
  printf("c abi smoke ok: %d receive rows\n", dest_offsets[R]);
  return 0;
}
