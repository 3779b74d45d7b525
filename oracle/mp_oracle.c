/*
 * mp_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-parallel layout / dispatch / combine path and the variable-size
 * reduce-scatterv / all-gatherv packing.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls
 * it.  Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared.
 * (-ffp-contract=off keeps every float add a separate IEEE binary32 add.)
 *
 * Sources followed (cited by page title and section):
 *  [EP]  "MSCCLPP EP implementation" (microsoft/mscclpp pull request #852):
 *        the port description (get_dispatch_layout computes counts and
 *        token-in-rank; intranode_dispatch / intranode_combine), the
 *        commit note on the bench byte accounting (the receive buffer holds
 *        one row per (token, source rank) pair) and the commit note that
 *        combine takes the dispatched rows back to their source tokens.
 *  [AGV] "Add pynccl all-gatherv and reducescatterv" (vllm-project/vllm pull
 *        request #20154): the all_gather / reduce_scatter code under review
 *        (per-root split along dim 0, offsets are running sums of sizes).
 *
 * Where the pages leave a step open, the readings below are used (each is
 * listed again in the design notes of the repository):
 *  - receive rows are ordered by destination rank, then source rank
 *    ascending, then token ascending; a token appears once per destination
 *    rank that owns at least one of its experts;
 *  - expert e lives on rank e / (E/R); topk_idx == -1 is a masked entry;
 *  - recv_topk_idx holds the local expert id (e - d*E/R) or -1 when the
 *    expert is not on the destination; recv_topk_weights holds the weight
 *    or 0.0f;
 *  - combine is the unweighted sum of a token's returned rows, accumulated
 *    in fp32 from +0.0f in ascending destination-rank order and rounded to
 *    bf16 once, round-to-nearest-even;
 *  - reduce-scatterv sums the R inputs in fp32 in ascending rank order and
 *    rounds once; all-gatherv concatenates the shards in rank order.
 *
 * Status bits returned (same meaning as the library's):
 *   8 = expert id outside [-1, E);  4 = receive capacity exceeded;
 *   1 = invalid argument.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORC_BAD_ARG 1
#define ORC_CAPACITY 4
#define ORC_BAD_EXPERT 8

/* ------------------------------------------------------------------ */
/* bf16 <-> binary32, from the IEEE-754 formats.                        */
/* bf16 is the top half of a binary32: widening is a 16-bit shift.      */
/* ------------------------------------------------------------------ */
float oracle_bf16_to_f32(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Narrowing keeps the top 16 bits and rounds on the 16 dropped bits:
 * above half -> up, below half -> down, exactly half -> to the even
 * (low bit 0) neighbour.  A carry out of the mantissa moves into the
 * exponent, which is what IEEE rounding wants (and reaches infinity from
 * the largest finite values).  NaN stays NaN: sign and payload top bits
 * kept, quiet bit forced so truncation cannot turn it into infinity. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint32_t exp_bits = u & 0x7f800000u, man_bits = u & 0x007fffffu;
  if (exp_bits == 0x7f800000u && man_bits != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xffffu;
  const uint32_t half = 0x8000u;
  if (dropped > half || (dropped == half && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* ------------------------------------------------------------------ */
/* Layout [EP, get_dispatch_layout: the counts and the token-in-rank   */
/* masks].                                                            */
/*   num_tokens_per_expert[s][e] = #(t,k) with topk_idx[s][t][k] == e   */
/*   is_token_in_rank[s][t]      = bit d set iff some k has its expert  */
/*                                 on rank d                            */
/*   num_tokens_per_rank[s][d]   = #t with bit d set                    */
/* ------------------------------------------------------------------ */
int oracle_layout(int R, int N, int K, int E, const int32_t *topk_idx,
                  int32_t *num_tokens_per_rank, int32_t *num_tokens_per_expert,
                  uint32_t *is_token_in_rank) {
  if (R < 1 || R > 32 || N < 0 || K < 1 || E < R || E % R != 0) return ORC_BAD_ARG;
  const int El = E / R;
  int status = 0;
  for (int64_t i = 0; i < (int64_t)R * R; ++i) num_tokens_per_rank[i] = 0;
  for (int64_t i = 0; i < (int64_t)R * E; ++i) num_tokens_per_expert[i] = 0;
  for (int s = 0; s < R; ++s) {
    for (int t = 0; t < N; ++t) {
      uint32_t mask = 0u;
      for (int k = 0; k < K; ++k) {
        int32_t e = topk_idx[((int64_t)s * N + t) * K + k];
        if (e == -1) continue; /* masked entry */
        if (e < -1 || e >= E) { status |= ORC_BAD_EXPERT; continue; }
        num_tokens_per_expert[(int64_t)s * E + e] += 1;
        mask |= 1u << (e / El);
      }
      is_token_in_rank[(int64_t)s * N + t] = mask;
      for (int d = 0; d < R; ++d)
        if ((mask >> d) & 1u) num_tokens_per_rank[(int64_t)s * R + d] += 1;
    }
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Dispatch [EP, intranode_dispatch; receive rows "one row per (token,  */
/* source rank) pair"].  Rows are appended in the literal loop order    */
/* for d, for s, for t -- that loop *is* the ordering definition.       */
/* Outputs besides the rows:                                            */
/*   dest_offsets[d]   first row of destination d; dest_offsets[R] =    */
/*                     total rows                                       */
/*   rank_prefix[s][d] rows that destination d received from ranks < s  */
/*   num_recv_tokens_per_expert[d][j] = #(s,t,k) with expert d*El+j     */
/*   send_row[s][t][d] row of (s,t) at d, or -1 (not sent / no room)    */
/* row_bytes is the payload size of one token row (bf16: 2H, e4m3: H);  */
/* scales_per_row floats of x_scales travel with each row (0 = none).   */
/* ------------------------------------------------------------------ */
int oracle_dispatch(int R, int N, int K, int E, int64_t row_bytes, int scales_per_row,
                    const uint8_t *x, const float *x_scales, const int32_t *topk_idx,
                    const float *topk_weights, const uint32_t *is_token_in_rank,
                    int64_t recv_capacity, uint8_t *recv_x, float *recv_scales,
                    int32_t *recv_src_rank, int32_t *recv_src_idx, int32_t *recv_topk_idx,
                    float *recv_topk_weights, int32_t *dest_offsets, int32_t *rank_prefix,
                    int32_t *num_recv_tokens_per_expert, int32_t *send_row) {
  if (R < 1 || R > 32 || N < 0 || K < 1 || E < R || E % R != 0 || row_bytes < 0 ||
      scales_per_row < 0 || recv_capacity < 0)
    return ORC_BAD_ARG;
  const int El = E / R;
  int status = 0;
  for (int64_t i = 0; i < (int64_t)R * N * R; ++i) send_row[i] = -1;

  int64_t row = 0;
  for (int d = 0; d < R; ++d) {
    dest_offsets[d] = (int32_t)row;
    for (int s = 0; s < R; ++s) {
      rank_prefix[(int64_t)s * R + d] = (int32_t)(row - dest_offsets[d]);
      for (int t = 0; t < N; ++t) {
        const int64_t tok = (int64_t)s * N + t;
        if (!((is_token_in_rank[tok] >> d) & 1u)) continue;
        if (row >= recv_capacity) { status |= ORC_CAPACITY; row += 1; continue; }
        memcpy(recv_x + row * row_bytes, x + tok * row_bytes, (size_t)row_bytes);
        for (int c = 0; c < scales_per_row; ++c)
          recv_scales[row * scales_per_row + c] = x_scales[tok * scales_per_row + c];
        recv_src_rank[row] = s;
        recv_src_idx[row] = t;
        for (int k = 0; k < K; ++k) {
          int32_t e = topk_idx[tok * K + k];
          int local = (e >= d * El && e < (d + 1) * El);
          recv_topk_idx[row * K + k] = local ? e - d * El : -1;
          recv_topk_weights[row * K + k] = local ? topk_weights[tok * K + k] : 0.0f;
        }
        send_row[tok * R + d] = (int32_t)row;
        row += 1;
      }
    }
  }
  dest_offsets[R] = (int32_t)row;

  for (int64_t i = 0; i < (int64_t)E; ++i) num_recv_tokens_per_expert[i] = 0;
  for (int64_t i = 0; i < (int64_t)R * N * K; ++i) {
    int32_t e = topk_idx[i];
    if (e >= 0 && e < E) num_recv_tokens_per_expert[e] += 1; /* [d][j] = e */
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Combine [EP, intranode_combine: the reverse of dispatch].            */
/*   out[s][t][h] = bf16( sum over d = 0..R-1 ascending, send_row >= 0, */
/*                        of float(y[send_row[s][t][d]][h]) )           */
/* accumulated in binary32 starting at +0.0f, rounded once.             */
/* ------------------------------------------------------------------ */
int oracle_combine(int R, int N, int H, const uint16_t *y, int64_t y_rows,
                   const int32_t *send_row, uint16_t *out) {
  if (R < 1 || R > 32 || N < 0 || H < 0 || y_rows < 0) return ORC_BAD_ARG;
  int status = 0;
  float *acc = (float *)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  if (!acc) return ORC_BAD_ARG;
  for (int s = 0; s < R; ++s) {
    for (int t = 0; t < N; ++t) {
      const int64_t tok = (int64_t)s * N + t;
      for (int h = 0; h < H; ++h) acc[h] = 0.0f;
      for (int d = 0; d < R; ++d) {
        int32_t r = send_row[tok * R + d];
        if (r < 0) continue;
        if ((int64_t)r >= y_rows) { status |= ORC_CAPACITY; continue; }
        const uint16_t *src = y + (int64_t)r * H;
        for (int h = 0; h < H; ++h) acc[h] = acc[h] + oracle_bf16_to_f32(src[h]);
      }
      uint16_t *dst = out + tok * H;
      for (int h = 0; h < H; ++h) dst[h] = oracle_f32_to_bf16(acc[h]);
    }
  }
  free(acc);
  return status;
}

/* ------------------------------------------------------------------ */
/* Reduce-scatterv [AGV, reduce_scatter with sizes: one reduce per      */
/* root r over rows [off_r, off_r + sizes[r]) of every rank's input].   */
/*   in  bf16 [R][S][H] (rank q's full input at q*S*H), S = sum(sizes)  */
/*   out bf16 [S][H]; rank r's shard is rows [off_r, off_r + sizes[r])  */
/*   out = bf16( sum over q ascending of float(in[q]) ), from +0.0f     */
/* ------------------------------------------------------------------ */
int oracle_reducescatterv(int R, int H, const int64_t *sizes, const uint16_t *in,
                          uint16_t *out) {
  if (R < 1 || H < 0) return ORC_BAD_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return ORC_BAD_ARG;
    S += sizes[r];
  }
  int64_t off = 0;
  for (int r = 0; r < R; ++r) {
    for (int64_t i = off; i < off + sizes[r]; ++i) {
      for (int h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int q = 0; q < R; ++q)
          acc = acc + oracle_bf16_to_f32(in[((int64_t)q * S + i) * H + h]);
        out[i * H + h] = oracle_f32_to_bf16(acc);
      }
    }
    off += sizes[r];
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* All-gatherv [AGV, all_gather with sizes: one broadcast per root r of */
/* its sizes[r] rows into rows [off_r, off_r + sizes[r]) of everyone's  */
/* output].                                                             */
/*   in  [S][row_bytes] -- shard r at rows [off_r, off_r + sizes[r])    */
/*   out [R][S][row_bytes] -- logical rank q's gathered copy at q*S     */
/* ------------------------------------------------------------------ */
int oracle_allgatherv(int R, int64_t row_bytes, const int64_t *sizes, const uint8_t *in,
                      uint8_t *out) {
  if (R < 1 || row_bytes < 0) return ORC_BAD_ARG;
  int64_t S = 0;
  for (int r = 0; r < R; ++r) {
    if (sizes[r] < 0) return ORC_BAD_ARG;
    S += sizes[r];
  }
  for (int q = 0; q < R; ++q) {
    int64_t off = 0;
    for (int r = 0; r < R; ++r) {
      for (int64_t i = off; i < off + sizes[r]; ++i)
        memcpy(out + ((int64_t)q * S + i) * row_bytes, in + i * row_bytes, (size_t)row_bytes);
      off += sizes[r];
    }
  }
  return 0;
}

/* Element-wise binary32 -> bf16 narrowing over an array (used by pins). */
void oracle_f32_to_bf16_array(int64_t n, const float *in, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 ("fn": no infinities, S.1111.111 is NaN, largest finite   */
/* 448 = 1.75 * 2^8, smallest normal 2^-6, subnormals k * 2^-9).      */
/* Narrowing from binary32 rounds to nearest, ties to even, on the    */
/* value's exact binary expansion, and saturates to +-448 (values at  */
/* or above 448 in magnitude give 448).  Written from the format,     */
/* with integer arithmetic on the binary32 fields.                    */
/* ------------------------------------------------------------------ */
static uint32_t rne_shift(uint32_t v, int sh) { /* round v / 2^sh to nearest, ties even */
  if (sh <= 0) return v << (-sh);
  if (sh >= 32) return 0u;
  uint32_t q = v >> sh, rem = v & ((1u << sh) - 1u), half = 1u << (sh - 1);
  if (rem > half || (rem == half && (q & 1u))) q += 1u;
  return q;
}

uint8_t oracle_f32_to_e4m3(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
  uint32_t ebits = (u >> 23) & 0xffu, mbits = u & 0x7fffffu;
  if (ebits == 0xffu && mbits) return (uint8_t)(sign | 0x7fu); /* NaN */
  if (ebits == 0xffu) return (uint8_t)(sign | 0x7eu);           /* +-inf saturate */
  if (ebits == 0u) return sign;  /* binary32 subnormals are far below 2^-10 */
  int e = (int)ebits - 127;      /* value = 1.m * 2^e */
  uint32_t sig = (1u << 23) | mbits; /* 24-bit significand */
  if (e >= -6) {
    /* normal range of the target: keep 3 fraction bits */
    uint32_t q = rne_shift(sig, 20); /* in [8, 16] */
    if (q == 16u) { q = 8u; e += 1; }
    if (e > 8 || (e == 8 && q > 14u)) return (uint8_t)(sign | 0x7eu); /* saturate to 448 */
    return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)(q - 8u));
  }
  /* below the normal range: units of 2^-9, value / 2^-9 = sig * 2^(e + 9 - 23) */
  uint32_t k = rne_shift(sig, 23 - (e + 9)); /* in [0, 8] */
  if (k >= 8u) return (uint8_t)(sign | 0x08u); /* rounds up to the smallest normal */
  return (uint8_t)(sign | (uint8_t)k);
}

float oracle_e4m3_to_f32(uint8_t b) {
  float s = (b & 0x80u) ? -1.0f : 1.0f;
  int e = (b >> 3) & 0xf, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) return s * (float)m * 0.001953125f; /* m * 2^-9 */
  return s * ldexpf(1.0f + (float)m / 8.0f, e - 7);
}

/* Per-block quantisation of bf16 rows to e4m3 (reading of the pages, which
 * name an FP8 E4M3 payload with FP32 scales but give no recipe): for each
 * token row and each block of 128 channels, amax = max |x|, scale =
 * amax / 448 (binary32 division; 1 when amax is 0), q = e4m3(x / scale)
 * (binary32 division, then the narrowing above).  Dequantised x ~ q * scale.
 *   x      bf16 [T][H], H a multiple of 128
 *   q      e4m3 [T][H]
 *   scales fp32 [T][H/128] */
int oracle_quantize_e4m3(int64_t T, int H, const uint16_t *x, uint8_t *q, float *scales) {
  if (T < 0 || H <= 0 || H % 128 != 0) return ORC_BAD_ARG;
  const int nb = H / 128;
  for (int64_t t = 0; t < T; ++t) {
    for (int b = 0; b < nb; ++b) {
      const uint16_t *xb = x + t * H + (int64_t)b * 128;
      float amax = 0.0f;
      for (int h = 0; h < 128; ++h) {
        float v = fabsf(oracle_bf16_to_f32(xb[h]));
        if (v > amax) amax = v;
      }
      const float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
      scales[t * nb + b] = scale;
      for (int h = 0; h < 128; ++h)
        q[t * H + (int64_t)b * 128 + h] = oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) / scale);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Receive-row expert ids in global numbering [EP, the later variant */
/* that returns global token-major expert ids with a configurable     */
/* invalid-expert sentinel]: for receive row r at destination d (the  */
/* d with dest_offsets[d] <= r < dest_offsets[d+1]) holding token     */
/* (s, t): out[r][k] = e when e = topk_idx[s][t][k] lives on d, else  */
/* `sentinel`.                                                        */
/* ------------------------------------------------------------------ */
int oracle_recv_topk_global(int R, int N, int K, int E, const int32_t *topk_idx,
                            const int32_t *recv_src_rank, const int32_t *recv_src_idx,
                            const int32_t *dest_offsets, int32_t sentinel, int32_t *out) {
  if (R < 1 || N < 0 || K < 1 || E < R || E % R != 0) return ORC_BAD_ARG;
  const int El = E / R;
  for (int d = 0; d < R; ++d) {
    for (int64_t r = dest_offsets[d]; r < dest_offsets[d + 1]; ++r) {
      const int64_t tok = (int64_t)recv_src_rank[r] * N + recv_src_idx[r];
      for (int k = 0; k < K; ++k) {
        const int32_t e = topk_idx[tok * K + k];
        out[r * K + k] = (e >= d * El && e < (d + 1) * El) ? e : sentinel;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Combined top-k weights [EP, intranode_combine returns the combined */
/* weights alongside the combined rows]: for token (s,t) and slot k,  */
/* the binary32 sum from +0.0f, over d = 0..R-1 ascending with        */
/* send_row[s][t][d] >= 0, of recv_topk_weights[send_row][k].         */
/* ------------------------------------------------------------------ */
int oracle_combine_weights(int R, int N, int K, const float *recv_topk_weights,
                           int64_t recv_rows, const int32_t *send_row, float *out) {
  if (R < 1 || N < 0 || K < 1 || recv_rows < 0) return ORC_BAD_ARG;
  int status = 0;
  for (int64_t tok = 0; tok < (int64_t)R * N; ++tok) {
    for (int k = 0; k < K; ++k) {
      float acc = 0.0f;
      for (int d = 0; d < R; ++d) {
        const int32_t r = send_row[tok * R + d];
        if (r < 0) continue;
        if ((int64_t)r >= recv_rows) { status |= ORC_CAPACITY; continue; }
        acc = acc + recv_topk_weights[(int64_t)r * K + k];
      }
      out[tok * K + k] = acc;
    }
  }
  return status;
}

/* ------------------------------------------------------------------ */
/* Low-latency expert-major layout [EP, low-latency dispatch/combine: */
/* per-expert receive buffers, one entry per (token, expert) pair].   */
/* Reading (the pages fix no order): expert e's rows are contiguous,  */
/* blocks in ascending e; inside a block rows are ordered by source   */
/* rank, then token, ascending.  A masked slot (-1) or an id outside  */
/* [0, E) gets no row.                                                */
/*   expert_offsets[e]    first row of expert e; [E] = total rows     */
/*   expert_src_offsets[e][s] rows of e from source ranks < s         */
/*   recv_src_token[row]  flattened source token s*N + t              */
/*   slot_row[s][t][k]    row of (s,t) at expert topk_idx[s][t][k], -1 */
/*   recv_x[row]          x[s][t] (row_bytes bytes)                   */
/* ------------------------------------------------------------------ */
int oracle_dispatch_ll(int R, int N, int K, int E, int64_t row_bytes, const uint8_t *x,
                       const int32_t *topk_idx, int64_t recv_capacity, uint8_t *recv_x,
                       int32_t *recv_src_token, int32_t *expert_offsets,
                       int32_t *expert_src_offsets, int32_t *slot_row) {
  if (R < 1 || N < 0 || K < 1 || E < 1 || row_bytes < 0 || recv_capacity < 0) return ORC_BAD_ARG;
  int status = 0;
  for (int64_t i = 0; i < (int64_t)R * N * K; ++i) slot_row[i] = -1;
  int64_t row = 0;
  for (int e = 0; e < E; ++e) {
    expert_offsets[e] = (int32_t)row;
    for (int s = 0; s < R; ++s) {
      expert_src_offsets[(int64_t)e * R + s] = (int32_t)(row - expert_offsets[e]);
      for (int t = 0; t < N; ++t) {
        const int64_t tok = (int64_t)s * N + t;
        for (int k = 0; k < K; ++k) {
          if (topk_idx[tok * K + k] != e) continue;
          if (row < recv_capacity) {
            memcpy(recv_x + row * row_bytes, x + tok * row_bytes, (size_t)row_bytes);
            recv_src_token[row] = (int32_t)tok;
            slot_row[tok * K + k] = (int32_t)row;
          } else {
            status |= ORC_CAPACITY;
          }
          row += 1;
        }
      }
    }
  }
  expert_offsets[E] = (int32_t)row;
  return status;
}

/* ------------------------------------------------------------------ */
/* Low-latency rank-major layout [EP, the pull request that adds      */
/* rank-major output to the low-latency path].  The same rows as the  */
/* expert-major layout (one per token and top-k slot with a valid     */
/* expert), grouped by the destination rank d = e / (E/R) that owns   */
/* the expert instead of by expert.  Reading (the pages fix no order  */
/* inside a group): rows of destination d are contiguous, groups in   */
/* ascending d; inside a group rows are ordered by source rank, then  */
/* token, then top-k slot, ascending.                                 */
/*   dest_offsets[d]      first row of destination d; [R] = total     */
/*   dest_src_offsets[d][s] rows of d from source ranks < s           */
/*   recv_src_token, slot_row, recv_x as in the expert-major layout   */
/* ------------------------------------------------------------------ */
int oracle_dispatch_ll_rank_major(int R, int N, int K, int E, int64_t row_bytes,
                                  const uint8_t *x, const int32_t *topk_idx,
                                  int64_t recv_capacity, uint8_t *recv_x,
                                  int32_t *recv_src_token, int32_t *dest_offsets,
                                  int32_t *dest_src_offsets, int32_t *slot_row) {
  if (R < 1 || N < 0 || K < 1 || E < R || E % R != 0 || row_bytes < 0 || recv_capacity < 0)
    return ORC_BAD_ARG;
  const int El = E / R;
  int status = 0;
  for (int64_t i = 0; i < (int64_t)R * N * K; ++i) slot_row[i] = -1;
  int64_t row = 0;
  for (int d = 0; d < R; ++d) {
    dest_offsets[d] = (int32_t)row;
    for (int s = 0; s < R; ++s) {
      dest_src_offsets[d * R + s] = (int32_t)(row - dest_offsets[d]);
      for (int t = 0; t < N; ++t) {
        const int64_t tok = (int64_t)s * N + t;
        for (int k = 0; k < K; ++k) {
          const int e = topk_idx[tok * K + k];
          if (e < d * El || e >= (d + 1) * El) continue;
          if (row < recv_capacity) {
            memcpy(recv_x + row * row_bytes, x + tok * row_bytes, (size_t)row_bytes);
            recv_src_token[row] = (int32_t)tok;
            slot_row[tok * K + k] = (int32_t)row;
          } else {
            status |= ORC_CAPACITY;
          }
          row += 1;
        }
      }
    }
  }
  dest_offsets[R] = (int32_t)row;
  return status;
}

/* Low-latency combine [EP, low-latency combine: the expert outputs of a   */
/* token are reduced with its top-k weights]: out[s][t] = bf16( sum over   */
/* k = 0..K-1 ascending with slot_row >= 0 of w[s][t][k] * float(y[row]) ), */
/* each product and each sum a separate binary32 operation, from +0.0f.    */
int oracle_combine_ll(int R, int N, int K, int H, const uint16_t *y, int64_t y_rows,
                      const int32_t *slot_row, const float *topk_weights, uint16_t *out) {
  if (R < 1 || N < 0 || K < 1 || H < 0 || y_rows < 0) return ORC_BAD_ARG;
  int status = 0;
  float *acc = (float *)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
  if (!acc) return ORC_BAD_ARG;
  for (int64_t tok = 0; tok < (int64_t)R * N; ++tok) {
    for (int h = 0; h < H; ++h) acc[h] = 0.0f;
    for (int k = 0; k < K; ++k) {
      const int32_t r = slot_row[tok * K + k];
      if (r < 0) continue;
      if ((int64_t)r >= y_rows) { status |= ORC_CAPACITY; continue; }
      const float w = topk_weights[tok * K + k];
      for (int h = 0; h < H; ++h) {
        const float p = w * oracle_bf16_to_f32(y[(int64_t)r * H + h]);
        acc[h] = acc[h] + p;
      }
    }
    for (int h = 0; h < H; ++h) out[tok * H + h] = oracle_f32_to_bf16(acc[h]);
  }
  free(acc);
  return status;
}

/* ------------------------------------------------------------------ */
/* MXFP8 block quantisation [EP, the later FP8 commits: E4M3 payloads */
/* with UE8M0 scale bytes per 32 elements, tiny non-zero blocks kept  */
/* at UE8M0 code zero].  Written from the microscaling definition:    */
/* per block of 32 channels, amax = max |x|, the shared scale is      */
/* X = 2^(floor(log2(amax)) - 8) (8 = exponent of E4M3's largest      */
/* normal), stored as the byte code = log2(X) + 127; codes below 0    */
/* are clamped to 0 (X = 2^-127) so a tiny non-zero block is still    */
/* encoded, and an all-zero block gets code 0.  Elements are          */
/* e4m3(x / X) with the narrowing above (saturating at +-448).        */
/*   x bf16 [T][H] (H % 32 == 0), q e4m3 [T][H], codes uint8 [T][H/32] */
/* ------------------------------------------------------------------ */
static int floor_log2_f32(float a) { /* a > 0, finite */
  uint32_t u;
  memcpy(&u, &a, sizeof u);
  int e = (int)((u >> 23) & 0xffu);
  if (e != 0) return e - 127;
  uint32_t m = u & 0x7fffffu; /* subnormal: m * 2^-149 */
  int p = 31;
  while (!((m >> p) & 1u)) --p;
  return p - 149;
}

int oracle_quantize_mxfp8(int64_t T, int H, const uint16_t *x, uint8_t *q, uint8_t *codes) {
  if (T < 0 || H <= 0 || H % 32 != 0) return ORC_BAD_ARG;
  const int nb = H / 32;
  for (int64_t t = 0; t < T; ++t) {
    for (int b = 0; b < nb; ++b) {
      const uint16_t *xb = x + t * H + (int64_t)b * 32;
      float amax = 0.0f;
      for (int h = 0; h < 32; ++h) {
        float v = fabsf(oracle_bf16_to_f32(xb[h]));
        if (v > amax) amax = v;
      }
      int code = 0;
      if (amax > 0.0f) {
        code = floor_log2_f32(amax) - 8 + 127;
        if (code < 0) code = 0;
        if (code > 254) code = 254;
      }
      codes[t * nb + b] = (uint8_t)code;
      const float X = ldexpf(1.0f, code - 127);
      for (int h = 0; h < 32; ++h)
        q[t * H + (int64_t)b * 32 + h] = oracle_f32_to_e4m3(oracle_bf16_to_f32(xb[h]) / X);
    }
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* MXFP4 block quantisation [AGV, the review note that gathering a    */
/* list of tensors lets the caller quantise to fp4 before the         */
/* all-gather; the pages name no fp4 format, so the microscaling one  */
/* of the EP page's MXFP8 scheme is used with E2M1 elements].         */
/* E2M1 (OCP FP4): sign bit 3, magnitude codes 0..7 stand for         */
/* 0, 0.5, 1, 1.5, 2, 3, 4, 6.  Narrowing picks the nearest magnitude,*/
/* a tie goes to the even code, magnitudes >= 6 saturate to 6, and    */
/* the sign is kept (a negative value that rounds to zero is -0).     */
/* Per block of 32 channels: code = clamp(floor(log2 amax) - 2 + 127, */
/* 0, 254) (2 = exponent of E2M1's largest normal, 6 = 1.5 * 2^2),    */
/* 0 for an all-zero block; X = 2^(code - 127); element e2m1(x / X).  */
/* Two elements per byte: channel 2j in bits 0-3, 2j+1 in bits 4-7.   */
/*   x bf16 [T][H] (H % 32 == 0), q uint8 [T][H/2], codes [T][H/32]   */
/* ------------------------------------------------------------------ */
static const float e2m1_mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

uint8_t oracle_f32_to_e2m1(float x) {
  const uint8_t sign = signbit(x) ? 8u : 0u;
  const double a = fabs((double)x);
  if (!(a < 6.0)) return (uint8_t)(sign | 7u); /* saturate (NaN never occurs in inputs) */
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = fabs(a - e2m1_mag[c]), db = fabs(a - e2m1_mag[best]);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  return (uint8_t)(sign | (uint8_t)best);
}

float oracle_e2m1_to_f32(uint8_t c) {
  const float m = e2m1_mag[c & 7u];
  return (c & 8u) ? -m : m;
}

int oracle_quantize_mxfp4(int64_t T, int H, const uint16_t *x, uint8_t *q, uint8_t *codes) {
  if (T < 0 || H <= 0 || H % 32 != 0) return ORC_BAD_ARG;
  const int nb = H / 32;
  for (int64_t t = 0; t < T; ++t) {
    for (int b = 0; b < nb; ++b) {
      const uint16_t *xb = x + t * H + (int64_t)b * 32;
      float amax = 0.0f;
      for (int h = 0; h < 32; ++h) {
        float v = fabsf(oracle_bf16_to_f32(xb[h]));
        if (v > amax) amax = v;
      }
      int code = 0;
      if (amax > 0.0f) {
        code = floor_log2_f32(amax) - 2 + 127;
        if (code < 0) code = 0;
        if (code > 254) code = 254;
      }
      codes[t * nb + b] = (uint8_t)code;
      const float X = ldexpf(1.0f, code - 127);
      uint8_t *qb = q + t * (H / 2) + (int64_t)b * 16;
      for (int h = 0; h < 32; h += 2) {
        const uint8_t lo = oracle_f32_to_e2m1(oracle_bf16_to_f32(xb[h]) / X);
        const uint8_t hi = oracle_f32_to_e2m1(oracle_bf16_to_f32(xb[h + 1]) / X);
        qb[h / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  return 0;
}
