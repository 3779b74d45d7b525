/*
 * mp_layout.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel
 * layout / dispatch / combine path and the variable-size
 * reduce-scatterv / all-gatherv packing.
 *
 * Problem statement.  R logical ranks each hold N tokens of hidden size H
 * (x[R][N][H]) routed to K of E experts (topk_idx[R][N][K], topk_weights
 * [R][N][K]); the E experts are split evenly, expert e living on rank
 * e / (E/R).  All R ranks' buffers live in the memory of ONE GPU, so every
 * step below is a single-device permutation or reduction done by this
 * library's own CUDA kernels.
 *
 * Conventions shared by every entry point.
 *  - Every pointer argument except `sizes` (host) is a DEVICE pointer.
 *    The caller owns every buffer, including the workspace; the library
 *    allocates nothing and keeps no state between calls.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and is asynchronous: outputs are valid once the stream
 *    has reached the point after the call.
 *  - The return value reports what the host can see before the launch:
 *    MP_ERR_INVALID_ARG for an argument that fails the checks listed with
 *    each call (nothing is launched), MP_ERR_CUDA when a launch fails.
 *  - Errors that depend on device data are OR-ed (atomicOr) into the
 *    caller's device word `dev_err` (int32, zero it before the first call,
 *    read it after synchronising).  Writes are clamped so that bad data never
 *    makes a kernel touch memory outside the buffers described here.
 *  - Arrays are dense row-major with the shapes given in brackets.
 *  - bf16 values are passed as their 16-bit patterns (uint16 storage),
 *    e4m3 values as bytes (OCP FP8 E4M3 "fn" encoding; only copied).
 *  - Kernels read their inputs with 16-byte vector loads: every payload
 *    pointer (x, recv_x, y, out, in) must be 16-byte aligned; the index
 *    arrays must be 4-byte aligned.
 *
 * Source pages, by title and section:
 *  [EP]  "MSCCLPP EP implementation", microsoft/mscclpp pull request #852:
 *        port scope (get_dispatch_layout, intranode_dispatch,
 *        intranode_combine), the intranode multirank validation note, the
 *        internode combine note (combine takes the dispatched rows back to
 *        their tokens), the bench byte-accounting notes (one receive row per
 *        (token, source rank) pair; combine moves as many bytes as
 *        dispatch) and the FP8 E4M3 payload with FP32 scales.
 *  [AGV] "Add pynccl all-gatherv and reducescatterv", vllm-project/vllm pull
 *        request #20154: all_gatherv / reduce_scatterv along dim 0 with
 *        per-rank sizes (one broadcast / reduce per root inside an NCCL
 *        group).
 * Where the pages leave a choice open, the plainest reading is used; each
 * is named at the call it affects.
 */
#ifndef MP_LAYOUT_H
#define MP_LAYOUT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *mp_stream_t;

/* Status bits: returned by the calls (host-visible errors) and OR-ed into
 * the caller's device error word (data-dependent errors). */
enum {
  MP_OK = 0,
  MP_ERR_INVALID_ARG = 1, /* argument check failed; nothing launched            */
  MP_ERR_CUDA = 2,        /* a CUDA launch or attribute call failed               */
  MP_ERR_CAPACITY = 4,    /* more receive rows than recv_capacity / y_rows        */
  MP_ERR_BAD_EXPERT = 8,  /* topk_idx entry outside [-1, E)                       */
  MP_ERR_TIMEOUT = 16     /* a bounded device-side wait gave up (about a second)  */
};

/* Payload element types of mp_dispatch. */
enum { MP_BF16 = 0, MP_E4M3 = 1 };

#define MP_MAX_RANKS 32     /* is_token_in_rank is one 32-bit mask per token  */
#define MP_MAX_TOPK 32
#define MP_MAX_EXPERTS 8192
#define MP_SCALE_BLOCK 128  /* channels per fp32 scale of an e4m3 payload     */

/* Human-readable text for one status bit (or the lowest bit set). */
const char *mp_status_string(int status);

/* Bytes of workspace that mp_layout and mp_dispatch need for R ranks, N
 * tokens per rank and E experts (their counters, the per-rank count
 * accumulators and the scan's tile records: R*(E+R)*4 bytes plus about
 * (4 + 8R) bytes per 128 tokens of each rank, 26 KB for R=8, N=4096,
 * E=256).  The caller allocates it (device memory), fills it with zeros
 * ONCE before the first call, and then passes the same buffer
 * to every call of the same (R, N, E): each call leaves it zero-filled
 * again for the next one.  Calls that share a workspace must be ordered on
 * one stream.  Returns 0 for arguments mp_layout would reject. */
size_t mp_workspace_size(int R, int N, int E);

/*
 * mp_layout -- [EP] get_dispatch_layout: the per-rank and per-expert
 * counts and the token-in-rank masks.
 *   in   topk_idx              int32 [R][N][K]; -1 marks a masked entry
 *   out  num_tokens_per_rank   int32 [R][R]  [s][d] = #tokens of s sent to d
 *   out  num_tokens_per_expert int32 [R][E]  [s][e] = #(t,k) of s with expert e
 *   out  is_token_in_rank      uint32 [R][N] bit d set iff token (s,t) has an
 *                                            expert on rank d
 * Checks: 1 <= R <= 32, N >= 0, 1 <= K <= 32, R <= E <= 8192, E % R == 0,
 *   R*N*K < 2^31, non-NULL pointers (topk_idx may be NULL when N == 0).
 * Device errors: MP_ERR_BAD_EXPERT (entry < -1 or >= E; the entry is
 *   ignored).
 */
int mp_layout(int R, int N, int K, int E, const int32_t *topk_idx,
              int32_t *num_tokens_per_rank, int32_t *num_tokens_per_expert,
              uint32_t *is_token_in_rank, int32_t *dev_err, void *workspace,
              mp_stream_t stream);

/*
 * mp_dispatch -- [EP] intranode_dispatch: the receive offsets (a single-pass
 * decoupled-lookback scan) and the row copy.
 * Receive layout (reading of the pages, which fix no order): one row per
 * (token, destination rank that owns at least one of the token's experts),
 * ordered by destination rank, then source rank, then token, ascending.
 *   in   x                 [R][N][H] payload, bf16 (dtype MP_BF16) or e4m3
 *                          (MP_E4M3)
 *   in   x_scales          fp32 [R][N][H/128] for MP_E4M3, NULL for MP_BF16
 *   in   topk_idx, topk_weights            as given to mp_layout
 *   in   is_token_in_rank, num_tokens_per_rank, num_tokens_per_expert
 *                          the outputs of mp_layout for the same topk_idx
 *   in   recv_capacity     rows available in the receive buffers
 *   out  recv_x            [recv_capacity][H] payload rows
 *   out  recv_scales       fp32 [recv_capacity][H/128] (MP_E4M3; else NULL)
 *   out  recv_src_rank, recv_src_idx   int32 [recv_capacity]: source (s, t)
 *   out  recv_topk_idx     int32 [recv_capacity][K]: local expert id
 *                          (e - d*E/R) when expert e is on the row's
 *                          destination d, else -1
 *   out  recv_topk_weights fp32 [recv_capacity][K]: the weight for a local
 *                          expert, else 0.0f
 *   out  dest_offsets      int32 [R+1]: first row of destination d;
 *                          dest_offsets[R] = total rows T_recv
 *   out  rank_prefix       int32 [R][R]: [s][d] = rows of destination d
 *                          that come from source ranks < s
 *   out  num_recv_tokens_per_expert int32 [R][E/R]
 *   out  send_row          int32 [R][N][R]: [s][t][d] = receive row of token
 *                          (s,t) at destination d, or -1 (not sent, or past
 *                          recv_capacity); this is the handle mp_combine needs
 * Rows past recv_capacity are not written (MP_ERR_CAPACITY).  A capacity of
 * R*N*min(R,K) can never overflow; the exact need is dest_offsets[R]
 * (= the sum of num_tokens_per_rank).
 * Checks: as mp_layout, plus H > 0, H % 8 == 0 (bf16) or H % 128 == 0
 *   (e4m3), x_scales/recv_scales non-NULL exactly for MP_E4M3,
 *   recv_capacity >= 0, 16-byte aligned payload pointers.
 * Device errors: MP_ERR_CAPACITY, MP_ERR_TIMEOUT (scan wait gave up),
 *   MP_ERR_INVALID_ARG (the workspace was not zero-filled before first use).
 */
int mp_dispatch(int R, int N, int K, int E, int H, int dtype, const void *x,
                const float *x_scales, const int32_t *topk_idx, const float *topk_weights,
                const uint32_t *is_token_in_rank, const int32_t *num_tokens_per_rank,
                const int32_t *num_tokens_per_expert, int64_t recv_capacity, void *recv_x,
                float *recv_scales, int32_t *recv_src_rank, int32_t *recv_src_idx,
                int32_t *recv_topk_idx, float *recv_topk_weights, int32_t *dest_offsets,
                int32_t *rank_prefix, int32_t *num_recv_tokens_per_expert, int32_t *send_row,
                int32_t *dev_err, void *workspace, mp_stream_t stream);

/*
 * mp_dispatch_offsets and mp_dispatch_rows -- the two steps of mp_dispatch as
 * separate calls, with the same argument meanings.  mp_dispatch is exactly
 * mp_dispatch_offsets followed by mp_dispatch_rows on the same stream.
 *
 * mp_dispatch_offsets: the receive-offset scan.  Writes dest_offsets,
 *   rank_prefix, num_recv_tokens_per_expert, send_row and the per-row
 *   metadata (recv_src_rank, recv_src_idx, recv_topk_idx, recv_topk_weights).
 *   Checks and device errors as mp_dispatch, minus those about the payload.
 * mp_dispatch_rows: the row copy.  recv_x[send_row[s][t][d]] = x[s][t] (and
 *   the row's scales for MP_E4M3) for every entry >= 0 and < recv_capacity.
 *   It reads only send_row, so one set of offsets can dispatch several
 *   payloads routed the same way (the offsets are computed once).
 *   Checks: 1 <= R <= 32, N >= 0, H and dtype as mp_dispatch, R*N*R < 2^31,
 *   16-byte aligned x / recv_x, x_scales/recv_scales non-NULL exactly for
 *   MP_E4M3.  No device errors.
 */
int mp_dispatch_offsets(int R, int N, int K, int E, const int32_t *topk_idx,
                        const float *topk_weights, const uint32_t *is_token_in_rank,
                        const int32_t *num_tokens_per_rank, const int32_t *num_tokens_per_expert,
                        int64_t recv_capacity, int32_t *recv_src_rank, int32_t *recv_src_idx,
                        int32_t *recv_topk_idx, float *recv_topk_weights, int32_t *dest_offsets,
                        int32_t *rank_prefix, int32_t *num_recv_tokens_per_expert,
                        int32_t *send_row, int32_t *dev_err, void *workspace,
                        mp_stream_t stream);
int mp_dispatch_rows(int R, int N, int H, int dtype, const void *x, const float *x_scales,
                     const int32_t *send_row, int64_t recv_capacity, void *recv_x,
                     float *recv_scales, mp_stream_t stream);

/*
 * mp_layout_and_offsets -- mp_layout followed by mp_dispatch_offsets in one
 * call (no counterpart in the pages: the same two steps, fused).  Where the
 * problem fits one resident grid (R * ceil(N / 128) tiles of 128 tokens, at
 * most 16 per block of the grid the GPU holds at once) the two steps run as
 * one cooperative launch: each tile computes its tokens' rank masks and
 * expert counts, publishes its per-destination counts and looks back over
 * its rank's earlier tiles; after one grid barrier every tile writes its
 * rows.  Otherwise the two launches of mp_layout and mp_dispatch_offsets run.
 *   Arguments: those of mp_layout (outputs num_tokens_per_rank,
 *   num_tokens_per_expert, is_token_in_rank) and of mp_dispatch_offsets
 *   (its receive-side outputs); the results are identical to the two calls.
 *   Checks and device errors as the two calls, plus MP_ERR_TIMEOUT when the
 *   grid barrier's bounded (~1 s) wait gives up (the workspace must then be
 *   zero-filled again).
 */
int mp_layout_and_offsets(int R, int N, int K, int E, const int32_t *topk_idx,
                          const float *topk_weights, int64_t recv_capacity,
                          int32_t *num_tokens_per_rank, int32_t *num_tokens_per_expert,
                          uint32_t *is_token_in_rank, int32_t *recv_src_rank,
                          int32_t *recv_src_idx, int32_t *recv_topk_idx,
                          float *recv_topk_weights, int32_t *dest_offsets, int32_t *rank_prefix,
                          int32_t *num_recv_tokens_per_expert, int32_t *send_row,
                          int32_t *dev_err, void *workspace, mp_stream_t stream);

/*
 * mp_layout_dispatch -- the whole dispatch in one call: mp_layout, then
 * mp_dispatch (receive offsets and row copy), from the routing and the token
 * rows ([EP] get_dispatch_layout followed by intranode_dispatch; fusing them
 * has no counterpart in the pages).  Up to 16,384 top-k ids (R*N*K) it is one
 * kernel whose blocks each read every id, place their own share of the tokens
 * (a token's row on destination d is dest_offsets[d] plus the number of
 * earlier tokens in source-rank, token order that go to d) and copy their
 * share of the rows, through shared memory by the bulk-copy engine when it
 * fits; the workspace is not used then.  Above that, where the problem fits
 * one resident grid (as for mp_layout_and_offsets), layout and offsets run as
 * one launch that writes send_row and the tables, and the row copy -- which
 * also writes the receive metadata -- is launched as its programmatic
 * dependent: its blocks start while the offsets are computed, load their first
 * token rows, and wait for the offsets before they store.  Otherwise the
 * launches of mp_layout and mp_dispatch run.
 *   Arguments: the layout outputs of mp_layout and every argument of
 *   mp_dispatch (same meaning, layout and ownership); the results are
 *   identical to those two calls.
 *   Checks and device errors: those of mp_layout and mp_dispatch, plus
 *   MP_ERR_TIMEOUT when a bounded (~1 s) device wait gives up: the grid
 *   barrier (the workspace must then be zero-filled again) or, in the
 *   one-kernel form, a block's wait for its bulk load of x.
 */
int mp_layout_dispatch(int R, int N, int K, int E, int H, int dtype, const void *x,
                       const float *x_scales, const int32_t *topk_idx,
                       const float *topk_weights, int64_t recv_capacity,
                       int32_t *num_tokens_per_rank, int32_t *num_tokens_per_expert,
                       uint32_t *is_token_in_rank, void *recv_x, float *recv_scales,
                       int32_t *recv_src_rank, int32_t *recv_src_idx, int32_t *recv_topk_idx,
                       float *recv_topk_weights, int32_t *dest_offsets, int32_t *rank_prefix,
                       int32_t *num_recv_tokens_per_expert, int32_t *send_row, int32_t *dev_err,
                       void *workspace, mp_stream_t stream);

/*
 * mp_dispatch_offsets_global -- mp_dispatch_offsets with the receive rows'
 * expert ids in global numbering ([EP] the later variant that returns
 * global token-major expert ids with a configurable invalid-expert
 * sentinel): recv_topk_idx[row][k] = e when topk expert e lives on the row's
 * destination, else `sentinel` (e.g. E).  Everything else as
 * mp_dispatch_offsets.
 */
int mp_dispatch_offsets_global(int R, int N, int K, int E, const int32_t *topk_idx,
                               const float *topk_weights, const uint32_t *is_token_in_rank,
                               const int32_t *num_tokens_per_rank,
                               const int32_t *num_tokens_per_expert, int64_t recv_capacity,
                               int32_t sentinel, int32_t *recv_src_rank, int32_t *recv_src_idx,
                               int32_t *recv_topk_idx, float *recv_topk_weights,
                               int32_t *dest_offsets, int32_t *rank_prefix,
                               int32_t *num_recv_tokens_per_expert, int32_t *send_row,
                               int32_t *dev_err, void *workspace, mp_stream_t stream);

/*
 * mp_combine_weights -- the combined top-k weights that accompany combine
 * ([EP] intranode_combine returns the combined weights with the rows).
 *   in   recv_topk_weights fp32 [recv_rows][K] (as written by dispatch, or
 *        updated by the experts)
 *   in   send_row int32 [R][N][R]
 *   out  combined_topk_weights fp32 [R][N][K]:
 *        [s][t][k] = sum over d = 0..R-1 ascending with send_row[s][t][d] >= 0
 *        of recv_topk_weights[send_row[s][t][d]][k], fp32 from +0.0f
 *        (for an un-modified dispatch: each valid slot's weight, +0 for masked)
 * Checks: 1 <= R <= 32, N >= 0, 1 <= K <= 32, recv_rows >= 0.
 * Device errors: MP_ERR_CAPACITY for a send_row entry >= recv_rows (skipped).
 */
int mp_combine_weights(int R, int N, int K, const float *recv_topk_weights, int64_t recv_rows,
                       const int32_t *send_row, float *combined_topk_weights, int32_t *dev_err,
                       mp_stream_t stream);

/*
 * mp_dispatch_rows_bulk -- the row copy of mp_dispatch_rows done by the
 * bulk-copy (TMA) engine instead of SM loads and stores (the north-star
 * design names cp.async.bulk row copies as one way to move the rows): each
 * block's single warp streams token rows through a ring of shared-memory
 * stages (cp.async.bulk global->shared, completion on an mbarrier) and
 * issues one contiguous shared->global bulk store per destination row.
 * Same arguments, checks and result as mp_dispatch_rows, plus `dev_err`
 * (non-NULL, 4-byte aligned).  On GB300 the SM-vector copy is faster for the
 * dsv3 rows (430 vs ~500 us); the bulk path leaves the SMs' load/store pipes
 * and registers free, for callers that run it beside compute kernels.
 * Device errors: MP_ERR_TIMEOUT if a bounded (~1 s) mbarrier wait gives up
 * (the block then waits, bounded, for its copies in flight and stops).
 */
int mp_dispatch_rows_bulk(int R, int N, int H, int dtype, const void *x, const float *x_scales,
                          const int32_t *send_row, int64_t recv_capacity, void *recv_x,
                          float *recv_scales, int32_t *dev_err, mp_stream_t stream);

/*
 * mp_dispatch_rows_e4m3 -- the row copy with in-kernel FP8 quantisation
 * ([EP] FP8 E4M3 payload with FP32 scales; the pages give no recipe, the
 * reading used: per block of 128 channels of a token row, amax = max |x|,
 * scale = amax / 448 in fp32 (1 when amax is 0), code = e4m3(x / scale) with
 * an fp32 division and round-to-nearest-even, saturating at +-448).
 *   in   x          bf16 [R][N][H], H % 128 == 0
 *   in   send_row   int32 [R][N][R] from mp_dispatch_offsets (or mp_dispatch)
 *   out  recv_x     e4m3 [recv_capacity][H]: the quantised row at every
 *                   destination row of the token
 *   out  recv_scales fp32 [recv_capacity][H/128]
 * Dequantised x is code * scale.  Checks: 1 <= R <= 32, N >= 0, H > 0,
 * H % 128 == 0, R*N*R < 2^31, 16-byte aligned x / recv_x.  No device errors.
 */
int mp_dispatch_rows_e4m3(int R, int N, int H, const void *x, const int32_t *send_row,
                          int64_t recv_capacity, void *recv_x, float *recv_scales,
                          mp_stream_t stream);

/*
 * mp_dispatch_rows_mxfp8 -- the row copy with in-kernel MXFP8 quantisation
 * ([EP] the later FP8 commits: E4M3 payloads with UE8M0 scale bytes per 32
 * elements, tiny non-zero blocks kept at UE8M0 code zero; read with the
 * microscaling definition): per block of 32 channels, amax = max |x|,
 * code = clamp(floor(log2 amax) - 8 + 127, 0, 254) (0 for an all-zero
 * block), X = 2^(code - 127), element codes e4m3(x / X) with round-to-
 * nearest-even, saturating at +-448 (values of x / X in (448, 512) clamp).
 *   in   x           bf16 [R][N][H], H % 32 == 0
 *   out  recv_x      e4m3 [recv_capacity][H]
 *   out  recv_scales uint8 [recv_capacity][H/32]: the UE8M0 codes
 * Dequantised x is element * 2^(code - 127).  Checks as mp_dispatch_rows_e4m3
 * with H % 32 == 0.  No device errors.
 */
int mp_dispatch_rows_mxfp8(int R, int N, int H, const void *x, const int32_t *send_row,
                           int64_t recv_capacity, void *recv_x, uint8_t *recv_scales,
                           mp_stream_t stream);

/*
 * mp_dispatch_rows_mxfp4 -- the row copy with in-kernel MXFP4 quantisation
 * ([AGV] the review note that a list all-gather lets the caller quantise to
 * fp4 first; the pages name no fp4 format, so the microscaling form of the
 * MXFP8 scheme above is used with E2M1 elements): per block of 32 channels,
 * code = clamp(floor(log2 amax) - 2 + 127, 0, 254) (0 for an all-zero
 * block), X = 2^(code - 127); each element is e2m1(x / X), round-to-nearest-
 * even over the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (saturating at 6; the
 * sign bit is kept, also on a zero), bit 3 the sign.
 *   in   x           bf16 [R][N][H], H % 32 == 0
 *   out  recv_x      uint8 [recv_capacity][H/2]: byte j of a row holds channel
 *                    2j in bits 0-3 and channel 2j+1 in bits 4-7
 *   out  recv_scales uint8 [recv_capacity][H/32]: the UE8M0 codes
 * Dequantised x is element * 2^(code - 127).  Checks as mp_dispatch_rows_mxfp8.
 * No device errors.
 */
int mp_dispatch_rows_mxfp4(int R, int N, int H, const void *x, const int32_t *send_row,
                           int64_t recv_capacity, void *recv_x, uint8_t *recv_scales,
                           mp_stream_t stream);

/*
 * mp_combine -- [EP] intranode_combine, the reverse of dispatch.
 *   in   y        bf16 [y_rows][H]: one row per receive row (for example the
 *                 expert outputs, or recv_x itself)
 *   in   send_row int32 [R][N][R] from mp_dispatch
 *   out  out      bf16 [R][N][H]:
 *        out[s][t] = bf16( sum over d = 0..R-1 ascending with
 *                          send_row[s][t][d] >= 0 of float(y[send_row[s][t][d]]) )
 *        accumulated in fp32 starting from +0.0f, rounded once to bf16 with
 *        round-to-nearest-even (reading of the pages, which fix neither the
 *        order nor the precision).  The sum is unweighted; a token with no
 *        destination gets +0.0.
 * Checks: 1 <= R <= 32, N >= 0, H > 0, H % 8 == 0, y_rows >= 0, aligned
 *   non-NULL pointers.
 * Device errors: MP_ERR_CAPACITY for a send_row entry >= y_rows (skipped).
 */
int mp_combine(int R, int N, int H, const void *y, int64_t y_rows, const int32_t *send_row,
               void *out, int32_t *dev_err, mp_stream_t stream);

/*
 * mp_reducescatterv -- [AGV] reduce_scatterv along dim 0 with per-rank sizes.
 *   sizes  HOST int64 [R]: rows of rank r's shard (>= 0); S = sum(sizes),
 *          off_r = sizes[0] + ... + sizes[r-1]
 *   in     bf16 [R][S][H]: logical rank q's full input at in + q*S*H
 *   out    bf16 [S][H]: rank r's shard is rows [off_r, off_r + sizes[r]),
 *          out[i] = bf16( sum over q = 0..R-1 ascending of float(in[q][i]) ),
 *          fp32 from +0.0f, rounded once (round-to-nearest-even).
 * Checks: R >= 1, H > 0, H % 8 == 0, sizes non-NULL with every entry >= 0,
 *   16-byte aligned non-NULL in/out when S > 0.
 */
int mp_reducescatterv(int R, int H, const int64_t *sizes, const void *in, void *out,
                      mp_stream_t stream);

/*
 * mp_allgatherv -- [AGV] all_gatherv along dim 0 with per-rank sizes.
 *   sizes      HOST int64 [R] as above
 *   row_bytes  bytes of one row (any element type; a multiple of 16)
 *   in         [S][row_bytes]: the R shards back to back, shard r at row off_r
 *   out        [R][S][row_bytes]: logical rank q's gathered copy at
 *              out + q*S*row_bytes; every copy is the shards in rank order.
 * Checks: R >= 1, row_bytes > 0, row_bytes % 16 == 0, sizes entries >= 0,
 *   16-byte aligned non-NULL in/out when S > 0.
 */
int mp_allgatherv(int R, int64_t row_bytes, const int64_t *sizes, const void *in, void *out,
                  mp_stream_t stream);

/*
 * mp_dispatch_noalloc -- mp_dispatch for callers that cannot allocate device
 * memory.  (The pages have no counterpart: this is a convenience of this
 * library.)
 * Some callers cannot call cudaMalloc for the workspace mp_dispatch needs:
 * a host application that reserves (nearly) all device memory for its own
 * pool at start-up, a plugin whose host framework owns every device
 * allocation, or a latency-critical loop in which cudaMalloc / cudaFree would
 * synchronise the device.  This call takes the same arguments as mp_dispatch
 * except the workspace, and computes the same outputs; it allocates nothing.
 * The scan's scratch lives instead in a fixed array of
 * MP_NOALLOC_SCRATCH_BYTES inside the library's device memory, which every
 * GPU that loads the library holds until the process exits.
 *  - Scope: only the dispatch step goes without a workspace.  Its inputs
 *    num_tokens_per_rank, num_tokens_per_expert and is_token_in_rank come
 *    from mp_layout, which still takes a caller-allocated workspace (a caller
 *    may also compute them by other means).
 *  - Limit: problems whose mp_workspace_size(R, N, E) exceeds
 *    MP_NOALLOC_SCRATCH_BYTES (1 MiB; with E=256 that allows up to 242,688
 *    tokens per rank at R=8 and 15,360 at R=32) are rejected with
 *    MP_ERR_INVALID_ARG before anything is launched; use mp_dispatch with a
 *    workspace for those.  Every other argument is checked as by mp_dispatch,
 *    also before anything is put on the stream.
 *  - Set-up: the first call on each device (with that device current), and
 *    the first call after that device's context was reset, finds the array's
 *    device address, zero-fills it on `stream` and waits for that stream
 *    (cudaStreamSynchronize), so the fill is complete before this or any
 *    later call uses the array.  Make that first call before any stream
 *    capture.
 *  - Every call on a device shares the one array and starts by clearing its
 *    counters on `stream`, so calls whose work overlaps on the GPU (other
 *    streams, other host threads) race and give wrong results: order them on
 *    one stream.
 * The caller still owns every input and output buffer, as for mp_dispatch.
 */
#define MP_NOALLOC_SCRATCH_BYTES (1u << 20)
int mp_dispatch_noalloc(int R, int N, int K, int E, int H, int dtype, const void *x,
                        const float *x_scales, const int32_t *topk_idx,
                        const float *topk_weights, const uint32_t *is_token_in_rank,
                        const int32_t *num_tokens_per_rank, const int32_t *num_tokens_per_expert,
                        int64_t recv_capacity, void *recv_x, float *recv_scales,
                        int32_t *recv_src_rank, int32_t *recv_src_idx, int32_t *recv_topk_idx,
                        float *recv_topk_weights, int32_t *dest_offsets, int32_t *rank_prefix,
                        int32_t *num_recv_tokens_per_expert, int32_t *send_row,
                        int32_t *dev_err, mp_stream_t stream);

/*
 * mp_allgatherv_e4m3 / _mxfp8 / _mxfp4 -- [AGV] all-gatherv with the
 * quantisation fused in (the page's note that gathering a list of tensors
 * lets a caller quantise before the all-gather; here data and scales leave
 * one launch together).  Each bf16 row of `in` is quantised once, exactly as
 * mp_dispatch_rows_e4m3 (one fp32 scale per 128 channels) or
 * mp_dispatch_rows_mxfp8 (one UE8M0 byte per 32 channels) quantise a token
 * row, and every logical rank q receives all S rows in order:
 *   sizes       HOST int64 [R], S = sum(sizes) (only S matters: every
 *               rank's gathered copy is the shards in rank order)
 *   in          bf16 [S][H]
 *   out         e4m3 [R][S][H]
 *   out_scales  fp32 [R][S][H/128] (e4m3) or uint8 [R][S][H/32] (mxfp8)
 * The result equals quantising `in` and then calling mp_allgatherv on the
 * codes and on the scales.
 * Checks: 1 <= R <= MP_MAX_RANKS, H > 0 and a multiple of the scale block,
 *   sizes >= 0, non-NULL in/out/out_scales when S > 0, in and out 16-byte
 *   aligned, fp32 scales 4-byte aligned.  No device errors.
 */
int mp_allgatherv_e4m3(int R, int H, const int64_t *sizes, const void *in, void *out,
                       float *out_scales, mp_stream_t stream);
int mp_allgatherv_mxfp8(int R, int H, const int64_t *sizes, const void *in, void *out,
                        uint8_t *out_scales, mp_stream_t stream);
/* The same with MXFP4 (as mp_dispatch_rows_mxfp4): out uint8 [R][S][H/2],
 * out_scales uint8 [R][S][H/32]. */
int mp_allgatherv_mxfp4(int R, int H, const int64_t *sizes, const void *in, void *out,
                        uint8_t *out_scales, mp_stream_t stream);

/*
 * mp_allgatherv_multi -- [AGV] all-gatherv of a list of tensors in one launch
 * (the page's motivation: gathering quantised data and its scales together).
 * Tensor j has row_bytes[j] bytes per row (a multiple of 16) and the same
 * per-rank row counts `sizes`; the result for each tensor is exactly
 * mp_allgatherv(R, row_bytes[j], sizes, in[j], out[j]).
 *   row_bytes  HOST int64 [ntensors]
 *   sizes      HOST int64 [R]
 *   in, out    HOST arrays of ntensors DEVICE pointers (in[j]: [S][row_bytes[j]],
 *              out[j]: [R][S][row_bytes[j]])
 * Checks: R >= 1, 1 <= ntensors <= MP_MAX_TENSORS, row_bytes as above,
 *   sizes >= 0, 16-byte aligned non-NULL pointers when S > 0.
 */
#define MP_MAX_TENSORS 8
int mp_allgatherv_multi(int R, int ntensors, const int64_t *row_bytes, const int64_t *sizes,
                        const void *const *in, void *const *out, mp_stream_t stream);

/*
 * Low-latency expert-major layout ([EP] the low-latency dispatch/combine:
 * per-expert receive buffers, one entry per (token, expert) pair, combine
 * reducing a token's expert outputs with its top-k weights).  Reading used
 * (the pages fix no order): expert e's rows are contiguous, blocks in
 * ascending e; inside a block rows are ordered by source rank, then token.
 * Meant for the small batches of the low-latency mode: the offsets kernel
 * runs one block per source rank (a stable counting sort of that rank's N*K
 * entries), so its time grows with N*K.
 *
 * mp_dispatch_ll_offsets
 *   in   topk_idx               int32 [R][N][K] (-1 = masked)
 *   in   num_tokens_per_expert  int32 [R][E] from mp_layout (same topk_idx), or
 *                               NULL: the call counts the experts itself (each
 *                               of its R blocks reads all R*N*K ids) and then
 *                               flags ids outside [-1, E) with
 *                               MP_ERR_BAD_EXPERT as mp_layout would; this saves
 *                               the mp_layout launch on small batches
 *   out  expert_offsets         int32 [E+1]: first row of expert e; [E] = total
 *   out  expert_src_offsets     int32 [E][R]: rows of e from source ranks < s
 *   out  recv_src_token         int32 [recv_capacity]: flattened s*N + t
 *   out  slot_row               int32 [R][N][K]: row of (s,t) at expert
 *                               topk_idx[s][t][k], or -1 (masked / no room)
 *   Device errors: MP_ERR_CAPACITY (rows past recv_capacity are dropped).
 * mp_dispatch_ll_rows: recv_x[slot_row[s][t][k]] = x[s][t] (and its scales
 *   for MP_E4M3), every entry >= 0 and < recv_capacity; x / recv_x / dtype /
 *   H as mp_dispatch_rows.
 * mp_combine_ll: out[s][t] = bf16( sum over k = 0..K-1 ascending with
 *   slot_row[s][t][k] >= 0 of topk_weights[s][t][k] * float(y[row]) ), each
 *   product and each sum a separate fp32 operation from +0.0f, rounded once
 *   to bf16 (round-to-nearest-even).  y: bf16 [y_rows][H].
 *   Device errors: MP_ERR_CAPACITY for a slot_row entry >= y_rows (skipped).
 */
int mp_dispatch_ll_offsets(int R, int N, int K, int E, const int32_t *topk_idx,
                           const int32_t *num_tokens_per_expert, int64_t recv_capacity,
                           int32_t *expert_offsets, int32_t *expert_src_offsets,
                           int32_t *recv_src_token, int32_t *slot_row, int32_t *dev_err,
                           mp_stream_t stream);
/*
 * mp_dispatch_ll_offsets_rank_major -- the low-latency layout with rank-major
 * output ([EP] the pull request adding rank-major output to the LL path).
 * The same rows as mp_dispatch_ll_offsets (one per token and top-k slot with
 * a valid expert), grouped by the rank d = e / (E/R) that owns the expert;
 * reading (the pages fix no order inside a group): groups in ascending d,
 * inside a group rows ordered by source rank, then token, then top-k slot.
 *   out  dest_offsets      int32 [R+1]: first row of destination d; [R] = total
 *   out  dest_src_offsets  int32 [R][R]: rows of d from source ranks < s
 *   other arguments, checks and device errors as mp_dispatch_ll_offsets
 *   (num_tokens_per_expert may be NULL in the same way).  mp_dispatch_ll_rows
 *   and mp_combine_ll take this slot_row unchanged.
 */
int mp_dispatch_ll_offsets_rank_major(int R, int N, int K, int E, const int32_t *topk_idx,
                                      const int32_t *num_tokens_per_expert,
                                      int64_t recv_capacity, int32_t *dest_offsets,
                                      int32_t *dest_src_offsets, int32_t *recv_src_token,
                                      int32_t *slot_row, int32_t *dev_err, mp_stream_t stream);
/*
 * mp_dispatch_ll -- the low-latency dispatch in one call: the results of
 * mp_dispatch_ll_offsets (rank_major = 0) or mp_dispatch_ll_offsets_rank_major
 * (rank_major = 1) followed by mp_dispatch_ll_rows, bit for bit ("MSCCLPP EP
 * implementation", the low-latency dispatch, one call that both places and
 * sends the tokens).  With num_tokens_per_expert NULL and up to 16,384 ids it
 * is one kernel whose blocks each read every id, place their share of the
 * entries (an entry's row is its bin's first row plus the number of earlier
 * entries of that bin in source-rank, token, slot order) and copy their share
 * of the rows (through shared memory by the bulk-copy engine for rows of 2 KB
 * or more).  Otherwise the row copy is launched as a programmatic dependent of
 * the sort, so its row loads overlap the sort.  Either way x must be complete
 * when the call is enqueued (as for every call, by stream order).
 *   bin_offsets / bin_src_offsets: expert_offsets / expert_src_offsets, or
 *   dest_offsets / dest_src_offsets for rank_major = 1; every other argument
 *   as in those calls (dtype MP_BF16 or MP_E4M3 with its scales).
 *   Device errors: as mp_dispatch_ll_offsets, plus MP_ERR_TIMEOUT if a
 *   block's bounded (~1 s) wait for its bulk load of x gives up.
 */
int mp_dispatch_ll(int R, int N, int K, int E, int H, int dtype, int rank_major, const void *x,
                   const float *x_scales, const int32_t *topk_idx,
                   const int32_t *num_tokens_per_expert, int64_t recv_capacity,
                   int32_t *bin_offsets, int32_t *bin_src_offsets, int32_t *recv_src_token,
                   int32_t *slot_row, void *recv_x, float *recv_scales, int32_t *dev_err,
                   mp_stream_t stream);
int mp_dispatch_ll_rows(int R, int N, int K, int H, int dtype, const void *x,
                        const float *x_scales, const int32_t *slot_row, int64_t recv_capacity,
                        void *recv_x, float *recv_scales, mp_stream_t stream);
int mp_combine_ll(int R, int N, int K, int H, const void *y, int64_t y_rows,
                  const int32_t *slot_row, const float *topk_weights, void *out,
                  int32_t *dev_err, mp_stream_t stream);

/*
 * Formats of the in-kernel quantisation on low-latency dispatch
 * (mp_dispatch_ll_quant, mp_dispatch_ll_rows_quant); each is the per-row
 * quantisation of mp_dispatch_rows_e4m3 / _mxfp8 / _mxfp4.
 *   MP_Q_E4M3   e4m3 codes [cap][H], one fp32 scale per 128 channels
 *               (recv_scales fp32 [cap][H/128]): scale = amax / 448 (1 for an
 *               all-zero block), code = e4m3(x / scale), saturating
 *   MP_Q_MXFP8  e4m3 codes [cap][H], one UE8M0 byte per 32 channels
 *               (recv_scales uint8 [cap][H/32])
 *   MP_Q_MXFP4  two e2m1 codes per byte [cap][H/2] (even channel in the low
 *               nibble), one UE8M0 byte per 32 channels (uint8 [cap][H/32])
 */
#define MP_Q_E4M3 0
#define MP_Q_MXFP8 1
#define MP_Q_MXFP4 2

/*
 * mp_dispatch_ll_rows_quant -- [EP] the low-latency dispatch with the FP8
 * quantisation done in the dispatch kernel (the page's file table lists FP8
 * E4M3 quantisation helpers for LL dispatch; its LL kernel list templates the
 * dispatch on FP8): each bf16 token row is quantised once and its codes and
 * scales are written to every slot row the LL offsets gave it.
 *   x            bf16 [R][N][H]
 *   slot_row     int32 [R][N][K] from mp_dispatch_ll_offsets(_rank_major)
 *   recv_x       codes and recv_scales scales, per qformat (MP_Q_*); rows at
 *                or past recv_capacity are not written
 * Checks: 1 <= R <= 32, 1 <= K <= 32, H a multiple of 128 (MP_Q_E4M3) or 32,
 *   16-byte aligned x / recv_x, non-NULL buffers where rows exist.
 * The result equals quantising x (the per-row definition above) and then
 * copying codes and scales to the slot rows (mp_dispatch_ll_rows).
 */
int mp_dispatch_ll_rows_quant(int R, int N, int K, int H, int qformat, const void *x,
                              const int32_t *slot_row, int64_t recv_capacity, void *recv_x,
                              void *recv_scales, mp_stream_t stream);

/*
 * mp_dispatch_ll_quant -- mp_dispatch_ll with the quantisation done in the row
 * copy: the LL offsets (expert-major, or rank-major with rank_major = 1) and
 * the quantising row copy of mp_dispatch_ll_rows_quant, bit for bit.  With
 * num_tokens_per_expert NULL and up to 16,384 ids (and x 32-byte aligned) one
 * kernel counts, places and quantises (as mp_dispatch_ll); otherwise the
 * quantising copy is launched as the sort's
 * programmatic dependent (its blocks start while the sort runs and wait for
 * its slot rows).  Arguments: those of mp_dispatch_ll, with qformat and
 * void *recv_scales in place of dtype, x_scales and the float scales (x is
 * bf16); checks and device errors as mp_dispatch_ll_offsets and
 * mp_dispatch_ll_rows_quant, plus MP_ERR_TIMEOUT as mp_dispatch_ll.
 */
int mp_dispatch_ll_quant(int R, int N, int K, int E, int H, int qformat, int rank_major,
                         const void *x, const int32_t *topk_idx,
                         const int32_t *num_tokens_per_expert, int64_t recv_capacity,
                         int32_t *bin_offsets, int32_t *bin_src_offsets, int32_t *recv_src_token,
                         int32_t *slot_row, void *recv_x, void *recv_scales, int32_t *dev_err,
                         mp_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MP_LAYOUT_H */
