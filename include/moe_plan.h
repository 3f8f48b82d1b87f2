/*
 * moe_plan.h: C ABI of the GB300 (sm_103a) MoE token dispatch / combine
 * library (libmoe_gb300.so).
 *
 * One GPU holds every expert.  A step is
 *   moe_plan      per-expert histogram, exclusive scan, stable slot map
 *   moe_dispatch  scatter each token row into its K per-expert buckets
 *                 (moe_plan_dispatch: both in one launch for small batches)
 *   (expert computation by the caller: packed rows -> expert output rows y)
 *   moe_combine   gather each token's K output rows, weighted f32 sum
 *                 (moe_combine_fold: unweighted or weighted, with the sum
 *                 of the forwarded weight vectors)
 * with a dedup variant (moe_group_plan, moe_dispatch_dedup,
 * moe_combine_dedup) that sends each token once per virtual expert group and
 * expands per expert from there.
 *
 * Sources (page title and the note on it):
 *   ROCm/mori "Draft: cco + flydsl dispatch/combine #448": PR description
 *     (ballot dedup, 16-byte scatter, gather combine reducing in f32), the
 *     StdMoE note (convert_dispatch_output repacks into packed_x[expert,slot]
 *     with packed_cnt, packed_src and an i64 slot map holding -1 for unused
 *     entries; convert_combine_input takes sum_k wts[k]*packed_x[slot_k]),
 *     the scale_dim note (scale rows forwarded verbatim with the token), the
 *     routing-handle note (per-expert token count; replay with a cached map).
 *   ROCm/mori "EPv2 internode dispatch/combine over CCO/GDA": the combine
 *     note on 16-byte load-first gathers and warp slices of whole vector
 *     steps; the config note requiring 16-byte token alignment.
 *   MoonshotAI/MoonEP "Drop cooperative launch from the CTA-independent
 *     local kernels": local kernels need no grid-wide synchronisation.
 *
 * Conventions for every call:
 *   - All buffer arguments are DEVICE pointers owned by the caller; the
 *     library allocates, frees and synchronises nothing and keeps no pointer
 *     after a call returns.  Work is enqueued on `stream` (NULL = legacy
 *     default stream) and runs asynchronously.
 *   - Arrays are dense and row-major.  S = tokens, K = experts per token
 *     (1..32), E = experts (1..1024), H = elements per row.
 *   - Return value: MOE_OK, or an error code.  MOE_EINVAL / MOE_EALIGN are
 *     detected on the host before anything is enqueued.  MOE_ECUDA means a
 *     CUDA call failed; moe_last_cuda_error() returns its error code.
 *     Data-dependent problems are never clamped: an expert id outside
 *     [0, E) is counted in *n_invalid and its entries are marked -1.
 *   - S = 0 is valid: moe_plan still writes zero counts/offsets; the other
 *     calls enqueue nothing.
 *   - No kernel waits for other CTAs or needs the whole GPU (no cooperative
 *     launch; MoonEP page above), so the calls share the GPU with work on
 *     other streams.  Beside a compute-bound kernel (an expert GEMM), a
 *     stream of high priority lets their CTAs take SMs first as they free up.
 */
#ifndef MOE_PLAN_H
#define MOE_PLAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* a cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_EINVAL = 1, /* null pointer, size out of range, bad dtype/group size   */
    MOE_EALIGN = 2, /* a row pointer or row size is not a multiple of 16 bytes */
    MOE_ECUDA = 3   /* a CUDA launch or attribute call failed                  */
} moe_status;

typedef enum {
    MOE_BF16 = 0,    /* bfloat16, 2 bytes                                 */
    MOE_F32 = 1,     /* IEEE binary32, 4 bytes                            */
    MOE_FP8_E4M3 = 2 /* OCP E4M3, 1 byte (dispatch only: a byte copy)     */
} moe_dtype;

/* Library ABI version (this header: 2). */
int moe_version(void);

/* Static text for a status code. */
const char *moe_status_string(int status);

/* The CUDA error code behind the last MOE_ECUDA returned on this host
 * thread (0 if none). */
int moe_last_cuda_error(void);

/* Device-side error bits of the kernels, OR-ed since the last call, which
 * clears them.  Kernels never fault on bad data: they skip the offending row
 * and set a bit instead.
 *   bit 0  dispatch: a bounded wait for a staged row ran out of time (the
 *          kernel stopped early; its output is incomplete)
 *   bit 1  dispatch (moe_dispatch*, moe_plan_dispatch): a map entry pointed
 *          outside the source or destination buffer (that row was not
 *          copied)
 *   bit 2  combine: a map entry pointed outside y, or a group row's source
 *          entry outside topk_w (that term was dropped)
 *   bit 3  reserved for a combine that waits on staged rows; the combine
 *          kernels of this version never wait and never set it
 * flags: HOST pointer to one uint32.  Synchronous: waits for the device. */
int moe_device_errors(uint32_t *flags);

/* Self-test of the bounded-wait path (the pages have no counterpart; the
 * dispatch kernels' mbarrier waits give up after 2 s and report instead of
 * hanging).  Enqueues one warp that waits, through the same bounded wait, on
 * an mbarrier phase that nothing will ever complete; after limit_ns
 * nanoseconds (1e3 .. 1e8, else MOE_EINVAL) it sets bit 0 of
 * moe_device_errors and returns.  No memory of the caller is touched and the
 * CUDA context stays usable.  Asynchronous on `stream`. */
int moe_selftest_wait_timeout(int64_t limit_ns, moe_stream_t stream);

/* Self-test of the number-format conversions the kernels use [mori #448:
 * Fp8BlockwiseQuant notes (the fp8 cast of each scaled element) and the
 * accumulator note (f32 sums stored back as bf16)]: for i in [0, count) the
 * binary32 value with bit pattern first + i is converted
 *   - to E4M3 exactly as the quantising dispatch casts its quotients (OCP
 *     OFP8 v1.0 E4M3, round to nearest even, saturated to +-448, NaN to a
 *     NaN code) into e4m3_out[i], when e4m3_out is not NULL;
 *   - to bfloat16 exactly as the combines store their f32 sums (round to
 *     nearest even) into bf16_out[i], when bf16_out is not NULL.
 * first and count: multiples of 4, first + count <= 2^32 (the whole
 * binary32 range in one call needs 4 GiB of e4m3_out and 8 GiB of bf16_out).
 * e4m3_out [count] u8, bf16_out [count] u16: DEVICE pointers, 16-byte
 * aligned, owned by the caller; at least one of them set.
 * Errors: MOE_EINVAL (ranges, both outputs NULL), MOE_EALIGN; asynchronous on
 * `stream`. */
int moe_selftest_convert(uint32_t first, int64_t count, uint8_t *e4m3_out, uint16_t *bf16_out,
                         moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Plan  [mori #448: StdMoE note (packed_cnt, packed_src, i64 slot map with
 * -1) and routing-handle note (local_expert_count)].
 *
 *   cnt[e]        = number of entries (s,k) with topk_idx[s,k] == e
 *   off[e]        = sum of cnt[e'] for e' < e; off[E] = valid entries
 *   tok_map[s,k]  = off[e] + (number of entries before (s,k) in (token, k)
 *                   order that chose the same expert), or -1 when topk_idx
 *                   [s,k] is outside [0, E)
 *   packed_src[r] = s*K + k of the entry whose packed row is r, r < off[E]
 *   n_invalid[0]  = number of entries outside [0, E)
 *
 * Slots are handed out in (token, k) order, so the result is a pure function
 * of topk_idx (the pages allocate slots with atomics; this library does not).
 *
 * topk_idx   int32 [S, K]            device, read
 * cnt        int32 [E]               device, written
 * off        int64 [E + 1]           device, written
 * packed_src int32 [S * K]           device, first off[E] entries written
 * tok_map    int64 [S, K]            device, written
 * n_invalid  int32 [1]               device, written
 * workspace  moe_plan_workspace_size(S, K, E) bytes of device scratch,
 *            256-byte aligned (NULL allowed when that size is 0); contents
 *            need no initialisation and are dead after the call.
 * Limits: S*K < 2^31, 1 <= K <= 32, 1 <= E <= 1024.
 * ---------------------------------------------------------------------- */
size_t moe_plan_workspace_size(int64_t S, int K, int E);

int moe_plan(const int32_t *topk_idx, int64_t S, int K, int E,
             int32_t *cnt, int64_t *off, int32_t *packed_src, int64_t *tok_map,
             int32_t *n_invalid, void *workspace, size_t workspace_bytes,
             moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Plan with a per-expert capacity  [mori #448 op-parity note: receive slots
 * are capped; over-cap tokens take the drop path, with no out-of-bounds
 * write].  Padded buckets: bucket e holds rows [e*capacity, (e+1)*capacity).
 * Entry (s,k) keeps the slot it has in moe_plan's order if that slot is
 * below capacity (earlier tokens first), else it is dropped:
 *   cnt[e]        = min(entries of e, capacity);   off[e] = e * capacity
 *   tok_map[s,k]  = e*capacity + slot, or -1 (dropped or id outside [0,E))
 *   packed_src[e*capacity + slot] = s*K + k for kept entries; rows at or
 *                   past cnt[e] in a bucket are left untouched
 *   n_dropped[0]  = valid entries that did not fit
 * packed_src int32 [E * capacity]; workspace as moe_plan_workspace_size.
 * dispatch/combine then take packed_rows = E * capacity.
 * Limits: as moe_plan; capacity >= 1 and E * capacity < 2^31.
 * ---------------------------------------------------------------------- */
int moe_plan_capacity(const int32_t *topk_idx, int64_t S, int K, int E, int64_t capacity,
                      int32_t *cnt, int64_t *off, int32_t *packed_src, int64_t *tok_map,
                      int32_t *n_invalid, int32_t *n_dropped, void *workspace,
                      size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Plan without a caller-supplied workspace.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory for
 * a workspace, such as a C or C++ host linking only this library with no
 * device allocator of its own, or a process whose device memory belongs to a
 * pool that forbids further cudaMalloc calls.
 *
 * Same arguments, outputs and errors as moe_plan, minus the workspace.  The
 * tile histograms live in a 256 KiB array inside the library image that
 * every GPU loading the library holds until the process exits; this call
 * allocates and frees nothing.  Plans whose moe_plan_workspace_size exceeds
 * 256 KiB are rejected with MOE_EINVAL (every plan with E <= 511 fits, and
 * so does every plan of up to 131,072 entries S*K, which needs no scratch).
 *
 * The first call on a device (with that device current) looks up the
 * array's device address once; make that first call before any stream
 * capture.  The address is kept for the rest of the process: do not call
 * cudaDeviceReset on a device after using this entry point on it.  All calls share the array and it keeps the last call's contents;
 * nothing in it needs to start at zero, because each call overwrites every
 * entry it reads.  Calls that overlap on the GPU (e.g. issued on two
 * streams, or from two host threads) race on the array: do not overlap them.
 * ---------------------------------------------------------------------- */
int moe_plan_static_scratch(const int32_t *topk_idx, int64_t S, int K, int E,
                            int32_t *cnt, int64_t *off, int32_t *packed_src,
                            int64_t *tok_map, int32_t *n_invalid, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Dedup plan  [mori #448: PR description (ballot dedup: one copy of a token
 * per destination) and StdMoE note (the receiver's i64 map holds -1 for the
 * token's experts that live elsewhere)].  Virtual group of expert e is
 * e / group_size; G = E / group_size groups.
 *
 * Entry (s,k) represents group g when topk_idx[s,k] is valid, lies in g, and
 * no earlier k' of token s lies in g.  Group rows are ordered by group, then
 * by token.
 *   gcnt[g]          = group rows of group g;  goff = exclusive prefix sum,
 *                      goff[G] = R, the number of group rows
 *   gtok_map[s,k]    = group row of (s,k) if it represents its group, else -1
 *   grp_src[r]       = s*K + k of the representative of group row r
 *   grp_tok_map[r,k] = tok_map[s,k] when expert (s,k) belongs to the group of
 *                      row r, else -1   (s = grp_src[r] / K)
 *
 * tok_map      int64 [S, K]  from moe_plan on the same topk_idx
 * gcnt         int32 [G]; goff int64 [G + 1]; gtok_map int64 [S, K]
 * grp_src      int32 [S * min(K, G)]        first R entries written
 * grp_tok_map  int64 [S * min(K, G), K]     first R rows written
 * workspace    moe_group_plan_workspace_size(S, K, E, group_size) bytes of
 *              device scratch, 256-byte aligned, contents dead after the
 *              call: the per-tile counts of a first kernel, so that each
 *              tile is counted once.  Up to 131072 entries S*K it may be NULL
 *              (or smaller); the plan then runs in one launch whose CTAs
 *              count all entries themselves, which is slower (26.6 against
 *              12.3 us at S=4096, K=8, 8 groups).
 * Limits: as moe_plan; group_size >= 1 divides E.
 * ---------------------------------------------------------------------- */
size_t moe_group_plan_workspace_size(int64_t S, int K, int E, int group_size);

int moe_group_plan(const int32_t *topk_idx, const int64_t *tok_map, int64_t S, int K,
                   int E, int group_size, int32_t *gcnt, int64_t *goff,
                   int64_t *gtok_map, int32_t *grp_src, int64_t *grp_tok_map,
                   void *workspace, size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Dispatch  [mori #448: PR description (16-byte scatter of each token row),
 * StdMoE note (packed_x[expert, slot]), scale_dim note (scale rows travel
 * verbatim)].
 *
 *   packed_x[tok_map[s,k], :] = x[s, :]          for every tok_map[s,k] >= 0
 *   packed_scales[tok_map[s,k], :] = x_scales[s, :]   (when n_scales > 0)
 * Rows of packed_x that no entry maps to are left untouched.
 *
 * x             [S, H] of `dtype` (a byte copy: any dtype of that size)
 * tok_map       int64 [S, K] from moe_plan or moe_plan_capacity
 * packed_x      [packed_rows, H] of `dtype`: off[E] rows suffice (S*K always
 *               do for moe_plan; E*capacity for moe_plan_capacity); a map
 *               entry at or past packed_rows is skipped and flagged (bit 1
 *               of moe_device_errors)
 * x_scales      f32 [S, n_scales] or NULL when n_scales == 0 (n_scales <= 256)
 * packed_scales f32 [packed_rows, n_scales] or NULL when n_scales == 0
 * Alignment: x, packed_x, x_scales, packed_scales 16-byte aligned; H*size
 * and n_scales*4 multiples of 16 (else MOE_EALIGN).
 * ---------------------------------------------------------------------- */
int moe_dispatch(const void *x, int64_t S, int64_t H, int dtype, int K,
                 const int64_t *tok_map, void *packed_x, int64_t packed_rows,
                 const float *x_scales, int64_t n_scales, float *packed_scales,
                 moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Quantising dispatch  [mori #448: Fp8BlockwiseQuant notes (per-block amax,
 * f32 scale, fp8 cast; block amax by a lane butterfly) and scale_dim note].
 * Reads each bf16 row once and writes it, quantised, to its K packed rows:
 *   for every block b of `block` elements of x[s]:
 *     scale = amax_b / 448 (1 if the block is all zero), IEEE f32 division
 *     packed_q[r, j]            = E4M3(x[s, j] / scale)  (nearest even,
 *                                 saturating to +-448; IEEE f32 division)
 *     packed_scales[r, b]       = scale
 *   for every r = tok_map[s,k] >= 0.  x must hold finite values.
 * x              bf16 [S, H]; H a multiple of block
 * block          16, 32, 64, 128 or 256
 * packed_q       uint8 [packed_rows, H] (E4M3 codes); off[E] rows suffice
 * packed_scales  f32 [packed_rows, H / block]
 * Alignment: x and packed_q 16-byte aligned, packed_scales 4-byte aligned.
 * ---------------------------------------------------------------------- */
int moe_dispatch_quant_fp8(const void *x, int64_t S, int64_t H, int K,
                           const int64_t *tok_map, int block, void *packed_q,
                           float *packed_scales, int64_t packed_rows, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Plan and dispatch in one call  [ROCm/mori "EPv2 internode dispatch/combine
 * over CCO/GDA": a throughput and a low-latency kernel family, chosen per
 * call below a token-count crossover (512 tokens on that page); mori #448
 * StdMoE note for the outputs].
 *
 * Computes exactly what moe_plan followed by moe_dispatch computes: the same
 * cnt, off, packed_src, tok_map, n_invalid, packed_x and packed_scales, with
 * the same arguments, layouts and rules as those two calls.  One kernel does
 * both when 0 < S*K <= moe_plan_dispatch_fused_max() (every CTA ranks all
 * entries in shared memory) and when S*K <= 131072 with at most 1024 entries
 * per SM's share of the tokens and at most 192 MiB of rows to copy (each CTA
 * owns a token range: it counts all entries, ranks its own and copies its
 * own rows); the workspace is then not used.  Otherwise the call enqueues
 * moe_plan then moe_dispatch (whose grid balances the copy across SMs), and
 * `workspace` follows moe_plan's rule (moe_plan_workspace_size).  All
 * arguments are checked before anything is enqueued.
 * ---------------------------------------------------------------------- */
int64_t moe_plan_dispatch_fused_max(void);
int moe_plan_dispatch(const int32_t *topk_idx, const void *x, int64_t S, int64_t H,
                      int dtype, int K, int E, const float *x_scales, int64_t n_scales,
                      int32_t *cnt, int64_t *off, int32_t *packed_src, int64_t *tok_map,
                      int32_t *n_invalid, void *packed_x, int64_t packed_rows,
                      float *packed_scales, void *workspace, size_t workspace_bytes,
                      moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Dedup dispatch  [mori #448: ballot-dedup send, then convert_dispatch_output
 * per (received token, k)].  Writes, on `stream`:
 *   grp_x[r, :]                = x[grp_src[r] / K, :]          r < R = goff[G]
 *   packed_x[grp_tok_map[r,k]] = grp_x[r, :]      for grp_tok_map[r,k] >= 0
 * gtok_map (moe_group_plan) gives each token's group rows.  For K <= 16 one
 * pass walks tokens: each chunk of x[s] is staged once and stored to the
 * token's group rows and to its experts' packed rows, so x is read once; for
 * 16 < K < 32 one pass walks group rows (x[s] is read once per group row);
 * K = 32 takes two passes, the second reading grp_x.
 * max_rows: rows allocated for grp_x (and grp_src/grp_tok_map); must be at
 * least S * min(K, G), which bounds R.
 * packed_x  [packed_rows, H] of `dtype`: the rows the plan behind grp_tok_map
 *           addresses (off[E] rows suffice; S*K for moe_plan, E*capacity for
 *           moe_plan_capacity); a map entry at or past packed_rows is skipped
 *           and flagged (bit 1 of moe_device_errors).  packed_rows >= 1.
 * Alignment as moe_dispatch.
 * ---------------------------------------------------------------------- */
int moe_dispatch_dedup(const void *x, int64_t S, int64_t H, int dtype, int K, int G,
                       const int64_t *goff, const int32_t *grp_src,
                       const int64_t *grp_tok_map, const int64_t *gtok_map,
                       int64_t max_rows, void *grp_x, void *packed_x, int64_t packed_rows,
                       moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine  [mori #448: PR description (gather each token's k expert outputs,
 * reduce in f32), StdMoE note (sum_k wts[k]*packed_x[slot_k]), accumulator
 * note (bf16/f32 widened to f32); mori EPv2 combine note (16-byte load-first
 * gather, whole vector steps per warp)].
 *
 *   out[s, j] = round_out( sum over k = 0..K-1 with tok_map[s,k] >= 0 of
 *                          topk_w[s,k] * y[tok_map[s,k], j] )
 * The sum is taken in f32 in increasing k, each product and each sum rounded
 * separately (no fused multiply-add); bf16 output rounds to nearest even.
 *
 * y       [y_rows, H] of in_dtype (MOE_BF16 or MOE_F32), 1 <= y_rows < 2^31;
 *         a map entry at or past y_rows, or below -1, drops its term and is
 *         flagged (bit 2)
 * topk_w  f32 [S, K]; tok_map int64 [S, K] from moe_plan
 * out     [S, H] of out_dtype (MOE_BF16 or MOE_F32)
 * Alignment: y, out 16-byte aligned; H a multiple of 8.
 * ---------------------------------------------------------------------- */
int moe_combine(const void *y, int64_t y_rows, int in_dtype, const float *topk_w,
                const int64_t *tok_map, int64_t S, int64_t H, int K, void *out,
                int out_dtype, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Dedup combine  [mori #448 StdMoE note: convert_combine_input per received
 * token, then the gather combine sums over destinations].  Two stages:
 *   gtok[r, j] = sum over k with grp_tok_map[r,k] >= 0 of
 *                topk_w[s,k] * y[grp_tok_map[r,k], j]     (f32, s = grp_src[r]/K)
 *   out[s, j]  = round_out( sum over k with gtok_map[s,k] >= 0 of
 *                           gtok[gtok_map[s,k], j] )      (f32, unweighted)
 * gtok: f32 [max_rows, H], written with the group-row sums (the per-group
 * result; it may be read afterwards).  For K <= 8 one pass computes both
 * sums from the same gathers, in the order above, and never reads gtok back
 * (the weights of a group row are then read from the token's own row, which
 * is grp_src[r] / K in a plan from moe_group_plan); larger K takes two
 * passes.
 * y        [y_rows, H] of in_dtype, the expert outputs in the packed order of
 *          the plan behind grp_tok_map (S*K rows for moe_plan, E*capacity for
 *          moe_plan_capacity), 1 <= y_rows < 2^31; an entry at or past y_rows
 *          drops its term and is flagged (bit 2)
 * max_rows >= S * min(K, G).  Alignment as moe_combine.
 * ---------------------------------------------------------------------- */
int moe_combine_dedup(const void *y, int64_t y_rows, int in_dtype, const float *topk_w,
                      const int64_t *goff, int G, const int32_t *grp_src,
                      const int64_t *grp_tok_map, const int64_t *gtok_map, int64_t S,
                      int64_t H, int K, int64_t max_rows, float *gtok, void *out,
                      int out_dtype, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine with the weight fold  [mori #448: the combine-weight-fold note (the
 * K per-token weight vectors forwarded with the copies are reduced into
 * out_weights, once per token in the gather's first part) and the op note
 * (identity round trip: comb == U*input, out_weights == U*wts, U = the
 * token's distinct destinations); mori EPv2 v2-native note (same golden)].
 *
 *   out[s, j]         = round_out( sum over k with map[s,k] >= 0 of
 *                                  c_k * y[map[s,k], j] )
 *                       c_k = topk_w[s,k] if weighted == 1; no factor if 0
 *   out_weights[s, i] = sum over k with map[s,k] >= 0 of topk_w[s, i]
 * Both sums in f32, increasing k, separately rounded; bf16 output rounds to
 * nearest even.  weighted == 1 with out_weights == NULL is moe_combine.
 *
 * map     int64 [S, K]: any token map into y -- tok_map from moe_plan (rows
 *         of y = expert outputs in packed order) or gtok_map from
 *         moe_group_plan (rows of y = one output row per (token, group),
 *         e.g. the group rows of moe_dispatch_dedup after a per-group stage)
 * y       [y_rows, H] of in_dtype (MOE_BF16 or MOE_F32), 1 <= y_rows < 2^31;
 *         an entry at or past y_rows drops its term and is flagged (bit 2)
 * topk_w  f32 [S, K]; may be NULL only when weighted == 0 and
 *         out_weights == NULL
 * out     [S, H] of out_dtype; out_weights f32 [S, K] (4-byte aligned) or
 *         NULL for no fold
 * Alignment as moe_combine.  weighted other than 0 or 1 is MOE_EINVAL.
 * ---------------------------------------------------------------------- */
int moe_combine_fold(const void *y, int64_t y_rows, int in_dtype, const float *topk_w,
                     int weighted, const int64_t *map, int64_t S, int64_t H, int K,
                     void *out, int out_dtype, float *out_weights, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_PLAN_H */
