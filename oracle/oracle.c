/*
 * CPU oracle for single-GPU MoE token dispatch and combine.
 *
 * TEST INFRASTRUCTURE.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark load it.  It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Every function is single-threaded and walks its loops in the order the
 * definition is written.  Compile with -ffp-contract=off so that every
 * multiply and add is a separately rounded f32 operation.
 *
 * Sources (page title, then the note on that page):
 *   [mori448]  ROCm/mori "Draft: cco + flydsl dispatch/combine #448":
 *              - PR description: dispatch scatters each token row once per
 *                destination; combine gathers each token's k expert outputs
 *                and reduces them in f32.
 *              - "Port mori/FlyDSL StdMoE ..." note: convert_dispatch_output
 *                repacks tokens into per-expert buckets packed_x[expert,slot]
 *                with packed_cnt / packed_src and an i64 slot map that holds
 *                -1 for entries that go nowhere; convert_combine_input takes
 *                sum_k wts[k]*packed_x[slot_k]; identity experts telescope to
 *                comb_out[s] == (sum_k wts[s][k]) * input[s].
 *              - "Combine accumulators ... per transport dtype" note: bf16
 *                and f32 inputs are widened to f32 and accumulated in f32.
 *              - "make_dispatch gains scale_dim ..." note: each token's scale
 *                block travels verbatim with its row.
 *              - "... routing handle, LEC, reset, replay" note: a per-expert
 *                token count (local_expert_count).
 *   [moonep34] MoonshotAI/MoonEP "Drop cooperative launch from the
 *              CTA-independent local kernels", "New test": dispatch outputs
 *              are compared bit-exactly against a CPU oracle.
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes):
 *   - slots inside a bucket are handed out in (token, k) order (the pages
 *     hand them out with atomics, whose order is not fixed);
 *   - packed_x is compact: the packed row of (s,k) is off[e] + slot, and
 *     off[] is the exclusive prefix sum of the per-expert counts;
 *   - the i64 token map holds that packed row, or -1 when topk_idx[s,k] is
 *     outside [0, E) (such entries are counted in n_invalid);
 *   - packed_src[row] holds the flat entry index s*K + k;
 *   - combine adds the K weighted terms in increasing k, in f32, with a
 *     separate multiply and add, then rounds to the output dtype (bf16:
 *     round to nearest even);
 *   - dedup groups: expert e belongs to group e / group_size; a token sends
 *     its row once per distinct group, represented by its first entry k in
 *     that group; group rows are ordered by group, then by token.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

enum { ODT_BF16 = 0, ODT_F32 = 1, ODT_FP8_E4M3 = 2 };

/* ------------------------------------------------------------------------
 * Number formats, written from their published definitions.
 * bfloat16: the upper 16 bits of an IEEE-754 binary32 value.
 * E4M3: OCP 8-bit Floating Point Specification (OFP8) v1.0, E4M3 encoding:
 *       1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
 *       is subnormal; S.1111.111 is NaN; there are no infinities.
 * ---------------------------------------------------------------------- */

ORACLE_API float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bfloat16, ties to even. */
ORACLE_API uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN stays NaN (quiet) */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;                        /* truncated result      */
    uint32_t rest = u & 0xffffu;                    /* discarded low half    */
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;                                 /* carries into exponent */
    return (uint16_t)keep;
}

ORACLE_API float oracle_e4m3_to_f32(uint8_t q)
{
    int sign = (q >> 7) & 1;
    int ex = (q >> 3) & 0xf;
    int man = q & 7;
    double v;
    if (ex == 0xf && man == 7)
        return NAN;
    if (ex == 0)
        v = (double)man / 8.0 * pow(2.0, -6);              /* subnormal */
    else
        v = (1.0 + (double)man / 8.0) * pow(2.0, ex - 7);  /* normal    */
    return (float)(sign ? -v : v);
}

/* Round a binary32 value to E4M3, to nearest with ties to even, saturating to
 * +-448 (the largest finite code); NaN maps to the NaN code.  Written from the
 * format definition: the representable magnitudes are m/8 * 2^-6 (m = 0..7,
 * subnormal) and (1 + m/8) * 2^(e-7) (e = 1..15, excluding e=15,m=7).  The
 * candidate codes are walked in increasing magnitude and the nearest is
 * taken; the exact midpoint goes to the code with an even mantissa. */
ORACLE_API uint8_t oracle_f32_to_e4m3(float f)
{
    if (f != f)
        return 0x7f;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    /* largest code whose magnitude is <= a, then compare with the next */
    uint8_t lo = 0;
    for (uint8_t c = 1; c <= 0x7e; ++c) {
        if ((double)oracle_e4m3_to_f32(c) <= a)
            lo = c;
        else
            break;
    }
    if (lo == 0x7e)
        return (uint8_t)(sign | lo);
    double vlo = oracle_e4m3_to_f32(lo);
    double vhi = oracle_e4m3_to_f32((uint8_t)(lo + 1));
    uint8_t code;
    if (a - vlo < vhi - a)
        code = lo;
    else if (a - vlo > vhi - a)
        code = (uint8_t)(lo + 1);
    else
        code = (lo & 1) ? (uint8_t)(lo + 1) : lo;  /* tie: even mantissa */
    return (uint8_t)(sign | code);
}

static float load_elem(const void *base, int dt, int64_t i)
{
    if (dt == ODT_BF16)
        return oracle_bf16_to_f32(((const uint16_t *)base)[i]);
    return ((const float *)base)[i];
}

static void store_elem(void *base, int dt, int64_t i, float v)
{
    if (dt == ODT_BF16)
        ((uint16_t *)base)[i] = oracle_f32_to_bf16(v);
    else
        ((float *)base)[i] = v;
}

/* ------------------------------------------------------------------------
 * Plan [mori448, StdMoE note and local_expert_count]:
 *   cnt[e]       = #{(s,k) : topk_idx[s,k] == e}
 *   off[e]       = sum_{e' < e} cnt[e'],  off[E] = number of valid entries
 *   tok_map[s,k] = off[e] + #{(s',k') before (s,k) in (token, k) order with
 *                  the same expert}, or -1 if topk_idx[s,k] is not in [0,E)
 *   packed_src[tok_map[s,k]] = s*K + k
 * Returns 0, or -1 if a scratch allocation fails.
 * ---------------------------------------------------------------------- */
ORACLE_API int oracle_plan(const int32_t *topk_idx, int64_t S, int K, int E,
                           int32_t *cnt, int64_t *off, int32_t *packed_src,
                           int64_t *tok_map, int32_t *n_invalid)
{
    int64_t n = S * (int64_t)K;
    int32_t invalid = 0;

    /* step 1: per-expert histogram */
    for (int e = 0; e < E; ++e)
        cnt[e] = 0;
    for (int64_t i = 0; i < n; ++i) {
        int32_t e = topk_idx[i];
        if (e >= 0 && e < E)
            cnt[e] += 1;
        else
            invalid += 1;
    }

    /* step 2: exclusive prefix sum */
    off[0] = 0;
    for (int e = 0; e < E; ++e)
        off[e + 1] = off[e] + cnt[e];

    /* step 3: walk entries in (token, k) order, each expert has a cursor */
    int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    if (!cursor)
        return -1;
    for (int e = 0; e < E; ++e)
        cursor[e] = off[e];
    for (int64_t s = 0; s < S; ++s) {
        for (int k = 0; k < K; ++k) {
            int64_t i = s * K + k;
            int32_t e = topk_idx[i];
            if (e >= 0 && e < E) {
                int64_t row = cursor[e];
                cursor[e] += 1;
                tok_map[i] = row;
                packed_src[row] = (int32_t)i;
            } else {
                tok_map[i] = -1;
            }
        }
    }
    free(cursor);
    *n_invalid = invalid;
    return 0;
}

/* ------------------------------------------------------------------------
 * Plan with a per-expert capacity [mori448 op-parity note: receive slots are
 * capped and over-cap tokens take the drop path, no out-of-bounds write].
 * Reading for one GPU: each expert's bucket holds `capacity` rows, bucket e
 * starts at row e*capacity; an entry keeps the slot it would get in the
 * uncapped plan if that slot is below capacity, else it is dropped (-1).
 *   cnt[e] = min(#{(s,k): idx == e}, capacity);  off[e] = e * capacity
 *   tok_map[s,k] = e*capacity + slot if slot < capacity, else -1
 *   packed_src[e*capacity + slot] = s*K + k for the kept entries
 *   n_dropped = valid entries that did not fit
 * ---------------------------------------------------------------------- */
ORACLE_API int oracle_plan_capacity(const int32_t *topk_idx, int64_t S, int K, int E,
                                    int64_t capacity, int32_t *cnt, int64_t *off,
                                    int32_t *packed_src, int64_t *tok_map,
                                    int32_t *n_invalid, int32_t *n_dropped)
{
    int32_t invalid = 0, dropped = 0;
    int64_t *seen = (int64_t *)malloc(sizeof(int64_t) * (size_t)(E > 0 ? E : 1));
    if (!seen)
        return -1;
    for (int e = 0; e < E; ++e)
        seen[e] = 0;
    for (int64_t s = 0; s < S; ++s) {
        for (int k = 0; k < K; ++k) {
            int64_t i = s * K + k;
            int32_t e = topk_idx[i];
            if (e < 0 || e >= E) {
                tok_map[i] = -1;
                invalid += 1;
                continue;
            }
            int64_t slot = seen[e];
            seen[e] += 1;
            if (slot < capacity) {
                tok_map[i] = e * capacity + slot;
                packed_src[e * capacity + slot] = (int32_t)i;
            } else {
                tok_map[i] = -1;
                dropped += 1;
            }
        }
    }
    for (int e = 0; e < E; ++e) {
        cnt[e] = (int32_t)(seen[e] < capacity ? seen[e] : capacity);
        off[e] = (int64_t)e * capacity;
    }
    off[E] = (int64_t)E * capacity;
    free(seen);
    *n_invalid = invalid;
    *n_dropped = dropped;
    return 0;
}

/* ------------------------------------------------------------------------
 * Dedup plan [mori448 PR description: ballot dedup sends a token once per
 * destination; StdMoE note: the receiver's i64 map holds -1 for the
 * token's experts that live elsewhere].  Groups play the destinations.
 *
 *   rep(s,k)  <=> topk_idx[s,k] valid and no k' < k of token s is valid with
 *                 the same group
 *   gcnt[g]   = #{(s,k) : rep(s,k), group(s,k) == g};  goff = exclusive sum
 *   gtok_map[s,k] = goff[g] + #{s' < s : token s' reaches g} if rep(s,k),
 *                   else -1
 *   grp_src[r]    = s*K + k of the representative entry of group row r
 *   grp_tok_map[r,k'] = tok_map[s,k'] if expert (s,k') is valid and in the
 *                       group of row r, else -1
 * ---------------------------------------------------------------------- */
static int group_of(int32_t e, int E, int group_size)
{
    return (e >= 0 && e < E) ? e / group_size : -1;
}

ORACLE_API int oracle_group_plan(const int32_t *topk_idx, const int64_t *tok_map,
                                 int64_t S, int K, int E, int group_size,
                                 int32_t *gcnt, int64_t *goff, int64_t *gtok_map,
                                 int32_t *grp_src, int64_t *grp_tok_map)
{
    int G = E / group_size;

    for (int g = 0; g < G; ++g)
        gcnt[g] = 0;
    for (int64_t s = 0; s < S; ++s) {
        for (int k = 0; k < K; ++k) {
            int g = group_of(topk_idx[s * K + k], E, group_size);
            if (g < 0)
                continue;
            int first = 1;
            for (int kp = 0; kp < k; ++kp)
                if (group_of(topk_idx[s * K + kp], E, group_size) == g)
                    first = 0;
            if (first)
                gcnt[g] += 1;
        }
    }

    goff[0] = 0;
    for (int g = 0; g < G; ++g)
        goff[g + 1] = goff[g] + gcnt[g];

    int64_t *cursor = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G > 0 ? G : 1));
    if (!cursor)
        return -1;
    for (int g = 0; g < G; ++g)
        cursor[g] = goff[g];
    for (int64_t s = 0; s < S; ++s) {
        for (int k = 0; k < K; ++k) {
            int64_t i = s * K + k;
            int g = group_of(topk_idx[i], E, group_size);
            int first = (g >= 0);
            for (int kp = 0; kp < k && first; ++kp)
                if (group_of(topk_idx[s * K + kp], E, group_size) == g)
                    first = 0;
            if (!first) {
                gtok_map[i] = -1;
                continue;
            }
            int64_t r = cursor[g];
            cursor[g] += 1;
            gtok_map[i] = r;
            grp_src[r] = (int32_t)i;
            for (int k2 = 0; k2 < K; ++k2) {
                int g2 = group_of(topk_idx[s * K + k2], E, group_size);
                grp_tok_map[r * K + k2] = (g2 == g) ? tok_map[s * K + k2] : -1;
            }
        }
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------------
 * Dispatch [mori448 PR description and StdMoE note]:
 *   packed[tok_map[s,k]] = rows[s] for every entry with tok_map >= 0.
 * A byte copy; the same call forwards fp8 scale rows [mori448 scale_dim
 * note] with row_bytes = scales per row * 4.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_dispatch(const uint8_t *rows, int64_t S, int64_t row_bytes, int K,
                                const int64_t *tok_map, uint8_t *packed)
{
    for (int64_t s = 0; s < S; ++s)
        for (int k = 0; k < K; ++k) {
            int64_t row = tok_map[s * K + k];
            if (row >= 0)
                memcpy(packed + row * row_bytes, rows + s * row_bytes, (size_t)row_bytes);
        }
}

/* ------------------------------------------------------------------------
 * Blockwise fp8 quantisation of bf16 rows [mori448 Fp8BlockwiseQuant note;
 * the note's formula is garbled, the reading taken: per block of `block`
 * elements, scale = amax / 448 (1 when the block is all zero) and
 * code = E4M3(v / scale), both divisions in f32].  The quantising dispatch
 * is this function followed by oracle_dispatch of the codes and the scales.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_quant_fp8(const uint16_t *x, int64_t S, int64_t H, int block,
                                 uint8_t *q, float *scales)
{
    int64_t nb = H / block;
    for (int64_t s = 0; s < S; ++s)
        for (int64_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int j = 0; j < block; ++j) {
                float v = fabsf(oracle_bf16_to_f32(x[s * H + b * block + j]));
                if (v > amax)
                    amax = v;
            }
            float scale = (amax > 0.0f) ? amax / 448.0f : 1.0f;
            scales[s * nb + b] = scale;
            for (int j = 0; j < block; ++j) {
                float v = oracle_bf16_to_f32(x[s * H + b * block + j]);
                q[s * H + b * block + j] = oracle_f32_to_e4m3(v / scale);
            }
        }
}

/* Dedup dispatch: one copy of x[s] per group row, then the per-expert
 * expansion out of the group rows. */
ORACLE_API void oracle_dispatch_dedup(const uint8_t *x, int64_t R, int64_t row_bytes, int K,
                                      const int32_t *grp_src, const int64_t *grp_tok_map,
                                      uint8_t *grp_x, uint8_t *packed)
{
    for (int64_t r = 0; r < R; ++r) {
        int64_t s = grp_src[r] / K;
        memcpy(grp_x + r * row_bytes, x + s * row_bytes, (size_t)row_bytes);
    }
    for (int64_t r = 0; r < R; ++r)
        for (int k = 0; k < K; ++k) {
            int64_t row = grp_tok_map[r * K + k];
            if (row >= 0)
                memcpy(packed + row * row_bytes, grp_x + r * row_bytes, (size_t)row_bytes);
        }
}

/* ------------------------------------------------------------------------
 * Combine [mori448 PR description, StdMoE and accumulator notes]:
 *   out[s,j] = round( sum_{k : tok_map[s,k] >= 0} w[s,k] * y[tok_map[s,k], j] )
 * with f32 accumulation in increasing k.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_combine(const void *y, int in_dt, const float *w,
                               const int64_t *tok_map, int64_t S, int64_t H, int K,
                               void *out, int out_dt)
{
    for (int64_t s = 0; s < S; ++s)
        for (int64_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t row = tok_map[s * K + k];
                if (row < 0)
                    continue;
                float term = w[s * K + k] * load_elem(y, in_dt, row * H + j);
                acc = acc + term;
            }
            store_elem(out, out_dt, s * H + j, acc);
        }
}

/* Dedup combine [mori448 StdMoE note]: each group row first takes the
 * weighted sum of its own experts' outputs (convert_combine_input); then the
 * token adds its group rows, unweighted, in the order of the token's
 * representative entries (the gather combine summing over destinations). */
ORACLE_API void oracle_combine_dedup(const void *y, int in_dt, const float *w,
                                     int64_t R, const int32_t *grp_src,
                                     const int64_t *grp_tok_map, const int64_t *gtok_map,
                                     int64_t S, int64_t H, int K, float *gtok,
                                     void *out, int out_dt)
{
    for (int64_t r = 0; r < R; ++r) {
        int64_t s = grp_src[r] / K;
        for (int64_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t row = grp_tok_map[r * K + k];
                if (row < 0)
                    continue;
                float term = w[s * K + k] * load_elem(y, in_dt, row * H + j);
                acc = acc + term;
            }
            gtok[r * H + j] = acc;
        }
    }
    for (int64_t s = 0; s < S; ++s)
        for (int64_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t r = gtok_map[s * K + k];
                if (r < 0)
                    continue;
                acc = acc + gtok[r * H + j];
            }
            store_elem(out, out_dt, s * H + j, acc);
        }
}

/* ------------------------------------------------------------------------
 * Combine with the weight fold [mori448 "Combine now reduces the K forwarded
 * per-token weight vectors" note, and the op note whose identity round trip
 * checks comb == U*input and out_weights == U*wts].  The token's whole weight
 * vector travels with every copy of its row; the combine sums the copies it
 * gathers, and folds the travelling weight vectors the same way:
 *   out[s,j] = round( sum_{k : map[s,k] >= 0} c_k * y[map[s,k], j] )
 *              with c_k = w[s,k] when `weighted`, else no factor at all;
 *   ow[s,i]  = sum_{k : map[s,k] >= 0} w[s,i]
 * both in f32, in increasing k.  `map` is any token map into y: tok_map over
 * packed rows, or gtok_map over group rows (one copy per destination group),
 * for which identity rows give out = U*x and ow = U*w, U being the number
 * of the token's groups.  ow may be NULL (no fold).
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_combine_fold(const void *y, int in_dt, const float *w, int weighted,
                                    const int64_t *map, int64_t S, int64_t H, int K,
                                    void *out, int out_dt, float *ow)
{
    for (int64_t s = 0; s < S; ++s)
        for (int64_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t row = map[s * K + k];
                if (row < 0)
                    continue;
                float v = load_elem(y, in_dt, row * H + j);
                acc = acc + (weighted ? w[s * K + k] * v : v);
            }
            store_elem(out, out_dt, s * H + j, acc);
        }
    if (!ow)
        return;
    for (int64_t s = 0; s < S; ++s)
        for (int i = 0; i < K; ++i) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k)
                if (map[s * K + k] >= 0)
                    acc = acc + w[s * K + i];
            ow[s * K + i] = acc;
        }
}

/* ------------------------------------------------------------------------
 * Synthetic expert stages (harness steps between dispatch and combine; not
 * part of the method, but the oracle runs its own copy so that no input of
 * its combine comes from the GPU).
 * ---------------------------------------------------------------------- */

/* y[r] = bf16(f32(packed[r]) * c[e]) for the rows of bucket e. */
ORACLE_API void oracle_expert_scale_bf16(const uint16_t *packed, const int64_t *off, int E,
                                         const float *c, int64_t H, uint16_t *y)
{
    for (int e = 0; e < E; ++e)
        for (int64_t r = off[e]; r < off[e + 1]; ++r)
            for (int64_t j = 0; j < H; ++j)
                y[r * H + j] = oracle_f32_to_bf16(oracle_bf16_to_f32(packed[r * H + j]) * c[e]);
}

/* y[r,j] = bf16(e4m3(q[r,j]) * scale[r, j / block]). */
ORACLE_API void oracle_expert_dequant_fp8(const uint8_t *q, const float *scales, int64_t R,
                                          int64_t H, int block, uint16_t *y)
{
    int64_t nb = H / block;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t j = 0; j < H; ++j)
            y[r * H + j] = oracle_f32_to_bf16(oracle_e4m3_to_f32(q[r * H + j]) *
                                              scales[r * nb + j / block]);
}
