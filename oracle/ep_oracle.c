/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for MoE token
 * dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file.  Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC.
 * -ffp-contract=off matters: every product and every sum below is rounded on
 * its own, exactly as written.
 *
 * What is computed, and where it comes from (the pages are the five DeepEP
 * web pages; the benchmark spec fixes the formulas the pages leave open):
 *
 *  - layout: per-expert token counts ("Redundant atomics in internode_ll",
 *    the quoted low-latency dispatch excerpt: counts kept per expert), expert
 *    to partition mapping by integer division of the expert id by the number
 *    of experts per partition (same excerpt: destination rank and local
 *    expert index), and an order that keeps the source order inside each
 *    expert ("Reasons for not calling NVSHMEM public APIs?", the answer on
 *    low-latency mode: data for one expert stays in order).
 *  - dispatch: each token's hidden row is copied to every expert it is routed
 *    to ("Pipeline direct NVLink dispatch with triple-buffered prefetch",
 *    Summary: hidden data, scale factors, metadata and routing travel per
 *    token); optionally cast to FP8 e4m3 with one fp32 scale per 128
 *    channels, scale = amax / 448 rounded to nearest in fp32.
 *  - combine: the weighted sum of a token's k expert outputs, accumulated in
 *    fp32 in slot order and rounded once to bf16 (same PR, Validation table:
 *    combine is the reverse of dispatch and is measured beside it).
 *
 * Every function is pinned by tests that do not re-type its formula: a
 * library stable sort, torch's own e4m3/bf16 conversions, an fp64
 * recomputation inside a derived error bound, invariants and hand-worked
 * examples.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* bf16: the upper 16 bits of an IEEE-754 binary32.                     */
/* ------------------------------------------------------------------ */

static float bf16_bits_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to the even bf16. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) {       /* NaN stays a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t dropped = u & 0xffffu;               /* the 16 bits cut off  */
    uint32_t kept = u >> 16;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) {
        kept += 1u;                               /* carries into exponent */
    }
    return (uint16_t)kept;
}

/* ------------------------------------------------------------------ */
/* FP8 e4m3 ("e4m3fn" in the OCP 8-bit float format): sign bit, 4       */
/* exponent bits with bias 7, 3 mantissa bits; no infinities; S.1111.111*/
/* is NaN; exponent field 0 holds subnormals m * 2^-9.  Largest finite  */
/* value 1.75 * 2^8 = 448.                                              */
/* ------------------------------------------------------------------ */

/* Value of a code, from the format definition.  NaN codes give NAN. */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int efield = (code >> 3) & 0xF;
    int m = code & 0x7;
    double mag;
    if (efield == 0xF && m == 0x7) {
        return NAN;
    }
    if (efield == 0) {
        mag = ldexp((double)m, -9);               /* subnormal: m/8 * 2^-6 */
    } else {
        mag = ldexp(1.0 + m / 8.0, efield - 7);
    }
    return sign ? -mag : mag;
}

/*
 * Round a binary32 to e4m3, nearest with ties to the even code, saturating
 * to +-448 instead of overflowing ("satfinite").  The non-negative finite
 * codes 0x00..0x7E are increasing in value, so the nearest code is found by
 * bisection over them and one midpoint comparison.  The sign is kept, also
 * for results that round to zero.
 */
uint8_t oracle_e4m3_encode(float v)
{
    if (isnan(v)) {
        return 0x7F;
    }
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) {
        /* Below 464 the nearest value is 448; 464 is a tie between 448 (even
         * mantissa) and 480 (not finite in this format); above it the result
         * overflows.  Saturation makes all of them 448. */
        return (uint8_t)(sign | 0x7E);
    }
    int lo = 0, hi = 0x7E;                       /* value(lo) <= a always  */
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_value((uint8_t)mid) <= a) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    int c = lo;                                  /* value(c) <= a < value(c+1) */
    double below = oracle_e4m3_value((uint8_t)c);
    double above = oracle_e4m3_value((uint8_t)(c + 1));
    double twice_a = 2.0 * a;                    /* exact in binary64      */
    double sum = below + above;                  /* exact: few mantissa bits */
    int code;
    if (twice_a < sum) {
        code = c;
    } else if (twice_a > sum) {
        code = c + 1;
    } else {
        code = (c % 2 == 0) ? c : c + 1;         /* tie: even mantissa     */
    }
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------ */
/* Layout                                                               */
/* ------------------------------------------------------------------ */

enum { ORACLE_PACKED = 0, ORACLE_CAPACITY = 1 };
enum { ORACLE_ERR_BAD_EXPERT = 1u, ORACLE_ERR_CAPACITY = 2u };

/*
 * topk_idx is [T, k] row-major.  An entry of -1 is a masked slot; any other
 * value outside [0, E) is an error (bit 0 of *err) and is treated as masked.
 *
 * counts[e]     = number of (t, j) routed to expert e (true demand).
 * offsets[e]    = sum of counts[e'] for e' < e; offsets[E] = total.
 * part_counts / part_offsets: the same over partitions of E/P consecutive
 *                 experts each.
 * Rows are handed out per expert in (t, j) row-major order.  The rank of a
 * copy is the number of earlier copies of the same expert.
 *   packed:   slot = offsets[e] + rank, R = T*k rows.
 *   capacity: slot = e*cap + rank if rank < cap, else -1 (bit 1 of *err);
 *             R = E*cap rows.
 * slot_of[t*k+j] = slot (-1 if masked or dropped); src_token[slot] = t and
 * src_k[slot] = j for every placed copy, -1 in rows that hold no copy.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_layout(int T, int E, int k, int P, int mode, int cap,
                  const int32_t *topk_idx,
                  int32_t *counts, int32_t *offsets,
                  int32_t *part_counts, int32_t *part_offsets,
                  int32_t *slot_of, int32_t *src_token, int32_t *src_k,
                  uint32_t *err)
{
    if (T < 0 || E < 1 || k < 1 || P < 1 || E % P != 0) return -1;
    if (mode == ORACLE_CAPACITY && cap < 1) return -1;
    long N = (long)T * k;
    long R = (mode == ORACLE_PACKED) ? N : (long)E * cap;
    *err = 0;

    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long n = 0; n < N; ++n) {
        int e = topk_idx[n];
        if (e == -1) continue;
        if (e < -1 || e >= E) { *err |= ORACLE_ERR_BAD_EXPERT; continue; }
        counts[e] += 1;
    }

    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];

    int per = E / P;
    part_offsets[0] = 0;
    for (int p = 0; p < P; ++p) {
        int s = 0;
        for (int e = p * per; e < (p + 1) * per; ++e) s += counts[e];
        part_counts[p] = s;
        part_offsets[p + 1] = part_offsets[p] + s;
    }

    for (long r = 0; r < R; ++r) { src_token[r] = -1; src_k[r] = -1; }

    int32_t *seen = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    if (!seen) return -1;
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            long n = (long)t * k + j;
            int e = topk_idx[n];
            if (e < 0 || e >= E) { slot_of[n] = -1; continue; }
            int rank = seen[e];
            seen[e] += 1;
            long slot;
            if (mode == ORACLE_PACKED) {
                slot = offsets[e] + rank;
            } else if (rank < cap) {
                slot = (long)e * cap + rank;
            } else {
                slot = -1;
                *err |= ORACLE_ERR_CAPACITY;
            }
            slot_of[n] = (int32_t)slot;
            if (slot >= 0) { src_token[slot] = t; src_k[slot] = j; }
        }
    }
    free(seen);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Dispatch                                                             */
/* ------------------------------------------------------------------ */

/*
 * bf16 dispatch: recv[slot_of[t,j], :] = x[t, :] bit for bit, for every
 * slot >= 0; recv_w[slot] = topk_w[t, j] when both pointers are given.
 * Rows of recv that receive no copy are not touched.
 */
void oracle_dispatch_bf16(int T, int H, int k, const uint16_t *x,
                          const int32_t *slot_of, const float *topk_w,
                          uint16_t *recv, float *recv_w)
{
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            long slot = slot_of[(long)t * k + j];
            if (slot < 0) continue;
            for (int i = 0; i < H; ++i) {
                recv[slot * H + i] = x[(long)t * H + i];
            }
            if (topk_w && recv_w) recv_w[slot] = topk_w[(long)t * k + j];
        }
    }
}

/*
 * fp8 dispatch.  For token t and channel block b (channels 128b .. 128b+127):
 *   amax = max |x[t,i]| over the block (exact),
 *   s    = max(amax, 1e-4) / 448       (fp32 division, round to nearest;
 *                                       the 1e-4 floor keeps s > 0 for an
 *                                       all-zero block, where q is then 0),
 *   q_i  = e4m3(x[t,i] / s)            (fp32 division, then nearest e4m3,
 *                                       ties to even, saturating).
 * q goes to recv_q[slot, 128b..] and s to recv_s[slot, b] (recv_s is
 * [R, H/128] row-major) for every slot of the token.  H % 128 == 0.
 */
void oracle_dispatch_fp8(int T, int H, int k, const uint16_t *x,
                         const int32_t *slot_of, const float *topk_w,
                         uint8_t *recv_q, float *recv_s, float *recv_w)
{
    int nb = H / 128;
    uint8_t q[128];
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t *xb = x + (long)t * H + (long)b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16_bits_to_f32(xb[i]));
                if (a > amax) amax = a;
            }
            float floor_amax = (amax > 1e-4f) ? amax : 1e-4f;
            float s = floor_amax / 448.0f;
            for (int i = 0; i < 128; ++i) {
                float v = bf16_bits_to_f32(xb[i]) / s;
                q[i] = oracle_e4m3_encode(v);
            }
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot < 0) continue;
                memcpy(recv_q + slot * H + (long)b * 128, q, 128);
                recv_s[slot * nb + b] = s;
            }
        }
        if (topk_w && recv_w) {
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot >= 0) recv_w[slot] = topk_w[(long)t * k + j];
            }
        }
    }
}

/*
 * fp8 dispatch with UE8M0 scales (an unsigned 8-bit exponent: the scale is a
 * power of two; "Redundant atomics in internode_ll" cross-references PR
 * "Support UE8M0 data format").  Per token t and block b:
 *   v  = max(amax, 1e-4) / 448               (fp32 division, round to nearest),
 *   s  = the smallest power of two >= v,
 *   q_i = e4m3(x[t,i] / s)                   (exact: s is a power of two),
 * recv_e[slot, b] = biased exponent of s (s = 2^(recv_e - 127)).
 */
void oracle_dispatch_fp8_ue8m0(int T, int H, int k, const uint16_t *x,
                               const int32_t *slot_of, const float *topk_w,
                               uint8_t *recv_q, uint8_t *recv_e, float *recv_w)
{
    int nb = H / 128;
    uint8_t q[128];
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t *xb = x + (long)t * H + (long)b * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float a = fabsf(bf16_bits_to_f32(xb[i]));
                if (a > amax) amax = a;
            }
            float v = ((amax > 1e-4f) ? amax : 1e-4f) / 448.0f;
            int ev;
            float mant = frexpf(v, &ev);          /* v = mant * 2^ev, mant in [0.5, 1) */
            float s = (mant == 0.5f) ? v : ldexpf(1.0f, ev);
            int es;
            (void)frexpf(s, &es);                 /* s = 0.5 * 2^es = 2^(es-1) */
            uint8_t e8 = (uint8_t)(es - 1 + 127);
            for (int i = 0; i < 128; ++i) {
                q[i] = oracle_e4m3_encode(bf16_bits_to_f32(xb[i]) / s);
            }
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot < 0) continue;
                memcpy(recv_q + slot * H + (long)b * 128, q, 128);
                recv_e[slot * nb + b] = e8;
            }
        }
        if (topk_w && recv_w) {
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot >= 0) recv_w[slot] = topk_w[(long)t * k + j];
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Combine                                                              */
/* ------------------------------------------------------------------ */

/*
 * out[t, i] = bf16( sum over j = 0..k-1 with slot = slot_of[t,j] >= 0 of
 *                   topk_w[t,j] * y[slot, i] ),
 * the sum taken in fp32 in increasing j starting from 0, each product and
 * each addition rounded on its own; a token with no valid slot gives 0.
 */
void oracle_combine(int T, int H, int k, const uint16_t *y,
                    const float *topk_w, const int32_t *slot_of,
                    uint16_t *out)
{
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < H; ++i) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot < 0) continue;
                float prod = topk_w[(long)t * k + j] * bf16_bits_to_f32(y[slot * H + i]);
                acc = acc + prod;
            }
            out[(long)t * H + i] = oracle_f32_to_bf16(acc);
        }
    }
}

/*
 * combine of fp8 expert outputs: y is e4m3 [R, H] with one scale per 128
 * channels, ys [R, H/128] (f32, or UE8M0 exponent bytes when ue8m0 != 0).
 * Each element is dequantised as v = value(q) * s (fp32 product, rounded to
 * nearest; value(q) is exact in fp32), then summed as in oracle_combine:
 * out[t, i] = bf16( sum over valid j of w[t,j] * v ), fp32, increasing j.
 * topk_w may be NULL (unweighted sum).
 */
void oracle_combine_fp8(int T, int H, int k, const uint8_t *y, const void *ys, int ue8m0,
                        const float *topk_w, const int32_t *slot_of, uint16_t *out)
{
    int nb = H / 128;
    for (int t = 0; t < T; ++t) {
        for (int i = 0; i < H; ++i) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                long slot = slot_of[(long)t * k + j];
                if (slot < 0) continue;
                float s;
                if (ue8m0) {
                    s = ldexpf(1.0f, (int)((const uint8_t *)ys)[slot * nb + i / 128] - 127);
                } else {
                    s = ((const float *)ys)[slot * nb + i / 128];
                }
                float v = (float)oracle_e4m3_value(y[slot * H + i]) * s;
                float w = topk_w ? topk_w[(long)t * k + j] : 1.0f;
                float prod = w * v;
                acc = acc + prod;
            }
            out[(long)t * H + i] = oracle_f32_to_bf16(acc);
        }
    }
}

/*
 * combine addressed from the expert side.  Row r of the expert-major buffer
 * y [R, H] carries the pair it was dispatched from, (src_token[r], src_k[r]),
 * or -1 when it holds no copy, and optionally its own weight row_w[r] (NULL:
 * every weight is 1).  Copy j of token t is the row whose pair is (t, j),
 * found by scanning the rows from 0 up (the first such row if several claim
 * it); a pair that no row holds (a dropped or masked copy) adds nothing.
 * out[t, i] = bf16( sum over j of w_r * y[r, i] ), fp32 in increasing j,
 * exactly as oracle_combine does with slot_of[t,j] = r.
 */
void oracle_combine_src(int T, int H, int k, long R, const uint16_t *y, const float *row_w,
                        const int32_t *src_token, const int32_t *src_k, uint16_t *out)
{
    long row_of_copy[64];
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            row_of_copy[j] = -1;
            for (long r = 0; r < R; ++r) {
                if (src_token[r] == t && src_k[r] == j) {
                    row_of_copy[j] = r;
                    break;
                }
            }
        }
        for (int i = 0; i < H; ++i) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                long r = row_of_copy[j];
                if (r < 0) continue;
                float w = row_w ? row_w[r] : 1.0f;
                float prod = w * bf16_bits_to_f32(y[r * H + i]);
                acc = acc + prod;
            }
            out[(long)t * H + i] = oracle_f32_to_bf16(acc);
        }
    }
}

/* Vector helpers for the tests (elementwise over n values). */
void oracle_e4m3_encode_n(const float *v, uint8_t *codes, long n)
{
    for (long i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(v[i]);
}

void oracle_f32_to_bf16_n(const float *v, uint16_t *b, long n)
{
    for (long i = 0; i < n; ++i) b[i] = oracle_f32_to_bf16(v[i]);
}
