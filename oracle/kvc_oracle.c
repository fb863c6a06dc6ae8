/*
 * kvc_oracle.c -- CPU oracle for the paged KV-cache decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously-correct C in fp64.  Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg load it; the
 * product path (the CUDA library) never does, and the two share no code,
 * header, table or constant.  Each function cites the passage it follows:
 *
 *   [P1] "KV cache: Generation state, latency, and allocation" (aisyseng.dev,
 *        chapter 21), sections 21.1, 21.5, 21.6, Eq. 21.1-21.3, 21.6, Table 21.1.
 *   [P2] "KV Cache Explained: The Memory Problem Behind Fast LLM Inference"
 *        (archcrux.com), sections "How much GPU memory does the KV cache use?",
 *        "Why PagedAttention allocates KV in blocks", "What changes when you
 *        use FP8 KV".
 *   [P3] the xf_kv_cache page (aicassindra.com), "The architecture: every
 *        piece explained", "End-to-end flow".
 *
 * Representations
 *   Logical list (Eq. 21.1, token-major): the stored scalars of one layer for
 *   a batch of sequences, concatenated: rows [cu[b], cu[b+1]) of an array
 *   [total][H_KV][d_h] hold sequence b's positions 0.. in logical order.  A
 *   stored scalar is a bf16 bit pattern (2 bytes) or an e4m3 code (1 byte).
 *   Pool image: a byte array laid out as the library documents it,
 *   element offset ((((l*N + p)*H_KV + h)*2 + kv)*bs + slot)*d_h + c, times
 *   the element size; kv = 0 for keys, 1 for values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Planted mistakes for the mutation test of the pins (tests/test_oracle_mutants.py):
 * built with -DORC_MUTANT=n, the oracle carries mistake n -- a dropped term, a
 * wrong constant, sign, index or operand -- and the pins must fail.  The oracle
 * proper is built without it (ORC_MUTANT 0: every ORC_MUT(n) is false). */
#ifndef ORC_MUTANT
#define ORC_MUTANT 0
#endif
#define ORC_MUT(n) (ORC_MUTANT == (n))

/* stored-scalar kinds: bf16 (2 bytes), OCP E4M3 (1 byte), int4 (half a byte in
 * the pool; one byte per element in logical lists) */
#define ORC_KIND_E4M3 1
#define ORC_KIND_BF16 2
#define ORC_KIND_INT4 3

static int logical_bytes(int kind) { return kind == ORC_KIND_BF16 ? 2 : 1; }

/* status codes (the oracle's own; the tests compare them by meaning) */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_BAD_BLOCK 3
#define ORC_ERR_RANGE 4

/* ---------------------------------------------------------------- bytes
 * [P1] Eq. 21.2: bytes = 2 * layers * B * H_KV * T * d_h * s  (the factor 2
 * counts keys and values; s = bytes per stored scalar).  Exact in uint64;
 * UINT64_MAX when a factor is negative or the product overflows. */
uint64_t orc_kv_bytes(int64_t layers, int64_t B, int64_t H_KV, int64_t T, int64_t d_h, int64_t s)
{
    const int64_t f[6] = {ORC_MUT(1) ? 1 : 2, layers, B, H_KV, T, d_h};   /* 1: keys only */
    uint64_t acc = (uint64_t)(s < 0 ? 0 : s);
    if (s < 0) return UINT64_MAX;
    for (int i = 0; i < 6; ++i) {
        if (f[i] < 0) return UINT64_MAX;
        const uint64_t x = (uint64_t)f[i];
        if (x != 0 && acc > UINT64_MAX / x) return UINT64_MAX;
        acc *= x;
    }
    return acc;
}

/* [P1] Eq. 21.3: growth for one more processed position in each of B requests. */
uint64_t orc_kv_bytes_growth(int64_t layers, int64_t B, int64_t H_KV, int64_t d_h, int64_t s)
{
    return orc_kv_bytes(layers, B, H_KV, ORC_MUT(2) ? 2 : 1, d_h, s);   /* 2: two positions */
}

/* ---------------------------------------------------------------- scalars
 * bf16 -> double: the bit pattern is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t bits)
{
    const uint32_t w = (uint32_t)bits << (ORC_MUT(3) ? 15 : 16);   /* 3: misplaced half */
    float f;
    memcpy(&f, &w, 4);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("FN" variant: no infinities): 1 sign bit,
 * 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0 encodes
 * subnormals m * 2^-9; S.1111.111 is NaN; the largest finite is
 * S.1111.110 = 1.75 * 2^8 = 448 (the constant the configuration's scales divide
 * by).  [P2] "What changes when you use FP8 KV": one byte per element, with
 * scales. */
double orc_e4m3_to_double(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, ORC_MUT(4) ? -10 : -9);              /* 4: subnormal step */
    else v = ldexp(8.0 + m, e - (ORC_MUT(5) ? 11 : 10));   /* (1 + m/8) * 2^(e-7); 5: bias 8 */
    return sign ? -v : v;
}

/* float -> e4m3 code: round to nearest, ties to even, saturating to +-448
 * (also for +-inf); NaN -> 0x7F with the input's sign bit.
 * Method: find the binade [2^e, 2^(e+1)) of |x| (the subnormal range shares
 * the binade e = -6), divide by that binade's spacing 2^(e-3) (exact), round
 * to an integer with ties to even; the codes of consecutive magnitudes are
 * consecutive integers, so the code is (e + 6) * 8 + that integer. */
uint8_t orc_e4m3_from_float(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return sign | 0x7F;
    const double a = fabs((double)x);
    if (a >= 448.0) return sign | (ORC_MUT(6) ? 0x7F : 0x7E);   /* 6: overflow to NaN */
    if (a == 0.0) return sign;
    int E;
    (void)frexp(a, &E);
    int e = E - 1;
    if (e < -6) e = -6;
    const double q = ORC_MUT(7) ? trunc(a / ldexp(1.0, e - 3))    /* 7: round toward zero */
                                : rint(a / ldexp(1.0, e - 3));    /* default rounding mode: ties to even */
    int code = (e + 6) * 8 + (int)q;
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

/* int4 ([P3] "The architecture: every piece explained": int4 with per-channel
 * scales; the pages fix nothing more, so the plainest symmetric reading):
 * q = round-half-even(y), clamped to [-7, 7], stored as the nibble q + 8;
 * NaN stores 0 (nibble 8). */
uint8_t orc_int4_encode(float y)
{
    if (isnan(y)) return 8;
    double r = rint((double)y);
    if (r > 7.0) r = 7.0;
    if (r < (ORC_MUT(8) ? -8.0 : -7.0)) r = ORC_MUT(8) ? -8.0 : -7.0;   /* 8: asymmetric clamp */
    return (uint8_t)(r + 8.0);
}

double orc_int4_decode(uint8_t nibble) { return (double)nibble - (ORC_MUT(9) ? 7.0 : 8.0); }   /* 9: bias 7 */

/* int4 scale for one channel: absmax over positions / 7 in fp32 (1 if 0). */
void orc_int4_scales(const uint16_t *x, int64_t n_tokens, int32_t H_KV, int32_t d_h, float *scale_out)
{
    for (int64_t hc = 0; hc < (int64_t)H_KV * d_h; ++hc) {
        float amax = 0.0f;
        for (int64_t t = 0; t < n_tokens; ++t) {
            const float v = fabsf((float)orc_bf16_to_double(x[t * H_KV * d_h + hc]));
            if (v > amax) amax = v;
        }
        scale_out[hc] = (amax > 0.0f) ? amax / (ORC_MUT(10) ? 8.0f : 7.0f) : 1.0f;   /* 10: /8 */
    }
}

/* fp8 scale for one channel, per the configuration: absmax over positions
 * divided by 448, in fp32; an all-zero channel gets scale 1. */
void orc_fp8_scales(const uint16_t *x, int64_t n_tokens, int32_t H_KV, int32_t d_h, float *scale_out)
{
    for (int64_t hc = 0; hc < (int64_t)H_KV * d_h; ++hc) {
        float amax = 0.0f;
        for (int64_t t = 0; t < n_tokens; ++t) {
            const float v = fabsf((float)orc_bf16_to_double(x[t * H_KV * d_h + hc]));
            if (v > amax) amax = v;
        }
        scale_out[hc] = (amax > 0.0f) ? amax / (ORC_MUT(11) ? 240.0f : 448.0f) : 1.0f;   /* 11: E4M3FNUZ max */
    }
}

/* Stored e4m3 codes of bf16 tokens x [n][H_KV][d_h] under scales [H_KV][d_h]:
 * e4m3(fp32(x) / scale), the same rule the append applies. */
void orc_quantize_e4m3(const uint16_t *x, int64_t n_tokens, int32_t H_KV, int32_t d_h, const float *scale,
                       uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int64_t hc = 0; hc < (int64_t)H_KV * d_h; ++hc) {
            const float xf = (float)orc_bf16_to_double(x[t * H_KV * d_h + hc]);
            out[t * H_KV * d_h + hc] = orc_e4m3_from_float(xf / scale[hc]);
        }
}

/* Stored int4 nibbles (one per byte) of bf16 tokens under scales [H_KV][d_h]. */
void orc_quantize_int4(const uint16_t *x, int64_t n_tokens, int32_t H_KV, int32_t d_h, const float *scale,
                       uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int64_t hc = 0; hc < (int64_t)H_KV * d_h; ++hc) {
            const float xf = (float)orc_bf16_to_double(x[t * H_KV * d_h + hc]);
            out[t * H_KV * d_h + hc] = orc_int4_encode(xf / scale[hc]);
        }
}

/* ---------------------------------------------------------------- tables
 * [P1] 21.5: position t lies in logical block floor(t / bs), slot t mod bs;
 * the block table supplies the physical block.  Entries past a sequence's
 * allocation are -1.  Returns ORC_ERR_RANGE when the logical block is past the
 * table row, ORC_ERR_BAD_BLOCK when the entry is not a block of the pool. */
int orc_locate(const int32_t *bt_row, int32_t max_blocks, int64_t t, int32_t bs, int64_t num_blocks,
               int64_t *phys, int32_t *slot)
{
    if (t < 0 || bs <= 0) return ORC_ERR_ARG;
    const int64_t lb = ORC_MUT(12) ? (t + 1) / bs : t / bs;   /* 12: off by one position */
    if (lb >= max_blocks) return ORC_ERR_RANGE;
    const int32_t p = bt_row[lb];
    if (p < 0 || (int64_t)p >= num_blocks) return ORC_ERR_BAD_BLOCK;
    *phys = p;
    *slot = (int32_t)(ORC_MUT(13) ? (bs - 1 - t % bs) : t % bs);   /* 13: slots reversed */
    return ORC_OK;
}

/* element offset of (layer, physical block, K|V, head, slot, channel) in the pool image */
uint64_t orc_pool_offset(int64_t num_blocks, int32_t bs, int32_t H_KV, int32_t d_h,
                         int32_t layer, int64_t phys, int32_t kv, int32_t h, int32_t slot, int32_t c)
{
    if (ORC_MUT(14))   /* 14: K|V outside the head index ([p][kv][h]) */
        return (((((uint64_t)layer * (uint64_t)num_blocks + (uint64_t)phys) * 2u + (uint64_t)kv) * (uint64_t)H_KV
                 + (uint64_t)h) * (uint64_t)bs + (uint64_t)slot) * (uint64_t)d_h + (uint64_t)c;
    return (((((uint64_t)layer * (uint64_t)num_blocks + (uint64_t)phys) * (uint64_t)H_KV + (uint64_t)h) * 2u
             + (uint64_t)kv) * (uint64_t)bs + (uint64_t)slot) * (uint64_t)d_h + (uint64_t)c;
}

/* ---------------------------------------------------------------- append
 * [P1] Eq. 21.6: cache_t = append(cache_{t-1}, K_t, V_t), one processed token
 * at a time, logical order preserved across nonconsecutive blocks
 * ([P1] Table 21.1 steps 1-2).  Sequence b receives tokens
 * k[cu[b] .. cu[b+1]) at positions start_pos[b], start_pos[b]+1, ...;
 * each lands at (block_table[b][t / bs], t mod bs).  Stored scalars (kind):
 * the bf16 bit pattern unchanged, or the e4m3 code / int4 nibble of
 * float(x) / scale[h][c] computed in fp32 (scales are the layer's
 * [2][H_KV][d_h] array, keys first).  int4 element e of the pool image is
 * nibble e mod 2 (0 = low) of byte e / 2.
 * A token whose slot cannot be located is skipped; the first such error is
 * returned and every other token is still written. */
int orc_write_tokens(uint8_t *img, int64_t num_blocks, int32_t bs, int32_t H_KV, int32_t d_h, int32_t kind,
                     int32_t layer, const int32_t *bt, int32_t max_blocks, int32_t B,
                     const int32_t *start_pos, const int64_t *cu, const uint16_t *k, const uint16_t *v,
                     const float *scales)
{
    int status = ORC_OK;
    for (int32_t b = 0; b < B; ++b) {
        for (int64_t i = cu[b]; i < cu[b + 1]; ++i) {
            const int64_t t = (int64_t)start_pos[b] + (i - cu[b]);
            int64_t phys;
            int32_t slot;
            const int st = orc_locate(bt + (int64_t)b * max_blocks, max_blocks, t, bs, num_blocks, &phys, &slot);
            if (st != ORC_OK) {
                if (status == ORC_OK) status = st;
                continue;
            }
            for (int32_t kv = 0; kv < 2; ++kv) {
                const uint16_t *src = (kv == 0 ? k : v) + i * H_KV * d_h;
                for (int32_t h = 0; h < H_KV; ++h)
                    for (int32_t c = 0; c < d_h; ++c) {
                        const uint64_t off = orc_pool_offset(num_blocks, bs, H_KV, d_h, layer, phys, kv, h, slot, c);
                        const uint16_t x = src[h * d_h + c];
                        const float xf = (float)orc_bf16_to_double(x);
                        const float sc = scales ? scales[((int64_t)kv * H_KV + h) * d_h + c] : 1.0f;
                        if (kind == ORC_KIND_BF16) {
                            img[2 * off] = (uint8_t)(x & 0xFF);      /* little-endian bf16 */
                            img[2 * off + 1] = (uint8_t)(x >> 8);
                        } else if (kind == ORC_KIND_E4M3) {
                            img[off] = orc_e4m3_from_float(xf / sc);
                        } else {
                            const uint8_t nib = orc_int4_encode(xf / sc);
                            const int shift = ((off % 2) ^ (ORC_MUT(15) ? 1 : 0)) ? 4 : 0;   /* 15: nibbles swapped */
                            img[off / 2] = (uint8_t)((img[off / 2] & ~(0x0F << shift)) | (nib << shift));
                        }
                    }
            }
        }
    }
    return status;
}

/* Read sequence b's first len positions back through its table: stored
 * scalars [len][H_KV][d_h] (keys to k_out, values to v_out). */
int orc_gather(const uint8_t *img, int64_t num_blocks, int32_t bs, int32_t H_KV, int32_t d_h, int32_t kind,
               int32_t layer, const int32_t *bt_row, int32_t max_blocks, int64_t len,
               uint8_t *k_out, uint8_t *v_out)
{
    for (int64_t t = 0; t < len; ++t) {
        int64_t phys;
        int32_t slot;
        const int st = orc_locate(bt_row, max_blocks, t, bs, num_blocks, &phys, &slot);
        if (st != ORC_OK) return st;
        for (int32_t kv = 0; kv < 2; ++kv)
            for (int32_t h = 0; h < H_KV; ++h)
                for (int32_t c = 0; c < d_h; ++c) {
                    const uint64_t off = orc_pool_offset(num_blocks, bs, H_KV, d_h, layer, phys, kv, h, slot, c);
                    const int lb = logical_bytes(kind);
                    uint8_t *dst = (kv == 0 ? k_out : v_out) + ((t * H_KV + h) * d_h + c) * lb;
                    if (kind == ORC_KIND_INT4)
                        *dst = (uint8_t)((img[off / 2] >> ((off % 2) ? 4 : 0)) & 0x0F);
                    else
                        memcpy(dst, img + off * lb, (size_t)lb);
                }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------- attention
 * Value of one stored scalar of a logical list: bf16 widened exactly, or the
 * e4m3 code / int4 nibble decoded times the channel's scale ([P2] FP8 and
 * [P3]: quantized values need scales). */
static double stored_value(const uint8_t *base, int64_t idx, int32_t kind, const float *scale_hc)
{
    if (kind == ORC_KIND_BF16) {
        const uint16_t bits = (uint16_t)(base[2 * idx] | (base[2 * idx + 1] << 8));
        return orc_bf16_to_double(bits);
    }
    if (kind == ORC_KIND_E4M3) return orc_e4m3_to_double(base[idx]) * (double)(*scale_hc);
    return orc_int4_decode(base[idx]) * (double)(*scale_hc);
}

/* One query head against one sequence's first n positions ([P1] 21.1: the new
 * query reads the cached keys and its own new key, normalises the scores and
 * mixes the values; padded or unfilled slots are never read):
 *   x_t  = scale * sum_c q_c K[t][h][c]             (t < n)
 *   m    = max_t x_t,  Z = sum_t exp(x_t - m)
 *   out_c = sum_t exp(x_t - m) V[t][h][c] / Z,   lse = m + ln Z
 * n = 0 gives out = 0 and lse = -inf.  x is caller scratch of n doubles. */
static void attend_one(const double *q, const uint8_t *K, const uint8_t *V, int64_t n,
                       int32_t H_KV, int32_t d_h, int32_t h, int32_t kind,
                       const float *sk, const float *sv, double scale, double *x, double *out, double *lse)
{
    if (n == 0) {
        for (int32_t c = 0; c < d_h; ++c) out[c] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    if (ORC_MUT(17) && n > 1) --n;   /* 17: the newest position masked out */
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int32_t c = 0; c < d_h; ++c) {
            const int64_t idx = (t * H_KV + h) * d_h + c;
            dot += q[c] * stored_value(K, idx, kind, sk ? &sk[h * d_h + c] : NULL);
        }
        x[t] = ORC_MUT(16) ? dot : scale * dot;   /* 16: softmax scale dropped */
        if (x[t] > m) m = x[t];
    }
    double Z = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        x[t] = exp(x[t] - m);          /* x now holds the unnormalised weights */
        if (ORC_MUT(22)) x[t] = exp(x[t]);   /* 22: exponentiated twice */
        Z += x[t];
    }
    for (int32_t c = 0; c < d_h; ++c) out[c] = 0.0;
    for (int64_t t = 0; t < n; ++t)
        for (int32_t c = 0; c < d_h; ++c) {
            const int64_t idx = (t * H_KV + h) * d_h + c;
            const float *svc = ORC_MUT(18) ? (sk ? &sk[h * d_h + c] : NULL) : (sv ? &sv[h * d_h + c] : NULL);
            out[c] += x[t] * stored_value(V, idx, kind, svc);   /* 18: values scaled by the key scales */
        }
    for (int32_t c = 0; c < d_h; ++c) out[c] /= ORC_MUT(23) ? (double)n : Z;   /* 23: mean, not softmax */
    *lse = m + (ORC_MUT(19) ? log2(Z) : log(Z));   /* 19: log base 2 */
}

/* Decode attention for a batch over logical lists.
 * q: bf16 bits [B][H_Q][d_h].  K, V: stored scalars, rows [cu[b], cu[b]+n[b])
 * belong to sequence b.  n[b] = positions attended (the post-append length).
 * GQA/MQA ([P1] 21.1; [P3] GQA head sharing): H_Q divisible by H_KV, query
 * head hq reads KV head hq / (H_Q / H_KV) (contiguous groups), and keeps its
 * own scores and value mixture.  scales: [2][H_KV][d_h] for e4m3, else NULL.
 * out: [B][H_Q][d_h], lse: [B][H_Q] (natural log of the scaled-score sum). */
int orc_decode(const uint16_t *q, const uint8_t *K, const uint8_t *V, const int64_t *cu, const int64_t *n,
               int32_t B, int32_t H_Q, int32_t H_KV, int32_t d_h, int32_t kind, const float *scales,
               double scale, double *out, double *lse)
{
    if (H_KV <= 0 || H_Q % H_KV != 0) return ORC_ERR_ARG;
    const int32_t g = H_Q / H_KV;
    const float *sk = scales, *sv = scales ? scales + (int64_t)H_KV * d_h : NULL;
    int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * H_Q; ++bh) {
        const int64_t b = bh / H_Q;
        const int32_t hq = (int32_t)(bh % H_Q), h = ORC_MUT(20) ? hq % H_KV : hq / g;   /* 20: interleaved groups */
        double *x = (double *)malloc(sizeof(double) * (size_t)(n[b] > 0 ? n[b] : 1));
        double qd[1024];
        if (!x || d_h > 1024) {
#pragma omp atomic write
            status = ORC_ERR_ARG;
            free(x);
            continue;
        }
        for (int32_t c = 0; c < d_h; ++c) qd[c] = orc_bf16_to_double(q[bh * d_h + c]);
        const int64_t row0 = cu[b] * H_KV * d_h * logical_bytes(kind);
        attend_one(qd, K + row0, V + row0, n[b], H_KV, d_h, h, kind, sk, sv, scale, x,
                   out + bh * d_h, lse + bh);
        free(x);
    }
    return status;
}

/* Prefill chunk over one sequence's logical list ([P1] 21.3 chunked prefill:
 * later portions keep the earlier positions; [P3] "End-to-end flow": the new
 * tokens attend to the shared prefix through the table).  Query i sits at
 * position q_start + i and, by causal visibility ([P1] 21.1), reads positions
 * 0 .. q_start + i.  q: [n_q][H_Q][d_h]; out/lse like orc_decode with B = n_q. */
int orc_prefill(const uint16_t *q, int64_t n_q, const uint8_t *K, const uint8_t *V, int64_t q_start,
                int32_t H_Q, int32_t H_KV, int32_t d_h, int32_t kind, const float *scales,
                double scale, double *out, double *lse)
{
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_q + 1));
    int64_t *n = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_q > 0 ? n_q : 1));
    if (!cu || !n) { free(cu); free(n); return ORC_ERR_ARG; }
    for (int64_t i = 0; i <= n_q; ++i) cu[i] = 0;        /* every query reads the same list */
    for (int64_t i = 0; i < n_q; ++i) n[i] = q_start + i + (ORC_MUT(21) ? 0 : 1);   /* 21: own key hidden */
    const int st = orc_decode(q, K, V, cu, n, (int32_t)n_q, H_Q, H_KV, d_h, kind, scales, scale, out, lse);
    free(cu);
    free(n);
    return st;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
