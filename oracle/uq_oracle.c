/*
 * uq_oracle.c -- plain, slow, fp64 CPU oracle for the UltraQuant 4-bit
 * KV-cache store and paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or constant with the CUDA path, and the CUDA path never calls it.
 *
 * Sources (vLLM API documentation pages):
 *   [ultraquant_attn]   vllm.v1.attention.backends.ultraquant_attn,
 *                       class UltraQuantAttentionImpl
 *   [flydsl_decode]     vllm.v1.attention.ops.flydsl_ultraquant_decode
 *   [tq_decode_v2]      vllm.v1.attention.ops.turboquant_soa.
 *                       triton_turboquant_decode_v2
 *
 * Every step follows the definition of what is computed, in the order the
 * pages give it, with no blocking, fusion or reordering.  Where the pages are
 * silent (block size of the UE8M0 scale, exponent rule, E2M1 rounding and
 * signed zero, slot byte layout, fp32 order of the K rotation) the function
 * says which reading it takes.
 *
 * Parity status of each function (what pins it, outside itself):
 *   uqo_hadamard        pinned: H.H = I, H = H^T, entries +-1/sqrt(D)
 *   uqo_fwht_f32        pinned: equals D^(1/2) H.x in fp64 to 1e-6; spike rows
 *   uqo_round_format    pinned: brute-force nearest-with-ties-to-even search,
 *                       torch's float8_e4m3fn / bfloat16 casts
 *   uqo_e2m1_encode     pinned: brute force over the 16-entry value table
 *   uqo_ue8m0_byte      pinned: amax = 2^k closed form, [4,8) range invariant
 *   uqo_quantize_slot   pinned: spike input closed form, error bound
 *   uqo_store           pinned: spike input at a chosen slot (address rule)
 *   uqo_query_prime     pinned: torch fp32 matmul + float8_e4m3fn cast
 *   uqo_decode          pinned: L=1, equal keys, dominant logit, head map,
 *                       page permutation invariance, numpy brute force
 *   uqo_decode (S > 0)  pinned: equals the single softmax to 1e-12
 *   uqo_decode_ex       pinned: window >= L equals no window; window 1 gives
 *                       the last token's v exactly; equal keys with a sink,
 *                       closed form; sink -> -inf equals no sink; split =
 *                       unsplit with both; numpy brute force
 *   uqo_full_dequant    pinned: numpy bit-level mirror on tiny caches, spike
 *                       slot, closed forms at scale bytes 0, 254 and 255,
 *                       page-permutation invariance
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

/* ------------------------------------------------------------------------- */
/* Number formats, written from their definitions.                            */
/* ------------------------------------------------------------------------- */

/* bf16 bit pattern -> exact double (bf16 is the top half of an IEEE fp32). */
double uqo_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round x to the nearest value of a binary floating-point format with
 * `mant_bits` explicit mantissa bits and minimum normal exponent `emin`,
 * ties to even (the integer significand that is even).  Values below the
 * normal range use the subnormal quantum 2^(emin - mant_bits).  If the
 * rounded magnitude exceeds `maxval`, it becomes `maxval` when `satfinite`
 * is set, else infinity.  Signed zero is kept.
 *
 *   E2M1 (FP4):  mant_bits 1, emin 0,    max 6
 *   E4M3 (fn):   mant_bits 3, emin -6,   max 448
 *   bf16:        mant_bits 7, emin -126, max (2 - 2^-7) 2^127
 */
double uqo_round_format(double x, int mant_bits, int emin, double maxval,
                        int satfinite)
{
    if (x == 0.0 || isnan(x))
        return x;
    double ax = fabs(x);
    int e2;
    (void)frexp(ax, &e2);           /* ax = f 2^e2, f in [0.5, 1) */
    int E = e2 - 1;                 /* floor(log2(ax)) */
    if (E < emin)
        E = emin;
    double quantum = ldexp(1.0, E - mant_bits);
    double q = rint(ax / quantum);  /* exact division; rint = ties to even */
    double r = q * quantum;
    if (r > maxval)
        r = satfinite ? maxval : INFINITY;
    return copysign(r, x);
}

/* bf16 round-to-nearest-even of a double, returned as a bit pattern. */
uint16_t uqo_bf16_round(double x)
{
    double r = uqo_round_format(x, 7, -126, ldexp(255.0, 120), 0);
    float f = (float)r;             /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* E4M3 ("fn" variant, max 448) round-to-nearest-even, saturating. */
double uqo_e4m3_round(double x)
{
    return uqo_round_format(x, 3, -6, 448.0, 1);
}

/*
 * FP4 E2M1 code -> value.  [flydsl_decode: _fp4_value_lut] the stored 4-bit
 * code indexes a 16-entry table whose entry is the dequantised value.  The
 * table follows the E2M1 bit layout s|e1 e0|m: codes 0..7 are
 * +{0, 0.5, 1, 1.5, 2, 3, 4, 6}, codes 8..15 the same values negated.
 */
double uqo_e2m1_value(int code)
{
    int mag = code & 7;
    int e = mag >> 1, m = mag & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return (code & 8) ? -v : v;
}

/*
 * Value -> E2M1 code: round to nearest E2M1 value, ties to the even code,
 * saturating at +-6; the sign bit follows the sign of y, so a negative value
 * that rounds to zero is stored as code 8 (reading: the pages are silent).
 */
int uqo_e2m1_encode(double y)
{
    double r = uqo_round_format(y, 1, 0, 6.0, 1);
    double ar = fabs(r);
    int mag;
    if (ar == 0.0)      mag = 0;
    else if (ar == 0.5) mag = 1;
    else if (ar == 1.0) mag = 2;
    else if (ar == 1.5) mag = 3;
    else if (ar == 2.0) mag = 4;
    else if (ar == 3.0) mag = 5;
    else if (ar == 4.0) mag = 6;
    else                mag = 7;    /* 6.0 */
    return (signbit(y) ? 8 : 0) | mag;
}

/*
 * UE8M0 block scale from a block's absolute maximum.  [ultraquant_attn:
 * class docstring] names "FP4 E2M1 + UE8M0" and nothing more.  Reading (the
 * MX convention): shared exponent se = floor(log2(amax)) - 2, where 2 is
 * E2M1's largest exponent, clamped to [-127, 127]; the byte is se + 127.
 * An all-zero block gets byte 0.
 */
int uqo_ue8m0_byte(double amax)
{
    if (!(amax > 0.0))
        return 0;
    int e2;
    (void)frexp(amax, &e2);
    int se = (e2 - 1) - 2;
    if (se < -127) se = -127;
    if (se > 127)  se = 127;
    return se + 127;
}

/* ------------------------------------------------------------------------- */
/* Hadamard rotation.                                                         */
/* ------------------------------------------------------------------------- */

/*
 * [ultraquant_attn: _ensure_on_device] the rotation is a pure Hadamard matrix,
 * orthonormal and symmetric (H = H^T).  Reading: Sylvester (natural) order,
 * H[i][j] = (-1)^popcount(i & j) / sqrt(D).  D must be a power of two.
 */
void uqo_hadamard(int D, double *H)
{
    double s = 1.0 / sqrt((double)D);
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j)
            H[(size_t)i * D + j] = (__builtin_popcount((unsigned)(i & j)) & 1) ? -s : s;
}

/*
 * Unnormalised fast Walsh-Hadamard transform in fp32, in the canonical stage
 * order: for h = 1, 2, 4, ..., D/2 every pair (i, i+h) with (i & h) == 0
 * becomes (a + b, a - b), a being the lower index.  The result equals
 * sqrt(D) H x up to fp32 rounding; this fixed order makes the fp32 result
 * unique (reading: the pages do not show the store kernel's arithmetic).
 */
void uqo_fwht_f32(float *x, int D)
{
    for (int h = 1; h < D; h <<= 1)
        for (int i = 0; i < D; ++i)
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/* ------------------------------------------------------------------------- */
/* Slot packing.                                                              */
/* ------------------------------------------------------------------------- */

/*
 * Slot layout for head dim D (reading; the pages give only the slot width as
 * kv_cache.shape[3]): bytes [0, D/2) K codes, [D/2, D) V codes,
 * [D, D + D/32) K scale bytes (one per 32-element block, block order),
 * [D + D/32, D + D/16) V scale bytes.  Byte j of a code region holds element
 * 2j in its low nibble and element 2j+1 in its high nibble.  D = 256 gives
 * 272 bytes.
 */
int uqo_slot_bytes(int D) { return D + D / 16; }

static void quantize_region(const float *x, int D, uint8_t *codes,
                            uint8_t *scales)
{
    memset(codes, 0, (size_t)D / 2);
    for (int blk = 0; blk < D / 32; ++blk) {
        double amax = 0.0;
        for (int i = 0; i < 32; ++i) {
            double a = fabs((double)x[blk * 32 + i]);
            if (a > amax) amax = a;
        }
        int byte = uqo_ue8m0_byte(amax);
        scales[blk] = (uint8_t)byte;
        int se = byte - 127;
        for (int i = 0; i < 32; ++i) {
            int d = blk * 32 + i;
            double y = ldexp((double)x[d], -se);    /* exact power-of-two scaling */
            int c = uqo_e2m1_encode(y);
            codes[d / 2] |= (uint8_t)((d & 1) ? (c << 4) : c);
        }
    }
}

/* Pack a rotated-K row and a V row (both fp32, length D) into one slot. */
void uqo_quantize_slot(const float *k_rot, const float *v, int D, uint8_t *slot)
{
    quantize_region(k_rot, D, slot, slot + D);
    quantize_region(v, D, slot + D / 2, slot + D + D / 32);
}

/* Dequantise one slot: x = LUT[code] * 2^(byte - 127). */
void uqo_dequant_slot(const uint8_t *slot, int D, double *k, double *v)
{
    for (int d = 0; d < D; ++d) {
        int kc = (slot[d / 2] >> ((d & 1) * 4)) & 15;
        int vc = (slot[D / 2 + d / 2] >> ((d & 1) * 4)) & 15;
        int kb = slot[D + d / 32];
        int vb = slot[D + D / 32 + d / 32];
        k[d] = ldexp(uqo_e2m1_value(kc), kb - 127);
        v[d] = ldexp(uqo_e2m1_value(vc), vb - 127);
    }
}

/* Byte offset of (slot, kv head) in the paged cache
 * kv_cache[num_blocks][block_size][Hk][slot_bytes]. */
static int64_t slot_offset(int64_t slot, int h, int Hk, int block_size,
                           int slot_bytes)
{
    int64_t page = slot / block_size, off = slot % block_size;
    return ((page * block_size + off) * Hk + h) * (int64_t)slot_bytes;
}

/*
 * [ultraquant_attn: _store_kv] rotate K by the Hadamard (k_rot = k.float() @
 * PiT, the same product the continuation path spells out) and pack K and V
 * into FP4/UE8M0 slots at slot_mapping.  V is not rotated (the continuation
 * path concatenates the raw value chunk).  The rotation is the canonical fp32
 * FWHT followed by the exact factor 1/sqrt(D) (D = 256: 1/16).  A negative
 * slot is skipped (vLLM's padding convention; reading).  Returns the number
 * of rows skipped because their slot was negative, or -1 if a slot is beyond
 * the cache.
 */
int64_t uqo_store(const uint16_t *key, const uint16_t *value,
                  const int64_t *slot_mapping, int64_t N, int Hk, int D,
                  int64_t key_stride_tok, int64_t value_stride_tok,
                  int num_blocks, int block_size, uint8_t *kv_cache)
{
    int sb = uqo_slot_bytes(D);
    float inv_sqrt_d = (float)(1.0 / sqrt((double)D));
    float *kr = (float *)malloc(sizeof(float) * D);
    float *vr = (float *)malloc(sizeof(float) * D);
    int64_t skipped = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) { ++skipped; continue; }
        if (slot >= (int64_t)num_blocks * block_size) { skipped = -1; break; }
        for (int h = 0; h < Hk; ++h) {
            const uint16_t *kp = key + n * key_stride_tok + (int64_t)h * D;
            const uint16_t *vp = value + n * value_stride_tok + (int64_t)h * D;
            for (int d = 0; d < D; ++d) {
                kr[d] = (float)uqo_bf16_to_double(kp[d]);
                vr[d] = (float)uqo_bf16_to_double(vp[d]);
            }
            uqo_fwht_f32(kr, D);
            for (int d = 0; d < D; ++d)
                kr[d] = kr[d] * inv_sqrt_d;
            uqo_quantize_slot(kr, vr, D,
                              kv_cache + slot_offset(slot, h, Hk, block_size, sb));
        }
    }
    free(kr);
    free(vr);
    return skipped;
}

/*
 * Quantise already-rotated fp32 K and fp32 V rows [N][Hk][D] into the cache
 * (no rotation).  Same slot rules as uqo_store.
 */
int64_t uqo_store_f32(const float *k_rot, const float *v,
                      const int64_t *slot_mapping, int64_t N, int Hk, int D,
                      int num_blocks, int block_size, uint8_t *kv_cache)
{
    int sb = uqo_slot_bytes(D);
    int64_t skipped = 0;
    for (int64_t n = 0; n < N; ++n) {
        int64_t slot = slot_mapping[n];
        if (slot < 0) { ++skipped; continue; }
        if (slot >= (int64_t)num_blocks * block_size) return -1;
        for (int h = 0; h < Hk; ++h)
            uqo_quantize_slot(k_rot + (n * Hk + h) * (int64_t)D,
                              v + (n * Hk + h) * (int64_t)D, D,
                              kv_cache + slot_offset(slot, h, Hk, block_size, sb));
    }
    return skipped;
}

/*
 * [ultraquant_attn: _ultraquant_continuation_prefill, the call to
 * ultraquant_full_dequant_kv] dequantise the cached prefix of one sequence
 * into bf16 buffers shaped (1, Hk, alloc_len, D), alloc_len = n_pages *
 * block_size (whole pages).  K stays Hadamard-rotated, as stored; V is in
 * the original space.  Token t of page p is slot block_table[p] * block_size
 * + t.  Each value is LUT[code] * 2^(byte - 127) in fp64 (a scale byte of 255
 * is read as 2^128 by the same formula; the store never writes it), then
 * bf16 round-to-nearest-even (inf on overflow).  Reading: a page id outside
 * [0, num_blocks) leaves its rows zero.  Returns the number of such pages.
 */
int uqo_full_dequant(const uint8_t *kv_cache, const int32_t *block_table, int n_pages,
                     int Hk, int D, int num_blocks, int block_size,
                     uint16_t *k_out, uint16_t *v_out)
{
    int sb = uqo_slot_bytes(D);
    int64_t alloc_len = (int64_t)n_pages * block_size;
    double *k = (double *)malloc(sizeof(double) * D);
    double *v = (double *)malloc(sizeof(double) * D);
    int bad = 0;
    for (int p = 0; p < n_pages; ++p) {
        int32_t pid = block_table[p];
        int ok = pid >= 0 && pid < num_blocks;
        if (!ok) ++bad;
        for (int t = 0; t < block_size; ++t) {
            int64_t slot = (int64_t)pid * block_size + t;
            int64_t row = (int64_t)p * block_size + t;
            for (int h = 0; h < Hk; ++h) {
                uint16_t *ko = k_out + ((int64_t)h * alloc_len + row) * D;
                uint16_t *vo = v_out + ((int64_t)h * alloc_len + row) * D;
                if (!ok) {
                    memset(ko, 0, sizeof(uint16_t) * D);
                    memset(vo, 0, sizeof(uint16_t) * D);
                    continue;
                }
                uqo_dequant_slot(kv_cache + slot_offset(slot, h, Hk, block_size, sb), D, k, v);
                for (int d = 0; d < D; ++d) {
                    ko[d] = uqo_bf16_round(k[d]);
                    vo[d] = uqo_bf16_round(v[d]);
                }
            }
        }
    }
    free(k);
    free(v);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Decode attention.                                                          */
/* ------------------------------------------------------------------------- */

/*
 * Query prologue, [flydsl_decode: flydsl_ultraquant_decode_attention, the
 * unfused prologue]: q_float = fp32(q); q_rot_fp32 = q_float @ PiT;
 * q_fp8 = e4m3(q_rot_fp32); q' = bf16(q_fp8).  The product is formed in fp64
 * and rounded once to fp32; the E4M3 cast is round-to-nearest-even and
 * saturates at +-448 (reading: the pages show no overflow rule); the bf16
 * cast of an E4M3 value is exact.  H is symmetric, so q @ PiT = H q.
 */
void uqo_query_prime(const uint16_t *q, int D, const double *H, double *qp)
{
    for (int i = 0; i < D; ++i) {
        double acc = 0.0;
        for (int j = 0; j < D; ++j)
            acc += uqo_bf16_to_double(q[j]) * H[(size_t)j * D + i];
        float r32 = (float)acc;
        qp[i] = uqo_e4m3_round((double)r32);
    }
}

typedef struct {
    const uint16_t *query;
    int64_t q_stride_seq, q_stride_head;
    const uint8_t *kv_cache;
    const int32_t *block_table;
    const int32_t *seq_lens;
    double scale;
    int B, Hq, Hk, D, num_blocks, block_size, max_blocks;
    int S;                      /* 0: one softmax over all tokens */
    const int32_t *rows;        /* (b, r) pairs, or NULL for all B*Hq rows */
    int n_rows;
    const double *sinks;        /* [Hq] sink logits, or NULL */
    int window;                 /* > 0: attend to the last `window` tokens only */
    const double *H;
    double *out;                /* [n_rows][D] */
    int status;
} decode_args;

/* Dequantised K and V of token t of sequence b, kv head g. */
static int token_kv(const decode_args *a, int b, int g, int t, double *k,
                    double *v)
{
    int sb = uqo_slot_bytes(a->D);
    int page = a->block_table[(int64_t)b * a->max_blocks + t / a->block_size];
    if (page < 0 || page >= a->num_blocks)
        return -1;
    int64_t slot = (int64_t)page * a->block_size + t % a->block_size;
    uqo_dequant_slot(a->kv_cache + slot_offset(slot, g, a->Hk, a->block_size, sb),
                     a->D, k, v);
    return 0;
}

/*
 * Softmax attention of one query row over tokens [t0, t1) of sequence b,
 * kv head g.  Returns (in fp64) the running max m, the sum l of exp(s - m)
 * and o = sum exp(s - m) v / l.  Empty ranges give m = -inf, l = 0, o = 0.
 */
static int attend_range(const decode_args *a, int b, int g, const double *qp,
                        int t0, int t1, double *m_out, double *l_out, double *o)
{
    int D = a->D;
    double *k = (double *)malloc(sizeof(double) * D);
    double *v = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (t1 > t0 ? t1 - t0 : 1));
    int rc = 0;
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t) {
        if (token_kv(a, b, g, t, k, v)) { rc = -1; break; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qp[d] * k[d];
        s[t - t0] = a->scale * dot;
        if (s[t - t0] > m) m = s[t - t0];
    }
    double l = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (rc == 0 && t1 > t0) {
        for (int t = t0; t < t1; ++t) {
            double p = exp(s[t - t0] - m);
            token_kv(a, b, g, t, k, v);
            l += p;
            for (int d = 0; d < D; ++d)
                o[d] += p * v[d];
        }
        for (int d = 0; d < D; ++d)
            o[d] /= l;
    }
    *m_out = m;
    *l_out = l;
    free(k); free(v); free(s);
    return rc;
}

/*
 * One output row (b, r).  Query head r reads kv head r / (Hq / Hk)
 * [ultraquant_attn: __init__, num_kv_groups].  Without splits this is plain
 * softmax(scale q'.k) v over the sequence's L_b tokens; L_b = 0 gives zeros
 * (reading).  [ultraquant_attn: sliding_window, sinks, passed on to the
 * unified attention, window_size = (sliding_window - 1, 0)] -- readings: a
 * window W > 0 keeps tokens [max(0, L - W), L); a sink logit z_r (same units
 * as scale q'.k) joins the softmax denominator only:
 * out = sum_t e^(s_t - m) v_t / (e^(z_r - m) + sum_t e^(s_t - m)).  With S splits, split s covers [s c, min((s+1) c, L)) with
 * c = ceil(L / S), each split keeps (m_s, l_s, o_s), and the splits are merged
 * with the log-sum-exp rule [tq_decode_v2: stage 2; flydsl_decode: reduce
 * partitions]: out = sum_s e^(m_s - M) l_s o_s / sum_s e^(m_s - M) l_s.
 */
static int decode_row(const decode_args *a, int b, int r, double *out)
{
    int D = a->D, QG = a->Hq / a->Hk, g = r / QG;
    int L = a->seq_lens[b];
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L <= 0)
        return 0;
    if ((int64_t)(L + a->block_size - 1) / a->block_size > a->max_blocks)
        return -1;
    uint16_t *q = (uint16_t *)malloc(sizeof(uint16_t) * D);
    double *qp = (double *)malloc(sizeof(double) * D);
    for (int d = 0; d < D; ++d)
        q[d] = a->query[(int64_t)b * a->q_stride_seq + (int64_t)r * a->q_stride_head + d];
    uqo_query_prime(q, D, a->H, qp);
    int rc = 0;
    int lo = (a->window > 0 && L > a->window) ? L - a->window : 0;
    if (a->S <= 0) {
        double m, l;
        rc = attend_range(a, b, g, qp, lo, L, &m, &l, out);
        if (rc == 0 && a->sinks) {
            double f = l / (l + exp(a->sinks[r] - m));
            for (int d = 0; d < D; ++d)
                out[d] *= f;
        }
    } else {
        int c = (L - lo + a->S - 1) / a->S;
        double M = -INFINITY;
        double *ms = (double *)malloc(sizeof(double) * a->S);
        double *ls = (double *)malloc(sizeof(double) * a->S);
        double *os = (double *)malloc(sizeof(double) * (size_t)a->S * D);
        for (int s = 0; s < a->S && rc == 0; ++s) {
            int t0 = lo + s * c, t1 = lo + (s + 1) * c < L ? lo + (s + 1) * c : L;
            if (t0 >= t1) { ms[s] = -INFINITY; ls[s] = 0.0; continue; }
            rc = attend_range(a, b, g, qp, t0, t1, &ms[s], &ls[s], os + (size_t)s * D);
            if (ms[s] > M) M = ms[s];
        }
        if (rc == 0) {
            double den = 0.0;
            for (int s = 0; s < a->S; ++s) {
                if (ls[s] == 0.0) continue;
                double w = exp(ms[s] - M) * ls[s];
                den += w;
                for (int d = 0; d < D; ++d)
                    out[d] += w * os[(size_t)s * D + d];
            }
            if (a->sinks)
                den += exp(a->sinks[r] - M);
            for (int d = 0; d < D; ++d)
                out[d] /= den;
        }
        free(ms); free(ls); free(os);
    }
    free(q); free(qp);
    return rc;
}

typedef struct {
    decode_args *a;
    int first, step;
} worker_args;

static void *decode_worker(void *p)
{
    worker_args *w = (worker_args *)p;
    decode_args *a = w->a;
    int total = a->rows ? a->n_rows : a->B * a->Hq;
    for (int i = w->first; i < total; i += w->step) {
        int b = a->rows ? a->rows[2 * i] : i / a->Hq;
        int r = a->rows ? a->rows[2 * i + 1] : i % a->Hq;
        if (decode_row(a, b, r, a->out + (size_t)i * a->D))
            a->status = -1;
    }
    return NULL;
}

/*
 * Decode attention for B sequences (or for the listed (b, r) rows).
 * query: bf16 bits, element (b, r, d) at b*q_stride_seq + r*q_stride_head + d.
 * kv_cache: uint8 [num_blocks][block_size][Hk][D + D/16].
 * block_table: int32 [B][max_blocks]; seq_lens: int32 [B].
 * out: fp64 [rows][D].  S = 0 computes one softmax per row; S > 0 uses the
 * split-then-combine variant.  Rows are spread over `nthreads` threads; the
 * arithmetic of a row does not depend on the thread count.
 * Returns 0, or -1 on an out-of-range page id or a table that is too short.
 */
int uqo_decode_ex(const uint16_t *query, int64_t q_stride_seq, int64_t q_stride_head,
                  const uint8_t *kv_cache, const int32_t *block_table,
                  const int32_t *seq_lens, double scale, int B, int Hq, int Hk,
                  int D, int num_blocks, int block_size, int max_blocks, int S,
                  const int32_t *rows, int n_rows, const double *sinks, int window,
                  int nthreads, double *out)
{
    if (Hk <= 0 || Hq % Hk != 0 || (D & (D - 1)) != 0 || D < 32)
        return -2;
    double *H = (double *)malloc(sizeof(double) * (size_t)D * D);
    uqo_hadamard(D, H);
    decode_args a = {query, q_stride_seq, q_stride_head, kv_cache, block_table,
                     seq_lens, scale, B, Hq, Hk, D, num_blocks, block_size,
                     max_blocks, S, rows, n_rows, sinks, window, H, out, 0};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    worker_args wa[256];
    for (int i = 0; i < nthreads; ++i) {
        wa[i].a = &a; wa[i].first = i; wa[i].step = nthreads;
        pthread_create(&tid[i], NULL, decode_worker, &wa[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        pthread_join(tid[i], NULL);
    free(H);
    return a.status;
}

/* uqo_decode_ex without sinks and without a window. */
int uqo_decode(const uint16_t *query, int64_t q_stride_seq, int64_t q_stride_head,
               const uint8_t *kv_cache, const int32_t *block_table,
               const int32_t *seq_lens, double scale, int B, int Hq, int Hk,
               int D, int num_blocks, int block_size, int max_blocks, int S,
               const int32_t *rows, int n_rows, int nthreads, double *out)
{
    return uqo_decode_ex(query, q_stride_seq, q_stride_head, kv_cache, block_table, seq_lens,
                         scale, B, Hq, Hk, D, num_blocks, block_size, max_blocks, S, rows,
                         n_rows, NULL, 0, nthreads, out);
}
