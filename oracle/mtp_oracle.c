/*
 * Plain CPU oracle for the GLM-5.3 MTP draft head ("Glm5NextMtpHead::forward_one").
 *
 * TEST INFRASTRUCTURE ONLY. This file is the reference the CUDA library is checked
 * against. Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * build, load or call it; the product path never does. It shares no code, header,
 * table or helper with the CUDA library, and includes nothing from it.
 *
 * It is slow and literal on purpose: double precision (fp64) for every sum and every
 * product, loops in the order the definitions state them, rounding to BF16 exactly at
 * the points where the source keeps BF16 storage, and a number-format codec written
 * from the format definitions (not from any library).
 *
 * Sources (titles and items of the pages this follows):
 *   [mtp]   "metrale_model_arch / glm5next_mtp_head.rs":
 *           module doc (the four-line math summary: x = eh_proj(concat(enorm(embed[token]),
 *           hnorm(target_hidden))); logits = lm_head(shared_head.norm(x)); draft = argmax),
 *           the proposer-state doc (BF16 concat [2, hidden], BF16 x [hidden]),
 *           the `head_fp8` doc (FP8 E4M3 copy of lm_head, drafting only),
 *           `norm` (rms_norm_vanilla launcher: x, w, out, n, eps),
 *           `forward_one` (embedding row read by pointer at token*hidden; enorm into
 *           concat[0:H], hnorm into concat[H:2H]; eh_proj gemv n=H, k=2H; final norm in
 *           place; lm_head gemv; argmax; `>=` tie rule of the cross-rank pick).
 *   [layer] "metrale_model_arch / glm5next_layer / mod.rs": module doc invariant that every
 *           norm is rms_norm_vanilla, x*w/rms, never the 1+w form.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *   - RMSNorm: rms = sqrt(mean(x^2) + eps), out = bf16(x * w / rms), one rounding.
 *   - BF16 rounding after enorm/hnorm (the concat), after eh_proj (x) and after the final
 *     norm (xhat); logits are kept unrounded (fp64 here; the GPU returns fp32).
 *   - argmax: lowest index among equal maxima; NaN never wins; an all-NaN row gives -1.
 *   - FP8 copy: OCP E4M3 ("fn": bias 7, subnormals, max 448, S.1111.111 = NaN, no Inf);
 *     per-row scale s = fp32(absmax / 448); code = RNE-to-E4M3 with saturation to +-448 of
 *     the fp32 quotient w / s; an all-zero row gives s = 0 and zero codes; any NaN or Inf
 *     weight fails the quantisation. The FP8 head's logits use the dequantised weights
 *     decode(code) * s, formed exactly in fp64.
 *   - An out-of-range token gives an all-zero x row and an error code (the source has no
 *     check at all).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off (no fast-math, no FMA
 * contraction, so the result is the same on every host).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define MO_OK 0
#define MO_ERR_NONFINITE (-6)
#define MO_ERR_TOKEN_RANGE (-7)

/* ------------------------------------------------------------------------------------ */
/* Rounding helper: round a non-negative double to the nearest integer, ties to even.   */
/* ------------------------------------------------------------------------------------ */
static double round_half_even(double q) {
    double f = floor(q);
    double r = q - f; /* exact: q and f share the exponent range of a double */
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* ------------------------------------------------------------------------------------ */
/* BF16: 1 sign bit, 8 exponent bits (bias 127), 7 mantissa bits; the upper half of an   */
/* IEEE binary32.                                                                        */
/* ------------------------------------------------------------------------------------ */
double mo_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest BF16 value (ties to even), one rounding. */
uint16_t mo_f64_to_bf16(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7FC0u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                  /* 2^(e-1) <= a < 2^e */
    int lead = e - 1;              /* exponent of the leading bit */
    /* spacing of BF16 values around a: 2^(lead-7) for normals, 2^-133 below 2^-126 */
    int quantum = (lead < -126) ? -133 : lead - 7;
    double units = round_half_even(ldexp(a, -quantum)); /* ldexp by a power of 2 is exact */
    double v = ldexp(units, quantum);
    if (v >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* rounds past the max */
    float f = (float)v; /* exact: v is a BF16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (uint16_t)(u >> 16));
}

/* ------------------------------------------------------------------------------------ */
/* FP8 E4M3 (OCP 8-bit floating point, E4M3 variant): sign, 4 exponent bits with bias 7, */
/* 3 mantissa bits. Exponent field 0 holds subnormals 2^-6 * m/8. Exponent field 15 with */
/* mantissa 7 is NaN; there is no infinity; the largest magnitude is 2^8 * 1.75 = 448.   */
/* ------------------------------------------------------------------------------------ */
double mo_e4m3_to_f64(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to the nearest E4M3 value, ties to even, saturating finite overflow to +-448.
 * NaN maps to the NaN code. Codes are contiguous in magnitude, so a mantissa that rounds
 * up to 2.0 carries into the next exponent by plain integer addition. */
uint8_t mo_f64_to_e4m3(double x) {
    uint8_t s = signbit(x) ? 0x80u : 0u;
    if (isnan(x)) return (uint8_t)(s | 0x7Fu);
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(s | 0x7Eu);
    int code;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: spacing 2^-9; 8 units is the smallest normal, code 0x08 */
        code = (int)round_half_even(ldexp(a, 9));
    } else {
        int e;
        frexp(a, &e);
        int lead = e - 1;                                         /* -6 .. 8 */
        int units = (int)round_half_even(ldexp(a, -(lead - 3)));  /* 8 .. 16 */
        code = (lead + 7) * 8 + (units - 8);
    }
    if (code > 0x7E) code = 0x7E;
    return (uint8_t)(s | (uint8_t)code);
}

/* Array forms (used by the tests to check the codecs against library conversions). */
void mo_bf16_to_f64_array(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = mo_bf16_to_f64(in[i]);
}
void mo_f64_to_bf16_array(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = mo_f64_to_bf16(in[i]);
}
void mo_e4m3_to_f64_array(const uint8_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = mo_e4m3_to_f64(in[i]);
}
void mo_f64_to_e4m3_array(const double* in, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = mo_f64_to_e4m3(in[i]);
}

/* ------------------------------------------------------------------------------------ */
/* rms_norm_vanilla: out = bf16( x * w / sqrt(mean(x^2) + eps) )   ([layer] invariant;  */
/* [mtp] `norm`). Never the (1 + w) form.                                                */
/* ------------------------------------------------------------------------------------ */
void mo_rms_norm(const uint16_t* x, const uint16_t* w, int64_t n, double eps, uint16_t* out) {
    double sum_sq = 0.0;
    for (int64_t k = 0; k < n; ++k) {
        double v = mo_bf16_to_f64(x[k]);
        sum_sq += v * v;
    }
    double rms = sqrt(sum_sq / (double)n + eps);
    for (int64_t k = 0; k < n; ++k) {
        out[k] = mo_f64_to_bf16(mo_bf16_to_f64(x[k]) * mo_bf16_to_f64(w[k]) / rms);
    }
}

/* ------------------------------------------------------------------------------------ */
/* Input stage for one sequence ([mtp] `forward_one`, before the block):                */
/*   e         = embed[token, :]            (row `token` of the [V, H] table)            */
/*   concat    = [ enorm(e) | hnorm(hidden) ]   ([2H], BF16)                             */
/*   x[n]      = bf16( sum_k eh_proj[n, k] * concat[k] ),  eh_proj is [H, 2H] row-major  */
/* concat_out (2H) and x_sum_out (H, the fp64 sums before the BF16 rounding) may be     */
/* NULL. Returns MO_ERR_TOKEN_RANGE (and a zero x) when token is outside [0, V).         */
/* ------------------------------------------------------------------------------------ */
int mo_input_stage(const uint16_t* embed, const uint16_t* enorm_w, const uint16_t* hnorm_w,
                   const uint16_t* eh_proj, int64_t token, const uint16_t* hidden,
                   int64_t H, int64_t V, double eps, uint16_t* concat_out, uint16_t* x_out,
                   double* x_sum_out, uint16_t* concat_scratch /* 2H */) {
    if (token < 0 || token >= V) {
        for (int64_t n = 0; n < H; ++n) x_out[n] = 0;
        if (x_sum_out) for (int64_t n = 0; n < H; ++n) x_sum_out[n] = 0.0;
        if (concat_out) memset(concat_out, 0, (size_t)(2 * H) * sizeof(uint16_t));
        return MO_ERR_TOKEN_RANGE;
    }
    uint16_t* c = concat_scratch;
    mo_rms_norm(embed + token * H, enorm_w, H, eps, c);
    mo_rms_norm(hidden, hnorm_w, H, eps, c + H);
    for (int64_t n = 0; n < H; ++n) {
        double acc = 0.0;
        const uint16_t* row = eh_proj + n * (2 * H);
        for (int64_t k = 0; k < 2 * H; ++k) acc += mo_bf16_to_f64(row[k]) * mo_bf16_to_f64(c[k]);
        x_out[n] = mo_f64_to_bf16(acc);
        if (x_sum_out) x_sum_out[n] = acc;
    }
    if (concat_out) memcpy(concat_out, c, (size_t)(2 * H) * sizeof(uint16_t));
    return MO_OK;
}

/* ------------------------------------------------------------------------------------ */
/* lm_head logits over rows [v0, v1) for one normalised vector xhat ([mtp] `forward_one`:*/
/* shared_head.norm, then the lm_head gemv over the whole vocabulary).                   */
/*   BF16 head : logit[v] = sum_k W[v, k] * xhat[k]                                      */
/*   FP8 head  : logit[v] = sum_k (decode(Q[v, k]) * s[v]) * xhat[k]  (dequantised head) */
/* w_dtype 0 = BF16 (W is uint16), 1 = FP8 E4M3 (W is uint8, scale required).            */
/* ------------------------------------------------------------------------------------ */
void mo_logits(int w_dtype, const void* W, const float* scale, const uint16_t* xhat,
               int64_t H, int64_t v0, int64_t v1, double* out) {
    for (int64_t v = v0; v < v1; ++v) {
        double acc = 0.0;
        if (w_dtype == 0) {
            const uint16_t* row = (const uint16_t*)W + v * H;
            for (int64_t k = 0; k < H; ++k) acc += mo_bf16_to_f64(row[k]) * mo_bf16_to_f64(xhat[k]);
        } else {
            const uint8_t* row = (const uint8_t*)W + v * H;
            double s = (double)scale[v];
            for (int64_t k = 0; k < H; ++k) acc += (mo_e4m3_to_f64(row[k]) * s) * mo_bf16_to_f64(xhat[k]);
        }
        out[v - v0] = acc;
    }
}

/* Logits of an explicit list of rows (for sampled checks at full size). */
void mo_logits_rows(int w_dtype, const void* W, const float* scale, const uint16_t* xhat,
                    int64_t H, const int64_t* rows, int64_t n_rows, double* out) {
    for (int64_t i = 0; i < n_rows; ++i) mo_logits(w_dtype, W, scale, xhat, H, rows[i], rows[i] + 1, out + i);
}

/* ------------------------------------------------------------------------------------ */
/* argmax with the lowest index winning among equal maxima (the `>=` rule of [mtp]       */
/* `forward_one`'s cross-rank pick, extended to every index). NaN never wins; -inf can   */
/* win only if nothing larger exists. Returns -1 when every entry is NaN or n == 0.      */
/* ------------------------------------------------------------------------------------ */
int64_t mo_argmax(const double* v, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
        if (isnan(v[i])) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best;
}

/* ------------------------------------------------------------------------------------ */
/* The pick over vocabulary shards ([mtp] the vocab-shard fields `head_rank`, `head_v0`, */
/* `head_n` and `forward_one`'s sharded branch: each rank sweeps its own row range and   */
/* the ranks' (max logit, global index) pairs decide the draft; `>=` lets the lower     */
/* rank, i.e. the lower row range, win a tie). Shard r offers (value[r], index[r]), its */
/* own lowest-index maximum as a global row index, or index < 0 when it has none (no    */
/* rows, or all NaN). Returns the index of the largest value, the lowest index among    */
/* equal values, or -1 when no shard offers anything. NaN never wins.                   */
/* ------------------------------------------------------------------------------------ */
int64_t mo_pick_combine(const double* value, const int64_t* index, int64_t R) {
    int64_t best = -1;
    double best_v = 0.0;
    for (int64_t r = 0; r < R; ++r) {
        if (index[r] < 0 || isnan(value[r])) continue;
        if (best < 0 || value[r] > best_v || (value[r] == best_v && index[r] < best)) {
            best = index[r];
            best_v = value[r];
        }
    }
    return best;
}

/* ------------------------------------------------------------------------------------ */
/* The source's own two-rank exchange ([mtp] `forward_one`, sharded branch, and the      */
/* `head_xchg` field of the proposer state): eight BF16 lanes,                           */
/*   lane 0, 1          the max logit of rank 0, rank 1 (BF16, as the source's logits)   */
/*   lane 2 + 3r + d    digit d (d = 0, 1, 2; base 256, least significant first) of rank */
/*                      r's global index, as a BF16 number                               */
/* Each rank writes only its own lanes and leaves the rest zero; a SUM all-reduce over   */
/* BF16 elements then hands every rank both ranks' lanes unchanged (adding zero is       */
/* exact), and BF16 holds the integers 0..256 exactly, hence the base-256 digits. The    */
/* winner is rank 0 when lane 0 >= lane 1, else rank 1, and its digits give the index.   */
/* ------------------------------------------------------------------------------------ */
void mo_xchg_pack(int rank, uint16_t value_bf16, int64_t global_index, uint16_t* lanes) {
    for (int i = 0; i < 8; ++i) lanes[i] = 0;
    lanes[rank] = value_bf16;
    for (int d = 0; d < 3; ++d) {
        double digit = (double)((global_index >> (8 * d)) & 0xFF);
        lanes[2 + rank * 3 + d] = mo_f64_to_bf16(digit);
    }
}

/* The SUM all-reduce of two ranks' lanes: each lane is the BF16 rounding of the sum. */
void mo_xchg_sum(const uint16_t* a, const uint16_t* b, uint16_t* out) {
    for (int i = 0; i < 8; ++i) out[i] = mo_f64_to_bf16(mo_bf16_to_f64(a[i]) + mo_bf16_to_f64(b[i]));
}

int64_t mo_xchg_pick(const uint16_t* lanes) {
    int win = (mo_bf16_to_f64(lanes[0]) >= mo_bf16_to_f64(lanes[1])) ? 0 : 1;
    int64_t index = 0;
    for (int d = 0; d < 3; ++d) index += (int64_t)mo_bf16_to_f64(lanes[2 + win * 3 + d]) << (8 * d);
    return index;
}

/* ------------------------------------------------------------------------------------ */
/* FP8 quantiser for one row ([mtp] `head_fp8` doc: the E4M3 copy of lm_head).          */
/*   s = fp32(absmax_k |w_k| / 448);  q_k = e4m3_rne_satfinite( fp32(w_k / s) )          */
/* A zero row gives s = 0 and zero codes. Returns MO_ERR_NONFINITE if any weight is NaN  */
/* or Inf (the copy is then unusable; the outputs are left as zero).                     */
/* The two divisions are IEEE binary32 divisions, as the reading of the scale states.    */
/* ------------------------------------------------------------------------------------ */
int mo_quantize_row(const uint16_t* w, int64_t H, uint8_t* q, float* scale) {
    float absmax = 0.0f;
    for (int64_t k = 0; k < H; ++k) {
        float f = (float)mo_bf16_to_f64(w[k]);
        if (isnan(f) || isinf(f)) {
            memset(q, 0, (size_t)H);
            *scale = 0.0f;
            return MO_ERR_NONFINITE;
        }
        float m = fabsf(f);
        if (m > absmax) absmax = m;
    }
    volatile float s = absmax / 448.0f; /* volatile: keep it a binary32 value */
    *scale = s;
    for (int64_t k = 0; k < H; ++k) {
        if (s == 0.0f) {
            q[k] = 0;
        } else {
            volatile float quotient = (float)mo_bf16_to_f64(w[k]) / s;
            q[k] = mo_f64_to_e4m3((double)quotient);
        }
    }
    return MO_OK;
}

int mo_quantize(const uint16_t* w, int64_t V, int64_t H, uint8_t* q, float* scale) {
    int status = MO_OK;
    for (int64_t v = 0; v < V; ++v) {
        int r = mo_quantize_row(w + v * H, H, q + v * H, scale + v);
        if (r != MO_OK) status = r;
    }
    return status;
}
