/*
 * Engram forward oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what one Engram layer
 * computes, written from the vLLM API pages for DeepSeek-V4.1 Engram:
 *   - "vllm.models.deepseek_v4_1.common.engram", class Engram (docstring,
 *     __init__, forward), class EngramLayout, class ParallelEngramEmbedding
 *     (lookup);
 *   - "vllm.models.deepseek_v41.amd.engram", _engram_gate_finish_kernel and
 *     _engram_gate_partials_kernel (the gate arithmetic; with one rank the
 *     finish kernel is the generic post-wkv kernel, per its docstring);
 *   - "vllm.models.deepseek_v41.amd.mono.attention.gemv", module docstring
 *     (MXFP8 weight layout: e4m3 [N, K] row-major, E8M0 scales per 32x32
 *     block, [N/32, K/32]).
 *
 * Every floating-point step runs in IEEE double.  Nothing here is blocked,
 * fused or reordered beyond the plain definition.  Only tests/, the smoke
 * check and the benchmark's CPU-baseline leg may load this library; the
 * product path never does.  It shares no code with the CUDA path.
 *
 * Pins (tests marked "not gpu"): layout primes against sympy.nextprime;
 * bf16/e4m3/E8M0 decoding against torch's dtype conversions and ldexp;
 * e4m3 and bf16 rounding against torch casts and constructed ties; the fp8
 * table gather against torch's e4m3 decode with exact power-of-two scaling; the
 * contraction against numpy's float64 matmul; the gate against closed
 * forms (identity projection, q = 0, sign symmetry, all-False mask).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP MX v1.0 E4M3 ("fn"): sign, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there
 * is no infinity.  (Engram table and wkv storage per the pages.) */
double oracle_e4m3_to_f64(uint8_t code) {
    int s = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* OCP MX v1.0 E8M0 scale: 2^(b - 127); 255 is NaN. */
double oracle_e8m0_to_f64(uint8_t b) {
    if (b == 255) return NAN;
    return ldexp(1.0, (int)b - 127);
}

/* Round an exact value to E4M3 with round-to-nearest, ties to even
 * mantissa, saturating to +-448 (never NaN).  Brute force: scan every
 * finite non-negative code and keep the nearest. */
uint8_t oracle_f64_to_e4m3_satfinite(double x) {
    double a = fabs(x);
    int best = 0;
    double best_err = INFINITY;
    if (isnan(x)) return 0x7F;
    if (a >= 448.0) return (uint8_t)((signbit(x) ? 0x80 : 0) | 0x7E);
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    /* the sign survives rounding, so a small negative value gives -0 */
    return (uint8_t)((signbit(x) ? 0x80 : 0) | best);
}

/* Round a double to bf16 (8 significant bits, 8 exponent bits), nearest,
 * ties to even.  Works from the exact value, so there is no double
 * rounding through binary32. */
uint16_t oracle_f64_to_bf16(double x) {
    uint32_t u;
    float f;
    double r;
    int e;
    if (isnan(x)) return 0x7FC0;
    if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
    if (fabs(x) < ldexp(1.0, -126)) {
        /* subnormal range: spacing 2^-133 */
        r = nearbyint(ldexp(x, 133));
        r = ldexp(r, -133);
    } else {
        (void)frexp(x, &e); /* x = f * 2^e, 0.5 <= |f| < 1 */
        r = nearbyint(ldexp(x, 8 - e)); /* 8 significant bits */
        r = ldexp(r, e - 8);
        /* largest finite bf16 is (2 - 2^-7) * 2^127 */
        if (fabs(r) > ldexp(255.0, 120)) r = x > 0 ? INFINITY : -INFINITY;
    }
    f = (float)r; /* exact: r has <= 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------ */
/* EngramLayout (class EngramLayout, __init__)                         */
/* ------------------------------------------------------------------ */

static int is_prime(int64_t n) {
    if (n < 2) return 0;
    if (n % 2 == 0) return n == 2;
    for (int64_t d = 3; d * d <= n; d += 2)
        if (n % d == 0) return 0;
    return 1;
}

/* Bucket sizes: for every layer, for every n-gram order 2..max, the
 * counter restarts at vocab_size - 1 and each head takes the next prime
 * strictly above the counter that no earlier (layer, order, head) took.
 * primes: [n_layers, (max_ngram_size-1)*n_heads]; offsets: the exclusive
 * cumulative sum within each layer.  Returns 0, or -1 on bad arguments. */
int oracle_layout(int64_t vocab_size, int max_ngram_size, int n_heads,
                  int n_layers, int64_t* primes, int64_t* offsets) {
    int cols = (max_ngram_size - 1) * n_heads;
    if (vocab_size < 1 || max_ngram_size < 2 || n_heads < 1 || n_layers < 1)
        return -1;
    for (int l = 0; l < n_layers; ++l) {
        for (int o = 0; o < max_ngram_size - 1; ++o) {
            int64_t current = vocab_size - 1;
            for (int h = 0; h < n_heads; ++h) {
                for (;;) {
                    int taken = 0;
                    ++current;
                    if (!is_prime(current)) continue;
                    /* skip primes already used by any earlier bucket */
                    for (int l2 = 0; l2 <= l && !taken; ++l2) {
                        int lim = (l2 < l) ? cols : o * n_heads + h;
                        for (int c = 0; c < lim; ++c)
                            if (primes[(int64_t)l2 * cols + c] == current) {
                                taken = 1;
                                break;
                            }
                    }
                    if (!taken) break;
                }
                primes[(int64_t)l * cols + o * n_heads + h] = current;
            }
        }
        int64_t acc = 0;
        for (int c = 0; c < cols; ++c) {
            offsets[(int64_t)l * cols + c] = acc;
            acc += primes[(int64_t)l * cols + c];
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Hash-row gather (ParallelEngramEmbedding.lookup, Engram.embed)      */
/* ------------------------------------------------------------------ */

/* rows[t, c, :] = table[row_offset[c] + ids[t, c], :] -- bytes copied.
 * ids are per-column local ids; an id outside [0, rows[c]) produces a
 * zero row and is counted in *n_bad.  table: bf16 bits [total_rows, E];
 * ids: int32, row stride ids_stride (elements); out: [T, C, E]. */
void oracle_gather(const uint16_t* table, const int64_t* row_offset,
                   const int64_t* rows, int64_t C, int64_t E,
                   const int32_t* ids, int64_t ids_stride, int64_t T,
                   uint16_t* out, int64_t* n_bad) {
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < C; ++c) {
            int64_t id = ids[t * ids_stride + c];
            uint16_t* dst = out + (t * C + c) * E;
            if (id < 0 || id >= rows[c]) {
                ++bad;
                for (int64_t j = 0; j < E; ++j) dst[j] = 0;
                continue;
            }
            const uint16_t* src = table + (row_offset[c] + id) * E;
            for (int64_t j = 0; j < E; ++j) dst[j] = src[j];
        }
    }
    if (n_bad) *n_bad = bad;
}

/* The same gather from an fp8 table (class ParallelEngramEmbedding: rows
 * stored as e4m3 with one ue8m0 scale per 32 consecutive elements,
 * dequantized on lookup into bf16): element j of a row is
 * e4m3(codes[row, j]) * 2^(scales[row, j / 32] - 127), rounded to bf16
 * (nearest, ties to even).  codes: [total_rows, E] bytes; scales:
 * [total_rows, E / 32] bytes; E a multiple of 32.  Bad ids as above. */
void oracle_gather_e4m3(const uint8_t* codes, const uint8_t* scales,
                        const int64_t* row_offset, const int64_t* rows, int64_t C,
                        int64_t E, const int32_t* ids, int64_t ids_stride, int64_t T,
                        uint16_t* out, int64_t* n_bad) {
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t c = 0; c < C; ++c) {
            int64_t id = ids[t * ids_stride + c];
            uint16_t* dst = out + (t * C + c) * E;
            if (id < 0 || id >= rows[c]) {
                ++bad;
                for (int64_t j = 0; j < E; ++j) dst[j] = 0;
                continue;
            }
            int64_t row = row_offset[c] + id;
            for (int64_t j = 0; j < E; ++j) {
                double v = oracle_e4m3_to_f64(codes[row * E + j]) *
                           oracle_e8m0_to_f64(scales[row * (E / 32) + j / 32]);
                dst[j] = oracle_f64_to_bf16(v);
            }
        }
    }
    if (n_bad) *n_bad = bad;
}

/* ------------------------------------------------------------------ */
/* wkv projection (Engram.__init__ wkv, Engram.forward)                */
/* ------------------------------------------------------------------ */

/* kv[t, n] = sum_k A[t, k] * W[n, k], A = the gathered rows flattened
 * [T, C*E] (k = c*E + j), W in the Linear layout [N, K].  bf16 weights. */
void oracle_wkv_bf16(const uint16_t* A, int64_t T, int64_t K,
                     const uint16_t* W, int64_t N, double* kv) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_f64(A[t * K + k]) *
                       oracle_bf16_to_f64(W[n * K + k]);
            kv[t * N + n] = acc;
        }
}

/* Same contraction with MXFP8 weights: W[n, k] = e4m3(code[n, k]) *
 * 2^(scale[n/32, k/32] - 127), scales [N/32, K/32] row-major. */
void oracle_wkv_mxfp8(const uint16_t* A, int64_t T, int64_t K,
                      const uint8_t* Wq, const uint8_t* Ws, int64_t N,
                      double* kv) {
    int64_t kb = K / 32;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double w = oracle_e4m3_to_f64(Wq[n * K + k]) *
                           oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);
                acc += oracle_bf16_to_f64(A[t * K + k]) * w;
            }
            kv[t * N + n] = acc;
        }
}

/* MXFP8 activation quantisation (the MXFP8 wkv chain quantises its input
 * rows).  Per token, per 32 consecutive k: amax over the block; the
 * scale is the smallest power of two 2^e with amax <= 448 * 2^e (amax = 0
 * gives e = 0), e clamped to [-127, 127]; codes = RTNE-satfinite e4m3 of
 * x / 2^e.  codes [T, K], scales [T, K/32] as E8M0 bytes (e + 127). */
void oracle_mx_quantize(const uint16_t* A, int64_t T, int64_t K,
                        uint8_t* codes, uint8_t* scales) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t b = 0; b < K / 32; ++b) {
            double amax = 0.0;
            int e = 0;
            for (int j = 0; j < 32; ++j) {
                double a = fabs(oracle_bf16_to_f64(A[t * K + b * 32 + j]));
                if (a > amax) amax = a;
            }
            if (amax > 0.0) {
                e = -127;
                while (e < 127 && amax > 448.0 * ldexp(1.0, e)) ++e;
            }
            scales[t * (K / 32) + b] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; ++j) {
                double x = oracle_bf16_to_f64(A[t * K + b * 32 + j]);
                codes[t * K + b * 32 + j] =
                    oracle_f64_to_e4m3_satfinite(ldexp(x, -e));
            }
        }
}

/* Contraction of MXFP8-quantised activations with MXFP8 weights: both
 * operands decoded to their exact values, products summed in double. */
void oracle_wkv_mxfp8_qact(const uint8_t* Aq, const uint8_t* As, int64_t T,
                           int64_t K, const uint8_t* Wq, const uint8_t* Ws,
                           int64_t N, double* kv) {
    int64_t kb = K / 32;
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = oracle_e4m3_to_f64(Aq[t * K + k]) *
                           oracle_e8m0_to_f64(As[t * kb + k / 32]);
                double w = oracle_e4m3_to_f64(Wq[n * K + k]) *
                           oracle_e8m0_to_f64(Ws[(n / 32) * kb + k / 32]);
                acc += a * w;
            }
            kv[t * N + n] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* Gate and residual (Engram.forward docstring; the finish kernel with */
/* one rank; the partials kernel for the per-hc sums)                  */
/* ------------------------------------------------------------------ */

/* For every token t and hc copy h:
 *   key   = kv[t, h*D : (h+1)*D],  value = kv[t, H*D : (H+1)*D]
 *   hr    = 1 / sqrt(sum_d hidden^2 / D + eps)
 *   kr    = 1 / sqrt(sum_d key^2 / D + eps)
 *   dot   = (sum_d hidden * q[h] * k[h] * key) * hr * kr / sqrt(D)
 *   gi    = sqrt(max(|dot|, clamp)), negated when dot < 0
 *   gate  = 1 / (1 + exp(-gi)), and 0 where token_mask is False
 *   out   = hidden + gate * value; masked positions copy hidden's bits.
 * hidden: bf16 bits, element (t, h, d) at t*hs[0] + h*hs[1] + d*hs[2];
 * kv: [T, (H+1)*D]; q, k: bf16 [H, D]; mask: one byte per token (0 =
 * False) or NULL (all True).  Outputs (each may be NULL): out_f64
 * [T, H, D], out_bf16 [T, H, D] (RTNE), gate [T, H], dot [T, H]. */
void oracle_gate(const uint16_t* hidden, const int64_t* hs, const double* kv,
                 const uint16_t* q, const uint16_t* k, const uint8_t* mask,
                 int64_t T, int64_t H, int64_t D, double eps, double clamp,
                 double* out_f64, uint16_t* out_bf16, double* gate_out,
                 double* dot_out) {
    int64_t N = (H + 1) * D;
    for (int64_t t = 0; t < T; ++t) {
        const double* value = kv + t * N + H * D;
        int active = mask ? (mask[t] != 0) : 1;
        for (int64_t h = 0; h < H; ++h) {
            const double* key = kv + t * N + h * D;
            const uint16_t* hid = hidden + t * hs[0] + h * hs[1];
            double s_hh = 0.0, s_kk = 0.0, s_hk = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                double x = oracle_bf16_to_f64(hid[d * hs[2]]);
                double qd = oracle_bf16_to_f64(q[h * D + d]);
                double kd = oracle_bf16_to_f64(k[h * D + d]);
                s_hh += x * x;
                s_kk += key[d] * key[d];
                s_hk += x * qd * kd * key[d];
            }
            double hr = 1.0 / sqrt(s_hh / (double)D + eps);
            double kr = 1.0 / sqrt(s_kk / (double)D + eps);
            double dot = s_hk * hr * kr / sqrt((double)D);
            double gi = sqrt(fmax(fabs(dot), clamp));
            if (dot < 0.0) gi = -gi;
            double gate = 1.0 / (1.0 + exp(-gi));
            if (!active) gate = 0.0;
            if (gate_out) gate_out[t * H + h] = gate;
            if (dot_out) dot_out[t * H + h] = dot;
            for (int64_t d = 0; d < D; ++d) {
                uint16_t xb = hid[d * hs[2]];
                int64_t o = (t * H + h) * D + d;
                if (!active) {
                    if (out_f64) out_f64[o] = oracle_bf16_to_f64(xb);
                    if (out_bf16) out_bf16[o] = xb; /* bits untouched */
                } else {
                    double y = oracle_bf16_to_f64(xb) + gate * value[d];
                    if (out_f64) out_f64[o] = y;
                    if (out_bf16) out_bf16[o] = oracle_f64_to_bf16(y);
                }
            }
        }
    }
}
