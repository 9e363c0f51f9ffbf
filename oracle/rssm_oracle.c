/*
 * ReplaySSM decode -- plain float64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library. The CUDA path never
 * does, and the two share no code.
 *
 * What it computes
 * ----------------
 * The pages ("ReplaySSM beschleunigt das Decoding von Hybridmodellen ...",
 * section "Wie es funktioniert"; the Turkish page, section "ReplaySSM nasil
 * calisir?") state that a replay decode produces the same outputs as the
 * conventional decode up to floating-point differences. The conventional decode
 * loads the state, decays and updates it, computes the output and stores the
 * state, one token at a time. So this oracle is that per-token recurrence,
 * written out in float64. It has no buffer, no checkpoint and no unrolling.
 *
 *   Mamba-2, per (sequence b, head h), group g = h / (H/G):
 *     a_t   = exp(dt_t * A_h)
 *     h_t   = a_t * h_{t-1} + dt_t * x_t (outer) B_t          (P x N)
 *     y_t   = h_t C_t + D_h * x_t                              (P)
 *   Gated DeltaNet, per (b, h), S in R^{d_v x d_k}:
 *     S_t   = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *           = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *     o_t   = S_t (scale * q_t)
 *
 * The output uses the post-update state, which is the reading the replay
 * output formula implies (its decay product includes a_t).
 *
 * Low-precision read copy (the Turkish page, section "Kuantizasyon hatasinin
 * sinirlandirilmasi"): the recurrence runs on the high-precision checkpoint,
 * and only output reads use the low-precision copy. The emulation below keeps
 * the exact float64 recurrence. It adds to each non-flush output the error of
 * the copy made at the last flush, carried forward by the decay since then.
 *
 * Quantisers follow the OCP 8-bit floating point specification (E4M3: bias 7,
 * max 448, no infinities, subnormals down to 2^-9) and the OCP Microscaling
 * (MX) v1.0 specification for FP4 E2M1 (values 0, 0.5, 1, 1.5, 2, 3, 4, 6).
 * Both round to nearest with ties to even and saturate to the largest finite
 * value. The scale arithmetic is done in float32, the precision the kernels
 * use, so the integer codes are decided in the same precision on both sides.
 *
 * Build with -ffp-contract=off: no fused multiply-add, on x86 or Arm.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL 1

int orc_version(void) { return 1; }

static void set_threads(int threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ======================================================================== */
/* Quantisers (float32 arithmetic, integer codes)                           */
/* ======================================================================== */

/* Round a non-negative float32 to the nearest integer, ties to even. */
static float rne_int(float r) {
    float fl = floorf(r);
    float diff = r - fl; /* exact: r and fl share the exponent range */
    if (diff > 0.5f) return fl + 1.0f;
    if (diff < 0.5f) return fl;
    return (fmodf(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

/* OCP FP8 E4M3: sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0.
 * Code magnitudes ordered by value. Between two adjacent binades the quantum is
 * 2^(e-3) and the code is (e+7)*8 + mantissa. So the integer
 * round(a / quantum) added to the binade's base code is the RNE code, and a
 * carry into the next binade falls out of the arithmetic. */
uint8_t orc_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    float a = fabsf(v);
    if (isnan(v)) return 0x7F;
    if (a >= 448.0f) return sign | 0x7E;             /* satfinite */
    int e;
    (void)frexpf(a, &e);                              /* a = f * 2^e, f in [0.5,1) */
    int ub = e - 1;                                   /* unbiased exponent of a */
    if (a == 0.0f || ub < -6) {
        /* subnormal binade: value = m * 2^-9, m in 0..7 ; m = 8 is 2^-6 */
        float q = rne_int(ldexpf(a, 9));
        return sign | (uint8_t)q;                     /* q <= 8, 8 = min normal */
    }
    float q = rne_int(ldexpf(a, 3 - ub));             /* in [8, 16] */
    int code = (ub + 7) * 8 + ((int)q - 8);
    if (code > 0x7E) code = 0x7E;
    return sign | (uint8_t)code;
}

double orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7) return NAN;
    double mag = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

/* OCP MX FP4 E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
uint8_t orc_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    float a = fabsf(v);
    if (isnan(v)) return 0x7;                         /* no NaN in E2M1: saturate */
    if (a >= 6.0f) return sign | 0x7;                 /* satfinite */
    if (a < 2.0f) {                                   /* quantum 0.5: codes 0..4 */
        float q = rne_int(a * 2.0f);
        return sign | (uint8_t)q;
    }
    if (a < 4.0f) {                                   /* quantum 1: 2,3,4 -> codes 4,5,6 */
        float q = rne_int(a);
        return sign | (uint8_t)(4 + ((int)q - 2));
    }
    float q = rne_int(a * 0.5f);                      /* quantum 2: 4,6 -> codes 6,7 */
    return sign | (uint8_t)(6 + ((int)q - 2));
}

double orc_e2m1_decode(uint8_t c) {
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[c & 7];
    return (c & 8) ? -v : v;
}

void orc_e4m3_encode_array(int64_t n, const float* src, uint8_t* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_e4m3_encode(src[i]);
}
void orc_e2m1_encode_array(int64_t n, const float* src, uint8_t* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_e2m1_encode(src[i]);
}

/* FP8 read copy of one tile of n float32 values:
 *   s = amax / 448, r = 1 / s (float32),  code_i = E4M3(x_i * r)  ;
 *   s == 0 -> all codes 0. */
static void quant_fp8_tile(int64_t n, const float* x, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
    float s = amax / 448.0f;
    *scale = s;
    float r = (s == 0.0f) ? 0.0f : 1.0f / s;
    for (int64_t i = 0; i < n; ++i) codes[i] = (s == 0.0f) ? 0 : orc_e4m3_encode(x[i] * r);
}

void orc_quant_fp8(int64_t tiles, int64_t n, const float* src, uint8_t* codes, float* scale) {
    for (int64_t t = 0; t < tiles; ++t) quant_fp8_tile(n, src + t * n, codes + t * n, scale + t);
}

void orc_dequant_fp8(int64_t tiles, int64_t n, const uint8_t* codes, const float* scale,
                     double* dst) {
    for (int64_t t = 0; t < tiles; ++t)
        for (int64_t i = 0; i < n; ++i)
            dst[t * n + i] = orc_e4m3_decode(codes[t * n + i]) * (double)scale[t];
}

/* NVFP4 read copy of one rows x cols tile (cols a multiple of 16):
 *   s_t  = amax_tile / (6*448)                      (float32, per tile)
 *   r6   = 1 / (6 * s_t)                            (float32, per tile)
 *   bs_j = E4M3( amax_block_j * r6 )                (per 16 consecutive elements of a row)
 *   es_j = decode(bs_j) * s_t, r_j = 1 / es_j       (float32)
 *   code = E2M1( x * r_j )    ; es_j == 0 -> code 0
 * Codes are packed two per byte, element 2i in the low nibble. */
static void quant_nvfp4_tile(int64_t rows, int64_t cols, const float* x, uint8_t* codes,
                             uint8_t* bscale, float* tscale) {
    int64_t n = rows * cols, nb = cols / 16;
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) { float a = fabsf(x[i]); if (a > amax) amax = a; }
    float st = amax / 2688.0f;
    *tscale = st;
    float st6 = 6.0f * st;
    float r6 = (st6 == 0.0f) ? 0.0f : 1.0f / st6;   /* one reciprocal per tile */
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t j = 0; j < nb; ++j) {
            const float* blk = x + r * cols + j * 16;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) { float a = fabsf(blk[i]); if (a > bmax) bmax = a; }
            uint8_t bs = (st6 == 0.0f) ? 0 : orc_e4m3_encode(bmax * r6);
            bscale[r * nb + j] = bs;
            float es = (float)orc_e4m3_decode(bs) * st;
            float rs = (es == 0.0f) ? 0.0f : 1.0f / es;
            uint8_t* out = codes + (r * cols + j * 16) / 2;
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = (es == 0.0f) ? 0 : orc_e2m1_encode(blk[i] * rs);
                uint8_t hi = (es == 0.0f) ? 0 : orc_e2m1_encode(blk[i + 1] * rs);
                out[i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

int orc_quant_nvfp4(int64_t tiles, int64_t rows, int64_t cols, const float* src,
                    uint8_t* codes, uint8_t* bscale, float* tscale) {
    if (cols % 16 != 0) return ORC_EINVAL;
    int64_t n = rows * cols;
    for (int64_t t = 0; t < tiles; ++t)
        quant_nvfp4_tile(rows, cols, src + t * n, codes + t * n / 2, bscale + t * n / 16,
                         tscale + t);
    return ORC_OK;
}

void orc_dequant_nvfp4(int64_t tiles, int64_t rows, int64_t cols, const uint8_t* codes,
                       const uint8_t* bscale, const float* tscale, double* dst) {
    int64_t n = rows * cols;
    for (int64_t t = 0; t < tiles; ++t)
        for (int64_t i = 0; i < n; ++i) {
            uint8_t byte = codes[(t * n + i) / 2];
            uint8_t c = (i & 1) ? (byte >> 4) : (byte & 0xF);
            double bs = orc_e4m3_decode(bscale[t * n / 16 + i / 16]);
            dst[t * n + i] = orc_e2m1_decode(c) * bs * (double)tscale[t];
        }
}

/* ======================================================================== */
/* Mamba-2 per-token recurrence                                             */
/* ======================================================================== */

/* One token for one (b, h) tile. h: P x N (row-major, N contiguous). */
static void m2_token(int64_t P, int64_t N, double A, double Dh, double* h, const double* x,
                     const double* Bv, const double* Cv, double dt, double* y) {
    double a = exp(dt * A);
    for (int64_t p = 0; p < P; ++p) {
        double* row = h + p * N;
        double dx = dt * x[p];
        double acc = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            row[n] = a * row[n] + dx * Bv[n];
            acc += row[n] * Cv[n];
        }
        y[p] = acc + Dh * x[p];
    }
}

/*
 * Run `steps` tokens of the Mamba-2 recurrence for every (b, h).
 *   h  [B][H][P][N]  in: state before the first token; out: after the last one
 *   x  [steps][B][H][P], Bm and C [steps][B][G][N], dt [steps][B][H]
 *   y  [steps][B][H][P]
 *   nsteps [B] or NULL: sequence b runs only its first nsteps[b] tokens
 *   (its later y entries are left untouched).
 */
int orc_m2_recurrence(int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, int64_t steps,
                      const double* A, const double* D, double* h, const double* x,
                      const double* Bm, const double* C, const double* dt,
                      const int32_t* nsteps, double* y, int threads) {
    if (B < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || steps < 0)
        return ORC_EINVAL;
    set_threads(threads);
    const int64_t hpg = H / G;
    const int64_t tiles = B * H;
#pragma omp parallel for schedule(static)
    for (int64_t tile = 0; tile < tiles; ++tile) {
        int64_t b = tile / H, hh = tile % H, g = hh / hpg;
        int64_t ns = nsteps ? nsteps[b] : steps;
        if (ns > steps) ns = steps;
        double* ht = h + tile * P * N;
        for (int64_t t = 0; t < ns; ++t) {
            const double* xt = x + ((t * B + b) * H + hh) * P;
            const double* bt = Bm + ((t * B + b) * G + g) * N;
            const double* ct = C + ((t * B + b) * G + g) * N;
            double dtt = dt[(t * B + b) * H + hh];
            m2_token(P, N, A[hh], D[hh], ht, xt, bt, ct, dtt, y + ((t * B + b) * H + hh) * P);
        }
    }
    return ORC_OK;
}

/* Quantise one float64 tile through float32 and return dequant - value. */
static void readcopy_delta(int fmt, int64_t P, int64_t N, const double* h, float* f32,
                           uint8_t* codes, uint8_t* bsc, double* deq, double* delta) {
    float ts;
    for (int64_t i = 0; i < P * N; ++i) f32[i] = (float)h[i];
    if (fmt == 1) {
        quant_fp8_tile(P * N, f32, codes, &ts);
        orc_dequant_fp8(1, P * N, codes, &ts, deq);
    } else {
        quant_nvfp4_tile(P, N, f32, codes, bsc, &ts);
        orc_dequant_nvfp4(1, P, N, codes, bsc, &ts, deq);
    }
    for (int64_t i = 0; i < P * N; ++i) delta[i] = deq[i] - h[i];
}

/*
 * Mamba-2 plain decode with a low-precision read copy (fmt 1 = FP8 E4M3 per
 * tile scale, 2 = NVFP4 with 16-element E4M3 block scales).
 *
 * The copy is made from the checkpoint at the start (count 0) and at every
 * flush, i.e. every k tokens. The checkpoint equals the exact state at that
 * point, rounded to float32. A non-flush token reads the copy in place of the
 * checkpoint, so its output is the exact output plus
 *     gamma * (copy - checkpoint) C_t,   gamma = product of a since the flush.
 * The flush token's output uses the exact state (it is computed from the
 * freshly folded high-precision checkpoint).
 */
int orc_m2_readcopy(int64_t B, int64_t H, int64_t P, int64_t N, int64_t G, int64_t steps,
                    const double* A, const double* D, double* h, const double* x,
                    const double* Bm, const double* C, const double* dt, int64_t k, int fmt,
                    double* y, int threads) {
    if (B < 0 || H <= 0 || P <= 0 || N <= 0 || G <= 0 || H % G != 0 || steps < 0 || k < 1 ||
        (fmt != 1 && fmt != 2) || (fmt == 2 && N % 16 != 0))
        return ORC_EINVAL;
    set_threads(threads);
    const int64_t hpg = H / G;
    const int64_t tiles = B * H;
    int err = ORC_OK;
#pragma omp parallel
    {
        float* f32 = (float*)malloc(sizeof(float) * P * N);
        uint8_t* codes = (uint8_t*)malloc(P * N);
        uint8_t* bsc = (uint8_t*)malloc(P * N / 16 + 1);
        double* deq = (double*)malloc(sizeof(double) * P * N);
        double* delta = (double*)malloc(sizeof(double) * P * N);
        double* yex = (double*)malloc(sizeof(double) * P);
        if (!f32 || !codes || !bsc || !deq || !delta || !yex) {
#pragma omp atomic write
            err = ORC_EINVAL;
        } else {
#pragma omp for schedule(static)
            for (int64_t tile = 0; tile < tiles; ++tile) {
                int64_t b = tile / H, hh = tile % H, g = hh / hpg;
                double* ht = h + tile * P * N;
                readcopy_delta(fmt, P, N, ht, f32, codes, bsc, deq, delta);
                double gamma = 1.0;
                int64_t count = 0;
                for (int64_t t = 0; t < steps; ++t) {
                    const double* xt = x + ((t * B + b) * H + hh) * P;
                    const double* bt = Bm + ((t * B + b) * G + g) * N;
                    const double* ct = C + ((t * B + b) * G + g) * N;
                    double dtt = dt[(t * B + b) * H + hh];
                    double* yt = y + ((t * B + b) * H + hh) * P;
                    m2_token(P, N, A[hh], D[hh], ht, xt, bt, ct, dtt, yex);
                    gamma *= exp(dtt * A[hh]);
                    count += 1;
                    if (count == k) {
                        for (int64_t p = 0; p < P; ++p) yt[p] = yex[p];
                        readcopy_delta(fmt, P, N, ht, f32, codes, bsc, deq, delta);
                        gamma = 1.0;
                        count = 0;
                    } else {
                        for (int64_t p = 0; p < P; ++p) {
                            double acc = 0.0;
                            for (int64_t n = 0; n < N; ++n) acc += delta[p * N + n] * ct[n];
                            yt[p] = yex[p] + gamma * acc;
                        }
                    }
                }
            }
        }
        free(f32); free(codes); free(bsc); free(deq); free(delta); free(yex);
    }
    return err;
}

/* ======================================================================== */
/* Gated DeltaNet per-token recurrence                                      */
/* ======================================================================== */

/*
 *   S  [B][H][DV][DK]  in/out
 *   q, k [steps][B][H][DK], v [steps][B][H][DV], alpha, beta [steps][B][H]
 *   o  [steps][B][H][DV]
 */
int orc_gdn_recurrence(int64_t B, int64_t H, int64_t DK, int64_t DV, int64_t steps,
                       double scale, double* S, const double* q, const double* k,
                       const double* v, const double* alpha, const double* beta,
                       const int32_t* nsteps, double* o, int threads) {
    if (B < 0 || H <= 0 || DK <= 0 || DV <= 0 || steps < 0) return ORC_EINVAL;
    set_threads(threads);
    const int64_t tiles = B * H;
    int err = ORC_OK;
#pragma omp parallel
    {
        double* sk = (double*)malloc(sizeof(double) * DV);
        if (!sk) {
#pragma omp atomic write
            err = ORC_EINVAL;
        } else {
#pragma omp for schedule(static)
            for (int64_t tile = 0; tile < tiles; ++tile) {
                int64_t b = tile / H, hh = tile % H;
                int64_t ns = nsteps ? nsteps[b] : steps;
                if (ns > steps) ns = steps;
                double* St = S + tile * DV * DK;
                for (int64_t t = 0; t < ns; ++t) {
                    int64_t bh = (t * B + b) * H + hh;
                    const double* qt = q + bh * DK;
                    const double* kt = k + bh * DK;
                    const double* vt = v + bh * DV;
                    double al = alpha[bh], be = beta[bh];
                    for (int64_t r = 0; r < DV; ++r) {          /* S_{t-1} k_t */
                        double acc = 0.0;
                        for (int64_t c = 0; c < DK; ++c) acc += St[r * DK + c] * kt[c];
                        sk[r] = acc;
                    }
                    double* ot = o + bh * DV;
                    for (int64_t r = 0; r < DV; ++r) {
                        double u = be * (vt[r] - al * sk[r]);
                        double acc = 0.0;
                        for (int64_t c = 0; c < DK; ++c) {
                            St[r * DK + c] = al * St[r * DK + c] + u * kt[c];
                            acc += St[r * DK + c] * (scale * qt[c]);
                        }
                        ot[r] = acc;
                    }
                }
            }
        }
        free(sk);
    }
    return err;
}
