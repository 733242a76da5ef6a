/*
 * oracle.c -- the CPU oracle for the attention forward and the Sage prepare.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; it is used by tests/, by the smoke check and by the benchmark's
 * CPU-baseline leg.  It shares no code, header, table or constant generator
 * with the CUDA library.
 *
 * It is deliberately plain and slow:
 *   - attention is the textbook definition O = softmax(scale * Q K^T) V
 *     evaluated per query row in FP64 (ai-infra handbook, "Kernel
 *     acceleration: attention, compilation and fusion", section "Attention:
 *     from O(N^2) memory to blocks", the `naive` form); no tiling, no online
 *     softmax;
 *   - the Sage prepare is the quantisation of the aiter pull request
 *     "gfx1201_sage_prepare / gfx1201_sage_attention" (commit message of
 *     gfx1201_sage_prepare; Technical Details), written step by step in IEEE
 *     binary32 with round-to-nearest-even and no fused multiply-add (this file
 *     must be compiled with -ffp-contract=off and without fast-math).  Where
 *     that page leaves a step open, the reading taken is written beside it.
 *
 * Tensors arrive as BF16 bit patterns (uint16) in contiguous [B, S, H, D]
 * order, D = 128 for everything but the attention definition, which takes any D.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- scalars */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* BF16 is the upper half of a binary32: widening is exact. */
float oracle_bf16_to_f32(uint16_t b) { return f32_from_bits((uint32_t)b << 16); }

/* Value of a BF16 magnitude pattern (sign bit clear) as a double, treating the
 * pattern one past the largest finite value as 2^128 (the next step of the
 * exponent scale) so that rounding near the top behaves like unbounded RNE. */
static double bf16_mag_value(uint32_t pat) {
    if (pat >= 0x7f80u) return ldexp(1.0, 128);
    return (double)f32_from_bits(pat << 16);
}

/* Round a finite binary32 to BF16, nearest, ties to the even pattern.
 * Brute force on the two neighbours: the pattern obtained by truncation and
 * the next one up in magnitude. */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u = bits_from_f32(f);
    uint32_t sign = u & 0x80000000u;
    uint32_t mag = u & 0x7fffffffu;
    if (mag > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);      /* NaN stays NaN */
    if (mag == 0x7f800000u) return (uint16_t)(u >> 16);                   /* +-inf */
    double a = fabs((double)f);
    uint32_t lo = mag >> 16, hi = lo + 1;
    double dl = a - bf16_mag_value(lo), dh = bf16_mag_value(hi) - a;
    uint32_t pick;
    if (dl < dh) pick = lo;
    else if (dh < dl) pick = hi;
    else pick = (lo & 1u) ? hi : lo;
    return (uint16_t)((sign >> 16) | pick);
}

/* FP8 e4m3 ("e4m3fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN.  Largest finite magnitude is
 * 1.75 * 2^8 = 448, smallest subnormal 2^-9. */
double oracle_e4m3_decode(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, e - 7);
    return s ? -v : v;
}

/* The 127 finite non-negative e4m3 magnitudes, indexed by code (they increase
 * with the code), filled from the definition above when the library is loaded,
 * before any thread can encode. */
static double e4m3_mag[127];
__attribute__((constructor)) static void e4m3_init(void) {
    for (int c = 0; c < 127; c++) e4m3_mag[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Encode a finite binary32 as e4m3: round to nearest, ties to the even code,
 * magnitudes at or above 448 saturate to 448 ("satfinite").  The sign of the
 * input is kept, zero included.  Bisection finds the two neighbouring finite
 * magnitudes; the nearer one wins, a tie goes to the even code. */
uint8_t oracle_e4m3_encode(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isnan(x)) return 0x7f;
    if (a >= 448.0) return sign | 126;
    int lo = 0, hi = 126;              /* invariant: mag[lo] <= a < mag[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_mag[mid] <= a) lo = mid; else hi = mid;
    }
    double dl = a - e4m3_mag[lo];
    double dh = e4m3_mag[hi] - a;
    int pick;
    if (dl < dh) pick = lo;
    else if (dh < dl) pick = hi;
    else pick = (lo & 1) ? hi : lo;
    return sign | (uint8_t)pick;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits with bias 15, 10 mantissa bits;
 * largest finite magnitude 65504, smallest subnormal 2^-24. */
double oracle_f16_decode(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
    if (e == 0) v = m * ldexp(1.0, -24);
    else v = (1.0 + m / 1024.0) * ldexp(1.0, e - 15);
    return s ? -v : v;
}

/* Round a finite double to binary16, nearest, ties to the even pattern (magnitudes
 * from halfway between 65504 and 2^16 up become infinity).  Bisection over the
 * 31744 finite magnitudes, which increase with the pattern. */
uint16_t oracle_f16_encode(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0x0000;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;
    int lo = 0, hi = 0x7c00;            /* invariant: value(lo) <= a < value(hi); value(0x7c00) := 2^16 */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (oracle_f16_decode((uint16_t)mid) <= a) lo = mid; else hi = mid;
    }
    double vh = (hi == 0x7c00) ? 65536.0 : oracle_f16_decode((uint16_t)hi);
    double dl = a - oracle_f16_decode((uint16_t)lo), dh = vh - a;
    int pick;
    if (dl < dh) pick = lo;
    else if (dh < dl) pick = hi;
    else pick = (lo & 1) ? hi : lo;
    return sign | (uint16_t)pick;
}

void oracle_f16_encode_array(const double* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f16_encode(x[i]);
}

void oracle_e4m3_encode_array(const float* x, uint8_t* out, int64_t n) {
    /* element by element; the threads only share the work (exhaustive checks encode
     * every binary32 of a range) */
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_encode(x[i]);
}
void oracle_e4m3_decode_array(const uint8_t* c, double* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_e4m3_decode(c[i]);
}
void oracle_f32_to_bf16_array(const float* x, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = oracle_f32_to_bf16(x[i]);
}

/* ------------------------------------------------------------- attention */

/* Threads for one call: nthreads if > 0, else all.  Passed as the parallel region's
 * num_threads clause, so a call never changes the count later calls see. */
static int oracle_team_size(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * O[b, s, h, :] = sum_j w_j V[b, j, h, :] / sum_j w_j,
 *   w_j = exp(t_j - max_j t_j),  t_j = scale * <Q[b, s, h, :], K[b, j, h, :]>,
 * all in FP64 from the exactly widened BF16 inputs.  Subtracting the row
 * maximum only keeps exp() finite; it cancels in the ratio.
 *
 * rows: optional list of flattened query rows r = (b*S + s)*H + h; NULL means
 * every row in order.  out: [n_rows, D] doubles.
 */
void oracle_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      int B, int S, int H, int D, double scale,
                      const int64_t* rows, int64_t n_rows, double* out, int nthreads) {
    int64_t total = rows ? n_rows : (int64_t)B * S * H;
    const int nt = oracle_team_size(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)S);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < total; i++) {
            int64_t r = rows ? rows[i] : i;
            int64_t h = r % H, s = (r / H) % S, b = r / ((int64_t)H * S);
            const uint16_t* qrow = q + ((b * S + s) * H + h) * D;
            for (int d = 0; d < D; d++) qd[d] = (double)oracle_bf16_to_f32(qrow[d]);
            double tmax = -INFINITY;
            for (int64_t j = 0; j < S; j++) {
                const uint16_t* krow = k + ((b * S + j) * H + h) * D;
                double dot = 0.0;
                for (int d = 0; d < D; d++) dot += qd[d] * (double)oracle_bf16_to_f32(krow[d]);
                t[j] = scale * dot;
                if (t[j] > tmax) tmax = t[j];
            }
            double wsum = 0.0;
            for (int d = 0; d < D; d++) acc[d] = 0.0;
            for (int64_t j = 0; j < S; j++) {
                double w = exp(t[j] - tmax);
                const uint16_t* vrow = v + ((b * S + j) * H + h) * D;
                wsum += w;
                for (int d = 0; d < D; d++) acc[d] += w * (double)oracle_bf16_to_f32(vrow[d]);
            }
            for (int d = 0; d < D; d++) out[i * D + d] = acc[d] / wsum;
        }
        free(t); free(qd); free(acc);
    }
}

/* ------------------------------------------------- Sage prepare: RMSNorm */

/*
 * RMSNorm of one 128-channel head row, with the BF16 rounding points of
 * PyTorch's eager ops (aiter pull request, gfx1201_sage_prepare commit message):
 *   y   = bf16( x * r ),   r = 1 / sqrt( mean(x^2) + eps )
 *   out = bf16( y * w )
 * with x widened from BF16 and every operation an IEEE binary32 operation.
 *
 * Reading (the page does not give a summation order): the sum of squares is
 * taken in eight partial sums, partial L = x[16L]^2 + ... + x[16L+15]^2 added
 * left to right, then combined pairwise like an XOR butterfly over the eight
 * partials with distances 4, 2, 1.  The mean is that sum times 1/128 (exact,
 * a power of two); sqrt and the reciprocal are each rounded once.
 */
static void rmsnorm_row(const uint16_t* x, const uint16_t* w, float eps, uint16_t* out) {
    float part[8];
    for (int L = 0; L < 8; L++) {
        float acc = 0.0f;
        for (int i = 0; i < 16; i++) {
            float xi = oracle_bf16_to_f32(x[16 * L + i]);
            float sq = xi * xi;
            acc = acc + sq;
        }
        part[L] = acc;
    }
    for (int dist = 4; dist >= 1; dist >>= 1) {
        float nxt[8];
        for (int L = 0; L < 8; L++) nxt[L] = part[L] + part[L ^ dist];
        memcpy(part, nxt, sizeof(part));
    }
    float sumsq = part[0];
    float ms = sumsq * (1.0f / 128.0f);
    float den = sqrtf(ms + eps);
    float r = 1.0f / den;
    for (int c = 0; c < 128; c++) {
        float xc = oracle_bf16_to_f32(x[c]);
        uint16_t y = oracle_f32_to_bf16(xc * r);
        float yw = oracle_bf16_to_f32(y) * oracle_bf16_to_f32(w[c]);
        out[c] = oracle_f32_to_bf16(yw);
    }
}

/*
 * Rotate-half RoPE on the first rope_dim channels of one head row at sequence
 * position s, for rope_dim of 32, 64, 96 or 128 (aiter pull request,
 * gfx1201_sage_prepare commit message).  With h = rope_dim / 2:
 *   rot[c] = -x[c + h] for c < h,   rot[c] = x[c - h] for h <= c < rope_dim
 *   out[c] = bf16( bf16(x[c] * cos[s, c]) + bf16(rot[c] * sin[s, c]) )
 * which is the eager BF16 sequence x*cos + rotate_half(x)*sin (each product
 * and the sum rounded to BF16).  Channels >= rope_dim pass through.
 */
static void rope_row(const uint16_t* x, const uint16_t* cosr, const uint16_t* sinr, int rope_dim,
                     uint16_t* out) {
    int h = rope_dim / 2;
    for (int c = 0; c < 128; c++) {
        if (c >= rope_dim) { out[c] = x[c]; continue; }
        float xc = oracle_bf16_to_f32(x[c]);
        float rot = (c < h) ? -oracle_bf16_to_f32(x[c + h]) : oracle_bf16_to_f32(x[c - h]);
        uint16_t a = oracle_f32_to_bf16(xc * oracle_bf16_to_f32(cosr[c]));
        uint16_t b = oracle_f32_to_bf16(rot * oracle_bf16_to_f32(sinr[c]));
        out[c] = oracle_f32_to_bf16(oracle_bf16_to_f32(a) + oracle_bf16_to_f32(b));
    }
}

/*
 * Optional fused pre-processing of Q or K: RMSNorm (when w != NULL), then RoPE
 * (when rope_dim > 0).  x, out: contiguous [B, S, H, 128]; cos/sin: [S, rope_dim].
 */
void oracle_norm_rope(const uint16_t* x, int B, int S, int H, const uint16_t* w, float eps,
                      const uint16_t* cos_t, const uint16_t* sin_t, int rope_dim, uint16_t* out) {
    int64_t nrow = (int64_t)B * S * H;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrow; r++) {
        int64_t s = (r / H) % S;
        uint16_t tmp[128];
        const uint16_t* src = x + r * 128;
        if (w) { rmsnorm_row(src, w, eps, tmp); src = tmp; }
        if (rope_dim > 0) {
            uint16_t tmp2[128];
            rope_row(src, cos_t + s * rope_dim, sin_t + s * rope_dim, rope_dim, tmp2);
            memcpy(out + r * 128, tmp2, sizeof(tmp2));
        } else {
            memcpy(out + r * 128, src, 128 * sizeof(uint16_t));
        }
    }
}

/* ---------------------------------------------- Sage prepare: Q/K to INT8 */

/*
 * INT8 codes for Q and K: each 32-row block of a (batch, head) has one FP32
 * scale, and Q's scales also hold softmax_scale * log2(e) (aiter pull request,
 * Technical Details).
 *
 * Readings: symmetric quantisation with the block's absolute maximum a over
 * its valid rows (rows < S):
 *   inv = 127 / a,  code = clamp(rint(x * inv), -127, 127)   (ties to even)
 *   scale = a / 127                    for K  (scale_mult = 1)
 *   scale = (a / 127) * scale_mult     for Q  (scale_mult = fl32(softmax_scale * log2 e))
 * a == 0 gives all-zero codes and scale 0.  The INT8 bytes therefore depend on
 * the tensor alone; the softmax factor lives in Q's scale.
 * With `mean` given ([B, H, 128], K smoothing, see oracle_k_mean) the value
 * quantised is fl32(x - mean[b, h, c]) in place of x, in both the block
 * maximum and the codes.
 * Output layout [B, H, S_pad, 128] (row-major); rows in [S, S_pad) are zero and
 * the scales of blocks wholly beyond S are zero.  scales: [B, H, S_pad / 32].
 */
void oracle_quant_qk(const uint16_t* x, int B, int S, int H, int64_t S_pad, float scale_mult,
                     const float* mean, int8_t* codes, float* scales) {
    int64_t nblk = S_pad / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            for (int64_t j = 0; j < nblk; j++) {
                int64_t r0 = 32 * j, r1 = r0 + 32 < S ? r0 + 32 : S;
                float a = 0.0f;
                const float* mu = mean ? mean + ((int64_t)b * H + h) * 128 : NULL;
                for (int64_t s = r0; s < r1; s++)
                    for (int c = 0; c < 128; c++) {
                        float xv = oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]);
                        if (mu) xv = xv - mu[c];
                        xv = fabsf(xv);
                        if (xv > a) a = xv;
                    }
                float inv = (a > 0.0f) ? 127.0f / a : 0.0f;
                for (int64_t s = r0; s < r0 + 32; s++) {
                    int8_t* dst = codes + (((int64_t)b * H + h) * S_pad + s) * 128;
                    for (int c = 0; c < 128; c++) {
                        if (s >= S || a == 0.0f) { dst[c] = 0; continue; }
                        float xv = oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]);
                        if (mu) xv = xv - mu[c];
                        float t = xv * inv;
                        float rq = rintf(t);
                        if (rq > 127.0f) rq = 127.0f;
                        if (rq < -127.0f) rq = -127.0f;
                        dst[c] = (int8_t)rq;
                    }
                }
                float sc = 0.0f;
                if (a > 0.0f) {
                    sc = a / 127.0f;
                    sc = sc * scale_mult;
                }
                scales[((int64_t)b * H + h) * nblk + j] = sc;
            }
        }
    }
}

/* ------------------------------------------- Sage prepare: K smoothing */

/*
 * SageAttention smooths K before quantising it: it subtracts the mean of K,
 * which takes out K's outlier channels (ai-infra handbook, "Kernel
 * acceleration: attention, compilation and fusion", section "SageAttention:
 * quantizing attention too").
 *
 * Reading: one mean per (batch, head, channel) over the S tokens of K (K after
 * the optional RMSNorm + RoPE, i.e. the tensor that is quantised), subtracted
 * before the INT8 quantisation (oracle_quant_qk with `mean`).  In exact
 * arithmetic the attention output does not change: every score of a query row
 * moves by the same q . mean, which the softmax cancels.
 *
 * The mean is a binary32 value that decides INT8 codes, so its summation
 * order is fixed (a deterministic function of K; the CUDA prepare follows the
 * same order).  For block j (rows 32j .. 32j+31, rows >= S skipped):
 *   P_g = (((0 + x[32j+g]) + x[32j+4+g]) + ...) + x[32j+28+g]     g = 0..3
 *   B_j = (P_0 + P_1) + (P_2 + P_3)
 *   total = ((0 + B_0) + B_1) + ... + B_{nblk-1},   mean = total / S
 * every + and the / in binary32, round to nearest even.
 * x: [B, S, H, 128] BF16 bits; mean: [B, H, 128].
 */
void oracle_k_mean(const uint16_t* x, int B, int S, int H, int64_t S_pad, float* mean) {
    int64_t nblk = S_pad / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            for (int c = 0; c < 128; c++) {
                float total = 0.0f;
                for (int64_t j = 0; j < nblk; j++) {
                    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    for (int g = 0; g < 4; g++)
                        for (int t = 0; t < 8; t++) {
                            int64_t s = 32 * j + 4 * t + g;
                            if (s < S) part[g] = part[g] + oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]);
                        }
                    float blk = (part[0] + part[1]) + (part[2] + part[3]);
                    total = total + blk;
                }
                mean[((int64_t)b * H + h) * 128 + c] = total / (float)S;
            }
        }
    }
}

/* ------------------------------------------- Sage prepare: Q smoothing */

/*
 * SageAttention subtracts the block means of Q as well as of K before the INT8
 * quantisation (ai-infra handbook, "Kernel acceleration: attention, compilation
 * and fusion", section "SageAttention: quantizing attention too").  For Q the
 * mean does not cancel in the softmax: with q = (q - qbar_B) + qbar_B,
 *   q . k_j = (q - qbar_B) . k_j + qbar_B . k_j,
 * and the second term, the correction, differs from key to key.  It is kept
 * with the block and added back in the score product.
 *
 * Readings (the page gives only the idea):
 *   - the block is the format's 32-row quantisation block (rows < S only); its
 *     mean per channel is summed in the order of oracle_k_mean's block sums,
 *       P_g = (((0 + x[32j+g]) + x[32j+4+g]) + ...) + x[32j+28+g],  g = 0..3,
 *       qbar[c] = ((P_0 + P_1) + (P_2 + P_3)) / n      (n = valid rows),
 *     every + and the / in binary32;
 *   - d = fl32(x - qbar[c]) is quantised like Q: a = max |d| over the block's
 *     valid rows, code = clamp(rint(fl32(d * inv)), -127, 127);
 *   - the mean is kept in units of the block's step, m[c] = qbar[c] * inv, as an
 *     IEEE binary16 value m16[c] = f16(fl32(qbar[c] * inv)): the score product
 *     takes Q's operand as the 16-bit value f16(code + m16) (see
 *     oracle_sage_attention), so that operand is exact only up to binary16;
 *   - to keep |m| within binary16's range the step is never below the block's
 *     largest |qbar| over 256 x 127: the block uses a_eff = max(a, fl32(max_c
 *     |qbar[c]| * 2^-8)), inv = fl32(127 / a_eff), scale = fl32(fl32(a_eff / 127)
 *     * scale_mult), so |m| <= 32512 (1 + 2^-23);
 *   - a block with a_eff = 0 (all zero), or whose 127 / a_eff overflows (a_eff
 *     below 127 / FLT_MAX: every score it touches is below 1e-34), is stored as
 *     zero codes, zero mean and scale 0; rows in [S, S_pad) are zero codes.
 * codes: [B, H, S_pad, 128]; scales: [B, H, S_pad/32]; mean16: [B, H, S_pad/32, 128]
 * binary16 bit patterns.
 */
void oracle_quant_q_smooth(const uint16_t* x, int B, int S, int H, int64_t S_pad, float scale_mult,
                           int8_t* codes, float* scales, uint16_t* mean16) {
    int64_t nblk = S_pad / 32;
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            for (int64_t j = 0; j < nblk; j++) {
                int64_t r0 = 32 * j, r1 = r0 + 32 < S ? r0 + 32 : S;
                int64_t n = r1 - r0;
                int8_t* dst0 = codes + (((int64_t)b * H + h) * S_pad + r0) * 128;
                uint16_t* m16 = mean16 + (((int64_t)b * H + h) * nblk + j) * 128;
                float* sc = scales + ((int64_t)b * H + h) * nblk + j;
                memset(dst0, 0, 32 * 128);
                for (int c = 0; c < 128; c++) m16[c] = 0;
                *sc = 0.0f;
                if (n <= 0) continue;
                float mu[128];
                for (int c = 0; c < 128; c++) {
                    float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    for (int g = 0; g < 4; g++)
                        for (int t = 0; t < 8; t++) {
                            int64_t s = r0 + 4 * t + g;
                            if (s < S) part[g] = part[g] + oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]);
                        }
                    float blk = (part[0] + part[1]) + (part[2] + part[3]);
                    mu[c] = blk / (float)n;
                }
                float a = 0.0f, cm = 0.0f;
                for (int64_t s = r0; s < r1; s++)
                    for (int c = 0; c < 128; c++) {
                        float d = oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]) - mu[c];
                        if (fabsf(d) > a) a = fabsf(d);
                    }
                for (int c = 0; c < 128; c++)
                    if (fabsf(mu[c]) > cm) cm = fabsf(mu[c]);
                float floor_step = cm * (1.0f / 256.0f);
                float ae = a > floor_step ? a : floor_step;
                if (!(ae > 0.0f)) continue;
                float inv = 127.0f / ae;
                if (isinf(inv)) continue;
                for (int64_t s = r0; s < r1; s++) {
                    int8_t* dst = codes + (((int64_t)b * H + h) * S_pad + s) * 128;
                    for (int c = 0; c < 128; c++) {
                        float d = oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]) - mu[c];
                        float t = d * inv;
                        float rq = rintf(t);
                        if (rq > 127.0f) rq = 127.0f;
                        if (rq < -127.0f) rq = -127.0f;
                        dst[c] = (int8_t)rq;
                    }
                }
                for (int c = 0; c < 128; c++) {
                    float m = mu[c] * inv;
                    m16[c] = oracle_f16_encode((double)m);
                }
                float st = ae / 127.0f;
                *sc = st * scale_mult;
            }
        }
    }
}

/* ----------------------------------------------- Sage prepare: V to e4m3 */

/*
 * e4m3 codes for V, stored channel-major as [B, H, 128, S_pad], each channel
 * with one FP32 scale (aiter pull request, Technical Details).
 *
 * Readings: one scale per (batch, head, channel) from the channel's absolute
 * maximum a over all valid positions s < S; inv = 448 / a (448 being the
 * largest e4m3 value); code = e4m3_rn_satfinite(v * inv); scale = a / 448.
 * a == 0 gives zero codes and scale 0.  Positions in [S, S_pad) are zero.
 * codes: [B, H, 128, S_pad]; scales: [B, H, 128].
 */
void oracle_quant_v(const uint16_t* x, int B, int S, int H, int64_t S_pad, uint8_t* codes, float* scales) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < H; h++) {
            for (int c = 0; c < 128; c++) {
                float a = 0.0f;
                for (int64_t s = 0; s < S; s++) {
                    float xv = fabsf(oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]));
                    if (xv > a) a = xv;
                }
                float inv = (a > 0.0f) ? 448.0f / a : 0.0f;
                uint8_t* dst = codes + (((int64_t)b * H + h) * 128 + c) * S_pad;
                for (int64_t s = 0; s < S_pad; s++) {
                    if (s >= S || a == 0.0f) { dst[s] = 0; continue; }
                    float xv = oracle_bf16_to_f32(x[(((int64_t)b * S + s) * H + h) * 128 + c]);
                    float t = xv * inv;
                    dst[s] = oracle_e4m3_encode(t);
                }
                scales[((int64_t)b * H + h) * 128 + c] = (a > 0.0f) ? a / 448.0f : 0.0f;
            }
        }
    }
}

/* ---------------------------------- the exact result of the Sage format */

/*
 * FP64 attention on prepared tensors, the function the Sage forward
 * approximates (aiter pull request "gfx1201_sage_prepare /
 * gfx1201_sage_attention", commit message of gfx1201_sage_attention: scores
 * from the INT8 codes, with softmax_scale * log2(e) inside Q's scales, V from
 * its e4m3 codes and per-channel scales):
 *   t_j = (sum_d q_i8[r, d] k_i8[j, d]) * q_scale[r / 32] * k_scale[j / 32]   (log2 units)
 *   O[r, d] = sum_{j < S} 2^(t_j - max t) v[j, d] / sum_{j < S} 2^(t_j - max t),
 *   v[j, d] = e4m3(v_fp8[d, j]) * v_scale[d]
 * with nothing rounded.  p_e4m3 != 0 adds the one rounding the forward's FP8
 * P V product needs (same commit message: "FP8 WMMA for P V"); reading: the
 * weights w_j = 2^(t_j - max t) in (0, 1] enter the numerator as
 * e4m3(448 w_j) / 448 while the denominator sums the unrounded w_j.
 * With Q smoothing (qm16 != NULL: [B, H, S_pad/32, 128] binary16 block means in
 * step units, oracle_quant_q_smooth) q_i8[r, d] above is replaced by Q's 16-bit
 * operand f16(q_i8[r, d] + qm16[r/32, d]) (q_operand), which carries the
 * correction term qbar . k_j.
 * abs_v != 0 evaluates the same weights on |v| instead (the weighted mean
 * magnitude the rounding bounds of the tests scale with).
 * Layouts: codes [B, H, S_pad, 128] and [B, H, 128, S_pad], scales
 * [B, H, S_pad/32] and [B, H, 128].  rows: flattened (b*S + s)*H + h.
 */
/* Q's operand of the score product for row r, channel d: the INT8 code, or with Q
 * smoothing (qm16 != NULL, see oracle_quant_q_smooth) the binary16 value
 * f16(code + m16[block, d]), the code and the block mean in step units summed
 * exactly and rounded once. */
static void q_operand(const int8_t* qrow, const uint16_t* qm16, double* qa) {
    for (int d = 0; d < 128; d++) {
        if (qm16) qa[d] = oracle_f16_decode(oracle_f16_encode((double)qrow[d] + oracle_f16_decode(qm16[d])));
        else qa[d] = (double)qrow[d];
    }
}

void oracle_sage_attention(const int8_t* q8, const int8_t* k8, const uint8_t* v8, const float* qs,
                           const float* ks, const float* vs, const uint16_t* qm16, int B, int S, int H,
                           int64_t S_pad, const int64_t* rows, int64_t n_rows, int abs_v, int p_e4m3, double* out,
                           int nthreads) {
    int64_t nblk = S_pad / 32;
    (void)B;
    const int nt = oracle_team_size(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)S);
        double acc[128];
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; i++) {
            int64_t r = rows[i];
            int64_t h = r % H, s = (r / H) % S, b = r / ((int64_t)H * S);
            int64_t bh = b * H + h;
            const int8_t* qrow = q8 + (bh * S_pad + s) * 128;
            double qa[128];
            q_operand(qrow, qm16 ? qm16 + (bh * nblk + s / 32) * 128 : NULL, qa);
            double fq = (double)qs[bh * nblk + s / 32];
            double tmax = -INFINITY;
            for (int64_t j = 0; j < S; j++) {
                const int8_t* krow = k8 + (bh * S_pad + j) * 128;
                /* binary64: exact for integer codes; with the 16-bit operand every product is
                   exact and the sum carries at most a 2^-53 relative rounding */
                double dot = 0.0;
                for (int d = 0; d < 128; d++) dot += qa[d] * (double)krow[d];
                t[j] = dot * fq * (double)ks[bh * nblk + j / 32];
                if (t[j] > tmax) tmax = t[j];
            }
            double wsum = 0.0;
            for (int d = 0; d < 128; d++) acc[d] = 0.0;
            for (int64_t j = 0; j < S; j++) {
                double w = exp2(t[j] - tmax);
                wsum += w;
                if (p_e4m3) w = oracle_e4m3_decode(oracle_e4m3_encode((float)(448.0 * w))) / 448.0;
                for (int d = 0; d < 128; d++) {
                    double vv = oracle_e4m3_decode(v8[(bh * 128 + d) * S_pad + j]) * (double)vs[bh * 128 + d];
                    acc[d] += w * (abs_v ? fabs(vv) : vv);
                }
            }
            for (int d = 0; d < 128; d++) out[i * 128 + d] = acc[d] / wsum;
        }
        free(t);
    }
}

/*
 * The same FP64 attention for the Sage mode whose P V product keeps V in 16-bit
 * precision: Q K^T on the INT8 codes as above, "P and V ... in FP8 or FP16"
 * (ai-infra handbook, "Kernel acceleration: attention, compilation and
 * fusion", section "SageAttention: quantizing attention too"), read here as
 * V taken from the BF16 input itself (no V quantisation):
 *   O[r, d] = sum_{j < S} 2^(t_j - max t) v[j, d] / sum_{j < S} 2^(t_j - max t),
 *   v[j, d] = the BF16 V of (b, j, h, d)
 * with t_j as in oracle_sage_attention (Q smoothing through qm16 as there) and
 * nothing rounded.  v: [B, S, H, 128] BF16 bits.  abs_v != 0 weights |v| instead.
 */
void oracle_sage_attention_v16(const int8_t* q8, const int8_t* k8, const float* qs, const float* ks,
                               const uint16_t* qm16, const uint16_t* v, int B, int S, int H, int64_t S_pad,
                               const int64_t* rows, int64_t n_rows, int abs_v, double* out, int nthreads) {
    int64_t nblk = S_pad / 32;
    (void)B;
    const int nt = oracle_team_size(nthreads);
    (void)nt;
#pragma omp parallel num_threads(nt)
    {
        double* t = (double*)malloc(sizeof(double) * (size_t)S);
        double acc[128];
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_rows; i++) {
            int64_t r = rows[i];
            int64_t h = r % H, s = (r / H) % S, b = r / ((int64_t)H * S);
            int64_t bh = b * H + h;
            const int8_t* qrow = q8 + (bh * S_pad + s) * 128;
            double qa[128];
            q_operand(qrow, qm16 ? qm16 + (bh * nblk + s / 32) * 128 : NULL, qa);
            double fq = (double)qs[bh * nblk + s / 32];
            double tmax = -INFINITY;
            for (int64_t j = 0; j < S; j++) {
                const int8_t* krow = k8 + (bh * S_pad + j) * 128;
                /* binary64: exact for integer codes; with the 16-bit operand every product is
                   exact and the sum carries at most a 2^-53 relative rounding */
                double dot = 0.0;
                for (int d = 0; d < 128; d++) dot += qa[d] * (double)krow[d];
                t[j] = dot * fq * (double)ks[bh * nblk + j / 32];
                if (t[j] > tmax) tmax = t[j];
            }
            double wsum = 0.0;
            for (int d = 0; d < 128; d++) acc[d] = 0.0;
            for (int64_t j = 0; j < S; j++) {
                double w = exp2(t[j] - tmax);
                wsum += w;
                const uint16_t* vrow = v + ((b * S + j) * H + h) * 128;
                for (int d = 0; d < 128; d++) {
                    double vv = (double)oracle_bf16_to_f32(vrow[d]);
                    acc[d] += w * (abs_v ? fabs(vv) : vv);
                }
            }
            for (int d = 0; d < 128; d++) out[i * 128 + d] = acc[d] / wsum;
        }
        free(t);
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
