/*
 * ROCmFP4 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 statement of what the ROCmFP4 block-quantised weight
 * product computes.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library; the product
 * path never does.  It shares no code, header, table or helper with the CUDA
 * library: everything below is written out again from the format's
 * definition.
 *
 * Source of the definitions: "Feasibility Report: Porting ROCmFP4 to Atlas",
 * section "What is ROCmFP4?", subsections "Block Layout", "Codebook10 Value
 * Table" and "Scale Format".
 *
 * Readings taken where that text is silent (each one is also pinned by the
 * CPU tests in tests/test_oracle.py):
 *   R1  nibble order inside qs[16]: byte j holds weight j in its low nibble
 *       and weight j+16 in its high nibble (the ggml Q4_0 order the type
 *       names Q4_0_ROCMFP4 / Q4_0_ROCMFP4_FAST point to).  Half 0 of a block
 *       is therefore the 16 low nibbles, half 1 the 16 high nibbles.
 *   R2  "decoded to half-scale values": the multiplier of a scale byte is
 *       one half of its unsigned-E4M3 value.
 *   R3  exponent field 0 decodes as an E4M3 subnormal, (M/8) * 2^-6.
 *   R4  a scale byte is finite iff it is below 0x7F: bit 7 set (no sign in
 *       an unsigned format) and 0x7F (exponent 15, mantissa 7) are rejected.
 *   R5  code 8 ("-0" in the table) is the value +0.
 *   R6  a row is K/32 blocks stored back to back, rows back to back, no
 *       padding; K must be a multiple of 32.
 * Parity with files written by the original implementation (R1, R2) is
 * parity unpinned: no such file or printed example exists to compare with.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Codebook10, as printed in the "Codebook10 Value Table" subsection. */
static const int8_t oracle_codebook10[16] = {
    0, 1, 2, 3, 4, 6, 8, 10,
    0, -1, -2, -3, -4, -6, -8, -10,
};

/* Block layout ("Block Layout" subsection): qs[16] followed by two scale
 * bytes (dual-scale, 18 B) or one (fast single-scale, 17 B). */
enum { ORACLE_DUAL = 0, ORACLE_FAST = 1 };
enum { ORACLE_ACT_F16 = 0, ORACLE_ACT_BF16 = 1 };

int oracle_block_bytes(int variant) {
  if (variant == ORACLE_DUAL) return 18;
  if (variant == ORACLE_FAST) return 17;
  return -1;
}

int oracle_codebook(int q) { return oracle_codebook10[q & 15]; }

/* Finite unsigned-E4M3 scale byte?  ("Scale Format": row validation rejects
 * non-finite scale bytes; reading R4.) */
int oracle_scale_is_valid(unsigned s) { return s < 0x7Fu; }

/* Unsigned E4M3 value of a scale byte: 4 exponent bits (bias 7) above 3
 * mantissa bits; exponent 0 is subnormal (reading R3). */
double oracle_ue4m3_value(unsigned s) {
  unsigned e = (s >> 3) & 0xFu;
  unsigned m = s & 7u;
  if (e == 0) return ldexp((double)m / 8.0, -6);
  return ldexp(1.0 + (double)m / 8.0, (int)e - 7);
}

/* Half-scale multiplier of a scale byte (reading R2). */
double oracle_halfscale(unsigned s) { return 0.5 * oracle_ue4m3_value(s); }

/* Nibble i (0..31) of a block's qs[16] (reading R1). */
static unsigned oracle_nibble(const uint8_t *qs, int i) {
  unsigned byte = qs[i % 16];
  return (i < 16) ? (byte & 0xFu) : (byte >> 4);
}

/* Decode one block into its 32 weights: w_i = Codebook10[q_i] * hs(scale of
 * the half that weight i belongs to). */
void oracle_decode_block(const uint8_t *blk, int variant, double w[32]) {
  const uint8_t *qs = blk;
  for (int i = 0; i < 32; ++i) {
    unsigned s = (variant == ORACLE_DUAL) ? blk[16 + i / 16] : blk[16];
    double c = (double)oracle_codebook10[oracle_nibble(qs, i)];
    w[i] = c * oracle_halfscale(s);
    if (w[i] == 0.0) w[i] = 0.0; /* reading R5: no negative zero */
  }
}

/* IEEE binary16 bits -> double (exact). */
static double oracle_f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = (m == 0) ? INFINITY : NAN;
  else v = ldexp((double)(1024 + m), e - 25);
  return sign ? -v : v;
}

/* bfloat16 bits (the upper half of an IEEE binary32) -> double (exact). */
static double oracle_bf16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int m = h & 0x7F;
  double v;
  if (e == 0) v = ldexp((double)m, -133);
  else if (e == 255) v = (m == 0) ? INFINITY : NAN;
  else v = ldexp((double)(128 + m), e - 134);
  return sign ? -v : v;
}

double oracle_act_value(uint16_t bits, int act) {
  return act == ORACLE_ACT_BF16 ? oracle_bf16_value(bits) : oracle_f16_value(bits);
}

static int oracle_check_shape(int64_t N, int64_t K, int variant) {
  if (N < 0 || K < 0 || K % 32 != 0) return -1;
  if (oracle_block_bytes(variant) < 0) return -1;
  return 0;
}

/* Dense weights: out[n*K + k] = w[n][k] (row-major, fp64). */
int oracle_dequant(const uint8_t *W, int64_t N, int64_t K, int variant, double *out) {
  if (oracle_check_shape(N, K, variant)) return -1;
  const int64_t bb = oracle_block_bytes(variant);
  const int64_t nb = K / 32;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t b = 0; b < nb; ++b)
      oracle_decode_block(W + (n * nb + b) * bb, variant, out + n * K + b * 32);
  return 0;
}

/* First block (row-major block index n*nb + b) holding a scale byte that is
 * not finite, or -1 when every scale byte is finite. */
int64_t oracle_validate(const uint8_t *W, int64_t N, int64_t K, int variant) {
  if (oracle_check_shape(N, K, variant)) return -2;
  const int64_t bb = oracle_block_bytes(variant);
  const int64_t nblk = N * (K / 32);
  const int nscale = (variant == ORACLE_DUAL) ? 2 : 1;
  for (int64_t i = 0; i < nblk; ++i)
    for (int j = 0; j < nscale; ++j)
      if (!oracle_scale_is_valid(W[i * bb + 16 + j])) return i;
  return -1;
}

/* Y[m][n] = sum_k w[n][k] * x[m][k], summed in fp64 in increasing k.
 * X holds M rows of K activation bit patterns (fp16 or bf16); Y is M x N.
 * Rows n are split over nthreads POSIX threads; each output is summed by one
 * thread in plain order, so the result does not depend on nthreads. */
typedef struct {
  const uint8_t *W;
  const uint16_t *X;
  double *Y;
  int64_t M, N, K, n0, n1;
  int variant, act;
  int status;
} oracle_gemm_job;

static void *oracle_gemm_worker(void *arg) {
  oracle_gemm_job *j = (oracle_gemm_job *)arg;
  const int64_t K = j->K;
  double *w = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  double *x = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  if (!w || !x) { j->status = -3; free(w); free(x); return NULL; }
  for (int64_t n = j->n0; n < j->n1; ++n) {
    oracle_dequant(j->W + n * (K / 32) * oracle_block_bytes(j->variant), 1, K, j->variant, w);
    for (int64_t m = 0; m < j->M; ++m) {
      const uint16_t *xr = j->X + m * K;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        x[k] = oracle_act_value(xr[k], j->act);
        acc += w[k] * x[k];
      }
      j->Y[m * j->N + n] = acc;
    }
  }
  free(w);
  free(x);
  j->status = 0;
  return NULL;
}

int oracle_gemm(const uint8_t *W, const uint16_t *X, int act, double *Y, int64_t M,
                int64_t N, int64_t K, int variant, int nthreads) {
  if (oracle_check_shape(N, K, variant) || M < 0) return -1;
  if (act != ORACLE_ACT_F16 && act != ORACLE_ACT_BF16) return -1;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > N) nthreads = (int)(N > 0 ? N : 1);
  oracle_gemm_job *jobs = (oracle_gemm_job *)calloc((size_t)nthreads, sizeof(*jobs));
  pthread_t *tid = (pthread_t *)calloc((size_t)nthreads, sizeof(*tid));
  if (!jobs || !tid) { free(jobs); free(tid); return -3; }
  for (int t = 0; t < nthreads; ++t) {
    oracle_gemm_job *j = &jobs[t];
    j->W = W; j->X = X; j->Y = Y; j->M = M; j->N = N; j->K = K;
    j->variant = variant; j->act = act; j->status = -4;
    j->n0 = N * t / nthreads;
    j->n1 = N * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&tid[t], NULL, oracle_gemm_worker, &jobs[t]) != 0) break;
    started = t;
  }
  oracle_gemm_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) oracle_gemm_worker(&jobs[t]); /* not started */
  int status = 0;
  for (int t = 0; t < nthreads; ++t) if (jobs[t].status != 0) status = jobs[t].status;
  free(jobs);
  free(tid);
  return status;
}

/* Fused gate/up product, the "gemv_gate_up" decode kernel type named in the
 * "Kernel System" section of the same report.  The report gives no formula;
 * the reading taken (R11) is the gated MLP of a decoder layer:
 *   W holds 2I rows, the I gate rows then the I up rows;
 *   g = (gate rows) . x,  u = (up rows) . x,  y[i] = SiLU(g[i]) * u[i],
 *   SiLU(g) = g / (1 + exp(-g)),
 * all in fp64.  The two products are oracle_gemm's, in full. */
static double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

int oracle_gemv_gate_up(const uint8_t *W, const uint16_t *X, int act, double *Y, int64_t M,
                        int64_t I, int64_t K, int variant, int nthreads) {
  if (oracle_check_shape(I, K, variant) || M < 0) return -1;
  double *gu = (double *)malloc(sizeof(double) * (size_t)(M * 2 * I > 0 ? M * 2 * I : 1));
  if (!gu) return -3;
  int status = oracle_gemm(W, X, act, gu, M, 2 * I, K, variant, nthreads);
  if (status == 0) {
    for (int64_t m = 0; m < M; ++m) {
      for (int64_t i = 0; i < I; ++i) {
        const double g = gu[m * 2 * I + i];
        const double u = gu[m * 2 * I + I + i];
        Y[m * I + i] = oracle_silu(g) * u;
      }
    }
  }
  free(gu);
  return status;
}

/* Decode attention over a ROCmFP4 K/V cache: the "ROCmFP4 K/V dequant inside
 * attention / FlashAttention" item of the report ("Why AMD is Different from
 * NVIDIA" lists FlashAttention among the kernels a ROCmFP4 port needs, and
 * Option 2 names the "FlashAttention K/V cache optimization").  The report
 * gives no formula; the reading taken (R12) is single-token decode attention:
 *   q      [B][H][D] activations (fp16 or bf16 bits);
 *   Kc, Vc [B][Hkv][Tmax] rows, each row D/32 blocks (D a multiple of 32);
 *   lens   [B] tokens held by sequence b (clamped to [0, Tmax]);
 *   head h reads KV head h / (H / Hkv);
 *   s_t = scale * sum_d q[b][h][d] K[b][hk][t][d],   t < lens[b];
 *   out[b][h][d] = sum_t exp(s_t - max s) V[b][hk][t][d] / sum_t exp(s_t - max s);
 *   a sequence with no tokens gives zeros.  Everything in fp64. */
int oracle_decode_attention(const uint16_t *q, int act, const uint8_t *Kc, const uint8_t *Vc,
                            const int32_t *lens, double *out, int64_t B, int64_t H, int64_t Hkv,
                            int64_t D, int64_t Tmax, double scale, int variant) {
  if (oracle_check_shape(1, D, variant) || B < 0 || H < 1 || Hkv < 1 || H % Hkv != 0 || Tmax < 0)
    return -1;
  if (act != ORACLE_ACT_F16 && act != ORACLE_ACT_BF16) return -1;
  const int64_t G = H / Hkv;
  const int64_t rb = D / 32 * oracle_block_bytes(variant);
  double *k = (double *)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
  double *v = (double *)malloc(sizeof(double) * (size_t)(D > 0 ? D : 1));
  double *s = (double *)malloc(sizeof(double) * (size_t)(Tmax > 0 ? Tmax : 1));
  if (!k || !v || !s) { free(k); free(v); free(s); return -3; }
  for (int64_t b = 0; b < B; ++b) {
    int64_t T = lens[b];
    if (T < 0) T = 0;
    if (T > Tmax) T = Tmax;
    for (int64_t h = 0; h < H; ++h) {
      const int64_t hk = h / G;
      const uint16_t *qr = q + (b * H + h) * D;
      double *o = out + (b * H + h) * D;
      for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
      if (T == 0) continue;
      double smax = -INFINITY;
      for (int64_t t = 0; t < T; ++t) {
        oracle_dequant(Kc + ((b * Hkv + hk) * Tmax + t) * rb, 1, D, variant, k);
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d) acc += oracle_act_value(qr[d], act) * k[d];
        s[t] = scale * acc;
        if (s[t] > smax) smax = s[t];
      }
      double denom = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        const double p = exp(s[t] - smax);
        denom += p;
        oracle_dequant(Vc + ((b * Hkv + hk) * Tmax + t) * rb, 1, D, variant, v);
        for (int64_t d = 0; d < D; ++d) o[d] += p * v[d];
      }
      for (int64_t d = 0; d < D; ++d) o[d] /= denom;
    }
  }
  free(k);
  free(v);
  free(s);
  return 0;
}

/* Quantiser fp16 / bf16 -> ROCmFP4 blocks, the inverse of the decode.  The
 * report defines the format ("What is ROCmFP4?") but no scale selection or
 * rounding rule; the reading taken (R13):
 *   - scale groups: the two 16-weight halves of a dual block, or the whole
 *     32 weights of a single-scale block;
 *   - a group's scale byte is the smallest e in 0x00 .. 0x7E whose half-scale
 *     covers the group's largest magnitude: 5 * E4M3(e) >= amax (Codebook10's
 *     largest magnitude is 10); none covers it -> 0x7E, codes saturate at 10;
 *     a group of zeros -> e = 0;
 *   - each weight takes the nearest Codebook10 magnitude m * hs, found by
 *     comparing |x| with the midpoints ((m_k + m_k+1) / 2) * hs; a tie goes to
 *     the smaller magnitude; a negative value sets the sign bit (code 8 + k);
 *     zero (and -0) is code 0;
 *   - non-finite inputs count as 0.
 * Every product and comparison here is exact (midpoint * hs has at most 9
 * significant bits), so fp32 and fp64 take the same decisions. */
static const double oracle_cb_mid[7] = {0.5, 1.5, 2.5, 3.5, 5.0, 7.0, 9.0};

static unsigned oracle_quant_scale(double amax) {
  if (!(amax > 0.0)) return 0u;
  for (unsigned e = 0; e <= 0x7Eu; ++e)
    if (5.0 * oracle_ue4m3_value(e) >= amax) return e;
  return 0x7Eu;
}

static unsigned oracle_quant_code(double x, double hs) {
  const double a = fabs(x);
  unsigned k = 0;
  while (k < 7 && a > oracle_cb_mid[k] * hs) ++k;
  if (k == 0) return 0u;
  return x < 0.0 ? 8u + k : k;
}

int oracle_quantize(const uint16_t *src, int act, uint8_t *W, int64_t N, int64_t K, int variant) {
  if (oracle_check_shape(N, K, variant)) return -1;
  if (act != ORACLE_ACT_F16 && act != ORACLE_ACT_BF16) return -1;
  const int bb = oracle_block_bytes(variant);
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t b = 0; b < K / 32; ++b) {
      double x[32];
      for (int i = 0; i < 32; ++i) {
        const double v = oracle_act_value(src[n * K + 32 * b + i], act);
        x[i] = isfinite(v) ? v : 0.0;
      }
      uint8_t *blk = W + (n * (K / 32) + b) * bb;
      unsigned code[32];
      const int groups = variant == ORACLE_DUAL ? 2 : 1, gsize = 32 / groups;
      for (int g = 0; g < groups; ++g) {
        double amax = 0.0;
        for (int i = g * gsize; i < (g + 1) * gsize; ++i) amax = fabs(x[i]) > amax ? fabs(x[i]) : amax;
        const unsigned e = oracle_quant_scale(amax);
        blk[16 + g] = (uint8_t)e;
        const double hs = oracle_halfscale(e);
        for (int i = g * gsize; i < (g + 1) * gsize; ++i) code[i] = hs > 0.0 ? oracle_quant_code(x[i], hs) : 0u;
      }
      for (int j = 0; j < 16; ++j) blk[j] = (uint8_t)(code[j] | (code[j + 16] << 4)); /* R1 */
    }
  }
  return 0;
}
