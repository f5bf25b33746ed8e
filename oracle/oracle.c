/*
 * MatMulNBits oracle: a plain, slow, double-precision CPU statement of the
 * weight-only INT4 blockwise-quantized MatMul.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; only the tests, the package smoke check and the CPU-baseline
 * leg of the benchmark use it. It shares no code, header, table or helper with
 * the CUDA library and includes nothing from it.
 *
 * What it computes (page "Qwen3 CPU Inference Critical Path", section "Exact
 * kernel inventory", row com.microsoft::MatMulNBits v1; section "Prepared
 * weight-only plan", paragraph on zero-point correction, scales and float32
 * accumulation):
 *
 *   Y[m,n] = sum_{k=0}^{K-1} A[m,k] * (q[n,k] - z[n,k/bs]) * s[n,k/bs] + bias[n]
 *
 * with the storage conventions below. Readings where the page is silent
 * (zero-point default 8, zero-point nibble packing, bias fp32, bf16 handling)
 * are the ones listed in the design notes; each is marked "reading" here.
 *
 *   B      uint8 [N, nb, bs/2], nb = ceil(K/bs). Element k of row n lives in
 *          byte (k mod bs)/2 of block k/bs; the low nibble holds the even
 *          element, the high nibble the odd one ("packed UINT8 storage
 *          containing 4-bit weights", low nibble first).  Nibbles past K in
 *          the last block are storage padding and never read.
 *   scales [N, nb], fp32 or bf16 (raw 16-bit patterns), widened exactly.
 *   zp     uint8 [N, ceil(nb/2)] or NULL. Reading: two blocks per byte, the
 *          even block in the low nibble; NULL means every zero point is 8.
 *   bias   fp32 [N] or NULL (reading: always fp32).
 *   A      [M, K] row-major, fp32 or bf16, widened exactly to double.
 *
 * Every product and sum is taken in double, in increasing k, with no
 * blocking or reordering. absdot[m,n] = sum_k |A[m,k] * w[n,k]| is returned
 * alongside Y because the acceptance bound is stated in terms of it.
 *
 * Parity status: pinned by the CPU tests (integer-exact brute force with an
 * independently written packer, a hand-worked fixture, invariants and a dense
 * float64 library GEMM).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2 /* activations only: an exact double input (e.g. a normalized row) */

/* Exact widening of one stored element to double. A bf16 value is the upper
 * half of the fp32 with the same bit pattern, so shifting the 16 stored bits
 * into the top of a 32-bit word reproduces it exactly. */
static double widen(const void *base, int64_t i, int dtype) {
  if (dtype == ORACLE_F32) {
    return (double)((const float *)base)[i];
  }
  if (dtype == ORACLE_F64) {
    return ((const double *)base)[i];
  }
  uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

static int64_t n_blocks(int64_t K, int bs) { return (K + bs - 1) / bs; }

/* The 4-bit code q[n,k]: byte (k mod bs)/2 of block k/bs of row n, low nibble
 * for even k. */
static int code_at(const uint8_t *B, int64_t n, int64_t k, int64_t nb, int bs) {
  int64_t b = k / bs;
  int64_t within = k % bs;
  uint8_t byte = B[(n * nb + b) * (bs / 2) + within / 2];
  return (within % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* The zero point z[n,b]. Reading: NULL means 8; otherwise byte b/2 of row n,
 * low nibble for even b. */
static int zero_point_at(const uint8_t *zp, int64_t n, int64_t b, int64_t nb) {
  if (zp == NULL) return 8;
  int64_t zbytes = (nb + 1) / 2;
  uint8_t byte = zp[n * zbytes + b / 2];
  return (b % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* Dequantized weight w[n,k] = (q - z) * s, in double. */
static double weight_at(const uint8_t *B, const void *scales, int scale_dtype,
                        const uint8_t *zp, int64_t n, int64_t k, int64_t nb,
                        int bs) {
  int64_t b = k / bs;
  int q = code_at(B, n, k, nb, bs);
  int z = zero_point_at(zp, n, b, nb);
  double s = widen(scales, n * nb + b, scale_dtype);
  return (double)(q - z) * s;
}

static int check_args(int64_t M, int64_t N, int64_t K, int bs, int a_dtype,
                      int scale_dtype) {
  if (M < 0 || N < 0 || K < 0) return -2;
  if (bs < 2 || (bs % 2) != 0) return -3;
  if ((a_dtype != ORACLE_F32 && a_dtype != ORACLE_BF16 && a_dtype != ORACLE_F64) ||
      (scale_dtype != ORACLE_F32 && scale_dtype != ORACLE_BF16))
    return -4;
  return 0;
}

/* W[n,k] for all n < N, k < K (row-major [N, K], double). */
int oracle_dequantize(const uint8_t *B, const void *scales, int scale_dtype,
                      const uint8_t *zp, int64_t N, int64_t K, int bs,
                      double *W) {
  int rc = check_args(0, N, K, bs, ORACLE_F32, scale_dtype);
  if (rc) return rc;
  int64_t nb = n_blocks(K, bs);
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      W[n * K + k] = weight_at(B, scales, scale_dtype, zp, n, k, nb, bs);
  return 0;
}

/* Y[i,j] for m = rows[i], n = cols[j]; rows/cols NULL means every row/column
 * in order. Y and absdot (may be NULL) are [n_rows, n_cols] row-major. */
int oracle_matmulnbits(const void *A, int a_dtype, const uint8_t *B,
                       const void *scales, int scale_dtype, const uint8_t *zp,
                       const float *bias, int64_t M, int64_t N, int64_t K,
                       int bs, const int64_t *rows, int64_t n_rows,
                       const int64_t *cols, int64_t n_cols, double *Y,
                       double *absdot) {
  int rc = check_args(M, N, K, bs, a_dtype, scale_dtype);
  if (rc) return rc;
  if (rows == NULL) n_rows = M;
  if (cols == NULL) n_cols = N;
  int64_t nb = n_blocks(K, bs);
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) return -2;
    for (int64_t j = 0; j < n_cols; ++j) {
      int64_t n = cols ? cols[j] : j;
      if (n < 0 || n >= N) return -2;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double a = widen(A, m * K + k, a_dtype);
        double w = weight_at(B, scales, scale_dtype, zp, n, k, nb, bs);
        acc += a * w;
        mag += fabs(a * w);
      }
      if (bias) acc += (double)bias[n];
      Y[i * n_cols + j] = acc;
      if (absdot) absdot[i * n_cols + j] = mag;
    }
  }
  return 0;
}

/*
 * The standard QDQ INT4 encoding (page "Qwen3 CPU Inference Critical Path",
 * section "qwen3-int4-qdq"): a logical UINT4 matrix stored ONNX row-major,
 * low nibble first (element i of the flattened matrix is nibble i of the
 * byte stream), DequantizeLinear with a block size along one axis, then
 * MatMul:
 *
 *   axis 0 (projections): the matrix is [K, N];  w[n,k] = (q[k,n] - z[k/bs,n]) * s[k/bs,n]
 *   axis 1 (tied LM head): the matrix is [N, K]; w[n,k] = (q[n,k] - z[n,k/bs]) * s[n,k/bs]
 *
 *   Y[m,n] = sum_k A[m,k] * w[n,k] + bias[n]
 *
 * Scales and zero points have the block-reduced shape ([ceil(K/bs), N] or
 * [N, ceil(K/bs)]); zero points are UINT4 stored like the codes, and absent
 * zero points are 0 (the DequantizeLinear default). Everything in double, in
 * increasing k.
 */
static int qdq_nibble(const uint8_t *p, int64_t i) {
  uint8_t byte = p[i / 2];
  return (i % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

static double qdq_weight_at(const uint8_t *Bq, const void *scales, int scale_dtype,
                            const uint8_t *zp, int axis, int64_t n, int64_t k,
                            int64_t N, int64_t K, int64_t nb, int bs) {
  int64_t b = k / bs;
  int64_t ci = axis == 0 ? k * N + n : n * K + k;   /* code element */
  int64_t si = axis == 0 ? b * N + n : n * nb + b;  /* scale / zero-point element */
  int q = qdq_nibble(Bq, ci);
  int z = zp ? qdq_nibble(zp, si) : 0;
  return (double)(q - z) * widen(scales, si, scale_dtype);
}

int oracle_qdq_matmul(const void *A, int a_dtype, const uint8_t *Bq,
                      const void *scales, int scale_dtype, const uint8_t *zp,
                      const float *bias, int axis, int64_t M, int64_t N,
                      int64_t K, int bs, const int64_t *rows, int64_t n_rows,
                      const int64_t *cols, int64_t n_cols, double *Y,
                      double *absdot) {
  int rc = check_args(M, N, K, bs, a_dtype, scale_dtype);
  if (rc) return rc;
  if (axis != 0 && axis != 1) return -2;
  if (rows == NULL) n_rows = M;
  if (cols == NULL) n_cols = N;
  int64_t nb = n_blocks(K, bs);
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) return -2;
    for (int64_t j = 0; j < n_cols; ++j) {
      int64_t n = cols ? cols[j] : j;
      if (n < 0 || n >= N) return -2;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double a = widen(A, m * K + k, a_dtype);
        double w = qdq_weight_at(Bq, scales, scale_dtype, zp, axis, n, k, N, K, nb, bs);
        acc += a * w;
        mag += fabs(a * w);
      }
      if (bias != NULL) acc += (double)bias[n];
      Y[i * n_cols + j] = acc;
      if (absdot) absdot[i * n_cols + j] = mag;
    }
  }
  return 0;
}

/*
 * RMS-style normalization of each activation row (page "Qwen3 CPU Inference
 * Critical Path": ai.onnx::SimplifiedLayerNormalization in the exact kernel
 * inventory, FP32 RMS-style normalization over the last axis with
 * epsilon 1e-6, and RMSNormalization v23 among the P1 operators; the fusion
 * list puts it into the packed projection input):
 *
 *   r[m]      = 1 / sqrt( (sum_k A[m,k]^2) / K + eps )
 *   out[m,k]  = A[m,k] * r[m] * gamma[k]        (gamma NULL: 1)
 *
 * in double, the sum in increasing k. out is [M, K] row-major double.
 */
int oracle_rms_normalize(const void *A, int a_dtype, const float *gamma, double eps,
                         int64_t M, int64_t K, double *out) {
  if (M < 0 || K < 1 || eps < 0.0) return -2;
  if (a_dtype != ORACLE_F32 && a_dtype != ORACLE_BF16 && a_dtype != ORACLE_F64) return -4;
  for (int64_t m = 0; m < M; ++m) {
    double sumsq = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double x = widen(A, m * K + k, a_dtype);
      sumsq += x * x;
    }
    double r = 1.0 / sqrt(sumsq / (double)K + eps);
    for (int64_t k = 0; k < K; ++k) {
      double g = gamma ? (double)gamma[k] : 1.0;
      out[m * K + k] = widen(A, m * K + k, a_dtype) * r * g;
    }
  }
  return 0;
}

/*
 * bitsandbytes-style 4-bit matrix (page "Qwen3 CPU Inference Critical Path",
 * com.microsoft operator inventory, row MatMulBnb4: an alternative
 * bitsandbytes-style 4-bit matrix format, to be adapted into the same
 * weight-only plan). The pages name the format and nothing more; readings:
 *
 *   B      uint8 [(N*K + 1) / 2]: the N x K weight (row n = output n)
 *          flattened row-major; element i is in byte i/2, in the HIGH
 *          nibble for even i (the first element of a pair high);
 *   absmax [ceil(N*K / bs)], fp32 or bf16: one scale per run of bs
 *          consecutive flattened elements;
 *   code   fp32 [16]: the 16-value code book (NF4, FP4 or any other);
 *
 *   w[n,k] = code[q(n*K + k)] * absmax[(n*K + k) / bs]
 *   Y[m,n] = sum_k A[m,k] * w[n,k] + bias[n]
 *
 * in double, in increasing k.
 */
static int bnb4_nibble(const uint8_t *B, int64_t i) {
  uint8_t byte = B[i / 2];
  return (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);
}

int oracle_bnb4_matmul(const void *A, int a_dtype, const uint8_t *B, const void *absmax,
                       int absmax_dtype, const float *code, const float *bias,
                       int64_t M, int64_t N, int64_t K, int bs, const int64_t *rows,
                       int64_t n_rows, const int64_t *cols, int64_t n_cols, double *Y,
                       double *absdot) {
  int rc = check_args(M, N, K, 2, a_dtype, absmax_dtype);  /* any block size >= 1 here */
  if (rc) return rc;
  if (bs < 1 || code == NULL) return -3;
  if (rows == NULL) n_rows = M;
  if (cols == NULL) n_cols = N;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t m = rows ? rows[i] : i;
    if (m < 0 || m >= M) return -2;
    for (int64_t j = 0; j < n_cols; ++j) {
      int64_t n = cols ? cols[j] : j;
      if (n < 0 || n >= N) return -2;
      double acc = 0.0, mag = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        int64_t flat = n * K + k;
        double w = (double)code[bnb4_nibble(B, flat)] * widen(absmax, flat / bs, absmax_dtype);
        double a = widen(A, m * K + k, a_dtype);
        acc += a * w;
        mag += fabs(a * w);
      }
      acc += bias ? (double)bias[n] : 0.0;
      Y[i * n_cols + j] = acc;
      if (absdot) absdot[i * n_cols + j] = mag;
    }
  }
  return 0;
}
