/*
 * oracle.c -- plain, slow CPU reference of the sub-bit weight products.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code,
 * header, table or constant with the CUDA path: it restates the format and
 * the products from their definitions, in FP64, one output at a time.
 *
 * What it computes (the plain definition of the method):
 *   y[m][n] = sum_k x[m][k] * s[n][floor(k/128)] * w[n][k],   w in {-1,0,+1}
 * -- one FP16 scale shared by each group of 128 weights along K
 *    ("1-bit diffusion ... WebGPU" page, section "1-bit 嘅數學"; OpenBonsai
 *    page, section "工作原理": FP16 group scale, one per 128 weights),
 * -- binary weights take values +1/-1 ("1-bit 嘅數學"), ternary ones
 *    -1/0/+1 (same section; "三值权重到底做了什么").
 * XNOR product ("1-bit 嘅數學": binary GEMM by XOR + popcount):
 *   D[m][n] = sum_k a[m][k] * w[n][k]   computed here from the unpacked +-1
 *   integers (not from popcount), so the popcount identity used on the GPU
 *   is checked rather than assumed;
 *   Y[m][n] = a_s[m] * sum_g s[n][g] * d_g,  d_g = sum_{k in g} a*w.
 * Activation binarisation (this library's reading; the pages give no rule):
 *   a = sign(x) with sign(0) = +1, a_s = mean |x| over the row.
 *
 * Byte layout (this library's reading; the pages give none):
 *   binary : bit (k % 32) of little-endian uint32 word k/32, bit 1 = +1.
 *   ternary: byte b = sum_{i<5} (w[5b+i] + 1) * 3^i; codes past k are 0;
 *            row padded to row_bytes with bytes 121 (five zero codes).
 *
 * Every product x*s*w is exact in double (11-bit x 11-bit significands);
 * the double sum adds at most k * 2^-53 relative to sum |x*s*w|.
 *
 * Parity status: the pages print no worked example of a packed byte or of a
 * product. Bit order, bit polarity and trit digit order are this library's
 * convention ("parity unpinned" by the pages); they are pinned by round trips,
 * single-hot codes and closed forms in the tests, not by page values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define O_OK 0
#define O_ERR_ARG 1
#define O_ERR_SHAPE 2
#define O_ERR_BAD_CODE 8

#define FMT_BINARY 1
#define FMT_TERNARY 2
#define GROUP 128

/* IEEE-754 binary16 -> double, exact: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 = subnormal f * 2^-24; exponent 31 = inf/NaN. */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double mag;
  if (e == 0)
    mag = ldexp((double)f, -24);
  else if (e == 31)
    mag = f ? NAN : INFINITY;
  else
    mag = ldexp((double)(1024 + f), e - 25);
  return sign ? -mag : mag;
}

int64_t oracle_row_bytes(int fmt, int64_t k) {
  if (k <= 0 || k % GROUP) return -1;
  if (fmt == FMT_BINARY) return k / 8;
  if (fmt == FMT_TERNARY) {
    int64_t data = (k + 4) / 5;
    return 64 * ((data + 63) / 64);
  }
  return -1;
}

/* ---------------- binary ---------------- */

int oracle_pack_binary(const int8_t* codes, int64_t rows, int64_t k,
                       uint8_t* out, int64_t row_bytes) {
  if (!codes || !out || rows < 0 || k <= 0) return O_ERR_ARG;
  if (k % 32 || row_bytes < k / 8) return O_ERR_SHAPE;
  for (int64_t r = 0; r < rows; ++r) {
    uint8_t* row = out + r * row_bytes;
    memset(row, 0, (size_t)row_bytes);
    for (int64_t j = 0; j < k / 32; ++j) {
      uint32_t word = 0;
      for (int i = 0; i < 32; ++i) {
        int8_t c = codes[r * k + 32 * j + i];
        if (c == 1)
          word |= (uint32_t)1 << i;
        else if (c != -1)
          return O_ERR_BAD_CODE;
      }
      for (int b = 0; b < 4; ++b) row[4 * j + b] = (uint8_t)(word >> (8 * b));
    }
  }
  return O_OK;
}

int oracle_unpack_binary(const uint8_t* packed, int64_t rows, int64_t k,
                         int64_t row_bytes, int8_t* codes) {
  if (!packed || !codes || rows < 0 || k <= 0) return O_ERR_ARG;
  if (k % 32 || row_bytes < k / 8) return O_ERR_SHAPE;
  for (int64_t r = 0; r < rows; ++r) {
    const uint8_t* row = packed + r * row_bytes;
    for (int64_t j = 0; j < k / 32; ++j) {
      uint32_t word = 0;
      for (int b = 0; b < 4; ++b) word |= (uint32_t)row[4 * j + b] << (8 * b);
      for (int i = 0; i < 32; ++i)
        codes[r * k + 32 * j + i] = ((word >> i) & 1u) ? 1 : -1;
    }
  }
  return O_OK;
}

/* ---------------- ternary ---------------- */

int oracle_pack_ternary(const int8_t* codes, int64_t rows, int64_t k,
                        uint8_t* out, int64_t row_bytes) {
  if (!codes || !out || rows < 0 || k <= 0) return O_ERR_ARG;
  if (row_bytes < (k + 4) / 5) return O_ERR_SHAPE;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < row_bytes; ++b) {
      int value = 0;
      for (int i = 4; i >= 0; --i) { /* Horner: most significant digit first */
        int64_t kk = 5 * b + i;
        int c = 0;
        if (kk < k) {
          c = codes[r * k + kk];
          if (c < -1 || c > 1) return O_ERR_BAD_CODE;
        }
        value = 3 * value + (c + 1);
      }
      out[r * row_bytes + b] = (uint8_t)value;
    }
  }
  return O_OK;
}

int oracle_unpack_ternary(const uint8_t* packed, int64_t rows, int64_t k,
                          int64_t row_bytes, int8_t* codes) {
  if (!packed || !codes || rows < 0 || k <= 0) return O_ERR_ARG;
  if (row_bytes < (k + 4) / 5) return O_ERR_SHAPE;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < (k + 4) / 5; ++b) {
      int value = packed[r * row_bytes + b];
      if (value > 242) return O_ERR_BAD_CODE;
      for (int i = 0; i < 5; ++i) {
        int digit = value % 3;
        value /= 3;
        int64_t kk = 5 * b + i;
        if (kk < k) codes[r * k + kk] = (int8_t)(digit - 1);
      }
    }
  }
  return O_OK;
}

static int unpack_row(int fmt, const uint8_t* packed, int64_t row_bytes,
                      int64_t row, int64_t k, int8_t* codes) {
  const uint8_t* p = packed + row * row_bytes;
  if (fmt == FMT_BINARY) return oracle_unpack_binary(p, 1, k, row_bytes, codes);
  if (fmt == FMT_TERNARY) return oracle_unpack_ternary(p, 1, k, row_bytes, codes);
  return O_ERR_ARG;
}

/* ---------------- products ---------------- */

/* y and norm are [m_cnt][n_cnt]:
 *   y[i][j]    = sum_k x[m_sel[i]][k] * s[n_sel[j]][k/128] * w[n_sel[j]][k]
 *   norm[i][j] = sum_k |x * s * w|                                        */
int oracle_linear(int fmt, const uint8_t* packed, int64_t row_bytes,
                  const uint16_t* scales, int64_t n, int64_t k,
                  const uint16_t* x, int64_t m,
                  const int64_t* n_sel, int64_t n_cnt,
                  const int64_t* m_sel, int64_t m_cnt,
                  double* y, double* norm) {
  if (!packed || !scales || !x || !n_sel || !m_sel || !y || !norm) return O_ERR_ARG;
  if (k <= 0 || k % GROUP) return O_ERR_SHAPE;
  int8_t* w = (int8_t*)malloc((size_t)k);
  if (!w) return O_ERR_ARG;
  const int64_t groups = k / GROUP;
  for (int64_t j = 0; j < n_cnt; ++j) {
    int64_t nn = n_sel[j];
    if (nn < 0 || nn >= n) { free(w); return O_ERR_ARG; }
    int st = unpack_row(fmt, packed, row_bytes, nn, k, w);
    if (st != O_OK) { free(w); return st; }
    for (int64_t i = 0; i < m_cnt; ++i) {
      int64_t mm = m_sel[i];
      if (mm < 0 || mm >= m) { free(w); return O_ERR_ARG; }
      double acc = 0.0, nrm = 0.0;
      for (int64_t kk = 0; kk < k; ++kk) {
        double xv = oracle_half_to_double(x[mm * k + kk]);
        double sv = oracle_half_to_double(scales[nn * groups + kk / GROUP]);
        double t = xv * sv * (double)w[kk];
        acc += t;
        nrm += fabs(t);
      }
      y[i * n_cnt + j] = acc;
      norm[i * n_cnt + j] = nrm;
    }
  }
  free(w);
  return O_OK;
}

/* Gated feed-forward input of a decode layer: the gate and up projections
 * of the same x, stored as ONE weight matrix of n = 2F rows whose 16-row
 * blocks hold 8 gate rows then the 8 up rows of the same features:
 *   gate row f -> stored row 16*(f/8) + f%8,  up row f -> that row + 8.
 * The pages run Qwen-family models (OpenBonsai page: Qwen3.5-9B) but do not
 * write the feed-forward block out; this library takes the SwiGLU form of
 * that family:
 *   g = x . (s (.) W_gate)^T,  u = x . (s (.) W_up)^T,
 *   h[m][f] = silu(g) * u,     silu(g) = g / (1 + exp(-g)).
 * h, g, u, norm_g, norm_u are [m_cnt][f_cnt]; norm_* are sum |x*s*w| of the
 * gate and up rows (the error scale of g and u). */
int oracle_swiglu(int fmt, const uint8_t* packed, int64_t row_bytes,
                  const uint16_t* scales, int64_t n, int64_t k,
                  const uint16_t* x, int64_t m,
                  const int64_t* f_sel, int64_t f_cnt,
                  const int64_t* m_sel, int64_t m_cnt,
                  double* h, double* g, double* u, double* norm_g, double* norm_u) {
  if (!f_sel || !h || !g || !u || !norm_g || !norm_u) return O_ERR_ARG;
  if (n <= 0 || n % 16) return O_ERR_SHAPE;
  const int64_t F = n / 2;
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(2 * f_cnt + 1));
  double* y = (double*)malloc(sizeof(double) * (size_t)(2 * f_cnt * m_cnt + 1));
  double* nr = (double*)malloc(sizeof(double) * (size_t)(2 * f_cnt * m_cnt + 1));
  if (!rows || !y || !nr) { free(rows); free(y); free(nr); return O_ERR_ARG; }
  int st = O_OK;
  for (int64_t j = 0; j < f_cnt; ++j) {
    const int64_t f = f_sel[j];
    if (f < 0 || f >= F) { st = O_ERR_ARG; break; }
    rows[j] = 16 * (f / 8) + f % 8;      /* gate */
    rows[f_cnt + j] = rows[j] + 8;       /* up   */
  }
  if (st == O_OK)
    st = oracle_linear(fmt, packed, row_bytes, scales, n, k, x, m, rows, 2 * f_cnt, m_sel,
                       m_cnt, y, nr);
  if (st == O_OK) {
    for (int64_t i = 0; i < m_cnt; ++i)
      for (int64_t j = 0; j < f_cnt; ++j) {
        const double gv = y[i * 2 * f_cnt + j], uv = y[i * 2 * f_cnt + f_cnt + j];
        const int64_t o = i * f_cnt + j;
        g[o] = gv;
        u[o] = uv;
        norm_g[o] = nr[i * 2 * f_cnt + j];
        norm_u[o] = nr[i * 2 * f_cnt + f_cnt + j];
        h[o] = gv / (1.0 + exp(-gv)) * uv;
      }
  }
  free(rows);
  free(y);
  free(nr);
  return st;
}

/* d, y, norm are [m_cnt][n_cnt]. a_bits rows are BINARY-packed, k/8 bytes. */
int oracle_xnor(const uint8_t* a_bits, const uint16_t* a_scale, int64_t m,
                const uint8_t* w_packed, int64_t row_bytes,
                const uint16_t* scales, int64_t n, int64_t k,
                const int64_t* n_sel, int64_t n_cnt,
                const int64_t* m_sel, int64_t m_cnt,
                int64_t* d, double* y, double* norm) {
  if (!a_bits || !a_scale || !w_packed || !scales || !n_sel || !m_sel || !d ||
      !y || !norm)
    return O_ERR_ARG;
  if (k <= 0 || k % GROUP) return O_ERR_SHAPE;
  int8_t* a = (int8_t*)malloc((size_t)k);
  int8_t* w = (int8_t*)malloc((size_t)k);
  if (!a || !w) { free(a); free(w); return O_ERR_ARG; }
  const int64_t groups = k / GROUP;
  int st = O_OK;
  for (int64_t i = 0; i < m_cnt && st == O_OK; ++i) {
    int64_t mm = m_sel[i];
    if (mm < 0 || mm >= m) { st = O_ERR_ARG; break; }
    st = oracle_unpack_binary(a_bits + mm * (k / 8), 1, k, k / 8, a);
    double as = oracle_half_to_double(a_scale[mm]);
    for (int64_t j = 0; j < n_cnt && st == O_OK; ++j) {
      int64_t nn = n_sel[j];
      if (nn < 0 || nn >= n) { st = O_ERR_ARG; break; }
      st = oracle_unpack_binary(w_packed + nn * row_bytes, 1, k, row_bytes, w);
      if (st != O_OK) break;
      int64_t total = 0;
      double acc = 0.0, sabs = 0.0;
      for (int64_t g = 0; g < groups; ++g) {
        int64_t dg = 0;
        for (int64_t kk = g * GROUP; kk < (g + 1) * GROUP; ++kk)
          dg += (int64_t)a[kk] * (int64_t)w[kk];
        double sg = oracle_half_to_double(scales[nn * groups + g]);
        total += dg;
        acc += sg * (double)dg;
        sabs += fabs(sg);
      }
      d[i * n_cnt + j] = total;
      y[i * n_cnt + j] = as * acc;
      norm[i * n_cnt + j] = fabs(as) * (double)GROUP * sabs;
    }
  }
  free(a);
  free(w);
  return st;
}

/* Activation binarisation, the A side of the XNOR product ("1-bit 嘅數學":
 * XOR + popcount needs both operands as +-1 bits). The pages say neither how
 * an FP16 activation row becomes +-1 codes nor which scale goes with it; this
 * library's reading:
 *   a[m][k]  = +1 if x[m][k] >= 0 (so +0 and -0 give +1), else -1;
 *              a NaN compares false and gives -1,
 *   a_s[m]   = (1/K) * sum_k |x[m][k]|,
 * the scale alpha that minimises sum_k (x[m][k] - alpha * a[m][k])^2 for these
 * codes (setting the derivative to zero: alpha * K = sum_k a*x = sum_k |x|).
 * bits is [m][k/8] bytes in the binary weight layout; a_scale is [m], exact
 * up to one rounding of the double sum. */
int oracle_binarize(const uint16_t* x, int64_t m, int64_t k, uint8_t* bits,
                    double* a_scale) {
  if (!x || !bits || !a_scale || m < 0 || k <= 0) return O_ERR_ARG;
  if (k % 32) return O_ERR_SHAPE;
  int8_t* a = (int8_t*)malloc((size_t)k);
  if (!a) return O_ERR_ARG;
  int st = O_OK;
  for (int64_t r = 0; r < m && st == O_OK; ++r) {
    double sum = 0.0;
    for (int64_t kk = 0; kk < k; ++kk) {
      const double v = oracle_half_to_double(x[r * k + kk]);
      a[kk] = (v >= 0.0) ? 1 : -1;
      sum += fabs(v);
    }
    a_scale[r] = sum / (double)k;
    st = oracle_pack_binary(a, 1, k, bits + r * (k / 8), k / 8);
  }
  free(a);
  return st;
}

/* Signed Hadamard rotation of activation rows. The OpenBonsai page
 * ("工作原理") lists a signed Hadamard rotation among its compression steps
 * (to tame weight outliers) but states neither its size nor where the
 * activation side is rotated. This library's reading: a block-diagonal
 * rotation along K with power-of-two blocks b (b | k), one +-1 sign per
 * input feature, orthonormal scaling:
 *   out[r][b0 + i] = b^(-1/2) * sum_{j<b} H[i][j] * s[b0 + j] * x[r][b0 + j],
 *   H[i][j] = (-1)^popcount(i & j)      (Sylvester's construction),
 * for each block start b0 = 0, b, 2b, ... The signs are bits in the binary
 * weight layout (bit (k%32) of word k/32, bit 1 = +1); NULL means all +1.
 * Written straight from the definition: O(b) work per output. */
int oracle_hadamard(const uint16_t* x, int64_t m, int64_t k, int64_t block,
                    const uint8_t* sign_bits, double* out) {
  if (!x || !out || m < 0 || k <= 0 || block <= 0) return O_ERR_ARG;
  if (block & (block - 1)) return O_ERR_SHAPE;
  if (k % block) return O_ERR_SHAPE;
  const double scale = 1.0 / sqrt((double)block);
  for (int64_t r = 0; r < m; ++r) {
    for (int64_t b0 = 0; b0 < k; b0 += block) {
      for (int64_t i = 0; i < block; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < block; ++j) {
          const int64_t kk = b0 + j;
          double v = oracle_half_to_double(x[r * k + kk]);
          if (sign_bits && !((sign_bits[kk >> 3] >> (kk & 7)) & 1)) v = -v;
          acc += (__builtin_popcountll((unsigned long long)(i & j)) & 1) ? -v : v;
        }
        out[r * k + b0 + i] = acc * scale;
      }
    }
  }
  return O_OK;
}

/* Acceptance: |y_gpu - y_ref| <= tol * norm; norm == 0 requires y_gpu = +-0;
 * a non-finite y_gpu always fails. Returns the number of failures; writes
 * the first failing index (or -1) and the largest |err|/norm seen. */
int64_t oracle_compare_f16(const uint16_t* y_gpu, const double* y_ref,
                           const double* norm, int64_t count, double tol,
                           int64_t* first_bad, double* worst) {
  int64_t bad = 0;
  double w = 0.0;
  if (first_bad) *first_bad = -1;
  for (int64_t i = 0; i < count; ++i) {
    double g = oracle_half_to_double(y_gpu[i]);
    int fail;
    if (!isfinite(g)) {
      fail = 1;
    } else if (norm[i] == 0.0) {
      fail = (g != 0.0);
    } else {
      double r = fabs(g - y_ref[i]) / norm[i];
      if (r > w) w = r;
      fail = r > tol;
    }
    if (fail) {
      if (bad == 0 && first_bad) *first_bad = i;
      ++bad;
    }
  }
  if (worst) *worst = w;
  return bad;
}
