/*
 * Oracle for the matrix-vector product c = B @ a  --  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  The product path (the CUDA library and its Python
 * binding) never calls it, and the two share no code: this file includes no
 * header of the CUDA path and the CUDA path includes nothing from here.
 *
 * What it computes (TileLang Case Studies, Case B "Background"): B has shape
 * (n, k) and is stored row-major, a has shape (k,), and
 *
 *     c_i = sum_{j=0}^{k-1} B[i, j] * a[j]            for i = 0 .. n-1.
 *
 * Inputs are 16-bit floats (IEEE-754 binary16 "fp16", or bfloat16, the upper
 * half of an IEEE-754 binary32).  Each element is decoded from its bit
 * pattern by the format definition (sign, biased exponent, fraction; zeros,
 * subnormals, infinities, NaN), widened to binary64, multiplied and summed in
 * ascending j, one row at a time, single-threaded.  Nothing is blocked, fused
 * or reordered.  Alongside c_i the oracle returns S_i = sum_j |B[i,j] a[j]|,
 * the scale against which the fp32-output tolerance is stated.
 *
 * Rounding of a binary64 value to an output format (fp16, bf16 or fp32) is
 * round-to-nearest, ties-to-even, written out from the definition: scale by
 * the format's quantum at that exponent, compare the remainder with one half.
 * Overflow goes to +-inf (what ties-to-even gives past the largest finite
 * value), NaN maps to the format's canonical quiet NaN.
 *
 * Compiled with -O2 -ffp-contract=off and without -ffast-math, so that every
 * product and every sum is one correctly rounded binary64 operation.
 *
 * The fused epilogue (the TileLang optimization guide, "Epilogue Fusion":
 * scaling, bias and activation applied to the result before it is stored)
 * is gemv_ref_epilogue(): y_i = act(alpha * c_i + beta * bias_i) in binary64
 * with act = identity, relu (max(y, 0), 0 for NaN), sigmoid 1/(1 + e^-y) or
 * silu y/(1 + e^-y), exp from the C library.
 *
 * gla_ref_decode() is one step of the gated-linear-attention recurrence
 * (Case D "Background"), written out the same way.
 *
 * Pins (tests/test_oracle.py): exhaustive decode of all 2^16 patterns of both
 * formats against torch's CPU casts; encode against numpy/torch casts and
 * constructed halfway and overflow cases; B = ones, a = ones gives k exactly;
 * identity-padded B gives c = a; exact rational (fractions.Fraction) sums on
 * 4x8 inputs; numpy float64 matmul within its error bound; linearity and row
 * permutation on integer-valued inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

/* dtype codes understood by this file (independent of the CUDA library's) */
#define REF_F16 0
#define REF_BF16 1
#define REF_F32 2

/* Format parameters: fraction bits and exponent bits. */
static void ref_format(int fmt, int *mbits, int *ebits) {
  if (fmt == REF_F16) {
    *mbits = 10;
    *ebits = 5;
  } else if (fmt == REF_BF16) {
    *mbits = 7;
    *ebits = 8;
  } else {
    *mbits = 23;
    *ebits = 8;
  }
}

/* Decode one binary interchange-format pattern (sign | exponent | fraction).
 * bias = 2^(ebits-1) - 1.  Exponent field 0: subnormal or zero, value
 * fraction * 2^(1 - bias - mbits).  All-ones exponent: inf (fraction 0) or NaN.
 * Otherwise (2^mbits + fraction) * 2^(e - bias - mbits). */
static double ref_decode_bits(uint32_t bits, int fmt) {
  int mbits, ebits;
  ref_format(fmt, &mbits, &ebits);
  const int bias = (1 << (ebits - 1)) - 1;
  const uint32_t emax_field = (1u << ebits) - 1u;
  const uint32_t sign = (bits >> (mbits + ebits)) & 1u;
  const uint32_t e = (bits >> mbits) & emax_field;
  const uint32_t m = bits & ((1u << mbits) - 1u);
  double v;
  if (e == 0) {
    v = ldexp((double)m, 1 - bias - mbits);
  } else if (e == emax_field) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
  }
  return sign ? -v : v;
}

/* Round a binary64 value to the nearest representable value of the format,
 * ties to even, and return its bit pattern. */
static uint32_t ref_encode_bits(double x, int fmt) {
  int mbits, ebits;
  ref_format(fmt, &mbits, &ebits);
  const int bias = (1 << (ebits - 1)) - 1;
  const uint32_t emax_field = (1u << ebits) - 1u;
  const uint32_t sign = signbit(x) ? (1u << (mbits + ebits)) : 0u;
  const uint32_t inf_bits = sign | (emax_field << mbits);
  if (isnan(x)) return (emax_field << mbits) | (1u << (mbits - 1)); /* quiet NaN */
  double ax = fabs(x);
  if (isinf(ax)) return inf_bits;
  if (ax == 0.0) return sign;
  /* Exponent of the leading bit: ax = f * 2^E with f in [1, 2). */
  int fe;
  (void)frexp(ax, &fe); /* ax = g * 2^fe, g in [0.5, 1) */
  int E = fe - 1;
  const int emin = 1 - bias; /* smallest normal exponent */
  /* Quantum (spacing of representable values) at this exponent. */
  int qexp = (E < emin) ? (emin - mbits) : (E - mbits);
  double m = ldexp(ax, -qexp); /* exact: power-of-two scaling */
  double fl = floor(m);
  double rem = m - fl; /* exact: m has at most 53 significant bits, fl < 2^(mbits+1) */
  double r;
  if (rem > 0.5) {
    r = fl + 1.0;
  } else if (rem < 0.5) {
    r = fl;
  } else {
    r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0; /* tie: to even */
  }
  /* r is the integer significand in units of the quantum. */
  uint64_t ri = (uint64_t)r;
  uint64_t out;
  if (E < emin) {
    /* subnormal (ri <= 2^mbits; ri == 2^mbits is the smallest normal) */
    out = ri;
  } else {
    /* normal: (E + bias) << mbits plus the fraction; a carry out of the
     * fraction (ri == 2^(mbits+1)) bumps the exponent by itself. */
    out = ((uint64_t)(E + bias) << mbits) + (ri - (1ull << mbits));
  }
  if ((out >> mbits) >= emax_field) return inf_bits; /* rounded past the largest finite */
  return sign | (uint32_t)out;
}

double gemv_ref_decode(uint32_t bits, int fmt) { return ref_decode_bits(bits, fmt); }

uint32_t gemv_ref_encode(double x, int fmt) { return ref_encode_bits(x, fmt); }

/* Decode a whole array of 16-bit patterns (for tests). */
void gemv_ref_decode_array(const uint16_t *bits, int64_t count, int fmt, double *out) {
  for (int64_t i = 0; i < count; ++i) out[i] = ref_decode_bits(bits[i], fmt);
}

/* Encode a whole array of binary64 values; out_fmt REF_F32 writes uint32
 * patterns, the 16-bit formats write uint16 patterns. */
void gemv_ref_encode_array(const double *x, int64_t count, int out_fmt, void *out) {
  for (int64_t i = 0; i < count; ++i) {
    uint32_t b = ref_encode_bits(x[i], out_fmt);
    if (out_fmt == REF_F32)
      ((uint32_t *)out)[i] = b;
    else
      ((uint16_t *)out)[i] = (uint16_t)b;
  }
}

/*
 * c_i = sum_j B[i,j] a[j] and S_i = sum_j |B[i,j] a[j]| in binary64,
 * ascending j, for every row i of the n x k row-major B.  in_fmt is REF_F16
 * or REF_BF16 (B and a share it).  Returns 0, or -1 for a bad argument.
 */
int gemv_ref(const uint16_t *B, const uint16_t *a, int64_t n, int64_t k, int in_fmt, double *c,
             double *s) {
  if (n < 0 || k < 0) return -1;
  if (in_fmt != REF_F16 && in_fmt != REF_BF16) return -1;
  if (n > 0 && (c == NULL || s == NULL)) return -1;
  if (n > 0 && k > 0 && (B == NULL || a == NULL)) return -1;
  for (int64_t i = 0; i < n; ++i) {
    double acc = 0.0;
    double acc_abs = 0.0;
    for (int64_t j = 0; j < k; ++j) {
      double p = ref_decode_bits(B[i * k + j], in_fmt) * ref_decode_bits(a[j], in_fmt);
      acc += p;
      acc_abs += fabs(p);
    }
    c[i] = acc;
    s[i] = acc_abs;
  }
  return 0;
}

/*
 * The same sums for a chosen subset of rows: rows[0..m-1] are row indices of
 * the n x k matrix B; c[r] and s[r] receive row rows[r]'s results.  Lets a
 * test check sampled rows of a matrix too large for the full oracle.
 */
int gemv_ref_rows(const uint16_t *B, const uint16_t *a, int64_t n, int64_t k, int in_fmt,
                  const int64_t *rows, int64_t m, double *c, double *s) {
  if (n < 0 || k < 0 || m < 0) return -1;
  for (int64_t r = 0; r < m; ++r) {
    if (rows[r] < 0 || rows[r] >= n) return -1;
    int rc = gemv_ref(B + rows[r] * k, a, 1, k, in_fmt, c + r, s + r);
    if (rc != 0) return rc;
  }
  return 0;
}

/* Activation codes (the same numbering as the library's, written here
 * independently). */
#define REF_ACT_NONE 0
#define REF_ACT_RELU 1
#define REF_ACT_SIGMOID 2
#define REF_ACT_SILU 3

static double ref_activation(double y, int act) {
  switch (act) {
    case REF_ACT_RELU: return y > 0.0 ? y : 0.0;
    case REF_ACT_SIGMOID: return 1.0 / (1.0 + exp(-y));
    case REF_ACT_SILU: return y / (1.0 + exp(-y));
    default: return y;
  }
}

/* Largest slope of each activation (bounds how an error in its argument
 * propagates): 1 for identity and relu, 1/4 for sigmoid, < 1.1 for silu. */
static double ref_activation_slope(int act) {
  switch (act) {
    case REF_ACT_SIGMOID: return 0.25;
    case REF_ACT_SILU: return 1.1;
    default: return 1.0;
  }
}

/*
 * y_i = act(alpha * c_i + beta * bias_i) for i < n, in binary64.  bias holds
 * n bit patterns of bias_fmt (REF_F16 or REF_BF16: uint16, REF_F32: uint32)
 * or is NULL (no bias).  scale_i = (|alpha| s_i + |beta bias_i|) * slope(act)
 * is the size against which the fp32-output tolerance is stated (s_i from
 * gemv_ref).  Returns 0, or -1 for a bad argument.
 */
int gemv_ref_epilogue(const double *c, const double *s, int64_t n, double alpha, double beta, const void *bias,
                      int bias_fmt, int act, double *y, double *scale) {
  if (n < 0 || act < REF_ACT_NONE || act > REF_ACT_SILU) return -1;
  if (bias != NULL && bias_fmt != REF_F16 && bias_fmt != REF_BF16 && bias_fmt != REF_F32) return -1;
  for (int64_t i = 0; i < n; ++i) {
    double b = 0.0;
    if (bias != NULL) {
      uint32_t bits = (bias_fmt == REF_F32) ? ((const uint32_t *)bias)[i] : ((const uint16_t *)bias)[i];
      b = ref_decode_bits(bits, bias_fmt);
    }
    double pre = alpha * c[i] + beta * b;
    y[i] = ref_activation(pre, act);
    scale[i] = (fabs(alpha) * s[i] + fabs(beta * b)) * ref_activation_slope(act);
  }
  return 0;
}

/*
 * One decode step of gated linear attention (TileLang Case Studies, Case D
 * "Background"), for bh independent heads:
 *
 *     S_new[i, j] = exp(gk[i]) * S[i, j] + k[i] * v[j]      (i < dk, j < dv)
 *     o[j]        = scale * sum_{i<dk} q[i] * S_new[i, j]
 *
 * Layout per head h: q, k, gk at h*dk, v and o at h*dv, S and S_new at
 * h*dk*dv (row i, column j at i*dv + j).  Inputs are bit patterns of fmt
 * (REF_F16, REF_BF16 or REF_F32; uint16 or uint32 arrays), decoded from the
 * format definitions; everything is computed in binary64, S_new before any
 * rounding feeds o.  Outputs: S_new and o in binary64, plus the tolerance
 * scales ss[h,i,j] = |exp(gk[i]) S[i,j]| + |k[i] v[j]| and
 * os[h,j] = |scale| * sum_i |q[i] S_new[i,j]|.  Returns 0, or -1.
 */
static double ref_load(const void *p, int64_t idx, int fmt) {
  uint32_t bits = (fmt == REF_F32) ? ((const uint32_t *)p)[idx] : ((const uint16_t *)p)[idx];
  return ref_decode_bits(bits, fmt);
}

int gla_ref_decode(const void *q, const void *k, const void *v, const void *gk, const void *S, int64_t bh,
                   int64_t dk, int64_t dv, double scale, int fmt, double *S_new, double *o, double *ss,
                   double *os) {
  if (bh < 0 || dk < 0 || dv < 0) return -1;
  if (fmt != REF_F16 && fmt != REF_BF16 && fmt != REF_F32) return -1;
  for (int64_t h = 0; h < bh; ++h) {
    for (int64_t j = 0; j < dv; ++j) {
      double acc = 0.0, acc_abs = 0.0;
      for (int64_t i = 0; i < dk; ++i) {
        const double decay = exp(ref_load(gk, h * dk + i, fmt));
        const double sij = ref_load(S, (h * dk + i) * dv + j, fmt);
        const double kv = ref_load(k, h * dk + i, fmt) * ref_load(v, h * dv + j, fmt);
        const double sn = decay * sij + kv;
        S_new[(h * dk + i) * dv + j] = sn;
        ss[(h * dk + i) * dv + j] = fabs(decay * sij) + fabs(kv);
        const double qi = ref_load(q, h * dk + i, fmt);
        acc += qi * sn;
        acc_abs += fabs(qi * sn);
      }
      o[h * dv + j] = scale * acc;
      os[h * dv + j] = fabs(scale) * acc_abs;
    }
  }
  return 0;
}
