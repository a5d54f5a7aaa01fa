/*
 * NVFP4 block-scaled GEMV oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU statement of what the GPU library
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it; the product path never does.  It shares no code, header,
 * table or constant with the CUDA sources.
 *
 * What is computed (kernelbot "nvfp4-gemv" submission 103289, `cute_kernel`:
 * the k-tile loop accumulates a*sfa*b*sfb per element in FP32, then stores
 * `res.to(Float16)`; submission 69953's docstring gives the shapes):
 *
 *   c[m,l] = fp16( sum_k  E2M1(a[m,k,l]) * E4M3(sfa[m,k/16,l])
 *                        * E2M1(b[k,l])   * E4M3(sfb[k/16,l]) )
 *
 * Memory layouts (submission 103289, `cute_jit_kernel`: A has stride
 * (k, 1, m*k), so it is [L][M][K/2] bytes; c has stride (1, 1, m), so it is
 * [L][M] fp16):
 *   a    uint8 [L][M][K/2]  two E2M1 codes per byte, low nibble = lower k
 *   b    uint8 [L][K/2]     same packing
 *   sfa  uint8 [L][M][K/16] one E4M3 code per 16-element K block
 *   sfb  uint8 [L][K/16]
 *   c    fp16 bits [L][M]
 *
 * Readings where the pages are silent (they name the types only:
 * `cutlass.Float4E2M1FN`, `cutlass.Float8E4M3FN`, submission 103289 kernel
 * configuration):
 *   - E2M1 is the OCP MX FP4 format: sign, 2 exponent bits (bias 1),
 *     1 mantissa bit, no Inf/NaN; code 0x8 is -0.
 *   - E4M3 "FN" is finite-only: sign, 4 exponent bits (bias 7), 3 mantissa
 *     bits, subnormals at exponent 0, exponent 15 with mantissa 7 is NaN.
 *   - The fp16 store rounds to nearest, ties to even; |x| >= 65520 -> +-Inf.
 *
 * Two independent summation paths are provided:
 *   oracle_gemv_f64   : table decode, fp64 accumulate (exact whenever the
 *                       partial sums need <= 53 significant bits, which
 *                       holds for all benchmark value distributions).
 *   oracle_gemv_exact : bit-field decode to integers, exact int64 sum of
 *                       term * 2^20, integer round-to-nearest-even to fp16.
 * Tests pin one against the other and both against hand-worked values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Element decoding (fp64 path): tables generated from the bit-field    */
/* definitions once, never typed by hand.                               */
/* ------------------------------------------------------------------ */

static double g_e2m1[16];
static double g_e4m3[256];
static int g_tables_ready = 0;

static double e2m1_from_code(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag;
  if (e == 0)
    mag = 0.5 * (double)m; /* subnormal: m/2 * 2^(1-1) */
  else
    mag = ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
  return s ? -mag : mag;
}

static double e4m3_from_code(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7); /* subnormal: m/8 * 2^(1-bias) */
  else
    mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

static void tables_init(void) {
  if (g_tables_ready) return;
  for (unsigned c = 0; c < 16; ++c) g_e2m1[c] = e2m1_from_code(c);
  for (unsigned c = 0; c < 256; ++c) g_e4m3[c] = e4m3_from_code(c);
  g_tables_ready = 1;
}

void oracle_e2m1_table(double* out16) {
  tables_init();
  memcpy(out16, g_e2m1, sizeof(g_e2m1));
}

void oracle_e4m3_table(double* out256) {
  tables_init();
  memcpy(out256, g_e4m3, sizeof(g_e4m3));
}

/* Nibble k of a packed row: byte k/2, low nibble for even k. */
static unsigned nibble(const uint8_t* row, int64_t k) {
  uint8_t byte = row[k / 2];
  return (k % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);
}

/* ------------------------------------------------------------------ */
/* IEEE-754 binary16 round-to-nearest-even from a double.               */
/* ------------------------------------------------------------------ */

uint16_t oracle_fp16_rne(double x) {
  if (isnan(x)) return 0x7E00u;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double ax = fabs(x);
  /* 65520 is the midpoint between the largest finite half (65504) and
   * 2^16; the tie goes to the even neighbour, which is 2^16 = overflow. */
  if (ax >= 65520.0) return (uint16_t)(sign | 0x7C00u);
  if (ax < ldexp(1.0, -14)) {
    /* subnormal range: fixed quantum 2^-24; rint() rounds half to even */
    double q = rint(ldexp(ax, 24));
    return (uint16_t)(sign | (uint16_t)q); /* q == 1024 encodes 2^-14 */
  }
  int e2;
  frexp(ax, &e2);     /* ax = f * 2^e2 with f in [0.5, 1) */
  int E = e2 - 1;     /* ax in [2^E, 2^(E+1)) */
  double q = rint(ldexp(ax, 10 - E)); /* 11-bit significand in [1024, 2048] */
  if (q == 2048.0) {
    q = 1024.0;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)(((unsigned)(E + 15) << 10) | ((unsigned)q - 1024u)));
}

void oracle_fp16_rne_array(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp16_rne(x[i]);
}

/* ------------------------------------------------------------------ */
/* fp64 path                                                            */
/* ------------------------------------------------------------------ */

/* One output c[m,l]: the plain definition, k in increasing order. */
static void one_output_f64(const uint8_t* a, const uint8_t* b, const uint8_t* sfa,
                           const uint8_t* sfb, int64_t M, int64_t K, int64_t m, int64_t l,
                           double* sum_out, double* sumabs_out) {
  const int64_t half_k = K / 2, blocks = K / 16;
  const uint8_t* arow = a + (l * M + m) * half_k;
  const uint8_t* brow = b + l * half_k;
  const uint8_t* sarow = sfa + (l * M + m) * blocks;
  const uint8_t* sbrow = sfb + l * blocks;
  double acc = 0.0, accabs = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double av = g_e2m1[nibble(arow, k)];
    double sa = g_e4m3[sarow[k / 16]];
    double bv = g_e2m1[nibble(brow, k)];
    double sb = g_e4m3[sbrow[k / 16]];
    double term = av * sa * bv * sb; /* exact: <= 12 significant bits */
    acc += term;
    accabs += fabs(term);
  }
  *sum_out = acc;
  *sumabs_out = accabs;
}

/* Full GEMV.  c_out: fp16 bits [L][M]; sum_out / sumabs_out (optional, may
 * be NULL): the fp64 sum and sum of |terms| per output. */
void oracle_gemv_f64(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb,
                     int64_t M, int64_t K, int64_t L, uint16_t* c_out, double* sum_out,
                     double* sumabs_out) {
  tables_init();
  for (int64_t l = 0; l < L; ++l)
    for (int64_t m = 0; m < M; ++m) {
      double s, sa;
      one_output_f64(a, b, sfa, sfb, M, K, m, l, &s, &sa);
      c_out[l * M + m] = oracle_fp16_rne(s);
      if (sum_out) sum_out[l * M + m] = s;
      if (sumabs_out) sumabs_out[l * M + m] = sa;
    }
}

/* Selected outputs only (m_idx[i], l_idx[i]), for sampled checks of
 * full-size problems. */
void oracle_gemv_f64_at(const uint8_t* a, const uint8_t* b, const uint8_t* sfa,
                        const uint8_t* sfb, int64_t M, int64_t K, int64_t L,
                        const int64_t* m_idx, const int64_t* l_idx, int64_t n, uint16_t* c_out,
                        double* sum_out, double* sumabs_out) {
  (void)L;
  tables_init();
  for (int64_t i = 0; i < n; ++i) {
    double s, sa;
    one_output_f64(a, b, sfa, sfb, M, K, m_idx[i], l_idx[i], &s, &sa);
    c_out[i] = oracle_fp16_rne(s);
    if (sum_out) sum_out[i] = s;
    if (sumabs_out) sumabs_out[i] = sa;
  }
}

/* ------------------------------------------------------------------ */
/* Exact integer path (independent decode, no tables, no floating point) */
/* ------------------------------------------------------------------ */

/* 2 * E2M1 value as an integer in [-12, 12]. */
static int64_t e2m1_times2(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  int64_t mag = (e == 0) ? (int64_t)m : ((int64_t)(2u + m) << (e - 1u));
  return s ? -mag : mag;
}

/* 2^9 * E4M3 value as an integer (|.| <= 229376); *is_nan set for NaN. */
static int64_t e4m3_times512(unsigned code, int* is_nan) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  if (e == 15 && m == 7) {
    *is_nan = 1;
    return 0;
  }
  int64_t mag = (e == 0) ? (int64_t)m : ((int64_t)(8u + m) << (e - 1u));
  return s ? -mag : mag;
}

static int msb_index(uint64_t v) {
  int i = -1;
  while (v) {
    v >>= 1;
    ++i;
  }
  return i;
}

/* fp16 bits of N * 2^-20, round to nearest even, by integer arithmetic. */
uint16_t oracle_fp16_from_scaled_int(int64_t N) {
  if (N == 0) return 0; /* +0: an fp64 accumulator starting at +0 ends at +0 */
  uint16_t sign = (N < 0) ? 0x8000u : 0u;
  uint64_t U = (N < 0) ? (uint64_t)(-(N + 1)) + 1u : (uint64_t)N;
  int p = msb_index(U);  /* U in [2^p, 2^(p+1)) */
  int E = p - 20;        /* value in [2^E, 2^(E+1)) */
  if (E < -14) {
    /* subnormal: quantum 2^-24 = 2^-4 units of 2^-20, so U*16 is exact */
    return (uint16_t)(sign | (uint16_t)(U << 4));
  }
  int sh = p - 10; /* keep 11 significant bits */
  uint64_t q;
  if (sh <= 0) {
    q = U << (-sh);
  } else {
    q = U >> sh;
    uint64_t rem = U & ((1ull << sh) - 1ull);
    uint64_t half = 1ull << (sh - 1);
    if (rem > half || (rem == half && (q & 1ull))) q += 1;
    if (q == 2048u) {
      q = 1024u;
      E += 1;
    }
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)(((unsigned)(E + 15) << 10) | (unsigned)(q - 1024u)));
}

/* Exact GEMV.  num_out: sum of terms times 2^20 (exact, int64); nan_out:
 * 1 where any scale on the row is NaN; c_out: fp16 bits.  Requires
 * K <= 2^20 so that the int64 sum cannot overflow (checked: returns -1). */
int oracle_gemv_exact(const uint8_t* a, const uint8_t* b, const uint8_t* sfa, const uint8_t* sfb,
                      int64_t M, int64_t K, int64_t L, int64_t* num_out, uint8_t* nan_out,
                      uint16_t* c_out) {
  if (K > (1ll << 20)) return -1;
  const int64_t half_k = K / 2, blocks = K / 16;
  for (int64_t l = 0; l < L; ++l)
    for (int64_t m = 0; m < M; ++m) {
      const uint8_t* arow = a + (l * M + m) * half_k;
      const uint8_t* brow = b + l * half_k;
      const uint8_t* sarow = sfa + (l * M + m) * blocks;
      const uint8_t* sbrow = sfb + l * blocks;
      int64_t total = 0;
      int nan = 0;
      for (int64_t k = 0; k < K; ++k) {
        int64_t a2 = e2m1_times2(nibble(arow, k));
        int64_t b2 = e2m1_times2(nibble(brow, k));
        int64_t sa = e4m3_times512(sarow[k / 16], &nan);
        int64_t sb = e4m3_times512(sbrow[k / 16], &nan);
        /* term * 2^20 = (a2/2)(b2/2)(sa/2^9)(sb/2^9) * 2^20 = a2*b2*sa*sb */
        total += a2 * b2 * sa * sb;
      }
      num_out[l * M + m] = total;
      nan_out[l * M + m] = (uint8_t)nan;
      c_out[l * M + m] = nan ? (uint16_t)0x7E00u : oracle_fp16_from_scaled_int(total);
    }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Scale repack: plain [L][rows][K/16] -> 128x4-atom pre-permuted.      */
/* ------------------------------------------------------------------ */

/*
 * The permuted tensor is [32, 4, rest_m, 4, rest_k, L] (submission 103289,
 * `permuted_to_blocked` docstring), and permuting it to
 * [rest_m, rest_k, 32, 4, 4] is a view of the blocked [-1, 32, 16] order that
 * submission 69953's `to_blocked_batch` builds with
 * view(rest_m,128,rest_k,4).permute(0,2,1,3).reshape(-1,4,32,4).transpose(1,2).
 * Stored with L outermost, byte (m, kb) of batch l lands at
 *
 *   ((l*rest_m + m/128)*rest_k + kb/4)*512 + (m%32)*16 + ((m/32)%4)*4 + kb%4
 *
 * with rest_m = ceil(rows/128) and rest_k = ceil(K/64): both helpers size the
 * blocked tensor with ceil_div (rows/128, (K/16)/4).  Rows m in
 * [rows, 128*rest_m) and, when K % 64 != 0, blocks kb in [K/16, 4*rest_k) are
 * padding and hold 0x00 (the pages fill neither; zero is the plainest reading,
 * and a zero scale adds nothing to any dot product).
 */
int64_t oracle_permuted_scale_bytes(int64_t rows, int64_t K, int64_t L) {
  int64_t rest_m = (rows + 127) / 128, rest_k = (K + 63) / 64;
  return L * rest_m * rest_k * 512;
}

void oracle_repack_scales(const uint8_t* src, uint8_t* dst, int64_t rows, int64_t K, int64_t L) {
  const int64_t blocks = K / 16, rest_m = (rows + 127) / 128, rest_k = (K + 63) / 64;
  memset(dst, 0, (size_t)oracle_permuted_scale_bytes(rows, K, L));
  for (int64_t l = 0; l < L; ++l)
    for (int64_t m = 0; m < rows; ++m)
      for (int64_t kb = 0; kb < blocks; ++kb) {
        int64_t off = ((l * rest_m + m / 128) * rest_k + kb / 4) * 512 + (m % 32) * 16 +
                      ((m / 32) % 4) * 4 + kb % 4;
        dst[off] = src[(l * rows + m) * blocks + kb];
      }
}
