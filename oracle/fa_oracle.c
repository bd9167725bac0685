/*
 * CPU oracle for the fused causal GQA attention forward and the q4_0 K/V cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously-correct statement of what the
 * GPU path computes.  Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg load it; the product library neither links nor calls it, and it shares no code, header or
 * table with the CUDA sources.
 *
 * Everything here is f64 (attention) or IEEE f32 with round-to-nearest-even (the quantizer, whose
 * f32 operation sequence is part of the format's definition).  It must be compiled without
 * floating-point contraction (-ffp-contract=off) and without fast-math.
 *
 * What is computed and where it comes from:
 *
 *  - attention: O[b,h,i,:] = sum_j softmax_j(scale * <Q[b,h,i,:], K[b,g(h),j,:]> + mask_ij) V[b,g(h),j,:]
 *    This is the "explicit matmul + softmax + matmul" reference that the page
 *    "perf(rocm): defer SDPA accumulator rescale, stage Q once per block (#2306)" tests its fused
 *    kernel against (Conversation, second paragraph; What changed), and the SDPA call of
 *    "Build FlashAttention (CK backend) on gfx90a" (Verification).  Grouped-query heads map query
 *    head h to key/value head g(h) = h / (Hq/Hkv) (contiguous groups; that page's GQA 32/8
 *    shape).  The causal mask hides key j from query row i when j > q_pos_offset + i, so a query
 *    chunk placed at positions Sk-Sq..Sk-1 is bottom-right aligned and the diagonal is visible.
 *    The deferred-rescale frame of the fused kernel is NOT modelled: the exact result does not
 *    depend on it.
 *
 *  - q4_0: the pages name the q4_0 cache type ("FlashAttention on gfx90a: Why It's Broken and How
 *    to Fix It", Impact of the V Dequant Patch: -ctk q4_0 -ctv q4_0) but do not fix its bits.  The
 *    format used throughout this library: blocks of 32 consecutive elements along the head
 *    dimension; per block an fp16 scale d = m / -8 where m is the signed element of largest
 *    magnitude (first one wins ties); codes q = min(15, trunc(x * (1/d) + 8.5)) in 4 bits; value
 *    x' = (q - 8) * d.  The f32 operation order (one multiply, one add, both rounded) is part of
 *    the definition, so the GPU quantizer can be bit-exact against this one.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary32/64, written out from the formats (no library conversion).        */
/* ------------------------------------------------------------------------------------------ */

/* Round an f32 to the nearest binary16 (ties to even).  Handles subnormals, overflow to inf
 * and NaN. */
uint16_t oracle_f32_to_f16_rn(float x) {
  uint32_t u;
  memcpy(&u, &x, 4);
  uint32_t sign = (u >> 16) & 0x8000u;
  uint32_t exp = (u >> 23) & 0xffu;
  uint32_t man = u & 0x7fffffu;
  if (exp == 0xffu) { /* inf or NaN */
    return (uint16_t)(sign | 0x7c00u | (man ? 0x200u : 0u));
  }
  /* value = 1.man * 2^(exp-127) for normal f32 */
  int32_t e = (int32_t)exp - 127;
  if (exp == 0) return (uint16_t)sign; /* f32 subnormals are far below the f16 range: +-0 */
  if (e > 15) return (uint16_t)(sign | 0x7c00u); /* overflow */
  uint32_t full = man | 0x800000u; /* 24-bit significand, value = full * 2^(e-23) */
  uint32_t shift;
  uint32_t h_exp;
  if (e >= -14) { /* normal f16: keep 11 significant bits */
    shift = 13;
    h_exp = (uint32_t)(e + 15);
  } else { /* subnormal f16: value = m * 2^-24, m = full * 2^(e-23+24) */
    int32_t s = 13 + (-14 - e);
    if (s > 25) return (uint16_t)sign; /* below half of the smallest subnormal */
    shift = (uint32_t)s;
    h_exp = 0;
  }
  uint32_t kept = full >> shift;
  uint32_t rem = full & ((1u << shift) - 1u);
  uint32_t half = 1u << (shift - 1);
  if (rem > half || (rem == half && (kept & 1u))) kept += 1u;
  uint32_t out;
  if (h_exp == 0) {
    out = kept; /* may carry into the smallest normal, which is the right encoding */
  } else {
    /* kept has the implicit bit at position 10; a carry to bit 11 bumps the exponent */
    if (kept & 0x800u) {
      kept >>= 1;
      h_exp += 1;
    }
    if (h_exp >= 31) return (uint16_t)(sign | 0x7c00u);
    out = (h_exp << 10) | (kept & 0x3ffu);
  }
  return (uint16_t)(sign | out);
}

/* Exact value of a binary16 bit pattern. */
double oracle_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int exp = (h >> 10) & 0x1f;
  int man = h & 0x3ff;
  double v;
  if (exp == 0) {
    v = ldexp((double)man, -24);
  } else if (exp == 31) {
    v = man ? NAN : INFINITY;
  } else {
    v = ldexp((double)(man | 0x400), exp - 25);
  }
  return sign ? -v : v;
}

/* ------------------------------------------------------------------------------------------ */
/* q4_0 quantize / dequantize (scalar, one 32-element block at a time).                        */
/* ------------------------------------------------------------------------------------------ */

enum { QK = 32 };

/* Quantize nblocks consecutive blocks of 32 f32 values.  nib receives 16 bytes per block (byte j
 * holds element j in its low nibble and element j+16 in its high nibble); scale receives the fp16
 * bit pattern of d. */
void oracle_quantize_q4_0(const float* x, int64_t nblocks, uint8_t* nib, uint16_t* scale) {
  for (int64_t b = 0; b < nblocks; ++b) {
    const float* xb = x + b * QK;
    /* m: the signed element of largest magnitude; a strict '>' keeps the first on ties */
    float amax = 0.0f;
    float m = 0.0f;
    for (int j = 0; j < QK; ++j) {
      float a = fabsf(xb[j]);
      if (a > amax) {
        amax = a;
        m = xb[j];
      }
    }
    float d = m / -8.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    uint8_t q[QK];
    for (int j = 0; j < QK; ++j) {
      float t = xb[j] * id; /* rounded f32 product */
      t = t + 8.5f;         /* rounded f32 sum */
      int qi = (int)t;      /* C conversion truncates toward zero */
      if (qi > 15) qi = 15;
      if (qi < 0) qi = 0;   /* unreachable for finite input: x*id >= -8 up to rounding */
      q[j] = (uint8_t)qi;
    }
    for (int j = 0; j < QK / 2; ++j) {
      nib[b * (QK / 2) + j] = (uint8_t)(q[j] | (q[j + QK / 2] << 4));
    }
    scale[b] = oracle_f32_to_f16_rn(d);
  }
}

/* Exact dequantized values (q - 8) * d16 of nblocks blocks, in f64. */
void oracle_dequantize_q4_0(const uint8_t* nib, const uint16_t* scale, int64_t nblocks,
                            double* out) {
  for (int64_t b = 0; b < nblocks; ++b) {
    double d = oracle_f16_to_f64(scale[b]);
    for (int j = 0; j < QK / 2; ++j) {
      uint8_t byte = nib[b * (QK / 2) + j];
      int lo = byte & 0x0f;
      int hi = byte >> 4;
      out[b * QK + j] = (double)(lo - 8) * d;
      out[b * QK + j + QK / 2] = (double)(hi - 8) * d;
    }
  }
}

/* ------------------------------------------------------------------------------------------ */
/* Attention, one query row at a time.                                                          */
/* ------------------------------------------------------------------------------------------ */

/* K/V source: either dense f64 [B, Hkv, Sk, D] or a q4_0 cache (nibble plane [B,Hkv,Sk,D/2],
 * fp16 scale plane [B,Hkv,Sk,D/32]) that is dequantized exactly, element by element. */
typedef struct {
  const double* dense;
  const uint8_t* nib;
  const uint16_t* scale;
} kv_src;

static double kv_at(const kv_src* s, int64_t row, int D, int d) {
  if (s->dense) return s->dense[row * D + d];
  const uint8_t byte = s->nib[row * (D / 2) + (d / QK) * (QK / 2) + (d % QK) % (QK / 2)];
  int code = (d % QK) < QK / 2 ? (byte & 0x0f) : (byte >> 4);
  double dd = oracle_f16_to_f64(s->scale[row * (D / QK) + d / QK]);
  return (double)(code - 8) * dd;
}

typedef struct {
  const double* q;
  kv_src k, v;
  double* o;     /* [nrows, D] */
  double* prob;  /* optional [nrows, Sk]: the softmax row */
  int B, Hq, Hkv, Sq, Sk, D, q_pos_offset, causal;
  double scale;
  const int64_t* rows;
  int64_t nrows;
  int64_t next; /* work counter */
  pthread_mutex_t mu;
} att_job;

static void one_row(att_job* J, int64_t r, double* s) {
  const int64_t flat = J->rows[r]; /* (b * Hq + h) * Sq + i */
  const int i = (int)(flat % J->Sq);
  const int64_t bh = flat / J->Sq;
  const int h = (int)(bh % J->Hq);
  const int b = (int)(bh / J->Hq);
  const int g = h / (J->Hq / J->Hkv);
  const int D = J->D;
  const double* qrow = J->q + flat * D;
  const int64_t kv_row0 = ((int64_t)b * J->Hkv + g) * J->Sk;
  const int64_t pos = (int64_t)J->q_pos_offset + i;

  /* scores, with masked keys at -inf */
  double m = -INFINITY;
  for (int j = 0; j < J->Sk; ++j) {
    if (J->causal && j > pos) {
      s[j] = -INFINITY;
      continue;
    }
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += qrow[d] * kv_at(&J->k, kv_row0 + j, D, d);
    s[j] = J->scale * acc;
    if (s[j] > m) m = s[j];
  }
  /* softmax with max subtraction */
  double l = 0.0;
  for (int j = 0; j < J->Sk; ++j) {
    s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
    l += s[j];
  }
  for (int j = 0; j < J->Sk; ++j) s[j] /= l;
  if (J->prob) memcpy(J->prob + r * J->Sk, s, sizeof(double) * (size_t)J->Sk);
  /* O = P V */
  double* orow = J->o + r * D;
  for (int d = 0; d < D; ++d) orow[d] = 0.0;
  for (int j = 0; j < J->Sk; ++j) {
    if (s[j] == 0.0) continue;
    for (int d = 0; d < D; ++d) orow[d] += s[j] * kv_at(&J->v, kv_row0 + j, D, d);
  }
}

static void* att_worker(void* arg) {
  att_job* J = (att_job*)arg;
  double* s = (double*)malloc(sizeof(double) * (size_t)J->Sk);
  if (!s) return NULL;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    int64_t r = J->next;
    J->next += 1;
    pthread_mutex_unlock(&J->mu);
    if (r >= J->nrows) break;
    one_row(J, r, s);
  }
  free(s);
  return NULL;
}

static int run_rows(att_job* J, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 512) nthreads = 512;
  pthread_t th[512];
  pthread_mutex_init(&J->mu, NULL);
  J->next = 0;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, att_worker, J) != 0) break;
    ++started;
  }
  if (started == 0) att_worker(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&J->mu);
  return started;
}

/* Attention rows over a dense f64 K/V.  rows[] holds flat indices (b*Hq + h)*Sq + i into the
 * query tensor; o receives one D-vector per listed row; prob (optional, may be NULL) receives
 * the softmax row of each listed row.  Returns the number of threads used. */
int oracle_attention_rows(const double* q, const double* k, const double* v, double* o,
                          double* prob, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                          int q_pos_offset, int causal, double scale, const int64_t* rows,
                          int64_t nrows, int nthreads) {
  att_job J;
  memset(&J, 0, sizeof(J));
  J.q = q;
  J.k.dense = k;
  J.v.dense = v;
  J.o = o;
  J.prob = prob;
  J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.Sq = Sq; J.Sk = Sk; J.D = D;
  J.q_pos_offset = q_pos_offset;
  J.causal = causal;
  J.scale = scale;
  J.rows = rows;
  J.nrows = nrows;
  return run_rows(&J, nthreads);
}

/* Same, with K and V read from q4_0 caches (exact dequantization per element). */
int oracle_attention_rows_q4_0(const double* q, const uint8_t* k_nib, const uint16_t* k_scale,
                               const uint8_t* v_nib, const uint16_t* v_scale, double* o,
                               double* prob, int B, int Hq, int Hkv, int Sq, int Sk, int D,
                               int q_pos_offset, int causal, double scale, const int64_t* rows,
                               int64_t nrows, int nthreads) {
  att_job J;
  memset(&J, 0, sizeof(J));
  J.q = q;
  J.k.nib = k_nib;
  J.k.scale = k_scale;
  J.v.nib = v_nib;
  J.v.scale = v_scale;
  J.o = o;
  J.prob = prob;
  J.B = B; J.Hq = Hq; J.Hkv = Hkv; J.Sq = Sq; J.Sk = Sk; J.D = D;
  J.q_pos_offset = q_pos_offset;
  J.causal = causal;
  J.scale = scale;
  J.rows = rows;
  J.nrows = nrows;
  return run_rows(&J, nthreads);
}
