/*
 * RoPE oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU statement of the two rotary-position-embedding
 * operators, written to be checked against the source pages by eye.  Only the
 * test-suite, the package smoke check and the benchmark's CPU-baseline leg
 * load it; the product path never calls, links or imports it.
 *
 * Arithmetic: every input element is widened exactly to binary64, the formula
 * is evaluated in binary64 in the pages' own order, and the result is rounded
 * once (round-to-nearest-even) to the output type.  No fusion, no blocking, no
 * reordering beyond what the formulas state.
 *
 * Sources (web pages, cited by title and section):
 *  [IPRM] "CANN ops-transformer 的 aclnnInplacePartialRotaryMul 算子：Inplace
 *         部分旋转位置编码接口详解与实现剖析"
 *  [RSCC] "CANN ops-transformer 旋转位置编码算子 RopeWithSinCosCache 深度解析：
 *         cache 化 RoPE 的计算原理与 aclnn 两段式调用实战"
 *
 * Readings taken where the pages are silent, garbled or ambiguous:
 *  (1) [IPRM §计算原理与公式] builds the rotated vector from the even members
 *      x1 = x[0::2] and odd members x2 = x[1::2] with a "cat" of (-x2, x1) and
 *      calls the mode "interleave".  Read as the interleaved rotation: the
 *      rotated vector holds -x2[p] at slot 2p and x1[p] at slot 2p+1 (a stack
 *      of the two, flattened), so every pair (2p, 2p+1) is rotated on its own.
 *      cos and sin multiply element-wise (their last dim equals the slice
 *      length), so slot 2p+1 uses cos[2p+1] and sin[2p+1].
 *      rotary_mode 0 ("half", declared by the page but not open there) is the
 *      same formula with x1, x2 the two halves of the slice (rotate_half).
 *  (2) [IPRM §partial_slice 局部旋转机制]: slice [0,0] (or no slice) means the
 *      whole D axis; any other start == end is a no-op.
 *  (3) [IPRM §约束说明]: cos/sin broadcast against x per dim (each of B, S, N
 *      is 1 or equal to x's); the per-platform layout lists are treated as
 *      platform limits.
 *  (4) [RSCC §rotate_interleaved]: the stacked pair (o1, o2) is flattened back
 *      to an interleaved row.
 *  (5) [RSCC §mrope 模式]: section k of mropeSection covers cos/sin indices
 *      [sum of sections before k, sum through k) of the R/2 indices; both the
 *      cos and the sin index i take row k of the positions.  The 3- and
 *      4-section forms mean the same thing.  mrope is on when the section is
 *      given and its first element is > 0 (the kernel test the page reports).
 *  (6) [RSCC §V2 接口：cacheMode 扩展] cacheMode 1, three sections: the result
 *      starts as row 0's cos (sin) and the indices 1, 4, 7, ... and 2, 5, 8, ...
 *      below 3*mropeSection[1] are replaced from rows 1 and 2.  The page bounds
 *      both runs by mropeSection[1]; taken literally.
 *  (7) [RSCC §约束说明 item 5] only says positions should be < maxSeqLen.  A
 *      token with any position outside [0, maxSeqLen) is left untouched and
 *      counted in the return value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORA_F32 = 0, ORA_F16 = 1, ORA_BF16 = 2 };

/* An IEEE-style binary format: precision p (significand bits with the hidden
 * one), exponent field width, bias = emax, emin = 1 - emax. */
typedef struct {
  int p;
  int ebits;
  int emax;
} fmt_t;

static fmt_t fmt_of(int dt) {
  fmt_t f;
  switch (dt) {
    case ORA_F16: f.p = 11; f.ebits = 5; f.emax = 15; break;   /* IEEE 754 binary16 */
    case ORA_BF16: f.p = 8; f.ebits = 8; f.emax = 127; break;  /* bfloat16: binary32's top half */
    default: f.p = 24; f.ebits = 8; f.emax = 127; break;       /* IEEE 754 binary32 */
  }
  return f;
}

static int bytes_of(int dt) { return dt == ORA_F32 ? 4 : 2; }

/* Bits -> exact value, from the format's definition. */
static double decode_bits(uint32_t bits, fmt_t f) {
  const int emin = 1 - f.emax;
  uint32_t sign = (bits >> (f.ebits + f.p - 1)) & 1u;
  uint32_t efield = (bits >> (f.p - 1)) & ((1u << f.ebits) - 1u);
  uint32_t frac = bits & ((1u << (f.p - 1)) - 1u);
  double v;
  if (efield == 0)
    v = ldexp((double)frac, emin - (f.p - 1)); /* zero / subnormal */
  else if (efield == (1u << f.ebits) - 1u)
    v = frac ? NAN : INFINITY;
  else
    v = ldexp((double)(frac | (1u << (f.p - 1))), (int)efield - f.emax - (f.p - 1));
  return sign ? -v : v;
}

/* Value -> bits, rounded to nearest, ties to even, from the format's
 * definition: scale the magnitude so that the last kept significand bit has
 * weight one, round that integer, then re-assemble (a carry out of the top
 * bit moves to the next binade; past emax the result is infinity). */
static uint32_t encode_bits(double v, fmt_t f) {
  const int emin = 1 - f.emax;
  const uint32_t sign = signbit(v) ? (1u << (f.ebits + f.p - 1)) : 0u;
  const uint32_t inf = ((1u << f.ebits) - 1u) << (f.p - 1);
  if (isnan(v)) return sign | inf | (1u << (f.p - 2)); /* quiet NaN */
  double a = fabs(v);
  if (isinf(a)) return sign | inf;
  if (a == 0.0) return sign;
  int e2;
  (void)frexp(a, &e2);
  int E = e2 - 1; /* a lies in [2^E, 2^(E+1)) */
  if (E < emin) E = emin;
  double m = nearbyint(ldexp(a, (f.p - 1) - E)); /* default rounding mode: nearest-even */
  if (m >= ldexp(1.0, f.p)) {                     /* rounded up into the next binade */
    m = ldexp(m, -1);
    E += 1;
  }
  if (E > f.emax) return sign | inf;
  uint32_t mi = (uint32_t)m;
  if (mi < (1u << (f.p - 1))) return sign | mi; /* subnormal: exponent field 0 */
  return sign | ((uint32_t)(E + f.emax) << (f.p - 1)) | (mi - (1u << (f.p - 1)));
}

static double load_elem(const void* buf, int dt, int64_t i) {
  if (dt == ORA_F32) {
    uint32_t u;
    memcpy(&u, (const char*)buf + 4 * i, 4);
    return decode_bits(u, fmt_of(dt));
  }
  uint16_t h;
  memcpy(&h, (const char*)buf + 2 * i, 2);
  return decode_bits(h, fmt_of(dt));
}

static void store_elem(void* buf, int dt, int64_t i, double v) {
  uint32_t u = encode_bits(v, fmt_of(dt));
  if (dt == ORA_F32) {
    memcpy((char*)buf + 4 * i, &u, 4);
  } else {
    uint16_t h = (uint16_t)u;
    memcpy((char*)buf + 2 * i, &h, 2);
  }
}

/* Exposed so that the tests can pin the conversions on their own. */
double oracle_decode(uint32_t bits, int dt) { return decode_bits(bits, fmt_of(dt)); }
uint32_t oracle_encode(double v, int dt) { return encode_bits(v, fmt_of(dt)); }
int oracle_elem_bytes(int dt) { return bytes_of(dt); }

/* The rotated vector x_rotate of [IPRM §计算原理与公式] for one slice of
 * length L.  mode 1 (interleave, reading (1)): slot 2p holds -v[2p+1] and slot
 * 2p+1 holds v[2p].  mode 0 (half): the formula's cat(-x2, x1) taken with x1,
 * x2 the two halves of the slice, i.e. rotate_half. */
static void rotated_vector(const double* v, double* out, int64_t L, int mode) {
  if (mode == 1) {
    for (int64_t p = 0; p < L / 2; ++p) {
      out[2 * p] = -v[2 * p + 1];
      out[2 * p + 1] = v[2 * p];
    }
  } else {
    for (int64_t i = 0; i < L / 2; ++i) {
      out[i] = -v[L / 2 + i];
      out[L / 2 + i] = v[i];
    }
  }
}

/*
 * In-place partial rotary multiply, forward or backward.
 * [IPRM §计算原理与公式, §partial_slice 局部旋转机制, §约束说明,
 *  §Python 接口与自动微分 (the backward op computes only x's gradient)]
 *
 * x:   [B, S, N, D] contiguous, type x_dt, rewritten in place on [start, end).
 *      For the backward it holds dL/dy on entry and dL/dx on return.
 * cos, sin: [cB, cS, cN, L] contiguous, type cs_dt, L = end - start; each of
 *      cB, cS, cN is 1 (broadcast) or equal to x's.
 * mode: 1 interleave, 0 half.
 * Forward:  y = x * cos + x_rotate * sin, element-wise.
 * Backward: the transpose of that linear map.  x_rotate = P x with P
 *      antisymmetric (P^T = -P), so dL/dx = dy * cos - P (dy * sin).
 * Returns 0 (the caller validates shapes), -1 on allocation failure.
 */
int oracle_inplace_partial_rope(void* x, int x_dt, const int64_t* x_shape, const void* cos, const void* sin,
                                int cs_dt, const int64_t* cs_shape, int64_t start, int64_t end, int mode,
                                int backward) {
  const int64_t B = x_shape[0], S = x_shape[1], N = x_shape[2], D = x_shape[3];
  if (start == 0 && end == 0) end = D; /* no slice: the whole D axis */
  if (start == end) return 0;          /* empty slice: no-op */
  const int64_t L = end - start;
  double* xs = (double*)malloc(sizeof(double) * (size_t)L);
  double* xrot = (double*)malloc(sizeof(double) * (size_t)L);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)L);
  if (!xs || !xrot || !tmp) {
    free(xs);
    free(xrot);
    free(tmp);
    return -1;
  }
  for (int64_t b = 0; b < B; ++b)
    for (int64_t s = 0; s < S; ++s)
      for (int64_t n = 0; n < N; ++n) {
        const int64_t xrow = ((b * S + s) * N + n) * D;
        const int64_t cb = cs_shape[0] == 1 ? 0 : b;
        const int64_t cs = cs_shape[1] == 1 ? 0 : s;
        const int64_t cn = cs_shape[2] == 1 ? 0 : n;
        const int64_t crow = ((cb * cs_shape[1] + cs) * cs_shape[2] + cn) * L;
        /* the rotated part x[..., start:end] */
        for (int64_t j = 0; j < L; ++j) xs[j] = load_elem(x, x_dt, xrow + start + j);
        if (!backward) {
          /* x = x * cos + x_rotate * sin, element-wise */
          rotated_vector(xs, xrot, L, mode);
          for (int64_t j = 0; j < L; ++j) {
            double c = load_elem(cos, cs_dt, crow + j);
            double sn = load_elem(sin, cs_dt, crow + j);
            double y = xs[j] * c + xrot[j] * sn;
            store_elem(x, x_dt, xrow + start + j, y);
          }
        } else {
          /* dx = dy * cos - P (dy * sin) */
          for (int64_t j = 0; j < L; ++j) tmp[j] = xs[j] * load_elem(sin, cs_dt, crow + j);
          rotated_vector(tmp, xrot, L, mode);
          for (int64_t j = 0; j < L; ++j) {
            double dx = xs[j] * load_elem(cos, cs_dt, crow + j) - xrot[j];
            store_elem(x, x_dt, xrow + start + j, dx);
          }
        }
      }
  free(xs);
  free(xrot);
  free(tmp);
  return 0;
}

/* Rotate the first R elements of one head in place; [R, head_size) pass through.
 * [RSCC §rotate_half（GPT-NeoX style）, §rotate_interleaved（GPT-J style）] */
static void rotate_head(void* buf, int dt, int64_t off, int64_t R, const double* cosv,
                        const double* sinv, int is_neox, double* xr, double* out) {
  const int64_t half = R / 2;
  for (int64_t i = 0; i < R; ++i) xr[i] = load_elem(buf, dt, off + i);
  for (int64_t i = 0; i < half; ++i) {
    double x1, x2;
    if (is_neox) { /* x1, x2 = the two halves of queryRot */
      x1 = xr[i];
      x2 = xr[half + i];
    } else { /* x1 = queryRot[0::2], x2 = queryRot[1::2] */
      x1 = xr[2 * i];
      x2 = xr[2 * i + 1];
    }
    double o1 = x1 * cosv[i] - x2 * sinv[i];
    double o2 = x2 * cosv[i] + x1 * sinv[i];
    if (is_neox) { /* cat(o1, o2) */
      out[i] = o1;
      out[half + i] = o2;
    } else { /* stack(o1, o2) flattened: o1 at even slots, o2 at odd slots */
      out[2 * i] = o1;
      out[2 * i + 1] = o2;
    }
  }
  for (int64_t i = 0; i < R; ++i) store_elem(buf, dt, off + i, out[i]);
}

/*
 * Cache-indexed rotary embedding, rope and mrope modes, applied in place.
 * [RSCC §设计动机 (three steps), §mrope 模式, §rope 模式, §rotate_half,
 *  §rotate_interleaved]
 *
 * positions: int64 [num_tokens] (rope) or [m, num_tokens] (mrope, m = section_len)
 * query: [num_tokens, q_cols], key: [num_tokens, k_cols]; q_cols and k_cols are
 *        multiples of head_size.  Both rewritten in place.
 * cache: [max_seq, R]; row = cos (first R/2) then sin (last R/2).
 * cache_mode (mrope only): 0 splices the sections in order (the V1 rule);
 * 1 is the V2 interleaved splice of [RSCC §V2 接口：cacheMode 扩展].
 * Returns the number of tokens left untouched for an out-of-range position,
 * or -1 on allocation failure.
 */
int64_t oracle_rope_with_sin_cos_cache(const int64_t* positions, const int64_t* mrope_section,
                                       int64_t section_len, void* query, int64_t q_cols, void* key,
                                       int64_t k_cols, int64_t num_tokens, const void* cache,
                                       int64_t max_seq, int64_t R, int dt, int64_t head_size,
                                       int is_neox, int cache_mode) {
  const int mrope = mrope_section != NULL && section_len > 0 && mrope_section[0] > 0;
  const int64_t rows = mrope ? section_len : 1;
  const int64_t half = R / 2;
  if (mrope) {
    int64_t total = 0;
    for (int64_t k = 0; k < section_len; ++k) total += mrope_section[k];
    if (2 * total != R) return -1; /* the sections must tile the R/2 indices */
  }
  double* cos_sin = (double*)malloc(sizeof(double) * (size_t)(rows * R));
  double* cosv = (double*)malloc(sizeof(double) * (size_t)half);
  double* sinv = (double*)malloc(sizeof(double) * (size_t)half);
  double* xr = (double*)malloc(sizeof(double) * (size_t)R);
  double* out = (double*)malloc(sizeof(double) * (size_t)R);
  if (!cos_sin || !cosv || !sinv || !xr || !out) {
    free(cos_sin); free(cosv); free(sinv); free(xr); free(out);
    return -1;
  }
  int64_t skipped = 0;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int bad = 0;
    for (int64_t r = 0; r < rows; ++r) {
      int64_t p = positions[r * num_tokens + t];
      if (p < 0 || p >= max_seq) bad = 1;
    }
    if (bad) {
      ++skipped;
      continue;
    }
    /* step 1: cosSin = cosSinCache[positions] (one row per positions row) */
    for (int64_t r = 0; r < rows; ++r) {
      int64_t p = positions[r * num_tokens + t];
      for (int64_t i = 0; i < R; ++i) cos_sin[r * R + i] = load_elem(cache, dt, p * R + i);
    }
    /* step 2: cos, sin = cosSin.chunk(2, -1); mrope splices section k from row k */
    if (!mrope) {
      for (int64_t i = 0; i < half; ++i) {
        cosv[i] = cos_sin[i];
        sinv[i] = cos_sin[half + i];
      }
    } else if (cache_mode == 1) {
      /* V2 interleaved splice: start from row 0, then indices 1, 4, 7, ... below
       * 3*mropeSection[1] take row 1 and indices 2, 5, 8, ... below the same
       * bound take row 2 */
      for (int64_t i = 0; i < half; ++i) {
        cosv[i] = cos_sin[i];
        sinv[i] = cos_sin[half + i];
      }
      for (int64_t i = 1; i < 3 * mrope_section[1] && i < half; i += 3) {
        cosv[i] = cos_sin[1 * R + i];
        sinv[i] = cos_sin[1 * R + half + i];
      }
      for (int64_t i = 2; i < 3 * mrope_section[1] && i < half; i += 3) {
        cosv[i] = cos_sin[2 * R + i];
        sinv[i] = cos_sin[2 * R + half + i];
      }
    } else {
      int64_t lo = 0;
      for (int64_t k = 0; k < section_len; ++k) {
        for (int64_t i = lo; i < lo + mrope_section[k]; ++i) {
          cosv[i] = cos_sin[k * R + i];
          sinv[i] = cos_sin[k * R + half + i];
        }
        lo += mrope_section[k];
      }
    }
    /* step 3: rotate queryRot = query[..., :R] of every head, then the same for key */
    for (int64_t h = 0; h < q_cols / head_size; ++h)
      rotate_head(query, dt, t * q_cols + h * head_size, R, cosv, sinv, is_neox, xr, out);
    for (int64_t h = 0; h < k_cols / head_size; ++h)
      rotate_head(key, dt, t * k_cols + h * head_size, R, cosv, sinv, is_neox, xr, out);
  }
  free(cos_sin); free(cosv); free(sinv); free(xr); free(out);
  return skipped;
}

/*
 * Fused QKV split + RMSNorm + RoPE + paged KV-cache write, in the order the
 * page gives it ["aclnnQkvRmsNormRopeCacheWithKScale" page, section 计算公式],
 * without its FP8 quantisation and its optional rotation matmul.
 *
 * Readings of the page, whose tables are garbled:
 *  - qkv is [T, (Nq + Nk + Nv) * D], split by heads of D elements;
 *  - RMSNorm is per head over its D elements, y = x / sqrt(mean(x^2) + eps) * gamma,
 *    with one gamma of length D per branch (q_gamma, k_gamma);
 *  - the position of token i of batch b is seqLens[b] - (qsl[b+1] - qsl[b]) + i,
 *    and cos/sin are the halves of cache row `position` of a [maxSeq, D] cos||sin
 *    table (the RopeWithSinCosCache convention);
 *  - RoPE is the page's concat(low*cos - high*sin, high*cos + low*sin) over the
 *    whole head; V gets neither norm nor RoPE;
 *  - q_out is [T, Nq * D]; K and V go to caches [numBlocks, N, BlockSize, D] at
 *    block slot/BlockSize, offset slot%BlockSize; a negative slot means "do not
 *    cache this token" (padding); everything is stored in the input type.
 * Tokens whose position falls outside the table leave q_out unwritten and
 * write no cache; slots at or past numBlocks*BlockSize are not written.
 * Returns (tokens with a bad position) + 2^32 * (tokens with a bad slot), or
 * -1 on allocation failure.
 */
int64_t oracle_qkv_rmsnorm_rope_cache(const void* qkv, int dt, int64_t T, int64_t nq, int64_t nk, int64_t nv,
                                      int64_t D, const void* q_gamma, const void* k_gamma, double eps,
                                      const void* cache, int64_t max_seq, const int64_t* seq_lens,
                                      const int64_t* qsl, int64_t B, const int64_t* slot_mapping,
                                      int64_t block_size, int64_t num_blocks, void* q_out, void* k_cache,
                                      void* v_cache) {
  const int64_t W = (nq + nk + nv) * D, half = D / 2;
  /* tokens of batch b are [qsl[b], qsl[b+1]): qsl must be non-decreasing inside [0, T] */
  for (int64_t b = 0; b <= B; ++b)
    if (qsl[b] < 0 || qsl[b] > T || (b > 0 && qsl[b] < qsl[b - 1])) return -2;
  double* x = (double*)malloc(sizeof(double) * (size_t)D);
  double* y = (double*)malloc(sizeof(double) * (size_t)D);
  double* o = (double*)malloc(sizeof(double) * (size_t)D);
  if (!x || !y || !o) {
    free(x); free(y); free(o);
    return -1;
  }
  int64_t bad_pos = 0, bad_slot = 0;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t t = qsl[b]; t < qsl[b + 1]; ++t) {
      const int64_t i = t - qsl[b];
      const int64_t position = seq_lens[b] - (qsl[b + 1] - qsl[b]) + i;
      if (position < 0 || position >= max_seq) {
        ++bad_pos;
        continue;
      }
      const int64_t slot = slot_mapping[t];
      const int cache_it = slot >= 0 && slot < num_blocks * block_size;
      if (slot >= num_blocks * block_size) ++bad_slot;
      const int64_t blk = cache_it ? slot / block_size : 0, off = cache_it ? slot % block_size : 0;
      for (int64_t h = 0; h < nq + nk + nv; ++h) {
        /* split: head h of qkv */
        for (int64_t j = 0; j < D; ++j) x[j] = load_elem(qkv, dt, t * W + h * D + j);
        if (h >= nq + nk) { /* V: stored as is */
          if (cache_it) {
            const int64_t vh = h - nq - nk;
            for (int64_t j = 0; j < D; ++j)
              store_elem(v_cache, dt, ((blk * nv + vh) * block_size + off) * D + j, x[j]);
          }
          continue;
        }
        /* RMSNorm over the head */
        const void* gamma = h < nq ? q_gamma : k_gamma;
        double ss = 0.0;
        for (int64_t j = 0; j < D; ++j) ss += x[j] * x[j];
        const double rms = sqrt(ss / (double)D + eps);
        for (int64_t j = 0; j < D; ++j) y[j] = x[j] / rms * load_elem(gamma, dt, j);
        /* RoPE: concat(low*cos - high*sin, high*cos + low*sin) */
        for (int64_t j = 0; j < half; ++j) {
          const double c = load_elem(cache, dt, position * D + j);
          const double s = load_elem(cache, dt, position * D + half + j);
          o[j] = y[j] * c - y[half + j] * s;
          o[half + j] = y[half + j] * c + y[j] * s;
        }
        if (h < nq) {
          for (int64_t j = 0; j < D; ++j) store_elem(q_out, dt, (t * nq + h) * D + j, o[j]);
        } else if (cache_it) {
          const int64_t kh = h - nq;
          for (int64_t j = 0; j < D; ++j)
            store_elem(k_cache, dt, ((blk * nk + kh) * block_size + off) * D + j, o[j]);
        }
      }
    }
  }
  free(x); free(y); free(o);
  return bad_pos + (bad_slot << 32);
}
