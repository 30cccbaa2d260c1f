/*
 * CPU oracle for the asymmetric low-bit KV cache and its decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file: only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * Plain, slow, literal code.  Build with -O2 -ffp-contract=off (no fast-math):
 * every fp32 step below is one IEEE round-to-nearest-even operation.
 *
 * What it computes, with the passages it follows (page title, section):
 *  - Uniform asymmetric integer quantizer: the group minimum is the zero
 *    point, the step is range/(2^B-1), every element rounds to the nearest
 *    step, so the element error is at most half a step.
 *    ("KV cache has a geometry problem, not a bit problem", section
 *    "Quantization error in practice".)
 *  - Keys grouped per channel over G tokens; values grouped per token over G
 *    channels.  (Same page, sections "Keys" and "Values"; KIVI summary page,
 *    section "Method".)
 *  - fp16 zero point and scale, G = 32 ("KIVI" summary page, "Experiments").
 *  - Per-vector dense-and-sparse keys: the largest-magnitude entries of each
 *    key vector are kept in fp16 and left out of the group ranges.
 *    (KVQuant review, "Proposed method", item on per-vector dense/sparse.)
 *  - Pre-RoPE keys: rotate after dequantization.  (unite.ai page, section
 *    "Rotary embeddings complicate keys"; KVQuant review, "Proposed method".)
 *  - Decode attention softmax(q.K^T*scale).V over the whole cache in fp64,
 *    and the log-sum-exp merge of partial results over token ranges.
 *
 * Readings where the pages are silent are stated beside the code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* IEEE binary16 codec (written here; the pages fix fp16 storage).      */
/* ------------------------------------------------------------------ */

double kvqo_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24);
  } else if (e == 31) {
    v = m ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + m), e - 25);
  }
  return sign ? -v : v;
}

float kvqo_half_to_float(uint16_t h) { return (float)kvqo_half_to_double(h); }

void kvqo_half_to_double_n(const uint16_t* h, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvqo_half_to_double(h[i]);
}

/* m >> s with round to nearest, ties to even (s >= 1). */
static uint32_t shift_rne(uint32_t m, int s) {
  if (s >= 26) return 0; /* m < 2^24 < half of 2^s */
  uint32_t q = m >> s;
  uint32_t rem = m & ((1u << s) - 1u);
  uint32_t half = 1u << (s - 1);
  if (rem > half || (rem == half && (q & 1u))) q++;
  return q;
}

/* fp32 -> fp16, round to nearest even; overflow gives infinity. */
uint16_t kvqo_float_to_half(float f) {
  uint32_t x;
  memcpy(&x, &f, sizeof x);
  uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7FFFFFFFu;
  if (ax >= 0x7F800000u) {
    if (ax > 0x7F800000u) return (uint16_t)(sign | 0x7E00u | ((ax >> 13) & 0x3FFu));
    return (uint16_t)(sign | 0x7C00u);
  }
  if (ax == 0) return sign;
  int e = (int)(ax >> 23) - 127;
  uint32_t m = ax & 0x7FFFFFu;
  if (e == -127) {
    e = -126; /* fp32 subnormal: no implicit bit */
  } else {
    m |= 0x800000u;
  }
  if (e >= -14) {
    uint32_t q = shift_rne(m, 13); /* 11 significant bits, maybe carried to 2^11 */
    int he = e + 15;
    if (q == 0x800u) {
      q = 0x400u;
      he++;
    }
    if (he >= 31) return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | (uint32_t)(he << 10) | (q & 0x3FFu));
  }
  /* half subnormal: units of 2^-24; a carry to 0x400 is the smallest normal */
  return (uint16_t)(sign | shift_rne(m, -e - 1));
}

void kvqo_float_to_half_n(const float* f, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = kvqo_float_to_half(f[i]);
}

/* ------------------------------------------------------------------ */
/* Quantizer for one group.                                            */
/* ------------------------------------------------------------------ */

/*
 * Quantize n fp16 values x[i*stride] with B = bits, L = 2^B - 1.  An entry
 * with excl[i*excl_stride] != 0 (a sparse outlier of its key vector) takes no
 * part: it does not enter the range and its code is 0.
 *
 * 1. mn, mx = min and max of the remaining entries (exact in fp32).  None
 *    remain: mn = mx = 0.  A minimum equal to zero is taken as +0 and a zero
 *    range as +0 (reading: the sign of a zero is not data).
 * 2. s32 = (mx - mn) / L: one fp32 subtraction, one fp32 division.
 * 3. zero point z = fp16(mn) (exact: mn is an input), scale s = fp16(s32),
 *    round to nearest even (reading: the pages only say "fp16").
 * 4. code = 0 when s == 0 or for an excluded entry; else
 *    clamp(rint((x - z) / s), 0, L) with z, s the stored fp16 values widened
 *    to fp32 (reading: codes are taken against the grid the decoder sees),
 *    a true fp32 division and rint rounding half to even.
 */
/*
 * Non-uniform levels (the nuqX datatype of the KVQuant review, "Proposed method", whose levels
 * come from a calibration the page does not give: here the caller's).  Reading: the zero point
 * and step stay those of steps 1-3; levels[0..L] are positions in steps, increasing from 0 to L;
 * a value takes the nearest level to y = (x - z) / s (fp32 quotient), found as the number of
 * decision thresholds t_j = fp32(levels[j] + levels[j+1]) * 0.5 (j < L) that y exceeds, so a value
 * on a threshold takes the lower level.  levels == NULL is the uniform quantizer of step 4.
 */
static uint8_t level_code(float y, const float* levels, int L) {
  uint8_t c = 0;
  for (int j = 0; j < L; ++j) {
    volatile float sum = levels[j] + levels[j + 1];
    volatile float t = sum * 0.5f;
    if (y > t) ++c;
  }
  return c;
}

void kvqo_quantize_group(const uint16_t* x, int64_t stride, int n, const uint8_t* excl,
                         int64_t excl_stride, int bits, uint16_t* z_out, uint16_t* s_out,
                         uint8_t* codes, int64_t code_stride, const float* levels) {
  const int L = (1 << bits) - 1;
  int any = 0;
  float mn = 0.0f, mx = 0.0f;
  for (int i = 0; i < n; ++i) {
    if (excl && excl[i * excl_stride]) continue;
    float v = kvqo_half_to_float(x[i * stride]);
    if (!any) {
      mn = v;
      mx = v;
      any = 1;
    } else {
      if (v < mn) mn = v;
      if (v > mx) mx = v;
    }
  }
  if (mn == 0.0f) mn = 0.0f; /* -0 -> +0 */
  volatile float range = mx - mn;
  if (!(range > 0.0f)) range = 0.0f;
  volatile float s32 = range / (float)L;
  uint16_t zb = kvqo_float_to_half(mn);
  uint16_t sb = kvqo_float_to_half(s32);
  *z_out = zb;
  *s_out = sb;
  float zf = kvqo_half_to_float(zb);
  float sf = kvqo_half_to_float(sb);
  for (int i = 0; i < n; ++i) {
    uint8_t code = 0;
    if (sf != 0.0f && !(excl && excl[i * excl_stride])) {
      float v = kvqo_half_to_float(x[i * stride]);
      volatile float d = v - zf;
      volatile float r = d / sf;
      if (levels) {
        code = level_code(r, levels, L);
      } else {
        float q = rintf(r);
        if (q < 0.0f) q = 0.0f;
        if (q > (float)L) q = (float)L;
        code = (uint8_t)q;
      }
    }
    codes[i * code_stride] = code;
  }
}

/* ------------------------------------------------------------------ */
/* Sparse outliers of one key vector.                                  */
/* ------------------------------------------------------------------ */

/*
 * Pick the nsp entries of x[0..D) with the largest |x|; ties go to the lower
 * channel.  idx/val are written sorted by channel; val holds the exact fp16.
 * (Per-vector dense-and-sparse quantization, KVQuant review.  Reading: the
 * count per vector is ceil(1% of D), chosen by the caller.)
 */
void kvqo_sparse_select(const uint16_t* x, int D, int nsp, uint8_t* idx, uint16_t* val) {
  uint8_t taken[1024];
  memset(taken, 0, sizeof taken);
  int chosen[64];
  for (int k = 0; k < nsp; ++k) {
    int best = -1;
    double bestv = -1.0;
    for (int c = 0; c < D; ++c) {
      if (taken[c]) continue;
      double a = fabs(kvqo_half_to_double(x[c]));
      if (a > bestv) {
        bestv = a;
        best = c;
      }
    }
    taken[best] = 1;
    chosen[k] = best;
  }
  /* sort ascending by channel (insertion sort, nsp is tiny) */
  for (int i = 1; i < nsp; ++i) {
    int v = chosen[i], j = i - 1;
    while (j >= 0 && chosen[j] > v) {
      chosen[j + 1] = chosen[j];
      --j;
    }
    chosen[j + 1] = v;
  }
  for (int k = 0; k < nsp; ++k) {
    idx[k] = (uint8_t)chosen[k];
    val[k] = x[chosen[k]];
  }
}

/* ------------------------------------------------------------------ */
/* Keys per channel, values per token, for one (batch, kv-head) unit.   */
/* ------------------------------------------------------------------ */

/*
 * Keys K[t][c] (fp16 bits), t in [0, Tq), Tq a multiple of G.  For every
 * group g of G consecutive tokens and every channel c, one (z, s) pair:
 * z[g*D + c], s[g*D + c].  codes[t*D + c] unpacked.  With nsp > 0 the sparse
 * entries of each token are chosen first and excluded from every group.
 */
int kvqo_quantize_keys(const uint16_t* K, int64_t Tq, int D, int G, int bits, int nsp,
                       uint8_t* codes, uint16_t* z, uint16_t* s, uint8_t* sp_idx, uint16_t* sp_val,
                       const float* levels) {
  if (Tq < 0 || G <= 0 || Tq % G || D <= 0 || D > 1024 || nsp < 0 || nsp > 64 || bits < 1 || bits > 8)
    return -1;
  uint8_t* excl = 0;
  if (nsp > 0) {
    excl = (uint8_t*)calloc((size_t)(Tq > 0 ? Tq : 1) * (size_t)D, 1);
    if (!excl) return -2;
    for (int64_t t = 0; t < Tq; ++t) {
      kvqo_sparse_select(K + t * D, D, nsp, sp_idx + t * nsp, sp_val + t * nsp);
      for (int k = 0; k < nsp; ++k) excl[t * D + sp_idx[t * nsp + k]] = 1;
    }
  }
  for (int64_t g = 0; g < Tq / G; ++g) {
    for (int c = 0; c < D; ++c) {
      const int64_t off = g * G * D + c;
      kvqo_quantize_group(K + off, D, G, excl ? excl + off : 0, D, bits, z + g * D + c, s + g * D + c,
                          codes + off, D, levels);
    }
  }
  free(excl);
  return 0;
}

/*
 * Values V[t][c], t in [0, Tq).  For every token t and every channel group of
 * G channels, one (z, s): z[t*(D/G) + j].  codes[t*D + c] unpacked.
 */
int kvqo_quantize_values(const uint16_t* V, int64_t Tq, int D, int G, int bits, uint8_t* codes,
                         uint16_t* z, uint16_t* s, const float* levels) {
  if (Tq < 0 || G <= 0 || D % G || bits < 1 || bits > 8) return -1;
  const int ng = D / G;
  for (int64_t t = 0; t < Tq; ++t)
    for (int j = 0; j < ng; ++j)
      kvqo_quantize_group(V + t * D + j * G, 1, G, 0, 0, bits, z + t * ng + j, s + t * ng + j,
                          codes + t * D + j * G, 1, levels);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Packing: little-endian bitstream.                                    */
/* ------------------------------------------------------------------ */

/*
 * Reading (the pages only say the codes are packed): the codes of one row
 * (the D channels of one token, for keys and for values) form a little-endian
 * bitstream; code i occupies bits [B*i, B*i + B) and word w holds bits
 * [32w, 32w + 32).  n*bits must be a multiple of 32.
 */
int kvqo_pack(const uint8_t* codes, int64_t n, int bits, uint32_t* words) {
  if ((n * bits) % 32) return -1;
  const int64_t nw = n * bits / 32;
  for (int64_t w = 0; w < nw; ++w) words[w] = 0;
  for (int64_t i = 0; i < n; ++i) {
    for (int b = 0; b < bits; ++b) {
      int64_t bit = i * bits + b;
      if ((codes[i] >> b) & 1u) words[bit / 32] |= 1u << (bit % 32);
    }
  }
  return 0;
}

int kvqo_unpack(const uint32_t* words, int64_t n, int bits, uint8_t* codes) {
  if ((n * bits) % 32) return -1;
  for (int64_t i = 0; i < n; ++i) {
    uint8_t v = 0;
    for (int b = 0; b < bits; ++b) {
      int64_t bit = i * bits + b;
      if ((words[bit / 32] >> (bit % 32)) & 1u) v |= (uint8_t)(1u << b);
    }
    codes[i] = v;
  }
  return 0;
}

/* ------------------------------------------------------------------ */
/* Rotary embedding (rotate-half), fp64.                               */
/* ------------------------------------------------------------------ */

/*
 * Rotate v[0..D) in place to absolute position t: for i < D/2,
 * theta_i = base^(-2i/D), (v_i, v_{i+D/2}) turns by the angle t*theta_i.
 * (Reading: the pages fix only the order, rotate after dequantizing.)
 */
void kvqo_rope(double* v, int D, double t, double base) {
  const int h = D / 2;
  for (int i = 0; i < h; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)D);
    double a = t * theta;
    double c = cos(a), s = sin(a);
    double x = v[i], y = v[i + h];
    v[i] = x * c - y * s;
    v[i + h] = y * c + x * s;
  }
}

/* ------------------------------------------------------------------ */
/* Dequantization of one token of a unit.                              */
/* ------------------------------------------------------------------ */

typedef struct {
  int D, G, nsp, rope;
  double rope_base;
  int64_t Tq, n_r;
  const uint8_t* kcodes;  /* [Tq][D] */
  const uint16_t* kz;     /* [Tq/G][D] */
  const uint16_t* ks;
  const uint8_t* sp_idx;  /* [Tq][nsp] */
  const uint16_t* sp_val;
  const uint8_t* vcodes;  /* [Tq][D] */
  const uint16_t* vz;     /* [Tq][D/G] */
  const uint16_t* vs;
  const uint16_t* wk;     /* [n_r][D] fp16 window keys (tokens n_s+Tq .. n_s+Tq+n_r) */
  const uint16_t* wv;
  int64_t n_s;            /* attention-sink tokens kept fp16 (tokens 0 .. n_s) */
  const uint16_t* sk;     /* [n_s][D] */
  const uint16_t* sv;
  const float* k_lev;     /* non-uniform levels of the key / value codes, or NULL (uniform) */
  const float* v_lev;
} kvqo_unit;

/* Token order: the n_s sink tokens, then the Tq quantized tokens, then the
   n_r window tokens; t is the absolute position, which is also the RoPE
   position. */

/* Key of token t as the decoder sees it: sink and window keys as stored,
   quantized keys z + s*code (exact in fp64) with their sparse entries
   restored, then RoPE at position t if asked. */
static void key_of(const kvqo_unit* u, int64_t t, double* k) {
  const int D = u->D;
  if (t < u->n_s) {
    for (int c = 0; c < D; ++c) k[c] = kvqo_half_to_double(u->sk[t * D + c]);
    if (u->rope) kvqo_rope(k, D, (double)t, u->rope_base);
    return;
  }
  const int64_t abs_t = t;
  t -= u->n_s;
  if (t < u->Tq) {
    const int64_t g = t / u->G;
    for (int c = 0; c < D; ++c)
      k[c] = kvqo_half_to_double(u->kz[g * D + c]) +
             kvqo_half_to_double(u->ks[g * D + c]) *
                 (u->k_lev ? (double)u->k_lev[u->kcodes[t * D + c]] : (double)u->kcodes[t * D + c]);
    for (int j = 0; j < u->nsp; ++j) k[u->sp_idx[t * u->nsp + j]] = kvqo_half_to_double(u->sp_val[t * u->nsp + j]);
  } else {
    for (int c = 0; c < D; ++c) k[c] = kvqo_half_to_double(u->wk[(t - u->Tq) * D + c]);
  }
  if (u->rope) kvqo_rope(k, D, (double)abs_t, u->rope_base);
}

static void value_of(const kvqo_unit* u, int64_t t, double* v) {
  const int D = u->D, ng = D / u->G;
  if (t < u->n_s) {
    for (int c = 0; c < D; ++c) v[c] = kvqo_half_to_double(u->sv[t * D + c]);
    return;
  }
  t -= u->n_s;
  if (t < u->Tq) {
    for (int c = 0; c < D; ++c) {
      const int j = c / u->G;
      v[c] = kvqo_half_to_double(u->vz[t * ng + j]) +
             kvqo_half_to_double(u->vs[t * ng + j]) *
                 (u->v_lev ? (double)u->v_lev[u->vcodes[t * D + c]] : (double)u->vcodes[t * D + c]);
    }
  } else {
    for (int c = 0; c < D; ++c) v[c] = kvqo_half_to_double(u->wv[(t - u->Tq) * D + c]);
  }
}

int kvqo_dequant_token(const kvqo_unit* u, int64_t t, double* k, double* v) {
  if (t < 0 || t >= u->n_s + u->Tq + u->n_r) return -1;
  if (k) key_of(u, t, k);
  if (v) value_of(u, t, v);
  return 0;
}

/* ------------------------------------------------------------------ */
/* Attention over a token range, and the merge of ranges.              */
/* ------------------------------------------------------------------ */

/*
 * Partial attention of Hg query heads q[h][c] (fp16) over tokens
 * [t_begin, t_end) of the unit, in fp64:
 *   sc_t = scale * sum_c q_c k_t,c;   m = max_t sc_t;
 *   l = sum_t exp(sc_t - m);          acc_c = sum_t exp(sc_t - m) v_t,c.
 * scale is the fp32 softmax scale widened to fp64.  Empty range: m = -inf,
 * l = 0, acc = 0.
 */
int kvqo_attention_partial(const kvqo_unit* u, const uint16_t* q, int Hg, float softmax_scale,
                           int64_t t_begin, int64_t t_end, double* m, double* l, double* acc) {
  const int D = u->D;
  const int64_t T = u->n_s + u->Tq + u->n_r;
  if (t_begin < 0 || t_end > T || t_begin > t_end || Hg <= 0) return -1;
  const int64_t n = t_end - t_begin;
  const double scale = (double)softmax_scale;
  double* qd = (double*)malloc(sizeof(double) * (size_t)Hg * D);
  double* sc = (double*)malloc(sizeof(double) * (size_t)Hg * (size_t)(n > 0 ? n : 1));
  double* k = (double*)malloc(sizeof(double) * D);
  if (!qd || !sc || !k) {
    free(qd); free(sc); free(k);
    return -2;
  }
  for (int i = 0; i < Hg * D; ++i) qd[i] = kvqo_half_to_double(q[i]);
  for (int h = 0; h < Hg; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0;
    for (int c = 0; c < D; ++c) acc[h * D + c] = 0.0;
  }
  for (int64_t i = 0; i < n; ++i) {
    key_of(u, t_begin + i, k);
    for (int h = 0; h < Hg; ++h) {
      double dot = 0.0;
      for (int c = 0; c < D; ++c) dot += qd[h * D + c] * k[c];
      sc[h * n + i] = scale * dot;
      if (sc[h * n + i] > m[h]) m[h] = sc[h * n + i];
    }
  }
  double* v = k; /* reuse */
  for (int64_t i = 0; i < n; ++i) {
    value_of(u, t_begin + i, v);
    for (int h = 0; h < Hg; ++h) {
      double p = exp(sc[h * n + i] - m[h]);
      l[h] += p;
      for (int c = 0; c < D; ++c) acc[h * D + c] += p * v[c];
    }
  }
  free(qd);
  free(sc);
  free(k);
  return 0;
}

/*
 * Merge S partials (m[s], l[s], acc[s][D]) of one head into the output
 * o_c = sum_s e^(m_s - M) acc_s,c / sum_s e^(m_s - M) l_s,  M = max_s m_s.
 */
int kvqo_combine(int S, int D, const double* m, const double* l, const double* acc, double* out) {
  double M = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (m[s] > M) M = m[s];
  if (!(M > -INFINITY)) return -1;
  double L = 0.0;
  for (int c = 0; c < D; ++c) out[c] = 0.0;
  for (int s = 0; s < S; ++s) {
    if (!(m[s] > -INFINITY)) continue;
    double w = exp(m[s] - M);
    L += w * l[s];
    for (int c = 0; c < D; ++c) out[c] += w * acc[s * D + c];
  }
  for (int c = 0; c < D; ++c) out[c] /= L;
  return 0;
}

/* Full decode attention of Hg heads over all T = n_s + Tq + n_r tokens. */
int kvqo_attention(const kvqo_unit* u, const uint16_t* q, int Hg, float softmax_scale, double* out) {
  const int D = u->D;
  double* m = (double*)malloc(sizeof(double) * Hg);
  double* l = (double*)malloc(sizeof(double) * Hg);
  double* acc = (double*)malloc(sizeof(double) * (size_t)Hg * D);
  if (!m || !l || !acc) {
    free(m); free(l); free(acc);
    return -2;
  }
  int rc = kvqo_attention_partial(u, q, Hg, softmax_scale, 0, u->n_s + u->Tq + u->n_r, m, l, acc);
  for (int h = 0; rc == 0 && h < Hg; ++h) rc = kvqo_combine(1, D, m + h, l + h, acc + h * D, out + h * D);
  free(m);
  free(l);
  free(acc);
  return rc;
}
