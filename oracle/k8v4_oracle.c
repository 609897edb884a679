/*
 * k8v4 CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct restatement of what the hybrid k8v4 KV cache
 * computes, written from the "--kv k8v4: hybrid KV cache -- INT8 K +
 * Hadamard-rotated Q4_0 V (816 B/cell)" pull request (sections "What", "How" and
 * "Tests") and the "kv: --kv k8v4 streams with --kv-resident" pull request
 * (section "How": three byte runs per block).  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load this library; the product
 * path never does.  It shares no code with the CUDA library.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - K: symmetric int8, one fp32 scale per 128-lane half, s = absmax / 127
 *    (IEEE fp32 division), code = clamp(rint_even(x / s), -127, 127); s == 0 gives
 *    all-zero codes.  (Tests section: int8 codes round half to even.)
 *  - V rotation: y_i = RN_fp32( (sum_j H[i][j] x_j) / 16 ), H the Sylvester
 *    Hadamard matrix H[i][j] = (-1)^popcount(i & j), the sum taken EXACTLY (a
 *    multi-limb integer) and rounded once.  (What section: V is stored as rotated q4_0.)
 *  - V Q4_0 per 32-lane block: m = the element of largest |y| (first index on
 *    ties), d = fp16_RN(m / -8) (fp32 division, then one rounding to fp16),
 *    code = clamp(rint_even(y / (float)d) + 8, 0, 15); d == 0 gives codes 8.
 *    Byte j of a block holds code j in the low nibble and code j+16 in the high.
 *  - Page layout (per page of P cells, H KV heads): K codes [P][H][256] int8,
 *    K scales [P][H][2] fp32, V nibbles [P][H][8][16], V scales [P][H][8] fp16:
 *    408 B per (cell, head), 816 B per cell at H = 2.
 *  - int8/int8 comparison format: V quantised like K (unrotated), 528 B per
 *    (cell, head): K codes, K scales, V codes [P][H][256], V scales [P][H][2].
 *  - q4_0 format (both K and V rotated Q4_0, the "--kv q4_0" format the k8v4
 *    pull request compares against, 576 B/cell): K is rotated and quantised
 *    exactly like V; runs K nibbles [P][H][8][16], K scales [P][H][8] fp16,
 *    V nibbles, V scales: 288 B per (cell, head).  Attention scores use
 *    q . Khat with Khat = (H/16) Khat_rot; since H/16 is symmetric and
 *    orthogonal this is (H/16 q) . Khat_rot, which the oracle evaluates (q
 *    rotated once per row in fp64).
 *  - Attention (fp64): s_j = sm_scale * sum_i q_i Khat_ji over the visible cells,
 *    softmax with max subtraction, o = sum_j p_j Vhat_j, and for k8v4 the output
 *    is brought back from rotated space by out = (H/16) o.  Khat = (float)c * s
 *    (fp32 multiply), Vhat_rot = (q - 8) * d.  Query head h reads KV head h / 8.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off (no fast-math: every fp32 division,
 * multiply and rint is the IEEE-754 operation in round-to-nearest-even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 256
#define GQA 8

/* ------------------------------------------------------------------------- */
/* fp16 <-> fp32, from the IEEE-754 binary16 definition                       */
/* ------------------------------------------------------------------------- */

static int bitlen64(uint64_t v) {
  int n = 0;
  while (v) { ++n; v >>= 1; }
  return n;
}

/* Round a finite fp32 to the nearest binary16 (ties to even). */
uint16_t orc_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t ef = (u >> 23) & 0xFFu, fr = u & 0x7FFFFFu;
  if (ef == 0xFF) return (uint16_t)(sign | 0x7C00u | (fr ? 0x200u : 0u));
  uint64_t M;
  int E; /* value = M * 2^E */
  if (ef == 0) { M = fr; E = -149; } else { M = fr | 0x800000u; E = (int)ef - 150; }
  if (M == 0) return sign;
  int top = bitlen64(M) - 1 + E;           /* exponent of the leading bit */
  int lsb = top >= -14 ? top - 10 : -24;   /* exponent of the result's last bit */
  int shift = lsb - E;                     /* bits of M below the result's last bit */
  uint64_t q;
  if (shift <= 0) {
    q = M << (-shift);
  } else if (shift > 40) {
    q = 0;
  } else {
    q = M >> shift;
    uint64_t rem = M & ((1ull << shift) - 1), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (q & 1))) ++q;
  }
  if (q == 0) return sign;
  if (q >= 2048) { q >>= 1; ++lsb; }
  if (q < 1024) return (uint16_t)(sign | q);          /* subnormal (lsb == -24) */
  int e = lsb + 10;
  if (e > 15) return (uint16_t)(sign | 0x7C00u);      /* overflow -> inf */
  return (uint16_t)(sign | ((uint32_t)(e + 15) << 10) | (uint32_t)(q - 1024));
}

void orc_f32_to_f16_array(const float* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

float orc_f16_to_f32(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m + 1024), e - 25);
  return (float)(s ? -v : v);
}

/* ------------------------------------------------------------------------- */
/* exact Hadamard rotation                                                     */
/* ------------------------------------------------------------------------- */

/* A signed fixed-point integer in units of 2^-149 (the smallest fp32
 * subnormal), held as ACC_LIMBS limbs of 32 bits (stored in int64 so that 256
 * additions need no carry handling until the end). */
#define ACC_LIMBS 10

static int hadamard_sign(int i, int j) { return (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1; }

int orc_hadamard_entry(int i, int j) { return hadamard_sign(i, j); }

static void acc_add(int64_t* acc, int sgn, uint32_t M, int k) {
  /* acc += sgn * M * 2^k  (k >= 0, M < 2^24) */
  uint64_t v = (uint64_t)M << (k & 31);
  int idx = k >> 5;
  acc[idx] += sgn * (int64_t)(v & 0xFFFFFFFFull);
  acc[idx + 1] += sgn * (int64_t)(v >> 32);
}

static void acc_normalize(int64_t* acc) {
  for (int i = 0; i < ACC_LIMBS - 1; ++i) {
    int64_t c = acc[i] >> 32; /* floor division by 2^32 */
    acc[i] -= c * 4294967296LL;
    acc[i + 1] += c;
  }
}

static int acc_bit(const int64_t* acc, int pos) {
  if (pos < 0) return 0;
  return (int)((acc[pos >> 5] >> (pos & 31)) & 1);
}

static int acc_any_below(const int64_t* acc, int pos) {
  for (int p = 0; p < pos; ++p)
    if (acc_bit(acc, p)) return 1;
  return 0;
}

/* Round sign * (acc * 2^-149) * 2^-extra to the nearest fp32, ties to even.
 * acc holds the magnitude, normalised, non-negative. */
static float acc_round(const int64_t* acc, int negative, int extra) {
  int b = 0; /* bit length */
  for (int i = ACC_LIMBS - 1; i >= 0 && b == 0; --i)
    if (acc[i]) b = 32 * i + bitlen64((uint64_t)acc[i]);
  if (b == 0) return 0.0f; /* an exact zero sum is +0 */
  /* value = mag * 2^-(149 + extra); result lsb is 2^-149 at least, i.e. bit
   * position `extra` of mag, or 24 significant bits, whichever is coarser. */
  int shift = b - 24 > extra ? b - 24 : extra;
  uint64_t q = 0;
  for (int p = 23; p >= 0; --p) q = (q << 1) | (uint64_t)acc_bit(acc, shift + p);
  int half = acc_bit(acc, shift - 1);
  int sticky = acc_any_below(acc, shift - 1);
  if (half && (sticky || (q & 1))) ++q;
  if (q == (1ull << 24)) { q >>= 1; ++shift; }
  /* fp32 bits: exponent field = shift - extra + 1 when q carries the implicit
   * bit (q >= 2^23); subnormal when shift == extra and q < 2^23. */
  int64_t ebits = (int64_t)(shift - extra);
  uint32_t bits;
  if (ebits + 1 >= 255 && q >= (1ull << 23)) bits = 0x7F800000u;
  else bits = (uint32_t)((uint64_t)ebits << 23) + (uint32_t)q;
  if (negative) bits |= 0x80000000u;
  float f;
  memcpy(&f, &bits, 4);
  return f;
}

/* y_i = RN_fp32( (sum_j H[i][j] * x_j) / 16 ), the sum exact. */
void orc_hadamard_rotate(const float* x, float* y) {
  uint32_t M[D];
  int k[D], sg[D];
  for (int j = 0; j < D; ++j) {
    uint32_t u;
    memcpy(&u, &x[j], 4);
    uint32_t ef = (u >> 23) & 0xFFu, fr = u & 0x7FFFFFu;
    sg[j] = (u >> 31) ? -1 : 1;
    if (ef == 0) { M[j] = fr; k[j] = 0; }                   /* 2^-149 units */
    else { M[j] = fr | 0x800000u; k[j] = (int)ef - 1; }      /* E + 149 */
  }
  for (int i = 0; i < D; ++i) {
    int64_t acc[ACC_LIMBS];
    memset(acc, 0, sizeof acc);
    for (int j = 0; j < D; ++j)
      if (M[j]) acc_add(acc, sg[j] * hadamard_sign(i, j), M[j], k[j]);
    acc_normalize(acc);
    int neg = acc[ACC_LIMBS - 1] < 0;
    if (neg) {
      for (int l = 0; l < ACC_LIMBS; ++l) acc[l] = -acc[l];
      acc_normalize(acc);
    }
    y[i] = acc_round(acc, neg, 4); /* divide by 16 */
  }
}

/* ------------------------------------------------------------------------- */
/* quantisers                                                                  */
/* ------------------------------------------------------------------------- */

/* Symmetric int8 over n lanes: s = absmax / 127, c = clamp(rint(x / s)). */
void orc_quant_int8(const float* x, int n, int8_t* c, float* s_out) {
  float a = 0.0f;
  for (int i = 0; i < n; ++i)
    if (fabsf(x[i]) > a) a = fabsf(x[i]);
  float s = a / 127.0f;
  *s_out = s;
  for (int i = 0; i < n; ++i) {
    if (s == 0.0f) { c[i] = 0; continue; }
    float r = rintf(x[i] / s);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    c[i] = (int8_t)r;
  }
}

/* Q4_0 over one block of 32 rotated values. */
void orc_quant_q4_block(const float* y, uint8_t* nib, uint16_t* d_bits) {
  int im = 0;
  for (int j = 1; j < 32; ++j)
    if (fabsf(y[j]) > fabsf(y[im])) im = j;
  float m = y[im];
  uint16_t db = orc_f32_to_f16(m / -8.0f);
  float d = orc_f16_to_f32(db);
  *d_bits = db;
  uint8_t q[32];
  for (int j = 0; j < 32; ++j) {
    if (d == 0.0f) { q[j] = 8; continue; }
    float r = rintf(y[j] / d) + 8.0f;
    if (r < 0.0f) r = 0.0f;
    if (r > 15.0f) r = 15.0f;
    q[j] = (uint8_t)r;
  }
  for (int j = 0; j < 16; ++j) nib[j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

/* ------------------------------------------------------------------------- */
/* page layout                                                                 */
/* ------------------------------------------------------------------------- */

enum { ORC_FMT_INT8 = 1, ORC_FMT_Q4 = 2, ORC_FMT_K8V4 = 3 };

int64_t orc_bytes_per_cell_head(int fmt) {
  if (fmt == ORC_FMT_K8V4) return 256 + 8 + 128 + 16;
  if (fmt == ORC_FMT_INT8) return 256 + 8 + 256 + 8;
  if (fmt == ORC_FMT_Q4) return 128 + 16 + 128 + 16;
  return -1;
}

typedef struct {
  uint8_t* pages;
  int fmt, P, H;
  const int32_t* pt;
  int64_t max_pages;
} cache_t;

/* Byte addresses of the four runs of (sequence b, logical cell c, head g). */
typedef struct { uint8_t *kc, *ks, *vq, *vs; } cell_ptrs;

static cell_ptrs cell_at(const cache_t* C, int b, int64_t c, int g) {
  int64_t page = C->pt[(int64_t)b * C->max_pages + c / C->P];
  int64_t slot = c % C->P;
  int64_t P = C->P, H = C->H, r = slot * H + g;
  uint8_t* base = C->pages + page * P * H * orc_bytes_per_cell_head(C->fmt);
  cell_ptrs p;
  if (C->fmt == ORC_FMT_Q4) {
    p.kc = base + r * 128;
    p.ks = base + 128 * H * P + r * 16;
    p.vq = base + 144 * H * P + r * 128;
    p.vs = base + 272 * H * P + r * 16;
    return p;
  }
  p.kc = base + r * 256;
  p.ks = base + 256 * H * P + r * 8;
  if (C->fmt == ORC_FMT_K8V4) {
    p.vq = base + 264 * H * P + r * 128;
    p.vs = base + 392 * H * P + r * 16;
  } else {
    p.vq = base + 264 * H * P + r * 256;
    p.vs = base + 520 * H * P + r * 8;
  }
  return p;
}

/* rotate a row and store it as eight Q4_0 blocks (nibbles + fp16 scales) */
static void write_rot_q4(const float* x, uint8_t* nib, uint8_t* scales) {
  float y[D];
  orc_hadamard_rotate(x, y);
  uint16_t dv[8];
  for (int blk = 0; blk < 8; ++blk) orc_quant_q4_block(y + 32 * blk, nib + 16 * blk, &dv[blk]);
  memcpy(scales, dv, 16);
}

/* the rotated-space values (q - 8) d of eight stored Q4_0 blocks */
static void read_q4(const uint8_t* nib, const uint8_t* scales, float* out) {
  uint16_t dv[8];
  memcpy(dv, scales, 16);
  for (int blk = 0; blk < 8; ++blk) {
    float d = orc_f16_to_f32(dv[blk]);
    for (int j = 0; j < 16; ++j) {
      uint8_t byte = nib[16 * blk + j];
      out[32 * blk + j] = (float)((int)(byte & 15) - 8) * d;
      out[32 * blk + j + 16] = (float)((int)(byte >> 4) - 8) * d;
    }
  }
}

static void write_cell(const cache_t* C, int b, int64_t c, int g, const float* kx, const float* vx) {
  cell_ptrs p = cell_at(C, b, c, g);
  if (C->fmt == ORC_FMT_Q4) {
    write_rot_q4(kx, p.kc, p.ks);
    write_rot_q4(vx, p.vq, p.vs);
    return;
  }
  int8_t codes[D];
  float s[2];
  orc_quant_int8(kx, 128, codes, &s[0]);
  orc_quant_int8(kx + 128, 128, codes + 128, &s[1]);
  memcpy(p.kc, codes, D);
  memcpy(p.ks, s, 8);
  if (C->fmt == ORC_FMT_K8V4) {
    float y[D];
    orc_hadamard_rotate(vx, y);
    uint16_t dv[8];
    for (int blk = 0; blk < 8; ++blk) orc_quant_q4_block(y + 32 * blk, p.vq + 16 * blk, &dv[blk]);
    memcpy(p.vs, dv, 16);
  } else {
    orc_quant_int8(vx, 128, codes, &s[0]);
    orc_quant_int8(vx + 128, 128, codes + 128, &s[1]);
    memcpy(p.vq, codes, D);
    memcpy(p.vs, s, 8);
  }
}

/* Khat = (float)c * s (Khat_rot = (q - 8) * d for q4_0);  Vhat = (q - 8) * d
 * (k8v4 and q4_0, rotated space) or c * s (int8). */
static void read_cell(const cache_t* C, int b, int64_t c, int g, float* kh, float* vh) {
  cell_ptrs p = cell_at(C, b, c, g);
  if (C->fmt == ORC_FMT_Q4) {
    read_q4(p.kc, p.ks, kh);
    read_q4(p.vq, p.vs, vh);
    return;
  }
  float s[2];
  memcpy(s, p.ks, 8);
  const int8_t* kc = (const int8_t*)p.kc;
  for (int i = 0; i < D; ++i) kh[i] = (float)kc[i] * s[i / 128];
  if (C->fmt == ORC_FMT_K8V4) {
    uint16_t dv[8];
    memcpy(dv, p.vs, 16);
    for (int blk = 0; blk < 8; ++blk) {
      float d = orc_f16_to_f32(dv[blk]);
      for (int j = 0; j < 16; ++j) {
        uint8_t byte = p.vq[16 * blk + j];
        vh[32 * blk + j] = (float)((int)(byte & 15) - 8) * d;
        vh[32 * blk + j + 16] = (float)((int)(byte >> 4) - 8) * d;
      }
    }
  } else {
    float sv[2];
    memcpy(sv, p.vs, 8);
    const int8_t* vc = (const int8_t*)p.vq;
    for (int i = 0; i < D; ++i) vh[i] = (float)vc[i] * sv[i / 128];
  }
}

/* ------------------------------------------------------------------------- */
/* a tiny parallel-for over independent items (rows or cells)                  */
/* ------------------------------------------------------------------------- */

typedef void (*item_fn)(void* ctx, int64_t i);
typedef struct { item_fn fn; void* ctx; int64_t n, lo, hi; } span_t;

static void* run_span(void* a) {
  span_t* s = (span_t*)a;
  for (int64_t i = s->lo; i < s->hi; ++i) s->fn(s->ctx, i);
  return NULL;
}

static void parallel_for(int n_threads, int64_t n, item_fn fn, void* ctx) {
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 256) n_threads = 256;
  if (n_threads == 1 || n < 2) {
    for (int64_t i = 0; i < n; ++i) fn(ctx, i);
    return;
  }
  pthread_t th[256];
  span_t sp[256];
  int made[256];
  for (int t = 0; t < n_threads; ++t) {
    sp[t].fn = fn; sp[t].ctx = ctx; sp[t].n = n;
    sp[t].lo = n * t / n_threads; sp[t].hi = n * (t + 1) / n_threads;
    made[t] = pthread_create(&th[t], NULL, run_span, &sp[t]) == 0;
    if (!made[t]) run_span(&sp[t]);
  }
  for (int t = 0; t < n_threads; ++t)
    if (made[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------- */
/* append                                                                      */
/* ------------------------------------------------------------------------- */

typedef struct {
  cache_t C;
  const int64_t* pos;
  int n_tok;
  const float *k, *v;
} append_ctx;

static void append_item(void* vctx, int64_t it) {
  append_ctx* a = (append_ctx*)vctx;
  int b = (int)(it / a->n_tok), t = (int)(it % a->n_tok);
  for (int g = 0; g < a->C.H; ++g) {
    int64_t off = ((it * a->C.H) + g) * D;
    write_cell(&a->C, b, a->pos[b] + t, g, a->k + off, a->v + off);
  }
}

/* k, v: [n_seqs][n_tok][H][256] float32; cell pos[b] + t of sequence b. */
int orc_append(uint8_t* pages, int fmt, int P, int H, const int32_t* pt, int64_t max_pages, int n_seqs,
               const int64_t* pos, int n_tok, const float* k, const float* v, int n_threads) {
  if (orc_bytes_per_cell_head(fmt) < 0) return -1;
  append_ctx a = {{pages, fmt, P, H, pt, max_pages}, pos, n_tok, k, v};
  parallel_for(n_threads, (int64_t)n_seqs * n_tok, append_item, &a);
  return 0;
}

/* Dequantise cells [start, start+n) of sequence b: Khat, Vhat (rotated space for
 * k8v4), and, when v_out is given, Vhat brought back by the exact rotation. */
int orc_dequant(const uint8_t* pages, int fmt, int P, int H, const int32_t* pt, int64_t max_pages, int b,
                int64_t start, int64_t n, float* k_out, float* v_rot_out, float* v_out) {
  cache_t C = {(uint8_t*)pages, fmt, P, H, pt, max_pages};
  for (int64_t c = 0; c < n; ++c)
    for (int g = 0; g < H; ++g) {
      int64_t off = (c * H + g) * D;
      read_cell(&C, b, start + c, g, k_out + off, v_rot_out + off);
      if (fmt == ORC_FMT_Q4) {             /* K back in the original basis */
        float kr[D];
        memcpy(kr, k_out + off, sizeof kr);
        orc_hadamard_rotate(kr, k_out + off);
      }
      if (v_out) {
        if (fmt != ORC_FMT_INT8) orc_hadamard_rotate(v_rot_out + off, v_out + off);
        else memcpy(v_out + off, v_rot_out + off, D * sizeof(float));
      }
    }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* attention (fp64)                                                            */
/* ------------------------------------------------------------------------- */

typedef struct {
  cache_t C;
  const int32_t *row_seq, *row_head, *row_vis;
  const float* q;
  double sm_scale;
  double* out;
  int rotate_back;
} attn_ctx;

/* Attention of one query row over cells [lo, hi) of sequence b, KV head g:
 * the scores s_j = (q . Khat_j) sm_scale, their maximum m and the sum l of
 * exp(s_j - m); acc = sum_j exp(s_j - m) Vhat_rot_j, divided by l when `norm`
 * (0 for an empty range); o = (H/16) acc when `rotate_back`, else acc. */
static void range_attention(const cache_t* C, int b, int g, int lo, int hi, const float* q32, double sm_scale,
                            int norm, int rotate_back, double* o, double* m_out, double* l_out) {
  double q[D];
  if (C->fmt == ORC_FMT_Q4) {            /* (H/16) q: scores against Khat_rot */
    for (int i = 0; i < D; ++i) {
      double s = 0.0;
      for (int j = 0; j < D; ++j) s += hadamard_sign(i, j) * (double)q32[j];
      q[i] = s / 16.0;
    }
  } else {
    for (int i = 0; i < D; ++i) q[i] = (double)q32[i];
  }
  int n = hi > lo ? hi - lo : 0;
  double* sc = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
  double acc[D];
  float kh[D], vh[D];
  memset(acc, 0, sizeof acc);
  double mx = -INFINITY;
  for (int j = 0; j < n; ++j) {
    read_cell(C, b, lo + j, g, kh, vh);
    double dot = 0.0;
    for (int i = 0; i < D; ++i) dot += q[i] * (double)kh[i];
    sc[j] = dot * sm_scale;
    if (sc[j] > mx) mx = sc[j];
  }
  double l = 0.0;
  for (int j = 0; j < n; ++j) {
    double p = exp(sc[j] - mx);
    l += p;
    read_cell(C, b, lo + j, g, kh, vh);
    for (int i = 0; i < D; ++i) acc[i] += p * (double)vh[i];
  }
  if (norm)
    for (int i = 0; i < D; ++i) acc[i] = n > 0 ? acc[i] / l : 0.0;
  if (rotate_back) {
    for (int i = 0; i < D; ++i) {
      double s = 0.0;
      for (int j = 0; j < D; ++j) s += hadamard_sign(i, j) * acc[j];
      o[i] = s / 16.0;
    }
  } else {
    memcpy(o, acc, sizeof acc);
  }
  *m_out = mx;
  *l_out = l;
  free(sc);
}

static void attn_row(void* vctx, int64_t r) {
  attn_ctx* a = (attn_ctx*)vctx;
  int b = a->row_seq[r], h = a->row_head[r], n = a->row_vis[r], g = h / GQA;
  double m, l;
  range_attention(&a->C, b, g, 0, n, a->q + r * D, a->sm_scale, 1, a->rotate_back, a->out + r * D, &m, &l);
}

/* Partial attention over a cell range (the cell-range split of one decode
 * across GPUs): for row r, cells [row_lo[r], row_hi[r]) of its sequence,
 *   m = max_j s_j,  l = sum_j exp(s_j - m),  o = (H/16) sum_j exp(s_j - m) Vhat_rot_j
 * (natural exponent; o un-rotated and unnormalised); an empty range gives
 * m = -inf, l = 0, o = 0.  Merging ranges: out = sum_r e^(m_r - M) o_r /
 * sum_r e^(m_r - M) l_r. */
typedef struct {
  cache_t C;
  const int32_t *row_seq, *row_head, *row_lo, *row_hi;
  const float* q;
  double sm_scale;
  double *o, *m, *l;
} part_ctx;

static void part_row(void* vctx, int64_t r) {
  part_ctx* a = (part_ctx*)vctx;
  const int b = a->row_seq[r], h = a->row_head[r];
  const int kv = h / GQA;                 /* query head h reads KV head h / 8 */
  range_attention(&a->C, b, kv, a->row_lo[r], a->row_hi[r], a->q + r * D, a->sm_scale, 0,
                  a->C.fmt != ORC_FMT_INT8, a->o + r * D, a->m + r, a->l + r);
}

int orc_attention_partial(const uint8_t* pages, int fmt, int P, int H, const int32_t* pt, int64_t max_pages,
                          int64_t n_rows, const int32_t* row_seq, const int32_t* row_head, const int32_t* row_lo,
                          const int32_t* row_hi, const float* q, double sm_scale, double* o, double* m, double* l,
                          int n_threads) {
  part_ctx a = {{(uint8_t*)pages, fmt, P, H, pt, max_pages}, row_seq, row_head, row_lo, row_hi, q, sm_scale, o, m, l};
  parallel_for(n_threads, n_rows, part_row, &a);
  return 0;
}

/* One output row per (sequence, head, visible count): out[r] = softmax-weighted
 * mean of the visible cells' V, in the original (un-rotated) basis.
 * rotate_back = 0 keeps the k8v4 result in rotated space (used by checks). */
int orc_attention(const uint8_t* pages, int fmt, int P, int H, const int32_t* pt, int64_t max_pages,
                  int64_t n_rows, const int32_t* row_seq, const int32_t* row_head, const int32_t* row_vis,
                  const float* q, double sm_scale, double* out, int rotate_back, int n_threads) {
  attn_ctx a = {{(uint8_t*)pages, fmt, P, H, pt, max_pages}, row_seq, row_head, row_vis, q, sm_scale, out,
                rotate_back && fmt != ORC_FMT_INT8};
  parallel_for(n_threads, n_rows, attn_row, &a);
  return 0;
}
