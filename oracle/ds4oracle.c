/*
 * ds4oracle.c -- CPU oracle for the routed MoE FFN of a DeepSeek-V4-Flash
 * layer. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never does.
 *
 * Plain scalar C, compiled -O2 -ffp-contract=off without fast-math, so every
 * float operation below is one IEEE-754 binary32 operation in the order
 * written (fmaf is the only fused operation, and it is written out).
 *
 * What it computes (sources, by page title and section):
 *  - Layer shape: "DeepSeek V4 Flash -- DFlash Integration", Model
 *    Architecture table: 256 routed experts top-6 + 1 shared, expert FFN
 *    2048, hidden 4096; first 3 layers hash routed (token ID -> expert
 *    table), the rest "top-k over learned router + optional bias".
 *  - Renormalisation of the kept experts' weights: same page, Execution
 *    Modes, --ds4-expert-top-k ("keeps the highest-ranked N routed experts
 *    and renormalizes their weights").
 *  - Router -> top-k -> gate/up -> weighted SwiGLU -> expert down, with the
 *    router returning "selected IDs and normalized weights" and F32 logits:
 *    "Baekpica/ds4 dfm Edition" README (two-bank batching notes).
 *  - Shared expert always on, Q8_0 for shared experts and router, 2-bit
 *    routed experts: DwarfStar README, Model Weights ("only the routed MoE
 *    experts are quantized ... shared experts, projections, routing are left
 *    untouched"), and the SExpQ8 file name.
 *  - Activations pre-quantised to int8 before the Q8_0 matmuls ("_preq"
 *    kernels): ds4-rocm fork README, __launch_bounds__ annotations list.
 *  - Final RMSNorm: DFlash Integration page, Forward Pass step 5.
 *  - Dense Q8_0 products beside the MoE (output head "OutQ8", attention
 *    projections) on pre-quantised int8 activations: ds4-rocm fork README,
 *    Performance optimizations (the matmul_q8_0_preq_* kernels) and the
 *    DwarfStar README, Model Weights (the OutQ8 model name).
 * The pages fix neither the bytes of the 2-bit format, nor the score
 * function, nor any float operation order. Those are fixed by the canonical
 * arithmetic spec (CAS) this file implements, stated at each function.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define FMT_F32 0
#define FMT_Q8_0 1
#define FMT_Q2S 2
#define FMT_Q4S 3
#define ROUTE_LEARNED 0
#define ROUTE_HASH 1

typedef struct {
  int32_t hidden, n_experts, top_k, ffn, n_shared;
  int32_t route, vocab;
  int32_t router_fmt, routed_fmt, shared_fmt;
  float route_scale;
  const void *router_w;       /* [E][H] router_fmt               (learned) */
  const float *router_bias;   /* [E]                             (learned) */
  const int32_t *hash_table;  /* [vocab][top_k]                  (hash)    */
  const uint8_t *gate, *up;   /* [E][F][H] routed_fmt                      */
  const uint8_t *down;        /* [E][H][F] routed_fmt                      */
  const uint8_t *sh_gate, *sh_up, *sh_down; /* [F][H],[F][H],[H][F]        */
} ora_layer;

/* ------------------------------------------------------------------------ */
/* Formats                                                                   */

/* IEEE binary16 -> binary32 (exact), by fields. */
float ora_half(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u, ex = (h >> 10) & 31u, man = h & 1023u;
  float v;
  if (ex == 0)
    v = ldexpf((float)man, -24); /* zero or subnormal: man * 2^-24 */
  else if (ex == 31)
    v = man ? NAN : INFINITY;
  else
    v = ldexpf((float)(man | 1024u), (int)ex - 25); /* (1024+man) * 2^(e-15-10) */
  return sign ? -v : v;
}

static inline uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q8_0 block, 34 bytes: fp16 d, int8 q[32]. w_i = d * q_i. */
void ora_q8_dequant(const uint8_t *blocks, int64_t n_blocks, float *out) {
  for (int64_t b = 0; b < n_blocks; b++) {
    const uint8_t *p = blocks + 34 * b;
    float d = ora_half(rd16(p));
    for (int i = 0; i < 32; i++) out[32 * b + i] = d * (float)(int8_t)p[2 + i];
  }
}

/* 2-bit superblock, 84 bytes: sm[16], qs[64], fp16 d, fp16 dmin.
 * Element i (0..255): group g = i/16, sc = sm[g] & 15, mn = sm[g] >> 4,
 * q = (qs[i/4] >> (2*(i%4))) & 3, w = d*sc*q - dmin*mn. Written out in
 * double so the value is exact (no rounding) for the pins. */
void ora_q2s_dequant_f64(const uint8_t *sbs, int64_t n_sb, double *out) {
  for (int64_t s = 0; s < n_sb; s++) {
    const uint8_t *p = sbs + 84 * s;
    double d = ora_half(rd16(p + 80)), dmin = ora_half(rd16(p + 82));
    for (int i = 0; i < 256; i++) {
      int g = i >> 4, sc = p[g] & 15, mn = p[g] >> 4;
      int q = (p[16 + (i >> 2)] >> (2 * (i & 3))) & 3;
      out[256 * s + i] = d * sc * q - dmin * mn;
    }
  }
}

/* Q4S superblock, 148 bytes: uint8 sm[16] | uint8 qs[128] | fp16 d | fp16
 * dmin (this library's own 4-bit layout: the pages name a 4-bit variant of
 * the routed experts, "q2 with the last 6 layers q4", without its bytes).
 * Group g = i / 16: sc = sm[g] & 15, mn = sm[g] >> 4;
 * q_i = (qs[i / 2] >> (4 * (i % 2))) & 15; w_i = d * sc * q_i - dmin * mn.
 * Evaluated in float64 (exact: every product of binary16 values and small
 * integers fits). */
void ora_q4s_dequant_f64(const uint8_t *sbs, int64_t n_sb, double *out) {
  for (int64_t s = 0; s < n_sb; s++) {
    const uint8_t *sb = sbs + 148 * s;
    double d = ora_half(rd16(sb + 144)), dmin = ora_half(rd16(sb + 146));
    for (int i = 0; i < 256; i++) {
      int g = i / 16, sc = sb[g] & 15, mn = sb[g] >> 4;
      int q = (sb[16 + i / 2] >> (4 * (i % 2))) & 15;
      out[256 * s + i] = d * sc * q - dmin * mn;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* CAS step 1: int8 quantisation per 32-block (activations x and SwiGLU h).  */
/*   amax = max|v|; dv = amax / 127; q = clamp(roundf(v / dv), +-127),       */
/*   q = 0 when dv == 0. gs[g] = sum of q over each 16-group (exact).        */

void ora_quantize(const float *v, int n, int8_t *q, float *dv, int16_t *gs) {
  for (int b = 0; b < n / 32; b++) {
    const float *x = v + 32 * b;
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
      float a = fabsf(x[i]);
      if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    dv[b] = d;
    for (int i = 0; i < 32; i++) {
      int qi = 0;
      if (d != 0.0f) {
        float r = roundf(x[i] / d);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        qi = (r == r) ? (int)r : 0;
      }
      q[32 * b + i] = (int8_t)qi;
    }
    for (int g = 0; g < 2; g++) {
      int s = 0;
      for (int i = 0; i < 16; i++) s += q[32 * b + 16 * g + i];
      gs[2 * b + g] = (int16_t)s;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* CAS step 2: exact integer block dots.                                     */

/* Q8_0: I = sum_i qw_i * qx_i over the 32 elements of one block. */
int32_t ora_q8_dot(const uint8_t *blk, const int8_t *xq) {
  int32_t s = 0;
  for (int i = 0; i < 32; i++) s += (int32_t)(int8_t)blk[2 + i] * (int32_t)xq[i];
  return s;
}

/* Q2S, 32-block j (0..7) of superblock sb; xq points at that block's 32
 * activations and gs at its two 16-group sums.
 *   A = sum over the two groups g of sc_g * sum_{i in g} q_i * qx_i
 *   B = sum over the two groups g of mn_g * gs_g                            */
void ora_q2s_dot(const uint8_t *sb, int j, const int8_t *xq, const int16_t *gs, int32_t *A,
                 int32_t *B) {
  int32_t a = 0, b = 0;
  for (int h = 0; h < 2; h++) {
    int g = 2 * j + h;
    int sc = sb[g] & 15, mn = sb[g] >> 4;
    int32_t dot = 0;
    for (int i = 0; i < 16; i++) {
      int e = 16 * g + i; /* element index within the superblock */
      int q = (sb[16 + (e >> 2)] >> (2 * (e & 3))) & 3;
      dot += q * (int32_t)xq[16 * h + i];
    }
    a += sc * dot;
    b += mn * (int32_t)gs[h];
  }
  *A = a;
  *B = b;
}

/* Q4S, 32-block j (0..7) of superblock sb: A and B as for Q2S, with 4-bit
 * codes. */
void ora_q4s_dot(const uint8_t *sb, int j, const int8_t *xq, const int16_t *gs, int32_t *A,
                 int32_t *B) {
  int32_t a = 0, b = 0;
  for (int h = 0; h < 2; h++) {
    int g = 2 * j + h;
    int sc = sb[g] & 15, mn = sb[g] >> 4;
    int32_t dot = 0;
    for (int i = 0; i < 16; i++) {
      int e = 16 * g + i; /* element index within the superblock */
      int q = (sb[16 + (e >> 1)] >> (4 * (e & 1))) & 15;
      dot += q * (int32_t)xq[16 * h + i];
    }
    a += sc * dot;
    b += mn * (int32_t)gs[h];
  }
  *A = a;
  *B = b;
}

/* ------------------------------------------------------------------------ */
/* CAS steps 3-4: block float terms and the row sum.                         */
/*   Q8_0: p_b = (d_b * dx_b) * (float)I_b                                   */
/*   Q2S : p_b = dx_b * fmaf(d_s, (float)A_b, -(dmin_s * (float)B_b))       */
/*   Q4S : the same, with A_b and B_b from the 4-bit codes                   */
/*   Row sum over nb blocks in S equal contiguous segments: each segment is  */
/*   acc = 0; acc = acc + p_b for increasing b; the segment sums are then    */
/*   added the same way in increasing segment order. Router rows: S = 8.     */
/*   Expert rows (routed and shared, gate/up/down): S = min(8, units), a     */
/*   unit being a superblock (Q2S) or a block (Q8_0) -- expert_segs().        */
/*   F32 rows (router only): each segment is acc = fmaf(w_i, x_i, acc) over  */
/*   its elements in increasing i.                                            */

static float row_q8(const uint8_t *row, int K, const int8_t *xq, const float *dx, int S) {
  int nb = K / 32, per = nb / S;
  float tot = 0.0f;
  for (int s = 0; s < S; s++) {
    float acc = 0.0f;
    for (int b = s * per; b < (s + 1) * per; b++) {
      const uint8_t *blk = row + 34 * b;
      float d = ora_half(rd16(blk));
      int32_t I = ora_q8_dot(blk, xq + 32 * b);
      float p = (d * dx[b]) * (float)I;
      acc = acc + p;
    }
    tot = tot + acc;
  }
  return tot;
}

static float row_q2s(const uint8_t *row, int K, const int8_t *xq, const float *dx,
                     const int16_t *gs, int S) {
  int nb = K / 32, per = nb / S;
  float tot = 0.0f;
  for (int s = 0; s < S; s++) {
    float acc = 0.0f;
    for (int b = s * per; b < (s + 1) * per; b++) {
      const uint8_t *sb = row + 84 * (b / 8);
      int32_t A, B;
      ora_q2s_dot(sb, b % 8, xq + 32 * b, gs + 2 * b, &A, &B);
      float d = ora_half(rd16(sb + 80)), dmin = ora_half(rd16(sb + 82));
      float m = dmin * (float)B;
      float p = dx[b] * fmaf(d, (float)A, -m);
      acc = acc + p;
    }
    tot = tot + acc;
  }
  return tot;
}

static float row_q4s(const uint8_t *row, int K, const int8_t *xq, const float *dx,
                     const int16_t *gs, int S) {
  int nb = K / 32, per = nb / S;
  float tot = 0.0f;
  for (int s = 0; s < S; s++) {
    float acc = 0.0f;
    for (int b = s * per; b < (s + 1) * per; b++) {
      const uint8_t *sb = row + 148 * (b / 8);
      int32_t A, B;
      ora_q4s_dot(sb, b % 8, xq + 32 * b, gs + 2 * b, &A, &B);
      float d = ora_half(rd16(sb + 144)), dmin = ora_half(rd16(sb + 146));
      float m = dmin * (float)B;
      float p = dx[b] * fmaf(d, (float)A, -m);
      acc = acc + p;
    }
    tot = tot + acc;
  }
  return tot;
}

static float row_f32(const float *w, int K, const float *x, int S) {
  int per = K / S;
  float tot = 0.0f;
  for (int s = 0; s < S; s++) {
    float acc = 0.0f;
    for (int i = s * per; i < (s + 1) * per; i++) acc = fmaf(w[i], x[i], acc);
    tot = tot + acc;
  }
  return tot;
}

static size_t row_bytes(int fmt, int K) {
  return fmt == FMT_Q2S ? (size_t)(K / 256) * 84 : fmt == FMT_Q4S ? (size_t)(K / 256) * 148
       : fmt == FMT_Q8_0 ? (size_t)(K / 32) * 34 : (size_t)K * 4;
}

/* One matrix row against one quantised activation vector. */
float ora_row(int fmt, const uint8_t *row, int K, const int8_t *xq, const float *dx,
              const int16_t *gs, int S) {
  return fmt == FMT_Q2S ? row_q2s(row, K, xq, dx, gs, S)
       : fmt == FMT_Q4S ? row_q4s(row, K, xq, dx, gs, S) : row_q8(row, K, xq, dx, S);
}

/* ------------------------------------------------------------------------ */
/* CAS step 5: exp, sigmoid, SiLU.                                           */
/* cas_exp(z): Cody & Waite argument reduction (Cody and Waite, Software     */
/* Manual for the Elementary Functions, 1980) with a degree-7 Taylor         */
/* polynomial. Constants are the binary32 roundings of:                      */
/*   log2(e); ln2 cut to 16 significant bits (so n*LN2_HI is exact for        */
/*   |n| <= 256) and the binary32 rounding of the remainder ln2 - LN2_HI;    */
/*   1/k! for k = 2..7.                                                       */

#define CAS_LOG2E 0x1.715476p+0f
#define CAS_LN2_HI 0x1.62e4p-1f
#define CAS_LN2_LO 0x1.7f7d1cp-20f
#define CAS_C2 0x1p-1f
#define CAS_C3 0x1.555556p-3f
#define CAS_C4 0x1.555556p-5f
#define CAS_C5 0x1.111112p-7f
#define CAS_C6 0x1.6c16c2p-10f
#define CAS_C7 0x1.a01a02p-13f

float ora_exp(float z) {
  if (z != z) return z;
  if (z < -87.0f) z = -87.0f;
  if (z > 88.0f) z = 88.0f;
  float n = rintf(z * CAS_LOG2E);          /* nearest integer, ties to even */
  float r = fmaf(-n, CAS_LN2_HI, z);
  r = fmaf(-n, CAS_LN2_LO, r);
  float p = CAS_C7;
  p = fmaf(p, r, CAS_C6);
  p = fmaf(p, r, CAS_C5);
  p = fmaf(p, r, CAS_C4);
  p = fmaf(p, r, CAS_C3);
  p = fmaf(p, r, CAS_C2);
  p = fmaf(p, r, 1.0f);
  p = fmaf(p, r, 1.0f);
  uint32_t bits = (uint32_t)((int)n + 127) << 23; /* 2^n, n in [-126, 127] */
  float s;
  memcpy(&s, &bits, 4);
  return p * s;
}

float ora_sigmoid(float z) { return 1.0f / (1.0f + ora_exp(-z)); }
float ora_silu(float g) { return g / (1.0f + ora_exp(-g)); }

/* ------------------------------------------------------------------------ */
/* CAS step 6: routing of one token.                                         */
/* learned: logit_e = router row e (S = 8); s_e = sigmoid(logit_e);          */
/*   key_e = s_e + bias_e; pick the k largest keys by repeated arg-max, ties */
/*   to the lower index, so ids come out in descending key order;           */
/*   sum = s_id0 + ... + s_id(k-1) in that order; w_j = (s_idj / sum)*scale.*/
/* hash: ids = table[token] in stored order; w_j = (1 / k) * scale.          */
/* Returns 0, or 1 when the token id is outside [0, vocab): ids are then -1  */
/* and weights 0.                                                             */

int ora_route_token(const ora_layer *L, const float *x, int32_t tok, int32_t *ids, float *w,
                    float *logits, float *keys) {
  int E = L->n_experts, k = L->top_k, H = L->hidden;
  if (L->route == ROUTE_HASH) {
    if (tok < 0 || tok >= L->vocab) {
      for (int j = 0; j < k; j++) ids[j] = -1, w[j] = 0.0f;
      return 1;
    }
    float wk = 1.0f / (float)k;
    for (int j = 0; j < k; j++) {
      ids[j] = L->hash_table[(int64_t)tok * k + j];
      w[j] = wk * L->route_scale;
    }
    return 0;
  }
  float *s = (float *)malloc(sizeof(float) * (size_t)E * 2);
  float *key = s + E;
  int8_t *xq = (int8_t *)malloc((size_t)H);
  float *dx = (float *)malloc(sizeof(float) * (size_t)(H / 32));
  int16_t *gs = (int16_t *)malloc(sizeof(int16_t) * (size_t)(H / 16));
  if (L->router_fmt != FMT_F32) ora_quantize(x, H, xq, dx, gs);
  for (int e = 0; e < E; e++) {
    float lg;
    if (L->router_fmt == FMT_F32)
      lg = row_f32((const float *)L->router_w + (int64_t)e * H, H, x, 8);
    else
      lg = ora_row(L->router_fmt, (const uint8_t *)L->router_w + (int64_t)e * row_bytes(L->router_fmt, H),
                   H, xq, dx, gs, 8);
    s[e] = ora_sigmoid(lg);
    key[e] = s[e] + L->router_bias[e];
    if (logits) logits[e] = lg;
    if (keys) keys[e] = key[e];
  }
  char *taken = (char *)calloc((size_t)E, 1);
  for (int j = 0; j < k; j++) {
    int best = -1;
    for (int e = 0; e < E; e++) {
      if (taken[e]) continue;
      if (best < 0 || key[e] > key[best]) best = e;
    }
    taken[best] = 1;
    ids[j] = best;
  }
  float sum = 0.0f;
  for (int j = 0; j < k; j++) sum = sum + s[ids[j]];
  for (int j = 0; j < k; j++) w[j] = (s[ids[j]] / sum) * L->route_scale;
  free(taken);
  free(gs);
  free(dx);
  free(xq);
  free(s);
  return 0;
}

/* ------------------------------------------------------------------------ */
/* One expert (e < E routed, e == E shared) for one token.                   */
/* g_j, u_j: gate/up rows j against (xq, dx, gs);                           */
/* h_j = silu(g_j) * u_j; (hq, dh, gsh) = CAS quantisation of h;              */
/* a_r: down row r against (hq, dh, gsh); every row in expert_segs segments. */
/* Any of g, u, h may be NULL.                                               */

typedef struct {
  const uint8_t *gate, *up, *down;
  int fmt;
} expert_w;

/* Row-sum segments of an expert row of K columns (CAS step 4). */
static int expert_segs(int fmt, int K) {
  int units = (fmt == FMT_Q2S || fmt == FMT_Q4S) ? K / 256 : K / 32;
  return units < 8 ? units : 8;
}

static expert_w expert_of(const ora_layer *L, int e) {
  expert_w x;
  int H = L->hidden, F = L->ffn;
  if (e == L->n_experts) {
    x.gate = L->sh_gate, x.up = L->sh_up, x.down = L->sh_down, x.fmt = L->shared_fmt;
  } else {
    size_t gu = (size_t)F * row_bytes(L->routed_fmt, H), dn = (size_t)H * row_bytes(L->routed_fmt, F);
    x.gate = L->gate + (size_t)e * gu, x.up = L->up + (size_t)e * gu, x.down = L->down + (size_t)e * dn;
    x.fmt = L->routed_fmt;
  }
  return x;
}

static void expert_gateup_rows(const ora_layer *L, int e, const int8_t *xq, const float *dx,
                               const int16_t *gs, int r0, int r1, float *g, float *u, float *h) {
  expert_w X = expert_of(L, e);
  int H = L->hidden;
  size_t rb = row_bytes(X.fmt, H);
  for (int j = r0; j < r1; j++) {
    float gj = ora_row(X.fmt, X.gate + (size_t)j * rb, H, xq, dx, gs, expert_segs(X.fmt, H));
    float uj = ora_row(X.fmt, X.up + (size_t)j * rb, H, xq, dx, gs, expert_segs(X.fmt, H));
    if (g) g[j] = gj;
    if (u) u[j] = uj;
    h[j] = ora_silu(gj) * uj;
  }
}

static void expert_down_rows(const ora_layer *L, int e, const int8_t *hq, const float *dh,
                             const int16_t *gsh, int r0, int r1, float *a) {
  expert_w X = expert_of(L, e);
  int F = L->ffn;
  size_t rb = row_bytes(X.fmt, F);
  for (int r = r0; r < r1; r++) a[r] = ora_row(X.fmt, X.down + (size_t)r * rb, F, hq, dh, gsh, expert_segs(X.fmt, F));
}

/* Full single expert for one token, exposing every intermediate. */
void ora_expert(const ora_layer *L, int e, const float *x, float *g, float *u, float *h,
                int8_t *hq, float *dh, int16_t *gsh, float *a) {
  int H = L->hidden, F = L->ffn;
  int8_t *xq = (int8_t *)malloc((size_t)H);
  float *dx = (float *)malloc(sizeof(float) * (size_t)(H / 32));
  int16_t *gs = (int16_t *)malloc(sizeof(int16_t) * (size_t)(H / 16));
  ora_quantize(x, H, xq, dx, gs);
  expert_gateup_rows(L, e, xq, dx, gs, 0, F, g, u, h);
  ora_quantize(h, F, hq, dh, gsh);
  expert_down_rows(L, e, hq, dh, gsh, 0, H, a);
  free(gs);
  free(dx);
  free(xq);
}

/* ------------------------------------------------------------------------ */
/* Whole layer: y[t] += MoE(x[t]) for T tokens.                              */
/* CAS step 7, per output element r of token t:                              */
/*   acc = 0; acc = acc + w_j * a_j[r] for j = 0..k-1 (descending key order);*/
/*   acc = acc + a_shared[r]; y[r] = y[r] + acc.                              */
/* A token whose hash id is out of range contributes nothing (y unchanged).  */
/* Work is split over nthreads threads by (token, expert slot, row chunk);  */
/* every element is computed by the same sequence of operations whatever the */
/* split. Returns the number of tokens with an out-of-range id.              */

typedef struct {
  const ora_layer *L;
  const float *x;
  const int32_t *tok;
  int T, ns; /* ns = expert slots per token = k + n_shared */
  float *y;
  int8_t *xq;
  float *dx;
  int16_t *gs;
  int32_t *ids;
  float *w;
  float *h;
  int8_t *hq;
  float *dh;
  int16_t *gsh;
  float *a;
  int *bad;
  int phase;
  int64_t n_items;
  int64_t next; /* shared work counter */
} fwd_ctx;

#define CHUNK 64

static void fwd_item(fwd_ctx *c, int64_t it) {
  const ora_layer *L = c->L;
  int H = L->hidden, F = L->ffn, k = L->top_k, ns = c->ns;
  if (c->phase == 0) { /* quantise + route token it */
    int t = (int)it;
    ora_quantize(c->x + (size_t)t * H, H, c->xq + (size_t)t * H, c->dx + (size_t)t * (H / 32),
                 c->gs + (size_t)t * (H / 16));
    c->bad[t] = ora_route_token(L, c->x + (size_t)t * H, c->tok ? c->tok[t] : 0, c->ids + (size_t)t * k,
                                c->w + (size_t)t * k, NULL, NULL);
  } else if (c->phase == 1) { /* gate/up rows of one (token, slot, chunk) */
    int nch = F / CHUNK;
    int t = (int)(it / ((int64_t)ns * nch)), rem = (int)(it % ((int64_t)ns * nch));
    int sl = rem / nch, ch = rem % nch;
    if (c->bad[t]) return;
    int e = sl < k ? c->ids[(size_t)t * k + sl] : L->n_experts;
    size_t ts = (size_t)t * ns + sl;
    expert_gateup_rows(L, e, c->xq + (size_t)t * H, c->dx + (size_t)t * (H / 32),
                       c->gs + (size_t)t * (H / 16), ch * CHUNK, (ch + 1) * CHUNK, NULL, NULL,
                       c->h + ts * F);
  } else if (c->phase == 2) { /* requantise h of one (token, slot) */
    int t = (int)(it / ns);
    if (c->bad[t]) return;
    size_t ts = (size_t)it;
    ora_quantize(c->h + ts * F, F, c->hq + ts * F, c->dh + ts * (F / 32), c->gsh + ts * (F / 16));
  } else if (c->phase == 3) { /* down rows of one (token, slot, chunk) */
    int nch = H / CHUNK;
    int t = (int)(it / ((int64_t)ns * nch)), rem = (int)(it % ((int64_t)ns * nch));
    int sl = rem / nch, ch = rem % nch;
    if (c->bad[t]) return;
    int e = sl < k ? c->ids[(size_t)t * k + sl] : L->n_experts;
    size_t ts = (size_t)t * ns + sl;
    expert_down_rows(L, e, c->hq + ts * F, c->dh + ts * (F / 32), c->gsh + ts * (F / 16), ch * CHUNK,
                     (ch + 1) * CHUNK, c->a + ts * H);
  } else { /* combine token it */
    int t = (int)it;
    if (c->bad[t]) return;
    float *y = c->y + (size_t)t * H;
    for (int r = 0; r < H; r++) {
      float acc = 0.0f;
      for (int j = 0; j < k; j++) acc = acc + c->w[(size_t)t * k + j] * c->a[((size_t)t * ns + j) * H + r];
      if (L->n_shared) acc = acc + c->a[((size_t)t * ns + k) * H + r];
      y[r] = y[r] + acc;
    }
  }
}

static void *fwd_worker(void *p) {
  fwd_ctx *c = (fwd_ctx *)p;
  for (;;) {
    int64_t it = __atomic_fetch_add(&c->next, 1, __ATOMIC_RELAXED);
    if (it >= c->n_items) break;
    fwd_item(c, it);
  }
  return NULL;
}

static void run_phase(fwd_ctx *c, int phase, int64_t n_items, int nthreads) {
  c->phase = phase;
  c->n_items = n_items;
  c->next = 0;
  if (nthreads <= 1) {
    fwd_worker(c);
    return;
  }
  pthread_t th[512];
  int n = nthreads > 512 ? 512 : nthreads, started = 0;
  for (int i = 0; i < n; i++) {
    if (pthread_create(&th[i], NULL, fwd_worker, c) != 0) break;
    started++;
  }
  fwd_worker(c);
  for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
}

int ora_forward(const ora_layer *L, const float *x, const int32_t *tok, int T, float *y,
                int32_t *ids_out, float *w_out, int nthreads) {
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  int H = L->hidden, F = L->ffn, k = L->top_k, ns = k + (L->n_shared ? 1 : 0);
  fwd_ctx c;
  memset(&c, 0, sizeof c);
  c.L = L, c.x = x, c.tok = tok, c.T = T, c.ns = ns, c.y = y;
  c.xq = (int8_t *)malloc((size_t)T * H);
  c.dx = (float *)malloc(sizeof(float) * (size_t)T * (H / 32));
  c.gs = (int16_t *)malloc(sizeof(int16_t) * (size_t)T * (H / 16));
  c.ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * k);
  c.w = (float *)malloc(sizeof(float) * (size_t)T * k);
  c.h = (float *)malloc(sizeof(float) * (size_t)T * ns * F);
  c.hq = (int8_t *)malloc((size_t)T * ns * F);
  c.dh = (float *)malloc(sizeof(float) * (size_t)T * ns * (F / 32));
  c.gsh = (int16_t *)malloc(sizeof(int16_t) * (size_t)T * ns * (F / 16));
  c.a = (float *)malloc(sizeof(float) * (size_t)T * ns * H);
  c.bad = (int *)calloc((size_t)T, sizeof(int));
  int ret = -1;
  if (c.xq && c.dx && c.gs && c.ids && c.w && c.h && c.hq && c.dh && c.gsh && c.a && c.bad) {
    run_phase(&c, 0, T, nthreads);
    run_phase(&c, 1, (int64_t)T * ns * (F / CHUNK), nthreads);
    run_phase(&c, 2, (int64_t)T * ns, nthreads);
    run_phase(&c, 3, (int64_t)T * ns * (H / CHUNK), nthreads);
    run_phase(&c, 4, T, nthreads);
    ret = 0;
    for (int t = 0; t < T; t++) ret += c.bad[t];
    if (ids_out) memcpy(ids_out, c.ids, sizeof(int32_t) * (size_t)T * k);
    if (w_out) memcpy(w_out, c.w, sizeof(float) * (size_t)T * k);
  }
  free(c.bad), free(c.a), free(c.gsh), free(c.dh), free(c.hq), free(c.h);
  free(c.w), free(c.ids), free(c.gs), free(c.dx), free(c.xq);
  return ret;
}

/* Routing only, for T tokens. Optional logits/keys are [T][E]. Returns the  */
/* number of tokens with an out-of-range hash id.                             */
int ora_route(const ora_layer *L, const float *x, const int32_t *tok, int T, int32_t *ids, float *w,
              float *logits, float *keys) {
  int bad = 0, E = L->n_experts, k = L->top_k;
  for (int t = 0; t < T; t++)
    bad += ora_route_token(L, x + (size_t)t * L->hidden, tok ? tok[t] : 0, ids + (size_t)t * k,
                           w + (size_t)t * k, logits ? logits + (size_t)t * E : NULL,
                           keys ? keys + (size_t)t * E : NULL);
  return bad;
}

/* ------------------------------------------------------------------------ */
/* CAS step 8: RMSNorm with unit gain, between stacked layers.               */
/*   ss = sum of v_i^2 in 32 equal contiguous segments (each a sequential     */
/*   fmaf chain; segment sums added in order); inv = 1 / sqrtf(ss / H + eps);*/
/*   out_i = v_i * inv.                                                       */

void ora_rmsnorm(const float *x, float *out, int T, int H, float eps) {
  int per = H / 32;
  for (int t = 0; t < T; t++) {
    const float *v = x + (size_t)t * H;
    float ss = 0.0f;
    for (int s = 0; s < 32; s++) {
      float acc = 0.0f;
      for (int i = s * per; i < (s + 1) * per; i++) acc = fmaf(v[i], v[i], acc);
      ss = ss + acc;
    }
    float inv = 1.0f / sqrtf(ss / (float)H + eps);
    for (int i = 0; i < H; i++) out[(size_t)t * H + i] = v[i] * inv;
  }
}

/* ------------------------------------------------------------------------ */
/* Dense Q8_0 product y = W x beside the MoE (output head, attention         */
/* projections): x quantised per 32-block (CAS step 1); each output row is   */
/* the CAS row sum (steps 2-4) of its Q8_0 blocks, with the row's blocks in  */
/* S = min(8, K/32) contiguous segments, as for an expert row.               */
/*   w [N][K] canonical Q8_0 rows, x [T][K] f32, y [T][N] f32 (overwritten). */
/* Rows are independent: nthreads > 1 splits them across threads, each row's */
/* arithmetic unchanged.                                                      */

typedef struct {
  const uint8_t *w;
  int N, K, T, nthreads, tid;
  const int8_t *xq;
  const float *dx;
  const int16_t *gs;
  float *y;
} dense_ctx;

static void *dense_worker(void *p) {
  dense_ctx *c = (dense_ctx *)p;
  const size_t rb = row_bytes(FMT_Q8_0, c->K);
  const int S = expert_segs(FMT_Q8_0, c->K);
  for (int n = c->tid; n < c->N; n += c->nthreads)
    for (int t = 0; t < c->T; t++)
      c->y[(size_t)t * c->N + n] = ora_row(FMT_Q8_0, c->w + (size_t)n * rb, c->K, c->xq + (size_t)t * c->K,
                                           c->dx + (size_t)t * (c->K / 32), c->gs + (size_t)t * (c->K / 16), S);
  return NULL;
}

void ora_dense_q8(const uint8_t *w, int N, int K, const float *x, int T, float *y, int nthreads) {
  int8_t *xq = (int8_t *)malloc((size_t)T * K);
  float *dx = (float *)malloc((size_t)T * (K / 32) * sizeof(float));
  int16_t *gs = (int16_t *)malloc((size_t)T * (K / 16) * sizeof(int16_t));
  for (int t = 0; t < T; t++)
    ora_quantize(x + (size_t)t * K, K, xq + (size_t)t * K, dx + (size_t)t * (K / 32), gs + (size_t)t * (K / 16));
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  pthread_t th[256];
  dense_ctx cs[256];
  for (int i = 0; i < nthreads; i++) {
    cs[i] = (dense_ctx){w, N, K, T, nthreads, i, xq, dx, gs, y};
    if (nthreads == 1) dense_worker(&cs[i]);
    else pthread_create(&th[i], NULL, dense_worker, &cs[i]);
  }
  if (nthreads > 1)
    for (int i = 0; i < nthreads; i++) pthread_join(th[i], NULL);
  free(xq);
  free(dx);
  free(gs);
}
