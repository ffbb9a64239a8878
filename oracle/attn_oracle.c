/*
 * Plain CPU oracle of one decode-attention step (the step before the
 * router), fp64 except where the method fixes a narrower type.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests and the benchmark's CPU-baseline
 * leg may load this library.  It shares no code, header, table or helper
 * with the CUDA path, and the product never calls it.
 *
 * Sources (page title, section):
 *   shilu.ai "drumih/turbo-fieldfare", section 推理引擎的工作原理: in every
 *     transformer layer the GPU computes attention and then the router from
 *     resident weights, and the router's top-8 ids drive the expert step
 *     (the router hand-off);
 *   the same page, section 状态和范围: 4-bit MLX affine attention weights;
 *     an FP16 KV store, bounded ring storage for the sliding-window layers and
 *     linear storage for the full-attention layers; exact split-K/V decode
 *     attention with distinct normalised K and V paths; RoPE and
 *     normalisation kernels.
 * The pages give no formulas or shapes.  Readings (each one plain):
 *   u = x / sqrt(mean(x^2) + 1e-6)                (unit-gain RMS pre-norm)
 *   q = Wq u, k = Wk u, v = Wv u                  (4-bit affine, dequantised)
 *   per head: q, k, v each divided by their RMS   (unit-gain, eps 1e-6)
 *   q, k rotated by RoPE at the token's position  (rotate-half pairs (i, i+d/2),
 *                                                  angle pos * theta^(-2i/d))
 *   k, v stored in fp16 (the FP16 KV store); the keys and values attended to
 *   are the stored fp16 values
 *   scores over the visible positions (all p <= pos for a full layer, the
 *   last `window` ones for a sliding layer), scaled by 1/sqrt(d);
 *   softmax; o_h = sum_p w_p v_p; y = Wo o (grouped-query: q head h reads
 *   kv head h / (Hq / Hkv)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  const uint8_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} ora_qt;

static double ora_half(uint16_t h) {
  _Float16 f;
  memcpy(&f, &h, sizeof f);
  return (double)f;
}

static uint16_t ora_to_half(double x) {
  _Float16 f = (_Float16)x; /* round to nearest even */
  uint16_t h;
  memcpy(&h, &f, sizeof h);
  return h;
}

static double ora_bf16(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* y[r] = sum_c (s q + b)[r][c] x[c] for a canonical 4-bit [rows][cols] tensor. */
static void ora_qgemv(const ora_qt* t, int64_t rows, int64_t cols, int group, const double* x,
                      double* y) {
  const int64_t ng = cols / group;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    double acc = 0.0;
    for (int64_t c = 0; c < cols; ++c) {
      const uint8_t byte = t->q[r * cols / 2 + c / 2];
      const int code = (c & 1) ? (byte >> 4) : (byte & 15);
      const double w = ora_half(t->scale[r * ng + c / group]) * code +
                       ora_half(t->bias[r * ng + c / group]);
      acc += w * x[c];
    }
    y[r] = acc;
  }
}

/* v / sqrt(mean(v^2) + eps), in place, over n values. */
void ora_rms(double* v, int n, double eps) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  const double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) v[i] *= r;
}

/* Rotary position embedding of one head vector of d values at `pos`: the
 * pairs (i, i + d/2) are rotated by the angle pos * theta^(-2i/d). */
void ora_rope(double* v, int d, int64_t pos, double theta) {
  const int h = d / 2;
  for (int i = 0; i < h; ++i) {
    const double ang = (double)pos * pow(theta, -2.0 * i / d);
    const double c = cos(ang), s = sin(ang);
    const double a = v[i], b = v[i + h];
    v[i] = a * c - b * s;
    v[i + h] = a * s + b * c;
  }
}

typedef struct {
  int d_model, n_heads, n_kv_heads, head_dim, group;
  ora_qt wq, wk, wv, wo; /* [Hq d][D], [Hkv d][D], [Hkv d][D], [D][Hq d] */
} ora_attn;

/*
 * One decode step of one layer for the token x (bf16 [D]) at position pos.
 * kcache / vcache: fp16 bits [Hkv][cap][d]; position p lives in slot p % cap
 * (a ring when cap == window, linear when cap > every position).  The step
 * writes its own k, v into slot pos % cap first, then attends to positions
 * max(0, pos - window + 1) .. pos (window <= 0: all of 0 .. pos).
 * y: [D] fp64, the attention block's output before the residual.
 * Returns 0, or -1 on bad arguments.
 */
int ora_attn_step(const ora_attn* A, const uint16_t* x_bf16, int64_t pos, int window, double theta,
                  uint16_t* kcache, uint16_t* vcache, int64_t cap, double* y) {
  const int D = A->d_model, Hq = A->n_heads, Hkv = A->n_kv_heads, d = A->head_dim;
  if (Hq % Hkv || d % 2 || cap < 1 || pos < 0 || (window > 0 && cap < window) ||
      (window <= 0 && pos >= cap))
    return -1;
  double* u = (double*)malloc(sizeof(double) * D);
  double* q = (double*)malloc(sizeof(double) * Hq * d);
  double* k = (double*)malloc(sizeof(double) * Hkv * d);
  double* v = (double*)malloc(sizeof(double) * Hkv * d);
  double* o = (double*)malloc(sizeof(double) * Hq * d);
  for (int c = 0; c < D; ++c) u[c] = ora_bf16(x_bf16[c]);
  ora_rms(u, D, 1e-6);
  ora_qgemv(&A->wq, (int64_t)Hq * d, D, A->group, u, q);
  ora_qgemv(&A->wk, (int64_t)Hkv * d, D, A->group, u, k);
  ora_qgemv(&A->wv, (int64_t)Hkv * d, D, A->group, u, v);
  for (int h = 0; h < Hq; ++h) {
    ora_rms(q + h * d, d, 1e-6);
    ora_rope(q + h * d, d, pos, theta);
  }
  const int64_t slot = pos % cap;
  for (int h = 0; h < Hkv; ++h) {
    ora_rms(k + h * d, d, 1e-6);
    ora_rope(k + h * d, d, pos, theta);
    ora_rms(v + h * d, d, 1e-6);
    for (int i = 0; i < d; ++i) {
      kcache[((int64_t)h * cap + slot) * d + i] = ora_to_half(k[h * d + i]);
      vcache[((int64_t)h * cap + slot) * d + i] = ora_to_half(v[h * d + i]);
    }
  }
  const int64_t first = (window > 0 && pos - window + 1 > 0) ? pos - window + 1 : 0;
  const int64_t n = pos - first + 1;
  double* s = (double*)malloc(sizeof(double) * n);
  const double scale = 1.0 / sqrt((double)d);
  for (int h = 0; h < Hq; ++h) {
    const int g = h / (Hq / Hkv);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      const int64_t sl = (first + j) % cap;
      double dot = 0.0;
      for (int i = 0; i < d; ++i) dot += q[h * d + i] * ora_half(kcache[((int64_t)g * cap + sl) * d + i]);
      s[j] = dot * scale;
      if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      s[j] = exp(s[j] - m);
      z += s[j];
    }
    for (int i = 0; i < d; ++i) o[h * d + i] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      const int64_t sl = (first + j) % cap;
      const double w = s[j] / z;
      for (int i = 0; i < d; ++i) o[h * d + i] += w * ora_half(vcache[((int64_t)g * cap + sl) * d + i]);
    }
  }
  ora_qgemv(&A->wo, D, (int64_t)Hq * d, A->group, o, y);
  free(u);
  free(q);
  free(k);
  free(v);
  free(o);
  free(s);
  return 0;
}
