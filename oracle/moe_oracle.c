/*
 * Plain CPU oracle of one Mixture-of-Experts layer step with MLX-style affine
 * 4-bit routed and shared experts and an 8-bit router.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the product never calls it.
 *
 * Arithmetic is fp64 throughout, except where the method turns floating point
 * into an integer decision: the router ranks fp32 logits (the precision of the
 * kernels), and the quantiser decides its codes in fp32.  Loops are plain and
 * unblocked; OpenMP only splits independent output rows or tokens.
 *
 * Sources (page title, section):
 *   [P1] blog.hypho.cn "TurboFieldfare gemma4 out-of-core inference",
 *        sections "它省的不是模型大小，而是常驻内存" and "为什么不用 mmap？".
 *   [P2] sh.edu-sjtu.cn "TurboFieldfare：8GB Mac 本地跑 Gemma 4 26B-A4B 的
 *        Swift + Metal 运行时", section "TurboFieldfare 把内存压到约 2GB 的三件事".
 *   [P4] shilu.ai "drumih/turbo-fieldfare", overview table (row 权重),
 *        sections "推理引擎的工作原理" and "状态和范围".
 * The pages give the structure (128 routed experts, top-8, a dense shared
 * branch, affine 4-bit g64 weights, 8-bit router, per-layer LFU slot cache,
 * chunked prefill) but no formulas; the readings taken where they are silent
 * are stated at each function.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- scalars */

/* IEEE binary16 bit pattern -> value (the compiler's _Float16 conversion). */
static double half_to_double(uint16_t h) {
  _Float16 f;
  memcpy(&f, &h, sizeof f);
  return (double)f;
}

/* fp32 -> IEEE binary16, round to nearest even (the compiler's conversion). */
static uint16_t float_to_half(float x) {
  _Float16 f = (_Float16)x;
  uint16_t h;
  memcpy(&h, &f, sizeof h);
  return h;
}

/* bfloat16 bit pattern -> value: the upper half of an fp32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Threads the OpenMP loops below use from now on (timing at 1 core and at all
 * cores); returns the count in effect.  Changes no result: every loop that
 * is split writes disjoint outputs. */
int orc_set_threads(int n) {
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
}

double orc_half_to_double(uint16_t h) { return half_to_double(h); }
double orc_bf16_to_double(uint16_t b) { return bf16_to_double(b); }

/*
 * tanh form of GELU (Hendrycks & Gimpel, "Gaussian Error Linear Units", 2016):
 *   gelu(x) = 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 * The activation on the gate projection; the pages do not name it.
 */
double orc_gelu_tanh(double x) {
  const double pi = 3.14159265358979323846;
  const double c = sqrt(2.0 / pi);
  return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

/* ------------------------------------------------------- quantised tensors */

/* One canonical affine-quantised matrix [rows][cols]: element (r, c) is
 * scale[r][c / group] * code(r, c) + bias[r][c / group].  4-bit codes sit two
 * per byte, column 2i in the low nibble of byte i; 8-bit codes one per byte.
 * ([P4] overview table, row 权重: MLX affine 4-bit, group 64; 8-bit router.) */
typedef struct {
  const uint8_t* q;
  const uint16_t* scale;
  const uint16_t* bias;
} orc_qt;

static int code_at(const uint8_t* q, int64_t cols, int bits, int64_t r, int64_t c) {
  if (bits == 8) return q[r * cols + c];
  uint8_t byte = q[r * (cols / 2) + c / 2];
  return (c & 1) ? (byte >> 4) : (byte & 15);
}

/* Dequantise row r of a matrix with `cols` columns into out[cols] (exact in fp64). */
void orc_dequant_row(const orc_qt* t, int64_t cols, int bits, int group, int64_t r,
                     double* out) {
  int64_t ng = cols / group;
  for (int64_t c = 0; c < cols; ++c) {
    double s = half_to_double(t->scale[r * ng + c / group]);
    double b = half_to_double(t->bias[r * ng + c / group]);
    out[c] = s * (double)code_at(t->q, cols, bits, r, c) + b;
  }
}

/* Whole-matrix dequantise into out[rows][cols]. */
void orc_dequant(const orc_qt* t, int64_t rows, int64_t cols, int bits, int group,
                 double* out) {
  for (int64_t r = 0; r < rows; ++r) orc_dequant_row(t, cols, bits, group, r, out + r * cols);
}

/*
 * Affine quantiser (the install-time repack; not on the layer step).  The
 * pages say only "MLX affine, group 64"; the reading: per group, min and max
 * in fp32, scale = fp16((max - min) / levels), bias = fp16(min), and
 * code = clamp(round_half_even((w - bias) / scale), 0, levels) in fp32, code 0
 * where the fp16 scale is 0.  Returns 0, or -1 on bad arguments.
 */
int orc_quantise(const float* w, int64_t rows, int64_t cols, int bits, int group,
                 uint8_t* q, uint16_t* scale, uint16_t* bias) {
  if ((bits != 4 && bits != 8) || group <= 0 || cols % group != 0) return -1;
  const int levels = (1 << bits) - 1;
  const int64_t ng = cols / group;
  if (bits == 4) memset(q, 0, (size_t)(rows * cols / 2));
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t g = 0; g < ng; ++g) {
      const float* wg = w + r * cols + g * group;
      float mn = wg[0], mx = wg[0];
      for (int i = 1; i < group; ++i) {
        if (wg[i] < mn) mn = wg[i];
        if (wg[i] > mx) mx = wg[i];
      }
      uint16_t s16 = float_to_half((mx - mn) / (float)levels);
      uint16_t b16 = float_to_half(mn);
      scale[r * ng + g] = s16;
      bias[r * ng + g] = b16;
      float sf = (float)half_to_double(s16), bf = (float)half_to_double(b16);
      for (int i = 0; i < group; ++i) {
        int code = 0;
        if (sf != 0.0f) {
          float t = nearbyintf((wg[i] - bf) / sf);
          code = t < 0.0f ? 0 : (t > (float)levels ? levels : (int)t);
        }
        int64_t c = g * group + i;
        if (bits == 8) {
          q[r * cols + c] = (uint8_t)code;
        } else {
          q[r * (cols / 2) + c / 2] |= (uint8_t)((c & 1) ? (code << 4) : code);
        }
      }
    }
  }
  return 0;
}

/* y[rows] = W x with W dequantised row by row (plain dot products in fp64). */
static void qgemv(const orc_qt* t, int64_t rows, int64_t cols, int bits, int group,
                  const double* x, double* y) {
#pragma omp parallel
  {
    double* row = (double*)malloc(sizeof(double) * (size_t)cols);
#pragma omp for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
      orc_dequant_row(t, cols, bits, group, r, row);
      double acc = 0.0;
      for (int64_t c = 0; c < cols; ++c) acc += row[c] * x[c];
      y[r] = acc;
    }
    free(row);
  }
}

/* --------------------------------------------------------------- the layer */

typedef struct {
  int d_model, n_experts, d_expert, top_k, d_shared, group;
  orc_qt router;                 /* 8-bit [E][D] */
  const float* logit_bias;       /* [E] or NULL */
  orc_qt shared_gate, shared_up; /* 4-bit [S][D] */
  orc_qt shared_down;            /* 4-bit [D][S] */
  orc_qt gate, up;               /* 4-bit, experts stacked: [E][I][D] */
  orc_qt down;                   /* 4-bit, experts stacked: [E][D][I] */
} orc_layer;

/* Expert e's slice of a stacked [E][rows][cols] 4-bit tensor. */
static orc_qt expert_slice(const orc_qt* t, int64_t e, int64_t rows, int64_t cols, int group) {
  orc_qt s;
  s.q = t->q + e * rows * cols / 2;
  s.scale = t->scale + e * rows * (cols / group);
  s.bias = t->bias + e * rows * (cols / group);
  return s;
}

/*
 * Router ([P2] 三件事, first bullet; [P4] 推理引擎的工作原理: the router picks
 * 8 of 128 experts per token): logit_e = sum_c Wr[e][c] x[c] in fp64, rounded
 * to fp32, then + logit_bias[e] in fp32 when a bias is given.  The ranking
 * uses these fp32 values, the precision the kernels rank in.
 */
void orc_router_logits(const orc_layer* L, const double* x, float* logits) {
  double* l = (double*)malloc(sizeof(double) * (size_t)L->n_experts);
  qgemv(&L->router, L->n_experts, L->d_model, 8, L->group, x, l);
  for (int e = 0; e < L->n_experts; ++e) {
    float v = (float)l[e];
    if (L->logit_bias) v = v + L->logit_bias[e];
    logits[e] = v;
  }
  free(l);
}

/* Top-k: order all experts by (logit descending, index ascending) with an
 * insertion sort and take the first k.  Equal logits go to the lower index. */
void orc_topk(const float* logits, int E, int k, int32_t* ids) {
  int* order = (int*)malloc(sizeof(int) * (size_t)E);
  for (int e = 0; e < E; ++e) order[e] = e;
  for (int i = 1; i < E; ++i) {
    int cur = order[i], j = i - 1;
    while (j >= 0 && (logits[order[j]] < logits[cur] ||
                      (logits[order[j]] == logits[cur] && order[j] > cur))) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = cur;
  }
  for (int i = 0; i < k; ++i) ids[i] = order[i];
  free(order);
}

/* Routing weights: softmax over the k chosen logits, which equals the full
 * softmax renormalised over the chosen set.  w_i = exp(l_i - m) / sum_j exp(l_j - m). */
void orc_routing_weights(const float* logits, const int32_t* ids, int k, double* w) {
  double m = -INFINITY, z = 0.0;
  for (int i = 0; i < k; ++i) m = fmax(m, (double)logits[ids[i]]);
  for (int i = 0; i < k; ++i) z += exp((double)logits[ids[i]] - m);
  for (int i = 0; i < k; ++i) w[i] = exp((double)logits[ids[i]] - m) / z;
}

/* One gated FFN: out[D] = Wd (gelu_tanh(Wg x) * (Wu x)), Wg/Wu [F][D], Wd [D][F]. */
void orc_ffn(const orc_qt* wg, const orc_qt* wu, const orc_qt* wd, int D, int F, int group,
             const double* x, double* out) {
  double* g = (double*)malloc(sizeof(double) * (size_t)F);
  double* u = (double*)malloc(sizeof(double) * (size_t)F);
  qgemv(wg, F, D, 4, group, x, g);
  qgemv(wu, F, D, 4, group, x, u);
  for (int j = 0; j < F; ++j) g[j] = orc_gelu_tanh(g[j]) * u[j];
  qgemv(wd, D, F, 4, group, g, out);
  free(g);
  free(u);
}

/*
 * Parameter-free RMS normalisation of a layer input: u = x / sqrt(mean(x^2) + eps).
 * [P4] 状态和范围 lists normalisation kernels beside the MoE kernels, and the
 * pages' model (Gemma 4) normalises the residual stream before each FFN block;
 * its learned gain is a trained weight, so the reading takes unit gain.
 */
void orc_rms_normalise(const double* x, int D, double eps, double* u) {
  double ss = 0.0;
  for (int c = 0; c < D; ++c) ss += x[c] * x[c];
  const double r = 1.0 / sqrt(ss / (double)D + eps);
  for (int c = 0; c < D; ++c) u[c] = x[c] * r;
}

#define ORC_PRENORM 1
#define ORC_RMS_EPS 1e-6

/*
 * One MoE layer step for T tokens ([P2] 三件事, first bullet; [P4]
 * 推理引擎的工作原理): per token, route to k experts, run them and the shared
 * expert, and combine.  The pages say only that the two outputs are combined
 * ("合并"); the reading is y = sum_i w_i expert_i(x) + shared(x).
 *
 * x_bf16: [T][D] bf16 bits.  forced_ids: [T][k] or NULL; when given, those
 * experts are used and the weights are the softmax over their logits.
 * flags & ORC_PRENORM: the router and the experts read orc_rms_normalise(x)
 * (eps 1e-6) instead of x.
 * Outputs: ids [T][k], w [T][k], logits [T][E] (fp32), y [T][D] (fp64).
 */
int orc_moe_layer(const orc_layer* L, const uint16_t* x_bf16, int T, const int32_t* forced_ids,
                  int flags, int32_t* ids, double* w, float* logits, double* y) {
  const int D = L->d_model, E = L->n_experts, I = L->d_expert, k = L->top_k;
  const int S = L->d_shared, G = L->group;
  if (k < 1 || k > E || D % G || I % G || S % G) return -1;
  double* x = (double*)malloc(sizeof(double) * (size_t)D);
  double* e_out = (double*)malloc(sizeof(double) * (size_t)D);
  for (int t = 0; t < T; ++t) {
    for (int c = 0; c < D; ++c) x[c] = bf16_to_double(x_bf16[(int64_t)t * D + c]);
    if (flags & ORC_PRENORM) orc_rms_normalise(x, D, ORC_RMS_EPS, x);
    float* lt = logits + (int64_t)t * E;
    int32_t* it = ids + (int64_t)t * k;
    double* wt = w + (int64_t)t * k;
    double* yt = y + (int64_t)t * D;
    orc_router_logits(L, x, lt);
    if (forced_ids) {
      for (int i = 0; i < k; ++i) {
        it[i] = forced_ids[(int64_t)t * k + i];
        if (it[i] < 0 || it[i] >= E) { free(x); free(e_out); return -1; }
      }
    } else {
      orc_topk(lt, E, k, it);
    }
    orc_routing_weights(lt, it, k, wt);
    orc_ffn(&L->shared_gate, &L->shared_up, &L->shared_down, D, S, G, x, yt);
    for (int i = 0; i < k; ++i) {
      orc_qt g = expert_slice(&L->gate, it[i], I, D, G);
      orc_qt u = expert_slice(&L->up, it[i], I, D, G);
      orc_qt d = expert_slice(&L->down, it[i], D, I, G);
      orc_ffn(&g, &u, &d, D, I, G, x, e_out);
      for (int c = 0; c < D; ++c) yt[c] += wt[i] * e_out[c];
    }
  }
  free(x);
  free(e_out);
  return 0;
}

/* ------------------------------------------------------------- bucketing */

/*
 * Token-to-expert bucketing for a prefill chunk ([P2] 三件事, third bullet;
 * [P4] 推理引擎的工作原理: one fetched expert serves many rows).  The pages
 * give no algorithm; the reading is a stable grouping of the T*k assignments
 * by expert.  Assignment a = t*k + j.  counts[e] = #{a : ids[a] = e};
 * offsets[0..E] is the exclusive prefix sum; perm lists the assignments in
 * (expert, t, j) order.  Written as a direct scan per expert.
 */
int orc_bucket(const int32_t* ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
               int32_t* perm) {
  const int64_t n = (int64_t)T * k;
  for (int64_t a = 0; a < n; ++a)
    if (ids[a] < 0 || ids[a] >= E) return -1;
  int64_t pos = 0;
  for (int e = 0; e < E; ++e) {
    offsets[e] = (int32_t)pos;
    int32_t c = 0;
    for (int64_t a = 0; a < n; ++a) {
      if (ids[a] == e) {
        perm[pos++] = (int32_t)a;
        ++c;
      }
    }
    counts[e] = c;
  }
  offsets[E] = (int32_t)pos;
  return 0;
}

/* --------------------------------------------------------- LFU slot cache */

/*
 * One step of a layer's expert-slot cache ([P4] 推理引擎的工作原理: the CPU
 * plans the router's top-8 against the layer's 16-slot LFU cache and fills the
 * misses; [P1] 为什么不用 mmap？: pre-allocated slots, a bounded per-layer
 * cache).  The pages name the policy (LFU) but not its tie-breaks; the reading:
 *   1. every id already resident is a hit: count += 1, last_use = step;
 *   2. the misses, in ascending expert id, each take the lowest-index empty
 *      slot, or else evict, among the slots this step has not used, the one
 *      with the smallest count, then the oldest last_use, then the lowest
 *      index; the newcomer starts at count 1, last_use = step.
 * Counts are forgotten on eviction.  Slot state: expert (-1 = empty), count,
 * last_use.  Per id i: hit[i] (0/1), slot[i], evicted[i] (expert id or -1).
 * Returns the number of misses, or -1 if ids repeat, are out of range, or
 * k > n_slots.
 */
int orc_lfu_step(int n_slots, int32_t* slot_expert, int64_t* slot_count, int64_t* slot_last,
                 int64_t step, const int32_t* ids, int k, int n_experts, int32_t* hit,
                 int32_t* slot, int32_t* evicted) {
  if (k > n_slots || k < 0) return -1;
  for (int i = 0; i < k; ++i) {
    if (ids[i] < 0 || ids[i] >= n_experts) return -1;
    for (int j = 0; j < i; ++j)
      if (ids[j] == ids[i]) return -1;
  }
  char* used = (char*)calloc((size_t)n_slots, 1);
  for (int i = 0; i < k; ++i) {
    hit[i] = 0;
    slot[i] = -1;
    evicted[i] = -1;
    for (int s = 0; s < n_slots; ++s) {
      if (slot_expert[s] == ids[i]) {
        hit[i] = 1;
        slot[i] = s;
        slot_count[s] += 1;
        slot_last[s] = step;
        used[s] = 1;
      }
    }
  }
  int misses = 0;
  for (;;) {
    /* next miss in ascending expert id */
    int best = -1;
    for (int i = 0; i < k; ++i)
      if (!hit[i] && slot[i] < 0 && (best < 0 || ids[i] < ids[best])) best = i;
    if (best < 0) break;
    int chosen = -1;
    for (int s = 0; s < n_slots && chosen < 0; ++s)
      if (slot_expert[s] < 0) chosen = s;
    if (chosen < 0) {
      for (int s = 0; s < n_slots; ++s) {
        if (used[s]) continue;
        if (chosen < 0 || slot_count[s] < slot_count[chosen] ||
            (slot_count[s] == slot_count[chosen] && slot_last[s] < slot_last[chosen]))
          chosen = s;
      }
    }
    evicted[best] = slot_expert[chosen];
    slot_expert[chosen] = ids[best];
    slot_count[chosen] = 1;
    slot_last[chosen] = step;
    used[chosen] = 1;
    slot[best] = chosen;
    ++misses;
  }
  free(used);
  return misses;
}
