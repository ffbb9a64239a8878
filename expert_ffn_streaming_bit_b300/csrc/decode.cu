// Persistent decode kernel: one token through one or more MoE layers.
//
// One CTA per SM (cooperative launch).  Warp 8 of each CTA is a producer: one
// lane walks the CTA's list of weight "stages" and brings each into a ring of
// shared-memory slots with bulk async copies (the copy engine, completion on
// an mbarrier).  Warps 0-7 consume the stages in the same order.
//
// Per layer l the CTA's stages are
//   BS  its share of the shared expert's gate/up row pairs   (weights known ahead)
//   BR  its share of the k routed experts' gate/up pairs     (needs ids(l))
//   C   its share of output rows: for each row the k routed down rows, the
//       shared down row and, when a next layer follows, the next router's
//       column block                                          (needs ids(l))
// and the data dependences are met with two grid barriers per layer:
//   after BS+BR: h = gelu(W_gate u) * (W_up u) complete for all k+1 branches;
//   after C: x_{l+1} and the next router's logits complete.  Each CTA adds
//   its rows' partial logits into one accumulator per expert as 64-bit fixed
//   point (integer addition, so the sum does not depend on arrival order);
//   after the barrier every CTA reads the E sums, and takes the top k and the
//   renormalised softmax itself (identical in every CTA).
// The producer runs ahead across barriers wherever the weights are already
// known, and prefetches into L2 the routed rows it will stream once the ids
// arrive, so HBM keeps working while the grid synchronises.  Every wait is
// bounded in time; a wait that runs out sets the status word and the CTA
// drains its in-flight copies and exits.
//
// Arithmetic (shilu.ai "drumih/turbo-fieldfare", overview table row 权重 and
// section 推理引擎的工作原理; sh.edu-sjtu.cn article, section 三件事):
//   router: logit_e = r * sum_c (s q + b) x_c in fp32, + bias_e (r = the
//           pre-norm scale or 1); top-k by (logit desc, index asc); w = softmax
//           over the chosen logits;
//   expert: h_j = gelu_tanh(g_j) u_j with g = W_gate u, u = W_up u;
//           e = W_down h; y = sum_i w_i e_i + shared(u); optional residual.
// Expert dot products are integer-exact: the activation vector is held as
// int16 X = rint(v / sigma) (sigma = max|v| / 32767 over the whole of x, or
// over each 32-value chunk of h), the 4-bit codes as bytes, and a 2-way
// integer dot product accumulates sum q X exactly in int32 per 32-column
// chunk; the chunk contributes s * sum(q X) + bias * sum(X), times sigma.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"
#include "qdot.cuh"

namespace moe {

namespace {

struct Part {
  int sh_lo, sh_hi;  // shared gate/up pairs
  int rt_lo, rt_hi;  // routed pairs, flattened k*I + j
  int c_lo, c_hi;    // output rows
};

__device__ __forceinline__ int split_at(int n, int c, int G) {
  return static_cast<int>(static_cast<int64_t>(n) * c / G);
}

enum : int { ST_R = 0, ST_BS = 1, ST_BR = 2, ST_C = 3 };

struct Stage {
  int kind;
  int a;  // first pair / first row
  int n;  // pairs / rows
  int k;  // routed slot (ST_BR)
};

// misc[] slots in shared memory
enum : int {
  M_IDS = 0,   // [32] ids of the current layer
  M_WTS = 32,  // [32] weights (float bits)
  M_ABORT = 64,
  M_LAST = 65,
  M_GEN = 66,
  M_ISSUED = 67,
  M_TARGET = 70,  // [2] next grid-barrier target (64-bit; 0 before the first barrier)
  M_RED = 72,  // [8] per-warp reduction scratch
  M_RED2 = 80, // [8] second per-warp reduction scratch
  M_COUNT = 136
};

struct Ctx {
  const DecodeParams* p;
  uint8_t* smem;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* ids_ready;
  volatile int* misc;
  Part part;
  int G;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  // round to nearest even; NaN stays a quiet NaN
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

__device__ __forceinline__ float gelu_tanh(float x) {
  // tanh form of GELU (Hendrycks & Gimpel 2016)
  const float c = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * x * (1.f + tanhf(c * (x + 0.044715f * x * x * x)));
}

__device__ __forceinline__ void csync() { named_sync(1, kConsumers); }

struct LayerPlan {
  int n_r, n_bs, n_br, n_c;  // stage counts
  int rc;                    // rows per C stage (balanced)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ LayerPlan layer_plan(const DecodeParams& p, const Part& pt, int li) {
  LayerPlan lp;
  lp.n_r = (li == 0 && (p.phases & PH_ROUTER) && pt.c_hi > pt.c_lo) ? 1 : 0;
  lp.n_bs = (p.phases & PH_BSHARED) ? ceil_div(pt.sh_hi - pt.sh_lo, kPairsPerStage) : 0;
  // routed pairs (flattened k*I + j): near-equal stages, which may span two experts
  lp.n_br = (p.phases & PH_BROUTED) ? ceil_div(pt.rt_hi - pt.rt_lo, kPairsPerStage) : 0;
  const int rows = pt.c_hi - pt.c_lo;
  lp.n_c = (p.phases & PH_C) ? ceil_div(rows, p.rc_max) : 0;
  lp.rc = lp.n_c ? ceil_div(rows, lp.n_c) : 0;
  return lp;
}

// The s-th stage of a layer (R, BS, BR, C in that order).
__device__ Stage stage_at(const DecodeParams& p, const Part& pt, const LayerPlan& lp, int s) {
  Stage st{0, 0, 0, 0};
  if (s < lp.n_r) {
    st.kind = ST_R;
    st.a = pt.c_lo;
    st.n = pt.c_hi - pt.c_lo;
    return st;
  }
  s -= lp.n_r;
  if (s < lp.n_bs) {
    st.kind = ST_BS;
    st.a = pt.sh_lo + s * kPairsPerStage;
    st.n = min(kPairsPerStage, pt.sh_hi - st.a);
    return st;
  }
  s -= lp.n_bs;
  if (s < lp.n_br) {
    const int len = pt.rt_hi - pt.rt_lo;
    st.kind = ST_BR;
    st.a = pt.rt_lo + static_cast<int>(static_cast<int64_t>(len) * s / lp.n_br);
    st.n = pt.rt_lo + static_cast<int>(static_cast<int64_t>(len) * (s + 1) / lp.n_br) - st.a;
    st.k = st.a / p.I;
    return st;
  }
  s -= lp.n_br;
  st.kind = ST_C;
  st.a = pt.c_lo + s * lp.rc;
  st.n = min(lp.rc, pt.c_hi - st.a);
  return st;
}

__device__ __forceinline__ const uint8_t* expert_blob(const DecodeParams& p, const LayerDev& L,
                                                      int slot_i, int id) {
  int b;
  if (p.use_slots) {
    b = p.slots[slot_i];
  } else {
    b = L.slot_of ? L.slot_of[id] : id;
  }
  return L.experts + static_cast<int64_t>(b) * p.blob_bytes;
}

// Does layer li's C stage carry the next layer's router block?
__device__ __forceinline__ bool c_has_router(const DecodeParams& p, int li) {
  return (p.phases & PH_ROUTER) && (p.phases & PH_C) && li + 1 < p.n_layers;
}

__device__ __forceinline__ bool needs_ids(const DecodeParams& p) {
  return (p.phases & (PH_BROUTED | PH_C)) != 0;
}

__device__ __forceinline__ int router_groups(int r0, int n) {
  return (r0 + n - 1) / kGroup - r0 / kGroup + 1;
}

__device__ uint32_t stage_bytes(const DecodeParams& p, const Stage& st, int li) {
  switch (st.kind) {
    case ST_R:
      return st.n * p.E + router_groups(st.a, st.n) * p.E * 4;
    case ST_BS:
    case ST_BR:
      return st.n * 2 * p.rbD;
    default: {
      uint32_t b = st.n * (p.K * p.rbI + p.rbS);
      if (c_has_router(p, li)) b += st.n * p.E + router_groups(st.a, st.n) * p.E * 4;
      return b;
    }
  }
}

__device__ void issue_stage(const Ctx& cx, const Stage& st, int li, uint8_t* dst, uint64_t* bar) {
  const DecodeParams& p = *cx.p;
  const int l = p.layer0 + li;
  const LayerDev& L = p.layers[l];
  auto router_block = [&](const LayerDev& R, uint8_t* d) {
    bulk_g2s(d, R.router_t + static_cast<int64_t>(st.a) * p.E, st.n * p.E, bar);
    d += st.n * p.E;
    const int g0 = st.a / kGroup, ng = router_groups(st.a, st.n);
    bulk_g2s(d, R.router_sb + static_cast<int64_t>(g0) * p.E, ng * p.E * 4, bar);
  };
  switch (st.kind) {
    case ST_R:
      router_block(L, dst);
      break;
    case ST_BS:
      bulk_g2s(dst, L.shared_gu + static_cast<int64_t>(st.a) * 2 * p.rbD, st.n * 2 * p.rbD, bar);
      break;
    case ST_BR: {
      // pairs [a, a+n) of the flattened k*I + j index; at most one expert boundary
      int q = st.a, left = st.n;
      uint8_t* d = dst;
      while (left > 0) {
        const int k = q / p.I, j = q % p.I;
        const int n = min(left, p.I - j);
        const uint8_t* blob = expert_blob(p, L, k, cx.misc[M_IDS + k]);
        bulk_g2s(d, blob + static_cast<int64_t>(j) * 2 * p.rbD, n * 2 * p.rbD, bar);
        d += n * 2 * p.rbD;
        q += n;
        left -= n;
      }
      break;
    }
    default: {
      uint8_t* d = dst;
      for (int k = 0; k < p.K; ++k) {
        const int id = cx.misc[M_IDS + k];
        const uint8_t* blob = expert_blob(p, L, k, id);
        bulk_g2s(d, blob + p.dn_off + static_cast<int64_t>(st.a) * p.rbI, st.n * p.rbI, bar);
        d += st.n * p.rbI;
      }
      bulk_g2s(d, L.shared_dn + static_cast<int64_t>(st.a) * p.rbS, st.n * p.rbS, bar);
      d += st.n * p.rbS;
      if (c_has_router(p, li)) router_block(p.layers[l + 1], d);
      break;
    }
  }
}

// ------------------------------------------------------------- producer

// L2 prefetches of the layer's weights that this CTA will stream later, so
// that HBM keeps working while the ring is full or the grid synchronises.
// Fixed weights (shared down rows, the next router's block) at the start of
// the layer; routed rows as soon as the layer's ids are known.
__device__ void prefetch_fixed(const Ctx& cx, int li) {
  const DecodeParams& p = *cx.p;
  if (!(p.phases & PH_C)) return;
  const int rows = cx.part.c_hi - cx.part.c_lo;
  if (rows <= 0) return;
  const int l = p.layer0 + li;
  prefetch_l2(p.layers[l].shared_dn + static_cast<int64_t>(cx.part.c_lo) * p.rbS, rows * p.rbS);
  if (c_has_router(p, li)) {
    const LayerDev& R = p.layers[l + 1];
    prefetch_l2(R.router_t + static_cast<int64_t>(cx.part.c_lo) * p.E, rows * p.E);
  }
}

// Routed gate/up pairs [q, rt_hi) of this CTA (only those stages the ring
// cannot take yet are worth a hint).
__device__ void prefetch_routed_gu(const Ctx& cx, int li, int q) {
  const DecodeParams& p = *cx.p;
  const LayerDev& L = p.layers[p.layer0 + li];
  while (q < cx.part.rt_hi) {
    const int k = q / p.I, j = q % p.I;
    const int n = min(cx.part.rt_hi - q, p.I - j);
    const uint8_t* blob = expert_blob(p, L, k, cx.misc[M_IDS + k]);
    prefetch_l2(blob + static_cast<int64_t>(j) * 2 * p.rbD, n * 2 * p.rbD);
    q += n;
  }
}

// The k routed experts' down rows of this CTA's output rows.
__device__ void prefetch_routed_dn(const Ctx& cx, int li) {
  const DecodeParams& p = *cx.p;
  const LayerDev& L = p.layers[p.layer0 + li];
  const int rows = cx.part.c_hi - cx.part.c_lo;
  if ((p.phases & PH_C) && rows > 0) {
    for (int k = 0; k < p.K; ++k) {
      const uint8_t* blob = expert_blob(p, L, k, cx.misc[M_IDS + k]);
      prefetch_l2(blob + p.dn_off + static_cast<int64_t>(cx.part.c_lo) * p.rbI, rows * p.rbI);
    }
  }
}

// Once the layer's ids are known the routed gate/up rows are needed first:
// their bulk copies go out at once, and only the stages that find no free
// ring slot are hinted into L2 ahead of their copies (with the down rows).
// Otherwise the down rows come with the C stages' own copies, which the ring
// issues while the gate/up stages are consumed, behind the gate/up data.
__device__ void producer(const Ctx& cx) {
  const DecodeParams& p = *cx.p;
  int st_idx = 0;
  for (int li = 0; li < p.n_layers; ++li) {
    const LayerPlan lp = layer_plan(p, cx.part, li);
    const int total = lp.n_r + lp.n_bs + lp.n_br + lp.n_c;
    bool gu_hinted = false;
    prefetch_fixed(cx, li);
    for (int s = 0; s <= total; ++s) {
      if (s == lp.n_r + lp.n_bs && needs_ids(p)) {
        // the routed stages' addresses need this layer's ids (one gate phase per layer)
        if (!mbar_wait(cx.ids_ready, li & 1, p.timeout_ns, &cx.misc[M_ABORT])) {
          cx.misc[M_ABORT] = 1;
          return;
        }
        if (lp.n_br == 0) prefetch_routed_dn(cx, li);
      }
      if (s == total) break;
      const Stage st = stage_at(p, cx.part, lp, s);
      const int slot = st_idx % p.nslots;
      const uint32_t round = st_idx / p.nslots;
      if (st.kind == ST_BR && !gu_hinted && !mbar_try_wait(&cx.empty[slot], (round & 1) ^ 1)) {
        prefetch_routed_gu(cx, li, st.a);
        prefetch_routed_dn(cx, li);
        gu_hinted = true;
      }
      if (!mbar_wait(&cx.empty[slot], (round & 1) ^ 1, p.timeout_ns, &cx.misc[M_ABORT])) {
        cx.misc[M_ABORT] = 1;
        return;
      }
      mbar_arrive_expect_tx(&cx.full[slot], stage_bytes(p, st, li));
      issue_stage(cx, st, li, cx.smem + static_cast<int64_t>(slot) * p.slot_bytes, &cx.full[slot]);
      ++st_idx;
      cx.misc[M_ISSUED] = st_idx;
    }
  }
}

// ------------------------------------------------------------- consumers

// Max of a value over all consumer threads.
// Max of a and sum of b over all consumer threads in one pass (fixed order).
__device__ void consumer_max_sum(const Ctx& cx, float& a, float& b) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  const int w = threadIdx.x >> 5;
  volatile float* ra = reinterpret_cast<volatile float*>(cx.misc) + M_RED;
  volatile float* rb = reinterpret_cast<volatile float*>(cx.misc) + M_RED2;
  if ((threadIdx.x & 31) == 0) {
    ra[w] = a;
    rb[w] = b;
  }
  csync();
  a = 0.f;
  b = 0.f;
  for (int i = 0; i < kConsumerWarps; ++i) {
    a = fmaxf(a, ra[i]);
    b += rb[i];
  }
  csync();
}

struct VecView {
  uint8_t* vec;   // int16 chunks, kChunkStride bytes each
  float* xsum;    // per-chunk sums
  float* vscale;  // dot products are multiplied by vscale[segment]
};

__device__ VecView vec_view(const Ctx& cx, int nchunks) {
  VecView v;
  v.vec = cx.smem + cx.p->off_vec;
  v.xsum = reinterpret_cast<float*>(v.vec + nchunks * kChunkStride);
  v.vscale = v.xsum + nchunks;
  return v;
}

// Layer input x (bf16 [D], global) -> int16 chunks.  One batch of 16-byte
// loads per thread (D <= 8 * kConsumers * kMaxXV); the CTA's own output rows
// [c_lo, c_hi) are also kept as fp32 in xres for the residual.
constexpr int kMaxXV = 2;  // D <= 8 * kConsumers * kMaxXV
constexpr int kMaxLogitLoads = 4;  // E <= 4 * kConsumers

// The layer input as loaded: this thread's bf16 words of x, the int16
// quantisation factor q and the pre-norm factor r.
struct XIn {
  uint4 r[kMaxXV];
  float q, rr;
  float hsc;  // h is held as fp16(h * hsc): hsc = 2^(-2 ceil(log2 max|r x|))
};

__device__ XIn prep_x(const Ctx& cx, const uint16_t* xg, const unsigned long long* lacc,
                      const float* logit_bias) {
  const DecodeParams& p = *cx.p;
  float* xres = reinterpret_cast<float*>(cx.smem + p.off_xres);
  const int nv = p.D / 8;
  XIn xin;
  uint4 (&r)[kMaxXV] = xin.r;
#pragma unroll
  for (int i = 0; i < kMaxXV; ++i) {
    const int idx = static_cast<int>(threadIdx.x) + i * kConsumers;
    r[i] = idx < nv ? __ldcg(reinterpret_cast<const uint4*>(xg) + idx) : make_uint4(0, 0, 0, 0);
  }
  long long lv[kMaxLogitLoads];  // the layer's raw router logits, in the same round trip
  float lb[kMaxLogitLoads];
  if (lacc) {
#pragma unroll
    for (int i = 0; i < kMaxLogitLoads; ++i) {
      const int e = static_cast<int>(threadIdx.x) + i * kConsumers;
      if (e < p.E) {
        lv[i] = static_cast<long long>(__ldcg(lacc + e));
        lb[i] = logit_bias ? __ldg(logit_bias + e) : 0.f;
      }
    }
  }
  float m = 0.f, ss = 0.f;  // max |x|, sum of x^2
#pragma unroll
  for (int i = 0; i < kMaxXV; ++i) {
    const int idx = static_cast<int>(threadIdx.x) + i * kConsumers;
    if (idx < nv) {
      const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = bf16_bits_to_f32(w[j] & 0xffffu), b = bf16_bits_to_f32(w[j] >> 16);
        m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
        ss = fmaf(a, a, fmaf(b, b, ss));
        const int col = idx * 8 + 2 * j;
        if (col >= cx.part.c_lo && col < cx.part.c_hi) xres[col - cx.part.c_lo] = a;
        if (col + 1 >= cx.part.c_lo && col + 1 < cx.part.c_hi) xres[col + 1 - cx.part.c_lo] = b;
      }
    }
  }
  consumer_max_sum(cx, m, ss);
  const float q = quant_factor(m);
  // r = 1 / sqrt(mean(x^2) + eps) with pre-norm, else 1 (the same value in every thread)
  const float rr = p.prenorm ? rsqrtf(ss / static_cast<float>(p.D) + p.rms_eps) : 1.f;
  if (lacc) {
    // logit_e = r * (sum of the fixed-point partials) + bias_e
    float* logits = reinterpret_cast<float*>(cx.smem + p.off_logits);
#pragma unroll
    for (int i = 0; i < kMaxLogitLoads; ++i) {
      const int e = static_cast<int>(threadIdx.x) + i * kConsumers;
      if (e < p.E) {
        float l = static_cast<float>(static_cast<double>(lv[i]) * 0x1p-32) * rr;
        if (logit_bias) l += lb[i];
        logits[e] = l;
      }
    }
  }
  xin.q = q;
  xin.rr = rr;
  {
    // the gated h grows like |u|^2 (u = r x): scaling it by 2^(-2e), e =
    // ceil(log2 max|u|), keeps fp16(h * hsc) in range for tiny and huge inputs
    const float umax = m * rr;
    int e = 0;
    if (umax > 0.f) e = max(-60, min(60, static_cast<int>(ceilf(log2f(umax)))));
    xin.hsc = ldexpf(1.f, -2 * e);
  }
  csync();  // the logits are read by every thread next
  return xin;
}

// x -> int16 chunks with their sums, in the activation region (after the
// routing, while the routed rows are in flight).
__device__ VecView pack_x(const Ctx& cx, const XIn& xin) {
  const DecodeParams& p = *cx.p;
  const int nc = p.D / 32, nv = p.D / 8;
  VecView v = vec_view(cx, nc);
  const float q = xin.q;
#pragma unroll
  for (int i = 0; i < kMaxXV; ++i) {
    const int idx = static_cast<int>(threadIdx.x) + i * kConsumers;
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (idx < nv) {
      const uint32_t w[4] = {xin.r[i].x, xin.r[i].y, xin.r[i].z, xin.r[i].w};
      uint32_t hv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j)
        hv[j] = pack_s16x2(bf16_bits_to_f32(w[j] & 0xffffu) * q, bf16_bits_to_f32(w[j] >> 16) * q);
      packed = make_uint4(hv[0], hv[1], hv[2], hv[3]);
      const int col = idx * 8;
      *reinterpret_cast<uint4*>(v.vec + (col >> 5) * kChunkStride + (col & 31) * 2) = packed;
    }
    // chunk sums: the 4 consecutive lanes holding idx 4c .. 4c+3 form chunk c
    int cs = sum8_s16(packed);
    cs += __shfl_xor_sync(0xffffffffu, cs, 1);
    cs += __shfl_xor_sync(0xffffffffu, cs, 2);
    if (idx < nv && (idx & 3) == 0) v.xsum[idx >> 2] = static_cast<float>(cs);
  }
  // dot products with X are q * (W x); the layer wants r * (W x)
  if (threadIdx.x == 0) v.vscale[0] = q > 0.f ? xin.rr / q : 0.f;
  csync();
  return v;
}

// The layer input, as each lane holds it for the B stages: chunks lane + 32 i
// (i < kXC) of the int16 vector, with their sums.
constexpr int kXC = 3;  // D <= 32 * 32 * kXC

struct XRegs {
  uint4 v[kXC][4];
  float s[kXC];
};

__device__ void load_xregs(const VecView& xv, int nc, XRegs& xr) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < kXC; ++i) {
    const int c = lane + 32 * i;
    if (c < nc) {
      const uint4* v = reinterpret_cast<const uint4*>(xv.vec + c * kChunkStride);
#pragma unroll
      for (int j = 0; j < 4; ++j) xr.v[i][j] = v[j];
      xr.s[i] = xv.xsum[c];
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) xr.v[i][j] = make_uint4(0, 0, 0, 0);
      xr.s[i] = 0.f;
    }
  }
}

// B stage: n gate/up row pairs -> h_out[pair].  Warp w owns pairs 2w and
// 2w+1; each lane takes its chunks of all four rows against the activation
// chunks it holds in registers, then a fixed-order warp sum per row.
__device__ __forceinline__ uint16_t h_bits(float h, float hsc) {
  return __half_as_ushort(__float2half_rn(fminf(fmaxf(h * hsc, -65504.f), 65504.f)));
}

__device__ void compute_b(const Ctx& cx, const uint8_t* buf, int n, const XRegs& xr, float vs,
                          float hsc, uint16_t* h_out) {
  const DecodeParams& p = *cx.p;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nc = p.D / 32, halfK = p.D / 2;
  const int p0 = 2 * warp;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // gate p0, up p0, gate p0+1, up p0+1
  // all code and scale words of this lane first (in flight together), then
  // the integer dot products
  uint4 wv[4][kXC];
  uint32_t sbv[4][kXC];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int i = 0; i < kXC; ++i) {
      const int c = lane + 32 * i;
      const bool ok = c < nc && p0 + (r >> 1) < n;
      const uint8_t* row = buf + (2 * p0 + r) * p.rbD;
      wv[r][i] = ok ? *reinterpret_cast<const uint4*>(row + c * 16) : make_uint4(0, 0, 0, 0);
      sbv[r][i] = ok ? *reinterpret_cast<const uint32_t*>(row + halfK + (c >> 1) * 4) : 0u;
    }
#pragma unroll
  for (int i = 0; i < kXC; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int tot = idot_chunk(wv[r][i], xr.v[i]);
      const __half2 sbh = *reinterpret_cast<const __half2*>(&sbv[r][i]);
      acc[r] += fmaf(__low2float(sbh), static_cast<float>(tot), __high2float(sbh) * xr.s[i]);
    }
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int o = 16; o; o >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], o);
  if (lane == 0) {
    if (p0 < n) h_out[p0] = h_bits(gelu_tanh(acc[0] * vs) * (acc[1] * vs), hsc);
    if (p0 + 1 < n) h_out[p0 + 1] = h_bits(gelu_tanh(acc[2] * vs) * (acc[3] * vs), hsc);
  }
}

// Router partial logits of rows [r0, r0+n) with the matching x values
// xr[0..n), accumulated into rpart[E].
__device__ void router_partial(const Ctx& cx, const uint8_t* blk, int r0, int n, const float* xr,
                               float* rpart) {
  const DecodeParams& p = *cx.p;
  const uint8_t* q = blk;
  const uint32_t* sb = reinterpret_cast<const uint32_t*>(blk + n * p.E);
  const int g0 = r0 / kGroup;
  for (int e = threadIdx.x; e < p.E; e += kConsumers) {
    float acc = 0.f;
    for (int r = 0; r < n; ++r) {
      const uint32_t w = sb[((r0 + r) / kGroup - g0) * p.E + e];
      const __half2 h2 = *reinterpret_cast<const __half2*>(&w);
      const float wv = fmaf(__low2float(h2), static_cast<float>(q[r * p.E + e]), __high2float(h2));
      acc = fmaf(wv, xr[r], acc);
    }
    rpart[e] += acc;
  }
}

// C phase: consumer thread t < ntask owns one (branch, chunk) task for the
// whole phase: chunk t of h (32 values; routed branch k = t / (I/32) for t <
// K*(I/32), the shared branch after that).  Each chunk is quantised on its
// own: X = rint(h * 32767 / m) with m the chunk's max |h|, so it carries its
// own scale sigma = m / 32767.  The task scale folds the routing weight
// (routed) and sigma.
struct HTask {
  uint4 v[4];
  float s;       // chunk sum of the int16 values
  float scale;   // w_k * sigma (routed) or sigma (shared)
  int k;         // branch (K = shared)
  int c;         // chunk within the branch
};

constexpr int kMaxHV = 4;  // K*I + S <= 8 * kConsumers * kMaxHV

// h (fp16 of h * hsc, global) -> the tasks' registers.  The loads are
// warp-contiguous (a warp instruction reads 512 consecutive bytes, which the
// L2 serves far faster than a line per thread); the 4 lanes that hold one
// chunk find its max and sum with shuffles, and the packed chunks pass
// through the activation region of shared memory to their task threads.
__device__ void load_htask(const Ctx& cx, HTask& ht, float hsc) {
  const DecodeParams& p = *cx.p;
  const int t = threadIdx.x;
  const int nh = p.K * p.I + p.S;
  const int n8 = nh / 8;                 // 16-byte groups of 8 fp16 values
  uint8_t* stage = cx.smem + p.off_vec;  // [nchunks] x kChunkStride bytes
  float* csig = reinterpret_cast<float*>(stage + (nh / 32) * kChunkStride);
  float* csum = csig + nh / 32;
  uint4 r[kMaxHV];
#pragma unroll
  for (int i = 0; i < kMaxHV; ++i) {
    const int idx = t + i * kConsumers;
    r[i] = idx < n8 ? __ldcg(reinterpret_cast<const uint4*>(p.h) + idx) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < kMaxHV; ++i) {
    const int idx = t + i * kConsumers;  // chunk idx / 4, part idx % 4
    const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
    float f[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&w[j]));
      f[2 * j] = v.x;
      f[2 * j + 1] = v.y;
    }
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const float q = quant_factor(m);
    const uint4 packed = make_uint4(pack_s16x2(f[0] * q, f[1] * q), pack_s16x2(f[2] * q, f[3] * q),
                                    pack_s16x2(f[4] * q, f[5] * q), pack_s16x2(f[6] * q, f[7] * q));
    int cs = sum8_s16(packed);
    cs += __shfl_xor_sync(0xffffffffu, cs, 1);
    cs += __shfl_xor_sync(0xffffffffu, cs, 2);
    if (idx < n8) {
      *reinterpret_cast<uint4*>(stage + (idx >> 2) * kChunkStride + (idx & 3) * 16) = packed;
      if ((idx & 3) == 0) {
        csig[idx >> 2] = m / 32767.f / hsc;  // back to units of h
        csum[idx >> 2] = static_cast<float>(cs);
      }
    }
  }
  csync();
  const int nch_i = p.I / 32;
  ht.k = -1;
  if (t < p.ntask) {
    const uint4* v = reinterpret_cast<const uint4*>(stage + t * kChunkStride);
#pragma unroll
    for (int j = 0; j < 4; ++j) ht.v[j] = v[j];
    ht.s = csum[t];
    const float sigma = csig[t];
    if (t < p.K * nch_i) {
      ht.k = t / nch_i;
      ht.c = t % nch_i;
      ht.scale = __int_as_float(cx.misc[M_WTS + ht.k]) * sigma;
    } else {
      ht.k = p.K;
      ht.c = t - p.K * nch_i;
      ht.scale = sigma;
    }
  }
}

constexpr int kRowBatch = 5;

// C stage: rows [r0, r0+n) of the layer output.  contrib (aliasing the
// activation region, free once the tasks are in registers) holds one partial
// per (row, task); then one warp per row sums them in a fixed order and adds
// the row's term of the next router's logits.
__device__ void compute_c(const Ctx& cx, const uint8_t* buf, int r0, int n, int li,
                          const HTask& ht, uint16_t* x_next, float* rpart) {
  const DecodeParams& p = *cx.p;
  float* contrib = reinterpret_cast<float*>(cx.smem + p.off_vec);  // [n][kConsumers]
  const int t = threadIdx.x;
  if (ht.k >= 0) {
    const bool shared = ht.k == p.K;
    const uint8_t* base = shared ? buf + static_cast<int64_t>(p.K) * n * p.rbI
                                 : buf + static_cast<int64_t>(ht.k) * n * p.rbI;
    const int rb = shared ? p.rbS : p.rbI;
    const int halfK = shared ? p.S / 2 : p.I / 2;
    // rows in batches of kRowBatch: the batch's code and scale words are in
    // flight together, then the integer dot products
    for (int r0b = 0; r0b < n; r0b += kRowBatch) {
      uint4 wv[kRowBatch];
      uint32_t sbv[kRowBatch];
#pragma unroll
      for (int k = 0; k < kRowBatch; ++k) {
        const int r = r0b + k;
        const uint8_t* row = base + r * rb;
        wv[k] = r < n ? *reinterpret_cast<const uint4*>(row + ht.c * 16) : make_uint4(0, 0, 0, 0);
        sbv[k] = r < n ? *reinterpret_cast<const uint32_t*>(row + halfK + (ht.c >> 1) * 4) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kRowBatch; ++k) {
        const int tot = idot_chunk(wv[k], ht.v);
        const __half2 sbh = *reinterpret_cast<const __half2*>(&sbv[k]);
        const int r = r0b + k;
        if (r < n)
          contrib[r * kConsumers + t] =
              fmaf(__low2float(sbh), static_cast<float>(tot), __high2float(sbh) * ht.s) * ht.scale;
      }
    }
  }
  csync();
  // One warp per row, two rows per warp at a time (rows rr and rr + 8, for
  // independent work in flight): a fixed-order tree sum of the row's task
  // partials, the output element, and the row's term of the next router's
  // logits, which each warp accumulates in its own row of rpart
  // ([kConsumerWarps][E]).
  const int warp = t >> 5, lane = t & 31;
  const bool nr = c_has_router(p, li);
  const uint8_t* rq = buf + static_cast<int64_t>(n) * (p.K * p.rbI + p.rbS);  // [n][E] codes
  const uint32_t* rsb = reinterpret_cast<const uint32_t*>(rq + n * p.E);     // [groups][E]
  const int g0 = r0 / kGroup;
  float* rp = rpart + warp * p.E;
  const float* xres = reinterpret_cast<const float*>(cx.smem + p.off_xres);
  constexpr int kPer = kConsumers / 32;  // task partials per lane and row
  for (int rb = warp; rb < n; rb += 2 * kConsumerWarps) {
    const int rr[2] = {rb, rb + kConsumerWarps};
    float y[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      float v[kPer];
#pragma unroll
      for (int i = 0; i < kPer; ++i) {
        const int j = lane + 32 * i;
        v[i] = (rr[q] < n && j < p.ntask) ? contrib[rr[q] * kConsumers + j] : 0.f;
      }
#pragma unroll
      for (int w = 1; w < kPer; w *= 2)
#pragma unroll
        for (int i = 0; i < kPer; i += 2 * w) v[i] += v[i + w];
      y[q] = v[0];
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      y[0] += __shfl_xor_sync(0xffffffffu, y[0], o);
      y[1] += __shfl_xor_sync(0xffffffffu, y[1], o);
    }
    float xd[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      xd[q] = 0.f;
      if (rr[q] < n) {
        const int d = r0 + rr[q];
        float out = y[q];
        if (p.residual) out += xres[d - cx.part.c_lo];
        const uint16_t ob = f32_to_bf16_bits(out);
        if (lane == 0) x_next[d] = ob;
        xd[q] = bf16_bits_to_f32(ob);
      }
    }
    if (nr) {
      const bool two = rr[1] < n;
      const uint32_t* sb0 = rsb + ((r0 + rr[0]) / kGroup - g0) * p.E;
      const uint32_t* sb1 = rsb + ((r0 + (two ? rr[1] : rr[0])) / kGroup - g0) * p.E;
      const uint8_t* q0 = rq + rr[0] * p.E;
      const uint8_t* q1 = rq + (two ? rr[1] : rr[0]) * p.E;
#pragma unroll 4
      for (int e = lane; e < p.E; e += 32) {
        const uint32_t w0 = sb0[e], w1 = sb1[e];
        const __half2 h0 = *reinterpret_cast<const __half2*>(&w0);
        const __half2 h1 = *reinterpret_cast<const __half2*>(&w1);
        const float wv0 = fmaf(__low2float(h0), static_cast<float>(q0[e]), __high2float(h0));
        const float wv1 = fmaf(__low2float(h1), static_cast<float>(q1[e]), __high2float(h1));
        const float acc = fmaf(wv0, xd[0], rp[e]);
        rp[e] = two ? fmaf(wv1, xd[1], acc) : acc;
      }
    }
  }
}

// Every CTA routes layer li itself from the raw logits that prep_x loaded
// into shared memory (identical in every CTA): apply the pre-norm factor r
// and the logit bias, take the top k (or the forced ids) and the softmax.  The
// ids and weights land in shared memory (M_IDS, M_WTS); CTA 0 also writes
// them to p.ids / p.wts for layer li.  Then the producer's gate for the
// layer's routed stages opens.
__device__ void route_all(const Ctx& cx, int li) {
  const DecodeParams& p = *cx.p;
  const float* logits = reinterpret_cast<const float*>(cx.smem + p.off_logits);
  const int t = threadIdx.x;
  // Top k in parallel: the rank of expert e is the number of experts before it
  // in (logit desc, index asc) order; the experts of rank < k are the choice,
  // in that order (or the forced ids).  Slot i's id goes to misc[M_IDS + i].
  if (li == 0 && p.forced) {
    if (t < p.K) cx.misc[M_IDS + t] = p.forced_ids[t];
  } else {
    // two threads per expert, each counting over half of the others (16-byte
    // broadcast reads of the logits when the halves are multiples of 4)
    const bool vec4 = (p.E & 7) == 0;
    for (int e2 = t; e2 < 2 * p.E; e2 += kConsumers) {
      const int e = e2 >> 1, half = e2 & 1;
      const float v = logits[e];
      const int f0 = half ? p.E / 2 : 0, f1 = half ? p.E : p.E / 2;
      int rank = 0;
      if (vec4) {
        const float4* l4 = reinterpret_cast<const float4*>(logits);
#pragma unroll 4
        for (int f = f0; f < f1; f += 4) {
          const float4 u = l4[f >> 2];
          rank += (u.x > v || (u.x == v && f < e)) ? 1 : 0;
          rank += (u.y > v || (u.y == v && f + 1 < e)) ? 1 : 0;
          rank += (u.z > v || (u.z == v && f + 2 < e)) ? 1 : 0;
          rank += (u.w > v || (u.w == v && f + 3 < e)) ? 1 : 0;
        }
      } else {
        for (int f = f0; f < f1; ++f) {
          const float u = logits[f];
          rank += (u > v || (u == v && f < e)) ? 1 : 0;
        }
      }
      rank += __shfl_xor_sync(0xffffffffu, rank, 1);
      if (!half && rank < p.K) cx.misc[M_IDS + rank] = e;
    }
  }
  csync();
  if (t < 32) {  // softmax over the k chosen logits (lanes 0..k-1)
    const int lane = t;
    int my_id = 0;
    float my_l = -INFINITY;
    if (lane < p.K) {
      my_id = cx.misc[M_IDS + lane];
      if (my_id < 0 || my_id >= p.E) {
        atomicCAS(p.bar + 2, DEV_OK, DEV_BAD_ID);
        my_id = 0;
      }
      my_l = logits[my_id];
    }
    float m = my_l;
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float ex = lane < p.K ? expf(my_l - m) : 0.f;
    float z = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    if (lane < p.K) {
      const float w = ex / z;
      cx.misc[M_IDS + lane] = my_id;
      cx.misc[M_WTS + lane] = __float_as_int(w);
      if (blockIdx.x == 0) {
        p.ids[li * p.K + lane] = my_id;
        p.wts[li * p.K + lane] = w;
      }
    }
  }
  csync();
  if (t == 0) mbar_arrive(cx.ids_ready);
}

// Grid barrier among the consumer groups of all CTAs on a monotonically
// increasing 64-bit arrival counter (bar[0..1]) that is a multiple of the grid
// size G between launches.  A CTA's first arrival in a launch is an atomic
// that returns the counter, from which it learns the launch's base multiple;
// the n-th barrier then completes when the counter reaches base + n G.  Later
// arrivals are fire-and-forget reductions, and each CTA polls the counter
// itself, so no arrival waits for a round trip before the others can see it.
// Returns false on timeout or abort.
__device__ bool grid_barrier(const Ctx& cx) {
  const DecodeParams& p = *cx.p;
  csync();
  if (threadIdx.x == 0) {
    // The CTA barrier above orders the other threads' writes before this
    // thread's release, which carries them (release is cumulative).
    unsigned long long* ctr = reinterpret_cast<unsigned long long*>(p.bar);
    const unsigned long long G = static_cast<unsigned long long>(cx.G);
    volatile unsigned long long* tgt = reinterpret_cast<volatile unsigned long long*>(cx.misc + M_TARGET);
    unsigned long long target;
    if (*tgt == 0ull) {
      const unsigned long long old = atom_add_acq_rel_gpu_u64(ctr, 1ull);
      target = (old / G + 1ull) * G + (p.stall_first_barrier ? G : 0ull);
    } else {
      red_add_release_gpu_u64(ctr, 1ull);
      target = *tgt + G;
    }
    *tgt = target;
    // Poll with relaxed loads of the counter and the status word issued
    // together (one round trip per poll); one acquire load once it is done.
    bool ok = false;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      const unsigned long long c = ld_relaxed_gpu_u64(ctr);
      const uint32_t st = ld_relaxed_gpu(p.bar + 2);
      if (c >= target) {
        (void)ld_acquire_gpu_u64(ctr);
        ok = true;
        break;
      }
      if (st != DEV_OK) break;
      if (globaltimer_ns() - t0 > p.timeout_ns) break;
    }
    if (!ok) {
      atomicCAS(p.bar + 2, DEV_OK, DEV_TIMEOUT);
      cx.misc[M_ABORT] = 1;
    }
  }
  csync();
  return !cx.misc[M_ABORT];
}

// Load ids/weights of layer li from global into shared memory and open the
// producer's gate for that layer's routed stages.
__device__ void publish_ids_local(const Ctx& cx, int li) {
  const DecodeParams& p = *cx.p;
  if (threadIdx.x < p.K) {
    int id = __ldcg(p.ids + li * p.K + threadIdx.x);
    if (id < 0 || id >= p.E) {
      atomicCAS(p.bar + 2, DEV_OK, DEV_BAD_ID);
      id = 0;
    }
    cx.misc[M_IDS + threadIdx.x] = id;
    cx.misc[M_WTS + threadIdx.x] = __float_as_int(__ldcg(p.wts + li * p.K + threadIdx.x));
  }
  csync();
  if (threadIdx.x == 0) mbar_arrive(cx.ids_ready);
}

__device__ bool wait_full(const Ctx& cx, int st_idx) {
  const DecodeParams& p = *cx.p;
  const int slot = st_idx % p.nslots;
  const uint32_t round = st_idx / p.nslots;
  if (threadIdx.x == 0) {
    if (!mbar_wait(&cx.full[slot], round & 1, p.timeout_ns, &cx.misc[M_ABORT]))
      cx.misc[M_ABORT] = 1;
  }
  csync();
  return !cx.misc[M_ABORT];
}

// Per-warp wait for a stage (no CTA barrier): every lane waits on the
// mbarrier phase itself, so each sees the copy engine's writes.  A timeout
// sets the abort flag; the warp then skips its work and the CTA leaves at its
// next CTA-wide check, so no warp is left waiting at a barrier.
__device__ bool wait_full_warp(const Ctx& cx, int st_idx) {
  const DecodeParams& p = *cx.p;
  const int slot = st_idx % p.nslots;
  const uint32_t round = st_idx / p.nslots;
  bool ok = mbar_wait(&cx.full[slot], round & 1, p.timeout_ns, &cx.misc[M_ABORT]);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) cx.misc[M_ABORT] = 1;
  return ok;
}

__device__ void release_slot(const Ctx& cx, int st_idx) {
  const int slot = st_idx % cx.p->nslots;
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&cx.empty[slot]);
}

// Add this CTA's partial logits (the sum of the warps' rows of rpart, in warp
// order) into the layer's accumulators: fp32 -> 64-bit fixed point in units
// of 2^-32 (|partial| < 2^31), integer atomic add.
__device__ void add_partials(const Ctx& cx, const float* rpart, unsigned long long* lacc) {
  const DecodeParams& p = *cx.p;
  for (int e = threadIdx.x; e < p.E; e += kConsumers) {
    float sum = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) sum += rpart[w * p.E + e];
    const long long v = __float2ll_rn(sum * 0x1p32f);
    red_add_gpu_u64(lacc + e, static_cast<unsigned long long>(v));
  }
}

__device__ __forceinline__ void trace(const Ctx& cx, int li, int ev) {
  const DecodeParams& p = *cx.p;
  if (p.trace && threadIdx.x == 0 && li < kTraceMaxLayers)
    p.trace[(static_cast<int64_t>(blockIdx.x) * p.n_layers + li) * kTraceEvents + ev] = globaltimer_ns();
}

__device__ void consumer(const Ctx& cx) {
  const DecodeParams& p = *cx.p;
  float* rpart = reinterpret_cast<float*>(cx.smem + p.off_rpart);
  float* xnext = reinterpret_cast<float*>(cx.smem + p.off_xnext);
  int st_idx = 0;
  for (int li = 0; li < p.n_layers; ++li) {
    const uint16_t* x_l = li == 0 ? p.x_in : p.xbuf + ((li - 1) & 1) * p.D;
    uint16_t* x_next = li + 1 == p.n_layers ? p.y_out : p.xbuf + (li & 1) * p.D;
    const LayerPlan lp = layer_plan(p, cx.part, li);
    // was layer li's routing computed in this launch (so we wait for its flag)?
    const bool routed_here = li > 0 || (p.phases & PH_ROUTER);
    int s = 0;
    trace(cx, li, 0);
    // ---- router of the launch's first layer (later layers: folded into C)
    if (li == 0 && (p.phases & PH_ROUTER)) {
      for (int e = threadIdx.x; e < kConsumerWarps * p.E; e += kConsumers) rpart[e] = 0.f;
      csync();
      if (lp.n_r) {
        if (!wait_full(cx, st_idx)) return;
        const Stage st = stage_at(p, cx.part, lp, s);
        for (int i = threadIdx.x; i < st.n; i += kConsumers)
          xnext[i] = bf16_bits_to_f32(__ldcg(x_l + st.a + i));
        csync();
        router_partial(cx, cx.smem + static_cast<int64_t>(st_idx % p.nslots) * p.slot_bytes,
                       st.a, st.n, xnext, rpart);
        csync();
        release_slot(cx, st_idx);
        ++st_idx;
        ++s;
      }
      add_partials(cx, rpart, p.lacc);
      if (!grid_barrier(cx)) return;
    }
    // ---- layer input (+ its router logits), routing, then the shared
    // expert's gate/up (which needs no ids) while the routed rows arrive
    unsigned long long* lacc_l = p.lacc + (li & 1) * p.E;
    const XIn xin = prep_x(cx, x_l, routed_here ? lacc_l : nullptr, p.layers[p.layer0 + li].logit_bias);
    trace(cx, li, 1);
    if (routed_here) route_all(cx, li);
    else if (needs_ids(p)) publish_ids_local(cx, li);  // ids from an earlier launch
    trace(cx, li, 2);
    const VecView xv = pack_x(cx, xin);
    XRegs xr;
    load_xregs(xv, p.D / 32, xr);
    const float vs = xv.vscale[0];
    // ---- shared gate/up stages, then the routed ones (one loop, so the dot
    // product code is emitted once)
    const int bs_end = lp.n_r + lp.n_bs, br_end = bs_end + lp.n_br;
    for (; s < br_end; ++s) {
      const Stage st = stage_at(p, cx.part, lp, s);
      const bool ok = wait_full_warp(cx, st_idx);
      if (s == lp.n_r) trace(cx, li, 3);
      if (s == bs_end) trace(cx, li, 5);
      if (s == br_end - 1) trace(cx, li, 6);
      const uint8_t* buf = cx.smem + static_cast<int64_t>(st_idx % p.nslots) * p.slot_bytes;
      if (ok) {
        compute_b(cx, buf, st.n, xr, vs, xin.hsc, p.h + (s < bs_end ? p.K * p.I : 0) + st.a);
        release_slot(cx, st_idx);
      }
      ++st_idx;
      if (s == bs_end - 1) trace(cx, li, 4);
    }
    trace(cx, li, 7);
    if (!(p.phases & PH_C)) {
      csync();  // the warps waited on their own: agree on the abort flag
      if (cx.misc[M_ABORT]) return;
      continue;
    }
    // ---- down + combine (+ next router's partial logits)
    if (!grid_barrier(cx)) return;
    trace(cx, li, 8);
    // every CTA has read layer li's logit accumulators: clear them for the
    // layer after next (their next additions come after the next barrier)
    if (blockIdx.x == 0)
      for (int e = threadIdx.x; e < p.E; e += kConsumers) lacc_l[e] = 0ull;
    HTask ht;
    load_htask(cx, ht, xin.hsc);
    trace(cx, li, 9);
    const bool nr = c_has_router(p, li);
    for (int e = threadIdx.x; e < kConsumerWarps * p.E; e += kConsumers) rpart[e] = 0.f;
    csync();  // the activation region is reused for the C-stage partials
    for (; s < lp.n_r + lp.n_bs + lp.n_br + lp.n_c; ++s) {
      const Stage st = stage_at(p, cx.part, lp, s);
      if (!wait_full(cx, st_idx)) return;
      if (s == lp.n_r + lp.n_bs + lp.n_br) trace(cx, li, 10);
      const uint8_t* buf = cx.smem + static_cast<int64_t>(st_idx % p.nslots) * p.slot_bytes;
      compute_c(cx, buf, st.a, st.n, li, ht, x_next, rpart);
      csync();
      release_slot(cx, st_idx);
      ++st_idx;
    }
    trace(cx, li, 11);
    if (nr) {
      add_partials(cx, rpart, p.lacc + ((li + 1) & 1) * p.E);
      if (!grid_barrier(cx)) return;
      trace(cx, li, 12);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  Ctx cx;
  cx.p = &p;
  cx.smem = smem;
  cx.full = reinterpret_cast<uint64_t*>(smem + p.off_bars);
  cx.empty = cx.full + kMaxSlots;
  cx.ids_ready = cx.empty + kMaxSlots;
  cx.misc = reinterpret_cast<volatile int*>(smem + p.off_misc);
  cx.G = gridDim.x;
  const int c = blockIdx.x, G = gridDim.x;
  cx.part.sh_lo = split_at(p.S, c, G);
  cx.part.sh_hi = split_at(p.S, c + 1, G);
  cx.part.rt_lo = split_at(p.K * p.I, c, G);
  cx.part.rt_hi = split_at(p.K * p.I, c + 1, G);
  cx.part.c_lo = split_at(p.D, c, G);
  cx.part.c_hi = split_at(p.D, c + 1, G);
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.nslots; ++i) {
      mbar_init(&cx.full[i], 1);
      mbar_init(&cx.empty[i], kConsumerWarps);
    }
    mbar_init(cx.ids_ready, 1);
    for (int i = 0; i < M_COUNT; ++i) cx.misc[i] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x >= kConsumers) {
    if (threadIdx.x == kConsumers) producer(cx);
  } else {
    consumer(cx);
    if (threadIdx.x == 0 && cx.misc[M_ABORT]) atomicCAS(p.bar + 2, DEV_OK, DEV_TIMEOUT);
  }
  __syncthreads();
  // Drain: copies issued but not consumed must land before the CTA exits.
  // Only the last stage issued on each slot can still be pending.
  if (threadIdx.x == 0) {
    const int issued = cx.misc[M_ISSUED];
    for (int st = issued - p.nslots < 0 ? 0 : issued - p.nslots; st < issued; ++st)
      mbar_wait(&cx.full[st % p.nslots], (st / p.nslots) & 1, p.timeout_ns, nullptr);
  }
  __syncthreads();
}

}  // namespace

int decode_smem_plan(DecodeParams* p, int max_smem) {
  const int nc_x = p->D / 32;
  auto vec_bytes = [](int nc, int nscale) { return nc * kChunkStride + nc * 8 + nscale * 4; };
  int vb = vec_bytes(nc_x, 1);  // the layer input's int16 chunks
  vb = (vb + 127) / 128 * 128;
  const int b_stage = kPairsPerStage * 2 * p->rbD;
  const int rsb = 2 * p->E * 4;
  const int c_stage = p->rc_max * (p->K * p->rbI + p->rbS + p->E) + rsb;
  int slot = b_stage > c_stage ? b_stage : c_stage;
  slot = (slot + 127) / 128 * 128;
  // fixed regions after the slot ring
  int fixed = 0;
  auto take = [&](int bytes) {
    const int o = fixed;
    fixed += (bytes + 127) / 128 * 128;
    return o;
  };
  if (vb < p->rc_max * kConsumers * 4) vb = (p->rc_max * kConsumers * 4 + 127) / 128 * 128;
  const int nc_h = (p->K * p->I + p->S) / 32;
  const int hb = nc_h * kChunkStride + 2 * nc_h * 4;  // staged int16 chunks of h + sigma, sum
  if (vb < hb) vb = (hb + 127) / 128 * 128;
  const int o_vec = take(vb);  // also h's staging and the C-stage partials [rc_max][kConsumers]
  const int o_rpart = take(kConsumerWarps * p->E * 4);
  const int o_xnext = take(256 * 4);
  const int o_xres = take(256 * 4);
  const int o_logits = take(p->E * 4);
  const int o_misc = take(M_COUNT * 4);
  const int o_bars = take((2 * kMaxSlots + 1) * 8);
  int ns = (max_smem - fixed) / slot;
  if (ns > kMaxSlots) ns = kMaxSlots;
  if (ns < 2) return -1;
  p->slot_bytes = slot;
  p->nslots = ns;
  const int base = ns * slot;
  p->off_vec = base + o_vec;
  p->off_rpart = base + o_rpart;
  p->off_xnext = base + o_xnext;
  p->off_xres = base + o_xres;
  p->off_logits = base + o_logits;
  p->off_misc = base + o_misc;
  p->off_bars = base + o_bars;
  p->smem_total = base + fixed;
  return p->smem_total <= max_smem ? 0 : -1;
}

int decode_launch(const DecodeParams& p, int grid, void* stream, bool cooperative) {
  const int e = set_smem_limit(reinterpret_cast<const void*>(decode_kernel), p.smem_total);
  if (e != 0) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.smem_total;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return static_cast<int>(cudaLaunchKernelEx(&cfg, decode_kernel, p));
}

}  // namespace moe
