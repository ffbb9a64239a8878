// Decode attention: the step before the router, one token per call.
//
// shilu.ai "drumih/turbo-fieldfare", sections 推理引擎的工作原理 and
// 状态和范围: in every layer the GPU computes attention and then the router
// from resident weights; attention weights are 4-bit MLX affine; the KV
// store is FP16, a bounded ring for the sliding-window layers and linear for
// the full-attention layers; decode attention is exact split-K/V with
// distinct normalised K and V paths.  The pages give no formulas; the
// readings (the same as the oracle's):
//   u = x / sqrt(mean(x^2) + 1e-6); q, k, v = Wq u, Wk u, Wv u;
//   per head q, k, v divided by their RMS (eps 1e-6); RoPE on q and k
//   (rotate-half pairs (i, i + d/2), angle pos * theta^(-2i/d));
//   k, v stored as fp16 in slot pos % capacity;
//   scores q . k / sqrt(d) over the visible positions, softmax, o = sum w v;
//   y = Wo o, optionally + x (residual), rounded to bf16.
//
// Launches per layer and token:
//   qgemv_kernel        q, k, v = W u (4-bit integer dot products; the
//                       pre-norm is a scale applied after the dot product)
//   attn_decode_kernel  (head, split) blocks: per-head RMS norms and RoPE, the
//                       fp16 KV append, scores and an online softmax over the
//                       split's positions; the head's last block merges the
//                       splits
//   qgemv_kernel        y = Wo o (+ x), bf16
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <string>
#include <vector>

#include "../../include/moe.h"
#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"
#include "qdot.cuh"
#include "repack.h"

namespace moe {
namespace {

constexpr int kGemvWarps = 8;
constexpr int kGemvMaxK = 4096;            // input length <= 4096
constexpr int kGemvXC = kGemvMaxK / 1024;  // activation chunks per lane
constexpr int kMaxSplits = 64;
constexpr int kSplitWarps = 8;

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

struct GemvArgs {
  const uint8_t* w;        // qrows [R] of K inputs, rb bytes each
  int R, K, rb;
  const uint16_t* x_bf16;  // input, bf16 [K] (or NULL)
  const float* x_f32;      // input, fp32 [K] (or NULL)
  int prenorm;             // dot products scaled by 1 / sqrt(mean(x^2) + eps)
  float eps;
  float* y_f32;            // output fp32 [R] (or NULL)
  uint16_t* y_bf16;        // output bf16 [R] = bf16(res + W x) (or NULL)
  const uint16_t* res;     // residual bf16 [R] for y_bf16 (or NULL)
};

// y = W x for a 4-bit matrix in qrows.  Every block quantises the whole
// input to int16 chunks in shared memory (one scale: max|x|), then each warp
// takes RPW rows: each lane loads its 32-column chunks of its rows (codes
// and scale/bias words, coalesced across the warp) and accumulates
// s * sum(q X) + b * sum(X) per chunk; a fixed-order warp sum finishes the row.
// The weight loads are issued before the input is prepared, so their
// latency overlaps the block's input reduction.
template <int RPW>  // rows per warp
__global__ void __launch_bounds__(kGemvWarps * 32) qgemv_kernel(GemvArgs a) {
  __shared__ __align__(16) uint8_t xs[(kGemvMaxK / 32) * 80];
  __shared__ float xsum[kGemvMaxK / 32];
  __shared__ float red[2][kGemvWarps];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int nc = a.K / 32, nv = a.K / 8;
  // ---- RPW rows per warp: their code and scale/bias words are requested
  // first, so that they are in flight while the input is prepared
  const int r0 = (blockIdx.x * kGemvWarps + w) * RPW;
  uint4 wv[RPW][kGemvXC];
  uint32_t sbv[RPW][kGemvXC];
#pragma unroll
  for (int k = 0; k < RPW; ++k) {
    const bool row_ok = r0 + k < a.R;
    const uint8_t* row = a.w + static_cast<int64_t>(row_ok ? r0 + k : 0) * a.rb;
#pragma unroll
    for (int i = 0; i < kGemvXC; ++i) {
      const int c = lane + 32 * i;
      const bool ok = row_ok && c < nc;
      wv[k][i] = ok ? __ldg(reinterpret_cast<const uint4*>(row + c * 16)) : make_uint4(0, 0, 0, 0);
      sbv[k][i] = ok ? __ldg(reinterpret_cast<const uint32_t*>(row + a.K / 2 + (c >> 1) * 4)) : 0u;
    }
  }
  // the input comes from the kernel before on the stream.  The next kernel
  // may start only once this one has passed its wait, so a kernel's early
  // reads (weights here, older cache rows in the attention kernel) overlap
  // at most the kernel right before it, which never writes them.
  grid_dep_wait();
  grid_dep_launch();
  // ---- the input, 8 values per thread and group of 256 threads
  float v[2][8];
  float m = 0.f, ss = 0.f;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int idx = t + 256 * g;
#pragma unroll
    for (int j = 0; j < 8; ++j) v[g][j] = 0.f;
    if (idx < nv) {
      if (a.x_bf16) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(a.x_bf16) + idx);
        const uint32_t ww[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[g][2 * j] = bf16_to_f32(ww[j] & 0xffffu);
          v[g][2 * j + 1] = bf16_to_f32(ww[j] >> 16);
        }
      } else {
        const float4 p0 = __ldg(reinterpret_cast<const float4*>(a.x_f32) + 2 * idx);
        const float4 p1 = __ldg(reinterpret_cast<const float4*>(a.x_f32) + 2 * idx + 1);
        v[g][0] = p0.x; v[g][1] = p0.y; v[g][2] = p0.z; v[g][3] = p0.w;
        v[g][4] = p1.x; v[g][5] = p1.y; v[g][6] = p1.z; v[g][7] = p1.w;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        m = fmaxf(m, fabsf(v[g][j]));
        ss = fmaf(v[g][j], v[g][j], ss);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    ss += __shfl_xor_sync(0xffffffffu, ss, o);
  }
  if (lane == 0) {
    red[0][w] = m;
    red[1][w] = ss;
  }
  __syncthreads();
  m = 0.f;
  ss = 0.f;
#pragma unroll
  for (int i = 0; i < kGemvWarps; ++i) {
    m = fmaxf(m, red[0][i]);
    ss += red[1][i];
  }
  const float q = quant_factor(m);
  const float r = a.prenorm ? rsqrtf(ss / static_cast<float>(a.K) + a.eps) : 1.f;
  const float vs = q > 0.f ? r / q : 0.f;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int idx = t + 256 * g;
    uint4 packed = make_uint4(0, 0, 0, 0);
    if (idx < nv) {
      packed = make_uint4(pack_s16x2(v[g][0] * q, v[g][1] * q), pack_s16x2(v[g][2] * q, v[g][3] * q),
                          pack_s16x2(v[g][4] * q, v[g][5] * q), pack_s16x2(v[g][6] * q, v[g][7] * q));
      *reinterpret_cast<uint4*>(xs + (idx >> 2) * 80 + (idx & 3) * 16) = packed;
    }
    // chunk sums: the 4 consecutive lanes holding idx 4c .. 4c+3 form chunk c
    int cs = sum8_s16(packed);
    cs += __shfl_xor_sync(0xffffffffu, cs, 1);
    cs += __shfl_xor_sync(0xffffffffu, cs, 2);
    if (idx < nv && (idx & 3) == 0) xsum[idx >> 2] = static_cast<float>(cs);
  }
  __syncthreads();
  float acc[RPW];
#pragma unroll
  for (int k = 0; k < RPW; ++k) acc[k] = 0.f;
#pragma unroll
  for (int i = 0; i < kGemvXC; ++i) {
    const int c = lane + 32 * i;
    if (c < nc) {
      uint4 xc[4];
      const uint4* src = reinterpret_cast<const uint4*>(xs + c * 80);
#pragma unroll
      for (int j = 0; j < 4; ++j) xc[j] = src[j];
      const float sx = xsum[c];
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        const int tot = idot_chunk(wv[k][i], xc);
        const __half2 sb = *reinterpret_cast<const __half2*>(&sbv[k][i]);
        acc[k] += fmaf(__low2float(sb), static_cast<float>(tot), __high2float(sb) * sx);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < RPW; ++k)
#pragma unroll
    for (int o = 16; o; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < RPW; ++k) {
      const int row = r0 + k;
      if (row >= a.R) continue;
      const float out = acc[k] * vs;
      if (a.y_f32) a.y_f32[row] = out;
      if (a.y_bf16) a.y_bf16[row] = f32_to_bf16((a.res ? bf16_to_f32(a.res[row]) : 0.f) + out);
    }
  }
}

struct AttnArgs {
  const float* qkv;         // raw projections: Hq query heads, Hkv key heads, Hkv value heads
  int Hq, Hkv, d;
  float eps;
  long long pos, cap;       // this token's position; the layer cache's capacity
  long long first, n;       // visible positions [first, first + n), the last one is pos
  int nsplit;
  float scale;              // 1 / sqrt(d)
  const double* freq_pi;    // [d/2] theta^(-2i/d) / pi of this layer
  __half* kc;               // this layer's key cache [Hkv][cap][d]
  __half* vc;               // this layer's value cache [Hkv][cap][d]
  float* part;              // [Hq][nsplit][d + 2]: unnormalised o, then max and sum
  unsigned int* done;       // [Hq] arrival counters (zero between calls)
  float* o;                 // [Hq][d] attention output
};

// A lane's PER fp16 values of one cache row, as loaded (8 values: 16 bytes).
template <int PER> struct Raw;
template <> struct Raw<8> { using T = uint4; };
template <> struct Raw<4> { using T = uint2; };
template <> struct Raw<2> { using T = uint32_t; };

template <int PER>
__device__ __forceinline__ typename Raw<PER>::T load_raw(const __half* p) {
  return *reinterpret_cast<const typename Raw<PER>::T*>(p);
}

template <int PER>
__device__ __forceinline__ void to_float(const typename Raw<PER>::T& r, float (&out)[PER]) {
  const uint32_t* ww = reinterpret_cast<const uint32_t*>(&r);
#pragma unroll
  for (int j = 0; j < PER / 2; ++j) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ww[j]));
    out[2 * j] = f.x;
    out[2 * j + 1] = f.y;
  }
}

// RoPE of one head vector held one value per thread (t < d) through shared
// memory: the pairs (i, i + d/2) rotate by the angle, in half turns,
// pos * theta^(-2i/d) / pi; formed in fp64 and reduced exactly to [-1, 1],
// then sine and cosine in fp32.
__device__ __forceinline__ float rope_value(float x0, float x1, int t, const AttnArgs& a) {
  const int h = a.d / 2, i = t < h ? t : t - h;
  const double turns = static_cast<double>(a.pos) * a.freq_pi[i];
  const float r = static_cast<float>(turns - 2.0 * rint(0.5 * turns));
  float sn, cs;
  sincospif(r, &sn, &cs);
  return t < h ? x0 * cs - x1 * sn : x0 * sn + x1 * cs;
}

// Decode attention of one layer for one token, block (h, s) = (query head,
// split of the visible positions); kv head g = h / (Hq / Hkv).
//  0. Each warp requests the cache rows of its first kBatch positions before
//     anything else, so their latency overlaps step 1.
//  1. q_h = RoPE(q_raw_h / RMS); the split that holds position pos (the last
//     one) also forms this token's key RoPE(k_raw_g / RMS) and value
//     v_raw_g / RMS, rounded to fp16 as the cache stores them, and the first
//     query head of the group writes them to cache slot pos % cap.  The three
//     norms share one block reduction and the two rotations one exchange.
//  2. Warp w takes the split's earlier positions lo + w, + 8, ... in batches
//     of kBatch (their key and value rows loaded together) with an online
//     softmax; warp 0 then folds in position pos from shared memory.  The 8
//     warps merge in a fixed order into the split's (o, max, sum).
//  3. The last block of head h to finish (an arrival counter) merges the
//     head's splits in split order: o_h = sum o_s e^(m_s - M) / sum l_s e^(m_s - M),
//     and clears the counter for the next call.
template <int PER>
__global__ void __launch_bounds__(kSplitWarps * 32) attn_decode_kernel(AttnArgs a) {
  constexpr int D = 32 * PER;
  constexpr int kBatch = 8;
  using RawT = typename Raw<PER>::T;
  __shared__ float bq[D], bk[D];
  __shared__ float red[3][kSplitWarps];
  __shared__ float qs[D];
  __shared__ __align__(16) __half kcur[D], vcur[D];
  __shared__ float wm[kSplitWarps], wl[kSplitWarps];
  __shared__ float wo[kSplitWarps][D];
  __shared__ unsigned int last;
  const int h = blockIdx.x, s = blockIdx.y, t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int grp = a.Hq / a.Hkv, g = h / grp;
  const long long lo = a.first + a.n * s / a.nsplit, hi = a.first + a.n * (s + 1) / a.nsplit;
  const bool has_pos = hi == a.pos + 1;  // the last split
  const long long hc = has_pos ? hi - 1 : hi;  // positions read from the cache
  const __half* kbase = a.kc + static_cast<int64_t>(g) * a.cap * D + lane * PER;
  const __half* vbase = a.vc + static_cast<int64_t>(g) * a.cap * D + lane * PER;
  // ---- 0. the first batch of cache rows
  RawT kr[kBatch], vr[kBatch];
  auto fetch = [&](long long p0) {
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const long long p = p0 + static_cast<long long>(b) * kSplitWarps;
      const long long slot = (p < hc ? p : lo) % a.cap;
      kr[b] = load_raw<PER>(kbase + slot * D);
      vr[b] = load_raw<PER>(vbase + slot * D);
    }
  };
  if (lo + w < hc) fetch(lo + w);
  // the projections come from the kernel before on the stream (the cache
  // rows fetched above were written two or more launches earlier)
  grid_dep_wait();
  grid_dep_launch();
  // ---- 1. this head's query, and (last split) this token's key and value
  {
    const float qv = t < D ? a.qkv[static_cast<int64_t>(h) * D + t] : 0.f;
    const float kv = has_pos && t < D ? a.qkv[static_cast<int64_t>(a.Hq + g) * D + t] : 0.f;
    const float vv = has_pos && t < D ? a.qkv[static_cast<int64_t>(a.Hq + a.Hkv + g) * D + t] : 0.f;
    float sq = qv * qv, sk = kv * kv, sv = vv * vv;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
      sv += __shfl_xor_sync(0xffffffffu, sv, o);
    }
    if (lane == 0) {
      red[0][w] = sq;
      red[1][w] = sk;
      red[2][w] = sv;
    }
    __syncthreads();
    sq = sk = sv = 0.f;
#pragma unroll
    for (int i = 0; i < kSplitWarps; ++i) {
      sq += red[0][i];
      sk += red[1][i];
      sv += red[2][i];
    }
    const float inv_d = 1.f / static_cast<float>(D);
    const float qn = qv * rsqrtf(sq * inv_d + a.eps), kn = kv * rsqrtf(sk * inv_d + a.eps);
    const float vn = vv * rsqrtf(sv * inv_d + a.eps);
    if (t < D) {
      bq[t] = qn;
      bk[t] = kn;
    }
    __syncthreads();
    if (t < D) {
      const int hh = D / 2, i = t < hh ? t : t - hh;
      qs[t] = rope_value(bq[i], bq[i + hh], t, a);
      if (has_pos) {
        kcur[t] = __float2half_rn(rope_value(bk[i], bk[i + hh], t, a));
        vcur[t] = __float2half_rn(vn);
        if (h % grp == 0) {
          const int64_t at = (static_cast<int64_t>(g) * a.cap + a.pos % a.cap) * D + t;
          a.kc[at] = kcur[t];
          a.vc[at] = vcur[t];
        }
      }
    }
    __syncthreads();
  }
  float q[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) q[i] = qs[lane * PER + i];
  // ---- 2. scores and online softmax
  float m = -INFINITY, l = 0.f, o[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) o[i] = 0.f;
  auto fold = [&](float dot, const float (&vf)[PER]) {
    const float sc = dot * a.scale;
    const float mn = fmaxf(m, sc);
    const float c = expf(m - mn), e = expf(sc - mn);
    l = l * c + e;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[i] = fmaf(o[i], c, e * vf[i]);
    m = mn;
  };
  for (long long p0 = lo + w; p0 < hc; p0 += kSplitWarps * kBatch) {
    if (p0 != lo + w) fetch(p0);
    float dot[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      float kf[PER];
      to_float<PER>(kr[b], kf);
      dot[b] = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) dot[b] = fmaf(q[i], kf[i], dot[b]);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1)
#pragma unroll
      for (int b = 0; b < kBatch; ++b) dot[b] += __shfl_xor_sync(0xffffffffu, dot[b], off);
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (p0 + static_cast<long long>(b) * kSplitWarps >= hc) break;
      float vf[PER];
      to_float<PER>(vr[b], vf);
      fold(dot[b], vf);
    }
  }
  if (has_pos && w == 0) {  // this token's own key and value
    float kf[PER], vf[PER];
    to_float<PER>(load_raw<PER>(kcur + lane * PER), kf);
    to_float<PER>(load_raw<PER>(vcur + lane * PER), vf);
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) dot = fmaf(q[i], kf[i], dot);
#pragma unroll
    for (int off = 16; off; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    fold(dot, vf);
  }
  if (lane == 0) {
    wm[w] = m;
    wl[w] = l;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) wo[w][lane * PER + i] = o[i];
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kSplitWarps; ++i) M = fmaxf(M, wm[i]);
  float* out = a.part + (static_cast<int64_t>(h) * a.nsplit + s) * (D + 2);
  for (int i = t; i < D; i += kSplitWarps * 32) {
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kSplitWarps; ++j)
      if (wl[j] > 0.f) acc = fmaf(wo[j][i], expf(wm[j] - M), acc);
    out[i] = acc;
  }
  if (t == 0) {
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kSplitWarps; ++j)
      if (wl[j] > 0.f) L = fmaf(wl[j], expf(wm[j] - M), L);
    out[D] = M;
    out[D + 1] = L;
  }
  // ---- 3. the head's last block merges its splits
  __threadfence();
  __syncthreads();
  if (t == 0) last = atomicAdd(a.done + h, 1u) == static_cast<unsigned int>(a.nsplit - 1);
  __syncthreads();
  if (!last) return;
  __threadfence();
  const float* ph = a.part + static_cast<int64_t>(h) * a.nsplit * (D + 2);
  // the splits' (max, sum) into shared memory, then each thread's column of
  // every split in batches of 8 independent loads, added in split order
  float* fm = bq;                   // reused: [kMaxSplits] <= D floats
  float* fl = &wo[0][0];            // reused: [kMaxSplits]
  if (t < a.nsplit) {
    fm[t] = __ldcg(ph + t * (D + 2) + D);
    fl[t] = __ldcg(ph + t * (D + 2) + D + 1);
  }
  __syncthreads();
  float Mh = -INFINITY;
  for (int j = 0; j < a.nsplit; ++j) Mh = fmaxf(Mh, fm[j]);
  if (t < D) {
    float L = 0.f, acc = 0.f;
    for (int j0 = 0; j0 < a.nsplit; j0 += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = j0 + k < a.nsplit ? __ldcg(ph + (j0 + k) * (D + 2) + t) : 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (j0 + k < a.nsplit) {
          const float f = expf(fm[j0 + k] - Mh);
          L = fmaf(fl[j0 + k], f, L);
          acc = fmaf(v[k], f, acc);
        }
      }
    }
    a.o[static_cast<int64_t>(h) * D + t] = acc / L;
  }
  if (t == 0) a.done[h] = 0u;
}

}  // namespace
}  // namespace moe

using namespace moe;

struct moe_attn {
  moe_attn_config cfg{};
  std::vector<int> sliding;
  std::vector<double> theta;
  std::vector<int64_t> cap, kv_off, next_pos;
  int device = 0;
  int64_t rbD = 0, rbQ = 0, wqkv_bytes = 0, layer_bytes = 0;
  uint8_t* w = nullptr;   // per layer: q/k/v qrows, then the output projection's qrows
  __half* kv = nullptr;   // per layer: keys [Hkv][cap][d], then values
  float* qkv = nullptr;   // [(Hq + 2 Hkv) d]
  float* qn = nullptr;    // [Hq d]
  float* part = nullptr;  // [Hq][kMaxSplits][d + 2]
  float* o = nullptr;     // [Hq d]
  uint16_t* xa = nullptr; // decode-step temporaries, bf16 [2][D]
  double* freq = nullptr; // [L][d/2] theta_l^(-2i/d) / pi
  unsigned int* done = nullptr;  // [Hq] arrival counters of the attention kernel
  std::string err;
};

namespace {

thread_local std::string g_attn_create_error;

moe_status afail(moe_attn* a, moe_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (a)
    a->err = buf;
  else
    g_attn_create_error = buf;
  return s;
}

void attn_free(moe_attn* a) {
  if (!a) return;
  if (a->w || a->kv) cudaDeviceSynchronize();
  cudaFree(a->w);
  cudaFree(a->kv);
  cudaFree(a->qkv);
  cudaFree(a->qn);
  cudaFree(a->part);
  cudaFree(a->o);
  cudaFree(a->xa);
  cudaFree(a->freq);
  cudaFree(a->done);
}

bool qt_ok(const moe_qtensor& t) { return t.q && t.scale && t.bias; }


// Rows per warp: 4 for tall matrices (one wave of blocks with their loads
// in flight), 2 otherwise (enough blocks to cover the SMs).
int launch_gemv(const GemvArgs& g, cudaStream_t s) {
  if (g.R >= 6144)
    return launch_pdl(qgemv_kernel<4>, dim3((g.R + 4 * kGemvWarps - 1) / (4 * kGemvWarps)),
                      dim3(kGemvWarps * 32), 0, s, g);
  return launch_pdl(qgemv_kernel<2>, dim3((g.R + 2 * kGemvWarps - 1) / (2 * kGemvWarps)),
                    dim3(kGemvWarps * 32), 0, s, g);
}

}  // namespace

#pragma GCC visibility push(default)
extern "C" {

moe_status moe_attn_create(const moe_attn_config* cfg, const moe_attn_weights* layers, moe_attn** out) {
  if (!out) return afail(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg || !layers) return afail(nullptr, MOE_ERR_INVALID_ARG, "cfg or layers is NULL");
  const moe_attn_config& c = *cfg;
  const int d = c.head_dim;
  if (c.group != kGroup || c.d_model <= 0 || c.d_model % 256 || c.d_model > kGemvMaxK ||
      c.n_heads < 1 || c.n_kv_heads < 1 || c.n_heads % c.n_kv_heads || (d != 64 && d != 128 && d != 256) ||
      c.n_heads * d > kGemvMaxK || (c.n_heads * d) % 256 || c.n_layers < 1 || c.window < 1 ||
      c.max_seq < 1)
    return afail(nullptr, MOE_ERR_INVALID_ARG, "unsupported attention configuration");
  for (int l = 0; l < c.n_layers; ++l) {
    const moe_attn_weights& w = layers[l];
    if (!qt_ok(w.wq) || !qt_ok(w.wk) || !qt_ok(w.wv) || !qt_ok(w.wo))
      return afail(nullptr, MOE_ERR_INVALID_ARG, "layer %d: missing attention weights", l);
    if (c.rope_theta && !(c.rope_theta[l] > 0.f))
      return afail(nullptr, MOE_ERR_INVALID_ARG, "layer %d: rope_theta must be positive", l);
  }
  std::unique_ptr<moe_attn> a(new moe_attn());
  a->cfg = c;
  a->cfg.sliding = nullptr;
  a->cfg.rope_theta = nullptr;
  const int L = c.n_layers, D = c.d_model, Hq = c.n_heads, Hkv = c.n_kv_heads;
  a->sliding.resize(L);
  a->theta.resize(L);
  a->cap.resize(L);
  a->kv_off.resize(L);
  a->next_pos.assign(L, 0);
  int64_t kv_total = 0;
  for (int l = 0; l < L; ++l) {
    a->sliding[l] = c.sliding ? (c.sliding[l] != 0) : 0;
    a->theta[l] = c.rope_theta ? c.rope_theta[l] : 10000.0;
    a->cap[l] = a->sliding[l] ? c.window : c.max_seq;
    a->kv_off[l] = kv_total;
    kv_total += 2 * int64_t(Hkv) * a->cap[l] * d;
  }
  a->rbD = qrow_bytes(D);
  a->rbQ = qrow_bytes(int64_t(Hq) * d);
  const int64_t R = int64_t(Hq + 2 * Hkv) * d;
  a->wqkv_bytes = R * a->rbD;
  a->layer_bytes = (a->wqkv_bytes + int64_t(D) * a->rbQ + 255) / 256 * 256;
#define ATRY(call)                                                                        \
  do {                                                                                    \
    const cudaError_t e_ = (call);                                                        \
    if (e_ != cudaSuccess) {                                                              \
      const moe_status st_ = afail(nullptr, e_ == cudaErrorMemoryAllocation ? MOE_ERR_OOM \
                                                                              : MOE_ERR_CUDA, \
                                   "%s: %s", #call, cudaGetErrorString(e_));              \
      attn_free(a.get());                                                                 \
      return st_;                                                                         \
    }                                                                                     \
  } while (0)
  ATRY(cudaGetDevice(&a->device));
  ATRY(cudaMalloc(&a->w, a->layer_bytes * L));
  ATRY(cudaMalloc(&a->kv, kv_total * sizeof(__half)));
  ATRY(cudaMemset(a->kv, 0, kv_total * sizeof(__half)));
  ATRY(cudaMalloc(&a->qkv, R * sizeof(float)));
  ATRY(cudaMalloc(&a->qn, int64_t(Hq) * d * sizeof(float)));
  ATRY(cudaMalloc(&a->part, int64_t(Hq) * kMaxSplits * (d + 2) * sizeof(float)));
  ATRY(cudaMalloc(&a->o, int64_t(Hq) * d * sizeof(float)));
  ATRY(cudaMalloc(&a->xa, 2 * int64_t(D) * sizeof(uint16_t)));
  ATRY(cudaMalloc(&a->done, Hq * sizeof(unsigned int)));
  ATRY(cudaMemset(a->done, 0, Hq * sizeof(unsigned int)));
  {
    std::vector<double> fr(static_cast<size_t>(L) * (d / 2));
    const double pi = 3.14159265358979323846;
    for (int l = 0; l < L; ++l)
      for (int i = 0; i < d / 2; ++i) fr[size_t(l) * (d / 2) + i] = std::pow(a->theta[l], -2.0 * i / d) / pi;
    ATRY(cudaMalloc(&a->freq, fr.size() * sizeof(double)));
    ATRY(cudaMemcpy(a->freq, fr.data(), fr.size() * sizeof(double), cudaMemcpyHostToDevice));
  }
  {
    std::vector<uint8_t> stage(static_cast<size_t>(a->layer_bytes));
    for (int l = 0; l < L; ++l) {
      const moe_attn_weights& w = layers[l];
      std::fill(stage.begin(), stage.end(), 0);
      repack_matrix(w.wq, int64_t(Hq) * d, D, stage.data());
      repack_matrix(w.wk, int64_t(Hkv) * d, D, stage.data() + int64_t(Hq) * d * a->rbD);
      repack_matrix(w.wv, int64_t(Hkv) * d, D, stage.data() + int64_t(Hq + Hkv) * d * a->rbD);
      repack_matrix(w.wo, D, int64_t(Hq) * d, stage.data() + a->wqkv_bytes);
      ATRY(cudaMemcpy(a->w + l * a->layer_bytes, stage.data(), stage.size(), cudaMemcpyHostToDevice));
    }
  }
#undef ATRY
  *out = a.release();
  return MOE_OK;
}

void moe_attn_destroy(moe_attn* a) {
  if (!a) return;
  attn_free(a);
  delete a;
}

const char* moe_attn_last_error(const moe_attn* a) {
  return a ? a->err.c_str() : g_attn_create_error.c_str();
}

moe_status moe_attn_reset(moe_attn* a) {
  if (!a) return MOE_ERR_INVALID_ARG;
  std::fill(a->next_pos.begin(), a->next_pos.end(), 0);
  return MOE_OK;
}

moe_status moe_attn_forward(moe_attn* a, int layer, const void* x, long long pos, void* y, int flags,
                            void* stream) {
  if (!a || !x || !y || x == y) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
    return afail(a, MOE_ERR_INVALID_ARG, "x and y must be 16-byte aligned");
  if (layer < 0 || layer >= a->cfg.n_layers) return afail(a, MOE_ERR_INVALID_ARG, "bad layer %d", layer);
  if (pos != 0 && pos != a->next_pos[layer])
    return afail(a, MOE_ERR_STATE, "layer %d expects position %lld (or 0 to restart), got %lld",
                 layer, static_cast<long long>(a->next_pos[layer]), pos);
  if (pos < 0 || (!a->sliding[layer] && pos >= a->cfg.max_seq))
    return afail(a, MOE_ERR_INVALID_ARG, "position %lld beyond max_seq of a full-attention layer", pos);
  const int D = a->cfg.d_model, Hq = a->cfg.n_heads, Hkv = a->cfg.n_kv_heads, d = a->cfg.head_dim;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* wl = a->w + layer * a->layer_bytes;
  __half* kc = a->kv + a->kv_off[layer];
  __half* vc = kc + int64_t(Hkv) * a->cap[layer] * d;
  // q, k, v projections of the pre-normed input
  GemvArgs g{};
  g.w = wl;
  g.R = (Hq + 2 * Hkv) * d;
  g.K = D;
  g.rb = static_cast<int>(a->rbD);
  g.x_bf16 = static_cast<const uint16_t*>(x);
  g.prenorm = 1;
  g.eps = 1e-6f;
  g.y_f32 = a->qkv;
  int e = launch_gemv(g, s);
  // norms, rotation, KV append, split-K/V attention and the merge: one launch
  const long long n = a->sliding[layer] ? (pos + 1 < a->cfg.window ? pos + 1 : a->cfg.window) : pos + 1;
  AttnArgs aa{};
  aa.qkv = a->qkv;
  aa.Hq = Hq;
  aa.Hkv = Hkv;
  aa.d = d;
  aa.eps = 1e-6f;
  aa.pos = pos;
  aa.cap = a->cap[layer];
  aa.first = pos + 1 - n;
  aa.n = n;
  aa.nsplit = static_cast<int>(std::min<long long>(kMaxSplits, (n + 63) / 64));
  aa.scale = 1.f / std::sqrt(static_cast<float>(d));
  aa.freq_pi = a->freq + int64_t(layer) * (d / 2);
  aa.kc = kc;
  aa.vc = vc;
  aa.part = a->part;
  aa.done = a->done;
  aa.o = a->o;
  if (!e) {
    const dim3 grid(Hq, aa.nsplit);
    if (d == 256) e = launch_pdl(attn_decode_kernel<8>, grid, dim3(kSplitWarps * 32), 0, s, aa);
    else if (d == 128) e = launch_pdl(attn_decode_kernel<4>, grid, dim3(kSplitWarps * 32), 0, s, aa);
    else e = launch_pdl(attn_decode_kernel<2>, grid, dim3(kSplitWarps * 32), 0, s, aa);
  }
  // output projection (+ residual), bf16
  GemvArgs go{};
  go.w = wl + a->wqkv_bytes;
  go.R = D;
  go.K = Hq * d;
  go.rb = static_cast<int>(a->rbQ);
  go.x_f32 = a->o;
  go.prenorm = 0;
  go.y_bf16 = static_cast<uint16_t*>(y);
  go.res = (flags & MOE_FWD_RESIDUAL) ? static_cast<const uint16_t*>(x) : nullptr;
  if (!e) e = launch_gemv(go, s);
  if (e) return afail(a, MOE_ERR_CUDA, "attention launch: %s", cudaGetErrorString(cudaError_t(e)));
  a->next_pos[layer] = pos + 1;
  return MOE_OK;
}

moe_status moe_decode_step(moe_attn* a, moe_handle* h, const void* x, long long pos, void* y,
                           int n_layers, void* stream) {
  if (!a || !h || !x || !y || x == y) return MOE_ERR_INVALID_ARG;
  if (n_layers < 1 || n_layers > a->cfg.n_layers)
    return afail(a, MOE_ERR_INVALID_ARG, "n_layers out of range for the attention handle");
  const int D = a->cfg.d_model;
  const void* cur = x;
  for (int l = 0; l < n_layers; ++l) {
    // attention (+ residual) into xa[0]; the MoE layer reads it directly
    // (the router hand-off) and writes x_{l+1} into xa[1] or y
    uint16_t* t0 = a->xa;
    uint16_t* t1 = a->xa + D;
    moe_status st = moe_attn_forward(a, l, cur, pos, t0, MOE_FWD_RESIDUAL, stream);
    if (st != MOE_OK) return st;
    void* dst = l + 1 == n_layers ? y : static_cast<void*>(t1);
    st = moe_layer_forward(h, l, t0, 1, dst, MOE_FWD_RESIDUAL | MOE_FWD_PRENORM, nullptr, stream,
                           nullptr);
    if (st != MOE_OK) return afail(a, st, "MoE layer %d: %s", l, moe_last_error(h));
    cur = t1;
  }
  return MOE_OK;
}

}  // extern "C"
#pragma GCC visibility pop
