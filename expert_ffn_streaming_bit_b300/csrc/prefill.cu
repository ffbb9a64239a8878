// Multi-token (prefill) layer step, SIMT parts: token preparation, the
// router's top-k and softmax, bucketing of the T*k (token, expert)
// assignments by expert together with the grouped GEMM's work units, and the
// gather combine.  The router GEMM and the grouped GEMMs run on the tensor
// cores (gemm_tc.cu).
//
// Passages (sh.edu-sjtu.cn article, section 三件事, third bullet; shilu.ai
// "drumih/turbo-fieldfare", section 推理引擎的工作原理): prompts are prefilled in
// chunks so that each expert brought in serves every row routed to it; the
// bucketing below is that grouping, done on the device.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf16f(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// ceil(log2(u)) for a positive float, exactly, from its bits (an infinity
// gives 128).
__device__ __forceinline__ int ceil_log2(float u) {
  const uint32_t b = __float_as_uint(u);
  const int ex = static_cast<int>((b >> 23) & 0xffu);
  const uint32_t mant = b & 0x7fffffu;
  if (ex == 0) {  // subnormal: u = mant 2^-149
    const int msb = 31 - __clz(mant);
    return msb - 149 + ((mant & (mant - 1u)) ? 1 : 0);
  }
  return ex - 127 + (mant ? 1 : 0);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------ token prep
// Per token (one warp): a power-of-two factor f with max|x| f in [2^14, 2^15)
// (1 for a zero row), x16 = fp16(f x) (exact for bf16 inputs in range), and
// the scales that turn dot products with x16 into dot products with the
// layer input u = r x (r = 1 / sqrt(mean(x^2) + eps) with the pre-norm, else 1).
// hscale = 2^(-2e), e = ceil(log2(max|u|)): the gated intermediate h grows
// like |u|^2, so it is held as fp16(h * hscale), inside fp16's normal range
// for tiny and huge inputs alike, and the down output is divided by hscale
// again (exact powers of two).  The row of x16 ends with its group sums
// (internal.h, kGsumCols): the sums of the fp16 values actually stored, in a
// fixed order.
constexpr int kPrepV = 12;  // D <= 8 * 32 * kPrepV

__global__ void __launch_bounds__(256) tok_prep_kernel(const uint16_t* __restrict__ x, int T, int D,
                                                       int prenorm, float eps,
                                                       __half* __restrict__ x16,
                                                       float* __restrict__ sigma,
                                                       float* __restrict__ rscale,
                                                       float* __restrict__ hscale) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const uint4* row = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * D);
  const int nv = D / 8;
  // the row is read once, all of a lane's loads in flight together
  uint4 rv[kPrepV];
#pragma unroll
  for (int k = 0; k < kPrepV; ++k) {
    const int i = lane + 32 * k;
    rv[k] = i < nv ? __ldg(row + i) : make_uint4(0, 0, 0, 0);
  }
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < kPrepV; ++k) {
    const uint32_t w[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) m = fmaxf(m, fmaxf(fabsf(bf16f(w[j] & 0xffffu)), fabsf(bf16f(w[j] >> 16))));
  }
  m = warp_max(m);
  int e = m > 0.f ? static_cast<int>((__float_as_uint(m) >> 23) & 0xffu) - 127 : 14;
  e = max(-100, min(100, e));
  const float f = ldexpf(1.f, 14 - e);
  const size_t pitch = static_cast<size_t>(D) + kGsumCols;
  uint4* out = reinterpret_cast<uint4*>(x16 + static_cast<size_t>(t) * pitch);
  float ss = 0.f;
  float part[kPrepV] = {};  // sum of the lane's 8 stored values per load
#pragma unroll
  for (int k = 0; k < kPrepV; ++k) {
    const int i = lane + 32 * k;
    if (i >= nv) break;
    const uint32_t w[4] = {rv[k].x, rv[k].y, rv[k].z, rv[k].w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16f(w[j] & 0xffffu) * f, b = bf16f(w[j] >> 16) * f;
      ss = fmaf(a, a, fmaf(b, b, ss));
      const __half2 h = __floats2half2_rn(a, b);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
      part[k] += __low2float(h) + __high2float(h);
    }
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  // group g (64 columns) = loads 8g .. 8g+7 = lanes 8j .. 8j+7 of load k,
  // g = 4k + j; D is a multiple of 128, so a group is wholly in or out
  __half* gs = x16 + static_cast<size_t>(t) * pitch + D;
#pragma unroll
  for (int k = 0; k < kPrepV; ++k) {
    float v = (lane + 32 * k < nv) ? part[k] : 0.f;
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    if ((lane & 7) == 0 && lane + 32 * k < nv) gs[4 * k + (lane >> 3)] = __float2half_rn(v * 0.015625f);
  }
  for (int g = D / 64 + lane; g < kGsumCols; g += 32) gs[g] = __float2half_rn(0.f);
  ss = warp_sum(ss);
  if (lane == 0) {
    // fp32 arithmetic: B300's fp64 pipe is narrow, and eight warps of a block
    // queue on it.  f = 2^k; the fp32 branch keeps f^2 and eps f^2 far inside
    // the float range (|k| <= 40, max|x| in [2^-26, 2^55)); other rows take
    // the fp64 one.
    const int k = 14 - e;
    float r = 1.f;
    if (prenorm) {
      if (k >= -40 && k <= 40) {
        r = f / sqrtf(ss / static_cast<float>(D) + eps * (f * f));
      } else {
        const double fd = static_cast<double>(f);
        r = static_cast<float>(fd / sqrt(static_cast<double>(ss) / D + static_cast<double>(eps) * fd * fd));
      }
    }
    sigma[t] = r / f;  // exact: f is a power of two and r / f stays normal
    rscale[t] = r;
    const float umax = m * r;
    const int eu = umax > 0.f ? max(-60, min(60, ceil_log2(umax))) : 0;  // 0 for a zero row
    hscale[t] = ldexpf(1.f, -2 * eu);
  }
}

// ------------------------------------------------------------ router top-k
// One warp per token: logits = sigma * (sum of the splits of w . x16, in
// order) + bias, sigma = r / f (so the logit is r * (w . x));
// top-k by (logit desc, index asc) (or the forced ids); softmax over the k.
// EPL = experts per lane (E <= 32 EPL); the loads of 48 / EPL splits for all
// of a lane's experts are in flight together.
template <int EPL>
__global__ void __launch_bounds__(256) router_topk_kernel(const float* __restrict__ partial,
                                                          int nsplit, int T, int E, int K,
                                                          const float* __restrict__ sigma,
                                                          const float* __restrict__ bias,
                                                          const int32_t* __restrict__ forced,
                                                          int32_t* __restrict__ ids,
                                                          float* __restrict__ wts) {
  grid_dep_wait();
  grid_dep_launch();
  constexpr int kB = 48 / EPL;  // splits per batch of loads
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float lv[EPL];
  const float r = sigma[t];
  // each expert's splits are summed in split order
#pragma unroll
  for (int i = 0; i < EPL; ++i) lv[i] = 0.f;
  for (int sp0 = 0; sp0 < nsplit; sp0 += kB) {
    float pv[kB][EPL];
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const float* row = partial + (static_cast<size_t>(sp0 + k) * T + t) * E;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        pv[k][i] = sp0 + k < nsplit && e < E ? row[e] : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kB; ++k)
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (sp0 + k < nsplit) lv[i] += pv[k][i];
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float v = -INFINITY;
    if (e < E) {
      v = lv[i] * r;
      if (bias) v += bias[e];
    }
    lv[i] = v;
  }
  // choice j is kept by lane j (K <= 32)
  int my_id = 0;
  float my_l = -INFINITY;
  for (int j = 0; j < K; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    if (forced) {
      bi = forced[t * K + j];
      float v = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == bi) v = lv[i];
      // the owner lane holds the value; others contribute 0 (one owner)
      bv = warp_sum((bi & 31) == lane ? v : 0.f);
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane + 32 * i;
        if (e < E && (lv[i] > bv || (lv[i] == bv && e < bi))) {
          bv = lv[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) {
          bv = ov;
          bi = oi;
        }
      }
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == bi) lv[i] = -INFINITY;
    }
    if (lane == j) {
      my_id = bi;
      my_l = bv;
    }
  }
  // softmax over the k chosen logits; the sum runs in choice order
  const float m = warp_max(lane < K ? my_l : -INFINITY);
  const float ex = lane < K ? expf(my_l - m) : 0.f;
  float z = 0.f;
  for (int j = 0; j < K; ++j) z += __shfl_sync(0xffffffffu, ex, j);
  if (lane < K) {
    ids[t * K + lane] = my_id;
    wts[t * K + lane] = ex / z;
  }
}

// -------------------------------------------------------------- bucketing
// Stable counting sort of the n = T*K assignments a = t*K + j by expert.  Up
// to kSmallN assignments, one block does it all (bk_small, below); above, it
// takes three launches so that no single SM carries the whole sort:
//   bk_hist   block b, warp w count the experts of their 256-assignment
//             segment -> hist[b][w][e];
//   bk_scan   one block: counts, offsets (exclusive scan over experts) and
//             the write base of every (block, warp, expert) in (block, warp)
//             order (in place in hist);
//   bk_place  block b, warp w place their segment in order with a
//             match/rank step: the result is in (expert, t, j) order; the
//             blocks then write the GEMM work units, a grid-strided share
//             each (one SM alone is limited by its store rate there).
// Work units: each expert's rows are cut into ceil(count / kUnitTokens)
// nearly equal token tiles, times the groups of kTilesPerUnit weight row
// tiles of the gate/up and of the down matrix; the shared expert's units (all
// T tokens) follow the routed ones.
constexpr int kBkWarps = 8;
constexpr int kBkThreads = 32 * kBkWarps;
constexpr int kBkPerLane = 8;                     // assignments per lane
constexpr int kBkWarpSeg = 32 * kBkPerLane;       // 256 per warp
constexpr int kBkBlockSeg = kBkWarps * kBkWarpSeg;  // 2048 per block

__global__ void __launch_bounds__(kBkThreads) bk_hist_kernel(BucketArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int h[kBkWarps][kMaxPrefillExperts];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, n = a.T * a.K;
  for (int i = tid; i < kBkWarps * kMaxPrefillExperts; i += kBkThreads) (&h[0][0])[i] = 0;
  __syncthreads();
  const int s0 = blockIdx.x * kBkBlockSeg + warp * kBkWarpSeg;
  int eb[kBkPerLane];
#pragma unroll
  for (int j = 0; j < kBkPerLane; ++j) {
    const int i = s0 + 32 * j + lane;
    eb[j] = i < n ? __ldg(a.ids + i) : 0;
  }
#pragma unroll
  for (int j = 0; j < kBkPerLane; ++j) {
    if (s0 + 32 * j + lane >= n) continue;
    int e = eb[j];
    if (e < 0 || e >= E) {
      atomicCAS(a.status, DEV_OK, DEV_BAD_ID);
      e = 0;
    }
    atomicAdd(&h[warp][e], 1);
  }
  __syncthreads();
  int* out = a.hist + static_cast<int64_t>(blockIdx.x) * kBkWarps * E;
  for (int i = tid; i < kBkWarps * E; i += kBkThreads) out[i] = h[i / E][i % E];
}

constexpr int kScanThreads = 1024;

// Exclusive scans over the experts, by one warp (lane = its lane): offsets of
// the assignments (off) and of the token tiles (toff), with the totals in
// off[E] and toff[E].
__device__ void scan_experts(int E, const int* cnt, int* off, int* toff, int lane) {
  int acc = 0, tacc = 0;
  for (int e0 = 0; e0 < E; e0 += 32) {
    const int ee = e0 + lane;
    const int c = ee < E ? cnt[ee] : 0;
    const int nt = (c + kUnitTokens - 1) / kUnitTokens;
    int x = c, y = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xs = __shfl_up_sync(0xffffffffu, x, o), ys = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) {
        x += xs;
        y += ys;
      }
    }
    if (ee < E) {
      off[ee] = acc + x - c;
      toff[ee] = tacc + y - nt;
    }
    acc += __shfl_sync(0xffffffffu, x, 31);
    tacc += __shfl_sync(0xffffffffu, y, 31);
  }
  if (lane == 0) {
    off[E] = acc;
    toff[E] = tacc;
  }
}

// The GEMM work units of both launches and their counts, from the per-expert
// counts and scans, by threads tid = 0 .. nthreads-1 of one block.
__device__ void emit_units(const BucketArgs& a, const int* cnt, const int* off, const int* toff,
                           int tid, int nthreads) {
  const int E = a.E;
  constexpr int kTU = kTilesPerUnit;
  const int pgu_r = (a.mt_gu_r + kTU - 1) / kTU, pdn = (a.mt_dn + kTU - 1) / kTU,
            pgu_s = (a.mt_gu_s + kTU - 1) / kTU;
  const int routed_tiles = toff[E];
  const int st = (a.T + kUnitTokens - 1) / kUnitTokens;  // shared token tiles
  if (tid == 0) {
    a.n_units[0] = routed_tiles * pgu_r + st * pgu_s;
    a.n_units[1] = (routed_tiles + st) * pdn;
  }
  // The shared expert's units come first: the CTAs take units in grid-stride
  // order, and its down units (K = d_shared) are the longest, so last they
  // would set the launch's tail.
  // routed: one thread per (token tile, weight group); the tile's expert is
  // found by a binary search over toff
  for (int idx = tid; idx < routed_tiles * (pgu_r + pdn); idx += nthreads) {
    const bool gu = idx < routed_tiles * pgu_r;
    const int j = gu ? idx : idx - routed_tiles * pgu_r;
    const int per = gu ? pgu_r : pdn;
    const int tile = j / per, m = j % per;
    int lo = 0, hi = E - 1;  // the last expert with toff[e] <= tile
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (toff[mid] <= tile) lo = mid;
      else hi = mid - 1;
    }
    const int ex = lo, tt = tile - toff[ex], nt = toff[ex + 1] - toff[ex];
    const int c = cnt[ex];
    const int r0t = c * tt / nt, r1t = c * (tt + 1) / nt;
    const int mt_all = gu ? a.mt_gu_r : a.mt_dn;
    GemmUnit u{0, kTU * m, ex, off[ex] + r0t, r1t - r0t, min(kTU, mt_all - kTU * m), {0, 0}};
    if (gu) a.units_gu[st * pgu_s + tile * pgu_r + m] = u;
    else a.units_dn[(st + tile) * pdn + m] = u;
  }
  for (int idx = tid; idx < st * (pgu_s + pdn); idx += nthreads) {
    const bool gu = idx < st * pgu_s;
    const int j = gu ? idx : idx - st * pgu_s;
    const int per = gu ? pgu_s : pdn;
    const int tt = j / per, m = j % per;
    const int r0t = a.T * tt / st, r1t = a.T * (tt + 1) / st;
    const int mt_all = gu ? a.mt_gu_s : a.mt_dn;
    GemmUnit u{1, kTU * m, 0, r0t, r1t - r0t, min(kTU, mt_all - kTU * m), {0, 0}};
    if (gu) a.units_gu[tt * pgu_s + m] = u;
    else a.units_dn[tt * pdn + m] = u;
  }
}

__global__ void __launch_bounds__(kScanThreads) bk_scan_kernel(BucketArgs a, int nb) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int part[kScanThreads];
  __shared__ int cnt[kMaxPrefillExperts];
  __shared__ int off[kMaxPrefillExperts + 1];
  __shared__ int toff[kMaxPrefillExperts + 1];
  const int tid = threadIdx.x;
  const int E = a.E;
  const int rows = nb * kBkWarps;          // (block, warp) rows of hist, in order
  const int np = kScanThreads / E;         // threads per expert (E <= 256 -> >= 4)
  const int e = tid % E, pi = tid / E;     // this thread: expert e, row chunk pi
  const bool active = pi < np;
  const int rper = (rows + np - 1) / np;
  const int r0 = min(rows, pi * rper), r1 = min(rows, r0 + rper);
  // per (expert, chunk) sums, loads in flight 8 at a time
  int sum = 0;
  if (active) {
    for (int r = r0; r < r1; r += 8) {
      int v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = r + k < r1 ? a.hist[static_cast<int64_t>(r + k) * E + e] : 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) sum += v[k];
    }
  }
  part[tid] = sum;
  __syncthreads();
  if (tid < E) {
    int c = 0;
    for (int q = 0; q < np; ++q) c += part[q * E + tid];
    cnt[tid] = c;
  }
  __syncthreads();
  if (tid < 32) scan_experts(E, cnt, off, toff, tid);
  __syncthreads();
  // write bases: chunk pi of expert e starts at off[e] + the earlier chunks' sums
  if (active) {
    int base = off[e];
    for (int q = 0; q < pi; ++q) base += part[q * E + e];
    for (int r = r0; r < r1; r += 8) {  // loads 8 at a time in flight
      int v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = r + k < r1 ? a.hist[static_cast<int64_t>(r + k) * E + e] : 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (r + k < r1) a.hist[static_cast<int64_t>(r + k) * E + e] = base;
        base += v[k];
      }
    }
  }
  if (tid < E) {
    a.counts[tid] = cnt[tid];
    a.offsets[tid] = off[tid];
  }
  if (tid == 0) a.offsets[E] = off[E];
}

// Places one warp's segment of assignments s0 + 32 j + lane (j < PER_LANE)
// in order: the lanes with the same expert take consecutive slots from
// base[e] (this warp's write base per expert) by their rank among their peers.
template <int PER_LANE>
__device__ __forceinline__ void place_segment(const BucketArgs& a, int* base,
                                              const int (&eb)[PER_LANE], int s0, int n, int lane) {
#pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int i = s0 + 32 * j + lane;
    const bool act = i < n;
    int e = eb[j];
    if (act && (e < 0 || e >= a.E)) e = 0;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const unsigned lower = peers & ((1u << lane) - 1u);
    if (act) {
      const int pos = base[e] + __popc(lower);
      a.perm[pos] = i;
      a.inv[i] = pos;
    }
    __syncwarp();
    if (act && lower == 0) base[e] += __popc(peers);
    __syncwarp();
  }
}

__global__ void __launch_bounds__(kBkThreads) bk_place_kernel(BucketArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int base[kBkWarps][kMaxPrefillExperts];
  __shared__ int cnt[kMaxPrefillExperts];
  __shared__ int off[kMaxPrefillExperts + 1];
  __shared__ int toff[kMaxPrefillExperts + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, n = a.T * a.K;
  const int* hb = a.hist + static_cast<int64_t>(blockIdx.x) * kBkWarps * E;
  for (int i = tid; i < kBkWarps * E; i += kBkThreads) base[i / E][i % E] = hb[i];
  for (int e = tid; e < E; e += kBkThreads) cnt[e] = a.counts[e];
  __syncthreads();
  if (tid < 32) scan_experts(E, cnt, off, toff, tid);  // for the units, below
  const int s0 = blockIdx.x * kBkBlockSeg + warp * kBkWarpSeg;
  int eb[kBkPerLane];
#pragma unroll
  for (int j = 0; j < kBkPerLane; ++j) {
    const int i = s0 + 32 * j + lane;
    eb[j] = i < n ? __ldg(a.ids + i) : -1;
  }
  place_segment(a, base[warp], eb, s0, n, lane);
  __syncthreads();
  emit_units(a, cnt, off, toff, blockIdx.x * kBkThreads + tid, gridDim.x * kBkThreads);
}

// n = T*K <= kSmallN: one launch of kSmallBlocks blocks.  Every block builds
// the histogram and the scans of all n assignments (cheap at this size) and
// writes a grid-strided share of the work units; block 0 alone writes the
// counts, the offsets and the placement, warp w holding the assignments
// [kSmallPerLane 32 w, kSmallPerLane 32 (w + 1)).  This saves the two extra
// launches and the global histogram round trip of the three-launch path,
// whose parallelism a chunk of ~128 tokens cannot use.
constexpr int kSmallWarps = kScanThreads / 32;
constexpr int kSmallPerLane = 2;
constexpr int kSmallN = kScanThreads * kSmallPerLane;
constexpr int kSmallBlocks = 8;

__global__ void __launch_bounds__(kScanThreads) bk_small_kernel(BucketArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int h[kSmallWarps][kMaxPrefillExperts];
  __shared__ int cnt[kMaxPrefillExperts];
  __shared__ int off[kMaxPrefillExperts + 1];
  __shared__ int toff[kMaxPrefillExperts + 1];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, n = a.T * a.K;
  const bool lead = blockIdx.x == 0;
  for (int i = tid; i < kSmallWarps * E; i += kScanThreads) h[i / E][i % E] = 0;
  const int s0 = warp * 32 * kSmallPerLane;
  int eb[kSmallPerLane];
#pragma unroll
  for (int j = 0; j < kSmallPerLane; ++j) {
    const int i = s0 + 32 * j + lane;
    int e = i < n ? __ldg(a.ids + i) : -1;
    if (i < n && (e < 0 || e >= E)) {
      if (lead) atomicCAS(a.status, DEV_OK, DEV_BAD_ID);
      e = 0;
    }
    eb[j] = e;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSmallPerLane; ++j)
    if (s0 + 32 * j + lane < n) atomicAdd(&h[warp][eb[j]], 1);
  __syncthreads();
  if (tid < E) {  // counts; each warp's row becomes its offset within the expert
    int c = 0;
    for (int w = 0; w < kSmallWarps; ++w) {
      const int v = h[w][tid];
      h[w][tid] = c;
      c += v;
    }
    cnt[tid] = c;
  }
  __syncthreads();
  if (tid < 32) scan_experts(E, cnt, off, toff, tid);
  __syncthreads();
  if (lead) {
    if (tid < E) {
      for (int w = 0; w < kSmallWarps; ++w) h[w][tid] += off[tid];
      a.counts[tid] = cnt[tid];
      a.offsets[tid] = off[tid];
    }
    if (tid == 0) a.offsets[E] = off[E];
    __syncthreads();
    place_segment(a, h[warp], eb, s0, n, lane);
  }
  emit_units(a, cnt, off, toff, blockIdx.x * kScanThreads + tid, gridDim.x * kScanThreads);
}

// ---------------------------------------------------------------- combine
// y[t] = bf16([x[t]] + s[t] + sum_j e[inv[t*K + j]]), summed in that order in
// fp32.  Each thread handles 8 consecutive columns.
__global__ void __launch_bounds__(128) combine_kernel(CombineArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int t = blockIdx.y;
  const int c8 = blockIdx.x * 128 + threadIdx.x;
  if (c8 * 8 >= a.D) return;
  const size_t base = static_cast<size_t>(t) * a.D + c8 * 8;
  float acc[8];
  const float4 s0 = __ldg(reinterpret_cast<const float4*>(a.s + base));
  const float4 s1 = __ldg(reinterpret_cast<const float4*>(a.s + base) + 1);
  acc[0] = s0.x; acc[1] = s0.y; acc[2] = s0.z; acc[3] = s0.w;
  acc[4] = s1.x; acc[5] = s1.y; acc[6] = s1.z; acc[7] = s1.w;
  // the k rows in order, their loads in flight together (8 at a time)
  for (int j0 = 0; j0 < a.K; j0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[j] = make_uint4(0, 0, 0, 0);
      if (j0 + j < a.K) {
        const int pos = __ldg(a.inv + t * a.K + j0 + j);
        v[j] = __ldg(reinterpret_cast<const uint4*>(a.e + static_cast<size_t>(pos) * a.D + c8 * 8));
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j0 + j >= a.K) break;
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16f(w[i] & 0xffffu);
        acc[2 * i + 1] += bf16f(w[i] >> 16);
      }
    }
  }
  if (a.residual) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.x + base));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] += bf16f(w[i] & 0xffffu);
      acc[2 * i + 1] += bf16f(w[i] >> 16);
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = static_cast<uint32_t>(f32_to_bf16(acc[2 * i])) |
           (static_cast<uint32_t>(f32_to_bf16(acc[2 * i + 1])) << 16);
  *reinterpret_cast<uint4*>(a.y + base) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace

int prefill_route(const RouteArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int e = launch_pdl(tok_prep_kernel, dim3((a.T + 7) / 8), dim3(256), 0, s, a.x, a.T, a.D,
                     a.prenorm, a.rms_eps, reinterpret_cast<__half*>(a.x16), a.sigma, a.rscale,
                     a.hscale);
  if (e) return e;
  e = router_tc_launch(*a.wmap, *a.xmap, a.T, a.E, a.D, a.nsplit, a.partials, a.status,
                       a.timeout_ns, stream);
  if (e) return e;
  const dim3 grid((a.T + 7) / 8);
  if (a.E <= 128)
    return launch_pdl(router_topk_kernel<4>, grid, dim3(256), 0, s, a.partials, a.nsplit, a.T, a.E,
                      a.K, a.sigma, a.logit_bias, a.forced, a.ids, a.wts);
  return launch_pdl(router_topk_kernel<kMaxPrefillExperts / 32>, grid, dim3(256), 0, s, a.partials,
                    a.nsplit, a.T, a.E, a.K, a.sigma, a.logit_bias, a.forced, a.ids, a.wts);
}

int bucket_blocks(int n) { return (n + kBkBlockSeg - 1) / kBkBlockSeg; }

int prefill_bucket(const BucketArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n = a.T * a.K;
  if (n <= kSmallN)
    return launch_pdl(bk_small_kernel, dim3(kSmallBlocks), dim3(kScanThreads), 0, s, a);
  const int nb = bucket_blocks(n);
  int e = launch_pdl(bk_hist_kernel, dim3(nb), dim3(kBkThreads), 0, s, a);
  if (!e) e = launch_pdl(bk_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, a, nb);
  if (!e) e = launch_pdl(bk_place_kernel, dim3(nb), dim3(kBkThreads), 0, s, a);
  return e;
}

int prefill_combine(const CombineArgs& a, void* stream) {
  const dim3 grid((a.D / 8 + 127) / 128, a.T);
  return launch_pdl(combine_kernel, grid, dim3(128), 0, static_cast<cudaStream_t>(stream), a);
}

}  // namespace moe
