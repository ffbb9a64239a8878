// Grouped GEMM of the multi-token layer step on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// One work unit = one 128-row tile of one 4-bit weight matrix (an expert's
// interleaved gate/up rows, its down rows, or the shared expert's) against the
// unit's activation rows: the tokens routed to that expert, in bucket order,
// or a tile of all tokens for the shared expert.  The weight tile is the MMA's
// M side (128) and the tokens its N side (16 up to the plan's width in steps
// of 16), so the tile shape follows the ragged per-expert token counts without
// padding M.  The kernel is a template over that width (Tile below: 160, 128
// or 32 tokens), chosen by the host from the batch size.
//
// The dequantised weights never touch shared memory: the dequantisation
// warps write them straight into tensor memory, and the MMA reads its A
// operand from there (only the activations come from shared memory).
// Tensor memory (512 columns): two accumulator sets (the epilogue drains one
// unit while the MMA fills the next) and the A stages.  The A and B rings
// advance in stages of two or four 64-column K blocks, so that each role
// synchronises once per stage.
//
// Per CTA (persistent, one per SM, 19 warps):
//   warp 0       weight loader: packed 4-bit codes (128 B x 128 rows, 128-byte
//                swizzle) and scale/bias words (16 B x 128 rows) of a
//                256-column slice of the weight tile -> P ring
//   warp 18      activation loader: the stage's tiles (64 fp16 columns x the
//                unit's rows, 128-byte swizzle, the UMMA K-major layout) -> B
//                ring, independent of the P ring
//   warp 1       MMA: the whole warp waits, one elected lane issues the
//                stage's tcgen05.mma kind::f16 (M=128, N=tokens, K=16, A in
//                tensor memory) and its commits; fp32 accumulators in tensor
//                memory
//   warps 2-9    dequantisation: the two warps of tensor-memory lane quarter
//                w%4 take the two 32-column halves of its 32 rows; per
//                64-column block each thread turns its codes into fp16 A
//                values (gate/up: fp16(s q), the biases entering through one
//                more K block of the tokens' group sums; down: fp16(s q + b))
//                and stores them into the A stage
//   warps 10-17  epilogue: tensor memory -> registers; gate/up units write
//                h = gelu(g) * u (fp16, times a per-token power of two that
//                keeps it in range), down units undo that factor and write the
//                routing-weighted expert output (bf16) or the shared output
//                (fp32), each chunk transposed through shared memory into
//                16-byte row-segment stores
// Rings are mbarrier-pipelined; every wait is bounded in time and a wait that
// runs out sets the status word and ends the CTA's work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "launch.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kTU = kTilesPerUnit;                 // weight tiles per unit
constexpr int kPCodeBytes = 128 * 128;             // 128 rows x 256 columns of 4-bit codes
constexpr int kPSbBytes = 128 * 16;                // 128 rows x 4 scale/bias words
constexpr int kPTile = kPCodeBytes + kPSbBytes;    // 18 KB per weight tile
constexpr int kPBytes = kTU * kPTile;              // the unit's weight tiles per P stage
constexpr int kTmemCols = 512;
constexpr int kAStage = kTU * 32;                  // per K block and tile: 32 columns (64 fp16)
// A and B rings advance by stages of several 64-column K blocks (the plan's
// kStageKB: two, or four = a whole weight slice), so that one wait, one pair
// of commits and one arrival per role cover them all; a unit's last stage of
// weight columns may hold fewer.
constexpr int kDqWarps = 8, kEpiWarps = 8;
constexpr int kGemmThreads = (3 + kDqWarps + kEpiWarps) * 32;  // + the activation loader warp
constexpr int kBLoadWarp = 2 + kDqWarps + kEpiWarps;
constexpr int kEpiWarp0 = 2 + kDqWarps;
constexpr int kStageBytes = 2048;                  // per epilogue warp: output transpose
// 64 b per row and group of the gate/up unit in flight, kept by the
// dequantisation threads for the group-sum K block (144-byte rows: the
// 16-byte loads stay aligned and the 2-byte stores of a warp's 32 rows spread
// over 8 banks).
constexpr int kGsumPitch = 144;
constexpr int kGsumBytes = 128 * kGsumPitch;

// The kernel's plan for units of up to kUT activation rows.  Tensor memory
// holds two accumulator sets of kUT columns and A stages in the rest; shared
// memory holds the P (weight), B (activation) and epilogue buffers.  Three
// plans: wide (kUT = 160, stages of two K blocks) for more than 128 tokens,
// medium (128) and narrow (32, for at most 32 tokens), both with stages of a
// whole 4-block weight slice.  A narrower plan turns the columns and bytes
// that wide units need into longer stages and deeper rings, which cut the
// per-block hand-offs that bound a unit of few tokens.
template <int kUT>
struct Tile {
  static constexpr int kUnit = kUT;
  static constexpr int kStageKB = kUT > 128 ? 2 : 4;  // K blocks per A/B stage
  static constexpr int kBBytes = kUT * 128;          // one K block's tile: tokens x 64 fp16
  static constexpr int kBStage = kStageKB * kBBytes;
  static constexpr int kAccCols = kUT;               // per tile
  static constexpr int kAccSet = kTU * kAccCols;     // one unit's accumulators
  static constexpr int kACol0 = 2 * kAccSet;         // A stages after the two sets
  static constexpr int kAStageCols = kStageKB * kAStage;
  static constexpr int kNA = (kTmemCols - kACol0) / kAStageCols;
  static constexpr int kNP = kUT > 128 ? 3 : (kUT > 32 ? 2 : 4);
  static constexpr int kNB = kUT > 128 ? 3 : (kUT > 32 ? 2 : 6);
  static_assert(kNA >= 2 && kACol0 + kNA * kAStageCols <= kTmemCols, "tensor memory plan");
  struct Bars {
    uint64_t p_full[kNP], p_empty[kNP];
    uint64_t a_full[kNA], a_empty[kNA];
    uint64_t b_full[kNB], b_empty[kNB];
    uint64_t acc_full[2], acc_empty[2];
    uint32_t tmem_base;
    int abort;
  };
  static constexpr int kMetaBytes = 2 * kUT * 4;     // per-column factors
  static constexpr int kSmemBytes = kNP * kPBytes + kNB * kBStage + kMetaBytes +
                                    kEpiWarps * kStageBytes + kGsumBytes +
                                    1024 /*Bars*/ + 1024 /*alignment slack*/;
  static_assert(sizeof(Bars) <= 1024, "barrier block");
};
using WideTile = Tile<kUnitTokens>;
using MediumTile = Tile<128>;
using NarrowTile = Tile<32>;
static_assert(WideTile::kSmemBytes <= 227 * 1024 && MediumTile::kSmemBytes <= 227 * 1024 &&
                  NarrowTile::kSmemBytes <= 227 * 1024,
              "shared memory plan");

__device__ __forceinline__ float gelu_tanh(float x) {
  const float c2 = 1.5957691216057308f;  // 2 sqrt(2/pi)
  const float u2 = c2 * fmaf(0.044715f * x, x * x, x);
  return __fdividef(x, 1.f + __expf(-u2));
}

// 16 consecutive per-column factors of the unit from shared memory into
// registers (broadcast vector loads), ahead of the chunk's stores to the
// staging tile, so that no factor load waits behind a store.
__device__ __forceinline__ void load16(const float* src, float (&d)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 v = reinterpret_cast<const float4*>(src)[i];
    d[4 * i] = v.x;
    d[4 * i + 1] = v.y;
    d[4 * i + 2] = v.z;
    d[4 * i + 3] = v.w;
  }
}

// Bounded mbarrier wait shared by all roles: on expiry record a timeout and
// make every role stop.
template <class BarsT>
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                         BarsT* bars) {
  if (mbar_wait(bar, parity, p.timeout_ns, &bars->abort)) return true;
  if (!bars->abort) atomicCAS(p.status, DEV_OK, DEV_TIMEOUT);
  bars->abort = 1;
  return false;
}

__device__ __forceinline__ int unit_nmma(int n) { return (n + 15) & ~15; }

// ---------------------------------------------------------------- roles

// Position in an mbarrier-pipelined ring of N stages: the stage and the
// parity of its current fill.
struct RingPos {
  int s = 0;
  uint32_t ph = 0;  // parity of the stage's current fill
  template <int N>
  __device__ __forceinline__ void next() {
    if (++s == N) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// K blocks in the A/B stage that starts at K block kb of unit `un`: the
// plan's kStageKB, fewer at the end of the weight columns, and one for the
// group-sum block.  The dequantisation forms the same stages inside each
// 4-block weight slice (only a unit's last slice holds fewer than four).
template <class T>
__device__ __forceinline__ int stage_blocks(const GemmUnit& un, const GemmParams& p, int kb) {
  const int nmain = p.K[un.kind] / 64;
  if (kb >= nmain) return 1;  // the group-sum block
  return min(T::kStageKB, nmain - kb);
}

// Two loader threads, so that neither ring waits for the other: the weight
// slices (P ring, one stage per 256 columns) and the activation tiles (B
// ring, one stage per 64-column block) are issued independently, each as far
// ahead as its ring allows.
template <class T>
__device__ void role_tma_p(const GemmParams& p, uint8_t* P, typename T::Bars* bars, int nU) {
  uint32_t pc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int np = (K + 255) / 256;
    const void* tc = &p.tm_code[un.kind];
    const void* ts = &p.tm_sb[un.kind];
    for (int sp = 0; sp < np; ++sp, ++pc) {
      const int st = pc % T::kNP;
      if (!wait_bar(&bars->p_empty[st], ((pc / T::kNP) & 1) ^ 1, p, bars)) return;
      uint8_t* dst = P + st * kPBytes;
      mbar_arrive_expect_tx(&bars->p_full[st], un.nmt * kPTile);
      const int xc = sp * 128, xs = K / 2 + sp * 16;
      for (int m = 0; m < un.nmt; ++m) {
        const int y = (un.mt + m) * 128;
        if (un.kind == 0) {
          tma_load_3d(dst + m * kPTile, tc, xc, y, un.expert, &bars->p_full[st]);
          tma_load_3d(dst + m * kPTile + kPCodeBytes, ts, xs, y, un.expert, &bars->p_full[st]);
        } else {
          tma_load_2d(dst + m * kPTile, tc, xc, y, &bars->p_full[st]);
          tma_load_2d(dst + m * kPTile + kPCodeBytes, ts, xs, y, &bars->p_full[st]);
        }
      }
    }
  }
  // drain: copies still in flight must land before the CTA exits
  for (uint32_t q = pc > T::kNP ? pc - T::kNP : 0; q < pc; ++q)
    mbar_wait(&bars->p_full[q % T::kNP], (q / T::kNP) & 1, p.timeout_ns, nullptr);
}

template <class T>
__device__ void role_tma_b(const GemmParams& p, uint8_t* B, typename T::Bars* bars, int nU) {
  uint32_t bc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int nkb = p.K[un.kind] / 64 + p.gsum;  // the group sums follow the K columns
    if (unit_nmma(un.n) > T::kUnit) {  // wider than this plan's stages (never launched so)
      if (!bars->abort) atomicCAS(p.status, DEV_OK, DEV_BAD_ID);
      bars->abort = 1;
      break;
    }
    int box = 0;  // the lowest tile that holds the MMA's rows
    while (box + 1 < kNBox && box_rows(box) < unit_nmma(un.n)) ++box;
    const void* tb = &p.tm_b[un.kind][box];
    const uint32_t bytes = box_rows(box) * 128;
    for (int kb = 0; kb < nkb; ++bc) {
      const int nb = stage_blocks<T>(un, p, kb);
      const int bs = bc % T::kNB;
      if (!wait_bar(&bars->b_empty[bs], ((bc / T::kNB) & 1) ^ 1, p, bars)) return;
      mbar_arrive_expect_tx(&bars->b_full[bs], nb * bytes);
      for (int i = 0; i < nb; ++i)
        tma_load_2d(B + bs * T::kBStage + i * T::kBBytes, tb, (kb + i) * 64, un.row0,
                    &bars->b_full[bs]);
      kb += nb;
    }
  }
  for (uint32_t q = bc > T::kNB ? bc - T::kNB : 0; q < bc; ++q)
    mbar_wait(&bars->b_full[q % T::kNB], (q / T::kNB) & 1, p.timeout_ns, nullptr);
}

// Dequantisation (8 warps): the two warps of tensor-memory lane quarter w%4
// take the two 32-column halves of its 32 rows.  Per 64-column block each
// thread turns its row's 32 codes into fp16 w = fp16(s q + b) (one rounding)
// and stores them into the block's A stage.  Blocks go two at a time while
// the weight slice holds two more: the warps are bound by latency (barrier
// waits, shared-memory loads, the tensor-memory store and its completion),
// and a pair overlaps those of two blocks and halves the synchronisation per
// block.
// One half K block (32 columns) of this thread's row as fp16 A values, from its
// packed codes and the group's scale/bias word.  kGsum: A = fp16(s q), as
// fp16((1024 + q) s - 1024 s) in one fused multiply-add (exact before its one
// rounding); otherwise A = fp16(s q + b) (q = (1024 + q) - 1024 exactly, then
// one fused multiply-add).
template <bool kGsum>
__device__ __forceinline__ void dequant32(const uint8_t* codes, const uint32_t* sbw, int row,
                                          int half, int sb, __half2 k1024, uint32_t (&o)[16]) {
  const uint32_t word = sbw[row * 4 + sb];
  const __half2 s2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(word & 0xffffu)));
  const __half2 b2 = kGsum ? __hmul2(s2, __hneg2(k1024))  // -1024 s, exact
                           : __half2half2(__ushort_as_half(static_cast<unsigned short>(word >> 16)));
  // packed chunk c (32 columns) of this row, stored at chunk c ^ (row & 7)
  const int c = 2 * sb + half;
  const uint4 wq = *reinterpret_cast<const uint4*>(codes + row * 128 + ((c ^ (row & 7)) << 4));
  const uint32_t ws[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    // word j: columns 8j..8j+7 of the chunk; byte i = col i (low) | col 4+i (high)
    const uint32_t lo = ws[j] & 0x0F0F0F0Fu;
    const uint32_t hi = (ws[j] >> 4) & 0x0F0F0F0Fu;
    // fp16 1024 + q pairs: bytes (q, 0x64) per half
    const uint32_t mm[4] = {__byte_perm(lo, 0x64646464u, 0x5140), __byte_perm(lo, 0x64646464u, 0x7362),
                            __byte_perm(hi, 0x64646464u, 0x5140), __byte_perm(hi, 0x64646464u, 0x7362)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 m = *reinterpret_cast<const __half2*>(&mm[i]);
      const __half2 v = kGsum ? __hfma2(m, s2, b2) : __hfma2(__hsub2(m, k1024), s2, b2);
      o[4 * j + i] = *reinterpret_cast<const uint32_t*>(&v);
    }
  }
}

// 64 b of group g (K block g) into this thread's row of the group-sum
// scratch, if g is in this thread's half of the K range.
__device__ __forceinline__ void keep_bias(const uint32_t* sbw, uint8_t* gsb, int row, int half,
                                          int g, int sb) {
  if ((g >> 5) != half) return;
  const __half b = __ushort_as_half(static_cast<unsigned short>(sbw[row * 4 + sb] >> 16));
  *reinterpret_cast<__half*>(gsb + row * kGsumPitch + 2 * g) = __hmul(b, __float2half(64.f));
}

// With kGsum (gate/up) each thread also keeps 64 b of the groups of its half
// of the K range (groups 32 half .. 32 half + 31) in its row of `gsb`, and after
// the unit's K blocks stores them as the group-sum block's A columns (zero
// past the last group); the activations' group sums form that block's B.
template <class T, bool kGsum>
__device__ void role_dequant(const GemmParams& p, const uint8_t* P, typename T::Bars* bars, int nU,
                             uint8_t* gsb) {
  static_assert(kTU == 1, "the dequantisation warps fill one weight tile per unit");
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = (w - 2) >> 2;       // 32-column half of the row
  const int qd = w & 3;                // tensor-memory lane quarter
  const int row = 32 * qd + lane;      // row of the weight tile
  const uint32_t tbase =
      bars->tmem_base + (static_cast<uint32_t>(32 * qd) << 16) + T::kACol0 + half * 16;
  static_assert(T::kStageKB == 2 || T::kStageKB == 4, "a stage is a pair or a weight slice");
  const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
  RingPos ra;
  uint32_t pc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int nkb = K / 64;
    const int np = (K + 255) / 256;
    for (int sp = 0; sp < np; ++sp, ++pc) {
      const int st = pc % T::kNP;
      if (!wait_bar(&bars->p_full[st], (pc / T::kNP) & 1, p, bars)) return;
      const int nsub = min(4, nkb - 4 * sp);
      const uint8_t* codes = P + st * kPBytes;
      const uint32_t* sbw = reinterpret_cast<const uint32_t*>(codes + kPCodeBytes);
      if constexpr (T::kStageKB == 4) {  // the slice is one stage: one wait, one arrival
        if (!wait_bar(&bars->a_empty[ra.s], ra.ph ^ 1u, p, bars)) return;
        const uint32_t ta = tbase + ra.s * T::kAStageCols;
        for (int sb = 0; sb < nsub; sb += 2) {
          uint32_t o0[16], o1[16];
          dequant32<kGsum>(codes, sbw, row, half, sb, k1024, o0);
          if (kGsum) keep_bias(sbw, gsb, row, half, 4 * sp + sb, sb);
          tmem_st16(ta + sb * kAStage, o0);
          if (sb + 1 < nsub) {
            dequant32<kGsum>(codes, sbw, row, half, sb + 1, k1024, o1);
            if (kGsum) keep_bias(sbw, gsb, row, half, 4 * sp + sb + 1, sb + 1);
            tmem_st16(ta + (sb + 1) * kAStage, o1);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->a_full[ra.s]);
        ra.next<T::kNA>();
      }
      for (int sb = 0; T::kStageKB == 2 && sb < nsub;) {
        if (sb + 1 < nsub) {  // a stage of two blocks
          if (!wait_bar(&bars->a_empty[ra.s], ra.ph ^ 1u, p, bars)) return;
          uint32_t o0[16], o1[16];
          dequant32<kGsum>(codes, sbw, row, half, sb, k1024, o0);
          dequant32<kGsum>(codes, sbw, row, half, sb + 1, k1024, o1);
          if (kGsum) keep_bias(sbw, gsb, row, half, 4 * sp + sb, sb);
          if (kGsum) keep_bias(sbw, gsb, row, half, 4 * sp + sb + 1, sb + 1);
          tmem_st16(tbase + ra.s * T::kAStageCols, o0);
          tmem_st16(tbase + ra.s * T::kAStageCols + kAStage, o1);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->a_full[ra.s]);
          ra.next<T::kNA>();
          sb += 2;
        } else {  // the unit's last block, alone in its stage
          if (!wait_bar(&bars->a_empty[ra.s], ra.ph ^ 1u, p, bars)) return;
          uint32_t o0[16];
          dequant32<kGsum>(codes, sbw, row, half, sb, k1024, o0);
          if (kGsum) keep_bias(sbw, gsb, row, half, 4 * sp + sb, sb);
          tmem_st16(tbase + ra.s * T::kAStageCols, o0);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->a_full[ra.s]);
          ra.next<T::kNA>();
          sb += 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_empty[st]);
    }
    if (kGsum) {  // the group-sum block: A columns 64 b_g of this half's groups
      const int ng = K / 64;
      if (!wait_bar(&bars->a_empty[ra.s], ra.ph ^ 1u, p, bars)) return;
      const uint4* src = reinterpret_cast<const uint4*>(gsb + row * kGsumPitch + half * 64);
      uint32_t o[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = src[i];
        o[4 * i] = v.x;
        o[4 * i + 1] = v.y;
        o[4 * i + 2] = v.z;
        o[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {  // column pair i holds groups 32 half + 2i, + 2i + 1
        const int g = 32 * half + 2 * i;
        if (g >= ng) o[i] = 0u;
        else if (g + 1 >= ng) o[i] &= 0xffffu;
      }
      tmem_st16(tbase + ra.s * T::kAStageCols, o);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->a_full[ra.s]);
      ra.next<T::kNA>();
    }
  }
}

// The MMA role runs on a whole warp: every lane waits, the warp stays
// converged, and one elected lane issues each K block's four MMAs and its two
// commits from a single instruction sequence.  A unit's K blocks run in a
// loop instantiated for its token count (the MMA's N, a multiple of 16), so
// the instruction descriptor is a constant, and the ring positions advance
// by increment: the warp shares its issue slots with dequantisation and
// epilogue warps, so every instruction it saves per K block keeps the tensor
// pipe fed.
template <class BarsT>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                          BarsT* bars) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, p, bars));
}


template <class T, int NMMA>
__device__ __forceinline__ bool mma_unit(const GemmParams& p, const GemmUnit& un,
                                         typename T::Bars* bars, uint32_t acc, uint32_t a_base,
                                         uint64_t bdesc0, int nkb, RingPos& ra, RingPos& rb) {
  constexpr uint32_t idesc = tc_idesc_f16(128, NMMA);
  for (int kb = 0; kb < nkb;) {
    const int nb = stage_blocks<T>(un, p, kb);
    // both stages are usually ready: probe them together, and take the
    // bounded waits only when one is not
    if (!__all_sync(0xffffffffu,
                    mbar_test_wait2(&bars->a_full[ra.s], ra.ph, &bars->b_full[rb.s], rb.ph))) {
      if (!warp_wait(&bars->a_full[ra.s], ra.ph, p, bars)) return false;
      if (!warp_wait(&bars->b_full[rb.s], rb.ph, p, bars)) return false;
    }
    tc_fence_after();
    const uint32_t a0 = a_base + ra.s * T::kAStageCols;
    const uint64_t b0 = bdesc0 + static_cast<uint64_t>(rb.s * (T::kBStage >> 4));
    if (T::kStageKB == 4 && nb > 2)  // blocks 0 and 1 first, without the commits
      tc_stage_ts_warp(acc, a0, b0, T::kBBytes >> 4, idesc, kb != 0, 1u, 0u, &bars->a_empty[ra.s],
                       &bars->b_empty[rb.s]);
    const int j0 = (T::kStageKB == 4 && nb > 2) ? 2 : 0;  // blocks j0, j0 + 1 (if any), commits
    tc_stage_ts_warp(acc, a0 + j0 * kAStage, b0 + static_cast<uint64_t>(j0 * (T::kBBytes >> 4)),
                     T::kBBytes >> 4, idesc, (kb + j0) != 0, nb - j0 == 2, 1u,
                     &bars->a_empty[ra.s], &bars->b_empty[rb.s]);
    ra.next<T::kNA>();
    rb.next<T::kNB>();
    kb += nb;
  }
  return true;
}

template <class T>
__device__ void role_mma(const GemmParams& p, uint8_t* B, typename T::Bars* bars, int nU) {
  static_assert(T::kUnit % 16 == 0 && T::kUnit <= 256, "unit token count");
  static_assert(kTU == 1, "the MMA loop issues one weight tile per unit");
  const uint32_t tmem = bars->tmem_base;
  const uint64_t bdesc0 = tc_desc_sw128(smem_u32(B));
  RingPos ra, rb;
  uint32_t uc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x, ++uc) {
    const GemmUnit un = p.units[u];
    const int nkb = p.K[un.kind] / 64 + p.gsum;  // + the group-sum block
    const uint32_t acc = tmem + (uc & 1) * T::kAccSet;  // this unit's accumulator set
    // (an injected stall waits for the phase before, which never completes)
    const uint32_t par = ((uc >> 1) & 1) ^ (p.stall ? 0u : 1u);
    if (!warp_wait(&bars->acc_empty[uc & 1], par, p, bars)) return;
    tc_fence_after();
    const uint32_t a_base = tmem + T::kACol0;
    const int n16 = unit_nmma(un.n) >> 4;
    if (n16 < 1 || 16 * n16 > T::kUnit) {  // never emitted by the bucketing
      if (!bars->abort) atomicCAS(p.status, DEV_OK, DEV_BAD_ID);
      bars->abort = 1;
      return;
    }
    bool ok = false;
    switch (n16) {
#define MOE_MMA_CASE(c)                                                                   \
  case c:                                                                                 \
    if constexpr (16 * (c) <= T::kUnit)                                                \
      ok = mma_unit<T, 16 * (c)>(p, un, bars, acc, a_base, bdesc0, nkb, ra, rb);         \
    break;
      MOE_MMA_CASE(1) MOE_MMA_CASE(2) MOE_MMA_CASE(3) MOE_MMA_CASE(4) MOE_MMA_CASE(5)
      MOE_MMA_CASE(6) MOE_MMA_CASE(7) MOE_MMA_CASE(8) MOE_MMA_CASE(9) MOE_MMA_CASE(10)
      MOE_MMA_CASE(11) MOE_MMA_CASE(12) MOE_MMA_CASE(13) MOE_MMA_CASE(14) MOE_MMA_CASE(15)
      MOE_MMA_CASE(16)
#undef MOE_MMA_CASE
      default: break;
    }
    if (!ok) return;  // a wait ran out
    tc_commit_warp(&bars->acc_full[uc & 1]);
  }
  // the last commits must complete before the CTA exits
  if (uc > 0) mbar_wait(&bars->acc_full[(uc - 1) & 1], ((uc - 1) >> 1) & 1, p.timeout_ns, nullptr);
}

// Epilogue (8 warps): warp w reads tensor-memory lanes of quarter w % 4 and
// the 32-column chunks of parity (w - 10) / 4.  Per unit, per-column (token)
// factors are first gathered into shared memory.  A thread holds one output
// feature for 32 tokens; the warp transposes each chunk through its own
// 2 KB of shared memory so that the global stores are 16-byte vectors
// covering whole output row segments (one token row per group of lanes).
__device__ __forceinline__ void epi_sync() { named_sync(1, kEpiWarps * 32); }

template <class T>
__device__ void role_epilogue(const GemmParams& p, typename T::Bars* bars, float* meta, uint8_t* stage,
                              int nU) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = w & 3;
  const int chalf = (w - kEpiWarp0) >> 2;
  const int te = threadIdx.x - kEpiWarp0 * 32;  // 0..255
  const uint32_t tmem = bars->tmem_base;
  uint8_t* stg = stage + (w - kEpiWarp0) * kStageBytes;
  uint32_t uc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x, ++uc) {
    const GemmUnit un = p.units[u];
    for (int col = te; col < un.n; col += kEpiWarps * 32) {
      const int brow = un.row0 + col;
      if (p.mode == 0) {
        const int tok = un.kind == 0 ? p.perm[brow] / p.topk : brow;
        meta[col] = p.sigma[tok];
        meta[T::kUnit + col] = p.hscale[tok];
      } else if (un.kind == 0) {
        const int a = p.perm[brow];
        meta[col] = p.wts[a] / p.hscale[a / p.topk];
      } else {
        meta[col] = 1.f / p.hscale[brow];
      }
    }
    if (!wait_bar(&bars->acc_full[uc & 1], (uc >> 1) & 1, p, bars)) return;
    tc_fence_after();
    epi_sync();
    const uint32_t acc = tmem + (uc & 1) * T::kAccSet;
    // the unit's 32-column chunks (3 per tile), alternating between the two
    // warps of this lane quarter
    constexpr int kChunks = T::kAccCols / 32;
    for (int idx = chalf; idx < un.nmt * kChunks; idx += 2) {
      const int m = idx / kChunks, c0 = (idx % kChunks) * 32;
      if (c0 >= un.n) continue;
      const int mt = un.mt + m;
      {
        uint32_t r[32];
        tmem_ld32(acc + (static_cast<uint32_t>(32 * q) << 16) + m * T::kAccCols + c0, r);
        tmem_ld_wait();
        if (p.mode == 0) {
          // rows 2j / 2j+1 of the tile are gate / up of output column j:
          // the even lane takes columns c0..c0+15, the odd lane c0+16..c0+31.
          // Stage: [32 tokens][16 columns] fp16 (32-byte rows).
          const int jj = lane >> 1;
          const bool odd = lane & 1;
          __half* sh = reinterpret_cast<__half*>(stg);
          float sgv[16], hsv[16];
          load16(meta + c0 + (odd ? 16 : 0), sgv);
          load16(meta + T::kUnit + c0 + (odd ? 16 : 0), hsv);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float mine_lo = __uint_as_float(r[i]), mine_hi = __uint_as_float(r[16 + i]);
            const float recv = __shfl_xor_sync(0xffffffffu, odd ? mine_lo : mine_hi, 1);
            const float g = odd ? recv : mine_lo;
            const float v = odd ? mine_hi : recv;
            const int tc = (odd ? 16 : 0) + i;  // token within the chunk
            const int col = c0 + tc;
            float h = 0.f;
            if (col < un.n) h = gelu_tanh(g * sgv[i]) * (v * sgv[i]) * hsv[i];
            sh[tc * 16 + jj] = __float2half_rn(fminf(fmaxf(h, -65504.f), 65504.f));
          }
          __syncwarp();
          __half* hout = reinterpret_cast<__half*>(p.hout[un.kind]);
          const int j0 = mt * 64 + 16 * q;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int tc = 16 * k + (lane >> 1);
            const int col = c0 + tc;
            if (col < un.n) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + tc * 32 + (lane & 1) * 16);
              *reinterpret_cast<uint4*>(hout + static_cast<int64_t>(un.row0 + col) * p.hld[un.kind] +
                                        j0 + (lane & 1) * 8) = v;
            }
          }
          __syncwarp();
        } else if (un.kind == 0) {
          // routed down: bf16 [32 tokens][32 features] (64-byte rows)
          const int d0 = mt * 128 + 32 * q;
          __nv_bfloat16* sb = reinterpret_cast<__nv_bfloat16*>(stg);
          float mv[2][16];
          load16(meta + c0, mv[0]);
          load16(meta + c0 + 16, mv[1]);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = c0 + i;
            const float v = col < un.n ? __uint_as_float(r[i]) * mv[i >> 4][i & 15] : 0.f;
            sb[i * 32 + lane] = __float2bfloat16_rn(v);
          }
          __syncwarp();
          __nv_bfloat16* eout = reinterpret_cast<__nv_bfloat16*>(p.eout);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int tc = 8 * k + (lane >> 2);
            const int col = c0 + tc;
            if (col < un.n) {
              const uint4 v = *reinterpret_cast<const uint4*>(stg + tc * 64 + (lane & 3) * 16);
              *reinterpret_cast<uint4*>(eout + static_cast<int64_t>(un.row0 + col) * p.D + d0 +
                                        (lane & 3) * 8) = v;
            }
          }
          __syncwarp();
        } else {
          // shared down: fp32 [16 tokens][32 features] (128-byte rows), twice
          const int d0 = mt * 128 + 32 * q;
          float* sf = reinterpret_cast<float*>(stg);
          float mv[2][16];
          load16(meta + c0, mv[0]);
          load16(meta + c0 + 16, mv[1]);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int col = c0 + 16 * hh + i;
              sf[i * 32 + lane] = col < un.n ? __uint_as_float(r[16 * hh + i]) * mv[hh][i] : 0.f;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int tc = 4 * k + (lane >> 3);
              const int col = c0 + 16 * hh + tc;
              if (col < un.n) {
                const uint4 v = *reinterpret_cast<const uint4*>(stg + tc * 128 + (lane & 7) * 16);
                *reinterpret_cast<uint4*>(p.sout + static_cast<int64_t>(un.row0 + col) * p.D + d0 +
                                          (lane & 7) * 4) = v;
              }
            }
            __syncwarp();
          }
        }
      }
    }
    tc_fence_before();
    epi_sync();  // all reads of this unit's accumulator and factors are done
    if (te == 0) mbar_arrive(&bars->acc_empty[uc & 1]);
  }
}

template <class T>
__global__ void __launch_bounds__(kGemmThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  uint8_t* P = smem;
  uint8_t* B = P + T::kNP * kPBytes;
  float* meta = reinterpret_cast<float*>(B + T::kNB * T::kBStage);
  uint8_t* stage = B + T::kNB * T::kBStage + T::kMetaBytes;
  uint8_t* gsb = stage + kEpiWarps * kStageBytes;
  typename T::Bars* bars = reinterpret_cast<typename T::Bars*>(gsb + kGsumBytes);
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < T::kNP; ++i) {
      mbar_init(&bars->p_full[i], 1);
      mbar_init(&bars->p_empty[i], kDqWarps);
    }
    for (int i = 0; i < T::kNA; ++i) {
      mbar_init(&bars->a_full[i], kDqWarps);
      mbar_init(&bars->a_empty[i], 1);
    }
    for (int i = 0; i < T::kNB; ++i) {
      mbar_init(&bars->b_full[i], 1);
      mbar_init(&bars->b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 1);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (w == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();  // the units, activations and factors come from the kernels before
  grid_dep_launch();
  const int nU = *p.n_units;
  if (w == 0) {
    if ((threadIdx.x & 31) == 0) role_tma_p<T>(p, P, bars, nU);
  } else if (w == kBLoadWarp) {
    if ((threadIdx.x & 31) == 0) role_tma_b<T>(p, B, bars, nU);
  } else if (w == 1) {
    role_mma<T>(p, B, bars, nU);
  } else if (w < kEpiWarp0) {
    if (p.gsum) role_dequant<T, true>(p, P, bars, nU, gsb);
    else role_dequant<T, false>(p, P, bars, nU, gsb);
  } else {
    role_epilogue<T>(p, bars, meta, stage, nU);
  }
  tc_fence_before();
  __syncthreads();
  if (w == 1) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------ router GEMM
// partial[split][t][e] = sum over the split's 64-column blocks of
// (Whi[e] + Wlo[e]) . x16[t], fp32 accumulation on the tensor cores.  The
// 8-bit router weight w = s q + b (fp32) is held as two fp16 parts, Whi =
// fp16(w) and Wlo = fp16(w - Whi), so the pair carries w to about 2^-22 of
// its size, and x16 = f_t x is exact: the logits come out as accurate as an
// fp32 product, which the exact top-k selection needs.  CTA = 128 experts x
// 128 tokens x one range of 64-column blocks; warp 0 lane 0 issues TMA
// loads, warp 1 lane 0 the MMAs (M=128, N=128, K=16, both operands in shared
// memory), then all four warps write their tensor-memory lane quarter.
constexpr int kRtStages = 4;
constexpr int kRtTile = 128 * 128;        // 128 rows x 64 fp16 (128-byte swizzle)
constexpr int kRtStage = 3 * kRtTile;     // Whi, Wlo, x16
constexpr int kRtSmem = kRtStages * kRtStage + 1024 /*bars*/ + 1024 /*alignment*/;

struct RtBars {
  uint64_t full[kRtStages], empty[kRtStages], done;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ bool rt_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns,
                                        RtBars* b, uint32_t* status) {
  if (mbar_wait(bar, parity, timeout_ns, &b->abort)) return true;
  if (!b->abort) atomicCAS(status, DEV_OK, DEV_TIMEOUT);
  b->abort = 1;
  return false;
}

__global__ void __launch_bounds__(128, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                     int T, int E, int Epad, int nkb, int kbs, float* __restrict__ partials,
                     uint32_t* status, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  RtBars* bars = reinterpret_cast<RtBars*>(smem + kRtStages * kRtStage);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128, mt = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * kbs, kb1 = min(nkb, kb0 + kbs);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (w == 0) {
    tmem_alloc(&bars->tmem, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t acc = bars->tmem;
  if (w == 0 && lane == 0) {
    // the weight tiles of the first stages depend on no earlier kernel: they
    // are requested before the wait for the token tiles
    const int npre = min(kRtStages, kb1 - kb0);
    for (int i = 0; i < npre; ++i) {
      uint8_t* dst = smem + i * kRtStage;
      mbar_arrive_expect_tx(&bars->full[i], kRtStage);
      tma_load_2d(dst, &wmap, (kb0 + i) * 64, mt * 128, &bars->full[i]);
      tma_load_2d(dst + kRtTile, &wmap, (kb0 + i) * 64, Epad + mt * 128, &bars->full[i]);
    }
    grid_dep_wait();
    grid_dep_launch();
    for (int kb = kb0; kb < kb1; ++kb) {
      const int i = kb - kb0, st = i % kRtStages;
      uint8_t* dst = smem + st * kRtStage;
      if (i >= npre) {
        if (!rt_wait(&bars->empty[st], ((i / kRtStages) & 1) ^ 1, timeout_ns, bars, status)) break;
        mbar_arrive_expect_tx(&bars->full[st], kRtStage);
        tma_load_2d(dst, &wmap, kb * 64, mt * 128, &bars->full[st]);
        tma_load_2d(dst + kRtTile, &wmap, kb * 64, Epad + mt * 128, &bars->full[st]);
      }
      tma_load_2d(dst + 2 * kRtTile, &xmap, kb * 64, t0, &bars->full[st]);
    }
  } else {
    grid_dep_wait();
    grid_dep_launch();
  }
  if (w == 1 && lane == 0) {
    const uint32_t idesc = tc_idesc_f16(128, 128);
    const uint64_t d0 = tc_desc_sw128(smem_u32(smem));
    bool ok = true;
    for (int kb = kb0; kb < kb1 && ok; ++kb) {
      const int i = kb - kb0, st = i % kRtStages;
      if (!rt_wait(&bars->full[st], (i / kRtStages) & 1, timeout_ns, bars, status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint64_t dh = d0 + static_cast<uint64_t>(st * (kRtStage >> 4));
      const uint64_t dl = dh + (kRtTile >> 4), dx = dh + 2 * (kRtTile >> 4);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        tc_mma_f16(acc, dh + 2 * kk, dx + 2 * kk, idesc, (i | kk) != 0);
        tc_mma_f16(acc, dl + 2 * kk, dx + 2 * kk, idesc, 1u);
      }
      tc_commit(&bars->empty[st]);
    }
    tc_commit(&bars->done);
  }
  // epilogue: warp w reads tensor-memory lanes 32w.. (experts), 32 tokens per load
  __syncwarp();
  const bool done = __all_sync(0xffffffffu, rt_wait(&bars->done, 0, timeout_ns, bars, status));
  if (done) {
    tc_fence_after();
    const int e = mt * 128 + 32 * w + lane;
    for (int c0 = 0; c0 < 128; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(acc + (static_cast<uint32_t>(32 * w) << 16) + c0, r);
      tmem_ld_wait();
      if (e < E) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = t0 + c0 + i;
          if (t < T) partials[(static_cast<int64_t>(split) * T + t) * E + e] = __uint_as_float(r[i]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (w == 0) {
    tc_fence_after();
    tmem_dealloc(acc, 128);
  }
}

// Token rows of x16 into bucket order (the routed gate/up activation operand).
// One warp per output row: a lane's 16-byte pieces of the row are all loaded
// before any is stored, so a row's reads are in flight together.
constexpr int kGatherWarps = 8, kGatherV = 13;  // rows of up to 32 * 13 uint4 (3,328 fp16)
__global__ void __launch_bounds__(kGatherWarps * 32) gather_rows_kernel(
    const uint4* __restrict__ x16, int D8, const int32_t* __restrict__ perm, int topk, int rows,
    uint4* __restrict__ out) {
  grid_dep_wait();
  grid_dep_launch();
  const int pos = blockIdx.x * kGatherWarps + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (pos >= rows) return;
  const int tok = perm[pos] / topk;
  const uint4* src = x16 + static_cast<int64_t>(tok) * D8;
  uint4* dst = out + static_cast<int64_t>(pos) * D8;
  uint4 v[kGatherV];
#pragma unroll
  for (int j = 0; j < kGatherV; ++j)
    if (lane + 32 * j < D8) v[j] = __ldg(src + lane + 32 * j);
#pragma unroll
  for (int j = 0; j < kGatherV; ++j)
    if (lane + 32 * j < D8) dst[lane + 32 * j] = v[j];
}

template <class T>
int launch_gemm(const GemmParams& p, int grid, cudaStream_t s) {
  const int e = set_smem_limit(reinterpret_cast<const void*>(gemm_tc_kernel<T>), T::kSmemBytes);
  if (e != 0) return e;
  return launch_pdl(gemm_tc_kernel<T>, dim3(grid), dim3(kGemmThreads), T::kSmemBytes, s, p);
}

}  // namespace

int gemm_tc_smem_bytes() {
  int m = WideTile::kSmemBytes;
  if (MediumTile::kSmemBytes > m) m = MediumTile::kSmemBytes;
  if (NarrowTile::kSmemBytes > m) m = NarrowTile::kSmemBytes;
  return m;
}

int gemm_tc_launch(const GemmParams& p, int grid, int max_rows, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (max_rows <= NarrowTile::kUnit) return launch_gemm<NarrowTile>(p, grid, s);
  if (max_rows <= MediumTile::kUnit) return launch_gemm<MediumTile>(p, grid, s);
  return launch_gemm<WideTile>(p, grid, s);
}

int router_tc_splits(int T, int E, int D, int num_sms) {
  const int tiles = ((T + 127) / 128) * ((E + 127) / 128);
  const int nkb = D / 64;
  int splits = num_sms / tiles;  // one wave: a partial second wave doubles the time
  const int cap = nkb / 4 > 1 ? nkb / 4 : 1;  // at least 4 blocks per split
  if (splits > cap) splits = cap;
  if (splits < 1) splits = 1;
  const int kbs = (nkb + splits - 1) / splits;
  return (nkb + kbs - 1) / kbs;
}

int router_tc_launch(const CUtensorMap& wmap, const CUtensorMap& xmap, int T, int E, int D,
                     int nsplit, float* partials, uint32_t* status, uint64_t timeout_ns, void* stream) {
  const int e = set_smem_limit(reinterpret_cast<const void*>(router_tc_kernel), kRtSmem);
  if (e != 0) return e;
  const int nkb = D / 64;
  const int kbs = (nkb + nsplit - 1) / nsplit;
  const int Epad = (E + 127) / 128 * 128;
  dim3 grid((T + 127) / 128, Epad / 128, nsplit);
  return launch_pdl(router_tc_kernel, grid, dim3(128), kRtSmem, static_cast<cudaStream_t>(stream),
                    wmap, xmap, T, E, Epad, nkb, kbs, partials, status, timeout_ns);
}

int gather_rows_launch(const void* x16, int D, const int32_t* perm, int topk, int rows, void* out,
                       void* stream) {
  if (rows <= 0) return 0;
  if (D / 8 > 32 * kGatherV || D % 8) return static_cast<int>(cudaErrorInvalidValue);
  return launch_pdl(gather_rows_kernel, dim3((rows + kGatherWarps - 1) / kGatherWarps),
                    dim3(kGatherWarps * 32), 0, static_cast<cudaStream_t>(stream),
                    static_cast<const uint4*>(x16), D / 8, perm, topk, rows, static_cast<uint4*>(out));
}

}  // namespace moe
