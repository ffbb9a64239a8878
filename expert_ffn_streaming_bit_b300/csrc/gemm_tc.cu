// Grouped GEMM of the multi-token layer step on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory).
//
// One work unit = a 128-row tile of one 4-bit weight matrix (an expert's
// interleaved gate/up rows, its down rows, or the shared expert's) against up
// to 256 activation rows (the tokens routed to that expert, or a tile of all
// tokens for the shared expert).  The weight tile is the MMA's M side (128),
// the tokens its N side (16..256 in steps of 16), so the tile shape follows
// the ragged per-expert token counts without padding M.
//
// Per CTA (persistent, one per SM, 18 warps):
//   warp 0       TMA: packed 4-bit codes (128 B x 128 rows, 128-byte swizzle)
//                and scale/bias words (16 B x 128 rows) of a 256-column slice
//                of the weight tile -> P ring (3 stages)
//   warp 1       MMA: one elected thread issues tcgen05.mma kind::f16
//                (M=128, N=tokens, K=16) x 4 per 64-column block, fp32
//                accumulators in tensor memory (2 x 256 columns)
//   warps 2-5    B producers: cp.async gather of the activation rows (fp16,
//                64 columns = 128 B per row) into the 128-byte swizzled
//                K-major layout -> B ring (3 stages)
//   warps 6-13   dequantisation: P stage -> fp16 weights w = s q + b (one
//                rounding) in the swizzled K-major layout -> A ring (3 stages)
//   warps 14-17  epilogue: tensor memory -> registers; gate/up units write
//                h = gelu(g) * u (fp16, times a per-token power of two that
//                keeps it in range), down units undo that factor and write the
//                routing-weighted expert output (bf16) or the shared output (fp32)
// Rings are mbarrier-pipelined; every wait is bounded in time and a wait that
// runs out sets the status word and ends the CTA's work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kNP = 3, kNA = 3, kNB = 3;
constexpr int kPCodeBytes = 128 * 128;           // 128 rows x 256 columns of 4-bit codes
constexpr int kPSbBytes = 128 * 16;              // 128 rows x 4 scale/bias words
constexpr int kPBytes = kPCodeBytes + kPSbBytes; // 18 KB per P stage (multiple of 1 KB)
constexpr int kABytes = 128 * 128;               // 128 rows x 64 fp16
constexpr int kBBytes = kUnitTokens * 128;       // 256 rows x 64 fp16
constexpr int kTmemCols = 512;                   // 2 accumulators x 256 columns
constexpr int kGemmThreads = 18 * 32;
constexpr int kBLag = kNB - 1;                   // cp.async groups kept in flight

struct Bars {
  uint64_t p_full[kNP], p_empty[kNP];
  uint64_t a_full[kNA], a_empty[kNA];
  uint64_t b_full[kNB], b_empty[kNB];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort;
};

constexpr int kStageBytes = 32 * 128 * 4;           // epilogue staging: 32 tokens x 128 fp32
constexpr int kMetaBytes = 2 * kUnitTokens * 4;     // per-column factors
constexpr int kSmemBytes = kNP * kPBytes + kNA * kABytes + kNB * kBBytes + kStageBytes +
                           kMetaBytes + 1024 /*Bars*/ + 1024 /*alignment slack*/;

__device__ __forceinline__ float gelu_tanh(float x) {
  const float c = 0.7978845608028654f;  // sqrt(2/pi)
  return 0.5f * x * (1.f + tanhf(c * (x + 0.044715f * x * x * x)));
}

// Bounded mbarrier wait shared by all roles: on expiry record a timeout and
// make every role stop.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const GemmParams& p,
                                         Bars* bars) {
  if (mbar_wait(bar, parity, p.timeout_ns, &bars->abort)) return true;
  if (!bars->abort) atomicCAS(p.status, DEV_OK, DEV_TIMEOUT);
  bars->abort = 1;
  return false;
}

__device__ __forceinline__ int unit_nmma(int n) { return (n + 15) & ~15; }

// ---------------------------------------------------------------- roles

__device__ void role_tma(const GemmParams& p, uint8_t* P, Bars* bars, int nU) {
  uint32_t pc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int np = (K + 255) / 256;
    const void* tc = &p.tm_code[un.kind];
    const void* ts = &p.tm_sb[un.kind];
    for (int sp = 0; sp < np; ++sp, ++pc) {
      const int st = pc % kNP;
      if (!wait_bar(&bars->p_empty[st], ((pc / kNP) & 1) ^ 1, p, bars)) return;
      uint8_t* dst = P + st * kPBytes;
      mbar_arrive_expect_tx(&bars->p_full[st], kPBytes);
      const int xc = sp * 128, xs = K / 2 + sp * 16, y = un.mt * 128;
      if (un.kind == 0) {
        tma_load_3d(dst, tc, xc, y, un.expert, &bars->p_full[st]);
        tma_load_3d(dst + kPCodeBytes, ts, xs, y, un.expert, &bars->p_full[st]);
      } else {
        tma_load_2d(dst, tc, xc, y, &bars->p_full[st]);
        tma_load_2d(dst + kPCodeBytes, ts, xs, y, &bars->p_full[st]);
      }
    }
  }
  // drain: the stages still in flight must land before the CTA exits
  for (uint32_t q = pc > kNP ? pc - kNP : 0; q < pc; ++q)
    mbar_wait(&bars->p_full[q % kNP], (q / kNP) & 1, p.timeout_ns, nullptr);
}

__device__ void role_dequant(const GemmParams& p, const uint8_t* P, uint8_t* A, Bars* bars,
                             int nU) {
  const int t = threadIdx.x - 6 * 32;  // 0..255
  const int row = t & 127, half = t >> 7;
  const int lane = threadIdx.x & 31;
  uint32_t pc = 0, ac = 0;
  const __half2 k1024 = __floats2half2_rn(1024.f, 1024.f);
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int nkb = K / 64;
    const int np = (K + 255) / 256;
    for (int sp = 0; sp < np; ++sp, ++pc) {
      const int st = pc % kNP;
      if (!wait_bar(&bars->p_full[st], (pc / kNP) & 1, p, bars)) return;
      const uint8_t* codes = P + st * kPBytes;
      const uint32_t* sbw = reinterpret_cast<const uint32_t*>(P + st * kPBytes + kPCodeBytes);
      const int nsub = min(4, nkb - 4 * sp);
      for (int sb = 0; sb < nsub; ++sb, ++ac) {
        const int as = ac % kNA;
        if (!wait_bar(&bars->a_empty[as], ((ac / kNA) & 1) ^ 1, p, bars)) return;
        // packed chunk c (32 columns) of this row, stored at chunk c ^ (row & 7)
        const int c = 2 * sb + half;
        const uint4 w = *reinterpret_cast<const uint4*>(codes + row * 128 + ((c ^ (row & 7)) << 4));
        const uint32_t word = sbw[row * 4 + sb];
        const __half2 s2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(word & 0xffffu)));
        const __half2 b2 = __half2half2(__ushort_as_half(static_cast<unsigned short>(word >> 16)));
        uint8_t* arow = A + as * kABytes + row * 128;
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // word j: columns 8j..8j+7 of the chunk; byte i = col i (low) | col 4+i (high)
          const uint32_t lo = ws[j] & 0x0F0F0F0Fu;
          const uint32_t hi = (ws[j] >> 4) & 0x0F0F0F0Fu;
          // fp16 1024 + q pairs: bytes (q, 0x64) per half
          const uint32_t m01 = __byte_perm(lo, 0x64646464u, 0x5140);
          const uint32_t m23 = __byte_perm(lo, 0x64646464u, 0x7362);
          const uint32_t m45 = __byte_perm(hi, 0x64646464u, 0x5140);
          const uint32_t m67 = __byte_perm(hi, 0x64646464u, 0x7362);
          uint32_t o[4];
          const uint32_t mm[4] = {m01, m23, m45, m67};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&mm[i]), k1024);
            const __half2 v = __hfma2(q, s2, b2);
            o[i] = *reinterpret_cast<const uint32_t*>(&v);
          }
          const int lc = 4 * half + j;  // logical 16-byte chunk in the 128-byte row
          *reinterpret_cast<uint4*>(arow + ((lc ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->a_full[as]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_empty[st]);
    }
  }
}

__device__ void role_bload(const GemmParams& p, uint8_t* B, Bars* bars, int nU) {
  const int t = threadIdx.x - 2 * 32;  // 0..127
  const int lane = threadIdx.x & 31;
  uint32_t bc = 0;        // blocks issued
  uint32_t signalled = 0; // blocks whose arrival has been signalled
  for (int u = blockIdx.x; u < nU; u += gridDim.x) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int nkb = K / 64;
    const __half* src[2] = {nullptr, nullptr};
    for (int h = 0; h < 2; ++h) {
      const int r = t + 128 * h;
      if (r < un.n) {
        int64_t srow;
        if (p.mode == 0 && un.kind == 0) srow = p.perm[un.row0 + r] / p.topk;  // token
        else srow = un.row0 + r;
        src[h] = reinterpret_cast<const __half*>(p.bsrc[un.kind]) + srow * p.bld[un.kind];
      }
    }
    for (int kb = 0; kb < nkb; ++kb, ++bc) {
      const int bs = bc % kNB;
      if (!wait_bar(&bars->b_empty[bs], ((bc / kNB) & 1) ^ 1, p, bars)) {
        cp_async_wait<0>();
        return;
      }
      uint8_t* dst = B + bs * kBBytes;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!src[h]) continue;
        const int r = t + 128 * h;
        const __half* s = src[h] + kb * 64;
#pragma unroll
        for (int c = 0; c < 8; ++c) cp_async16(dst + r * 128 + ((c ^ (r & 7)) << 4), s + c * 8);
      }
      cp_async_commit();
      if (bc >= static_cast<uint32_t>(kBLag)) {
        cp_async_wait<kBLag>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->b_full[signalled % kNB]);
        ++signalled;
      }
    }
  }
  cp_async_wait<0>();
  fence_proxy_async_smem();
  __syncwarp();
  for (; signalled < bc; ++signalled)
    if (lane == 0) mbar_arrive(&bars->b_full[signalled % kNB]);
}

__device__ void role_mma(const GemmParams& p, uint8_t* A, uint8_t* B, Bars* bars, int nU) {
  const uint32_t tmem = bars->tmem_base;
  uint32_t ac = 0, bc = 0, uc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x, ++uc) {
    const GemmUnit un = p.units[u];
    const int K = p.K[un.kind];
    const int nkb = K / 64;
    const uint32_t idesc = tc_idesc_f16(128, unit_nmma(un.n));
    const int acc = uc & 1;
    if (!wait_bar(&bars->acc_empty[acc], ((uc >> 1) & 1) ^ 1, p, bars)) return;
    tc_fence_after();
    const uint32_t d_tmem = tmem + acc * 256;
    for (int kb = 0; kb < nkb; ++kb, ++ac, ++bc) {
      const int as = ac % kNA, bs = bc % kNB;
      if (!wait_bar(&bars->a_full[as], (ac / kNA) & 1, p, bars)) return;
      if (!wait_bar(&bars->b_full[bs], (bc / kNB) & 1, p, bars)) return;
      tc_fence_after();
      const uint32_t a0 = smem_u32(A + as * kABytes), b0 = smem_u32(B + bs * kBBytes);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        tc_mma_f16(d_tmem, tc_desc_sw128(a0 + 32 * kk), tc_desc_sw128(b0 + 32 * kk), idesc,
                   (kb | kk) != 0);
      tc_commit(&bars->a_empty[as]);
      tc_commit(&bars->b_empty[bs]);
    }
    tc_commit(&bars->acc_full[acc]);
  }
  // the last commits must complete before the CTA exits
  if (uc > 0) {
    const uint32_t last = uc - 1;
    mbar_wait(&bars->acc_full[last & 1], (last >> 1) & 1, p.timeout_ns, nullptr);
  }
}

// Epilogue (warps 14-17, 128 threads).  Per unit: per-column (token) scale
// factors are gathered into shared memory once; then per 32-column chunk the
// accumulator is read from tensor memory, the values are finished (GELU for
// gate/up; routing weight and range factor for down) and staged in shared
// memory, and the 4 warps write the chunk's output rows with 16-byte stores.
__device__ __forceinline__ void epi_sync() { named_sync(1, 128); }

__device__ void role_epilogue(const GemmParams& p, Bars* bars, uint8_t* stage, float* meta, int nU) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = w & 3;  // tensor-memory lane quarter this warp may access
  const int te = threadIdx.x - 14 * 32;  // 0..127
  const uint32_t tmem = bars->tmem_base;
  uint32_t uc = 0;
  for (int u = blockIdx.x; u < nU; u += gridDim.x, ++uc) {
    const GemmUnit un = p.units[u];
    const int acc = uc & 1;
    // per-column factors (independent of the accumulator: overlap the wait)
    for (int col = te; col < un.n; col += 128) {
      const int brow = un.row0 + col;
      if (p.mode == 0) {
        const int tok = un.kind == 0 ? p.perm[brow] / p.topk : brow;
        meta[col] = p.sigma[tok];
        meta[kUnitTokens + col] = p.hscale[tok];
      } else if (un.kind == 0) {
        const int a = p.perm[brow];
        meta[col] = p.wts[a] / p.hscale[a / p.topk];
      } else {
        meta[col] = 1.f / p.hscale[brow];
      }
    }
    if (!wait_bar(&bars->acc_full[acc], (uc >> 1) & 1, p, bars)) return;
    tc_fence_after();
    epi_sync();
    for (int c0 = 0; c0 < un.n; c0 += 32) {
      uint32_t r[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + acc * 256 + c0, r);
      tmem_ld_wait();
      const int nrow = min(32, un.n - c0);
      if (p.mode == 0) {
        // rows 2j / 2j+1 of the tile are gate / up of output column j:
        // the even lane takes columns c0..c0+15, the odd lane c0+16..c0+31
        const int jl = 16 * q + (lane >> 1);  // column within the tile's 64
        const bool odd = lane & 1;
        __half* st = reinterpret_cast<__half*>(stage);  // [32 tokens][64]
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float mine_lo = __uint_as_float(r[i]), mine_hi = __uint_as_float(r[16 + i]);
          const float recv = __shfl_xor_sync(0xffffffffu, odd ? mine_lo : mine_hi, 1);
          const float g = odd ? recv : mine_lo;
          const float v = odd ? mine_hi : recv;
          const int cl = (odd ? 16 : 0) + i;
          const int col = c0 + cl;
          if (col < un.n) {
            const float sg = meta[col];
            const float h = gelu_tanh(g * sg) * (v * sg) * meta[kUnitTokens + col];
            st[cl * 64 + jl] = __float2half_rn(fminf(fmaxf(h, -65504.f), 65504.f));
          }
        }
        epi_sync();
        // 32 rows x 128 bytes: 4 threads per row, 32 bytes each
        {
          const int rr = te >> 2, part = te & 3;
          if (rr < nrow) {
            const uint4* src = reinterpret_cast<const uint4*>(st + rr * 64 + part * 16);
            __half* dst = reinterpret_cast<__half*>(p.hout[un.kind]) +
                          static_cast<int64_t>(un.row0 + c0 + rr) * p.hld[un.kind] + un.mt * 64 + part * 16;
            reinterpret_cast<uint4*>(dst)[0] = src[0];
            reinterpret_cast<uint4*>(dst)[1] = src[1];
          }
        }
        epi_sync();
      } else if (un.kind == 0) {
        __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(stage);  // [32 tokens][128]
        const int dl = 32 * q + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < un.n) st[i * 128 + dl] = __float2bfloat16_rn(__uint_as_float(r[i]) * meta[c0 + i]);
        epi_sync();
        {  // 32 rows x 256 bytes: 4 threads per row, 64 bytes each
          const int rr = te >> 2, part = te & 3;
          if (rr < nrow) {
            const uint4* src = reinterpret_cast<const uint4*>(st + rr * 128 + part * 32);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.eout) +
                                                  static_cast<int64_t>(un.row0 + c0 + rr) * p.D +
                                                  un.mt * 128 + part * 32);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = src[k];
          }
        }
        epi_sync();
      } else {
        float* st = reinterpret_cast<float*>(stage);  // [32 tokens][128]
        const int dl = 32 * q + lane;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < un.n) st[i * 128 + dl] = __uint_as_float(r[i]) * meta[c0 + i];
        epi_sync();
        {  // 32 rows x 512 bytes: 4 threads per row, 128 bytes each
          const int rr = te >> 2, part = te & 3;
          if (rr < nrow) {
            const uint4* src = reinterpret_cast<const uint4*>(st + rr * 128 + part * 32);
            uint4* dst = reinterpret_cast<uint4*>(p.sout + static_cast<int64_t>(un.row0 + c0 + rr) * p.D +
                                                  un.mt * 128 + part * 32);
#pragma unroll
            for (int k = 0; k < 8; ++k) dst[k] = src[k];
          }
        }
        epi_sync();
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
  }
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base & 1023u)) & 1023u);
  uint8_t* P = smem;
  uint8_t* A = P + kNP * kPBytes;
  uint8_t* B = A + kNA * kABytes;
  uint8_t* stage = B + kNB * kBBytes;
  float* meta = reinterpret_cast<float*>(stage + kStageBytes);
  Bars* bars = reinterpret_cast<Bars*>(stage + kStageBytes + kMetaBytes);
  const int w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNP; ++i) {
      mbar_init(&bars->p_full[i], 1);
      mbar_init(&bars->p_empty[i], 8);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&bars->a_full[i], 8);
      mbar_init(&bars->a_empty[i], 1);
    }
    for (int i = 0; i < kNB; ++i) {
      mbar_init(&bars->b_full[i], 4);
      mbar_init(&bars->b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 4);
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
  const int nU = *p.n_units;
  if (w == 0) {
    if ((threadIdx.x & 31) == 0) role_tma(p, P, bars, nU);
  } else if (w == 1) {
    if ((threadIdx.x & 31) == 0) role_mma(p, A, B, bars, nU);
  } else if (w < 6) {
    role_bload(p, B, bars, nU);
  } else if (w < 14) {
    role_dequant(p, P, A, bars, nU);
  } else {
    role_epilogue(p, bars, stage, meta, nU);
  }
  tc_fence_before();
  __syncthreads();
  if (w == 1) {
    tc_fence_after();
    tmem_dealloc(bars->tmem_base, kTmemCols);
  }
}

}  // namespace

int gemm_tc_smem_bytes() { return kSmemBytes; }

int gemm_tc_launch(const GemmParams& p, int grid, void* stream) {
  static bool attr = false;
  if (!attr) {
    const cudaError_t e =
        cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return static_cast<int>(e);
    attr = true;
  }
  gemm_tc_kernel<<<grid, kGemmThreads, kSmemBytes, static_cast<cudaStream_t>(stream)>>>(p);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace moe
