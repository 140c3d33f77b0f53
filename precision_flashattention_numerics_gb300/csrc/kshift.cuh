// Online pseudo-average shifting of the keys (the first PASA step).
//
// "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM Inference"
// (arXiv 2503.01873), Abstract: every key block is shifted by a pseudo-average along the
// sequence so that a large bias of K along the sequence cannot drive the fp16 scores past
// 65504; the offsets q_i . m_j are added back later ("global recovering") in fp32, which
// keeps the result equal to plain attention. The abstract does not define the
// pseudo-average; this library uses the following reading (the oracle implements the same
// reading independently, in numpy):
//
//   for key block j (block_rows_for(D) rows, n valid) and channel d:
//     M = max_r |K[r,d]|            g = fp16 spacing at M (2^(E-25), or 2^-24 if E = 0)
//     t_r = rint_even(K[r,d] / g)   m = g * rint_even(sum_r t_r / n)   (exact integers)
//     m = 0 when M >= 2^15 or the block/channel holds inf or NaN
//     K'[r,d] = fp16_rn(K[r,d] - m)
//
// m lies on the grid of the block maximum, so K - m is exact in fp16 for most elements.
//
// PLAIN (the alternative reading, fp16 output only): m = fp16_rn(exact mean of the n
// values). Every fp16 value is an integer multiple of 2^-24 below 2^15, so the block sum S
// is an exact 64-bit integer in units of 2^-24; fp16_rn(fp64(S / n) * 2^-24) is one
// rounding of the exact mean, because an exact mean that is not an fp16 tie lies at least
// 2^-32 from every tie while the fp64 division errs by at most 2^-38. The guard is the same.
//
// FP8 score modes: the same kernel can instead write e4m3 codes of K' (or of the raw keys,
// without the shift) with one scale per block: a = max |K'| over the block (all channels),
// inv = fp32(448 / a), code = e4m3_rn_satfinite(fp32(K' * inv)), scale = fp32(a / 448)
// (a = 0: inv = scale = 1). 448 is the largest finite e4m3 value.
//
// Kernel shape: one CTA of 256 threads per (batch*kv-head, key block). A block's rows are
// contiguous, so one thread stages the whole block into shared memory with a single
// untiled bulk copy (cp.async.bulk, completing on an mbarrier); each thread owns one 16-byte
// unit (8 channels) of up to ceil(block rows / row groups) rows and reads them from shared
// memory in each pass. The per-channel max and integer sums are reduced with warp shuffles
// and a small shared-memory exchange across the 8 warps. Keeping the block in shared
// memory instead of registers leaves room for several CTAs per SM, so one CTA's loads
// overlap another's reductions and stores. The block is read from HBM once and K' written
// once (HBM-bound: 2 * rows * D * 2 bytes per block).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace pasa {

// Keys per block: the block the pseudo-average is taken over, which is also the attention
// kernel's key tile (the N of its score MMA). 128 for both supported head dims.
__host__ __device__ constexpr int block_rows_for(int D) { return D == 128 || D == 64 ? 128 : 0; }
constexpr int kShiftThreads = 256;

// Output of kshift_kernel.
enum KshiftOut : int {
  kShiftF16 = 0,    // K' in fp16 (+ means)
  kShiftFp8 = 1,    // e4m3 codes of K' with one scale per block (+ means)
  kRawFp8 = 2,      // e4m3 codes of the raw keys with one scale per block (no shift)
};

// Two fp32 values -> two e4m3 codes, lo in the low byte (round to nearest even, saturating).
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// round-half-even(s / n) for integers, n > 0.
__device__ __forceinline__ int rne_div(int s, int n) {
  const int a = s < 0 ? -s : s;
  int q = a / n;
  const int r = a - q * n;
  if (2 * r > n || (2 * r == n && (q & 1))) ++q;
  return s < 0 ? -q : q;
}

template <int D, int BN, int OUT = kShiftF16, bool PLAIN = false>
__global__ void __launch_bounds__(kShiftThreads)
kshift_kernel(const __half* __restrict__ k, void* __restrict__ kshift, __half* __restrict__ means,
              float* __restrict__ kscale, int Sk, int nb, int j0, int cap, int nb_cap) {
  constexpr int U = D / 8;                       // 16-byte units per row
  constexpr int R = kShiftThreads / U;           // row groups
  constexpr int RPT = (BN + R - 1) / R;          // rows per thread (upper bound)
  constexpr int NW = kShiftThreads / 32;
  static_assert(32 % U == 0 || U % 32 == 0, "unit layout");
  static_assert(U <= 32, "D <= 256");

  __shared__ __align__(128) uint4 sh_blk[BN * U];   // the block, row-major, rows >= n zeroed
  __shared__ uint64_t sh_bar;
  __shared__ int sh_abort;
  __shared__ uint32_t sh_max[NW][U][4];
  __shared__ uint32_t sh_nf[NW][U][4];
  static_assert(!PLAIN || OUT == kShiftF16, "the plain-mean reading has the fp16 output only");
  __shared__ int sh_sum[PLAIN ? 1 : NW][U][8];
  __shared__ long long sh_sum64[PLAIN ? NW : 1][U][8];
  __shared__ uint32_t sh_amax[NW];

  // blocks [j0, nb) of the Sk valid rows; planes are cap rows (means: nb_cap blocks) apart.
  // j0 > 0 refreshes the tail of a key cache after an append. A decode launch queued behind
  // a refresh may start now: it reads the refreshed blocks only after griddep_wait().
  griddep_launch_dependents();
  const int j = j0 + blockIdx.x;
  const int bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int u = tid % U;
  const int rg = tid / U;
  const int warp = tid / 32;
  const int row0 = j * BN;
  const int n = min(BN, Sk - row0);

  uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(kshift) + (static_cast<size_t>(bh) * cap + row0) * D) + u;

  // 0. stage the block: n contiguous rows of D fp16 (n * D * 2 bytes, a multiple of 16)
  if (tid == 0) {
    sh_abort = 0;
    mbar_init(&sh_bar, 1);
    fence_mbar_init();
  }
  for (int r = n + tid / U; r < BN; r += R) sh_blk[r * U + u] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // One thread waits for the copy (256 polling threads per CTA would crowd the shared-memory
  // pipe that the other resident CTAs' passes use); the rest wait at the CTA barrier.
  if (tid == 0) {
    const uint32_t bytes = static_cast<uint32_t>(n) * D * 2;
    mbar_arrive_expect_tx(&sh_bar, bytes);
    bulk_load_1d(sh_blk, k + (static_cast<size_t>(bh) * cap + row0) * D, bytes, &sh_bar);
    if (!mbar_wait(&sh_bar, 0, &sh_abort, 0x4B530000u | static_cast<uint32_t>(blockIdx.y & 0xFFFF))) {
      // give the copy in flight a last bounded chance to land before the CTA leaves
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&sh_bar, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
  }
  __syncthreads();
  if (sh_abort) return;
  const uint4* blk = sh_blk + u;

  // 1. per-channel max |K| over finite values, and a non-finite flag (16-bit lanes)
  uint32_t mx[4] = {0, 0, 0, 0}, nf[4] = {0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const uint4 xi = blk[(rg + i * R) * U];
    const uint32_t w[4] = {xi.x, xi.y, xi.z, xi.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t a = w[c] & 0x7FFF7FFFu;
      const uint32_t bad = __vcmpgeu2(a, 0x7C007C00u);  // inf or NaN (rows >= n are zero)
      nf[c] |= bad;
      mx[c] = __vmaxu2(mx[c], a & ~bad);
    }
  }
#pragma unroll
  for (int off = U; off < 32; off *= 2) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      mx[c] = __vmaxu2(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
      nf[c] |= __shfl_xor_sync(0xffffffffu, nf[c], off);
    }
  }
  if ((tid % 32) < U) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      sh_max[warp][u][c] = mx[c];
      sh_nf[warp][u][c] = nf[c];
    }
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t m = 0, f = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      m = __vmaxu2(m, sh_max[w][u][c]);
      f |= sh_nf[w][u][c];
    }
    mx[c] = m;
    nf[c] = f;
  }

  // 2. grid step per channel and the quantised sum
  float inv_g[8], g[8];
  bool guard[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const uint32_t a = (mx[h / 2] >> (16 * (h & 1))) & 0xFFFFu;
    const int E = static_cast<int>(a >> 10);
    const int e = E >= 1 ? E - 25 : -24;            // g = 2^e
    g[h] = __int_as_float((e + 127) << 23);
    inv_g[h] = __int_as_float((127 - e) << 23);
    guard[h] = (E >= 30) || (((nf[h / 2] >> (16 * (h & 1))) & 0xFFFFu) != 0);
  }
  if constexpr (PLAIN) {
    // exact sums in units of 2^-24 (f * 2^24 is exact in fp32: an fp16 value has 11 bits)
    long long sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const uint4 xi = blk[(rg + i * R) * U];
      const __half* hv = reinterpret_cast<const __half*>(&xi);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float f = __half2float(hv[h]);
        sum[h] += isfinite(f) ? __float2ll_rn(f * 16777216.0f) : 0ll;
      }
    }
#pragma unroll
    for (int off = U; off < 32; off *= 2) {
#pragma unroll
      for (int h = 0; h < 8; ++h) sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], off);
    }
    if ((tid % 32) < U) {
#pragma unroll
      for (int h = 0; h < 8; ++h) sh_sum64[warp][u][h] = sum[h];
    }
  } else {
    // t = K / g is exact (a power-of-two scale) and |t| < 2^11 in every channel that is not
    // guarded (|K| <= M < 2^11 g), so fp32(t + 1.5 * 2^23) is rint_even(t) + 1.5 * 2^23
    // exactly and its bit pattern minus that of 1.5 * 2^23 is rint_even(t): one FFMA and one
    // integer add per element. Rows >= n hold zeros. A guarded channel (non-finite values, or
    // M >= 2^15) gets a meaningless sum that is discarded below; the sums are unsigned so
    // that it wraps harmlessly.
    constexpr float kRound = 12582912.0f;      // 1.5 * 2^23
    constexpr uint32_t kRoundBits = 0x4B400000u;
    uint32_t sum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const uint4 xi = blk[(rg + i * R) * U];
      const __half2* hv = reinterpret_cast<const __half2*>(&xi);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = __half22float2(hv[c]);
        sum[2 * c] += __float_as_uint(__fmaf_rn(f.x, inv_g[2 * c], kRound)) - kRoundBits;
        sum[2 * c + 1] += __float_as_uint(__fmaf_rn(f.y, inv_g[2 * c + 1], kRound)) - kRoundBits;
      }
    }
#pragma unroll
    for (int off = U; off < 32; off *= 2) {
#pragma unroll
      for (int h = 0; h < 8; ++h) sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], off);
    }
    if ((tid % 32) < U) {
#pragma unroll
      for (int h = 0; h < 8; ++h) sh_sum[warp][u][h] = static_cast<int>(sum[h]);
    }
  }
  __syncthreads();

  // 3. pseudo-average, then 4. K' = fp16_rn(K - m)
  float mf[8];
  __half mh[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if constexpr (PLAIN) {
      long long s = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) s += sh_sum64[w][u][h];
      mh[h] = guard[h] ? __float2half_rn(0.0f) : __double2half(static_cast<double>(s) / n * 0x1p-24);
      mf[h] = __half2float(mh[h]);
    } else {
      uint32_t su = 0;
#pragma unroll
      for (int w = 0; w < NW; ++w) su += static_cast<uint32_t>(sh_sum[w][u][h]);
      const int s = static_cast<int>(su);  // |s| < 128 * 2^11 wherever it is used
      const int mu = guard[h] ? 0 : rne_div(s, n);
      mf[h] = (guard[h] || OUT == kRawFp8) ? 0.0f : static_cast<float>(mu) * g[h];  // exact, an fp16 value
      mh[h] = __float2half_rn(mf[h]);
    }
  }
  if (OUT != kRawFp8 && rg == 0) {
    uint4 mv;
    __half* mp = reinterpret_cast<__half*>(&mv);
#pragma unroll
    for (int h = 0; h < 8; ++h) mp[h] = mh[h];
    reinterpret_cast<uint4*>(means + (static_cast<size_t>(bh) * nb_cap + j) * D)[u] = mv;
  }
  if constexpr (OUT == kShiftF16) {
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg + i * R;
      if (r < n) {
        uint4 o;
        const uint4 xi = blk[r * U];
        const __half2* hv = reinterpret_cast<const __half2*>(&xi);
        __half2* op = reinterpret_cast<__half2*>(&o);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = __half22float2(hv[c]);
          op[c] = __floats2half2_rn(f.x - mf[2 * c], f.y - mf[2 * c + 1]);  // each rounded once, RN
        }
        dst[static_cast<size_t>(r) * U] = o;
      }
    }
  } else {
    // K' (rounded to fp16, as the fp16 modes use it) over the block's own shared-memory
    // copy (each thread rewrites only the units it reads), and its block maximum
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg + i * R;
      uint4 xi = blk[r * U];
      __half* hv = reinterpret_cast<__half*>(&xi);
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        hv[h] = r < n ? __float2half_rn(__half2float(hv[h]) - mf[h]) : __ushort_as_half(0);
        amax = max(amax, static_cast<uint32_t>(__half_as_ushort(hv[h]) & 0x7FFFu));
      }
      sh_blk[r * U + u] = xi;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((tid % 32) == 0) sh_amax[warp] = amax;
    __syncthreads();
    amax = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) amax = max(amax, sh_amax[w]);
    const float a = __half2float(__ushort_as_half(static_cast<unsigned short>(amax)));
    const float inv = a > 0.0f ? __fdiv_rn(448.0f, a) : 1.0f;
    if (tid == 0) kscale[static_cast<size_t>(bh) * nb_cap + j] = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
    uint2* dst8 = reinterpret_cast<uint2*>(static_cast<uint8_t*>(kshift) + (static_cast<size_t>(bh) * cap + row0) * D) + u;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int r = rg + i * R;
      if (r < n) {
        const uint4 xi = blk[r * U];
        const __half* hv = reinterpret_cast<const __half*>(&xi);
        uint16_t c[4];
#pragma unroll
        for (int h = 0; h < 4; ++h)
          c[h] = pack_e4m3x2(__fmul_rn(__half2float(hv[2 * h]), inv), __fmul_rn(__half2float(hv[2 * h + 1]), inv));
        dst8[static_cast<size_t>(r) * U] = make_uint2(c[0] | (static_cast<uint32_t>(c[1]) << 16),
                                                      c[2] | (static_cast<uint32_t>(c[3]) << 16));
      }
    }
  }
}

// The fp16 grid-mean shift (kShiftF16, the prefill path) held in registers instead of
// shared memory: thread (u, rg) owns the 16-byte unit u (channels 8u .. 8u + 7) of the block
// rows rg, rg + RG, rg + 2 RG, ...; it loads them straight from global memory (a warp reads
// whole rows, so the loads are coalesced), reduces the per-channel maximum and integer sums
// with one shuffle level and an exchange across the CTA's warps, and writes K' from the same
// registers. No staging pass over shared memory, so nothing but HBM bounds it. The reading
// is kshift_kernel's; K' is one rounding of K - m (sub.rn.f16x2), which is what that
// kernel's fp32 subtraction and fp16 rounding give (checked bit for bit in the tests).
constexpr int kShiftRegThreads = 128;

template <int D, int BN>
__global__ void __launch_bounds__(kShiftRegThreads)
kshift_reg_kernel(const __half* __restrict__ k, __half* __restrict__ kshift, __half* __restrict__ means, int Sk,
                  int nb, int j0, int cap, int nb_cap) {
  constexpr int U = D / 8;                       // 16-byte units per row
  constexpr int RG = kShiftRegThreads / U;       // row groups
  constexpr int RPT = BN / RG;                   // rows per thread
  constexpr int NW = kShiftRegThreads / 32;
  static_assert(BN % RG == 0 && 32 % U == 0, "layout");
  __shared__ uint32_t sh_max[NW][U][4];
  __shared__ uint32_t sh_sum[NW][U][8];

  griddep_launch_dependents();   // as in kshift_kernel: a queued decode launch may start
  const int j = j0 + blockIdx.x;
  const int bh = blockIdx.y;
  const int tid = threadIdx.x;
  const int u = tid % U;
  const int rg = tid / U;
  const int warp = tid / 32;
  const int row0 = j * BN;
  const int n = min(BN, Sk - row0);
  const uint4* src = reinterpret_cast<const uint4*>(k + (static_cast<size_t>(bh) * cap + row0) * D) + u;
  uint4* dst = reinterpret_cast<uint4*>(kshift + (static_cast<size_t>(bh) * cap + row0) * D) + u;

  uint4 x[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * RG;
    x[i] = r < n ? __ldg(src + static_cast<size_t>(r) * U) : make_uint4(0, 0, 0, 0);
  }
  // 1. per-channel max |K| (16-bit lanes); an inf or NaN makes it >= 0x7C00
  uint32_t mx[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    mx[0] = __vmaxu2(mx[0], x[i].x & 0x7FFF7FFFu);
    mx[1] = __vmaxu2(mx[1], x[i].y & 0x7FFF7FFFu);
    mx[2] = __vmaxu2(mx[2], x[i].z & 0x7FFF7FFFu);
    mx[3] = __vmaxu2(mx[3], x[i].w & 0x7FFF7FFFu);
  }
#pragma unroll
  for (int off = U; off < 32; off *= 2)
#pragma unroll
    for (int c = 0; c < 4; ++c) mx[c] = __vmaxu2(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], off));
  if ((tid % 32) < U) {
#pragma unroll
    for (int c = 0; c < 4; ++c) sh_max[warp][u][c] = mx[c];
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t m = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) m = __vmaxu2(m, sh_max[w][u][c]);
    mx[c] = m;
  }
  // 2. grid step per channel; guard (m = 0) from 2^15 up and for inf/NaN
  float g[8], inv_g[8];
  bool guard[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const uint32_t a = (mx[h / 2] >> (16 * (h & 1))) & 0xFFFFu;
    const int E = static_cast<int>(a >> 10);
    const int e = E >= 1 ? E - 25 : -24;
    g[h] = __int_as_float((e + 127) << 23);
    inv_g[h] = __int_as_float((127 - e) << 23);
    guard[h] = E >= 30;
  }
  // 3. exact integer sums of rint_even(K / g) (rows >= n are zeros); see kshift_kernel
  constexpr float kRound = 12582912.0f;      // 1.5 * 2^23
  constexpr uint32_t kRoundBits = 0x4B400000u;
  uint32_t sum[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const __half2* hv = reinterpret_cast<const __half2*>(&x[i]);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float2 f = __half22float2(hv[c]);
      sum[2 * c] += __float_as_uint(__fmaf_rn(f.x, inv_g[2 * c], kRound)) - kRoundBits;
      sum[2 * c + 1] += __float_as_uint(__fmaf_rn(f.y, inv_g[2 * c + 1], kRound)) - kRoundBits;
    }
  }
#pragma unroll
  for (int off = U; off < 32; off *= 2)
#pragma unroll
    for (int h = 0; h < 8; ++h) sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], off);
  if ((tid % 32) < U) {
#pragma unroll
    for (int h = 0; h < 8; ++h) sh_sum[warp][u][h] = sum[h];
  }
  __syncthreads();
  // 4. m = g * rint_even(sum / n), then K' = fp16_rn(K - m) from the registers
  uint32_t m2[4];
  float mf[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    uint32_t su = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) su += sh_sum[w][u][h];
    const int si = static_cast<int>(su);
    int mu;
    if (n == BN && (BN & (BN - 1)) == 0) {
      constexpr int kShift = BN == 128 ? 7 : (BN == 64 ? 6 : 0);
      const int fl = si >> kShift, rm = si & (BN - 1);
      mu = fl + ((2 * rm > BN || (2 * rm == BN && (fl & 1))) ? 1 : 0);
    } else {
      mu = rne_div(si, n);
    }
    mf[h] = guard[h] ? 0.0f : static_cast<float>(mu) * g[h];   // exact, an fp16 value
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __half2 h2 = __floats2half2_rn(mf[2 * c], mf[2 * c + 1]);
    m2[c] = *reinterpret_cast<const uint32_t*>(&h2);
  }
  if (rg == 0) reinterpret_cast<uint4*>(means + (static_cast<size_t>(bh) * nb_cap + j) * D)[u] =
      make_uint4(m2[0], m2[1], m2[2], m2[3]);
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = rg + i * RG;
    if (r < n) {
      uint4 o;
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.x) : "r"(x[i].x), "r"(m2[0]));
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.y) : "r"(x[i].y), "r"(m2[1]));
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.z) : "r"(x[i].z), "r"(m2[2]));
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(o.w) : "r"(x[i].w), "r"(m2[3]));
      dst[static_cast<size_t>(r) * U] = o;
    }
  }
}

}  // namespace pasa
