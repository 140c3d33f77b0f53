// PASA attention forward, the variant for D = 64: two softmax warp sets taking alternate key
// blocks.
//
// Method as in attn_fwd_kernel ("Online Pseudo-average Shifting Attention (PASA) for Robust
// Low-precision LLM Inference", arXiv 2503.01873, Abstract: shifted keys K', fp16 scores,
// the offsets q_i . m_j added back in fp32 in the online softmax).
//
// At D = 64 the tensor work per 128 x 128 block halves while the softmax work (one thread
// per query row, ~1800 cycles a block) stays the same, so one softmax warpgroup leaves the
// tensor core idle half the time. Here eight softmax warps form two sets of four that take
// alternate key blocks: warp w handles query rows 32 (w mod 4) .. +31 (the TMEM lanes of its
// sub-partition) for the blocks j with j mod 2 = w div 4, so each warp has two block periods
// for one block's dependent chain, and the two warps on a sub-partition overlap their
// latencies. The running max and row sum of a row pass from one set to the other through
// shared memory after each block; P is double-buffered (p_free per block parity).
//
// Warp roles (352 threads): warps 0-7 softmax + epilogue (two sets), warp 8 TMA producer
// (Q once, K' one block ahead of V, 16-block means chunks), warp 9 TMEM owner and the score /
// offsets MMAs, warp 10 the PV MMAs. TMEM: two score buffers S_0, S_1, O, P, two offsets
// buffers and the Q tile (D / 2 columns). The score and offsets MMAs read Q from TMEM: a
// tcgen05 MMA with A in TMEM runs at ~67 cycles per M = 128, N <= 128 step against ~86 with
// both operands in shared memory. Every wait is bounded (ptx.cuh).
//
// Used for D = 64 prefill in modes 0-3 (pasa_lib.cu); the diagnostic, fp16-PV, FP8 and
// split-key (decode) work stays on attn_fwd_kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "attn_fwd.cuh"
#include "kshift.cuh"
#include "ptx.cuh"

namespace pasa {
namespace twoset {

constexpr int kTileRows = 128;       // query rows per CTA (MMA M)
constexpr int kChunkBlocks = 16;     // key blocks per offsets MMA (its N)
constexpr int kAttnThreads = 352;
constexpr int kSoftmaxWarps = 8;
constexpr float kRescaleLog2 = 8.0f;

using AttnParams = ::pasa::AttnParams;   // its leading fields are the ones read here

// TMEM column map (see the header comment).
template <int D, int BN>
struct TmemMap {
  __host__ __device__ static constexpr int s(int b) { return b * BN; }
  static constexpr int o = 2 * BN;
  static constexpr int p = 2 * BN + D;
  __host__ __device__ static constexpr int c(int b) { return 2 * BN + D + BN / 2 + b * kChunkBlocks; }
  static constexpr int q = 2 * BN + D + BN / 2 + 2 * kChunkBlocks;   // Q as the A operand
  static constexpr int total = q + D / 2;
  static_assert(total <= 512, "TMEM budget");
  static_assert(BN % 32 == 0 && BN <= 256, "key block");
  static_assert(D == 64 || D == 128, "head dim");
};

template <int D, int BN, int KST, int VST>
struct AttnSmem {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr int kQTile = kTileRows * D * 2;
  static constexpr int kKTile = BN * D * 2;
  static constexpr int kMTile = kChunkBlocks * D * 2;
  static constexpr int kQChunk = kTileRows * 128;
  static constexpr int kKChunk = BN * 128;
  static constexpr int kMChunk = kChunkBlocks * 128;
  alignas(1024) uint8_t q[kQTile];   // also the O staging buffer
  alignas(1024) uint8_t k[KST][kKTile];
  alignas(1024) uint8_t v[VST][kKTile];
  alignas(1024) uint8_t m[2][kMTile];
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t m_full[2], m_empty[2];
  uint64_t s_full[2];   // QK(j) done: S_(j mod 2) (and C) hold block j
  uint64_t s_free[2];   // the softmax has loaded S_(j mod 2) and C of block j (4 warps)
  uint64_t p_full;      // the softmax has written P of block j (4 warps)
  uint64_t p_free[2];   // PV(j) done (barrier j mod 2): P may be rewritten, O is stable.
                        // One per block parity: set t publishes m of block j before it
                        // waits for PV(j-1), so the other set can reach its wait for PV(j)
                        // while PV(j-1) still runs; with a single barrier that wait would
                        // see the phase of PV(j-2), of the same parity, as complete.
  uint64_t o_full;
  uint64_t drain[2];
  uint64_t mxf[4][2];            // [row group][set]: the set has published m of its block
  float xm[2][kTileRows];        // m of the last block of each set
  float xsum[4][2][kTileRows];   // epilogue: row sum, its max and the diagnostics per set
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float half_lo_to_float(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}

// Bounded wait by all lanes of a warp, with one result for the whole warp: a lane whose
// deadline passes just as the phase completes cannot leave the others behind.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t site) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, site));
}

// In-place tree reductions over a fully unrolled register array.
template <int N>
__device__ __forceinline__ float tree_max3(float* a) {
#pragma unroll
  for (int stride = 1; stride < N; stride *= 3)
#pragma unroll
    for (int i = 0; i < N; i += 3 * stride)
      a[i] = fmax3(a[i], i + stride < N ? a[i + stride] : -INFINITY,
                   i + 2 * stride < N ? a[i + 2 * stride] : -INFINITY);
  return a[0];
}

template <int N>
__device__ __forceinline__ float tree_min3(float* a) {
#pragma unroll
  for (int stride = 1; stride < N; stride *= 3)
#pragma unroll
    for (int i = 0; i < N; i += 3 * stride)
      a[i] = fmin3(a[i], i + stride < N ? a[i + stride] : INFINITY, i + 2 * stride < N ? a[i + 2 * stride] : INFINITY);
  return a[0];
}

template <int N, bool MAX>
__device__ __forceinline__ uint32_t tree_h2(uint32_t* a) {
#pragma unroll
  for (int stride = 1; stride < N; stride *= 2)
#pragma unroll
    for (int i = 0; i + stride < N; i += 2 * stride) a[i] = MAX ? hmax2(a[i], a[i + stride]) : hmin2(a[i], a[i + stride]);
  return a[0];
}

// Load BN/2 registers of packed fp16 scores (BN columns) from TMEM.
template <int BN>
__device__ __forceinline__ void tmem_ld_scores_f16(uint32_t taddr, uint32_t* hp) {
  static_assert(BN % 16 == 0, "BN");
#pragma unroll
  for (int c = 0; c + 32 <= BN; c += 32) tmem_ld_x16_pack16(taddr + c, hp + c / 2);
  if constexpr (BN % 32 != 0) tmem_ld_x8_pack16(taddr + (BN / 32) * 32, hp + (BN / 32) * 16);
}

template <int D, int BN, bool F16ACC, bool SHIFT, bool CAUSAL, int KST, int VST, bool STATS = false>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_fwd_2set_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                const __grid_constant__ CUtensorMap mapM, const AttnParams p) {
  using Smem = AttnSmem<D, BN, KST, VST>;
  using TM = TmemMap<D, BN>;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Work item: heavy (late) query tiles first across all heads; neighbouring CTAs share a
  // kv head so K/V stay in L2.
  const int lin = blockIdx.x;
  const int hb = lin % (p.Hq * p.B);
  const int qb = p.n_qblk - 1 - lin / (p.Hq * p.B);
  const int hq = hb % p.Hq;
  const int b = hb / p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const int q0 = qb * kTileRows;

  int nblk;
  {
    const int last = min(p.Sq, q0 + kTileRows) - 1;
    const int kv_end = CAUSAL ? min(p.Sk, last + p.Sk - p.Sq + 1) : p.Sk;
    nblk = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
  }

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < KST; ++i) { mbar_init(&s.k_full[i], 1); mbar_init(&s.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&s.v_full[i], 1); mbar_init(&s.v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.m_full[i], 1);
      mbar_init(&s.m_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);
    }
    mbar_init(&s.p_full, 4);
    for (int q4 = 0; q4 < 4; ++q4) {
      mbar_init(&s.mxf[q4][0], 1);
      mbar_init(&s.mxf[q4][1], 1);
    }
    mbar_init(&s.p_free[0], 1);
    mbar_init(&s.p_free[1], 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.drain[0], 1);
    mbar_init(&s.drain[1], 1);
    s.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 8) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      if (SHIFT) tma_prefetch_desc(&mapM);
      const int qz = b * p.Hq + hq;
      const int kz = b * p.Hkv + hk;
      mbar_arrive_expect_tx(&s.q_full, Smem::kQTile);
#pragma unroll
      for (int c = 0; c < Smem::kChunks; ++c)
        tma_load_3d(s.q + c * Smem::kQChunk, &mapQ, &s.q_full, c * 64, q0, qz);
      int k_issued = 0, v_issued = 0, m_issued = 0;
      // Issue order K_0, K_1, V_0, K_2, V_1, ...: each K runs one block ahead of V, matching
      // the MMA thread, whose loop step j takes K_j and V_(j-1).
      auto load_k = [&](int j) -> bool {
        if (SHIFT && (j % kChunkBlocks) == 0) {
          const int ci = j / kChunkBlocks, slot = ci & 1;
          if (!mbar_wait(&s.m_empty[slot], ((ci >> 1) & 1) ^ 1, abort_flag, 0x101)) return false;
          mbar_arrive_expect_tx(&s.m_full[slot], Smem::kMTile);
#pragma unroll
          for (int c = 0; c < Smem::kChunks; ++c)
            tma_load_3d(s.m[slot] + c * Smem::kMChunk, &mapM, &s.m_full[slot], c * 64, j, kz);
          m_issued = ci + 1;
        }
        const int ks = j % KST;
        if (!mbar_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, abort_flag, 0x102)) return false;
        mbar_arrive_expect_tx(&s.k_full[ks], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.k[ks] + c * Smem::kKChunk, &mapK, &s.k_full[ks], c * 64, j * BN, kz);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int vs = j % VST;
        if (!mbar_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, abort_flag, 0x103)) return false;
        mbar_arrive_expect_tx(&s.v_full[vs], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.v[vs] + c * Smem::kKChunk, &mapV, &s.v_full[vs], c * 64, j * BN, kz);
        v_issued = j + 1;
        return true;
      };
      // The keys and means may come from the shift kernel queued just ahead of this launch
      // (launched with programmatic dependence on it): wait for it before the first load of
      // either. Q is not written by it and is already on its way.
      griddep_wait();
      bool pok = nblk == 0 || load_k(0);
      for (int j = 0; pok && j < nblk; ++j) {
        if (j + 1 < nblk && !load_k(j + 1)) break;
        if (!load_v(j)) break;
      }
      if (*abort_flag) {
        // Let every copy this warp issued land before the CTA's shared memory goes away.
        const uint64_t t0 = globaltimer_ns();
        auto drain = [&](uint64_t* bar, uint32_t parity) {
          while (!mbar_try_wait(bar, parity) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
          }
        };
        drain(&s.q_full, 0);
        for (int j = max(0, k_issued - KST); j < k_issued; ++j) drain(&s.k_full[j % KST], (j / KST) & 1);
        for (int j = max(0, v_issued - VST); j < v_issued; ++j) drain(&s.v_full[j % VST], (j / VST) & 1);
        for (int ci = max(0, m_issued - 2); ci < m_issued; ++ci) drain(&s.m_full[ci & 1], (ci >> 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------------ QK issuer
    // QK(j) goes into S_(j mod 2) once the softmax has loaded block j-2 from that buffer; at
    // the start of a 16-block chunk the offsets of the chunk go into C_(chunk mod 2), which
    // was last read with block 16*(chunk-1)-1 <= j-2 and so is free as well.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(kTileRows, BN, !F16ACC, false);
      constexpr uint32_t id_c = idesc_f16(kTileRows, kChunkBlocks, true, false);
      // Descriptor words: the high word is one constant per layout, the low word of every
      // operand is its buffer's base word plus a compile-time offset.
      constexpr uint32_t hi_kmaj = sdesc_hi_sw128(1024);
      const uint32_t q_lo = sdesc_lo(smem_u32(s.q), 16);
      const uint32_t k_lo0 = sdesc_lo(smem_u32(s.k[0]), 16);
      const uint32_t m_lo0 = sdesc_lo(smem_u32(s.m[0]), 16);
      constexpr uint32_t kKStride = sizeof(s.k[0]) >> 4;  // descriptor units per ring slot
      constexpr uint32_t kMStride = sizeof(s.m[0]) >> 4;
      uint32_t qd[D / 16];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) qd[kk] = q_lo + (((kk / 4) * Smem::kQChunk + (kk % 4) * 32) >> 4);
      const uint32_t tQ = tmem + TM::q;
      bool ok = mbar_wait(&s.q_full, 0, abort_flag, 0x201);
      if (ok && nblk > 0) {
        // Q into TMEM once. Only with key blocks: without them the epilogue rewrites the Q
        // buffer as soon as Q has landed, and no MMA completion would cover this copy.
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) tmem_cp_128x256b(tQ + kk * 8, qd[kk], hi_kmaj);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        const int ks = j % KST;
        const int ci = j / kChunkBlocks;
        const int sb = j & 1;
        const bool chunk_start = SHIFT && (j % kChunkBlocks) == 0;
        uint32_t kd[D / 16];
        const uint32_t k_lo = k_lo0 + ks * kKStride;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) kd[kk] = k_lo + (((kk / 4) * Smem::kKChunk + (kk % 4) * 32) >> 4);
        if (!mbar_wait(&s.k_full[ks], (j / KST) & 1, abort_flag, 0x202)) break;
        if (!mbar_wait(&s.v_full[j % VST], (j / VST) & 1, abort_flag, 0x207)) break;
        if (chunk_start && !mbar_wait(&s.m_full[ci & 1], (ci >> 1) & 1, abort_flag, 0x203)) break;
        if (j >= 2 && !mbar_wait(&s.s_free[sb], ((j >> 1) - 1) & 1, abort_flag, 0x206)) break;
        tc_fence_after();
        if (chunk_start) {
          const uint32_t m_lo = m_lo0 + (ci & 1) * kMStride;
          const uint32_t tC = tmem + TM::c(ci & 1);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_m = ((kk / 4) * Smem::kMChunk + (kk % 4) * 32) >> 4;
            mma_ts_w(tC, tQ + kk * 8, m_lo + off_m, hi_kmaj, id_c, kk > 0 ? 1u : 0u);
          }
        }
        const uint32_t tS = tmem + TM::s(sb);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) mma_ts_w(tS, tQ + kk * 8, kd[kk], hi_kmaj, id_s, kk > 0 ? 1u : 0u);
        mma_commit(&s.s_full[sb]);
        mma_commit(&s.k_empty[ks]);
        if (chunk_start) mma_commit(&s.m_empty[ci & 1]);
      }
      // all MMAs issued by this thread complete before TMEM can be released
      mma_commit(&s.drain[0]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain[0], 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  } else if (warp == 10) {
    // ------------------------------------------------------------------ PV issuer
    // PV(j) once the softmax has written P of block j. V_j has landed by then: the QK thread
    // waited for it before issuing QK(j), and the softmax loads S_j (after QK(j) completes)
    // before it writes P of block j. Waiting here as well cost ~1% (one more barrier poll
    // on the path from the P store to the PV MMAs).
    if (lane == 0) {
      constexpr uint32_t id_o = idesc_f16(kTileRows, D, true, true);
      constexpr uint32_t hi_v = sdesc_hi_sw128(1024);
      const uint32_t v_lo0 = sdesc_lo(smem_u32(s.v[0]), Smem::kKChunk);
      constexpr uint32_t kVStride = sizeof(s.v[0]) >> 4;
      const uint32_t tO = tmem + TM::o;
      const uint32_t tP = tmem + TM::p;
      for (int j = 0; j < nblk; ++j) {
        const int vs = j % VST;
        uint32_t vd[BN / 16];
        const uint32_t v_lo = v_lo0 + vs * kVStride;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) vd[kk] = v_lo + kk * (2048 >> 4);
        if (!mbar_wait(&s.p_full, j & 1, abort_flag, 0x205)) break;
        tc_fence_after();
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) mma_ts_w(tO, tP + kk * 8, vd[kk], hi_v, id_o, kk > 0 ? 1u : acc0);
        mma_commit(&s.p_free[j & 1]);
        mma_commit(&s.v_empty[vs]);
        if (j == nblk - 1) mma_commit(&s.o_full);
      }
      mma_commit(&s.drain[1]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain[1], 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    // Two warp sets: set 0 (warps 0-3) takes the even key blocks (score buffer S_0), set 1
    // (warps 4-7) the odd ones (S_1); warp w handles query rows 32*(w mod 4) .. +31, the TMEM
    // lanes of its sub-partition. The running max m is handed from block j-1 to block j
    // through shared memory (xm, barriers mxf); each set keeps the row sum of its own blocks
    // with the max it was last scaled to, and the epilogue combines the two sums.
    const int quad = warp & 3;
    const int set = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int kOCols = D / 2;         // O columns this warp normalises and stores
    const uint32_t tO = tmem + lane_base + TM::o;
    const uint32_t tP = tmem + lane_base + TM::p;
    const uint32_t tS = tmem + lane_base + TM::s(set);
    const int i = q0 + r;
    const int limit = (i < p.Sq) ? (CAUSAL ? min(p.Sk, max(0, i + p.Sk - p.Sq + 1)) : p.Sk) : 0;
    const float sl2 = p.scale_log2;
    constexpr int kPairs = BN / 2;
    float m_w = -INFINITY, l_w = 0.0f;   // this set's row sum and the max it is scaled to
    float st_acc = 0.0f, st_rec = 0.0f;  // STATS: max |accumulated score|, max |S' + c|
    bool ok = true;

    for (int j = set; j < nblk; j += 2) {
      if (!warp_wait(&s.s_full[set], (j >> 1) & 1, abort_flag, 0x300)) { ok = false; break; }
      tc_fence_after();
      // Load the block's scores and offset, wait once, fence the registers, and release the
      // score buffer to the QK thread before any arithmetic. fp16 scores (F16ACC) are loaded
      // two per register; their max is taken in f16x2 and each score enters fp32 through one
      // mixed-precision add. fp32 scores are used as loaded.
      uint32_t hp[F16ACC ? kPairs : 1];
      float sv[F16ACC ? 1 : BN];
      uint32_t cw = 0;
      if constexpr (F16ACC) {
        tmem_ld_scores_f16<BN>(tS, hp);
      } else {
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) tmem_ld_x16(tS + c * 16, reinterpret_cast<uint32_t*>(sv) + c * 16);
      }
      if (SHIFT) tmem_ld_x1(tmem + lane_base + TM::c((j / kChunkBlocks) & 1) + (j % kChunkBlocks), cw);
      tmem_ld_wait();
      if constexpr (F16ACC) reg_fence<kPairs>(hp);
      else reg_fence<BN>(reinterpret_cast<uint32_t*>(sv));
      reg_fence<1>(&cw);
      tc_fence_before();
      __syncwarp();
      mbar_arrive_if(&s.s_free[set], lane == 0);

      const int cmax = limit - j * BN;
      const float c_raw = SHIFT ? __uint_as_float(cw) : 0.0f;
      float mx, mn = 0.0f;
      if constexpr (F16ACC) {
        if constexpr (STATS) {
          uint32_t tmp[kPairs];
#pragma unroll
          for (int c = 0; c < kPairs; ++c)
            tmp[c] = ((2 * c < cmax) ? (hp[c] & 0xFFFFu) : 0x7C00u) |
                     ((2 * c + 1 < cmax) ? (hp[c] & 0xFFFF0000u) : 0x7C000000u);  // +inf when masked
          const uint32_t n1 = tree_h2<kPairs, false>(tmp);
          mn = fminf(half_lo_to_float(n1), half_lo_to_float(n1 >> 16));
        }
        if (cmax < BN) {
#pragma unroll
          for (int c = 0; c < kPairs; ++c)
            hp[c] = ((2 * c < cmax) ? (hp[c] & 0xFFFFu) : 0xFC00u) |
                    ((2 * c + 1 < cmax) ? (hp[c] & 0xFFFF0000u) : 0xFC000000u);  // -inf when masked
        }
        uint32_t tmp[kPairs];
#pragma unroll
        for (int c = 0; c < kPairs; ++c) tmp[c] = hp[c];
        const uint32_t m1 = tree_h2<kPairs, true>(tmp);
        mx = fmaxf(half_lo_to_float(m1), half_lo_to_float(m1 >> 16));
      } else {
        if (cmax < BN) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c >= cmax) sv[c] = -INFINITY;
        }
        float tmp[BN];
#pragma unroll
        for (int c = 0; c < BN; ++c) tmp[c] = sv[c];
        mx = tree_max3<BN>(tmp);
        if constexpr (STATS) {
#pragma unroll
          for (int c = 0; c < BN; ++c) tmp[c] = c < cmax ? sv[c] : INFINITY;
          mn = tree_min3<BN>(tmp);
        }
      }
      if constexpr (STATS) {
        if (cmax > 0) {
          st_acc = fmaxf(st_acc, fmaxf(fabsf(mx), fabsf(mn)));
          st_rec = fmaxf(st_rec, fmaxf(fabsf(mx + c_raw), fabsf(mn + c_raw)));
        }
      }
      const float bm = (mx == -INFINITY) ? -INFINITY : (mx + c_raw) * sl2;
      // The max block j-1 was computed with (the other set's), then the lazy rescale
      // decision: m only moves when this block raises it by more than kRescaleLog2.
      float m_prev = -INFINITY;
      if (j > 0) {
        if (!warp_wait(&s.mxf[quad][set ^ 1], ((j - 1) >> 1) & 1, abort_flag, 0x340)) { ok = false; break; }
        m_prev = s.xm[set ^ 1][r];
      }
      const float m_new = fmaxf(m_prev, bm);
      const bool need = j > 0 && m_new > m_prev + kRescaleLog2;
      const float m_cur = (j == 0 || need) ? m_new : m_prev;
      const bool rescale = __any_sync(0xffffffffu, need);
      const float alpha = need ? ex2_approx(m_prev - m_new) : 1.0f;
      s.xm[set][r] = m_cur;
      __syncwarp();
      mbar_arrive_if(&s.mxf[quad][set], lane == 0);

      // p = exp2((S' + c) * scale*log2e - m): MUFU ex2 per element, packed fp32 arithmetic per
      // pair, row sums in four independent pair accumulators.
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kPairs];
      if constexpr (F16ACC) {
        // x = (S' + (c - m / sl2)) * sl2
        const float b16 = (m_cur == -INFINITY) ? 0.0f : c_raw - m_cur * p.inv_scale_log2;
#pragma unroll
        for (int c = 0; c < kPairs; ++c) {
          float y0, y1, x0, x1;
          add_f16x2_f32(y0, y1, hp[c], b16);
          fmul2(x0, x1, y0, y1, sl2, sl2);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          const int a = (c & 3) * 2;
          fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
          pk[c] = pack_half2(p0, p1);
        }
      } else {
        const float bias = (m_cur == -INFINITY) ? 0.0f : c_raw * sl2 - m_cur;
#pragma unroll
        for (int c = 0; c < kPairs; ++c) {
          float x0, x1;
          ffma2(x0, x1, sv[2 * c], sv[2 * c + 1], sl2, sl2, bias, bias);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          const int a = (c & 3) * 2;
          fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
          pk[c] = pack_half2(p0, p1);
        }
      }
      const float rowsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
      if (m_w != m_cur) l_w *= ex2_approx(m_w - m_cur);  // 0 while this set has no blocks yet
      l_w += rowsum;
      m_w = m_cur;
      // PV(j-1) has to be done before O is rescaled or P rewritten; the exponentials above
      // overlap it.
      if (j >= 1 && !warp_wait(&s.p_free[(j - 1) & 1], ((j - 1) >> 1) & 1, abort_flag, 0x320)) { ok = false; break; }
      tc_fence_after();
      if (rescale) {
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          tmem_ld_x16(tO + c * 16, w);
          tmem_ld_wait();
          reg_fence<16>(w);
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(w[e]) * alpha);
          tmem_st_x16(tO + c * 16, w);
        }
      }
#pragma unroll
      for (int c = 0; c < BN / 16; ++c) tmem_st_x8(tP + c * 8, pk + c * 8);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_if(&s.p_full, lane == 0);
    }

    // epilogue: combine the two sets' row sums, O / l -> fp16 -> swizzled staging (the Q
    // buffer; each set writes half of the columns) -> TMA store
    s.xsum[0][set][r] = l_w;
    s.xsum[1][set][r] = m_w;
    if constexpr (STATS) {
      s.xsum[2][set][r] = st_acc;
      s.xsum[3][set][r] = st_rec;
    }
    named_bar_sync(1, 32 * kSoftmaxWarps);
    const float l_o = s.xsum[0][set ^ 1][r];
    const float m_o = s.xsum[1][set ^ 1][r];
    const float m_f = fmaxf(m_w, m_o);  // the max O is scaled to (that of the last block)
    const float l_tot = (m_f == -INFINITY) ? 0.0f
                                           : l_w * ex2_approx(m_w - m_f) + l_o * ex2_approx(m_o - m_f);
    const bool have_o = ok && nblk > 0;
    if (have_o && !warp_wait(&s.o_full, 0, abort_flag, 0x310)) ok = false;
    // A tile without key blocks reaches here before any MMA: its Q load (into the buffer
    // reused as staging) must have landed before the staging is written.
    if (!have_o && !warp_wait(&s.q_full, 0, abort_flag, 0x330)) ok = false;
    tc_fence_after();
    const float inv_l = (l_tot > 0.0f) ? 1.0f / l_tot : 0.0f;
    uint8_t* stage = s.q;
#pragma unroll
    for (int c = 0; c < kOCols / 16; ++c) {
      uint32_t w[16];
      if (have_o && ok) {
        tmem_ld_x16(tO + set * kOCols + c * 16, w);
        tmem_ld_wait();
        reg_fence<16>(w);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = 0u;
      }
      uint32_t hh[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        hh[e] = pack_half2(__uint_as_float(w[2 * e]) * inv_l, __uint_as_float(w[2 * e + 1]) * inv_l);
      const int col = set * kOCols + c * 16;
      const int chunk = col / 64;
      const int u0 = (col % 64) / 8;
      uint8_t* rowp = stage + chunk * Smem::kQChunk + r * 128;
      *reinterpret_cast<uint4*>(rowp + ((u0 ^ (r & 7)) * 16)) = make_uint4(hh[0], hh[1], hh[2], hh[3]);
      *reinterpret_cast<uint4*>(rowp + (((u0 + 1) ^ (r & 7)) * 16)) = make_uint4(hh[4], hh[5], hh[6], hh[7]);
    }
    fence_proxy_async_smem();
    named_bar_sync(2, 32 * kSoftmaxWarps);
    if (warp == 0 && lane == 0) {
#pragma unroll
      for (int c = 0; c < Smem::kChunks; ++c) tma_store_3d(&mapO, stage + c * Smem::kQChunk, c * 64, q0, b * p.Hq + hq);
      tma_store_commit();
      tma_store_wait_all();
    }
    if (set == 0 && i < p.Sq) {
      if constexpr (STATS) {
        float* st = p.stats + ((static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i) * 2;
        st[0] = fmaxf(st_acc, s.xsum[2][1][r]);
        st[1] = fmaxf(st_rec, s.xsum[3][1][r]);
      }
      if (p.lse != nullptr) {
        const float lse = (l_tot > 0.0f) ? (m_f + log2f(l_tot)) * 0.69314718055994531f : -INFINITY;
        p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace twoset
}  // namespace pasa
