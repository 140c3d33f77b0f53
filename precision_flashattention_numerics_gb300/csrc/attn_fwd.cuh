// PASA attention forward on sm_103a: TMA -> shared memory -> tcgen05.mma -> TMEM, with the
// online softmax, the global-recovering offsets and the final rescale in the softmax warps.
//
// Method: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
// Inference" (arXiv 2503.01873), Abstract: FlashAttention in half precision where every key
// block K_j is shifted by its pseudo-average m_j before the fp16 score GEMM and the per-row
// offsets q_i . m_j are carried in fp32 and folded back into the online max and sum
// ("global recovering"). The shifted keys and the block means come from kshift_kernel.
//
// One CTA owns 256 query rows of one (batch, query head) as two 128-row tiles and walks the
// key blocks (kBlockRows = 112 keys) of its kv head. Warp roles (352 threads):
//   warps 0-3  softmax + epilogue for tile 0   (thread r <-> query row r <-> TMEM lane r)
//   warps 4-7  softmax + epilogue for tile 1
//   warp  8    TMA producer: Q once, then K'_j / V_j rings and 16-block chunks of means
//   warp  9    TMEM owner and MMA issuer for tile 0 (one thread)
//   warp 10    MMA issuer for tile 1 (one thread)
// TMEM (512 columns): S_t at t*128 (112 columns, P_t packed fp16 aliased onto its first
// 56), C_t at t*128+112 (16 columns: offsets of 16 consecutive key blocks), O_t at 256+t*128.
// Per key block j each tile's MMA thread issues PV_t(j-1) then QK_t(j), so the tensor core
// works on one tile while the softmax warps of the other tile run (ping-pong).
//
// Score modes: the QK^T accumulator is fp16 (F16ACC, the PASA regime) or fp32. SHIFT
// selects shifted keys + offsets (PASA) or raw keys (no shift: the naive fp16 kernel or the
// plain fp32-accumulate FlashAttention). P is rounded to fp16 and PV accumulates in fp32.
//
// Online softmax in log2 units: x = (S' + c) * scale * log2(e). The running max is only
// moved when a block raises it by more than kRescaleLog2 (so P <= 2^kRescaleLog2 in fp16);
// moving it rescales l and the O accumulator in TMEM by exp2(m_old - m_new).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "kshift.cuh"
#include "ptx.cuh"

namespace pasa {

constexpr int kTileRows = 128;       // query rows per tile (MMA M)
constexpr int kCtaRows = 256;        // two tiles per CTA
constexpr int kChunkBlocks = 16;     // key blocks per offsets MMA (its N)
constexpr int kAttnThreads = 352;
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  float* lse;        // [B, Hq, Sq] fp32 or nullptr
  int B, Hq, Hkv, Sq, Sk;
  int n_qblk;        // ceil(Sq / kCtaRows)
  float scale_log2;  // softmax scale * log2(e)
  float inv_scale_log2;  // 1 / scale_log2
};

template <int D, int KST, int VST>
struct AttnSmem {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr int kQTile = kTileRows * D * 2;
  static constexpr int kKTile = kBlockRows * D * 2;
  static constexpr int kMTile = kChunkBlocks * D * 2;
  static constexpr int kQChunk = kTileRows * 128;
  static constexpr int kKChunk = kBlockRows * 128;
  static constexpr int kMChunk = kChunkBlocks * 128;
  alignas(1024) uint8_t q[2][kQTile];   // also the O staging buffer of each tile
  alignas(1024) uint8_t k[KST][kKTile];
  alignas(1024) uint8_t v[VST][kKTile];
  alignas(1024) uint8_t m[2][kMTile];
  uint64_t q_full;
  uint64_t k_full[KST], k_empty[KST];  // empty barriers: one arrival per MMA warp
  uint64_t v_full[VST], v_empty[VST];
  uint64_t m_full[2], m_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain[2];
  uint64_t issued[2];  // MMA warp t has issued its batch for block j (phase j)
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float half_lo_to_float(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}

template <int D, bool F16ACC, bool SHIFT, bool CAUSAL, int KST, int VST>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                const __grid_constant__ CUtensorMap mapM, const AttnParams p) {
  using Smem = AttnSmem<D, KST, VST>;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Work item: heavy (late) query blocks first across all heads; neighbouring CTAs share a
  // kv head so K/V stay in L2.
  const int lin = blockIdx.x;
  const int hb = lin % (p.Hq * p.B);
  const int qb = p.n_qblk - 1 - lin / (p.Hq * p.B);
  const int hq = hb % p.Hq;
  const int b = hb / p.Hq;
  const int hk = hq / (p.Hq / p.Hkv);
  const int q0 = qb * kCtaRows;

  int nblk[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int lo = q0 + t * kTileRows;
    if (lo >= p.Sq) {
      nblk[t] = 0;
    } else {
      const int last = min(p.Sq, lo + kTileRows) - 1;
      const int kv_end = CAUSAL ? min(p.Sk, last + p.Sk - p.Sq + 1) : p.Sk;
      nblk[t] = kv_end > 0 ? (kv_end + kBlockRows - 1) / kBlockRows : 0;
    }
  }
  const int nblk_max = max(nblk[0], nblk[1]);

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < KST; ++i) { mbar_init(&s.k_full[i], 1); mbar_init(&s.k_empty[i], 2); }
    for (int i = 0; i < VST; ++i) { mbar_init(&s.v_full[i], 1); mbar_init(&s.v_empty[i], 2); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.m_full[i], 1);
      mbar_init(&s.m_empty[i], 2);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.o_full[i], 1);
    }
    mbar_init(&s.drain[0], 1);
    mbar_init(&s.drain[1], 1);
    mbar_init(&s.issued[0], 1);
    mbar_init(&s.issued[1], 1);
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
      mbar_arrive_expect_tx(&s.q_full, 2 * Smem::kQTile);
#pragma unroll
      for (int t = 0; t < 2; ++t)
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.q[t] + c * Smem::kQChunk, &mapQ, &s.q_full, c * 64, q0 + t * kTileRows, qz);
      int k_issued = 0, v_issued = 0, m_issued = 0;
      // Issue order K_0, K_1, V_0, K_2, V_1, ...: each K runs one block ahead of V, so an
      // MMA warp's wait for K_(j+1) never sits behind V_j. A slot is reused once both MMA
      // warps have released its previous block.
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
          tma_load_3d(s.k[ks] + c * Smem::kKChunk, &mapK, &s.k_full[ks], c * 64, j * kBlockRows, kz);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int vs = j % VST;
        if (!mbar_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, abort_flag, 0x103)) return false;
        mbar_arrive_expect_tx(&s.v_full[vs], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.v[vs] + c * Smem::kKChunk, &mapV, &s.v_full[vs], c * 64, j * kBlockRows, kz);
        v_issued = j + 1;
        return true;
      };
      bool pok = nblk_max == 0 || load_k(0);
      for (int j = 0; pok && j < nblk_max; ++j) {
        if (j + 1 < nblk_max && !load_k(j + 1)) break;
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
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 9 issues tile 0's MMAs and warp 10 tile 1's, one thread each, so one tile's waits
    // (for its softmax, or for a K/V tile) overlap the other tile's MMA issue. Both warps
    // walk every key block: for a block its tile does not use, a warp still waits for the
    // block to be loaded and then arrives on the slot's release barrier without a commit.
    // Each release barrier takes one arrival per warp, and a warp only releases a slot after
    // seeing its current block loaded, so slots are never released early.
    // The two warps pass a token so that the tensor core still alternates between the tiles
    // (tile 0's batch for block j after tile 1's batch for block j-1, tile 1's after tile
    // 0's for block j): one tile's softmax runs while the other tile's batch executes. A
    // warp does all its other waits while the other warp's batch is executing.
    const int t = warp - 9;
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(kTileRows, kBlockRows, !F16ACC, false);
      constexpr uint32_t id_c = idesc_f16(kTileRows, kChunkBlocks, true, false);
      constexpr uint32_t id_o = idesc_f16(kTileRows, D, true, true);
      // Descriptor words: the high word is one constant per layout, the low word of every
      // operand is its buffer's base word plus a compile-time offset (one add per MMA).
      constexpr uint32_t hi_kmaj = sdesc_hi_sw128(1024);
      constexpr uint32_t hi_v = sdesc_hi_sw128(1024);
      const uint32_t q_lo = sdesc_lo(smem_u32(s.q[t]), 16);
      const uint32_t k_lo0 = sdesc_lo(smem_u32(s.k[0]), 16);
      const uint32_t v_lo0 = sdesc_lo(smem_u32(s.v[0]), Smem::kKChunk);
      const uint32_t m_lo0 = sdesc_lo(smem_u32(s.m[0]), 16);
      constexpr uint32_t kKStride = sizeof(s.k[0]) >> 4;  // descriptor units per ring slot
      constexpr uint32_t kVStride = sizeof(s.v[0]) >> 4;
      constexpr uint32_t kMStride = sizeof(s.m[0]) >> 4;
      const int my_nblk = t == 0 ? nblk[0] : nblk[1];
      const uint32_t tS = tmem + t * 128;
      const uint32_t tO = tmem + 256 + t * 128;
      // Every descriptor word of a batch is formed before the waits that gate it, so once
      // the gate opens the thread issues nothing but the MMAs (the softmax warps sharing its
      // SMSP are at their busiest then).
      uint32_t qd[D / 16];
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) qd[kk] = q_lo + (((kk / 4) * Smem::kQChunk + (kk % 4) * 32) >> 4);
      bool ok = mbar_wait(&s.q_full, 0, abort_flag, 0x201 + 0x10 * t);
      tc_fence_after();
      for (int j = 0; ok && j <= nblk_max; ++j) {
        uint32_t vd[kBlockRows / 16], kd[D / 16];
        {
          const uint32_t v_lo = v_lo0 + ((j + VST - 1) % VST) * kVStride;
          const uint32_t k_lo = k_lo0 + (j % KST) * kKStride;
#pragma unroll
          for (int kk = 0; kk < kBlockRows / 16; ++kk) vd[kk] = v_lo + kk * (2048 >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) kd[kk] = k_lo + (((kk / 4) * Smem::kKChunk + (kk % 4) * 32) >> 4);
        }
        if (j < nblk_max) {
          const int ci = j / kChunkBlocks;
          if (!mbar_wait(&s.k_full[j % KST], (j / KST) & 1, abort_flag, 0x202 + 0x10 * t)) break;
          if (SHIFT && (j % kChunkBlocks) == 0 &&
              !mbar_wait(&s.m_full[ci & 1], (ci >> 1) & 1, abort_flag, 0x203 + 0x10 * t))
            break;
        }
        if (j >= 1 && !mbar_wait(&s.v_full[(j - 1) % VST], ((j - 1) / VST) & 1, abort_flag, 0x204 + 0x10 * t)) break;
        if (j >= 1 && j - 1 < my_nblk && !mbar_wait(&s.p_full[t], (j - 1) & 1, abort_flag, 0x205 + 0x10 * t)) break;
        // token: tile 0 waits for tile 1's batch of block j-1, tile 1 for tile 0's of block j
        if (t == 0 && j >= 1 && !mbar_wait(&s.issued[1], (j - 1) & 1, abort_flag, 0x208)) break;
        if (t == 1 && !mbar_wait(&s.issued[0], j & 1, abort_flag, 0x218)) break;
        tc_fence_after();
        if (j >= 1) {
          const int vs = (j - 1) % VST;
          if (j - 1 < my_nblk) {
            const uint32_t acc0 = j - 1 > 0 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kBlockRows / 16; ++kk)
              mma_ts_w(tO, tS + kk * 8, vd[kk], hi_v, id_o, kk > 0 ? 1u : acc0);
            if (j - 1 == my_nblk - 1) mma_commit(&s.o_full[t]);
            mma_commit(&s.v_empty[vs]);
          } else {
            mbar_arrive(&s.v_empty[vs]);
          }
        }
        if (j < nblk_max) {
          const int ks = j % KST;
          const int ci = j / kChunkBlocks;
          const bool chunk_start = SHIFT && (j % kChunkBlocks) == 0;
          if (j < my_nblk) {
            if (chunk_start) {
              const uint32_t m_lo = m_lo0 + (ci & 1) * kMStride;
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off_q = ((kk / 4) * Smem::kQChunk + (kk % 4) * 32) >> 4;
                const uint32_t off_m = ((kk / 4) * Smem::kMChunk + (kk % 4) * 32) >> 4;
                mma_ss_w(tS + kBlockRows, q_lo + off_q, hi_kmaj, m_lo + off_m, hi_kmaj, id_c, kk > 0 ? 1u : 0u);
              }
            }
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) mma_ss_w(tS, qd[kk], hi_kmaj, kd[kk], hi_kmaj, id_s, kk > 0 ? 1u : 0u);
            mma_commit(&s.s_full[t]);
            mma_commit(&s.k_empty[ks]);
            if (chunk_start) mma_commit(&s.m_empty[ci & 1]);
          } else {
            mbar_arrive(&s.k_empty[ks]);
            if (chunk_start) mbar_arrive(&s.m_empty[ci & 1]);
          }
        }
        mbar_arrive(&s.issued[t]);
      }
      // all MMAs issued by this thread complete before TMEM can be released
      mma_commit(&s.drain[t]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain[t], 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * 128;
    const uint32_t tC = tS + kBlockRows;
    const uint32_t tO = tmem + lane_base + 256 + t * 128;
    const int i = q0 + t * kTileRows + r;
    const int limit = (i < p.Sq) ? (CAUSAL ? min(p.Sk, max(0, i + p.Sk - p.Sq + 1)) : p.Sk) : 0;
    const float sl2 = p.scale_log2;
    const int my_nblk = t == 0 ? nblk[0] : nblk[1];  // keeps nblk in registers
    float m_run = -INFINITY, l_run = 0.0f;
    bool ok = true;

    for (int j = 0; j < my_nblk; ++j) {
      if (!mbar_wait(&s.s_full[t], j & 1, abort_flag, 0x300 + t)) { ok = false; break; }
      tc_fence_after();
      // All loads of this block in flight, one wait, then a register fence so no use of the
      // loaded registers is scheduled before the wait. fp16 scores (F16ACC) are loaded two per
      // register; their row max is taken in f16x2 and each score enters fp32 through one
      // mixed-precision add (no separate conversion). fp32 scores are used as loaded.
      constexpr int kPairs = kBlockRows / 2;
      uint32_t hp[F16ACC ? kPairs : 1];
      float sv[F16ACC ? 1 : kBlockRows];
      uint32_t cw = 0;
      const int cmax = limit - j * kBlockRows;
      float mx;
      if constexpr (F16ACC) {
        static_assert(kBlockRows == 112, "load split below");
        tmem_ld_x16_pack16(tS + 0, hp + 0);
        tmem_ld_x16_pack16(tS + 32, hp + 16);
        tmem_ld_x16_pack16(tS + 64, hp + 32);
        tmem_ld_x8_pack16(tS + 96, hp + 48);
        if (SHIFT) tmem_ld_x1(tC + (j % kChunkBlocks), cw);
        tmem_ld_wait();
        reg_fence<kPairs>(hp);
        reg_fence<1>(&cw);
        if (cmax < kBlockRows) {
#pragma unroll
          for (int c = 0; c < kPairs; ++c) {
            const uint32_t lo = (2 * c < cmax) ? (hp[c] & 0xFFFFu) : 0xFC00u;        // -inf
            const uint32_t hi = (2 * c + 1 < cmax) ? (hp[c] & 0xFFFF0000u) : 0xFC000000u;
            hp[c] = lo | hi;
          }
        }
        // f16x2 max tree: 56 -> 28 -> 14 -> 7 -> 4 -> 2 -> 1
        uint32_t m28[28], m14[14], m7[7];
#pragma unroll
        for (int c = 0; c < 28; ++c) m28[c] = hmax2(hp[2 * c], hp[2 * c + 1]);
#pragma unroll
        for (int c = 0; c < 14; ++c) m14[c] = hmax2(m28[2 * c], m28[2 * c + 1]);
#pragma unroll
        for (int c = 0; c < 7; ++c) m7[c] = hmax2(m14[2 * c], m14[2 * c + 1]);
        const uint32_t m4a = hmax2(m7[0], m7[1]), m4b = hmax2(m7[2], m7[3]), m4c = hmax2(m7[4], m7[5]);
        const uint32_t m1 = hmax2(hmax2(m4a, m4b), hmax2(m4c, m7[6]));
        mx = fmaxf(half_lo_to_float(m1), half_lo_to_float(m1 >> 16));
      } else {
#pragma unroll
        for (int c = 0; c < kBlockRows / 16; ++c) tmem_ld_x16(tS + c * 16, reinterpret_cast<uint32_t*>(sv) + c * 16);
        if (SHIFT) tmem_ld_x1(tC + (j % kChunkBlocks), cw);
        tmem_ld_wait();
        reg_fence<kBlockRows>(reinterpret_cast<uint32_t*>(sv));
        reg_fence<1>(&cw);
        if (cmax < kBlockRows) {
#pragma unroll
          for (int c = 0; c < kBlockRows; ++c)
            if (c >= cmax) sv[c] = -INFINITY;
        }
        // fp32 max tree with three-input max: 112 -> 38 -> 13 -> 5 -> 2 -> 1
        float m38[38], m13[13];
#pragma unroll
        for (int c = 0; c < 37; ++c) m38[c] = fmax3(sv[3 * c], sv[3 * c + 1], sv[3 * c + 2]);
        m38[37] = sv[111];
#pragma unroll
        for (int c = 0; c < 12; ++c) m13[c] = fmax3(m38[3 * c], m38[3 * c + 1], m38[3 * c + 2]);
        m13[12] = fmaxf(m38[36], m38[37]);
        const float m5a = fmax3(m13[0], m13[1], m13[2]), m5b = fmax3(m13[3], m13[4], m13[5]);
        const float m5c = fmax3(m13[6], m13[7], m13[8]), m5d = fmax3(m13[9], m13[10], m13[11]);
        mx = fmaxf(fmax3(m5a, m5b, m5c), fmaxf(m5d, m13[12]));
      }
      const float c_raw = SHIFT ? __uint_as_float(cw) : 0.0f;
      const float bm = (mx == -INFINITY) ? -INFINITY : (mx + c_raw) * sl2;
      const float m_new = fmaxf(m_run, bm);
      if (j == 0) {
        m_run = m_new;
      } else {
        const bool need = m_new > m_run + kRescaleLog2;
        if (__any_sync(0xffffffffu, need)) {
          const float alpha = need ? ex2_approx(m_run - m_new) : 1.0f;
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
          if (need) {
            l_run *= alpha;
            m_run = m_new;
          }
        }
      }
      // p = exp2((S' + c) * scale*log2e - m): MUFU ex2 per element, packed fp32 arithmetic per
      // pair, row sums in four independent pair accumulators.
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kPairs];
      if constexpr (F16ACC) {
        // x = (S' + (c - m / sl2)) * sl2
        const float b16 = (m_run == -INFINITY) ? 0.0f : c_raw - m_run * p.inv_scale_log2;
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
        const float bias = (m_run == -INFINITY) ? 0.0f : c_raw * sl2 - m_run;
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
      l_run += rowsum;
#pragma unroll
      for (int c = 0; c < kBlockRows / 16; ++c) tmem_st_x8(tS + c * 8, pk + c * 8);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.p_full[t]);
    }

    // epilogue: O / l -> fp16 -> swizzled staging (the tile's Q buffer) -> TMA store
    const bool have_o = ok && my_nblk > 0;
    if (have_o && !mbar_wait(&s.o_full[t], 0, abort_flag, 0x310 + t)) ok = false;
    // A tile without key blocks reaches here before any MMA: its Q load (into the buffer
    // reused as staging) must have landed before the staging is written.
    if (!have_o && !mbar_wait(&s.q_full, 0, abort_flag, 0x320 + t)) ok = false;
    tc_fence_after();
    const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    uint8_t* stage = s.q[t];
#pragma unroll
    for (int c = 0; c < D / 16; ++c) {
      uint32_t w[16];
      if (have_o && ok) {
        tmem_ld_x16(tO + c * 16, w);
        tmem_ld_wait();
        reg_fence<16>(w);
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = 0u;
      }
      uint32_t h[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        h[e] = pack_half2(__uint_as_float(w[2 * e]) * inv_l, __uint_as_float(w[2 * e + 1]) * inv_l);
      const int col = c * 16;
      const int chunk = col / 64;
      const int u0 = (col % 64) / 8;
      uint8_t* rowp = stage + chunk * Smem::kQChunk + r * 128;
      *reinterpret_cast<uint4*>(rowp + ((u0 ^ (r & 7)) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(rowp + (((u0 + 1) ^ (r & 7)) * 16)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + t, 128);
    if (r == 0 && q0 + t * kTileRows < p.Sq) {
#pragma unroll
      for (int c = 0; c < Smem::kChunks; ++c)
        tma_store_3d(&mapO, stage + c * Smem::kQChunk, c * 64, q0 + t * kTileRows, b * p.Hq + hq);
      tma_store_commit();
      tma_store_wait_all();
    }
    if (p.lse != nullptr && i < p.Sq) {
      const float lse = (l_run > 0.0f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i] = lse;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

}  // namespace pasa
