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
// key blocks (kBlockRows = 112 keys) of its kv head. Warp roles (320 threads):
//   warps 0-3  softmax + epilogue for tile 0   (thread r <-> query row r <-> TMEM lane r)
//   warps 4-7  softmax + epilogue for tile 1
//   warp  8    TMA producer: Q once, then K'_j / V_j rings and 16-block chunks of means
//   warp  9    TMEM owner and MMA issuer (one thread)
// TMEM (512 columns): S_t at t*128 (112 columns, P_t packed fp16 aliased onto its first
// 56), C_t at t*128+112 (16 columns: offsets of 16 consecutive key blocks), O_t at 256+t*128.
// Per key block j the MMA thread issues, for each tile, PV_t(j-1) then QK_t(j), so the tensor
// core works on one tile while the softmax warps of the other tile run (ping-pong).
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
constexpr int kAttnThreads = 320;
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  float* lse;        // [B, Hq, Sq] fp32 or nullptr
  int B, Hq, Hkv, Sq, Sk;
  int n_qblk;        // ceil(Sq / kCtaRows)
  float scale_log2;  // softmax scale * log2(e)
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
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t m_full[2], m_empty[2];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t drain;
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
    for (int i = 0; i < KST; ++i) { mbar_init(&s.k_full[i], 1); mbar_init(&s.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&s.v_full[i], 1); mbar_init(&s.v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.m_full[i], 1);
      mbar_init(&s.m_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 4);
      mbar_init(&s.o_full[i], 1);
    }
    mbar_init(&s.drain, 1);
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
      for (int j = 0; j < nblk_max; ++j) {
        if (SHIFT && (j % kChunkBlocks) == 0) {
          const int ci = j / kChunkBlocks, slot = ci & 1;
          if (!mbar_wait(&s.m_empty[slot], ((ci >> 1) & 1) ^ 1, abort_flag, 0x101)) break;
          mbar_arrive_expect_tx(&s.m_full[slot], Smem::kMTile);
#pragma unroll
          for (int c = 0; c < Smem::kChunks; ++c)
            tma_load_3d(s.m[slot] + c * Smem::kMChunk, &mapM, &s.m_full[slot], c * 64, j, kz);
          m_issued = ci + 1;
        }
        const int ks = j % KST;
        if (!mbar_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, abort_flag, 0x102)) break;
        mbar_arrive_expect_tx(&s.k_full[ks], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.k[ks] + c * Smem::kKChunk, &mapK, &s.k_full[ks], c * 64, j * kBlockRows, kz);
        k_issued = j + 1;
        const int vs = j % VST;
        if (!mbar_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, abort_flag, 0x103)) break;
        mbar_arrive_expect_tx(&s.v_full[vs], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.v[vs] + c * Smem::kKChunk, &mapV, &s.v_full[vs], c * 64, j * kBlockRows, kz);
        v_issued = j + 1;
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
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16(kTileRows, kBlockRows, !F16ACC, false);
      constexpr uint32_t id_c = idesc_f16(kTileRows, kChunkBlocks, true, false);
      constexpr uint32_t id_o = idesc_f16(kTileRows, D, true, true);
      const uint32_t q_addr[2] = {smem_u32(s.q[0]), smem_u32(s.q[1])};
      bool ok = mbar_wait(&s.q_full, 0, abort_flag, 0x201);
      tc_fence_after();
      for (int j = 0; ok && j <= nblk_max; ++j) {
        const bool has_k = j < nblk_max;
        const int ks = j % KST;
        const int ci = j / kChunkBlocks;
        const bool chunk_start = SHIFT && has_k && (j % kChunkBlocks) == 0;
        if (has_k && !mbar_wait(&s.k_full[ks], (j / KST) & 1, abort_flag, 0x202)) break;
        if (chunk_start && !mbar_wait(&s.m_full[ci & 1], (ci >> 1) & 1, abort_flag, 0x203)) break;
        bool v_waited = false;
        const int vs = (j + VST - 1) % VST;  // slot of block j-1
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t tS = tmem + t * 128;
          const uint32_t tO = tmem + 256 + t * 128;
          if (j >= 1 && j - 1 < nblk[t]) {
            if (!v_waited) {
              if (!mbar_wait(&s.v_full[vs], ((j - 1) / VST) & 1, abort_flag, 0x204)) { ok = false; break; }
              v_waited = true;
            }
            if (!mbar_wait(&s.p_full[t], (j - 1) & 1, abort_flag, 0x205)) { ok = false; break; }
            tc_fence_after();
            const uint32_t v_addr = smem_u32(s.v[vs]);
#pragma unroll
            for (int kk = 0; kk < kBlockRows / 16; ++kk) {
              const uint64_t vd = sdesc_sw128(v_addr + kk * 2048, Smem::kKChunk, 1024);
              mma_ts(tO, tS + kk * 8, vd, id_o, (j - 1 > 0 || kk > 0) ? 1u : 0u);
            }
            if (j - 1 == nblk[t] - 1) mma_commit(&s.o_full[t]);
          }
          if (has_k && j < nblk[t]) {
            if (chunk_start) {
              const uint32_t m_addr = smem_u32(s.m[ci & 1]);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint64_t ad = sdesc_sw128(q_addr[t] + (kk / 4) * Smem::kQChunk + (kk % 4) * 32, 16, 1024);
                const uint64_t md = sdesc_sw128(m_addr + (kk / 4) * Smem::kMChunk + (kk % 4) * 32, 16, 1024);
                mma_ss(tS + kBlockRows, ad, md, id_c, kk > 0 ? 1u : 0u);
              }
            }
            const uint32_t k_addr = smem_u32(s.k[ks]);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t ad = sdesc_sw128(q_addr[t] + (kk / 4) * Smem::kQChunk + (kk % 4) * 32, 16, 1024);
              const uint64_t kd = sdesc_sw128(k_addr + (kk / 4) * Smem::kKChunk + (kk % 4) * 32, 16, 1024);
              mma_ss(tS, ad, kd, id_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&s.s_full[t]);
          }
        }
        if (!ok) break;
        if (has_k) mma_commit(&s.k_empty[ks]);
        if (chunk_start) mma_commit(&s.m_empty[ci & 1]);
        if (v_waited) mma_commit(&s.v_empty[vs]);
      }
      // all MMAs issued by this thread complete before TMEM can be released
      mma_commit(&s.drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
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
      // all loads of this block in flight, one wait, then a register fence so no use of
      // the loaded registers is scheduled before the wait
      uint32_t sr[kBlockRows];
#pragma unroll
      for (int c = 0; c < kBlockRows / 16; ++c) tmem_ld_x16(tS + c * 16, sr + c * 16);
      uint32_t cw = 0;
      if (SHIFT) tmem_ld_x1(tC + (j % kChunkBlocks), cw);
      tmem_ld_wait();
      reg_fence<kBlockRows>(sr);
      reg_fence<1>(&cw);
      float sv[kBlockRows];
#pragma unroll
      for (int c = 0; c < kBlockRows; ++c) sv[c] = F16ACC ? half_lo_to_float(sr[c]) : __uint_as_float(sr[c]);
      const float c_raw = SHIFT ? __uint_as_float(cw) : 0.0f;
      const int cmax = limit - j * kBlockRows;
      if (cmax < kBlockRows) {
#pragma unroll
        for (int c = 0; c < kBlockRows; ++c)
          if (c >= cmax) sv[c] = -INFINITY;
      }
      // row max: three-input max, four independent chains
      float mxa = sv[0], mxb = sv[1], mxc = sv[2], mxd = sv[3];
#pragma unroll
      for (int c = 4; c + 8 <= kBlockRows; c += 8) {
        mxa = fmax3(mxa, sv[c], sv[c + 1]);
        mxb = fmax3(mxb, sv[c + 2], sv[c + 3]);
        mxc = fmax3(mxc, sv[c + 4], sv[c + 5]);
        mxd = fmax3(mxd, sv[c + 6], sv[c + 7]);
      }
      mxa = fmax3(mxa, sv[kBlockRows - 4], sv[kBlockRows - 3]);
      mxb = fmax3(mxb, sv[kBlockRows - 2], sv[kBlockRows - 1]);
      const float mx = fmaxf(fmaxf(mxa, mxb), fmaxf(mxc, mxd));
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
      const float bias = (m_run == -INFINITY) ? 0.0f : c_raw * sl2 - m_run;
      // p = exp2(S' * scale*log2e + (c * scale*log2e - m)): one packed FMA per pair, MUFU
      // ex2 per element, packed fp32 row sums in four independent accumulators
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[kBlockRows / 2];
#pragma unroll
      for (int c = 0; c < kBlockRows / 2; ++c) {
        float x0, x1;
        ffma2(x0, x1, sv[2 * c], sv[2 * c + 1], sl2, sl2, bias, bias);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        const int a = (c & 3) * 2;
        fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
        pk[c] = pack_half2(p0, p1);
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
