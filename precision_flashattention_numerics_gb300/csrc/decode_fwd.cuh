// PASA decode attention on sm_103a: a few query rows per kv head against a key cache, with
// the MMA operands swapped so that the 128 keys of a block fill the tcgen05 M dimension.
//
// Method: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
// Inference" (arXiv 2503.01873), Abstract: FlashAttention in half precision where each key
// block K_j is shifted by its pseudo-average m_j before the fp16 score GEMM, and the offsets
// q . m_j are added back in fp32 to the online max and sum. The method targets long-sequence
// inference; there a kv head meets only rows = g * Sq query rows per step (the g query heads
// that share it, Sq new tokens each), far fewer than the 128 rows of a tcgen05 MMA. This
// kernel therefore computes the transposed products, with NQ = 16 or 32 >= rows (the packed
// query rows, zero-padded by TMA):
//   S'^T (128 keys x NQ) = K'_j Q^T        A = K'_j  (K-major, as TMA writes it)
//                                          B = Q     (K-major)
//   O^T  (128 dims x NQ) += V_j^T P_j^T    A = V_j   (MN-major: the same tile, read along D)
//                                          B = P_j   (K-major, fp16, written by the softmax)
// Thread t of the four softmax warps owns TMEM lane t: key t of the current block for the
// scores and output dim t for O. The max of a query column over the block's keys is a
// reduction across the 128 threads: in each warp a reduce-scatter over shuffles (each level
// halves the values a lane holds, so NQ values take NQ + 0-1 shuffles instead of 5 NQ), then
// the four warps' results through shared memory. Each thread sums the probabilities of its
// own key (rescaled with its column's max); the 128 partial sums are reduced once at the end.
// The offsets q . m_j of a 16-block chunk are computed on the CUDA cores (NQ x 16 dot
// products of length 128 in fp32) when the chunk's means arrive.
//
// Score modes as in attn_fwd_kernel: F16ACC (fp16 score accumulator) or fp32, SHIFT (K' and
// offsets) or raw keys, F16PV (fp16 O accumulator and fp16 per-thread row sums, added in
// fp32 across threads at the end and rounded to fp16 once). Lazy rescaling: a column's max
// moves only when a block raises it by more than kRescaleLog2; every thread takes the same
// decision from the same shared maxima.
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue; warp 4 TMA producer (Q once, K'_j
// one block ahead of V_j, 16-block means chunks); warp 5 TMEM owner, one thread issuing
// QK(j+1) before PV(j). Split keys (grid.y) as in attn_fwd_kernel: a split writes O / l in
// fp32 and m + log2 l for combine_splits_kernel; or, with `cluster`, the splits of a kv head
// run as one thread-block cluster: each leaves its unnormalised O (in the shared memory of
// its first K' slot), m and l, and after a cluster barrier the CTA of rank r merges the rows
// q = r, r + splits, ... reading every split's values through distributed shared memory.
//
// Every wait is bounded (see ptx.cuh). The softmax warps meet at named barriers inside the
// block loop, so after a failed wait they keep iterating (skipping the work, not the
// barriers) instead of leaving the loop early.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "attn_fwd.cuh"
#include "ptx.cuh"

namespace pasa {

// Threads of a decode CTA with G softmax warpgroups: 4 G softmax warps, the TMA producer
// and the TMEM-owning MMA warp.
__host__ __device__ constexpr int dec_threads(int G) { return 32 * (4 * G + 2); }

struct DecodeParams {
  __half* o;          // [planes][rows][128] fp16 (the [B, Hq, Sq, D] output)
  float* lse;         // [planes * rows] natural-log LSE, or nullptr (unsplit launches)
  float* part_o;      // split keys: [splits][planes * rows][128] fp32 O / l, else nullptr
  float* part_lse;    // split keys: [splits][planes * rows] m + log2 l
  int rows;           // packed query rows per kv head, g * sq <= NQ
  int sq;             // query rows per head: packed row r is query r mod sq of head r / sq
  int Sk, nbt;        // keys in the cache and key blocks, ceil(Sk / 128)
  int bps;            // key blocks per split, 0 = one CTA per kv head
  int causal;
  float scale_log2;   // softmax scale * log2(e)
  int cluster;        // 1: the splits of a kv head form one thread-block cluster (grid.y) and
                      // merge their partial results through distributed shared memory
  const float* kscale;  // FP8: [planes][kstride] fp32 e4m3 scale of each key block
  int kstride;
  // The first key block (global index) that the kernel queued ahead of this launch rewrites
  // (a cache refresh, with this launch's programmatic dependence on it): its keys, means and
  // scales, and those of every later block, are read only after griddep_wait(). INT_MAX:
  // nothing to wait for.
  int dep_block;
};

template <int NQ, int KST, int VST, bool FP8 = false, int G = 1>
struct DecodeSmem {
  static constexpr int D = 128, BN = 128;
  static constexpr int kTile = BN * D * 2;            // one fp16 block of V (or K')
  static constexpr int kKTile = BN * D * (FP8 ? 1 : 2);   // one block of keys: fp16, or e4m3 codes
  static constexpr int kKChunks = FP8 ? 1 : 2;        // 128-byte atom columns of a key row
  static constexpr int kChunk = BN * 128;             // one 64-column (128-byte) atom column of it
  static constexpr int kQTile = NQ * D * 2, kQChunk = NQ * 128;
  static constexpr int kPTile = NQ * BN * 2, kPChunk = NQ * 128;
  static constexpr int kMTile = kChunkBlocks * D * 2, kMChunk = kChunkBlocks * 128;
  alignas(1024) uint8_t k[KST][kKTile];
  alignas(1024) uint8_t v[VST][kTile];
  alignas(1024) uint8_t q[kQTile];
  alignas(1024) uint8_t q8[FP8 ? NQ * 128 : 16];        // FP8: e4m3 codes of Q, one atom per row
  alignas(1024) uint8_t pt[G][2][kPTile];             // per group: P_j (rows = queries, K = keys), 2 buffers
  alignas(1024) uint8_t m[2][kMTile];
  alignas(16) float cv[G][2][kChunkBlocks][NQ];       // per group: offsets q . m_j of a chunk, by chunk parity
  alignas(16) float red[G][2][4][NQ];                 // per group: per-warp column maxima, 2 buffers
  float exm[NQ], exl[NQ];                             // G = 2: group 1's m (log2) and l for the merge
  float cm[NQ], cl[NQ];                               // cluster merge: this split's m (log2) and l
  float sqs[NQ];                                      // FP8: the e4m3 scale of each query row
  uint64_t q_full;
  uint64_t q8_full;                                   // FP8: the softmax warps wrote Q's codes (4)
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t m_full[2], m_empty[2];
  uint64_t s_full[G][2], s_free[G][2];
  uint64_t p_full[G][2], p_free[G][2];
  uint64_t o_full[G], drain;
  uint32_t tmem_base;
  int abort_flag;
};

// Bounded wait by every lane of a warp; the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, uint32_t site) {
  const bool ok = mbar_wait(bar, parity, abort_flag, site);
  return __all_sync(0xffffffffu, ok);
}

// Warp reduce-scatter of NQ per-lane values (NQ = 16 or 32), one shuffle level per call: at
// lane offset OFF (16, 8, ..., 1) a lane keeps the half of its values selected by its lane
// bit OFF and receives the other half from lane ^ OFF. The result, left in v[0], is the
// reduction over all 32 lanes of column lane >> 1 (NQ = 16) or lane (NQ = 32).
template <int NQ, bool MAX, int OFF>
__device__ __forceinline__ void reduce_scatter_level(float* v, int lane) {
  constexpr int n = NQ * OFF / 16;   // values a lane still holds
  if constexpr (n >= 2) {
    constexpr int h = n / 2;
    const bool hi = (lane & OFF) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = hi ? v[i] : v[i + h];
      const float keep = hi ? v[i + h] : v[i];
      const float got = __shfl_xor_sync(0xffffffffu, send, OFF);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  } else {
    const float got = __shfl_xor_sync(0xffffffffu, v[0], OFF);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
  if constexpr (OFF > 1) reduce_scatter_level<NQ, MAX, OFF / 2>(v, lane);
}

template <int NQ, bool MAX>
__device__ __forceinline__ float warp_reduce_scatter(float* v, int lane) {
  static_assert(NQ == 16 || NQ == 32, "columns");
  reduce_scatter_level<NQ, MAX, 16>(v, lane);
  return v[0];
}

template <int NQ, bool F16ACC, bool SHIFT, bool F16PV, int KST, int VST, bool FP8 = false, int G = 1>
__global__ void __launch_bounds__(dec_threads(G), 1)
decode_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                  const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapM,
                  const DecodeParams p) {
  static_assert(!F16PV || F16ACC, "fp16 PV accumulation is a variant of the fp16-score mode");
  static_assert(!FP8 || (!F16ACC && !F16PV), "FP8 scores accumulate in fp32");
  static_assert(G == 1 || G == 2, "softmax groups");
  using Smem = DecodeSmem<NQ, KST, VST, FP8, G>;
  static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory per CTA");
  constexpr int D = 128, BN = 128;
  // per group: S_0, S_1 and O, NQ columns each, from column 3 NQ g
  constexpr uint32_t kTmemCols = G * 3 * NQ <= 64 ? 64 : (G * 3 * NQ <= 128 ? 128 : 256);
  constexpr int kProdWarp = 4 * G, kMmaWarp = 4 * G + 1;
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int plane = blockIdx.x;          // b * Hkv + kv head
  const int split = blockIdx.y;
  const int jb0 = split * p.bps;
  const int nblk = p.bps > 0 ? max(0, min(p.bps, p.nbt - jb0)) : p.nbt;

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    mbar_init(&s.q8_full, 4);
    for (int i = 0; i < KST; ++i) { mbar_init(&s.k_full[i], 1); mbar_init(&s.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&s.v_full[i], 1); mbar_init(&s.v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.m_full[i], 1);
      mbar_init(&s.m_empty[i], 4 * G);
      for (int g = 0; g < G; ++g) {
        mbar_init(&s.s_full[g][i], 1);
        mbar_init(&s.s_free[g][i], 4);
        mbar_init(&s.p_full[g][i], 4);
        mbar_init(&s.p_free[g][i], 1);
      }
    }
    for (int g = 0; g < G; ++g) mbar_init(&s.o_full[g], 1);
    mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == kProdWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      if (SHIFT) tma_prefetch_desc(&mapM);
      mbar_arrive_expect_tx(&s.q_full, Smem::kQTile);
#pragma unroll
      for (int c = 0; c < 2; ++c) tma_load_3d(s.q + c * Smem::kQChunk, &mapQ, &s.q_full, c * 64, 0, plane);
      int k_issued = 0, v_issued = 0, m_issued = 0;
      bool dep_done = false;
      auto dep_wait = [&](int first_global_block) {   // before reading a refreshed block
        if (!dep_done && first_global_block >= p.dep_block) {
          griddep_wait();
          dep_done = true;
        }
      };
      auto load_k = [&](int j) -> bool {
        if (SHIFT && (j % kChunkBlocks) == 0) {
          const int ci = j / kChunkBlocks, slot = ci & 1;
          dep_wait(jb0 + j + kChunkBlocks - 1);   // the chunk's last block
          if (!mbar_wait(&s.m_empty[slot], ((ci >> 1) & 1) ^ 1, abort_flag, 0x501)) return false;
          mbar_arrive_expect_tx(&s.m_full[slot], Smem::kMTile);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(s.m[slot] + c * Smem::kMChunk, &mapM, &s.m_full[slot], c * 64, jb0 + j, plane);
          m_issued = ci + 1;
        }
        const int ks = j % KST;
        dep_wait(jb0 + j);
        if (!mbar_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, abort_flag, 0x502)) return false;
        mbar_arrive_expect_tx(&s.k_full[ks], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kKChunks; ++c)
          tma_load_3d(s.k[ks] + c * Smem::kChunk, &mapK, &s.k_full[ks], c * 64, (jb0 + j) * BN, plane);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int vs = j % VST;
        if (!mbar_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, abort_flag, 0x503)) return false;
        mbar_arrive_expect_tx(&s.v_full[vs], Smem::kTile);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          tma_load_3d(s.v[vs] + c * Smem::kChunk, &mapV, &s.v_full[vs], c * 64, (jb0 + j) * BN, plane);
        v_issued = j + 1;
        return true;
      };
      // K runs G blocks ahead of V, matching the MMA thread (QK(j + G) before PV(j))
      bool pok = true;
      for (int j = 0; pok && j < G && j < nblk; ++j) pok = load_k(j);
      for (int j = 0; pok && j < nblk; ++j) {
        if (j + G < nblk && !load_k(j + G)) break;
        if (!load_v(j)) break;
      }
      if (*abort_flag) {
        // every copy this thread issued lands before the CTA's shared memory goes away
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
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA thread
    // Block j belongs to softmax group j mod G (its local index i = j / G picks the S and P
    // buffers); QK(j + G) is issued before PV(j).
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_f16_ab(BN, NQ, !F16ACC, false, false);
      constexpr uint32_t id_o = idesc_f16_ab(D, NQ, !F16PV, true, false);
      constexpr uint32_t hi = sdesc_hi_sw128(1024);
      const uint32_t q_lo = sdesc_lo(smem_u32(s.q), 16);
      const uint32_t k_lo0 = sdesc_lo(smem_u32(s.k[0]), 16);
      const uint32_t v_lo0 = sdesc_lo(smem_u32(s.v[0]), Smem::kChunk);   // MN-major: atoms along D are kChunk apart
      const uint32_t p_lo0 = sdesc_lo(smem_u32(s.pt[0]), 16);
      const uint32_t q8_lo = sdesc_lo(smem_u32(s.q8), 16);
      constexpr uint32_t id_s8 = idesc_e4m3(BN, NQ);
      constexpr uint32_t kKStride = sizeof(s.k[0]) >> 4, kVStride = sizeof(s.v[0]) >> 4;
      constexpr uint32_t kPStride = sizeof(s.pt[0][0]) >> 4;
      auto qk = [&](int j) -> bool {
        const int g = j % G, i = j / G;
        const int ks = j % KST, sb = i & 1;
        if (!mbar_wait(&s.k_full[ks], (j / KST) & 1, abort_flag, 0x601)) return false;
        if (i >= 2 && !mbar_wait(&s.s_free[g][sb], ((i >> 1) - 1) & 1, abort_flag, 0x602)) return false;
        const uint32_t tS = tmem + g * 3 * NQ + sb * NQ;
        tc_fence_after();
        const uint32_t k_lo = k_lo0 + ks * kKStride;
        if constexpr (FP8) {
          // e4m3 codes of K and Q, one 128-byte atom per row: four K-steps of 32 (32 bytes)
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_w(tS, k_lo + ((kk * 32) >> 4), hi, q8_lo + ((kk * 32) >> 4), hi, id_s8, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_k = ((kk / 4) * Smem::kChunk + (kk % 4) * 32) >> 4;
            const uint32_t off_q = ((kk / 4) * Smem::kQChunk + (kk % 4) * 32) >> 4;
            mma_ss_w(tS, k_lo + off_k, hi, q_lo + off_q, hi, id_s, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&s.s_full[g][sb]);
        mma_commit(&s.k_empty[ks]);
        return true;
      };
      auto pv = [&](int j) -> bool {
        const int g = j % G, i = j / G;
        const int vs = j % VST, pb = i & 1;
        if (!mbar_wait(&s.v_full[vs], (j / VST) & 1, abort_flag, 0x603)) return false;
        if (!mbar_wait(&s.p_full[g][pb], (i >> 1) & 1, abort_flag, 0x604)) return false;
        tc_fence_after();
        const uint32_t v_lo = v_lo0 + vs * kVStride, p_lo = p_lo0 + (g * 2 + pb) * kPStride;
        const uint32_t tO = tmem + g * 3 * NQ + 2 * NQ;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t off_p = ((kk / 4) * Smem::kPChunk + (kk % 4) * 32) >> 4;
          mma_ss_w(tO, v_lo + kk * (2048 >> 4), hi, p_lo + off_p, hi, id_o, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&s.p_free[g][pb]);
        mma_commit(&s.v_empty[vs]);
        if (j + G >= nblk) mma_commit(&s.o_full[g]);   // the group's last block
        return true;
      };
      bool ok = mbar_wait(FP8 ? &s.q8_full : &s.q_full, 0, abort_flag, 0x600);
      for (int j = 0; ok && j < G && j < nblk; ++j) ok = qk(j);
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + G < nblk && !qk(j + G)) break;
        if (!pv(j)) break;
      }
      // every MMA issued here completes before TMEM is released
      mma_commit(&s.drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain, 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    // Group g takes blocks g, g + G, ...; with G = 2 the two groups' results are merged by
    // group 0 at the end.
    const int g = warp >> 2;
    const int t = tid & 127;   // TMEM lane: key t of a block, output dim t
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tG = tmem + lane_base + g * 3 * NQ;   // this group's S_0, S_1, O
    const float sl2 = p.scale_log2;
    constexpr int kLaneShift = NQ == 16 ? 1 : 0;
    const int q_of_lane = lane >> kLaneShift;              // column held after a reduce-scatter
    const bool writer = (lane & ((1 << kLaneShift) - 1)) == 0;
    // keys visible to every query row (causal: row r sees keys < Sk - sq + 1 + r mod sq)
    const int kv_all = p.causal ? p.Sk - p.sq + 1 : p.Sk;
    float m_run[NQ], lsum[NQ];
    uint32_t lsum_h[NQ / 2];   // F16PV: fp16 partial row sums, two per register
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      m_run[q] = -INFINITY;
      lsum[q] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < NQ / 2; ++e) lsum_h[e] = 0u;
    bool ok = true;
    if (SHIFT || FP8) ok = warp_wait(&s.q_full, 0, abort_flag, 0x700);
    float sqv[FP8 ? NQ : 1];   // FP8: the e4m3 scale of each query row
    if constexpr (FP8) {
      if (g == 0) {
      // quantise Q to e4m3, one scale per row: sq = fp32(a / 448), a = max |q_row|,
      // code = e4m3_rn_satfinite(fp32(q * fp32(448 / a))) (a = 0: both 1). TPR consecutive
      // threads share a row, EPT elements each; the row maximum is a shuffle reduction.
      constexpr int TPR = 128 / NQ, EPT = D / TPR;
      const int qr = t / TPR, part = t % TPR;
      uint4 xv[EPT / 8];
#pragma unroll
      for (int i = 0; i < EPT / 8; ++i) {
        const int u = part * (EPT / 8) + i;   // 16-byte unit of the fp16 row
        xv[i] = *reinterpret_cast<const uint4*>(s.q + (u / 8) * Smem::kQChunk + qr * 128 + (((u % 8) ^ (qr & 7)) << 4));
      }
      uint32_t amax = 0;
#pragma unroll
      for (int i = 0; i < EPT / 8; ++i) {
        const uint32_t w4[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = __vmaxu2(amax, w4[e] & 0x7FFF7FFFu);
      }
      amax = max(amax & 0xFFFFu, amax >> 16);
#pragma unroll
      for (int off = 1; off < TPR; off <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float a = __half2float(__ushort_as_half(static_cast<unsigned short>(amax)));
      const float inv = a > 0.0f ? __fdiv_rn(448.0f, a) : 1.0f;
      if (part == 0) s.sqs[qr] = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
#pragma unroll
      for (int i = 0; i < EPT / 16; ++i) {   // 16 codes (one 16-byte unit of the e4m3 row) each
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half* h = reinterpret_cast<const __half*>(&xv[2 * i + e / 2]) + (e % 2) * 4;
          const uint16_t c01 = pack_e4m3x2(__fmul_rn(__half2float(h[0]), inv), __fmul_rn(__half2float(h[1]), inv));
          const uint16_t c23 = pack_e4m3x2(__fmul_rn(__half2float(h[2]), inv), __fmul_rn(__half2float(h[3]), inv));
          w[e] = c01 | (static_cast<uint32_t>(c23) << 16);
        }
        const int wu = part * (EPT / 16) + i;
        *reinterpret_cast<uint4*>(s.q8 + qr * 128 + ((wu ^ (qr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.q8_full);
      }
      named_bar_sync(3, 128 * G);   // every row's scale is in shared memory
#pragma unroll
      for (int q = 0; q < NQ; ++q) sqv[q] = s.sqs[q];
    }

    // FP8: block scales, loaded one block ahead so the load is off the score path
    const float* kscale_row = FP8 ? p.kscale + static_cast<size_t>(plane) * p.kstride : nullptr;
    bool dep_done = false;   // FP8: the block scales of refreshed blocks after griddep_wait()
    auto scale_of = [&](int global_block) {
      if (!dep_done && global_block >= p.dep_block) {
        griddep_wait();
        dep_done = true;
      }
      return __ldg(kscale_row + global_block);
    };
    float sk_next = (FP8 && g < nblk) ? scale_of(jb0 + g) : 1.0f;
    for (int j = g; j < nblk; j += G) {
      const int i = j / G;   // the group's local block index
      const int sb = i & 1;
      const int jg = jb0 + j;
      float sk = 1.0f;
      if constexpr (FP8) {
        sk = sk_next;
        if (j + G < nblk) sk_next = scale_of(jg + G);
      }
      if (SHIFT && (j % kChunkBlocks) == g) {   // the group's first block of a chunk
        // offsets of the chunk's 16 blocks: thread t takes block t % 16 and the query rows
        // t / 16 + 8 e; fp32 dot products over the 128 dims (both tiles 128-byte swizzled)
        const int ci = j / kChunkBlocks;
        if (ok) ok = warp_wait(&s.m_full[ci & 1], (ci >> 1) & 1, abort_flag, 0x701);
        if (ok) {
          const int blk = t & 15, qg = t >> 4;
          const uint8_t* mrow = s.m[ci & 1] + blk * 128;
          float acc[NQ / 8];
#pragma unroll
          for (int e = 0; e < NQ / 8; ++e) acc[e] = 0.0f;
#pragma unroll 4
          for (int u = 0; u < 16; ++u) {
            const int c = u >> 3, uu = u & 7;
            const uint4 mv = *reinterpret_cast<const uint4*>(mrow + c * Smem::kMChunk + ((uu ^ (blk & 7)) << 4));
            const __half2* mh = reinterpret_cast<const __half2*>(&mv);
#pragma unroll
            for (int e = 0; e < NQ / 8; ++e) {
              const int qr = qg + 8 * e;
              const uint4 qv =
                  *reinterpret_cast<const uint4*>(s.q + c * Smem::kQChunk + qr * 128 + ((uu ^ (qr & 7)) << 4));
              const __half2* qh = reinterpret_cast<const __half2*>(&qv);
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const float2 mf = __half22float2(mh[h]);
                const float2 qf = __half22float2(qh[h]);
                acc[e] = fmaf(qf.x, mf.x, acc[e]);
                acc[e] = fmaf(qf.y, mf.y, acc[e]);
              }
            }
          }
#pragma unroll
          for (int e = 0; e < NQ / 8; ++e) s.cv[g][ci & 1][blk][qg + 8 * e] = acc[e];
        }
        named_bar_sync(1 + g, 128);
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.m_empty[ci & 1]);
      }

      // scores of block j: this thread's key against the NQ query columns
      if (ok) ok = warp_wait(&s.s_full[g][sb], (i >> 1) & 1, abort_flag, 0x702);
      tc_fence_after();
      float y[NQ];
      {
        const uint32_t tS = tG + sb * NQ;
        if constexpr (F16ACC) {
          uint32_t h[NQ / 2];
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_ld_x8_pack16(tS + c * 16, h + c * 8);
          tmem_ld_wait();
          reg_fence<NQ / 2>(h);
#pragma unroll
          for (int e = 0; e < NQ / 2; ++e) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[e]));
            y[2 * e] = f.x;
            y[2 * e + 1] = f.y;
          }
        } else {
          uint32_t w[NQ];
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_ld_x16(tS + c * 16, w + c * 16);
          tmem_ld_wait();
          reg_fence<NQ>(w);
#pragma unroll
          for (int q = 0; q < NQ; ++q) y[q] = __uint_as_float(w[q]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.s_free[g][sb]);

      // recovered scores in log2 units, masked
      if constexpr (FP8) {   // dequantise: S = sq_q * sk_j * (codes product)
#pragma unroll
        for (int q = 0; q < NQ; ++q) y[q] *= sqv[q] * sk;
      }
      if constexpr (SHIFT) {
        const float4* cr = reinterpret_cast<const float4*>(s.cv[g][(j / kChunkBlocks) & 1][j % kChunkBlocks]);
#pragma unroll
        for (int c4 = 0; c4 < NQ / 4; ++c4) {
          const float4 c = cr[c4];
          y[4 * c4] = (y[4 * c4] + c.x) * sl2;
          y[4 * c4 + 1] = (y[4 * c4 + 1] + c.y) * sl2;
          y[4 * c4 + 2] = (y[4 * c4 + 2] + c.z) * sl2;
          y[4 * c4 + 3] = (y[4 * c4 + 3] + c.w) * sl2;
        }
      } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) y[q] *= sl2;
      }
      const int key = jg * BN + t;
      if ((jg + 1) * BN > kv_all) {   // a block some row does not see whole (uniform branch)
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const int lim = p.causal ? min(p.Sk, kv_all + q % p.sq) : p.Sk;
          if (key >= lim) y[q] = -INFINITY;
        }
      }

      // column maxima over the block's 128 keys
      {
        float v[NQ];
#pragma unroll
        for (int q = 0; q < NQ; ++q) v[q] = y[q];
        const float mx = warp_reduce_scatter<NQ, true>(v, lane);
        if (writer) s.red[g][sb][warp & 3][q_of_lane] = mx;
      }
      named_bar_sync(1 + g, 128);
      float alpha[NQ];
      bool resc = false;
      {
        const float4* r4 = reinterpret_cast<const float4*>(s.red[g][sb]);
#pragma unroll
        for (int c4 = 0; c4 < NQ / 4; ++c4) {
          const float4 a = r4[c4], b = r4[NQ / 4 + c4], c = r4[2 * (NQ / 4) + c4], d = r4[3 * (NQ / 4) + c4];
          const float bm[4] = {fmaxf(fmaxf(a.x, b.x), fmaxf(c.x, d.x)), fmaxf(fmaxf(a.y, b.y), fmaxf(c.y, d.y)),
                               fmaxf(fmaxf(a.z, b.z), fmaxf(c.z, d.z)), fmaxf(fmaxf(a.w, b.w), fmaxf(c.w, d.w))};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int q = 4 * c4 + e;
            alpha[q] = 1.0f;
            if (bm[e] > m_run[q] + kRescaleLog2) {   // also when m_run is still -inf
              alpha[q] = ex2_approx(m_run[q] - bm[e]);
              m_run[q] = bm[e];
              resc = true;
            }
          }
        }
      }

      // probabilities, this thread's row sums, and P_j (fp16) into shared memory
      float pe[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) pe[q] = ex2_approx(y[q] - (m_run[q] == -INFINITY ? 0.0f : m_run[q]));
      uint32_t ph[NQ / 2];
#pragma unroll
      for (int e = 0; e < NQ / 2; ++e) ph[e] = pack_half2(pe[2 * e], pe[2 * e + 1]);
      if constexpr (F16PV) {
#pragma unroll
        for (int e = 0; e < NQ / 2; ++e) {
          const uint32_t l2 = resc ? hmul2(lsum_h[e], pack_half2(alpha[2 * e], alpha[2 * e + 1])) : lsum_h[e];
          lsum_h[e] = hadd2(l2, ph[e]);
        }
      } else {
#pragma unroll
        for (int q = 0; q < NQ; ++q) lsum[q] = (resc ? lsum[q] * alpha[q] : lsum[q]) + pe[q];
      }
      // P_(j-2) (same buffer) has been consumed by PV(j-2); a rescale of O needs PV(j-1) done
      if (ok && i >= 2) ok = warp_wait(&s.p_free[g][sb], ((i >> 1) - 1) & 1, abort_flag, 0x703);
      if (resc && i >= 1) {
        if (ok) ok = warp_wait(&s.p_free[g][sb ^ 1], ((i - 1) >> 1) & 1, abort_flag, 0x704);
        tc_fence_after();
        const uint32_t tO = tG + 2 * NQ;
        if constexpr (F16PV) {
          uint32_t w[NQ / 2];
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_ld_x8_pack16(tO + c * 16, w + c * 8);
          tmem_ld_wait();
          reg_fence<NQ / 2>(w);
#pragma unroll
          for (int e = 0; e < NQ / 2; ++e) w[e] = hmul2(w[e], pack_half2(alpha[2 * e], alpha[2 * e + 1]));
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_st_x8_unpack16(tO + c * 16, w + c * 8);
        } else {
          uint32_t w[NQ];
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_ld_x16(tO + c * 16, w + c * 16);
          tmem_ld_wait();
          reg_fence<NQ>(w);
#pragma unroll
          for (int q = 0; q < NQ; ++q) w[q] = __float_as_uint(__uint_as_float(w[q]) * alpha[q]);
#pragma unroll
          for (int c = 0; c < NQ / 16; ++c) tmem_st_x16(tO + c * 16, w + c * 16);
        }
        tmem_st_wait();
      }
      {
        // element (query q, key t) of the K-major, 128-byte swizzled P tile
        uint8_t* prow = s.pt[g][sb] + (t >> 6) * Smem::kPChunk + (t & 7) * 2;
        const int u = (t & 63) >> 3;
#pragma unroll
        for (int e = 0; e < NQ / 2; ++e) {
          const int q0 = 2 * e;
          *reinterpret_cast<__half*>(prow + q0 * 128 + ((u ^ (q0 & 7)) << 4)) =
              __ushort_as_half(static_cast<unsigned short>(ph[e] & 0xFFFFu));
          *reinterpret_cast<__half*>(prow + (q0 + 1) * 128 + ((u ^ ((q0 + 1) & 7)) << 4)) =
              __ushort_as_half(static_cast<unsigned short>(ph[e] >> 16));
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.p_full[g][sb]);
    }

    // ------------------------------------------------------------------ epilogue
    const int nmine = nblk > g ? (nblk - g + G - 1) / G : 0;   // this group's blocks
    if (ok && nmine > 0) ok = warp_wait(&s.o_full[g], 0, abort_flag, 0x705);
    tc_fence_after();
    // row sums: the 128 threads' partial sums per column (F16PV: fp16 partials added in
    // fp32, the total rounded to fp16)
    float lt[NQ];
    {
      float v[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if constexpr (F16PV) {
          const uint32_t w = lsum_h[q / 2];
          v[q] = __half2float(__ushort_as_half(static_cast<unsigned short>((q & 1) ? (w >> 16) : (w & 0xFFFFu))));
        } else {
          v[q] = lsum[q];
        }
      }
      const float sum = warp_reduce_scatter<NQ, false>(v, lane);
      if (writer) s.red[g][nmine & 1][warp & 3][q_of_lane] = sum;
      named_bar_sync(1 + g, 128);
      const float4* r4 = reinterpret_cast<const float4*>(s.red[g][nmine & 1]);
#pragma unroll
      for (int c4 = 0; c4 < NQ / 4; ++c4) {
        const float4 a = r4[c4], b = r4[NQ / 4 + c4], c = r4[2 * (NQ / 4) + c4], d = r4[3 * (NQ / 4) + c4];
        lt[4 * c4] = (a.x + b.x) + (c.x + d.x);
        lt[4 * c4 + 1] = (a.y + b.y) + (c.y + d.y);
        lt[4 * c4 + 2] = (a.z + b.z) + (c.z + d.z);
        lt[4 * c4 + 3] = (a.w + b.w) + (c.w + d.w);
      }
      if constexpr (F16PV) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) lt[q] = __half2float(__float2half_rn(lt[q]));
      }
    }
    // O^T lane t is output dim t of every query column
    // O^T in TMEM (fp32, or fp16 with F16PV) -> NQ fp32 values of output dim t
    auto load_o = [&](uint32_t tO, float* out) {
      if constexpr (F16PV) {
        uint32_t w[NQ / 2];
#pragma unroll
        for (int c = 0; c < NQ / 16; ++c) tmem_ld_x8_pack16(tO + c * 16, w + c * 8);
        tmem_ld_wait();
        reg_fence<NQ / 2>(w);
#pragma unroll
        for (int e = 0; e < NQ / 2; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          out[2 * e] = f.x;
          out[2 * e + 1] = f.y;
        }
      } else {
        uint32_t w[NQ];
#pragma unroll
        for (int c = 0; c < NQ / 16; ++c) tmem_ld_x16(tO + c * 16, w + c * 16);
        tmem_ld_wait();
        reg_fence<NQ>(w);
#pragma unroll
        for (int q = 0; q < NQ; ++q) out[q] = __uint_as_float(w[q]);
      }
    };
    float ov[NQ];
    if (ok && nmine > 0) {
      load_o(tG + 2 * NQ, ov);
    } else {
#pragma unroll
      for (int q = 0; q < NQ; ++q) ov[q] = 0.0f;
    }
    if constexpr (G == 2) {
      // group 1 hands m and l to group 0, which merges the two partial results:
      // O = a0 O0 + a1 O1, l = a0 l0 + a1 l1, a_x = 2^(m_x - M), M = max(m0, m1)
      if (g == 1) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (t == q) {
            s.exm[q] = lt[q] > 0.0f ? m_run[q] : -INFINITY;
            s.exl[q] = lt[q];
          }
        }
      }
      named_bar_sync(3, 256);
      if (g == 0) {
        const int n1 = nblk / 2;   // group 1's blocks
        float o1[NQ];
        if (ok && n1 > 0) ok = warp_wait(&s.o_full[1], 0, abort_flag, 0x706);
        tc_fence_after();
        if (ok && n1 > 0) {
          load_o(tmem + lane_base + 3 * NQ + 2 * NQ, o1);
        } else {
#pragma unroll
          for (int q = 0; q < NQ; ++q) o1[q] = 0.0f;
        }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          const float m0 = lt[q] > 0.0f ? m_run[q] : -INFINITY;
          const float m1 = s.exm[q], l1 = s.exl[q];
          const float M = fmaxf(m0, m1);
          if (M != -INFINITY) {
            const float a0 = m0 == -INFINITY ? 0.0f : ex2_approx(m0 - M);
            const float a1 = m1 == -INFINITY ? 0.0f : ex2_approx(m1 - M);
            ov[q] = a0 * ov[q] + a1 * o1[q];
            lt[q] = a0 * lt[q] + a1 * l1;
            m_run[q] = M;
          }
        }
      }
    }
    if (g == 0) {
    const size_t rows_total = static_cast<size_t>(gridDim.x) * p.rows;
    const size_t row0 = static_cast<size_t>(plane) * p.rows;
    if (p.cluster) {
      // this split's unnormalised O (column q, dim t), m and l, for the cluster merge below;
      // every load and MMA that used the first K' slot is done
      float* po = reinterpret_cast<float*>(s.k[0]);
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        po[q * D + t] = ov[q];
        if (t == q) {
          s.cm[q] = lt[q] > 0.0f ? m_run[q] : -INFINITY;
          s.cl[q] = lt[q];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      if (q < p.rows && !p.cluster) {
        const float inv_l = lt[q] > 0.0f ? 1.0f / lt[q] : 0.0f;
        const float val = ov[q] * inv_l;
        const float l2 = lt[q] > 0.0f ? m_run[q] + log2f(lt[q]) : -INFINITY;
        if (p.part_o != nullptr) {
          const size_t idx = static_cast<size_t>(split) * rows_total + row0 + q;
          p.part_o[idx * D + t] = val;
          if (t == q) p.part_lse[idx] = l2;
        } else {
          p.o[(row0 + q) * D + t] = __float2half_rn(val);
          if (t == q && p.lse != nullptr) p.lse[row0 + q] = l2 * 0.69314718055994531f;
        }
      }
    }
    }  // group 0
  }

  if (p.cluster) {
    // merge of the cluster's splits: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,
    // M = max_s m_s; LSE = ln 2 * (M + log2 of the denominator)
    cluster_sync_all();
    if (warp < 4) {
      const int t = tid;
      const int ns = static_cast<int>(gridDim.y);
      const uint32_t po = smem_u32(s.k[0]), pm = smem_u32(s.cm), pl = smem_u32(s.cl);
      const size_t row0 = static_cast<size_t>(plane) * p.rows;
      for (int q = static_cast<int>(cluster_ctarank()); q < p.rows; q += ns) {
        float ms[8], ls[8];
        float M = -INFINITY;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          ms[r] = -INFINITY;
          ls[r] = 0.0f;
          if (r < ns) {
            ms[r] = ld_shared_cluster_f32(mapa_shared(pm + q * 4, r));
            ls[r] = ld_shared_cluster_f32(mapa_shared(pl + q * 4, r));
            if (ls[r] > 0.0f) M = fmaxf(M, ms[r]);
          }
        }
        float num = 0.0f, den = 0.0f;
        if (M != -INFINITY) {
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            if (r < ns && ls[r] > 0.0f) {
              const float wgt = ex2_approx(ms[r] - M);
              den = fmaf(wgt, ls[r], den);
              num = fmaf(wgt, ld_shared_cluster_f32(mapa_shared(po + (q * D + t) * 4, r)), num);
            }
          }
        }
        p.o[(row0 + q) * D + t] = __float2half_rn(den > 0.0f ? num / den : 0.0f);
        if (t == 0 && p.lse != nullptr)
          p.lse[row0 + q] = den > 0.0f ? (M + log2f(den)) * 0.69314718055994531f : -INFINITY;
      }
    }
    cluster_sync_all();   // no CTA leaves while another still reads its shared memory
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace pasa
