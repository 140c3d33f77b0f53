// PASA attention forward on sm_103a: TMA -> shared memory -> tcgen05.mma -> TMEM, with the
// online softmax, the global-recovering offsets and the final rescale in the softmax warps.
//
// Method: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
// Inference" (arXiv 2503.01873), Abstract: FlashAttention in half precision where every key
// block K_j is shifted by its pseudo-average m_j before the fp16 score GEMM and the per-row
// offsets q_i . m_j are carried in fp32 and folded back into the online max and sum
// ("global recovering"). The shifted keys and the block means come from kshift_kernel.
//
// One CTA owns one 128-row query tile of one (batch, query head) and walks the key blocks
// (BN = 128 keys each) of its kv head. Warp roles (224 threads):
//   warps 0-3  softmax + epilogue          (thread r <-> query row r <-> TMEM lane r)
//   warp  4    TMA producer: Q once, then K'_j (one block ahead of V) / V_j rings and
//              16-block chunks of means
//   warp  5    TMEM owner; one thread issues the score MMAs QK(j) (and the offsets)
//   warp  6    one thread issues the PV MMAs
// The two MMA streams touch disjoint TMEM (S, C versus P, O), so they need no ordering
// between them; each thread's barrier waits overlap the other's MMAs on the tensor pipe.
//
// TMEM (512 columns) holds two score buffers S_0, S_1 (BN columns each), the output
// accumulator O (D columns), the probabilities P (BN/2 columns, two fp16 per column) and two
// buffers of offsets C (16 columns each: q_i . m_j for 16 consecutive key blocks) and, in the
// columns left, the Q tile (at D = 128 the 32 columns left hold its first 64 channels), all
// disjoint. The score and offsets
// MMAs take those K-steps with A in TMEM (a tcgen05 MMA with M = 128, N <= 128 runs at ~67
// cycles with A in TMEM against ~86 with both operands in shared memory) and the rest with
// both operands in shared memory. Key block j uses S_(j mod 2), so the score MMA of block j+1 is issued while the
// softmax still works on block j-1 and S_(j+1) is ready before the softmax reaches it: once
// running, the softmax never waits for scores and the tensor pipe always has the next
// block's work queued. The softmax releases an S buffer (s_free) as soon as it has loaded
// it, and waits for the previous block's PV MMA (p_free) only right before it rescales O or
// rewrites P.
//
// Score modes: the QK^T accumulator is fp16 (F16ACC, the PASA regime) or fp32. SHIFT
// selects shifted keys + offsets (PASA) or raw keys (no shift: the naive fp16 kernel or the
// plain fp32-accumulate FlashAttention). P is rounded to fp16 and PV accumulates in fp32,
// except with F16PV (half precision throughout the FlashAttention loop, Abstract): the PV
// accumulator O is fp16 in TMEM (tcgen05 F16 D format, rescaled in f16x2 arithmetic) and
// the running row sum is fp16 (each block's probabilities summed in f16x2, then added in
// fp16). The running max, the offsets and the final division stay fp32.
//
// STATS (diagnostic build): per query row, the largest |score| the score accumulator held
// (S' with the shift, S without; fp16 values in the fp16-accumulate modes, inf if one
// overflowed) and the largest |S' + c| (the recovered raw score; equal to the first without
// the shift). A block's min and max of S' give both, since c is constant per row and block.
// The same two magnitudes are also reduced over the query rows of each key block (a warp
// max, then one atomicMax per warp on the fp32 bits, which order like the values since
// both are >= 0) into per-(head, block) maxima.
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

constexpr int kTileRows = 128;       // query rows per CTA (MMA M)
constexpr int kChunkBlocks = 16;     // key blocks per offsets MMA (its N)
constexpr int kAttnThreads = 224;
constexpr int kAttnThreadsFused = 352;   // + four shift warps (7-10) in the FUSED kernels
constexpr int kShiftBar = 3;             // named barrier of the shift warps
constexpr float kRescaleLog2 = 8.0f;

// The softmax's exponentials of a block: pair c (two scores) runs on the FMA pipe
// (exp2_fma2) when bit (c mod 16) of kPolyMask is set and on MUFU (ex2.approx) otherwise.
// On GB300 MUFU retires ex2.approx.f32 at 8 lanes a clock per SM sub-partition (4 cycles per
// warp instruction, 32 per clock per SM), so a block's 128 exponentials per row take 512
// cycles of MUFU time against ~1100 cycles of MMA: MUFU is not what bounds the softmax,
// while the FMA-pipe form costs 7 FMA-pipe lane operations per value (1.75x MUFU's pipe
// time) and lengthens the softmax's chain. Measured on the 32K causal and the D = 64
// resonance workloads, 1, 2 and 5 pairs of 16 on the FMA pipe all ran slower than none
// (e.g. 5 of 16: 1225 vs 1365 and 690 vs 775 TFLOP/s), so the mask is empty.
constexpr uint32_t kPolyMask = 0x0000u;

__device__ __forceinline__ void exp2_split(float& p0, float& p1, float x0, float x1, int c) {
  if ((kPolyMask >> (c & 15)) & 1u) {
    exp2_fma2(p0, p1, x0, x1);
  } else {
    p0 = ex2_approx(x0);
    p1 = ex2_approx(x1);
  }
}

struct AttnParams {
  float* lse;            // [B, Hq, Sq] fp32 or nullptr
  int B, Hq, Hkv, Sq, Sk;
  int n_qblk;            // ceil(Sq / kTileRows)
  float scale_log2;      // softmax scale * log2(e)
  float inv_scale_log2;  // 1 / scale_log2
  float* stats;          // STATS kernels: [B, Hq, Sq, 2] fp32 score magnitudes per row
  unsigned* bstats;      // STATS kernels, or nullptr: [B, Hq, nbt, 2] per key block, fp32 bits
  int nbt;               // key blocks per head, ceil(Sk / BN)
  const float* kscale;   // FP8 kernels: [B, Hkv, nbt] fp32 e4m3 scale of each key block
  // Decode layout. sq_mod: query rows per head for the causal mask; equal to Sq, except
  // when the g = Hq/Hkv heads of a kv group are packed into one row range ("Hq" = Hkv,
  // "Sq" = g * sq_mod rows, row r holding query r mod sq_mod of head r / sq_mod).
  int sq_mod;
  // Split keys: blockIdx.y selects key blocks [y * bps, (y + 1) * bps) (0 = no split).
  // Then each CTA writes O / l in fp32 to part_o [split][row][D] and
  // m + log2 l to part_lse [split][row] instead of o and lse; a combine kernel merges them.
  int bps;
  float* part_o;
  float* part_lse;
  // FUSED kernels, optional (nullptr: not written): the shifted keys [B, Hkv, Sk, D] and the
  // block means [B, Hkv, nbt, D] the kernel computed, for checking them against the pre-pass
  __half* kshift_out;
  __half* means_out;
};

// TMEM column map (see the header comment).
template <int D, int BN>
struct TmemMap {
  __host__ __device__ static constexpr int s(int b) { return b * BN; }
  static constexpr int o = 2 * BN;
  static constexpr int p = 2 * BN + D;
  __host__ __device__ static constexpr int c(int b) { return 2 * BN + D + BN / 2 + b * kChunkBlocks; }
  // The first kQtSteps K-steps of the Q tile as the A operand (8 columns per K-step of 16):
  // as many as the 512 columns leave room for.
  static constexpr int q = 2 * BN + D + BN / 2 + 2 * kChunkBlocks;
  static constexpr int kQtSteps = (512 - q) / 8 < D / 16 ? (512 - q) / 8 : D / 16;
  static constexpr int total = q + 8 * kQtSteps;
  static_assert(total <= 512, "TMEM budget");
  static_assert(BN % 32 == 0 && BN <= 256, "key block");
  static_assert(D == 64 || D == 128, "head dim");
};

template <int D, int BN, int KST, int VST, bool FP8 = false, bool FUSED = false>
struct AttnSmem {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms along D (fp16)
  static constexpr int kKB = FP8 ? 1 : 2;                // bytes per key element
  static constexpr int kKChunks = D * kKB / 128;         // 128-byte swizzle atoms of a key row
  static constexpr int kQTile = kTileRows * D * 2;
  static constexpr int kKTile = BN * D * kKB;
  static constexpr int kVTile = BN * D * 2;              // V stays fp16 in every mode
  static constexpr int kMTile = kChunkBlocks * D * 2;
  static constexpr int kQChunk = kTileRows * 128;
  static constexpr int kKChunk = BN * 128;                 // bytes of one 128-byte-wide atom column
  static constexpr int kVChunk = BN * 128;
  static constexpr int kMChunk = kChunkBlocks * 128;
  alignas(1024) uint8_t q[kQTile];   // also the O staging buffer
  alignas(1024) uint8_t q8[FP8 ? kTileRows * D : 16];  // FP8: e4m3 codes of Q (one 128-byte atom per row)
  alignas(1024) uint8_t k[KST][kKTile];
  alignas(1024) uint8_t v[VST][kVTile];
  alignas(1024) uint8_t m[FUSED ? 1 : 2][FUSED ? 16 : kMTile];
  // FUSED: offsets ring (one c per query row and K slot), the block's means in fp32, and the
  // shift warps' exchange of per-channel maxima and integer sums (4 warps x 16 units)
  float cs[FUSED ? KST : 1][FUSED ? kTileRows : 1];
  float mf[FUSED ? D : 1];
  uint32_t red_max[FUSED ? 4 : 1][FUSED ? D / 8 : 1][4];
  uint32_t red_sum[FUSED ? 4 : 1][FUSED ? D / 8 : 1][8];
  uint64_t sh_full[FUSED ? KST : 1];   // K'_j shifted in place and c_j written (4 shift warps)
  uint64_t c_free[FUSED ? KST : 1];    // the softmax has read c_j (4 warps)
  uint64_t q_full;
  uint64_t q8_full;     // FP8: the softmax warps have written the e4m3 Q tile (4 warps)
  uint64_t k_full[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t m_full[2], m_empty[2];
  uint64_t s_full[2];   // QK(j) done: S_(j mod 2) (and C) hold block j
  uint64_t s_free[2];   // the softmax has loaded S_(j mod 2) and C of block j (4 warps)
  uint64_t p_full;      // the softmax has written P of block j (4 warps)
  uint64_t p_free;      // PV(j) done: P may be rewritten, O is stable
  uint64_t o_full;
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ANDs a predicate over the nthreads participants: every thread
// leaves with the same answer, so a group can decide together to stop.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Two fp16 values minus two fp16 values, each difference rounded once to fp16 (round to
// nearest even, subnormals kept).
__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float half_lo_to_float(uint32_t w) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
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

template <int D, int BN, bool F16ACC, bool SHIFT, bool CAUSAL, int KST, int VST, bool STATS = false,
          bool F16PV = false, bool FP8 = false, bool FUSED = false>
__global__ void __launch_bounds__(FUSED ? kAttnThreadsFused : kAttnThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
                const __grid_constant__ CUtensorMap mapM, const AttnParams p) {
  static_assert(!F16PV || F16ACC, "fp16 PV accumulation is a variant of the fp16-score mode");
  static_assert(!FP8 || (D == 128 && !F16ACC && !STATS && !F16PV), "FP8 scores: D = 128, fp32 accumulation");
  static_assert(!FUSED || (D == 128 && SHIFT && !FP8 && !STATS), "the fused shift: D = 128, shifted fp16 keys");
  using Smem = AttnSmem<D, BN, KST, VST, FP8, FUSED>;
  static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory per CTA");
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

  // Key blocks of this CTA: [jb0, jb0 + nblk). The loops below count j from 0 (offsets
  // chunks and ring slots are local to the CTA); data addresses (key rows, block means,
  // block scales, the causal mask) use the global block jb0 + j.
  const int split = blockIdx.y;
  const int jb0 = split * p.bps;
  int nblk;
  {
    const int last = min(p.Sq, q0 + kTileRows) - 1;
    const int i_last = p.sq_mod == p.Sq ? last : min(p.sq_mod - 1, last);   // packed rows: an upper bound
    const int kv_end = CAUSAL ? min(p.Sk, i_last + p.Sk - p.sq_mod + 1) : p.Sk;
    nblk = kv_end > 0 ? (kv_end + BN - 1) / BN : 0;
    if (p.bps > 0) nblk = max(0, min(p.bps, nblk - jb0));
  }

  if (tid == 0) {
    mbar_init(&s.q_full, 1);
    mbar_init(&s.q8_full, 4);
    for (int i = 0; i < KST; ++i) { mbar_init(&s.k_full[i], 1); mbar_init(&s.k_empty[i], 1); }
    for (int i = 0; i < VST; ++i) { mbar_init(&s.v_full[i], 1); mbar_init(&s.v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.m_full[i], 1);
      mbar_init(&s.m_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 4);
    }
    mbar_init(&s.p_full, 4);
    mbar_init(&s.p_free, 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.drain[0], 1);
    mbar_init(&s.drain[1], 1);
    if constexpr (FUSED) {
      for (int i = 0; i < KST; ++i) {
        mbar_init(&s.sh_full[i], 4);
        mbar_init(&s.c_free[i], 4);
      }
    }
    s.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp == 4) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      if (SHIFT && !FUSED) tma_prefetch_desc(&mapM);
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
        if (SHIFT && !FUSED && (j % kChunkBlocks) == 0) {
          const int ci = j / kChunkBlocks, slot = ci & 1;
          if (!mbar_wait(&s.m_empty[slot], ((ci >> 1) & 1) ^ 1, abort_flag, 0x101)) return false;
          mbar_arrive_expect_tx(&s.m_full[slot], Smem::kMTile);
#pragma unroll
          for (int c = 0; c < Smem::kChunks; ++c)
            tma_load_3d(s.m[slot] + c * Smem::kMChunk, &mapM, &s.m_full[slot], c * 64, jb0 + j, kz);
          m_issued = ci + 1;
        }
        const int ks = j % KST;
        if (!mbar_wait(&s.k_empty[ks], ((j / KST) & 1) ^ 1, abort_flag, 0x102)) return false;
        mbar_arrive_expect_tx(&s.k_full[ks], Smem::kKTile);
#pragma unroll
        for (int c = 0; c < Smem::kKChunks; ++c)
          tma_load_3d(s.k[ks] + c * Smem::kKChunk, &mapK, &s.k_full[ks], c * (128 / Smem::kKB), (jb0 + j) * BN, kz);
        k_issued = j + 1;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int vs = j % VST;
        if (!mbar_wait(&s.v_empty[vs], ((j / VST) & 1) ^ 1, abort_flag, 0x103)) return false;
        mbar_arrive_expect_tx(&s.v_full[vs], Smem::kVTile);
#pragma unroll
        for (int c = 0; c < Smem::kChunks; ++c)
          tma_load_3d(s.v[vs] + c * Smem::kVChunk, &mapV, &s.v_full[vs], c * 64, (jb0 + j) * BN, kz);
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
  } else if (warp == 5) {
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
      // FP8: e4m3 Q (written by the softmax warps), K = 32 per MMA, 32 bytes along the row
      constexpr uint32_t id_s8 = idesc_e4m3(kTileRows, BN);
      const uint32_t q8_lo = sdesc_lo(smem_u32(s.q8), 16);
      bool ok = mbar_wait(FP8 ? &s.q8_full : &s.q_full, 0, abort_flag, 0x201);
      const uint32_t tQ = tmem + TM::q;
      constexpr int kQt = FP8 ? 0 : TM::kQtSteps;   // FP8 keeps the fp16 Q (offsets) in shared memory
      if (kQt > 0 && ok && nblk > 0) {
        // Q's first K-steps into TMEM once. Only with key blocks: without them the epilogue
        // rewrites the Q buffer as soon as Q has landed, and no MMA completion would cover
        // this copy.
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kQt; ++kk) tmem_cp_128x256b(tQ + kk * 8, qd[kk], hi_kmaj);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        const int ks = j % KST;
        const int ci = j / kChunkBlocks;
        const int sb = j & 1;
        const bool chunk_start = SHIFT && !FUSED && (j % kChunkBlocks) == 0;
        uint32_t kd[D / 16];
        const uint32_t k_lo = k_lo0 + ks * kKStride;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) kd[kk] = k_lo + (((kk / 4) * Smem::kKChunk + (kk % 4) * 32) >> 4);
        // (FP8: the first D / 32 of these are the e4m3 K-steps of the single 128-byte atom)
        // FUSED: the shift warps have shifted the raw tile in place (K'_j), else TMA brought K'_j
        if (!mbar_wait(FUSED ? &s.sh_full[ks] : &s.k_full[ks], (j / KST) & 1, abort_flag, 0x202)) break;
        if (chunk_start && !mbar_wait(&s.m_full[ci & 1], (ci >> 1) & 1, abort_flag, 0x203)) break;
        if (j >= 2 && !mbar_wait(&s.s_free[sb], ((j >> 1) - 1) & 1, abort_flag, 0x206)) break;
        tc_fence_after();
        if (chunk_start) {
          const uint32_t m_lo = m_lo0 + (ci & 1) * kMStride;
          const uint32_t tC = tmem + TM::c(ci & 1);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off_m = ((kk / 4) * Smem::kMChunk + (kk % 4) * 32) >> 4;
            if (kk < kQt) mma_ts_w(tC, tQ + kk * 8, m_lo + off_m, hi_kmaj, id_c, kk > 0 ? 1u : 0u);
            else mma_ss_w(tC, qd[kk], hi_kmaj, m_lo + off_m, hi_kmaj, id_c, kk > 0 ? 1u : 0u);
          }
        }
        const uint32_t tS = tmem + TM::s(sb);
        if constexpr (FP8) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_w(tS, q8_lo + ((kk * 32) >> 4), hi_kmaj, kd[kk], hi_kmaj, id_s8, kk > 0 ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            if (kk < kQt) mma_ts_w(tS, tQ + kk * 8, kd[kk], hi_kmaj, id_s, kk > 0 ? 1u : 0u);
            else mma_ss_w(tS, qd[kk], hi_kmaj, kd[kk], hi_kmaj, id_s, kk > 0 ? 1u : 0u);
          }
        }
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
  } else if (warp == 6) {
    // ------------------------------------------------------------------ PV issuer
    // PV(j) once the softmax has written P of block j and V_j has landed.
    if (lane == 0) {
      constexpr uint32_t id_o = idesc_f16(kTileRows, D, !F16PV, true);
      constexpr uint32_t hi_v = sdesc_hi_sw128(1024);
      const uint32_t v_lo0 = sdesc_lo(smem_u32(s.v[0]), Smem::kVChunk);
      constexpr uint32_t kVStride = sizeof(s.v[0]) >> 4;
      const uint32_t tO = tmem + TM::o;
      const uint32_t tP = tmem + TM::p;
      for (int j = 0; j < nblk; ++j) {
        const int vs = j % VST;
        uint32_t vd[BN / 16];
        const uint32_t v_lo = v_lo0 + vs * kVStride;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) vd[kk] = v_lo + kk * (2048 >> 4);
        if (!mbar_wait(&s.v_full[vs], (j / VST) & 1, abort_flag, 0x204)) break;
        if (!mbar_wait(&s.p_full, j & 1, abort_flag, 0x205)) break;
        tc_fence_after();
        const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) mma_ts_w(tO, tP + kk * 8, vd[kk], hi_v, id_o, kk > 0 ? 1u : acc0);
        mma_commit(&s.p_free);
        mma_commit(&s.v_empty[vs]);
        if (j == nblk - 1) mma_commit(&s.o_full);
      }
      mma_commit(&s.drain[1]);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(&s.drain[1], 0) && globaltimer_ns() - t0 < kWaitTimeoutNs) {
      }
    }
    __syncwarp();
  } else if (FUSED && warp >= 7) {
    // ------------------------------------------------------------------ shift warps (FUSED)
    // The pseudo-average shift of each raw K tile, in place in shared memory as it lands,
    // then the tile's offsets for the 128 query rows. The same reading of the pseudo-average
    // as kshift_kernel (exact integer sums on the grid of the block maximum, one rounding of
    // K - m), so K' and m are the pre-pass's bit for bit. Thread st owns channels
    // 8u .. 8u + 7 (one 16-byte unit) of the tile rows rg, rg + 8, ..., rg + 120; in the
    // 128-byte swizzle those rows hold the unit at the same position (row mod 8 = rg).
    if constexpr (FUSED) {
      const int st = tid - 7 * 32;      // 0..127
      const int sw = st >> 5;           // shift warp 0..3
      const int u = st & 15;
      const int rg = st >> 4;           // 0..7
      static_assert(D / 8 == 16, "16 units per key row");
      const uint32_t uoff = (u >> 3) * Smem::kKChunk + ((((u & 7) ^ rg)) << 4);
      constexpr float kRound = 12582912.0f;      // 1.5 * 2^23
      constexpr uint32_t kRoundBits = 0x4B400000u;
      const int kz = b * p.Hkv + hk;
      bool ok = named_bar_and(kShiftBar, 128, mbar_wait(&s.q_full, 0, abort_flag, 0x360));
      for (int j = 0; ok && j < nblk; ++j) {
        const int ks = j % KST;
        // every decision to stop is taken by all 128 threads together (no one is left at a
        // named barrier)
        if (!named_bar_and(kShiftBar, 128, mbar_wait(&s.k_full[ks], (j / KST) & 1, abort_flag, 0x361))) {
          ok = false;
          break;
        }
        uint8_t* tile = s.k[ks];
        uint4 x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = *reinterpret_cast<const uint4*>(tile + (rg + 8 * i) * 128 + uoff);
        // 1. per-channel max |K| (16-bit lanes); an inf or NaN makes it >= 0x7C00
        uint32_t mx[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          mx[0] = __vmaxu2(mx[0], x[i].x & 0x7FFF7FFFu);
          mx[1] = __vmaxu2(mx[1], x[i].y & 0x7FFF7FFFu);
          mx[2] = __vmaxu2(mx[2], x[i].z & 0x7FFF7FFFu);
          mx[3] = __vmaxu2(mx[3], x[i].w & 0x7FFF7FFFu);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) mx[c] = __vmaxu2(mx[c], __shfl_xor_sync(0xffffffffu, mx[c], 16));
        if (lane < 16) {
#pragma unroll
          for (int c = 0; c < 4; ++c) s.red_max[sw][u][c] = mx[c];
        }
        named_bar_sync(kShiftBar, 128);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          mx[c] = __vmaxu2(__vmaxu2(s.red_max[0][u][c], s.red_max[1][u][c]),
                           __vmaxu2(s.red_max[2][u][c], s.red_max[3][u][c]));
        // 2. grid step g = fp16 spacing at the maximum; guard: m = 0 from 2^15 up (and inf/NaN)
        float g[8], inv_g[8];
        bool guard[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const uint32_t a = (mx[h >> 1] >> (16 * (h & 1))) & 0xFFFFu;
          const int E = static_cast<int>(a >> 10);
          const int e = E >= 1 ? E - 25 : -24;
          g[h] = __int_as_float((e + 127) << 23);
          inv_g[h] = __int_as_float((127 - e) << 23);
          guard[h] = E >= 30;
        }
        // 3. sums of rint_even(K / g): K / g is exact and below 2^11 where not guarded, so
        //    fp32(K / g + 1.5 * 2^23) holds the rounded integer in its low bits
        uint32_t sm[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __half2* hv = reinterpret_cast<const __half2*>(&x[i]);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float2 f = __half22float2(hv[c]);
            sm[2 * c] += __float_as_uint(__fmaf_rn(f.x, inv_g[2 * c], kRound)) - kRoundBits;
            sm[2 * c + 1] += __float_as_uint(__fmaf_rn(f.y, inv_g[2 * c + 1], kRound)) - kRoundBits;
          }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) sm[h] += __shfl_xor_sync(0xffffffffu, sm[h], 16);
        if (lane < 16) {
#pragma unroll
          for (int h = 0; h < 8; ++h) s.red_sum[sw][u][h] = sm[h];
        }
        named_bar_sync(kShiftBar, 128);
        // 4. m = g * rint_even(sum / n) over the n valid rows of the block (0 where guarded)
        const int n = min(BN, p.Sk - (jb0 + j) * BN);
        float mv[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const int su = static_cast<int>(s.red_sum[0][u][h] + s.red_sum[1][u][h] + s.red_sum[2][u][h] +
                                          s.red_sum[3][u][h]);
          int mu;
          if (n == BN) {
            // rint_even(su / 128): floor plus the half-even decision on the remainder
            const int fl = su >> 7, rm = su & 127;
            mu = fl + ((rm > 64 || (rm == 64 && (fl & 1))) ? 1 : 0);
          } else {
            mu = rne_div(su, n);
          }
          mv[h] = guard[h] ? 0.0f : static_cast<float>(mu) * g[h];  // exact
        }
        uint32_t m2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) m2[c] = pack_half2(mv[2 * c], mv[2 * c + 1]);   // exact
        // 5. K' = fp16_rn(K - m) in place
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          x[i] = make_uint4(hsub2_rn(x[i].x, m2[0]), hsub2_rn(x[i].y, m2[1]), hsub2_rn(x[i].z, m2[2]),
                            hsub2_rn(x[i].w, m2[3]));
          *reinterpret_cast<uint4*>(tile + (rg + 8 * i) * 128 + uoff) = x[i];
        }
        if (rg == 0) {
#pragma unroll
          for (int h = 0; h < 8; ++h) s.mf[8 * u + h] = mv[h];
        }
        if (p.kshift_out != nullptr) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int row = rg + 8 * i;
            if (row < n)
              *reinterpret_cast<uint4*>(p.kshift_out + (static_cast<size_t>(kz) * p.Sk + (jb0 + j) * BN + row) * D +
                                        8 * u) = x[i];
          }
        }
        if (p.means_out != nullptr && rg == 0)
          *reinterpret_cast<uint4*>(p.means_out + (static_cast<size_t>(kz) * p.nbt + jb0 + j) * D + 8 * u) =
              make_uint4(m2[0], m2[1], m2[2], m2[3]);
        fence_proxy_async_smem();   // the MMA reads K' through the async proxy
        // 6. the offsets c = q_st . m_j of query row st (fp32; the products are exact), once
        //    the softmax has read the last offsets of this ring slot; the barrier also makes
        //    every thread's means visible
        const bool cf = j < KST || mbar_wait(&s.c_free[ks], ((j / KST) & 1) ^ 1, abort_flag, 0x362);
        if (!named_bar_and(kShiftBar, 128, cf)) {
          ok = false;
          break;
        }
        float ca[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // four independent pair chains
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const uint4 qv = *reinterpret_cast<const uint4*>(s.q + (v >> 3) * Smem::kQChunk + st * 128 +
                                                           ((((v & 7) ^ (st & 7))) << 4));
          const float4 ma = *reinterpret_cast<const float4*>(s.mf + 8 * v);
          const float4 mb = *reinterpret_cast<const float4*>(s.mf + 8 * v + 4);
          const __half2* qh = reinterpret_cast<const __half2*>(&qv);
          const float2 q0f = __half22float2(qh[0]), q1f = __half22float2(qh[1]);
          const float2 q2f = __half22float2(qh[2]), q3f = __half22float2(qh[3]);
          ffma2(ca[0], ca[1], q0f.x, q0f.y, ma.x, ma.y, ca[0], ca[1]);
          ffma2(ca[2], ca[3], q1f.x, q1f.y, ma.z, ma.w, ca[2], ca[3]);
          ffma2(ca[4], ca[5], q2f.x, q2f.y, mb.x, mb.y, ca[4], ca[5]);
          ffma2(ca[6], ca[7], q3f.x, q3f.y, mb.z, mb.w, ca[6], ca[7]);
        }
        s.cs[ks][st] = ((ca[0] + ca[1]) + (ca[2] + ca[3])) + ((ca[4] + ca[5]) + (ca[6] + ca[7]));
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.sh_full[ks]);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int r = tid;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + TM::o;
    const uint32_t tP = tmem + lane_base + TM::p;
    const int i = q0 + r;
    const int i_mask = i % p.sq_mod;   // the query's position within its head
    const int limit = (i < p.Sq) ? (CAUSAL ? min(p.Sk, max(0, i_mask + p.Sk - p.sq_mod + 1)) : p.Sk) : 0;
    const float sl2 = p.scale_log2;
    constexpr int kPairs = BN / 2;
    float m_run = -INFINITY, l_run = 0.0f;
    float st_acc = 0.0f, st_rec = 0.0f;  // STATS: max |accumulated score|, max |S' + c|
    bool ok = true;

    // FP8: quantise this thread's Q row to e4m3 with the row scale sq = a / 448 (a = max |q|,
    // inv = 448 / a, code = e4m3_rn_satfinite(q * inv), all fp32 with one rounding each) into
    // the e4m3 Q tile, whose rows are single 128-byte swizzle atoms. Score dequantisation:
    // S = sq * sk_j * (Q8 . K8_j), folded into the softmax's scale per block.
    float sq = 1.0f;
    const float* kscale_row = FP8 ? p.kscale + static_cast<size_t>(b * p.Hkv + hk) * p.nbt : nullptr;
    float sk_next = 1.0f;
    if constexpr (FP8) {
      griddep_wait();   // the block scales come from the key preparation queued just ahead
      if (nblk > 0) sk_next = __ldg(kscale_row + jb0);
      if (!mbar_wait(&s.q_full, 0, abort_flag, 0x340)) ok = false;
      uint4 qrow[D / 8];
#pragma unroll
      for (int u = 0; u < D / 8; ++u)
        qrow[u] = *reinterpret_cast<const uint4*>(s.q + (u / 8) * Smem::kQChunk + r * 128 + (((u % 8) ^ (r & 7)) * 16));
      uint32_t amax = 0;
#pragma unroll
      for (int u = 0; u < D / 8; ++u) {
        const uint32_t w4[4] = {qrow[u].x, qrow[u].y, qrow[u].z, qrow[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) amax = __vmaxu2(amax, w4[e] & 0x7FFF7FFFu);  // per fp16 lane
      }
      amax = max(amax & 0xFFFFu, amax >> 16);
      const float a = __half2float(__ushort_as_half(static_cast<unsigned short>(amax)));
      const float inv = a > 0.0f ? __fdiv_rn(448.0f, a) : 1.0f;
      sq = a > 0.0f ? __fdiv_rn(a, 448.0f) : 1.0f;
#pragma unroll
      for (int u = 0; u < D / 16; ++u) {   // 16 codes (16 bytes) per iteration
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half* h = reinterpret_cast<const __half*>(&qrow[2 * u + e / 2]) + (e % 2) * 4;
          const uint16_t c01 = pack_e4m3x2(__fmul_rn(__half2float(h[0]), inv), __fmul_rn(__half2float(h[1]), inv));
          const uint16_t c23 = pack_e4m3x2(__fmul_rn(__half2float(h[2]), inv), __fmul_rn(__half2float(h[3]), inv));
          w[e] = c01 | (static_cast<uint32_t>(c23) << 16);
        }
        *reinterpret_cast<uint4*>(s.q8 + r * 128 + ((u ^ (r & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.q8_full);
    }

    for (int j = 0; ok && j < nblk; ++j) {
      const int sb = j & 1;
      float fsc = 1.0f;   // FP8: dequantisation factor sq * sk_j of this block's scores
      if constexpr (FP8) {
        fsc = sq * sk_next;
        if (j + 1 < nblk) sk_next = __ldg(kscale_row + jb0 + j + 1);
      }
      if (!mbar_wait(&s.s_full[sb], (j >> 1) & 1, abort_flag, 0x300)) { ok = false; break; }
      // FUSED: the offset of block j comes from the shift warps through shared memory; their
      // arrival on sh_full (complete before QK(j) could start) orders the write
      if (FUSED && !mbar_wait(&s.sh_full[j % KST], (j / KST) & 1, abort_flag, 0x301)) { ok = false; break; }
      tc_fence_after();
      // Load the block's scores and offset, wait once, fence the registers, and release the
      // score buffer to the MMA thread before any arithmetic. fp16 scores (F16ACC) are
      // loaded two per register; their row max is taken in f16x2 and each score enters fp32
      // through one mixed-precision add. fp32 scores are used as loaded.
      const uint32_t tS = tmem + lane_base + TM::s(sb);
      uint32_t hp[F16ACC ? kPairs : 1];
      float sv[F16ACC ? 1 : BN];
      uint32_t cw = 0;
      if constexpr (F16ACC) {
        tmem_ld_scores_f16<BN>(tS, hp);
      } else {
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) tmem_ld_x16(tS + c * 16, reinterpret_cast<uint32_t*>(sv) + c * 16);
      }
      if (SHIFT && !FUSED) tmem_ld_x1(tmem + lane_base + TM::c((j / kChunkBlocks) & 1) + (j % kChunkBlocks), cw);
      if constexpr (FUSED) cw = __float_as_uint(s.cs[j % KST][r]);
      tmem_ld_wait();
      if constexpr (F16ACC) reg_fence<kPairs>(hp);
      else reg_fence<BN>(reinterpret_cast<uint32_t*>(sv));
      reg_fence<1>(&cw);
      tc_fence_before();
      __syncwarp();
      mbar_arrive_if(&s.s_free[sb], lane == 0);
      if constexpr (FUSED) mbar_arrive_if(&s.c_free[j % KST], lane == 0);

      const int cmax = limit - (jb0 + j) * BN;
      const float c_raw = SHIFT ? __uint_as_float(cw) : 0.0f;
      float mx, mn = 0.0f;
      if constexpr (F16ACC) {
        if constexpr (STATS) {
          // block min in eight f16x2 accumulators (+inf where masked)
          auto masked = [&](int c) {
            return ((2 * c < cmax) ? (hp[c] & 0xFFFFu) : 0x7C00u) |
                   ((2 * c + 1 < cmax) ? (hp[c] & 0xFFFF0000u) : 0x7C000000u);
          };
          uint32_t tmp[8];
          if (cmax >= BN) {   // no key of the block is masked for this row
#pragma unroll
            for (int k = 0; k < 8; ++k) tmp[k] = hp[k];
#pragma unroll
            for (int c = 8; c < kPairs; ++c) tmp[c & 7] = hmin2(tmp[c & 7], hp[c]);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) tmp[k] = masked(k);
#pragma unroll
            for (int c = 8; c < kPairs; ++c) tmp[c & 7] = hmin2(tmp[c & 7], masked(c));
          }
          const uint32_t n1 = tree_h2<8, false>(tmp);
          mn = fminf(half_lo_to_float(n1), half_lo_to_float(n1 >> 16));
        }
        if (cmax < BN) {
#pragma unroll
          for (int c = 0; c < kPairs; ++c)
            hp[c] = ((2 * c < cmax) ? (hp[c] & 0xFFFFu) : 0xFC00u) |
                    ((2 * c + 1 < cmax) ? (hp[c] & 0xFFFF0000u) : 0xFC000000u);  // -inf when masked
        }
        uint32_t tmp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) tmp[k] = hp[k];
#pragma unroll
        for (int c = 8; c < kPairs; ++c) tmp[c & 7] = hmax2(tmp[c & 7], hp[c]);
        const uint32_t m1 = tree_h2<8, true>(tmp);
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
        const float a_acc = cmax > 0 ? fmaxf(fabsf(mx), fabsf(mn)) : 0.0f;
        const float a_rec = cmax > 0 ? fmaxf(fabsf(mx + c_raw), fabsf(mn + c_raw)) : 0.0f;
        st_acc = fmaxf(st_acc, a_acc);
        st_rec = fmaxf(st_rec, a_rec);
        if (p.bstats != nullptr) {
          const unsigned u_acc = __reduce_max_sync(0xffffffffu, __float_as_uint(a_acc));
          const unsigned u_rec = __reduce_max_sync(0xffffffffu, __float_as_uint(a_rec));
          if (lane == 0) {
            unsigned* bs = p.bstats + ((static_cast<size_t>(b) * p.Hq + hq) * p.nbt + j) * 2;
            atomicMax(bs, u_acc);
            atomicMax(bs + 1, u_rec);
          }
        }
      }
      const float bm = (mx == -INFINITY) ? -INFINITY : (FP8 ? fmaf(mx, fsc, c_raw) : mx + c_raw) * sl2;
      const float m_new = fmaxf(m_run, bm);
      // Lazy rescale decision, with selects instead of branches; the O rescale itself waits
      // for PV(j-1) further down. Block 0 takes its max as the running max and leaves l and O.
      const bool need = m_new > m_run + kRescaleLog2;
      const bool later = j > 0;
      const float alpha_n = ex2_approx(m_run - m_new);
      const float alpha = need ? alpha_n : 1.0f;
      if constexpr (F16PV) {
        const float l_s = __half2float(__hmul(__float2half_rn(l_run), __float2half_rn(alpha_n)));
        l_run = (need && later) ? l_s : l_run;
      } else {
        l_run = (need && later) ? l_run * alpha_n : l_run;
      }
      m_run = (need || !later) ? m_new : m_run;
      const bool rescale = __any_sync(0xffffffffu, need) && later;
      // p = exp2((S' + c) * scale*log2e - m): MUFU ex2 per element, packed fp32 arithmetic per
      // pair, row sums in four independent pair accumulators.
      float rs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t hs[4] = {0u, 0u, 0u, 0u};  // F16PV: fp16 row-sum accumulators (f16x2)
      uint32_t pk[kPairs];
      if constexpr (F16ACC) {
        // x = (S' + (c - m / sl2)) * sl2
        const float b16 = (m_run == -INFINITY) ? 0.0f : c_raw - m_run * p.inv_scale_log2;
#pragma unroll
        for (int c = 0; c < kPairs; ++c) {
          float y0, y1, x0, x1;
          add_f16x2_f32(y0, y1, hp[c], b16);
          fmul2(x0, x1, y0, y1, sl2, sl2);
          float p0, p1;
          exp2_split(p0, p1, x0, x1, c);
          pk[c] = pack_half2(p0, p1);
          if constexpr (F16PV) {
            hs[c & 3] = hadd2(hs[c & 3], pk[c]);
          } else {
            const int a = (c & 3) * 2;
            fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
          }
        }
      } else {
        const float bias = (m_run == -INFINITY) ? 0.0f : c_raw * sl2 - m_run;
        const float mul = FP8 ? fsc * sl2 : sl2;
#pragma unroll
        for (int c = 0; c < kPairs; ++c) {
          float x0, x1;
          ffma2(x0, x1, sv[2 * c], sv[2 * c + 1], mul, mul, bias, bias);
          float p0, p1;
          exp2_split(p0, p1, x0, x1, c);
          const int a = (c & 3) * 2;
          fadd2(rs[a], rs[a + 1], rs[a], rs[a + 1], p0, p1);
          pk[c] = pack_half2(p0, p1);
        }
      }
      if constexpr (F16PV) {
        const uint32_t h = hadd2(hadd2(hs[0], hs[1]), hadd2(hs[2], hs[3]));
        const __half rsum = __hadd(__ushort_as_half(static_cast<unsigned short>(h & 0xFFFFu)),
                                   __ushort_as_half(static_cast<unsigned short>(h >> 16)));
        l_run = __half2float(__hadd(__float2half_rn(l_run), rsum));
      } else {
        const float rowsum = ((rs[0] + rs[1]) + (rs[2] + rs[3])) + ((rs[4] + rs[5]) + (rs[6] + rs[7]));
        l_run += rowsum;
      }
      // PV(j-1) has to be done before O is rescaled or P rewritten; the exponentials above
      // overlap it.
      if (j >= 1 && !mbar_wait(&s.p_free, (j - 1) & 1, abort_flag, 0x320)) { ok = false; break; }
      tc_fence_after();
      // P first: its stores do not depend on the rescale, and their latency overlaps it (not
      // in the fused kernel, where that order makes the 168-register code spill)
      if constexpr (!FUSED) {
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) tmem_st_x8(tP + c * 8, pk + c * 8);
      }
      if (rescale) {
        if constexpr (F16PV) {
          uint32_t w[16];
          const uint32_t a2 = pack_half2(alpha, alpha);
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            tmem_ld_x16_pack16(tO + c * 32, w);
            tmem_ld_wait();
            reg_fence<16>(w);
#pragma unroll
            for (int e = 0; e < 16; ++e) w[e] = hmul2(w[e], a2);
            tmem_st_x16_unpack16(tO + c * 32, w);
          }
        } else {
          // kRc columns per load round, one wait each (a heavy-tailed workload rescales in
          // about a fifth of its warp-blocks, inside the softmax's chain); the fused kernel,
          // at 168 registers, keeps rounds of 16
          constexpr int kRc = FUSED ? 16 : 64;
#pragma unroll
          for (int b0 = 0; b0 < D; b0 += kRc) {
            uint32_t w[kRc];
#pragma unroll
            for (int c = 0; c < kRc / 16; ++c) tmem_ld_x16(tO + b0 + c * 16, w + c * 16);
            tmem_ld_wait();
            reg_fence<kRc>(w);
#pragma unroll
            for (int e = 0; e < kRc; e += 2) {
              float a, b;
              fmul2(a, b, __uint_as_float(w[e]), __uint_as_float(w[e + 1]), alpha, alpha);
              w[e] = __float_as_uint(a);
              w[e + 1] = __float_as_uint(b);
            }
#pragma unroll
            for (int c = 0; c < kRc / 16; ++c) tmem_st_x16(tO + b0 + c * 16, w + c * 16);
          }
        }
      }
      if constexpr (FUSED) {
#pragma unroll
        for (int c = 0; c < BN / 16; ++c) tmem_st_x8(tP + c * 8, pk + c * 8);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      mbar_arrive_if(&s.p_full, lane == 0);
    }

    // epilogue: O / l -> fp16 -> swizzled staging (the Q buffer) -> TMA store
    const bool have_o = ok && nblk > 0;
    if (have_o && !mbar_wait(&s.o_full, 0, abort_flag, 0x310)) ok = false;
    // A tile without key blocks reaches here before any MMA: its Q load (into the buffer
    // reused as staging) must have landed before the staging is written.
    if (!have_o && !mbar_wait(&s.q_full, 0, abort_flag, 0x330)) ok = false;
    tc_fence_after();
    const float inv_l = (l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    if (p.part_o != nullptr) {
      // split keys: this CTA's O / l in fp32 and m + log2 l for the combine kernel (the TMEM
      // loads are warp-wide; only rows that exist are stored)
      const size_t rows_total = static_cast<size_t>(p.B) * p.Hq * p.Sq;
      const size_t row = (static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i;
      float* dst = p.part_o + (static_cast<size_t>(split) * rows_total + row) * D;
      const bool live = i < p.Sq;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float f[32];
        uint32_t w[16];
        if (have_o && ok) {
          if constexpr (F16PV) {
            tmem_ld_x16_pack16(tO + c * 32, w);
            tmem_ld_wait();
            reg_fence<16>(w);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              f[2 * e] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[e] & 0xFFFFu))) * inv_l;
              f[2 * e + 1] = __half2float(__ushort_as_half(static_cast<unsigned short>(w[e] >> 16))) * inv_l;
            }
          } else {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              tmem_ld_x16(tO + c * 32 + hh * 16, w);
              tmem_ld_wait();
              reg_fence<16>(w);
#pragma unroll
              for (int e = 0; e < 16; ++e) f[hh * 16 + e] = __uint_as_float(w[e]) * inv_l;
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) f[e] = 0.0f;
        }
        if (live) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            reinterpret_cast<float4*>(dst + c * 32)[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
        }
      }
      if (live) p.part_lse[static_cast<size_t>(split) * rows_total + row] = (l_run > 0.0f) ? m_run + log2f(l_run) : -INFINITY;
    } else {
    uint8_t* stage = s.q;
    // 16 output columns starting at col, as 8 packed fp16 pairs, into the swizzled staging
    auto stage16 = [&](int col, const uint32_t* h) {
      const int chunk = col / 64;
      const int u0 = (col % 64) / 8;
      uint8_t* rowp = stage + chunk * Smem::kQChunk + r * 128;
      *reinterpret_cast<uint4*>(rowp + ((u0 ^ (r & 7)) * 16)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(rowp + (((u0 + 1) ^ (r & 7)) * 16)) = make_uint4(h[4], h[5], h[6], h[7]);
    };
    if constexpr (F16PV) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t w[16];
        if (have_o && ok) {
          tmem_ld_x16_pack16(tO + c * 32, w);
          tmem_ld_wait();
          reg_fence<16>(w);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = 0u;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t h[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t v2 = w[half * 8 + e];
            const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(v2 & 0xFFFFu)));
            const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(v2 >> 16)));
            h[e] = pack_half2(lo * inv_l, hi * inv_l);
          }
          stage16(c * 32 + half * 16, h);
        }
      }
    } else {
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
        stage16(c * 16, h);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 128);
    if (r == 0) {
#pragma unroll
      for (int c = 0; c < Smem::kChunks; ++c) tma_store_3d(&mapO, stage + c * Smem::kQChunk, c * 64, q0, b * p.Hq + hq);
      tma_store_commit();
      tma_store_wait_all();
    }
    if constexpr (STATS) {
      if (i < p.Sq) {
        float* st = p.stats + ((static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i) * 2;
        st[0] = st_acc;
        st[1] = st_rec;
      }
    }
    if (p.lse != nullptr && i < p.Sq) {
      const float lse = (l_run > 0.0f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
      p.lse[(static_cast<size_t>(b) * p.Hq + hq) * p.Sq + i] = lse;
    }
    }  // not split
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

// Merge of split-key partials: for each row, with lse_s = m_s + log2 l_s (log2 units) and
// O_s = O / l of split s, O = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M) and
// LSE = ln 2 * (M + log2 sum_s 2^(lse_s - M)), M = max_s lse_s (a row no split saw gets
// O = 0 and LSE = -inf). One warp per row, D / 32 columns per lane; HBM-bound and small.
template <int D>
__global__ void __launch_bounds__(256) combine_splits_kernel(const float* __restrict__ part_o,
                                                             const float* __restrict__ part_lse, int splits,
                                                             long long rows, __half* __restrict__ o,
                                                             float* __restrict__ lse) {
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float mx = -INFINITY;
  for (int s2 = 0; s2 < splits; ++s2) mx = fmaxf(mx, part_lse[s2 * rows + row]);
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (mx != -INFINITY) {
    for (int s2 = 0; s2 < splits; ++s2) {
      const float ls = part_lse[s2 * rows + row];
      if (ls == -INFINITY) continue;
      const float w = exp2f(ls - mx);
      wsum += w;
      const float* src = part_o + (s2 * rows + row) * D + lane * kPer;
#pragma unroll
      for (int e = 0; e < kPer; ++e) acc[e] = fmaf(w, src[e], acc[e]);
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int e = 0; e < kPer; ++e) o[row * D + lane * kPer + e] = __float2half_rn(acc[e] * inv);
  if (lane == 0 && lse != nullptr) lse[row] = wsum > 0.0f ? (mx + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace pasa
