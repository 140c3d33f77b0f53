// libpasa.so: the C ABI declared in include/pasa.h. Host-side argument validation, TMA
// descriptor encoding, workspace layout and kernel dispatch. Compiled as one translation
// unit for sm_103a.
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/pasa.h"
#include "attn_fwd.cuh"
#include "attn_fwd2s.cuh"
#include "decode_fwd.cuh"
#include "kshift.cuh"
#include "ptx.cuh"

namespace pasa {

// Site tag the self-test below records in the device error word.
constexpr uint32_t kSelftestSite = 0x5E1F7E57u;

// The failure-detection path without a fault: thread 0 waits, through the bounded mbarrier
// wait every kernel of this library uses, on a barrier that nothing arrives on. The wait
// gives up after kWaitTimeoutNs, records the timeout in the device error word and returns;
// the CTA holds no TMA copy and no tensor memory, so it simply ends.
__global__ void wait_selftest_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    (void)mbar_wait(&bar, 0, &abort_flag, kSelftestSite);
  }
}

// Element i: the FMA-pipe exponential the softmax uses for part of its scores (poly) and the
// MUFU one it uses for the rest (mufu), both of x[i]; pairs go through exp2_fma2 together.
__global__ void exp2_selftest_kernel(const float* __restrict__ x, float* __restrict__ poly, float* __restrict__ mufu,
                                     int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i];
  const float x1 = i + 1 < n ? x[i + 1] : 0.0f;
  float p0, p1;
  exp2_fma2(p0, p1, x0, x1);
  poly[i] = p0;
  mufu[i] = ex2_approx(x0);
  if (i + 1 < n) {
    poly[i + 1] = p1;
    mufu[i + 1] = ex2_approx(x1);
  }
}

}  // namespace pasa

namespace {

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return PASA_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 3-D fp16 view [planes, rows, D] of a contiguous tensor, 128-byte swizzled boxes of
// 64 x box_rows x 1 elements.
// 3-D map (D, rows, planes) with 128-byte rows per box chunk: 64 fp16 or 128 one-byte elements.
// 3-D map over [planes][rows][D] with planes stride_rows rows apart (0: rows, dense).
int make_map(CUtensorMap* m, const void* base, int D, long long rows, long long planes, int box_rows,
             int elem_bytes = 2, long long stride_rows = 0) {
  auto enc = encode_fn();
  if (!enc) return cuda_fail(cudaErrorNotSupported);
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(planes)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem_bytes, static_cast<cuuint64_t>(stride_rows > 0 ? stride_rows : rows) * D * elem_bytes};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
  return PASA_OK;
}

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  return pasa_device_supported(dev) ? PASA_OK : PASA_ERR_UNSUPPORTED;
}

bool fp8_mode(int mode) { return mode == PASA_MODE_SHIFT_FP8 || mode == PASA_MODE_NAIVE_FP8; }

// Modes that shift the keys (and so need the block means).
bool shift_mode(int mode) {
  return mode == PASA_MODE_SHIFT_F16ACC || mode == PASA_MODE_SHIFT_F32ACC || mode == PASA_MODE_SHIFT_F16ALL ||
         mode == PASA_MODE_SHIFT_FP8;
}

// Workspace: the keys the attention kernel reads (fp16 K', or e4m3 codes in the FP8 modes),
// the block means [B,Hkv,nb,D] fp16 and, in the FP8 modes, the block scales [B,Hkv,nb] fp32;
// each part 256-byte aligned.
struct WorkspaceLayout {
  size_t kshift_off, means_off, kscale_off, total;
};

WorkspaceLayout workspace_layout(int B, int Hkv, int Sk, int D, int mode) {
  const int bn = pasa::block_rows_for(D);
  const size_t nb = (static_cast<size_t>(Sk) + bn - 1) / bn;
  const size_t eb = fp8_mode(mode) ? 1 : 2;
  WorkspaceLayout w;
  w.kshift_off = 0;
  w.means_off = align_up(static_cast<size_t>(B) * Hkv * Sk * D * eb, 256);
  w.kscale_off = align_up(w.means_off + static_cast<size_t>(B) * Hkv * nb * D * 2, 256);
  w.total = fp8_mode(mode) ? align_up(w.kscale_off + static_cast<size_t>(B) * Hkv * nb * 4, 256) : w.kscale_off;
  return w;
}

template <int D, int OUT, bool PLAIN = false>
int launch_kshift(const void* k, void* ks, void* means, float* kscale, int B, int H, int Sk, cudaStream_t st,
                  int first_block = 0, int cap = 0) {
  constexpr int BN = pasa::block_rows_for(D);
  const int nb = (Sk + BN - 1) / BN;
  if (cap <= 0) cap = Sk;
  dim3 grid(nb - first_block, B * H);
  if constexpr (OUT == pasa::kShiftF16 && !PLAIN) {
    // the fp16 grid-mean shift: the register-resident kernel
    pasa::kshift_reg_kernel<D, BN><<<grid, pasa::kShiftRegThreads, 0, st>>>(
        static_cast<const __half*>(k), static_cast<__half*>(ks), static_cast<__half*>(means), Sk, nb, first_block,
        cap, (cap + BN - 1) / BN);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PASA_OK : cuda_fail(e);
  }
  pasa::kshift_kernel<D, BN, OUT, PLAIN><<<grid, pasa::kShiftThreads, 0, st>>>(
      static_cast<const __half*>(k), ks, static_cast<__half*>(means), kscale, Sk, nb, first_block, cap,
      (cap + BN - 1) / BN);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

// fp16 K' for the fp16 modes; e4m3 codes (of K', or of K in the naive FP8 mode) otherwise.
// The key preparation of `mode` (fp16 shift, or e4m3 codes and scales) for key blocks
// [first_block, ceil(Sk / BN)) of heads holding cap (>= Sk) rows each.
int kshift_dispatch(const void* k, void* ks, void* means, float* kscale, int B, int H, int Sk, int D, int mode,
                    cudaStream_t st, int first_block = 0, int cap = 0) {
  if (mode == PASA_MODE_SHIFT_FP8)
    return launch_kshift<128, pasa::kShiftFp8>(k, ks, means, kscale, B, H, Sk, st, first_block, cap);
  if (mode == PASA_MODE_NAIVE_FP8)
    return launch_kshift<128, pasa::kRawFp8>(k, ks, means, kscale, B, H, Sk, st, first_block, cap);
  return D == 64 ? launch_kshift<64, pasa::kShiftF16>(k, ks, means, nullptr, B, H, Sk, st, first_block, cap)
                 : launch_kshift<128, pasa::kShiftF16>(k, ks, means, nullptr, B, H, Sk, st, first_block, cap);
}

// Launch `kern` on `st`; with pdl, by programmatic stream serialization: the kernel may start
// while the kernel queued just ahead of it (the key preparation of the same call) still
// runs, and waits for it with griddep_wait() before reading what it writes.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, int smem, cudaStream_t st, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, bool F16ACC, bool SHIFT, bool CAUSAL, bool STATS, bool F16PV = false, bool FP8 = false>
int launch_attn(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                const CUtensorMap& mm, const pasa::AttnParams& p, cudaStream_t st, bool pdl = false) {
  constexpr int BN = pasa::block_rows_for(D);
  // ring slots: D = 128 fp16 keys: 3 K + 2 V (201 KB of shared memory); e4m3 keys: 4 + 3
  constexpr int KST = D == 128 ? (FP8 ? 4 : 3) : 4;
  constexpr int VST = D == 128 ? (FP8 ? 3 : 2) : 4;
  using Smem = pasa::AttnSmem<D, BN, KST, VST, FP8>;
  auto kern = pasa::attn_fwd_kernel<D, BN, F16ACC, SHIFT, CAUSAL, KST, VST, STATS, F16PV, FP8>;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  const long long ctas = static_cast<long long>(p.n_qblk) * p.Hq * p.B;
  const unsigned splits = p.bps > 0 ? static_cast<unsigned>((p.nbt + p.bps - 1) / p.bps) : 1u;
  e = launch_kernel(kern, dim3(static_cast<unsigned>(ctas), splits), dim3(pasa::kAttnThreads), smem, st, pdl, mq, mk, mv,
                    mo, mm, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

// The fused-shift kernel (D = 128, modes 0, 1, 4): raw keys in, shift warps in the kernel.
template <bool F16ACC, bool CAUSAL, bool F16PV>
int launch_attn_fused(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                      const pasa::AttnParams& p, cudaStream_t st) {
  constexpr int D = 128, BN = 128, KST = 3, VST = 2;
  using Smem = pasa::AttnSmem<D, BN, KST, VST, false, true>;
  auto kern = pasa::attn_fwd_kernel<D, BN, F16ACC, true, CAUSAL, KST, VST, false, F16PV, false, true>;
  const int smem = static_cast<int>(sizeof(Smem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  const long long ctas = static_cast<long long>(p.n_qblk) * p.Hq * p.B;
  kern<<<static_cast<unsigned>(ctas), pasa::kAttnThreadsFused, smem, st>>>(mq, mk, mv, mo, mk, p);
  e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

template <int D, bool STATS>
int attn_dispatch(int mode, int causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                  const CUtensorMap& mo, const CUtensorMap& mm, const pasa::AttnParams& p, cudaStream_t st,
                  bool pdl = false) {
#define PASA_CASE(MODE, F16, SH)                                                        \
  case MODE:                                                                            \
    return causal ? launch_attn<D, F16, SH, true, STATS>(mq, mk, mv, mo, mm, p, st, pdl)     \
                  : launch_attn<D, F16, SH, false, STATS>(mq, mk, mv, mo, mm, p, st, pdl);
  switch (mode) {
    PASA_CASE(PASA_MODE_SHIFT_F16ACC, true, true)
    PASA_CASE(PASA_MODE_SHIFT_F32ACC, false, true)
    PASA_CASE(PASA_MODE_NAIVE_F16ACC, true, false)
    PASA_CASE(PASA_MODE_NOSHIFT_F32ACC, false, false)
    case PASA_MODE_SHIFT_F16ALL:
      return causal ? launch_attn<D, true, true, true, STATS, true>(mq, mk, mv, mo, mm, p, st, pdl)
                    : launch_attn<D, true, true, false, STATS, true>(mq, mk, mv, mo, mm, p, st, pdl);
    case PASA_MODE_SHIFT_FP8:
    case PASA_MODE_NAIVE_FP8:
      if constexpr (D == 128 && !STATS) {
        if (mode == PASA_MODE_SHIFT_FP8)
          return causal ? launch_attn<D, false, true, true, false, false, true>(mq, mk, mv, mo, mm, p, st, pdl)
                        : launch_attn<D, false, true, false, false, false, true>(mq, mk, mv, mo, mm, p, st, pdl);
        return causal ? launch_attn<D, false, false, true, false, false, true>(mq, mk, mv, mo, mm, p, st, pdl)
                      : launch_attn<D, false, false, false, false, false, true>(mq, mk, mv, mo, mm, p, st, pdl);
      }
      return PASA_ERR_UNSUPPORTED;
    default:
      return PASA_ERR_UNSUPPORTED;
  }
#undef PASA_CASE
}

int validate_shape(int B, int Hq, int Hkv, int Sq, int Sk, int D, int mode) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || Hq % Hkv != 0) return PASA_ERR_SHAPE;
  if (D != 64 && D != 128) return PASA_ERR_UNSUPPORTED;
  if (mode < PASA_MODE_SHIFT_F16ACC || mode > PASA_MODE_NAIVE_FP8) return PASA_ERR_UNSUPPORTED;
  if (fp8_mode(mode) && D != 128) return PASA_ERR_UNSUPPORTED;
  // grid size, TMA plane counts and flat LSE indices fit in 32-bit signed integers
  const long long n_qblk = (static_cast<long long>(Sq) + pasa::kTileRows - 1) / pasa::kTileRows;
  if (n_qblk * Hq * B > 0x7fffffffLL) return PASA_ERR_SHAPE;
  if (static_cast<long long>(B) * Hq > 0x7fffffffLL || static_cast<long long>(B) * Hkv > 0x7fffffffLL)
    return PASA_ERR_SHAPE;
  return PASA_OK;
}

int validate(const void* q, const void* k, const void* v, const void* o, const float* lse, int B, int Hq, int Hkv,
             int Sq, int Sk, int D, int mode) {
  if (!q || !k || !v || !o) return PASA_ERR_NULLPTR;
  const int rc = validate_shape(B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned16(lse)))
    return PASA_ERR_ALIGN;
  return PASA_OK;
}

// D = 64 prefill, modes 0-3: two softmax warp sets on alternate key blocks.
template <bool F16ACC, bool SHIFT, bool CAUSAL>
int launch_2set(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mo,
                const CUtensorMap& mm, const pasa::AttnParams& p, cudaStream_t st, bool pdl = false) {
  constexpr int KST = 4, VST = 4;
  auto kern = pasa::twoset::attn_fwd_2set_kernel<64, 128, F16ACC, SHIFT, CAUSAL, KST, VST, false>;
  const int smem = static_cast<int>(sizeof(pasa::twoset::AttnSmem<64, 128, KST, VST>)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  const long long ctas = static_cast<long long>(p.n_qblk) * p.Hq * p.B;
  e = launch_kernel(kern, dim3(static_cast<unsigned>(ctas)), dim3(pasa::twoset::kAttnThreads), smem, st, pdl, mq, mk,
                    mv, mo, mm, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

int twoset_dispatch(int mode, int causal, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                    const CUtensorMap& mo, const CUtensorMap& mm, const pasa::AttnParams& p, cudaStream_t st,
                    bool pdl = false) {
#define PASA_2S_CASE(MODE, F16, SH)                                                   \
  case MODE:                                                                          \
    return causal ? launch_2set<F16, SH, true>(mq, mk, mv, mo, mm, p, st, pdl)        \
                  : launch_2set<F16, SH, false>(mq, mk, mv, mo, mm, p, st, pdl);
  switch (mode) {
    PASA_2S_CASE(PASA_MODE_SHIFT_F16ACC, true, true)
    PASA_2S_CASE(PASA_MODE_SHIFT_F32ACC, false, true)
    PASA_2S_CASE(PASA_MODE_NAIVE_F16ACC, true, false)
    PASA_2S_CASE(PASA_MODE_NOSHIFT_F32ACC, false, false)
    default:
      return PASA_ERR_UNSUPPORTED;
  }
#undef PASA_2S_CASE
}

// The swapped-operand decode kernel (D = 128, at most 32 packed query rows per kv head).
// pdl: launch with programmatic stream serialization, so the kernel may start while the
// refresh queued ahead of it still runs (it waits for it before reading p.dep_block on).
template <int NQ, bool F16ACC, bool SHIFT, bool F16PV, bool FP8 = false>
int launch_decode(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const CUtensorMap& mm,
                         const pasa::DecodeParams& p, long long planes, int splits, cudaStream_t st, bool pdl) {
  // e4m3 keys at 16 columns: two softmax warpgroups (even and odd key blocks) and rings of
  // 4 K + 3 V; fp16 keys: one group with 3 K' + 3 V (16 columns) or 3 + 2 (32 columns).
  // (Measured on the 8 x 32K-key cache: two groups lift the e4m3 cache by 7%, while the fp16
  // cache gains more from the third V slot that two groups leave no room for.)
  constexpr int G = (FP8 && NQ == 16) ? 2 : 1;
  constexpr int KST = FP8 ? 4 : 3, VST = (FP8 || NQ == 16) ? 3 : 2;
  auto kern = pasa::decode_fwd_kernel<NQ, F16ACC, SHIFT, F16PV, KST, VST, FP8, G>;
  const int smem = static_cast<int>(sizeof(pasa::DecodeSmem<NQ, KST, VST, FP8, G>)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_fail(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(planes), static_cast<unsigned>(splits));
  cfg.blockDim = dim3(pasa::dec_threads(G));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (p.cluster) {
    // the splits of a kv head as one cluster (at most 8: the portable cluster size)
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 1;
    attr[na].val.clusterDim.y = static_cast<unsigned>(splits);
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (na > 0) {
    cfg.attrs = attr;
    cfg.numAttrs = na;
  }
  e = cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mm, p);
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

template <int NQ>
int decode_dispatch(int mode, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const CUtensorMap& mm, const pasa::DecodeParams& p, long long planes, int splits,
                           cudaStream_t st, bool pdl) {
#define PASA_DEC_CASE(MODE, ...) \
  case MODE: return launch_decode<NQ, __VA_ARGS__>(mq, mk, mv, mm, p, planes, splits, st, pdl);
  switch (mode) {
    PASA_DEC_CASE(PASA_MODE_SHIFT_F16ACC, true, true, false)
    PASA_DEC_CASE(PASA_MODE_SHIFT_F32ACC, false, true, false)
    PASA_DEC_CASE(PASA_MODE_NAIVE_F16ACC, true, false, false)
    PASA_DEC_CASE(PASA_MODE_NOSHIFT_F32ACC, false, false, false)
    PASA_DEC_CASE(PASA_MODE_SHIFT_F16ALL, true, true, true)
    PASA_DEC_CASE(PASA_MODE_SHIFT_FP8, false, true, false, true)
    PASA_DEC_CASE(PASA_MODE_NAIVE_FP8, false, false, false, true)
    default: return PASA_ERR_UNSUPPORTED;
  }
#undef PASA_DEC_CASE
}

}  // namespace

extern "C" {

int pasa_block_rows(int D) { return pasa::block_rows_for(D); }

int pasa_last_cuda_error(void) { return t_last_cuda_error; }

int pasa_device_supported(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess) return 0;
  return (major == 10 && minor == 3) ? 1 : 0;
}

const char* pasa_strerror(int status) {
  switch (status) {
    case PASA_OK: return "ok";
    case PASA_ERR_NULLPTR: return "a required pointer is NULL";
    case PASA_ERR_SHAPE: return "invalid sizes (<= 0, Hq % Hkv != 0, or too large)";
    case PASA_ERR_UNSUPPORTED: return "unsupported head dim, mode or device (needs D in {64,128}, sm_103)";
    case PASA_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case PASA_ERR_CUDA: return "a CUDA call failed";
    case PASA_ERR_TIMEOUT: return "a device pipeline wait timed out";
    case PASA_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

size_t pasa_attn_fwd_workspace_bytes(int B, int Hkv, int Sk, int D, int mode) {
  if (B <= 0 || Hkv <= 0 || Sk <= 0 || pasa::block_rows_for(D) == 0) return 0;
  if (!shift_mode(mode) && !fp8_mode(mode)) return 0;
  if (fp8_mode(mode) && D != 128) return 0;
  return workspace_layout(B, Hkv, Sk, D, mode).total;
}

int pasa_kshift(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int D, void* stream) {
  if (!k || !k_shifted || !means) return PASA_ERR_NULLPTR;
  if (B <= 0 || H <= 0 || Sk <= 0) return PASA_ERR_SHAPE;
  if (D != 64 && D != 128) return PASA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return PASA_ERR_SHAPE;  // grid.y
  if (!aligned16(k) || !aligned16(k_shifted) || !aligned16(means)) return PASA_ERR_ALIGN;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  return kshift_dispatch(k, k_shifted, means, nullptr, B, H, Sk, D, PASA_MODE_SHIFT_F16ACC,
                         static_cast<cudaStream_t>(stream));
}

int pasa_kshift_mean(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int D, int mean_rule,
                     void* stream) {
  if (mean_rule == PASA_MEAN_GRID) return pasa_kshift(k, k_shifted, means, B, H, Sk, D, stream);
  if (mean_rule != PASA_MEAN_PLAIN) return PASA_ERR_UNSUPPORTED;
  if (!k || !k_shifted || !means) return PASA_ERR_NULLPTR;
  if (B <= 0 || H <= 0 || Sk <= 0) return PASA_ERR_SHAPE;
  if (D != 64 && D != 128) return PASA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return PASA_ERR_SHAPE;  // grid.y
  if (!aligned16(k) || !aligned16(k_shifted) || !aligned16(means)) return PASA_ERR_ALIGN;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_kshift<64, pasa::kShiftF16, true>(k, k_shifted, means, nullptr, B, H, Sk, st)
                 : launch_kshift<128, pasa::kShiftF16, true>(k, k_shifted, means, nullptr, B, H, Sk, st);
}

int pasa_kprep_fp8(const void* k, void* k8, void* means, float* kscale, int B, int H, int Sk, int D, int mode,
                   void* stream) {
  if (!k || !k8 || !kscale || (mode == PASA_MODE_SHIFT_FP8 && !means)) return PASA_ERR_NULLPTR;
  if (B <= 0 || H <= 0 || Sk <= 0) return PASA_ERR_SHAPE;
  if (D != 128 || !fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return PASA_ERR_SHAPE;  // grid.y
  if (!aligned16(k) || !aligned16(k8) || (means && !aligned16(means)) || !aligned16(kscale)) return PASA_ERR_ALIGN;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  return kshift_dispatch(k, k8, means, kscale, B, H, Sk, D, mode, static_cast<cudaStream_t>(stream));
}

int pasa_kshift_blocks(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int Sk_cap, int D,
                       int first_block, void* stream) {
  if (!k || !k_shifted || !means) return PASA_ERR_NULLPTR;
  if (B <= 0 || H <= 0 || Sk <= 0 || Sk_cap < Sk) return PASA_ERR_SHAPE;
  if (D != 64 && D != 128) return PASA_ERR_UNSUPPORTED;
  const int nb = (Sk + pasa::block_rows_for(D) - 1) / pasa::block_rows_for(D);
  if (first_block < 0 || first_block >= nb) return PASA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 65535) return PASA_ERR_SHAPE;  // grid.y
  if (!aligned16(k) || !aligned16(k_shifted) || !aligned16(means)) return PASA_ERR_ALIGN;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return D == 64 ? launch_kshift<64, pasa::kShiftF16>(k, k_shifted, means, nullptr, B, H, Sk, st, first_block, Sk_cap)
                 : launch_kshift<128, pasa::kShiftF16>(k, k_shifted, means, nullptr, B, H, Sk, st, first_block, Sk_cap);
}

// Launch the attention kernel on (possibly shifted) keys `kk` and block means `mm`.
// pdl: the key preparation of the same call was launched just before on `st` (see
// launch_kernel); never with the diagnostic outputs, whose zeroing sits in between.
static int attn_launch(const void* q, const void* kk, const void* mm, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode, cudaStream_t st,
                       float* stats = nullptr, float* block_stats = nullptr, const float* kscale = nullptr,
                       bool pdl = false) {
  const bool shift = shift_mode(mode);
  if (!(scale > 0.0f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  const int bn = pasa::block_rows_for(D);
  const int nb = (Sk + bn - 1) / bn;
  int rc;
  CUtensorMap mq, mk, mv, mo, mmeans;
  if ((rc = make_map(&mq, q, D, Sq, static_cast<long long>(B) * Hq, pasa::kTileRows)) != PASA_OK) return rc;
  if ((rc = make_map(&mk, kk, D, Sk, static_cast<long long>(B) * Hkv, bn, fp8_mode(mode) ? 1 : 2)) != PASA_OK)
    return rc;
  if ((rc = make_map(&mv, v, D, Sk, static_cast<long long>(B) * Hkv, bn)) != PASA_OK) return rc;
  if ((rc = make_map(&mo, o, D, Sq, static_cast<long long>(B) * Hq, pasa::kTileRows)) != PASA_OK) return rc;
  if (shift) {
    if ((rc = make_map(&mmeans, mm, D, nb, static_cast<long long>(B) * Hkv, pasa::kChunkBlocks)) != PASA_OK)
      return rc;
  } else {
    mmeans = mk;  // unused by the no-shift kernels
  }
  pasa::AttnParams p;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.n_qblk = (Sq + pasa::kTileRows - 1) / pasa::kTileRows;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.inv_scale_log2 = 1.0f / p.scale_log2;
  p.stats = stats;
  p.bstats = reinterpret_cast<unsigned*>(block_stats);
  p.nbt = nb;
  p.kscale = kscale;
  p.sq_mod = Sq;
  p.bps = 0;
  p.part_o = nullptr;
  p.part_lse = nullptr;
  p.kshift_out = nullptr;
  p.means_out = nullptr;
  if (block_stats) {
    const cudaError_t e = cudaMemsetAsync(block_stats, 0, static_cast<size_t>(B) * Hq * nb * 2 * sizeof(float), st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (stats)
    return D == 64 ? attn_dispatch<64, true>(mode, causal, mq, mk, mv, mo, mmeans, p, st)
                   : attn_dispatch<128, true>(mode, causal, mq, mk, mv, mo, mmeans, p, st);
  if (D == 64 && mode <= PASA_MODE_NOSHIFT_F32ACC)
    return twoset_dispatch(mode, causal, mq, mk, mv, mo, mmeans, p, st, pdl);
  return D == 64 ? attn_dispatch<64, false>(mode, causal, mq, mk, mv, mo, mmeans, p, st, pdl)
                 : attn_dispatch<128, false>(mode, causal, mq, mk, mv, mo, mmeans, p, st, pdl);
}

int pasa_attn_fwd_shifted(const void* q, const void* k_shifted, const void* means, const void* v, void* o,
                          float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                          int mode, void* stream) {
  int rc = validate(q, k_shifted, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;  // the FP8 modes read e4m3 keys, not fp16 K'
  const bool shift = shift_mode(mode);
  if (shift && !means) return PASA_ERR_NULLPTR;
  if (shift && !aligned16(means)) return PASA_ERR_ALIGN;
  rc = check_device();
  if (rc != PASA_OK) return rc;
  return attn_launch(q, k_shifted, shift ? means : k_shifted, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode,
                     static_cast<cudaStream_t>(stream));
}

int pasa_attn_fwd_fp8(const void* q, const void* k8, const void* means, const float* kscale, const void* v, void* o,
                      float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode,
                      void* stream) {
  int rc = validate(q, k8, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (!fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;
  if (!kscale || (mode == PASA_MODE_SHIFT_FP8 && !means)) return PASA_ERR_NULLPTR;
  if (!aligned16(kscale) || (means && !aligned16(means))) return PASA_ERR_ALIGN;
  rc = check_device();
  if (rc != PASA_OK) return rc;
  return attn_launch(q, k8, mode == PASA_MODE_SHIFT_FP8 ? means : k8, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale,
                     mode, static_cast<cudaStream_t>(stream), nullptr, nullptr, kscale);
}

// Decode path: key-block split and its partial-result workspace. By default at most one
// wave of CTAs (152 SMs, one CTA each) and at least eight key blocks per split, so that a
// CTA's fixed start-up and pipeline fill stay small against its streaming time.
static int decode_split(int B, int Hkv, int Sk, int D, int splits_req, int* splits_out) {
  const int bn = pasa::block_rows_for(D);
  const int nb = (Sk + bn - 1) / bn;
  const long long units = static_cast<long long>(B) * Hkv;
  int splits = splits_req > 0 ? splits_req : static_cast<int>(std::min<long long>(152 / units, nb / 8));
  splits = std::max(1, std::min(std::min(splits, nb), 65535));   // grid.y
  const int bps = (nb + splits - 1) / splits;
  splits = (nb + bps - 1) / bps;
  *splits_out = splits;
  return splits > 1 ? bps : 0;
}

// The swapped-operand decode kernel merges up to 8 splits of a kv head inside one cluster.
static bool decode_cluster_merge(int D, long long rows, int splits) {
  return D == 128 && rows <= 32 && splits >= 2 && splits <= 8;
}

size_t pasa_attn_fwd_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Sk <= 0 || Hq % Hkv != 0 || pasa::block_rows_for(D) == 0) return 0;
  int sp = 1;
  if (decode_split(B, Hkv, Sk, D, splits, &sp) == 0) return 0;
  if (decode_cluster_merge(D, static_cast<long long>(Hq / Hkv) * Sq, sp)) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * Sq;
  return align_up(static_cast<size_t>(sp) * rows * D * 4, 256) + align_up(static_cast<size_t>(sp) * rows * 4, 256);
}

// Decode on a key cache: fp16 keys (K' or K) for modes 0-4, e4m3 codes with block scales
// `kscale` for modes 5 and 6. dep_block < nb: the kernel queued just ahead on the stream
// rewrites key blocks [dep_block, nb) (a refresh); the swapped-operand decode kernel then
// starts while it runs and waits for it only before reading those blocks.
static int decode_impl(const void* q, const void* k_shifted, const void* means, const float* kscale, const void* v,
                       void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal,
                       float scale, int mode, int splits, void* workspace, size_t workspace_bytes, void* stream,
                       int dep_block = INT_MAX) {
  int rc = validate(q, k_shifted, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (Sk_cap < Sk) return PASA_ERR_SHAPE;
  if (splits < 0) return PASA_ERR_UNSUPPORTED;
  const int g = Hq / Hkv;
  if (static_cast<long long>(g) * Sq > pasa::kTileRows) return PASA_ERR_UNSUPPORTED;  // one tile per kv group
  const bool fp8 = fp8_mode(mode);
  // e4m3 keys run on the swapped-operand decode kernel only (D = 128, up to 32 packed rows)
  if (fp8 && (D != 128 || static_cast<long long>(g) * Sq > 32)) return PASA_ERR_UNSUPPORTED;
  if (fp8 && !kscale) return PASA_ERR_NULLPTR;
  if (fp8 && !aligned16(kscale)) return PASA_ERR_ALIGN;
  const bool shift = shift_mode(mode);
  if (shift && !means) return PASA_ERR_NULLPTR;
  if (shift && !aligned16(means)) return PASA_ERR_ALIGN;
  int sp = 1;
  const int bps = decode_split(B, Hkv, Sk, D, splits, &sp);
  const size_t need = pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, splits);
  const bool cluster = bps > 0 && decode_cluster_merge(D, static_cast<long long>(g) * Sq, sp);
  if (bps > 0 && !cluster) {
    if (!workspace || workspace_bytes < need) return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PASA_ERR_ALIGN;
  }
  rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!(scale > 0.0f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  const int bn = pasa::block_rows_for(D);
  const int nb = (Sk + bn - 1) / bn;
  // Q and O viewed as [B * Hkv, g * Sq, D]: the query rows of a kv group's g heads, contiguous
  const int rows = g * Sq;
  const long long planes = static_cast<long long>(B) * Hkv;
  const size_t nrows = static_cast<size_t>(B) * Hq * Sq;
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (bps > 0 && !cluster) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    part_o = reinterpret_cast<float*>(ws);
    part_lse = reinterpret_cast<float*>(ws + align_up(static_cast<size_t>(sp) * nrows * D * 4, 256));
  }
  CUtensorMap mq, mk, mv, mo, mmeans;
  // the cache: Sk valid rows of Sk_cap per head (reads past Sk are zero-filled and masked)
  if ((rc = make_map(&mk, k_shifted, D, Sk, planes, bn, fp8 ? 1 : 2, Sk_cap)) != PASA_OK) return rc;
  if ((rc = make_map(&mv, v, D, Sk, planes, bn, 2, Sk_cap)) != PASA_OK) return rc;
  if (shift) {
    if ((rc = make_map(&mmeans, means, D, nb, planes, pasa::kChunkBlocks, 2, (Sk_cap + bn - 1) / bn)) != PASA_OK)
      return rc;
  } else {
    mmeans = mk;
  }
  if (D == 128 && rows <= 32) {
    // few rows: keys on the MMA's M side (decode_fwd_kernel)
    const int nq = rows <= 16 ? 16 : 32;
    if ((rc = make_map(&mq, q, D, rows, planes, nq)) != PASA_OK) return rc;
    pasa::DecodeParams dp;
    dp.o = static_cast<__half*>(o);
    dp.lse = lse;
    dp.part_o = part_o;
    dp.part_lse = part_lse;
    dp.rows = rows;
    dp.sq = Sq;
    dp.Sk = Sk;
    dp.nbt = nb;
    dp.bps = bps;
    dp.causal = causal ? 1 : 0;
    dp.scale_log2 = scale * 1.4426950408889634f;
    dp.cluster = cluster ? 1 : 0;
    dp.kscale = kscale;
    dp.kstride = (Sk_cap + bn - 1) / bn;
    dp.dep_block = dep_block;
    const bool pdl = dep_block < nb;
    rc = nq == 16 ? decode_dispatch<16>(mode, mq, mk, mv, mmeans, dp, planes, sp, st, pdl)
                  : decode_dispatch<32>(mode, mq, mk, mv, mmeans, dp, planes, sp, st, pdl);
  } else {
    // query rows on the MMA's M side: the attention kernel on the packed [g * Sq] rows
    if ((rc = make_map(&mq, q, D, rows, planes, pasa::kTileRows)) != PASA_OK) return rc;
    if ((rc = make_map(&mo, o, D, rows, planes, pasa::kTileRows)) != PASA_OK) return rc;
    pasa::AttnParams p;
    p.lse = lse;
    p.B = B;
    p.Hq = Hkv;
    p.Hkv = Hkv;
    p.Sq = rows;
    p.Sk = Sk;
    p.n_qblk = 1;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.inv_scale_log2 = 1.0f / p.scale_log2;
    p.stats = nullptr;
    p.bstats = nullptr;
    p.nbt = nb;
    p.kscale = nullptr;
    p.sq_mod = Sq;
    p.bps = bps;
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.kshift_out = nullptr;
    p.means_out = nullptr;
    rc = D == 64 ? attn_dispatch<64, false>(mode, causal, mq, mk, mv, mo, mmeans, p, st)
                 : attn_dispatch<128, false>(mode, causal, mq, mk, mv, mo, mmeans, p, st);
  }
  if (rc != PASA_OK || bps == 0 || cluster) return rc;
  const unsigned cblocks = static_cast<unsigned>((nrows + 7) / 8);
  if (D == 64)
    pasa::combine_splits_kernel<64><<<cblocks, 256, 0, st>>>(part_o, part_lse, sp, static_cast<long long>(nrows),
                                                             static_cast<__half*>(o), lse);
  else
    pasa::combine_splits_kernel<128><<<cblocks, 256, 0, st>>>(part_o, part_lse, sp, static_cast<long long>(nrows),
                                                              static_cast<__half*>(o), lse);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

int pasa_attn_fwd_decode(const void* q, const void* k_shifted, const void* means, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal, float scale, int mode,
                         int splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;   // e4m3 caches: pasa_attn_fwd_decode_fp8
  return decode_impl(q, k_shifted, means, nullptr, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode,
                     splits, workspace, workspace_bytes, stream);
}

int pasa_attn_fwd_decode_step(const void* q, const void* k, void* k_shifted, void* means, const void* v, void* o,
                              float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal,
                              float scale, int mode, int first_block, int splits, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;   // e4m3 caches: pasa_kprep_fp8_blocks + _decode_fp8
  if (!shift_mode(mode)) {
    // raw-key modes keep no shifted copy: nothing to refresh
    return decode_impl(q, k_shifted, means, nullptr, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode,
                       splits, workspace, workspace_bytes, stream);
  }
  // argument checks of both calls before anything is enqueued
  if (!k) return PASA_ERR_NULLPTR;
  if (!aligned16(k)) return PASA_ERR_ALIGN;
  int rc = validate(q, k_shifted, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (!means) return PASA_ERR_NULLPTR;
  if (!aligned16(means)) return PASA_ERR_ALIGN;
  if (Sk_cap < Sk || splits < 0) return Sk_cap < Sk ? PASA_ERR_SHAPE : PASA_ERR_UNSUPPORTED;
  const int nb = (Sk + pasa::block_rows_for(D) - 1) / pasa::block_rows_for(D);
  if (first_block < 0 || first_block >= nb || static_cast<long long>(B) * Hkv > 65535) return PASA_ERR_SHAPE;
  if (static_cast<long long>(Hq / Hkv) * Sq > pasa::kTileRows) return PASA_ERR_UNSUPPORTED;
  int sp = 1;
  const int bps = decode_split(B, Hkv, Sk, D, splits, &sp);
  if (bps > 0 && !decode_cluster_merge(D, static_cast<long long>(Hq / Hkv) * Sq, sp)) {
    if (!workspace || workspace_bytes < pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, splits))
      return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PASA_ERR_ALIGN;
  }
  rc = pasa_kshift_blocks(k, k_shifted, means, B, Hkv, Sk, Sk_cap, D, first_block, stream);
  if (rc != PASA_OK) return rc;
  return decode_impl(q, k_shifted, means, nullptr, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode,
                     splits, workspace, workspace_bytes, stream, first_block);
}

int pasa_attn_fwd_decode_step_fp8(const void* q, const void* k, void* k8, void* means, float* kscale, const void* v,
                                  void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D,
                                  int causal, float scale, int mode, int first_block, int splits, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  if (!fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;   // fp16 caches: pasa_attn_fwd_decode_step
  // argument checks of both calls before anything is enqueued
  if (!k || !kscale || (mode == PASA_MODE_SHIFT_FP8 && !means)) return PASA_ERR_NULLPTR;
  if (!aligned16(k) || !aligned16(kscale) || (means && !aligned16(means))) return PASA_ERR_ALIGN;
  int rc = validate(q, k8, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (D != 128 || static_cast<long long>(Hq / Hkv) * Sq > 32) return PASA_ERR_UNSUPPORTED;
  if (Sk_cap < Sk || splits < 0) return Sk_cap < Sk ? PASA_ERR_SHAPE : PASA_ERR_UNSUPPORTED;
  const int nb = (Sk + 127) / 128;
  if (first_block < 0 || first_block >= nb || static_cast<long long>(B) * Hkv > 65535) return PASA_ERR_SHAPE;
  int sp = 1;
  const int bps = decode_split(B, Hkv, Sk, D, splits, &sp);
  if (bps > 0 && !decode_cluster_merge(D, static_cast<long long>(Hq / Hkv) * Sq, sp)) {
    if (!workspace || workspace_bytes < pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, splits))
      return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PASA_ERR_ALIGN;
  }
  rc = pasa_kprep_fp8_blocks(k, k8, means, kscale, B, Hkv, Sk, Sk_cap, D, mode, first_block, stream);
  if (rc != PASA_OK) return rc;
  return decode_impl(q, k8, means, kscale, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode, splits,
                     workspace, workspace_bytes, stream, first_block);
}

int pasa_attn_fwd_decode_fp8(const void* q, const void* k8, const void* means, const float* kscale, const void* v,
                             void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal,
                             float scale, int mode, int splits, void* workspace, size_t workspace_bytes, void* stream) {
  if (!fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;
  return decode_impl(q, k8, means, kscale, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode, splits,
                     workspace, workspace_bytes, stream);
}

int pasa_kprep_fp8_blocks(const void* k, void* k8, void* means, float* kscale, int B, int H, int Sk, int Sk_cap, int D,
                          int mode, int first_block, void* stream) {
  if (!k || !k8 || !kscale || (mode == PASA_MODE_SHIFT_FP8 && !means)) return PASA_ERR_NULLPTR;
  if (B <= 0 || H <= 0 || Sk <= 0 || Sk_cap < Sk) return PASA_ERR_SHAPE;
  if (D != 128 || !fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;
  const int nb = (Sk + 127) / 128;
  if (first_block < 0 || first_block >= nb) return PASA_ERR_SHAPE;
  if (static_cast<long long>(B) * H > 65535) return PASA_ERR_SHAPE;  // grid.y
  if (!aligned16(k) || !aligned16(k8) || !aligned16(kscale) || (means && !aligned16(means))) return PASA_ERR_ALIGN;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return mode == PASA_MODE_SHIFT_FP8
             ? launch_kshift<128, pasa::kShiftFp8>(k, k8, means, kscale, B, H, Sk, st, first_block, Sk_cap)
             : launch_kshift<128, pasa::kRawFp8>(k, k8, means, kscale, B, H, Sk, st, first_block, Sk_cap);
}

int pasa_attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int causal, float scale, int mode, void* workspace,
                     size_t workspace_bytes, void* stream) {
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  const bool prep = shift_mode(mode) || fp8_mode(mode);  // the shift kernel runs first
  const WorkspaceLayout wl = workspace_layout(B, Hkv, Sk, D, mode);
  if (prep) {
    if (!workspace || workspace_bytes < wl.total) return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PASA_ERR_ALIGN;
    if (static_cast<long long>(B) * Hkv > 65535) return PASA_ERR_SHAPE;  // kshift grid.y
  }
  rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* kk = k;
  const void* mm = k;
  float* kscale = nullptr;
  if (prep) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    void* ks = ws + wl.kshift_off;
    void* means = ws + wl.means_off;
    if (fp8_mode(mode)) kscale = reinterpret_cast<float*>(ws + wl.kscale_off);
    rc = kshift_dispatch(k, ks, means, kscale, B, Hkv, Sk, D, mode, st);
    if (rc != PASA_OK) return rc;
    kk = ks;
    mm = means;
  }
  return attn_launch(q, kk, mm, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, st, nullptr, nullptr, kscale,
                     prep);
}

int pasa_attn_fwd_stats(const void* q, const void* k, const void* v, void* o, float* lse, float* stats,
                        float* block_stats, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                        int mode, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (!stats) return PASA_ERR_NULLPTR;
  if ((reinterpret_cast<uintptr_t>(stats) & 7u) != 0) return PASA_ERR_ALIGN;
  if (block_stats && (reinterpret_cast<uintptr_t>(block_stats) & 7u) != 0) return PASA_ERR_ALIGN;
  if (fp8_mode(mode)) return PASA_ERR_UNSUPPORTED;  // no diagnostic build of the FP8 kernels
  const bool shift = shift_mode(mode);
  const WorkspaceLayout wl = workspace_layout(B, Hkv, Sk, D, mode);
  if (shift) {
    if (!workspace || workspace_bytes < wl.total) return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return PASA_ERR_ALIGN;
    if (static_cast<long long>(B) * Hkv > 65535) return PASA_ERR_SHAPE;
  }
  rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* kk = k;
  const void* mm = k;
  if (shift) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    rc = kshift_dispatch(k, ws + wl.kshift_off, ws + wl.means_off, nullptr, B, Hkv, Sk, D, mode, st);
    if (rc != PASA_OK) return rc;
    kk = ws + wl.kshift_off;
    mm = ws + wl.means_off;
  }
  return attn_launch(q, kk, mm, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, st, stats, block_stats);
}

int pasa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                  int Sq, int Sk, int D, int causal, float scale, int mode, void* stream) {
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  const size_t bytes = pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (bytes > 0) {
    rc = check_device();
    if (rc != PASA_OK) return rc;
    cudaError_t e = cudaMallocAsync(&ws, bytes, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  rc = pasa_attn_fwd_ws(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, ws, bytes, stream);
  if (ws) {
    cudaError_t e = cudaFreeAsync(ws, st);
    if (rc == PASA_OK && e != cudaSuccess) rc = cuda_fail(e);
  }
  return rc;
}

int pasa_attn_fwd_fused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, int D, int causal, float scale, int mode, void* k_shifted_out,
                        void* means_out, void* stream) {
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (D != 128) return PASA_ERR_UNSUPPORTED;
  if (mode != PASA_MODE_SHIFT_F16ACC && mode != PASA_MODE_SHIFT_F32ACC && mode != PASA_MODE_SHIFT_F16ALL)
    return PASA_ERR_UNSUPPORTED;
  if ((k_shifted_out && !aligned16(k_shifted_out)) || (means_out && !aligned16(means_out))) return PASA_ERR_ALIGN;
  rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!(scale > 0.0f) || !std::isfinite(scale)) scale = 1.0f / std::sqrt(static_cast<float>(D));
  const int bn = pasa::block_rows_for(D);
  CUtensorMap mq, mk, mv, mo;
  if ((rc = make_map(&mq, q, D, Sq, static_cast<long long>(B) * Hq, pasa::kTileRows)) != PASA_OK) return rc;
  if ((rc = make_map(&mk, k, D, Sk, static_cast<long long>(B) * Hkv, bn)) != PASA_OK) return rc;
  if ((rc = make_map(&mv, v, D, Sk, static_cast<long long>(B) * Hkv, bn)) != PASA_OK) return rc;
  if ((rc = make_map(&mo, o, D, Sq, static_cast<long long>(B) * Hq, pasa::kTileRows)) != PASA_OK) return rc;
  pasa::AttnParams p = {};
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.n_qblk = (Sq + pasa::kTileRows - 1) / pasa::kTileRows;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.inv_scale_log2 = 1.0f / p.scale_log2;
  p.nbt = (Sk + bn - 1) / bn;
  p.sq_mod = Sq;
  p.kshift_out = static_cast<__half*>(k_shifted_out);
  p.means_out = static_cast<__half*>(means_out);
  switch (mode) {
    case PASA_MODE_SHIFT_F16ACC:
      return causal ? launch_attn_fused<true, true, false>(mq, mk, mv, mo, p, st)
                    : launch_attn_fused<true, false, false>(mq, mk, mv, mo, p, st);
    case PASA_MODE_SHIFT_F32ACC:
      return causal ? launch_attn_fused<false, true, false>(mq, mk, mv, mo, p, st)
                    : launch_attn_fused<false, false, false>(mq, mk, mv, mo, p, st);
    default:
      return causal ? launch_attn_fused<true, true, true>(mq, mk, mv, mo, p, st)
                    : launch_attn_fused<true, false, true>(mq, mk, mv, mo, p, st);
  }
}

int pasa_selftest_wait_timeout(void* stream) {
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  pasa::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

int pasa_selftest_exp2(const float* x, float* poly, float* mufu, int n, void* stream) {
  if (!x || !poly || !mufu) return PASA_ERR_NULLPTR;
  if (n <= 0) return PASA_ERR_SHAPE;
  int rc = check_device();
  if (rc != PASA_OK) return rc;
  const int pairs = (n + 1) / 2;
  pasa::exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, poly, mufu, n);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}

int pasa_check_device_error(void* stream, unsigned long long* info) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  int word = 0;
  unsigned long long inf = 0;
  e = cudaMemcpyFromSymbol(&word, pasa::g_device_error, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e);
  e = cudaMemcpyFromSymbol(&inf, pasa::g_device_error_info, sizeof(inf));
  if (e != cudaSuccess) return cuda_fail(e);
  if (word == pasa::kDeviceOk) return PASA_OK;
  const int zero = 0;
  const unsigned long long zero64 = 0;
  cudaMemcpyToSymbol(pasa::g_device_error, &zero, sizeof(int));
  cudaMemcpyToSymbol(pasa::g_device_error_info, &zero64, sizeof(zero64));
  if (info) *info = inf;
  return PASA_ERR_TIMEOUT;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free variant of pasa_attn_fwd.
//
// Some callers may not call cudaMalloc at all: a process whose device memory is owned by a
// framework or server allocator that reserves the whole GPU up front, or a latency-bound
// loop where an allocation (and the synchronisation it can imply) is not allowed. For them
// the shifted keys and block means live in one file-scope device array instead of a
// workspace. The array is part of this library's device image, so every GPU that loads
// the library holds it until the process exits.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device. The host-side name of the
// array is only a stand-in, so the address is looked up once per device (with that device
// current) and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PASA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PASA_OK;
}

}  // namespace

extern "C" int pasa_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                     int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode,
                                     void* stream) {
  int rc = validate(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  const size_t need = pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode);
  if (need > kNoAllocScratchBytes) return PASA_ERR_WORKSPACE;
  rc = check_device();
  if (rc != PASA_OK) return rc;
  void* ws = nullptr;
  if (need > 0) {
    rc = noalloc_scratch(&ws);
    if (rc != PASA_OK) return rc;
  }
  return pasa_attn_fwd_ws(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, ws,
                          need > 0 ? kNoAllocScratchBytes : 0, stream);
}

// ---------------------------------------------------------------------------------------
// Host-buffer forward: q, k, v in host memory, o and lse back to host memory, with the
// copies overlapped with the attention kernels.
//
// The (batch, kv head) pairs are the units of work: a unit's query heads, keys, values and
// outputs are contiguous in the [B, H, S, D] layouts, and a run of consecutive units is
// itself a problem of n units with one kv head, n standing in for B. The work is cut into
// pieces; piece i's host->device copies run on one side stream, its shift and attention
// kernels on the caller's stream once they have landed, and its device->host copies on a
// second side stream once they have finished. Copy engines and SMs then work at the same
// time, and only the first piece's inputs and the last piece's outputs are not hidden
// behind computation.
//
// To keep those two small, the automatic plan also cuts the first and the last unit along
// the query rows, in pieces that halve towards the ends ([0, Sq/8), [Sq/8, Sq/4),
// [Sq/4, Sq/2), ... for the first unit, mirrored for the last). A row piece [r0, r1) is the
// problem with Sq' = r1 - r0 query rows and, under the causal mask, the key prefix
// Sk' = r1 + Sk - Sq it can see: row r0 + i' sees key j iff j <= i' + Sk' - Sq', the same
// keys as before. With r0 on a 128-row tile boundary and Sk' on a 128-key block boundary
// (or Sk' = Sk) every query tile meets the same key blocks with the same pseudo-averages,
// so the results stay bit-identical to the single call. The unit's keys are copied once,
// in the slices each row piece adds.
// ---------------------------------------------------------------------------------------
#include <vector>

namespace {

constexpr int kHostMaxChunks = 64;
constexpr long long kHostMinChunkTiles = 256;  // query tiles of 128 rows a unit chunk keeps
constexpr long long kHostMinRowTiles = 128;    // ... and the smallest row piece keeps
constexpr int kHostMaxHalvings = 3;

struct HostPiece {
  int u0 = 0, n = 0;    // units [u0, u0 + n)
  int r0 = 0, r1 = 0;   // query rows [r0, r1) of each unit
  int k0 = 0, k1 = 0;   // keys this piece copies in; it attends keys [0, k1)
  bool rowcut = false;  // one of the query-row pieces of a unit
  size_t q_off = 0, kv_off = 0, o_off = 0, lse_off = 0;  // slots in the device buffer
  size_t prep_off = 0;  // rowcut with a key preparation: the unit's prepared keys (all Sk rows)
};

struct HostPlan {
  std::vector<HostPiece> pieces;
  int max_units = 0;  // units in the largest piece that is not a row piece
  size_t ws_off = 0, ws_bytes = 0, total = 0;
};

// Row boundaries for one unit: halving pieces at the front and/or the back, on 128-row
// tiles, the smallest with at least kHostMinRowTiles tiles over the unit's g heads.
std::vector<int> host_row_cuts(int Sq, int g, bool front, bool back) {
  std::vector<int> cuts{0};
  int halvings = 0;
  while (halvings < kHostMaxHalvings) {
    const long long rows = (static_cast<long long>(Sq) >> (halvings + 1)) / 128 * 128;
    if (rows <= 0 || static_cast<long long>(g) * (rows / 128) < kHostMinRowTiles) break;
    ++halvings;
  }
  if (halvings == 0 || (!front && !back)) {
    cuts.push_back(Sq);
    return cuts;
  }
  auto tile = [](long long r) { return static_cast<int>(r / 128 * 128); };
  if (front)
    for (int h = halvings; h >= 1; --h) cuts.push_back(tile(static_cast<long long>(Sq) >> h));
  else
    cuts.push_back(tile(static_cast<long long>(Sq) >> 1));
  if (back)
    for (int h = 2; h <= halvings; ++h) cuts.push_back(tile(Sq - (static_cast<long long>(Sq) >> h)));
  cuts.push_back(Sq);
  std::vector<int> out{0};
  for (size_t i = 1; i < cuts.size(); ++i)
    if (cuts[i] > out.back()) out.push_back(cuts[i]);
  return out;
}

// Pieces: the units cut into chunks (the requested count clamped to [1, min(units, 64)];
// 0 asks for as many as keep every chunk at >= 256 query tiles, at most 8). Only the
// automatic plan cuts the first and last unit into row pieces, and only where the row
// pieces keep the computation tile-for-tile the same (see above).
HostPlan host_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, int mode, int chunks) {
  HostPlan hp;
  const int units = B * Hkv;
  const int g = Hq / Hkv;
  const int cap = units < kHostMaxChunks ? units : kHostMaxChunks;
  const bool automatic = chunks <= 0;
  if (automatic) {
    const long long tiles = static_cast<long long>(g) * ((static_cast<long long>(Sq) + 127) / 128);
    int c = cap < 8 ? cap : 8;
    while (c > 1 && (units / c) * tiles < kHostMinChunkTiles) --c;
    chunks = c;
  }
  chunks = chunks < cap ? chunks : cap;
  const bool rows_ok = automatic && (!causal || (Sk >= Sq && (Sk - Sq) % 128 == 0));
  for (int c = 0; c < chunks; ++c) {
    const int a = static_cast<int>(static_cast<long long>(c) * units / chunks);
    const int b = static_cast<int>(static_cast<long long>(c + 1) * units / chunks);
    for (int u = a; u < b;) {
      const bool first = u == 0, last = u == units - 1;
      std::vector<int> cuts{0, Sq};
      if (rows_ok && (first || last)) cuts = host_row_cuts(Sq, g, first, last);
      if (cuts.size() > 2) {
        int kprev = 0;
        for (size_t i = 0; i + 1 < cuts.size(); ++i) {
          HostPiece pc;
          pc.u0 = u, pc.n = 1, pc.r0 = cuts[i], pc.r1 = cuts[i + 1], pc.rowcut = true;
          pc.k1 = causal ? pc.r1 + (Sk - Sq) : Sk;
          pc.k0 = kprev;
          kprev = pc.k1;
          hp.pieces.push_back(pc);
        }
        ++u;
        continue;
      }
      // a run of whole units up to the chunk's end or the next unit that is cut into rows
      int e = u + 1;
      while (e < b && !(rows_ok && e == units - 1 && host_row_cuts(Sq, g, false, true).size() > 2)) ++e;
      HostPiece pc;
      pc.u0 = u, pc.n = e - u, pc.r0 = 0, pc.r1 = Sq, pc.k0 = 0, pc.k1 = Sk;
      hp.pieces.push_back(pc);
      u = e;
    }
  }
  // slots: q and o [n, g, rows, D], lse [n, g, rows], and the keys/values [n, Sk, D] of a
  // unit once (row pieces after the first of a unit reuse it), with, for a unit cut into
  // row pieces, its prepared keys (shifted keys and means, or e4m3 codes and scales, for
  // all Sk rows): each row piece prepares only the key blocks it newly sees, the blocks
  // before them being final once written (a block's preparation reads that block only);
  // each slot 256-byte aligned
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  const size_t prep_bytes = align_up(pasa_attn_fwd_workspace_bytes(1, 1, Sk, D, mode), 256);
  size_t off = 0, kv_last = 0, prep_last = 0;
  int kv_unit = -1;
  for (HostPiece& pc : hp.pieces) {
    const size_t nrows = static_cast<size_t>(pc.n) * g * (pc.r1 - pc.r0);
    pc.q_off = off;   off += align_up(nrows * row_bytes, 256);
    pc.o_off = off;   off += align_up(nrows * row_bytes, 256);
    pc.lse_off = off; off += align_up(nrows * 4, 256);
    if (pc.n == 1 && pc.k0 > 0 && kv_unit == pc.u0) {
      pc.kv_off = kv_last;
      pc.prep_off = prep_last;
    } else {
      pc.kv_off = kv_last = off;
      kv_unit = pc.n == 1 ? pc.u0 : -1;
      off += 2 * align_up(static_cast<size_t>(pc.n) * Sk * row_bytes, 256);
      if (pc.rowcut && prep_bytes > 0) {
        pc.prep_off = prep_last = off;
        off += prep_bytes;
      }
    }
    if (!pc.rowcut && pc.n > hp.max_units) hp.max_units = pc.n;
  }
  // one shift workspace per compute stream (pieces alternate between two), for the pieces of
  // whole units
  hp.ws_off = off;
  hp.ws_bytes = hp.max_units > 0 ? align_up(pasa_attn_fwd_workspace_bytes(hp.max_units, 1, Sk, D, mode), 256) : 0;
  hp.total = off + (hp.pieces.size() > 1 ? 2 : 1) * hp.ws_bytes;
  return hp;
}

// Three non-blocking side streams per device (host->device copies, device->host copies, a
// second compute stream), created on first use and kept for the life of the process. Calls
// from several host threads may share them: every wait a call enqueues refers to work that
// call has already enqueued, so the order stays acyclic.
std::mutex g_side_mutex;
cudaStream_t g_side_streams[kNoAllocMaxDevices][3] = {};

int side_streams(cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PASA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_side_mutex);
  for (int j = 0; j < 3; ++j) {
    if (g_side_streams[dev][j] == nullptr) {
      e = cudaStreamCreateWithFlags(&g_side_streams[dev][j], cudaStreamNonBlocking);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    out[j] = g_side_streams[dev][j];
  }
  return PASA_OK;
}

// `height` rows of `width` bytes between pitched buffers; one plain copy when both sides
// are contiguous.
cudaError_t copy_rows(void* dst, size_t dpitch, const void* src, size_t spitch, size_t width, size_t height,
                      cudaMemcpyKind kind, cudaStream_t st) {
  if (width == 0 || height == 0) return cudaSuccess;
  if (dpitch == width && spitch == width) return cudaMemcpyAsync(dst, src, width * height, kind, st);
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, height, kind, st);
}

}  // namespace

extern "C" int pasa_release_host_streams(void) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kNoAllocMaxDevices) return PASA_OK;   // none were ever created there
  std::lock_guard<std::mutex> lock(g_side_mutex);
  cudaError_t first = cudaSuccess;
  for (int j = 0; j < 3; ++j) {
    cudaStream_t& st = g_side_streams[dev][j];
    if (st == nullptr) continue;
    e = cudaStreamSynchronize(st);
    if (e == cudaSuccess) e = cudaStreamDestroy(st);
    if (e != cudaSuccess && first == cudaSuccess) first = e;
    st = nullptr;   // a failed destroy leaves the handle to the runtime; never reuse it
  }
  return first == cudaSuccess ? PASA_OK : cuda_fail(first);
}

extern "C" size_t pasa_attn_fwd_host_device_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal,
                                                   int mode, int chunks) {
  if (chunks < 0 || validate_shape(B, Hq, Hkv, Sq, Sk, D, mode) != PASA_OK) return 0;
  return host_plan(B, Hq, Hkv, Sq, Sk, D, causal, mode, chunks).total;
}

extern "C" int pasa_attn_fwd_host_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, int mode,
                                       int chunks, int* pieces, int max_pieces) {
  if (chunks < 0 || max_pieces < 0 || (max_pieces > 0 && !pieces)) return chunks < 0 ? PASA_ERR_SHAPE : PASA_ERR_NULLPTR;
  const int rc = validate_shape(B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  const HostPlan hp = host_plan(B, Hq, Hkv, Sq, Sk, D, causal, mode, chunks);
  const int np = static_cast<int>(hp.pieces.size());
  for (int i = 0; i < np && i < max_pieces; ++i) {
    const HostPiece& pc = hp.pieces[i];
    int* r = pieces + 6 * static_cast<size_t>(i);
    r[0] = pc.u0, r[1] = pc.n, r[2] = pc.r0, r[3] = pc.r1, r[4] = pc.k0, r[5] = pc.k1;
  }
  return np;
}

extern "C" int pasa_attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                                  int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode, int chunks,
                                  void* device_buffer, size_t device_buffer_bytes, void* stream) {
  if (!q || !k || !v || !o) return PASA_ERR_NULLPTR;
  int rc = validate_shape(B, Hq, Hkv, Sq, Sk, D, mode);
  if (rc != PASA_OK) return rc;
  if (chunks < 0) return PASA_ERR_SHAPE;
  const HostPlan hp = host_plan(B, Hq, Hkv, Sq, Sk, D, causal, mode, chunks);
  if (device_buffer) {
    if (device_buffer_bytes < hp.total) return PASA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0) return PASA_ERR_ALIGN;
  }
  rc = check_device();
  if (rc != PASA_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStream_t side[3] = {};
  rc = side_streams(side);
  if (rc != PASA_OK) return rc;
  cudaStream_t s_in = side[0], s_out = side[1];
  cudaStream_t s_run[2] = {st, side[2]};  // piece i computes on s_run[i % 2]

  // events: [0] start on st, [1] h2d stream done, [2] d2h stream done, [3] second compute
  // stream done, [4 + i] piece i's inputs landed, [4 + np + i] piece i's kernels finished,
  // [4 + 2 np + i] a row piece's key blocks, and those of its unit's earlier pieces, prepared
  const int np = static_cast<int>(hp.pieces.size());
  std::vector<cudaEvent_t> ev(4 + 3 * static_cast<size_t>(np), nullptr);
  cudaError_t e = cudaSuccess;
  size_t made = 0;
  for (; made < ev.size(); ++made) {
    e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
    if (e != cudaSuccess) break;
  }
  uint8_t* buf = static_cast<uint8_t*>(device_buffer);
  bool owned = false;
  if (e == cudaSuccess && !buf) {
    e = cudaMallocAsync(reinterpret_cast<void**>(&buf), hp.total, st);
    owned = e == cudaSuccess;
  }
  if (e != cudaSuccess) {
    for (size_t j = 0; j < made; ++j) cudaEventDestroy(ev[j]);
    return cuda_fail(e);
  }

  // Everything below is enqueued on st, s_in or s_out; on the first failure the rest is
  // skipped, but the side streams are still joined back to st before the buffer is freed.
  auto step = [&](cudaError_t err) {
    if (e == cudaSuccess && err != cudaSuccess) e = err;
    return e == cudaSuccess;
  };
  const int g = Hq / Hkv;
  const size_t row_bytes = static_cast<size_t>(D) * 2;
  const size_t q_unit = static_cast<size_t>(g) * Sq * row_bytes;  // bytes of one unit's q (and o)
  const size_t kv_unit = static_cast<size_t>(Sk) * row_bytes;
  const size_t lse_unit = static_cast<size_t>(g) * Sq * 4;
  const uint8_t* qh = static_cast<const uint8_t*>(q);
  const uint8_t* kh = static_cast<const uint8_t*>(k);
  const uint8_t* vh = static_cast<const uint8_t*>(v);
  uint8_t* oh = static_cast<uint8_t*>(o);
  uint8_t* lh = reinterpret_cast<uint8_t*>(lse);

  // the buffer may still be in use by work the caller queued on st before this call
  step(cudaEventRecord(ev[0], st));
  step(cudaStreamWaitEvent(s_in, ev[0], 0));
  step(cudaStreamWaitEvent(s_out, ev[0], 0));
  step(cudaStreamWaitEvent(s_run[1], ev[0], 0));
  for (int i = 0; i < np && e == cudaSuccess; ++i) {
    const HostPiece& pc = hp.pieces[i];
    const size_t kv_bytes = align_up(static_cast<size_t>(pc.n) * kv_unit, 256);
    uint8_t* kd = buf + pc.kv_off;
    uint8_t* vd = kd + kv_bytes;
    // whole units: all their keys; a row piece: the keys [k0, k1) its rows newly see
    const size_t kb0 = static_cast<size_t>(pc.k0) * row_bytes;
    const size_t nb = pc.n == 1 ? static_cast<size_t>(pc.k1 - pc.k0) * row_bytes : pc.n * kv_unit;
    step(copy_rows(kd + kb0, nb, kh + pc.u0 * kv_unit + kb0, nb, nb, 1, cudaMemcpyHostToDevice, s_in));
    step(copy_rows(vd + kb0, nb, vh + pc.u0 * kv_unit + kb0, nb, nb, 1, cudaMemcpyHostToDevice, s_in));
    const size_t w = static_cast<size_t>(pc.r1 - pc.r0) * row_bytes;
    step(copy_rows(buf + pc.q_off, w, qh + pc.u0 * q_unit + pc.r0 * row_bytes, static_cast<size_t>(Sq) * row_bytes,
                   w, static_cast<size_t>(pc.n) * g, cudaMemcpyHostToDevice, s_in));
    step(cudaEventRecord(ev[4 + i], s_in));
  }
  const bool prep = shift_mode(mode) || fp8_mode(mode);
  const WorkspaceLayout pl = workspace_layout(1, 1, Sk, D, mode);   // a row-cut unit's prepared keys
  const int bn = pasa::block_rows_for(D);
  for (int i = 0; i < np && e == cudaSuccess; ++i) {
    const HostPiece& pc = hp.pieces[i];
    const size_t kv_bytes = align_up(static_cast<size_t>(pc.n) * kv_unit, 256);
    const int rows = pc.r1 - pc.r0;
    cudaStream_t run = s_run[i & 1];
    if (!step(cudaStreamWaitEvent(run, ev[4 + i], 0))) break;
    int krc = PASA_OK;
    if (pc.rowcut && prep) {
      // prepare this piece's new key blocks [k0, k1) into the unit's slot, then wait until
      // the unit's earlier pieces have prepared theirs (on either compute stream)
      uint8_t* pb = buf + pc.prep_off;
      float* kscale = fp8_mode(mode) ? reinterpret_cast<float*>(pb + pl.kscale_off) : nullptr;
      if (pc.k1 > pc.k0) krc = kshift_dispatch(buf + pc.kv_off, pb + pl.kshift_off, pb + pl.means_off, kscale, 1, 1,
                                               pc.k1, D, mode, run, pc.k0 / bn, Sk);
      if (krc == PASA_OK && i > 0 && hp.pieces[i - 1].rowcut && hp.pieces[i - 1].u0 == pc.u0)
        step(cudaStreamWaitEvent(run, ev[4 + 2 * np + i - 1], 0));
      step(cudaEventRecord(ev[4 + 2 * np + i], run));
      if (krc == PASA_OK && e == cudaSuccess)
        krc = attn_launch(buf + pc.q_off, pb + pl.kshift_off, pb + pl.means_off, buf + pc.kv_off + kv_bytes,
                          buf + pc.o_off, lse ? reinterpret_cast<float*>(buf + pc.lse_off) : nullptr, 1, g, 1, rows,
                          pc.k1, D, causal, scale, mode, run, nullptr, nullptr, kscale);
    } else {
      krc = pasa_attn_fwd_ws(buf + pc.q_off, buf + pc.kv_off, buf + pc.kv_off + kv_bytes, buf + pc.o_off,
                             lse ? reinterpret_cast<float*>(buf + pc.lse_off) : nullptr, pc.n, g, 1, rows, pc.k1, D,
                             causal, scale, mode, hp.ws_bytes ? buf + hp.ws_off + (i & 1) * hp.ws_bytes : nullptr,
                             hp.ws_bytes, run);
    }
    if (krc != PASA_OK) {
      rc = krc;
      break;
    }
    step(cudaEventRecord(ev[4 + np + i], run));
    step(cudaStreamWaitEvent(s_out, ev[4 + np + i], 0));
    const size_t w = static_cast<size_t>(rows) * row_bytes;
    const size_t h = static_cast<size_t>(pc.n) * g;
    step(copy_rows(oh + pc.u0 * q_unit + pc.r0 * row_bytes, static_cast<size_t>(Sq) * row_bytes, buf + pc.o_off, w,
                   w, h, cudaMemcpyDeviceToHost, s_out));
    if (lse)
      step(copy_rows(lh + pc.u0 * lse_unit + static_cast<size_t>(pc.r0) * 4, static_cast<size_t>(Sq) * 4,
                     buf + pc.lse_off, static_cast<size_t>(rows) * 4, static_cast<size_t>(rows) * 4, h,
                     cudaMemcpyDeviceToHost, s_out));
  }
  // join: st continues only after the side streams have drained this call's work
  cudaError_t je = cudaSuccess;
  for (int j = 0; j < 3 && je == cudaSuccess; ++j) {
    je = cudaEventRecord(ev[1 + j], side[j]);
    if (je == cudaSuccess) je = cudaStreamWaitEvent(st, ev[1 + j], 0);
  }
  if (je != cudaSuccess) {
    // st cannot be ordered after the side streams: wait for them here before freeing
    for (int j = 0; j < 3; ++j) cudaStreamSynchronize(side[j]);
    step(je);
  }
  if (owned) step(cudaFreeAsync(buf, st));
  for (cudaEvent_t x : ev) cudaEventDestroy(x);
  if (rc != PASA_OK) return rc;
  return e == cudaSuccess ? PASA_OK : cuda_fail(e);
}
