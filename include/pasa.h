/*
 * pasa.h — C ABI of the PASA attention forward library (libpasa.so, sm_103a / GB300).
 *
 * PASA: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
 * Inference: Algorithms and Numerical Analysis" (arXiv 2503.01873), Abstract. A
 * FlashAttention forward pass in half precision in which each key block is shifted by its
 * pseudo-average along the sequence before the fp16 score GEMM ("online pseudo-average
 * shifting") and the per-row offsets q_i . m_j are added back in fp32 inside the online
 * softmax ("global recovering"). The result equals plain attention
 *     O = softmax(scale * Q K^T) V,   LSE_i = ln sum_j exp(scale * q_i . k_j)
 * up to rounding, while the fp16 scores stay far from the fp16 limit 65504.
 *
 * Conventions shared by every entry point:
 *   - Tensors are device pointers to contiguous row-major arrays, fp16 = IEEE binary16:
 *       q, o  [B, Hq,  Sq, D]      k, v  [B, Hkv, Sk, D]      lse [B, Hq, Sq] fp32
 *     Query head h reads key/value head h / (Hq / Hkv) (grouped-query attention).
 *   - Every device pointer must be 16-byte aligned (TMA), else PASA_ERR_ALIGN.
 *   - The caller owns all buffers; entry points never free or keep them.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is enqueued
 *     asynchronously: a PASA_OK return means "validated and launched", like a CUDA kernel
 *     launch. Argument errors are detected on the host before anything is enqueued.
 *   - Device-side failures (a pipeline wait that timed out) are latched in a device error
 *     word and reported by pasa_check_device_error(). No entry point reads that word by
 *     itself: the launch that timed out returned PASA_OK, and its outputs are invalid. A
 *     timeout ends only the CTA it happened in (each CTA of a broken launch gives up at its
 *     own 2 s limit); other launches run normally, whether or not the word has been read.
 *   - Supported: D in {64, 128}; B, Hq, Hkv, Sq, Sk >= 1; Hq % Hkv == 0; a GPU of compute
 *     capability 10.3 (sm_103a). Anything else returns an error and launches nothing.
 *   - Causal masking is bottom-right aligned: key j is visible to query i iff
 *     j <= i + Sk - Sq. A query row with no visible key gets O = 0 and LSE = -inf.
 */
#ifndef PASA_H_
#define PASA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (return values). */
#define PASA_OK 0
#define PASA_ERR_NULLPTR (-1)     /* a required pointer is NULL */
#define PASA_ERR_SHAPE (-2)       /* a size is <= 0, Hq % Hkv != 0, or a size overflows */
#define PASA_ERR_UNSUPPORTED (-3) /* D not in {64,128}, unknown mode, or not an sm_103 GPU */
#define PASA_ERR_ALIGN (-4)       /* a pointer is not 16-byte aligned */
#define PASA_ERR_CUDA (-5)        /* a CUDA runtime/driver call failed (see pasa_last_cuda_error) */
#define PASA_ERR_TIMEOUT (-6)     /* a device-side pipeline wait gave up (pasa_check_device_error) */
#define PASA_ERR_WORKSPACE (-7)   /* workspace NULL or smaller than pasa_attn_fwd_workspace_bytes */

/* Score modes (the `mode` argument). */
#define PASA_MODE_SHIFT_F16ACC 0   /* PASA: shifted keys, fp16-accumulated scores, fp32 offsets */
#define PASA_MODE_SHIFT_F32ACC 1   /* PASA shift with fp32-accumulated scores */
#define PASA_MODE_NAIVE_F16ACC 2   /* no shift, fp16-accumulated scores: shows the fp16 overflow */
#define PASA_MODE_NOSHIFT_F32ACC 3 /* no shift, fp32-accumulated scores: plain FlashAttention */
/* PASA with half precision throughout the loop ("Online Pseudo-average Shifting Attention
 * (PASA) for Robust Low-precision LLM Inference", Abstract: half-precision computation
 * throughout FlashAttention): mode 0, plus an fp16 PV accumulator and an fp16 running row
 * sum. The running max, the offsets and the final division stay fp32. */
#define PASA_MODE_SHIFT_F16ALL 4
/* FP8 scores (D = 128 only). Each query row of Q and each 128-key block of keys is quantised
 * to e4m3 (largest value 448) with one fp32 scale (row or block absolute maximum / 448);
 * the score GEMM takes e4m3 operands and accumulates in fp32; the rest is mode 1. Mode 5
 * quantises the shifted keys K' (PASA, offsets carried as in mode 1), mode 6 the raw keys
 * (no shift, the naive 8-bit kernel). Not available in pasa_attn_fwd_shifted or
 * pasa_attn_fwd_stats. */
#define PASA_MODE_SHIFT_FP8 5
#define PASA_MODE_NAIVE_FP8 6

/* Keys per block for head dim D: the block the pseudo-average is taken over, which is also
 * the attention kernel's key tile (128 for D = 64 and D = 128; 0 for other D). */
int pasa_block_rows(int D);

/*
 * PASA attention forward (the whole hot path: pseudo-average shift of K, then the fused
 * attention kernel). Abstract of the PASA paper: "online pseudo-average shifting" and
 * "global recovering" inside a FlashAttention forward pass.
 *
 *   q, k, v   fp16 inputs (layout above); o fp16 output [B, Hq, Sq, D].
 *   lse       fp32 output [B, Hq, Sq], natural-log sum of exp of the scaled scores; may
 *             be NULL to skip it.
 *   causal    0 or 1 (bottom-right aligned mask).
 *   scale     softmax scale; <= 0 selects 1/sqrt(D).
 *   mode      PASA_MODE_* above. Modes 0, 1, 4, 5 and 6 need a workspace for the shifted keys and
 *             block means: this entry point takes it from the CUDA stream-ordered allocator
 *             (cudaMallocAsync / cudaFreeAsync on `stream`); use pasa_attn_fwd_ws to pass
 *             your own.
 * Overflow in mode 2 is not an error: it shows up as inf/NaN in o, which is the point of
 * that mode.
 */
int pasa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                  int Sq, int Sk, int D, int causal, float scale, int mode, void* stream);

/*
 * PASA attention forward with the pseudo-average shift fused into the attention kernel
 * (Abstract of the PASA paper: "online pseudo-average shifting"): one launch, raw keys in,
 * no workspace. Each CTA reduces every raw key tile in shared memory as it lands (per
 * channel: the maximum |K|, its fp16 spacing g, the exact sum of rint_even(K / g)), shifts
 * the tile in place to K' = fp16_rn(K - m) with m = g * rint_even(sum / n), and computes
 * the fp32 offsets q_i . m_j itself; the rest is the pasa_attn_fwd kernel. K' and m are
 * those of pasa_kshift bit for bit. The offsets are summed in another order than the
 * pre-pass path's (on the CUDA cores instead of the tensor core), so o and lse agree with
 * pasa_attn_fwd to fp32 rounding, not bit for bit.
 *   - Arguments as in pasa_attn_fwd; D must be 128 and mode 0, 1 or 4, else
 *     PASA_ERR_UNSUPPORTED.
 *   - k_shifted_out [B, Hkv, Sk, D] and means_out [B, Hkv, ceil(Sk / 128), D], fp16 device
 *     buffers, may be NULL; when given, the kernel also writes the K' and m it computed
 *     there (every CTA of a kv head writes the same values), for checking.
 *   - Every CTA of a kv head repeats the shift of each key block it reads (ceil(Sq / 128)
 *     query tiles times Hq / Hkv heads), where pasa_attn_fwd shifts each block once in a
 *     separate kernel: this entry point trades that work for a launch and a workspace.
 */
int pasa_attn_fwd_fused(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                        int Sq, int Sk, int D, int causal, float scale, int mode, void* k_shifted_out,
                        void* means_out, void* stream);

/*
 * pasa_attn_fwd for callers that cannot allocate device memory. (The paper has no
 * counterpart: this is a library convenience.) Some callers may not call cudaMalloc at
 * all, for instance a process whose GPU memory is reserved up front by a framework or
 * serving allocator, or a latency-bound loop in which an allocation is not allowed. This
 * entry point allocates nothing: the shifted keys and block means go to one 64 MiB array
 * compiled into the library, which every GPU that loads the library holds until exit.
 *   - Arguments and results as in pasa_attn_fwd.
 *   - Returns PASA_ERR_WORKSPACE, and launches nothing, when the problem needs more than
 *     64 MiB of scratch, i.e. when pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode)
 *     exceeds 67108864 (modes 2 and 3 need none).
 *   - The first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current); make that first call before any
 *     stream capture.
 *   - All calls share the one array. Every call writes the part it reads before reading
 *     it, so nothing has to start at zero, but calls whose work overlaps on the GPU (other
 *     streams, other host threads) race on the array: order them, e.g. on one stream.
 */
int pasa_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                          int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode, void* stream);

/*
 * pasa_attn_fwd on HOST buffers: the PASA forward pass ("Online Pseudo-average Shifting
 * Attention (PASA) for Robust Low-precision LLM Inference", Abstract) computed exactly as
 * pasa_attn_fwd computes it, for inputs and outputs in host memory. (The paper has no
 * counterpart: this is a library convenience. It is the one entry point whose tensors are
 * host pointers.)
 *   q, k, v   HOST fp16 inputs in the layout above; o HOST fp16 [B, Hq, Sq, D]; lse HOST
 *             fp32 [B, Hq, Sq] or NULL. No alignment is required. For the copies to
 *             overlap with the kernels they must be page-locked (cudaHostAlloc /
 *             cudaHostRegister); pageable memory gives the same results, slower.
 *   chunks    0 = automatic, else the number of pieces the B * Hkv (batch, kv head) units
 *             are cut into, clamped to [1, min(B * Hkv, 64)]; negative is an error. The
 *             automatic plan takes the largest count <= min(B * Hkv, 8) that leaves every
 *             piece at least 256 query tiles of 128 rows, and also cuts the first and the
 *             last unit along the query rows into pieces that halve towards the ends
 *             (Sq/2, Sq/4, Sq/8 rows; the smallest keeps >= 128 query tiles), so that
 *             little of the copying waits on, or is waited on by, the kernels. Row pieces
 *             start on 128-row tiles and, under the causal mask, see a key prefix ending
 *             on a 128-key block; they are used only where that holds (not causal, or
 *             Sk >= Sq with Sk - Sq a multiple of 128).
 *   device_buffer, device_buffer_bytes
 *             device memory of at least pasa_attn_fwd_host_device_bytes(...) bytes, 256-byte
 *             aligned: it stages the whole problem (q, k, v, o, lse), the prepared
 *             keys of each unit cut into query-row pieces (each piece prepares only the
 *             key blocks it newly sees) and two shift workspaces for the other pieces,
 *             one per compute stream. Its contents on entry do not matter.
 *             NULL: the call takes it from the stream-ordered allocator on `stream` and
 *             frees it there.
 *   stream    the stream the kernels run on. The call only enqueues: o and lse hold the
 *             result once `stream` has reached the end of this call's work (synchronize
 *             it, or record an event after the call). Work queued on `stream` earlier is
 *             finished before any copy of this call starts.
 * Per piece: its q, k and v go host->device on a side stream; its shift and attention
 * kernels run once they have landed, pieces alternating between `stream` and a second
 * compute stream so that one piece's last tiles overlap the next piece's first; its o and
 * lse go device->host on another side stream once the kernels are done. A piece is a
 * problem of n (batch, kv head) units with one kv head, or query rows [r0, r1) of one unit
 * with the keys they see, and every query tile meets the same key blocks and
 * pseudo-averages as in one call: the results are bit-identical to pasa_attn_fwd on the
 * same inputs. The three side streams are non-blocking streams the library creates on
 * first use per device and keeps until pasa_release_host_streams. Errors: as
 * pasa_attn_fwd (shapes and mode), PASA_ERR_WORKSPACE when the buffer is too small,
 * PASA_ERR_ALIGN when it is not 256-byte aligned; a failure after enqueueing began still
 * orders `stream` after all work already queued.
 */
int pasa_attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                       int Sq, int Sk, int D, int causal, float scale, int mode, int chunks, void* device_buffer,
                       size_t device_buffer_bytes, void* stream);

/* Destroys the three side streams pasa_attn_fwd_host created on the current device, after
 * synchronizing each, so that the library holds no CUDA object of its own there; the next
 * pasa_attn_fwd_host call on the device creates them again. The library has no counterpart
 * in the paper: this is resource management of the host-buffer entry point. Call it only
 * while no other host thread is inside pasa_attn_fwd_host on the same device (their calls
 * would enqueue on a stream being destroyed). Returns PASA_OK (also when there was nothing
 * to release) or PASA_ERR_CUDA (pasa_last_cuda_error gives the cudaError_t); the handles
 * are dropped either way. */
int pasa_release_host_streams(void);

/* The pieces pasa_attn_fwd_host runs for these arguments, in order: writes min(count,
 * max_pieces) records of six ints (u0, n, r0, r1, k0, k1) to `pieces` (host memory) and
 * returns the count, or a negative status (argument errors as pasa_attn_fwd_host; NULL
 * pieces with max_pieces > 0 is PASA_ERR_NULLPTR). A record stands for query rows [r0, r1)
 * of the units [u0, u0 + n) attending keys [0, k1); its copy-in adds keys [k0, k1). */
int pasa_attn_fwd_host_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, int mode, int chunks,
                            int* pieces, int max_pieces);

/* Device bytes pasa_attn_fwd_host needs for these sizes, masking, mode and chunk request (0
 * when the arguments are invalid). */
size_t pasa_attn_fwd_host_device_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, int mode,
                                       int chunks);

/* Workspace bytes pasa_attn_fwd_ws needs for these sizes and mode (0 for modes 2 and 3, and
 * for the FP8 modes with D != 128). */
size_t pasa_attn_fwd_workspace_bytes(int B, int Hkv, int Sk, int D, int mode);

/*
 * Same as pasa_attn_fwd with a caller-owned device workspace of at least
 * pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode) bytes, 256-byte aligned. Its
 * contents on entry do not matter; it must not be used by other work until the stream
 * has passed this call.
 */
int pasa_attn_fwd_ws(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                     int Sq, int Sk, int D, int causal, float scale, int mode, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * pasa_attn_fwd_ws plus an overflow diagnostic. The Abstract traces fp16 overflow (> 65504)
 * in attention scores to a large sequence-dimension bias of K and to Q/K resonance; this
 * call reports, for every query row, what the score accumulator actually held:
 *   stats[b, h, i, 0] = max over visible keys of |accumulated score|: the shifted score
 *                       S' = q_i . k'_j for modes 0/1/4, the raw score q_i . k_j for modes
 *                       2/3; in the fp16-accumulate modes this is the fp16 value (inf if the
 *                       accumulator overflowed);
 *   stats[b, h, i, 1] = max over visible keys of |S' + q_i . m_j|, the recovered raw score
 *                       (modes 0/1/4; equal to [0] for modes 2/3).
 * stats is fp32 [B, Hq, Sq, 2], 8-byte aligned; rows with no visible key get 0.
 * block_stats, if not NULL, is fp32 [B, Hq, ceil(Sk / pasa_block_rows(D)), 2], 8-byte
 * aligned, and gets the same two magnitudes per key block, as the max over all query rows
 * that see the block (0 for a block no row sees). Their ratio tells the Abstract's two
 * causes apart: a sequence-dimension bias of K is removed by the shift ([0] << [1] in the
 * PASA modes), Q/K resonance within a block is not ([0] close to [1]). The call zeroes
 * block_stats on the stream before the kernel. o and lse are written as in
 * pasa_attn_fwd_ws. Runs a separately compiled variant of the attention kernel that also
 * tracks the per-block minimum score.
 */
int pasa_attn_fwd_stats(const void* q, const void* k, const void* v, void* o, float* lse, float* stats,
                        float* block_stats, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                        int mode, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The attention kernel alone, on keys already shifted by pasa_kshift (for modes 0, 1 and 4:
 * k_shifted and means exactly as pasa_kshift wrote them for the same k) or on raw keys
 * (modes 2 and 3: pass k as k_shifted; means is ignored and may be NULL). This is the
 * second half of pasa_attn_fwd; callers that keep shifted keys (a KV cache) skip the shift.
 * Arguments as in pasa_attn_fwd; means is fp16 [B, Hkv, ceil(Sk / pasa_block_rows(D)), D].
 */
int pasa_attn_fwd_shifted(const void* q, const void* k_shifted, const void* means, const void* v, void* o,
                          float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale,
                          int mode, void* stream);

/*
 * The pseudo-average shift step alone (PASA Abstract, "online pseudo-average shifting"),
 * exposed for testing and diagnostics. For every key block j of pasa_block_rows(D) rows
 * (the last block may be shorter) and channel d it writes
 *     means[b, h, j, d]   the block's pseudo-average m_j[d] (fp16)
 *     k_shifted[b, h, r, d] = fp16_rn(k[b, h, r, d] - m_j[d])
 * where m_j[d] = g * round_half_even(sum_r round_half_even(k[r,d] / g) / n), g the fp16
 * spacing at max_r |k[r,d]| and n the block's row count; m_j[d] = 0 when that maximum is
 * >= 32768 or the block/channel holds inf or NaN.
 *   k          fp16 [B, H, Sk, D]        k_shifted  fp16 [B, H, Sk, D]
 *   means      fp16 [B, H, ceil(Sk / pasa_block_rows(D)), D]
 */
int pasa_kshift(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int D, void* stream);

/* Rules for the block average (the `mean_rule` argument of pasa_kshift_mean). */
#define PASA_MEAN_GRID 0   /* the pseudo-average of pasa_kshift (the library's reading) */
#define PASA_MEAN_PLAIN 1  /* the exact block mean rounded once to fp16 (ties to even) */

/*
 * pasa_kshift with a choice of the Abstract's undefined "pseudo-average". PASA_MEAN_GRID
 * is pasa_kshift itself. PASA_MEAN_PLAIN writes m_j[d] = fp16_rn(sum_r k[r,d] / n), the
 * plain fp16-rounded mean of the block's n valid rows, with the same guard (m = 0 when
 * max |k| >= 32768 or the block/channel holds inf or NaN) and the same shift
 * k_shifted = fp16_rn(k - m). Both keep attention exact up to rounding, since the offsets
 * q . m_j are added back; they differ in how often k - m is exact in fp16 (the grid reading
 * keeps it exact far more often when the mean is small against the block maximum). The
 * output feeds pasa_attn_fwd_shifted / pasa_attn_fwd_decode unchanged. Other arguments and
 * errors as pasa_kshift; an unknown rule is PASA_ERR_UNSUPPORTED.
 */
int pasa_kshift_mean(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int D, int mean_rule,
                     void* stream);

/*
 * Key preparation of the FP8 score modes (D = 128): per key block j of 128 rows, with
 * a = max |x| over the block (all channels) of x = K' (mode 5, PASA_MODE_SHIFT_FP8: the
 * shifted keys exactly as pasa_kshift rounds them to fp16) or x = K (mode 6,
 * PASA_MODE_NAIVE_FP8), it writes
 *     kscale[b, h, j]      = fp32(a / 448)        (1 when a = 0)
 *     k8[b, h, r, d]       = e4m3 code of fp32(x[r, d] * fp32(448 / a)), round to nearest
 *                            even, saturating at 448 (one byte, the OCP e4m3 encoding)
 *     means[b, h, j, d]    = the pseudo-average m_j[d] as in pasa_kshift (mode 5 only; may
 *                            be NULL in mode 6)
 * 448 is the largest finite e4m3 value: the Abstract's overflow concern at 8 bits, where
 * a sequence-dimension bias of K spends the 3-bit mantissa on the bias instead of the part
 * of K that varies. Layouts: k fp16 [B, H, Sk, D]; k8 bytes [B, H, Sk, D]; kscale fp32
 * [B, H, ceil(Sk / 128)]; means fp16 [B, H, ceil(Sk / 128), D]; all 16-byte aligned. The
 * results can be kept as an FP8 key cache for pasa_attn_fwd_fp8. Returns
 * PASA_ERR_UNSUPPORTED for other modes or D != 128.
 */
int pasa_kprep_fp8(const void* k, void* k8, void* means, float* kscale, int B, int H, int Sk, int D, int mode,
                   void* stream);

/*
 * The attention kernel of the FP8 modes alone, on keys from pasa_kprep_fp8 (same mode).
 * Q is quantised inside the kernel, per query row r: sq = fp32(a / 448) with a = max |q_r|,
 * codes e4m3(fp32(q * fp32(448 / a))); the score GEMM multiplies e4m3 codes and accumulates
 * in fp32, and the scores are sq * kscale_j * (codes product) (+ q . m_j in mode 5). Other
 * arguments and errors as pasa_attn_fwd_shifted; means may be NULL in mode 6.
 */
int pasa_attn_fwd_fp8(const void* q, const void* k8, const void* means, const float* kscale, const void* v, void* o,
                      float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int D, int causal, float scale, int mode,
                      void* stream);

/*
 * Refresh of a shifted key cache after an append ("Online Pseudo-average Shifting Attention
 * (PASA) for Robust Low-precision LLM Inference", Abstract: long-sequence inference). The
 * pseudo-average of a key block depends on that block's rows only, so when rows are
 * appended to a cache of Sk keys, only the blocks from first_block on change. This call
 * recomputes exactly pasa_kshift's output for key blocks [first_block, ceil(Sk / BN)), BN =
 * pasa_block_rows(D), and leaves every earlier block of k_shifted and means untouched.
 * The cache holds Sk valid keys of Sk_cap allocated rows per head (Sk_cap >= Sk; pass Sk
 * for a dense tensor): k and k_shifted fp16 [B, H, Sk_cap, D], means fp16 [B, H,
 * ceil(Sk_cap / BN), D]; rows and blocks past Sk are neither read nor written. Other
 * arguments as pasa_kshift; first_block outside [0, ceil(Sk / BN)), Sk_cap < Sk or
 * B * H > 65535 is PASA_ERR_SHAPE.
 */
int pasa_kshift_blocks(const void* k, void* k_shifted, void* means, int B, int H, int Sk, int Sk_cap, int D,
                       int first_block, void* stream);

/*
 * Bytes of workspace pasa_attn_fwd_decode(_fp8) needs for these sizes and `splits` (0 =
 * the automatic choice): 0 when the call runs unsplit or merges its splits inside a
 * thread-block cluster (D = 128, g * Sq <= 32, 2 to 8 splits), else splits * B * Hq * Sq *
 * (D + 1) fp32 values (partial outputs and log-sum-exps, each part 256-byte aligned).
 * Returns 0 for invalid sizes as well.
 */
size_t pasa_attn_fwd_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int D, int splits);

/*
 * Decode attention on a key cache (the inference use of PASA, same citation as
 * pasa_kshift_blocks): a few new query rows per head against Sk cached keys, already
 * shifted by pasa_kshift / pasa_kshift_blocks (modes 0, 1, 4) or raw (modes 2, 3; means may
 * be NULL; FP8 caches: pasa_attn_fwd_decode_fp8). The result equals pasa_attn_fwd_shifted's
 * on the same arguments up to the
 * rounding: the split merge, and in the decode kernel the order of the row sums and the
 * offsets (fp32 dot products on the CUDA cores instead of the tensor cores).
 * Two changes of work layout serve the small Sq:
 *  - the g = Hq / Hkv query heads sharing a kv head are packed into rows = g * Sq query
 *    rows (requires rows <= 128, else PASA_ERR_UNSUPPORTED), so each key block is read
 *    once per kv head instead of once per query head. With D = 128 and rows <= 32 a
 *    decode kernel puts the 128 keys of a block on the MMA's M side and the packed rows
 *    (padded to 16 or 32) on its N side; otherwise the attention kernel runs on the
 *    packed rows as one 128-row tile;
 *  - the key blocks are split across `splits` CTAs per kv head (0 = automatic: at most one
 *    CTA per SM, at least eight key blocks per split), merged by their log-sum-exps:
 *    O = sum_s w_s O_s / sum_s w_s, w_s = 2^(lse_s - max lse). On the swapped-operand
 *    kernel with up to 8 splits the splits of a kv head run as one thread-block cluster and
 *    merge through distributed shared memory (no workspace); otherwise each split writes
 *    its O / l (fp32) and m + log2 l to the workspace and a second kernel merges them.
 * The causal mask is bottom-right aligned per head, as in pasa_attn_fwd. q, o: fp16
 * [B, Hq, Sq, D]; the cache holds Sk valid keys of Sk_cap allocated rows per head
 * (Sk_cap >= Sk, else PASA_ERR_SHAPE; pass Sk for dense tensors): k_shifted, v fp16
 * [B, Hkv, Sk_cap, D], means fp16 [B, Hkv, ceil(Sk_cap / pasa_block_rows(D)), D]; rows
 * past Sk are not read. lse: fp32 [B, Hq, Sq] or NULL. workspace: device,
 * 256-byte aligned, at least pasa_attn_fwd_decode_workspace_bytes(...) bytes (may be NULL
 * when that is 0); the caller owns it and it is only used on `stream`. FP8 modes and
 * splits < 0 are PASA_ERR_UNSUPPORTED; a short workspace is PASA_ERR_WORKSPACE.
 */
int pasa_attn_fwd_decode(const void* q, const void* k_shifted, const void* means, const void* v, void* o, float* lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal, float scale, int mode,
                         int splits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One decode step on a shifted fp16 key cache: the refresh of pasa_kshift_blocks(k,
 * k_shifted, means, B, Hkv, Sk, Sk_cap, D, first_block) followed by pasa_attn_fwd_decode on
 * the refreshed cache, in one call (same citation as pasa_kshift_blocks; the library's
 * pairing of the two has no counterpart in the paper). Results are bit-identical to the two
 * calls in sequence. The difference is scheduling: the decode kernel is launched with
 * programmatic dependence on the refresh, starts while the refresh still runs, and waits
 * for it (griddepcontrol.wait) only before it reads key blocks first_block and later (their
 * K', means and scales), which every split reaches last, so the refresh is hidden. The
 * decode kernels that do not take this schedule (more than 32 packed rows, or D = 64) run
 * after the refresh in stream order.
 *   k          the raw fp16 key cache [B, Hkv, Sk_cap, D] the refresh reads
 *   k_shifted, means   the shifted cache and its block means, rewritten from first_block on
 *   other arguments as pasa_attn_fwd_decode; modes 2 and 3 (no shifted cache) only run
 *   the decode, and the FP8 modes are PASA_ERR_UNSUPPORTED (pasa_attn_fwd_decode_step_fp8
 *   covers them). Errors: as the two calls; all arguments are
 *   checked before anything is enqueued.
 */
int pasa_attn_fwd_decode_step(const void* q, const void* k, void* k_shifted, void* means, const void* v, void* o,
                              float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal,
                              float scale, int mode, int first_block, int splits, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Decode on an FP8 key cache (modes 5 and 6; the FP8 score modes of pasa_attn_fwd_fp8 on
 * the decode work layout of pasa_attn_fwd_decode). The cache holds e4m3 codes k8 [B, Hkv,
 * Sk_cap, D] uint8 with one fp32 scale per 128-key block, kscale [B, Hkv,
 * ceil(Sk_cap / 128)], as pasa_kprep_fp8 / pasa_kprep_fp8_blocks write them, plus (mode 5)
 * the block means [B, Hkv, ceil(Sk_cap / 128), D] fp16; v fp16 [B, Hkv, Sk_cap, D]. The new
 * query rows are quantised in the kernel exactly as in pasa_attn_fwd_fp8 (one scale per
 * row). Only the swapped-operand decode kernel takes e4m3 keys: D = 128 and g * Sq <= 32,
 * else PASA_ERR_UNSUPPORTED; kscale NULL is PASA_ERR_NULLPTR. Workspace, splits, causal
 * mask and other arguments as pasa_attn_fwd_decode (pasa_attn_fwd_decode_workspace_bytes
 * applies unchanged).
 */
int pasa_attn_fwd_decode_fp8(const void* q, const void* k8, const void* means, const float* kscale, const void* v,
                             void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D, int causal,
                             float scale, int mode, int splits, void* workspace, size_t workspace_bytes, void* stream);

/* One decode step on an e4m3 key cache: pasa_kprep_fp8_blocks(k, k8, means, kscale, B, Hkv,
 * Sk, Sk_cap, D, mode, first_block) followed by pasa_attn_fwd_decode_fp8 on the refreshed
 * cache, in one call, with the schedule of pasa_attn_fwd_decode_step (the decode kernel
 * overlaps the refresh and waits for it only before the refreshed blocks, their codes,
 * means and scales). Bit-identical to the two calls. Modes 5 and 6 only (other modes:
 * PASA_ERR_UNSUPPORTED); D = 128 with at most 32 packed rows, as pasa_attn_fwd_decode_fp8.
 * Errors: as the two calls, all checked before anything is enqueued. */
int pasa_attn_fwd_decode_step_fp8(const void* q, const void* k, void* k8, void* means, float* kscale, const void* v,
                                  void* o, float* lse, int B, int Hq, int Hkv, int Sq, int Sk, int Sk_cap, int D,
                                  int causal, float scale, int mode, int first_block, int splits, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * pasa_kprep_fp8 for key blocks [first_block, ceil(Sk / 128)) of a cache of Sk valid keys in
 * Sk_cap allocated rows per head (the FP8 counterpart of pasa_kshift_blocks): after an
 * append only the blocks it wrote into change. k fp16 [B, H, Sk_cap, D]; k8 uint8 [B, H,
 * Sk_cap, D]; kscale fp32 [B, H, ceil(Sk_cap / 128)]; means (mode 5) fp16 [B, H,
 * ceil(Sk_cap / 128), D]. Earlier blocks and rows past Sk are left untouched. Errors as
 * pasa_kprep_fp8, plus PASA_ERR_SHAPE for first_block outside [0, ceil(Sk / 128)) or
 * Sk_cap < Sk.
 */
int pasa_kprep_fp8_blocks(const void* k, void* k8, void* means, float* kscale, int B, int H, int Sk, int Sk_cap, int D,
                          int mode, int first_block, void* stream);

/*
 * Synchronise `stream` and read the device error word. Returns PASA_OK, PASA_ERR_TIMEOUT
 * (a pipeline wait gave up; `info`, if not NULL, receives the CTA index << 32 | wait site)
 * or PASA_ERR_CUDA. Reading the word clears it.
 */
int pasa_check_device_error(void* stream, unsigned long long* info);

/* Human-readable text for a status code (static storage). */
const char* pasa_strerror(int status);

/* The cudaError_t of the most recent failed CUDA call in this thread (0 if none). */
int pasa_last_cuda_error(void);

/* 1 if `device` can run this library (compute capability 10.3), else 0. */
int pasa_device_supported(int device);

/*
 * Exercises the failure-detection path without a fault. (The paper has no counterpart: this
 * is a library test hook.) It launches one CTA whose thread 0 waits, through the same
 * bounded mbarrier wait every kernel of the library uses, on a barrier that nothing arrives
 * on. After the library's wait limit (2 s of %globaltimer) the wait gives up and records a
 * timeout in the device error word, with site tag 0x5E1F7E57 as the low 32 bits of the
 * info word, and the kernel returns. It holds no TMA copy and no tensor memory, so the GPU
 * context stays usable: pasa_check_device_error(stream, &info) then returns
 * PASA_ERR_TIMEOUT with that tag and clears the word. If the word already holds an unread
 * error, the wait still runs to its limit and the word keeps the first error's info.
 *   stream  where the CTA runs. Returns PASA_OK once launched; errors as for every entry
 *           point (no supported device: PASA_ERR_UNSUPPORTED; a failed launch:
 *           PASA_ERR_CUDA).
 */
int pasa_selftest_wait_timeout(void* stream);

/*
 * Evaluates the two exponentials the attention kernels' softmax uses, for testing. (The paper
 * has no counterpart: the softmax's exp2 is an implementation detail of this library.) For
 * each of the n fp32 values x[i] (device pointers, n >= 1):
 *   poly[i] = 2^x[i] on the FMA pipe: Cody-Waite split x = rint(x) + f, f in [-1/2, 1/2],
 *             a cubic fitted to 2^f (max relative error 7.5e-5) times 2^rint(x) built in the
 *             exponent field; x <= -126 (or -inf) gives a value in [0, 2^-125]; NaN gives
 *             NaN; x must be <= 127 (+inf gives NaN).
 *   mufu[i] = ex2.approx.ftz.f32 of x[i] (the MUFU exponential).
 * The kernels compute a fixed share of each key block's probabilities with the first and
 * the rest with the second. Errors: PASA_ERR_NULLPTR, PASA_ERR_SHAPE (n <= 0),
 * PASA_ERR_UNSUPPORTED (device), PASA_ERR_CUDA (launch). Asynchronous on `stream`.
 */
int pasa_selftest_exp2(const float* x, float* poly, float* mufu, int n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PASA_H_ */
