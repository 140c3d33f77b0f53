"""PASA attention forward for GB300 (sm_103a): Python binding of libpasa.so.

The binding only marshals arguments: it checks dtypes/devices, allocates outputs and the
workspace with PyTorch, and calls the C ABI (include/pasa.h) on the current CUDA stream.
Every step of the computation runs in the library's CUDA kernels. If libpasa.so is missing
the calls raise; there is no fallback.

Method: "Online Pseudo-average Shifting Attention (PASA) for Robust Low-precision LLM
Inference" (arXiv 2503.01873), Abstract.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "MODE_SHIFT_F16ACC", "MODE_SHIFT_F32ACC", "MODE_NAIVE_F16ACC", "MODE_NOSHIFT_F32ACC", "MODE_SHIFT_F16ALL", "MODE_SHIFT_FP8", "MODE_NAIVE_FP8", "kprep_fp8", "attn_fwd_fp8",
    "PasaError", "attn_fwd", "attn_fwd_alloc", "attn_fwd_fused", "attn_fwd_shifted", "attn_fwd_stats", "kshift", "workspace_bytes", "check_device_error", "block_rows",
    "library", "library_path",
]

MODE_SHIFT_F16ACC = 0
MODE_SHIFT_F32ACC = 1
MODE_NAIVE_F16ACC = 2
MODE_NOSHIFT_F32ACC = 3
MODE_SHIFT_F16ALL = 4   # mode 0 with an fp16 PV accumulator and an fp16 running row sum
MODE_SHIFT_FP8 = 5      # e4m3 Q and shifted keys, fp32 score accumulation (D = 128)
MODE_NAIVE_FP8 = 6      # e4m3 Q and raw keys, no shift (D = 128)
MEAN_GRID = 0           # block average rules for kshift
MEAN_PLAIN = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libpasa.so")
_lock = threading.Lock()
_lib = None

# exported symbols and their ctypes signatures, mirroring include/pasa.h
_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "pasa_block_rows": ([_I], _I),
    "pasa_attn_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "pasa_attn_fwd_noalloc": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "pasa_attn_fwd_fused": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _P, _P], _I),
    "pasa_attn_fwd_workspace_bytes": ([_I, _I, _I, _I, _I], _SZ),
    "pasa_attn_fwd_ws": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_stats": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_shifted": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "pasa_kshift": ([_P, _P, _P, _I, _I, _I, _I, _P], _I),
    "pasa_kshift_mean": ([_P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "pasa_kprep_fp8": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "pasa_attn_fwd_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "pasa_kshift_blocks": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "pasa_attn_fwd_decode_workspace_bytes": ([_I, _I, _I, _I, _I, _I, _I], _SZ),
    "pasa_attn_fwd_decode": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_decode_step": ([_P, _P, _P, _P, _P, _P, _P] + [_I] * 8 + [_F, _I, _I, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_decode_step_fp8": ([_P] * 8 + [_I] * 8 + [_F, _I, _I, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_decode_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P, _SZ, _P],
                                 _I),
    "pasa_kprep_fp8_blocks": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P], _I),
    "pasa_attn_fwd_host": ([_P, _P, _P, _P, _P] + [_I] * 7 + [_F, _I, _I, _P, _SZ, _P], _I),
    "pasa_attn_fwd_host_device_bytes": ([_I] * 9, _SZ),
    "pasa_attn_fwd_host_plan": ([_I] * 9 + [_P, _I], _I),
    "pasa_release_host_streams": ([], _I),
    "pasa_check_device_error": ([_P, ctypes.POINTER(ctypes.c_ulonglong)], _I),
    "pasa_selftest_wait_timeout": ([_P], _I),
    "pasa_selftest_exp2": ([_P, _P, _P, _I, _P], _I),
    "pasa_strerror": ([_I], ctypes.c_char_p),
    "pasa_last_cuda_error": ([], _I),
    "pasa_device_supported": ([_I], _I),
}


class PasaError(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = library()
        msg = lib.pasa_strerror(status).decode()
        if status == -5:
            msg += f" (cudaError {lib.pasa_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {status}]")
        self.status = status


def library():
    """Load libpasa.so (built by __graft_entry__.build()); raises if it is not there."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(f"{library_path} is missing: build it with "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(library_path)
            for name, (args, res) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(x: torch.Tensor, name: str):
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float16 or not x.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA fp16 tensor")


def block_rows(D: int) -> int:
    """Keys per pseudo-average block (and attention key tile) for head dim D."""
    return library().pasa_block_rows(D)


def workspace_bytes(B: int, Hkv: int, Sk: int, D: int, mode: int) -> int:
    return int(library().pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode))


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, mode: int = MODE_SHIFT_F16ACC,
             out=None, lse=None, return_lse: bool = True, workspace=None):
    """O, LSE of softmax(scale * Q K^T) V via libpasa (q [B,Hq,Sq,D], k/v [B,Hkv,Sk,D], fp16).

    Returns (o fp16 [B,Hq,Sq,D], lse fp32 [B,Hq,Sq] or None). ``mode`` is one of the MODE_*
    constants. The workspace (modes 0/1/4) is taken from PyTorch's allocator unless given.
    """
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(v, "v")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,D] and k, v [B,Hkv,Sk,D]")
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Sk, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("q and k disagree on B or D")
    if out is None:
        out = torch.empty_like(q)
    if return_lse and lse is None:
        lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    if not return_lse:
        lse = None
    nbytes = int(lib.pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode))
    if nbytes and workspace is None:
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_ws(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                              int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode),
                              _ptr(workspace) if nbytes else None,
                              workspace.numel() * workspace.element_size() if nbytes else 0, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_ws")
    return out, lse


def attn_fwd_fused(q, k, v, causal: bool = False, scale: float | None = None, mode: int = MODE_SHIFT_F16ACC,
                   out=None, lse=None, return_shift: bool = False):
    """Like attn_fwd, through pasa_attn_fwd_fused: the pseudo-average shift runs inside the
    attention kernel (one launch, no workspace; D = 128, modes 0, 1 and 4). With
    return_shift=True it also returns the shifted keys and block means the kernel computed:
    (o, lse, k_shifted, means)."""
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(v, "v")
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,Hq,Sq,D] and k, v [B,Hkv,Sk,D]")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    ks = means = None
    if return_shift:
        bn = block_rows(D)
        ks = torch.empty_like(k)
        means = torch.empty((B, Hkv, (Sk + bn - 1) // bn, D), device=k.device, dtype=torch.float16)
    rc = lib.pasa_attn_fwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                 int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode),
                                 _ptr(ks), _ptr(means), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_fused")
    return (out, lse, ks, means) if return_shift else (out, lse)


def attn_fwd_alloc(q, k, v, causal: bool = False, scale: float | None = None, mode: int = MODE_SHIFT_F16ACC,
                   out=None, lse=None):
    """Like attn_fwd, through pasa_attn_fwd (the library takes its own stream-ordered workspace)."""
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    rc = lib.pasa_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                           int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd")
    return out, lse


def _check_host(x: torch.Tensor, name: str, dtype=torch.float16):
    if not isinstance(x, torch.Tensor) or x.is_cuda or x.dtype != dtype or not x.is_contiguous():
        raise TypeError(f"{name} must be a contiguous host (CPU) {dtype} tensor")


def host_device_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, causal: bool, mode: int,
                      chunks: int = 0) -> int:
    return int(library().pasa_attn_fwd_host_device_bytes(B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), mode, chunks))


def host_plan(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, causal: bool, mode: int, chunks: int = 0):
    """The pieces attn_fwd_host runs: a list of (u0, n, r0, r1, k0, k1)."""
    lib = library()
    args = (B, Hq, Hkv, Sq, Sk, D, int(bool(causal)), int(mode), int(chunks))
    count = lib.pasa_attn_fwd_host_plan(*args, None, 0)
    if count < 0:
        raise PasaError(count, "pasa_attn_fwd_host_plan")
    rec = (ctypes.c_int * (6 * max(count, 1)))()
    lib.pasa_attn_fwd_host_plan(*args, ctypes.cast(rec, ctypes.c_void_p), count)
    return [tuple(rec[6 * i:6 * i + 6]) for i in range(count)]


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, mode: int = MODE_SHIFT_F16ACC,
                  out=None, lse=None, chunks: int = 0, device_buffer=None, sync: bool = True):
    """pasa_attn_fwd_host: q, k, v and the outputs are HOST fp16/fp32 tensors (pin them for
    the copies to overlap the kernels); the library stages them on the current device in
    pieces of (batch, kv head) units. With sync=False the call only enqueues on the current
    stream and out/lse are complete once that stream has been synchronized."""
    lib = library()
    _check_host(q, "q"), _check_host(k, "k"), _check_host(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float16, pin_memory=True)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, pin_memory=True)
    _check_host(out, "out"), _check_host(lse, "lse", torch.float32)
    nbytes = 0
    if device_buffer is not None:
        if not device_buffer.is_cuda or not device_buffer.is_contiguous():
            raise TypeError("device_buffer must be a contiguous CUDA tensor")
        nbytes = device_buffer.numel() * device_buffer.element_size()
    rc = lib.pasa_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D,
                                int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode),
                                int(chunks), _ptr(device_buffer), nbytes, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_host")
    if sync:
        torch.cuda.current_stream().synchronize()
    return out, lse


def release_host_streams() -> None:
    """pasa_release_host_streams: destroy the side streams attn_fwd_host created on the
    current device (recreated by the next attn_fwd_host call)."""
    rc = library().pasa_release_host_streams()
    if rc != 0:
        raise PasaError(rc, "pasa_release_host_streams")


def attn_fwd_stats(q, k, v, causal: bool = False, scale: float | None = None, mode: int = MODE_SHIFT_F16ACC,
                   block_stats: bool = False):
    """attn_fwd plus score magnitudes: returns (o, lse, stats [B,Hq,Sq,2] fp32), and with
    block_stats=True also the per-key-block maxima [B,Hq,ceil(Sk/128),2] fp32.

    [..., 0] = max |score held by the accumulator| (S' for modes 0/1/4, S for 2/3),
    [..., 1] = max |S' + q.m| (the recovered raw score; = [..., 0] for modes 2/3).
    """
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k.shape
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    stats = torch.empty((B, Hq, Sq, 2), device=q.device, dtype=torch.float32)
    nbt = -(-Sk // lib.pasa_block_rows(D))
    bstats = torch.empty((B, Hq, nbt, 2), device=q.device, dtype=torch.float32) if block_stats else None
    nbytes = int(lib.pasa_attn_fwd_workspace_bytes(B, Hkv, Sk, D, mode))
    ws = torch.empty(max(nbytes, 1), device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(stats),
                                 _ptr(bstats) if bstats is not None else None, B, Hq, Hkv, Sq, Sk,
                                 D, int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode),
                                 _ptr(ws) if nbytes else None, nbytes, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_stats")
    if bstats is not None:
        return out, lse, stats, bstats
    return out, lse, stats


def attn_fwd_shifted(q, k_shifted, means, v, causal: bool = False, scale: float | None = None,
                     mode: int = MODE_SHIFT_F16ACC, out=None, lse=None):
    """The attention kernel alone on keys from :func:`kshift` (modes 0/1/4) or raw keys (2/3)."""
    lib = library()
    _check(q, "q"), _check(k_shifted, "k_shifted"), _check(v, "v")
    if means is not None:
        _check(means, "means")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = k_shifted.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32)
    rc = lib.pasa_attn_fwd_shifted(_ptr(q), _ptr(k_shifted), _ptr(means), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                   Hkv, Sq, Sk, D, int(bool(causal)),
                                   float(scale) if scale is not None else 0.0, int(mode), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_shifted")
    return out, lse


def kshift(k, out=None, means=None, mean_rule: int = 0):
    """The pseudo-average shift step alone: returns (k_shifted [B,H,Sk,D], means [B,H,nb,D]).
    mean_rule: MEAN_GRID (0, the pseudo-average) or MEAN_PLAIN (1, the fp16-rounded mean)."""
    lib = library()
    _check(k, "k")
    B, H, Sk, D = k.shape
    bn = lib.pasa_block_rows(D)
    nb = (Sk + bn - 1) // bn
    ks = torch.empty_like(k) if out is None else out
    if means is None:
        means = torch.empty((B, H, nb, D), device=k.device, dtype=torch.float16)
    if mean_rule == MEAN_GRID:
        rc = lib.pasa_kshift(_ptr(k), _ptr(ks), _ptr(means), B, H, Sk, D, _stream())
    else:
        rc = lib.pasa_kshift_mean(_ptr(k), _ptr(ks), _ptr(means), B, H, Sk, D, int(mean_rule), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_kshift")
    return ks, means


def kprep_fp8(k, mode: int = MODE_SHIFT_FP8):
    """FP8 key preparation (D = 128): returns (k8 [B,H,Sk,D] uint8 e4m3 codes, means
    [B,H,nb,D] fp16 or None in mode 6, kscale [B,H,nb] fp32)."""
    lib = library()
    _check(k, "k")
    B, H, Sk, D = k.shape
    nb = -(-Sk // 128)
    k8 = torch.empty((B, H, Sk, D), device=k.device, dtype=torch.uint8)
    means = torch.empty((B, H, nb, D), device=k.device, dtype=torch.float16) if mode == MODE_SHIFT_FP8 else None
    kscale = torch.empty((B, H, nb), device=k.device, dtype=torch.float32)
    rc = lib.pasa_kprep_fp8(_ptr(k), _ptr(k8), _ptr(means) if means is not None else None, _ptr(kscale), B, H, Sk,
                            D, int(mode), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_kprep_fp8")
    return k8, means, kscale


def attn_fwd_fp8(q, k8, means, kscale, v, causal: bool = False, scale: float | None = None,
                 mode: int = MODE_SHIFT_FP8, out=None, lse=None):
    """The FP8 attention kernel alone on keys from :func:`kprep_fp8`: returns (o, lse)."""
    lib = library()
    _check(q, "q"), _check(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, Sk, _ = v.shape
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32) if lse is None else lse
    rc = lib.pasa_attn_fwd_fp8(_ptr(q), _ptr(k8), _ptr(means) if means is not None else None, _ptr(kscale), _ptr(v),
                               _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, D, int(bool(causal)),
                               float(scale) if scale is not None else 0.0, int(mode), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_fp8")
    return out, lse


def kshift_blocks(k, k_shifted, means, first_block: int, length: int | None = None):
    """Recompute :func:`kshift`'s output in place for key blocks first_block.. of a cache
    k [B,H,cap,D] holding `length` valid rows (default cap): the blocks an append touched;
    earlier blocks are left as they are."""
    lib = library()
    _check(k, "k"), _check(k_shifted, "k_shifted"), _check(means, "means")
    B, H, cap, D = k.shape
    Sk = cap if length is None else int(length)
    rc = lib.pasa_kshift_blocks(_ptr(k), _ptr(k_shifted), _ptr(means), B, H, Sk, cap, D, int(first_block),
                                _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_kshift_blocks")
    return k_shifted, means


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Sk: int, D: int, splits: int = 0) -> int:
    return library().pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, splits)


def attn_fwd_decode(q, k_shifted, means, v, causal: bool = False, scale: float | None = None,
                    mode: int = MODE_SHIFT_F16ACC, splits: int = 0, out=None, lse=None, workspace=None,
                    length: int | None = None):
    """Decode attention on a shifted key cache (modes 0/1/4) or raw keys (2/3): packed GQA
    rows, keys split across CTAs and merged. k_shifted / v are [B,Hkv,cap,D] caches with
    `length` valid rows (default cap). Returns (o, lse)."""
    lib = library()
    _check(q, "q"), _check(k_shifted, "k_shifted"), _check(v, "v")
    if means is not None:
        _check(means, "means")
    B, Hq, Sq, D = q.shape
    _, Hkv, cap, _ = k_shifted.shape
    Sk = cap if length is None else int(length)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32) if lse is None else lse
    nbytes = lib.pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(splits))
    if nbytes and (workspace is None or workspace.numel() * workspace.element_size() < nbytes):
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_decode(_ptr(q), _ptr(k_shifted), _ptr(means) if means is not None else None, _ptr(v),
                                  _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, cap, D, int(bool(causal)),
                                  float(scale) if scale is not None else 0.0, int(mode), int(splits),
                                  _ptr(workspace) if nbytes else None, nbytes, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_decode")
    return out, lse


def attn_fwd_decode_step(q, k, k_shifted, means, v, first_block: int, causal: bool = False,
                         scale: float | None = None, mode: int = MODE_SHIFT_F16ACC, splits: int = 0, out=None,
                         lse=None, workspace=None, length: int | None = None):
    """pasa_attn_fwd_decode_step: refresh key blocks first_block.. of the shifted cache
    (k_shifted, means) from the raw cache k, then decode on it, in one call (the decode kernel
    overlaps the refresh). Arguments as :func:`attn_fwd_decode` plus the raw cache k
    [B,Hkv,cap,D] and first_block. Returns (o, lse)."""
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(k_shifted, "k_shifted"), _check(v, "v")
    if means is not None:
        _check(means, "means")
    B, Hq, Sq, D = q.shape
    _, Hkv, cap, _ = k_shifted.shape
    Sk = cap if length is None else int(length)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32) if lse is None else lse
    nbytes = lib.pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(splits))
    if nbytes and (workspace is None or workspace.numel() * workspace.element_size() < nbytes):
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_decode_step(_ptr(q), _ptr(k), _ptr(k_shifted), _ptr(means) if means is not None else None,
                                       _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, cap, D, int(bool(causal)),
                                       float(scale) if scale is not None else 0.0, int(mode), int(first_block),
                                       int(splits), _ptr(workspace) if nbytes else None, nbytes, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_decode_step")
    return out, lse


def attn_fwd_decode_step_fp8(q, k, k8, means, kscale, v, first_block: int, causal: bool = False,
                             scale: float | None = None, mode: int = MODE_SHIFT_FP8, splits: int = 0, out=None,
                             lse=None, workspace=None, length: int | None = None):
    """pasa_attn_fwd_decode_step_fp8: refresh key blocks first_block.. of the e4m3 cache (k8,
    means, kscale) from the raw cache k, then decode on it, in one call. Returns (o, lse)."""
    lib = library()
    _check(q, "q"), _check(k, "k"), _check(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, cap, _ = k8.shape
    Sk = cap if length is None else int(length)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32) if lse is None else lse
    nbytes = lib.pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(splits))
    if nbytes and (workspace is None or workspace.numel() * workspace.element_size() < nbytes):
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_decode_step_fp8(_ptr(q), _ptr(k), _ptr(k8), _ptr(means) if means is not None else None,
                                           _ptr(kscale), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, cap, D,
                                           int(bool(causal)), float(scale) if scale is not None else 0.0, int(mode),
                                           int(first_block), int(splits), _ptr(workspace) if nbytes else None, nbytes,
                                           _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_decode_step_fp8")
    return out, lse


def kprep_fp8_blocks(k, k8, means, kscale, first_block: int, mode: int = MODE_SHIFT_FP8, length: int | None = None):
    """:func:`kprep_fp8` in place for key blocks first_block.. of a cache k [B,H,cap,D] holding
    `length` valid rows (default cap)."""
    lib = library()
    _check(k, "k")
    B, H, cap, D = k.shape
    Sk = cap if length is None else int(length)
    rc = lib.pasa_kprep_fp8_blocks(_ptr(k), _ptr(k8), _ptr(means) if means is not None else None, _ptr(kscale), B, H,
                                   Sk, cap, D, int(mode), int(first_block), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_kprep_fp8_blocks")
    return k8, means, kscale


def attn_fwd_decode_fp8(q, k8, means, kscale, v, causal: bool = False, scale: float | None = None,
                        mode: int = MODE_SHIFT_FP8, splits: int = 0, out=None, lse=None, workspace=None,
                        length: int | None = None):
    """Decode on an e4m3 key cache from :func:`kprep_fp8` (k8 [B,Hkv,cap,D] uint8, kscale
    [B,Hkv,ceil(cap/128)], means for mode 5) with `length` valid rows. Returns (o, lse)."""
    lib = library()
    _check(q, "q"), _check(v, "v")
    B, Hq, Sq, D = q.shape
    _, Hkv, cap, _ = v.shape
    Sk = cap if length is None else int(length)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, Hq, Sq), device=q.device, dtype=torch.float32) if lse is None else lse
    nbytes = lib.pasa_attn_fwd_decode_workspace_bytes(B, Hq, Hkv, Sq, Sk, D, int(splits))
    if nbytes and (workspace is None or workspace.numel() * workspace.element_size() < nbytes):
        workspace = torch.empty(nbytes, device=q.device, dtype=torch.uint8)
    rc = lib.pasa_attn_fwd_decode_fp8(_ptr(q), _ptr(k8), _ptr(means) if means is not None else None, _ptr(kscale),
                                      _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Sk, cap, D, int(bool(causal)),
                                      float(scale) if scale is not None else 0.0, int(mode), int(splits),
                                      _ptr(workspace) if nbytes else None, nbytes, _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_attn_fwd_decode_fp8")
    return out, lse


def selftest_wait_timeout():
    """Launch the failure-detection self-test on the current stream (pasa_selftest_wait_timeout):
    one CTA waits on a barrier nothing arrives on until the library's wait limit (2 s) and
    records a timeout in the device error word. check_device_error() then raises it."""
    rc = library().pasa_selftest_wait_timeout(_stream())
    if rc != 0:
        raise PasaError(rc, "pasa_selftest_wait_timeout")


def selftest_exp2(x):
    """(poly, mufu): the softmax's two exponentials 2^x of a CUDA fp32 tensor
    (pasa_selftest_exp2): the FMA-pipe polynomial and MUFU ex2.approx."""
    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32 or not x.is_contiguous():
        raise TypeError("x must be a contiguous CUDA fp32 tensor")
    poly = torch.empty_like(x)
    mufu = torch.empty_like(x)
    rc = library().pasa_selftest_exp2(_ptr(x), _ptr(poly), _ptr(mufu), x.numel(), _stream())
    if rc != 0:
        raise PasaError(rc, "pasa_selftest_exp2")
    return poly, mufu


def check_device_error():
    """Synchronise the current stream; raise PasaError if a kernel reported a timeout."""
    info = ctypes.c_ulonglong(0)
    rc = library().pasa_check_device_error(_stream(), ctypes.byref(info))
    if rc != 0:
        err = PasaError(rc, f"device (info {info.value:#x})")
        raise err
