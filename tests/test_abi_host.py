"""Host-only checks of the C ABI: the library builds, loads and exports every function
include/pasa.h declares, and argument errors are reported before any launch.

Every call below is rejected by host-side validation, so none reaches a CUDA launch
(the pointers passed are never dereferenced).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from precision_flashattention_numerics_gb300 import build

    build.build()
    import precision_flashattention_numerics_gb300 as pasa

    return pasa.library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "pasa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pasa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    import precision_flashattention_numerics_gb300 as pasa

    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in pasa.SIGNATURES, f"binding has no signature for {n}"


def test_block_rows_and_strings(lib):
    # the key tile (and shift block): 128 keys for both supported head dims
    assert lib.pasa_block_rows(64) == 128
    assert lib.pasa_block_rows(128) == 128
    assert lib.pasa_block_rows(96) == 0
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.pasa_strerror(code)
    assert lib.pasa_strerror(12345) == b"unknown status"


FAKE = 1 << 20          # 16-byte aligned, never dereferenced
FAKE_MIS = FAKE + 8     # misaligned


def call(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Sq=64, Sk=64, D=64,
         causal=0, scale=0.0, mode=3, ws=None, ws_bytes=0):
    P = ctypes.c_void_p
    return lib.pasa_attn_fwd_ws(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, Sq, Sk, D, causal, scale, mode,
                                P(ws) if ws is not None else None, ws_bytes, None)


def test_argument_errors(lib):
    assert call(lib, q=0) == -1
    assert call(lib, o=0) == -1
    assert call(lib, B=0) == -2
    assert call(lib, Sk=-3) == -2
    assert call(lib, Hq=3, Hkv=2) == -2
    assert call(lib, D=96) == -3
    assert call(lib, D=256) == -3
    assert call(lib, mode=7) == -3
    assert call(lib, mode=-1) == -3
    assert call(lib, mode=5, D=64) == -3               # FP8 score modes: D = 128 only
    assert call(lib, mode=6, D=128, ws=None) == -7     # they prepare e4m3 keys in the workspace
    assert call(lib, mode=4, ws=None) == -7          # mode 4 shifts the keys: it needs the workspace
    assert call(lib, k=FAKE_MIS) == -4
    assert call(lib, lse=FAKE_MIS) == -4
    # modes with the shift need a workspace of the advertised size
    assert call(lib, mode=0, ws=None) == -7
    need = lib.pasa_attn_fwd_workspace_bytes(1, 1, 64, 64, 0)
    assert call(lib, mode=1, ws=FAKE, ws_bytes=need - 1) == -7
    assert call(lib, mode=1, ws=FAKE + 16, ws_bytes=need) == -4   # workspace must be 256-byte aligned
    # grid overflow is a shape error
    assert call(lib, B=65536, Hq=65536, Hkv=1, Sq=1 << 20) == -2


def test_kshift_argument_errors(lib):
    P = ctypes.c_void_p
    # pasa_kshift_mean(k, k_shifted, means, B, H, Sk, D, mean_rule, stream)
    assert lib.pasa_kshift_mean(P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 64, 2, None) == -3
    assert lib.pasa_kshift_mean(P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 64, -1, None) == -3
    assert lib.pasa_kshift_mean(None, P(FAKE), P(FAKE), 1, 1, 64, 64, 1, None) == -1
    assert lib.pasa_kshift_mean(P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 96, 1, None) == -3
    assert lib.pasa_kshift_mean(P(FAKE_MIS), P(FAKE), P(FAKE), 1, 1, 64, 64, 1, None) == -4
    assert lib.pasa_kshift_mean(P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 64, 0, None) == lib.pasa_kshift(
        P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 64, None)   # rule 0 is pasa_kshift (no device here)
    assert lib.pasa_kshift(None, P(FAKE), P(FAKE), 1, 1, 64, 64, None) == -1
    assert lib.pasa_kshift(P(FAKE), P(FAKE), P(FAKE), 1, 1, 0, 64, None) == -2
    assert lib.pasa_kshift(P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 32, None) == -3
    assert lib.pasa_kshift(P(FAKE_MIS), P(FAKE), P(FAKE), 1, 1, 64, 64, None) == -4


def test_workspace_bytes(lib):
    # shifted keys [B,Hkv,Sk,D] fp16 + means [B,Hkv,ceil(Sk/128),D] fp16, each 256-aligned
    def expect(B, H, Sk, D):
        a = -(-(B * H * Sk * D * 2) // 256) * 256
        nb = -(-Sk // 128)
        return -(-(a + B * H * nb * D * 2) // 256) * 256

    for (B, H, Sk, D) in [(1, 4, 4096, 128), (2, 5, 9216, 64), (1, 1, 1, 64), (4, 8, 8192, 128)]:
        for mode in (0, 1, 4):
            assert lib.pasa_attn_fwd_workspace_bytes(B, H, Sk, D, mode) == expect(B, H, Sk, D)
        for mode in (2, 3):
            assert lib.pasa_attn_fwd_workspace_bytes(B, H, Sk, D, mode) == 0
        # FP8 modes (D = 128): e4m3 keys [B,H,Sk,D] bytes + means fp16 + block scales fp32
        nb = -(-Sk // 128)
        fp8 = (-(-(-(-(-(-(B * H * Sk * D) // 256) * 256 + B * H * nb * D * 2) // 256) * 256 + B * H * nb * 4) // 256)
               * 256)
        for mode in (5, 6):
            assert lib.pasa_attn_fwd_workspace_bytes(B, H, Sk, D, mode) == (fp8 if D == 128 else 0)


def test_no_device_here_is_reported_not_launched(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.pasa_device_supported(0) == 0
    # the failure-detection self-test launches nothing without a supported device
    assert lib.pasa_selftest_wait_timeout(None) in (-3, -5)


def test_fp8_entry_points_check_arguments(lib):
    P = ctypes.c_void_p
    # pasa_kprep_fp8(k, k8, means, kscale, B, H, Sk, D, mode, stream)
    assert lib.pasa_kprep_fp8(P(FAKE), P(FAKE), None, P(FAKE), 1, 1, 64, 128, 5, None) == -1   # mode 5 needs means
    assert lib.pasa_kprep_fp8(P(FAKE), P(FAKE), None, None, 1, 1, 64, 128, 6, None) == -1
    assert lib.pasa_kprep_fp8(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 64, 5, None) == -3
    assert lib.pasa_kprep_fp8(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 128, 0, None) == -3
    assert lib.pasa_kprep_fp8(P(FAKE_MIS), P(FAKE), P(FAKE), P(FAKE), 1, 1, 64, 128, 5, None) == -4
    # pasa_attn_fwd_fp8(q, k8, means, kscale, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, stream)
    args = [P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 2, 1, 64, 64, 128, 0, 0.0]
    assert lib.pasa_attn_fwd_fp8(*args, 1, None) == -3            # not an FP8 mode
    args[3] = None
    assert lib.pasa_attn_fwd_fp8(*args, 5, None) == -1            # no block scales
    # the fp16-key entry points refuse the FP8 modes
    assert lib.pasa_attn_fwd_shifted(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 2, 1, 64, 64, 128, 0, 0.0,
                                     5, None) == -3


def test_decode_entry_points_check_arguments(lib):
    P = ctypes.c_void_p

    # pasa_attn_fwd_decode(q, k_shifted, means, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale, mode,
    #                      splits, workspace, workspace_bytes, stream)
    def dec(q=FAKE, means=FAKE, B=1, Hq=8, Hkv=1, Sq=1, Sk=5000, cap=5000, D=128, mode=0, splits=0, ws=None,
            ws_bytes=0):
        return lib.pasa_attn_fwd_decode(P(q), P(FAKE), P(means) if means else None, P(FAKE), P(FAKE), P(FAKE), B, Hq,
                                        Hkv, Sq, Sk, cap, D, 1, 0.0, mode, splits, P(ws) if ws else None, ws_bytes,
                                        None)

    assert dec(q=0) == -1
    assert dec(cap=4999) == -2                 # the cache holds fewer rows than Sk
    assert dec(Sq=17) == -3                    # 8 heads x 17 rows do not fit one 128-row tile
    assert dec(mode=5) == -3 and dec(mode=6) == -3
    assert dec(splits=-1) == -3
    assert dec(means=0) == -1                  # the shift modes read the block means
    assert dec(means=FAKE_MIS) == -4
    # 40 key blocks in 10 splits: more than one cluster holds, so the partials need a workspace
    assert dec(mode=3, means=0, splits=10) == -7
    need = lib.pasa_attn_fwd_decode_workspace_bytes(1, 8, 1, 1, 5000, 128, 10)
    assert need > 0
    assert dec(splits=10, ws=FAKE, ws_bytes=need - 1) == -7
    assert dec(splits=10, ws=FAKE + 16, ws_bytes=need) == -4   # 256-byte aligned
    # up to 8 splits of at most 32 packed rows at D = 128 merge inside a cluster: no workspace
    assert lib.pasa_attn_fwd_decode_workspace_bytes(1, 8, 1, 1, 5000, 128, 8) == 0
    # pasa_kshift_blocks(k, k_shifted, means, B, H, Sk, Sk_cap, D, first_block, stream)
    kb = lib.pasa_kshift_blocks
    assert kb(None, P(FAKE), P(FAKE), 1, 1, 300, 300, 128, 0, None) == -1
    assert kb(P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 299, 128, 0, None) == -2
    assert kb(P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 128, 3, None) == -2   # 300 rows: blocks 0..2
    assert kb(P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 128, -1, None) == -2
    assert kb(P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 96, 0, None) == -3
    assert kb(P(FAKE), P(FAKE_MIS), P(FAKE), 1, 1, 300, 300, 128, 0, None) == -4


def test_decode_step_checks_arguments(lib):
    """pasa_attn_fwd_decode_step checks the arguments of both of its calls before it enqueues
    anything (nothing here reaches a device)."""
    P = ctypes.c_void_p

    # pasa_attn_fwd_decode_step(q, k, k_shifted, means, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal,
    #                           scale, mode, first_block, splits, workspace, workspace_bytes, stream)
    def step(k=FAKE, means=FAKE, Sk=5000, cap=5000, D=128, mode=0, first=39, splits=0, ws=None, ws_bytes=0):
        return lib.pasa_attn_fwd_decode_step(P(FAKE), P(k) if k else None, P(FAKE), P(means) if means else None,
                                             P(FAKE), P(FAKE), P(FAKE), 1, 8, 1, 1, Sk, cap, D, 1, 0.0, mode, first,
                                             splits, P(ws) if ws else None, ws_bytes, None)

    assert step(k=0) == -1                     # the refresh reads the raw cache
    assert step(k=FAKE_MIS) == -4
    assert step(means=0) == -1 and step(means=FAKE_MIS) == -4
    assert step(mode=5) == -3 and step(mode=6) == -3   # e4m3 caches: kprep_fp8_blocks + decode_fp8
    assert step(first=40) == -2 and step(first=-1) == -2   # 5000 keys: blocks 0..39
    assert step(cap=4999) == -2
    assert step(D=96) == -3
    assert step(splits=-1) == -3
    need = lib.pasa_attn_fwd_decode_workspace_bytes(1, 8, 1, 1, 5000, 128, 10)
    assert step(splits=10, ws=FAKE, ws_bytes=need - 1) == -7
    assert step(splits=10, ws=FAKE + 16, ws_bytes=need) == -4


def test_decode_step_fp8_checks_arguments(lib):
    P = ctypes.c_void_p

    # pasa_attn_fwd_decode_step_fp8(q, k, k8, means, kscale, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D,
    #                               causal, scale, mode, first_block, splits, workspace, workspace_bytes, stream)
    def step(k=FAKE, means=FAKE, kscale=FAKE, Sq=1, Sk=5000, D=128, mode=5, first=39):
        return lib.pasa_attn_fwd_decode_step_fp8(P(FAKE), P(k) if k else None, P(FAKE), P(means) if means else None,
                                                 P(kscale) if kscale else None, P(FAKE), P(FAKE), P(FAKE), 1, 8, 1,
                                                 Sq, Sk, Sk, D, 1, 0.0, mode, first, 0, None, 0, None)

    assert step(mode=0) == -3 and step(mode=3) == -3   # fp16 caches: pasa_attn_fwd_decode_step
    assert step(k=0) == -1 and step(kscale=0) == -1
    assert step(means=0) == -1                          # mode 5 keeps block means
    assert step(k=FAKE_MIS) == -4 and step(kscale=FAKE_MIS) == -4
    assert step(D=64) == -3
    assert step(Sq=5) == -3                             # 40 packed rows: beyond the decode kernel
    assert step(first=40) == -2 and step(first=-1) == -2


def test_decode_workspace_bytes(lib):
    # split choice: `splits` if given, else at most one CTA per SM (152) over the B * Hkv
    # kv heads and at least eight key blocks per split; blocks spread evenly; no workspace
    # when that leaves one split. Partials: fp32 O [splits, B*Hq*Sq, D] and lse, 256-aligned.
    def expect(B, Hq, Hkv, Sq, Sk, D, splits):
        nb = -(-Sk // 128)
        sp = splits if splits > 0 else min(152 // (B * Hkv), nb // 8)
        sp = max(1, min(sp, nb, 65535))
        bps = -(-nb // sp)
        sp = -(-nb // bps)
        if sp == 1:
            return 0
        if D == 128 and (Hq // Hkv) * Sq <= 32 and sp <= 8:
            return 0      # merged inside a thread-block cluster
        rows = B * Hq * Sq
        a = lambda x: -(-x // 256) * 256
        return a(sp * rows * D * 4) + a(sp * rows * 4)

    for args in [(1, 8, 8, 1, 32768, 128, 0), (8, 28, 4, 1, 32768, 128, 0), (1, 8, 8, 1, 640, 128, 0),
                 (4, 32, 8, 4, 8192, 64, 0), (1, 8, 8, 1, 32768, 128, 5), (1, 28, 4, 1, 131072, 128, 0),
                 (1, 8, 8, 1, 128, 128, 0), (1, 2, 1, 64, 777, 128, 100), (200, 8, 1, 1, 4096, 128, 0),
                 (1, 8, 1, 1, 5000, 128, 12), (2, 28, 4, 4, 3001, 128, 0), (1, 16, 2, 8, 2049, 64, 0)]:
        assert lib.pasa_attn_fwd_decode_workspace_bytes(*args) == expect(*args), args
    assert lib.pasa_attn_fwd_decode_workspace_bytes(1, 3, 2, 1, 100, 128, 0) == 0   # Hq % Hkv != 0


def test_fp8_decode_entry_points_check_arguments(lib):
    P = ctypes.c_void_p

    # pasa_attn_fwd_decode_fp8(q, k8, means, kscale, v, o, lse, B, Hq, Hkv, Sq, Sk, Sk_cap, D, causal, scale,
    #                          mode, splits, workspace, workspace_bytes, stream)
    def dec8(means=FAKE, kscale=FAKE, Hq=8, Hkv=1, Sq=1, D=128, mode=5, cap=5000):
        return lib.pasa_attn_fwd_decode_fp8(P(FAKE), P(FAKE), P(means) if means else None,
                                            P(kscale) if kscale else None, P(FAKE), P(FAKE), P(FAKE), 1, Hq, Hkv, Sq,
                                            5000, cap, D, 1, 0.0, mode, 0, None, 0, None)

    assert dec8(mode=0) == -3 and dec8(mode=3) == -3     # fp16 modes: pasa_attn_fwd_decode
    assert dec8(D=64) == -3                              # e4m3 keys: D = 128 only
    assert dec8(Sq=5) == -3                              # 40 packed rows: beyond the decode kernel
    assert dec8(kscale=0) == -1
    assert dec8(means=0) == -1 and dec8(mode=6, means=0) != -1
    assert dec8(kscale=FAKE_MIS) == -4
    assert dec8(cap=4999) == -2
    # the fp16 decode entry refuses the FP8 modes
    assert lib.pasa_attn_fwd_decode(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 8, 1, 1, 5000, 5000, 128,
                                    1, 0.0, 5, 0, None, 0, None) == -3
    # pasa_kprep_fp8_blocks(k, k8, means, kscale, B, H, Sk, Sk_cap, D, mode, first_block, stream)
    kb = lib.pasa_kprep_fp8_blocks
    assert kb(P(FAKE), P(FAKE), None, P(FAKE), 1, 1, 300, 300, 128, 5, 0, None) == -1   # mode 5 needs means
    assert kb(P(FAKE), P(FAKE), None, None, 1, 1, 300, 300, 128, 6, 0, None) == -1
    assert kb(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 128, 5, 3, None) == -2
    assert kb(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 299, 128, 5, 0, None) == -2
    assert kb(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 64, 5, 0, None) == -3
    assert kb(P(FAKE), P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 128, 1, 0, None) == -3
    assert kb(P(FAKE_MIS), P(FAKE), P(FAKE), P(FAKE), 1, 1, 300, 300, 128, 6, 0, None) == -4


def test_host_buffer_entry_checks_arguments(lib):
    P = ctypes.c_void_p
    # pasa_attn_fwd_host(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, causal, scale, mode, chunks, buf, buf_bytes, stream)
    def host(q=FAKE, o=FAKE, B=1, Hq=8, Hkv=2, Sq=300, Sk=300, D=128, mode=0, chunks=0, buf=FAKE, nbytes=None):
        if nbytes is None:
            nbytes = lib.pasa_attn_fwd_host_device_bytes(B, Hq, Hkv, Sq, Sk, D, 1, mode, chunks)
        return lib.pasa_attn_fwd_host(P(q) if q else None, P(FAKE), P(FAKE), P(o) if o else None, None, B, Hq, Hkv,
                                      Sq, Sk, D, 1, 0.0, mode, chunks, P(buf) if buf else None, nbytes, None)

    assert host(q=0) == -1 and host(o=0) == -1
    assert host(Hq=7) == -2 and host(Sk=0) == -2 and host(chunks=-1) == -2
    assert host(D=96) == -3 and host(mode=9) == -3 and host(D=64, mode=5) == -3
    nbytes = lib.pasa_attn_fwd_host_device_bytes(1, 8, 2, 300, 300, 128, 1, 0, 0)
    assert host(nbytes=nbytes - 1) == -7                 # buffer too small
    assert host(buf=FAKE + 128, nbytes=nbytes) == -4     # buffer not 256-byte aligned
    # host pointers need no alignment: a misaligned q gets past argument checks to the
    # device query, which fails here (no GPU) instead of reporting PASA_ERR_ALIGN
    assert host(q=FAKE_MIS) != -4


def test_host_buffer_device_bytes(lib):
    nb = lib.pasa_attn_fwd_host_device_bytes
    assert nb(1, 8, 2, 300, 300, 128, 1, 0, -1) == 0 and nb(1, 7, 2, 300, 300, 128, 1, 0, 0) == 0
    for (B, Hq, Hkv, Sq, Sk, D) in [(1, 28, 4, 32768, 32768, 128), (2, 5, 5, 9216, 9216, 64), (8, 28, 4, 1, 4096, 128),
                                    (3, 6, 3, 129, 257, 64), (1, 64, 1, 2048, 2048, 128)]:
        units = B * Hkv
        problem = 2 * B * Hq * Sq * D * 2 + 2 * B * Hkv * Sk * D * 2 + B * Hq * Sq * 4
        for mode in (0, 2, 5):
            if mode == 5 and D != 128:
                continue
            for causal in (0, 1):
                for chunks in (1, 2, 3, units, units + 5):
                    n = min(chunks, units)
                    biggest = -(-units // n)
                    got = nb(B, Hq, Hkv, Sq, Sk, D, causal, mode, chunks)
                    # whole problem staged + a workspace for each of the two compute streams
                    # (one when there is one piece), slots 256-byte aligned
                    ws = -(-lib.pasa_attn_fwd_workspace_bytes(biggest, 1, Sk, D, mode) // 256) * 256
                    ws *= 2 if n > 1 else 1
                    assert problem + ws <= got <= problem + ws + 5 * 256 * n, (B, Hq, Sq, mode, chunks)
                    assert got % 256 == 0
                # the automatic plan (row pieces included) stages the same problem, once
                auto = nb(B, Hq, Hkv, Sq, Sk, D, causal, mode, 0)
                ws1 = lib.pasa_attn_fwd_workspace_bytes(1, 1, Sk, D, mode)
                assert problem + ws1 <= auto <= problem + 2 * lib.pasa_attn_fwd_workspace_bytes(units, 1, Sk, D, mode) \
                    + 5 * 256 * (units + 8) + 512


def host_plan_checks(B, Hq, Hkv, Sq, Sk, D, causal, chunks):
    """Every (unit, query row) in exactly one piece, in unit order; each unit's keys copied
    once, in order, up to what its rows see; row pieces on 128-row tiles with their key
    prefix ending on a 128-key block or at Sk (the conditions for tile-for-tile equality)."""
    import precision_flashattention_numerics_gb300 as pasa

    plan = pasa.host_plan(B, Hq, Hkv, Sq, Sk, D, causal, 0, chunks)
    units = B * Hkv
    covered = {}
    keys = {}
    for (u0, n, r0, r1, k0, k1) in plan:
        assert n >= 1 and 0 <= r0 < r1 <= Sq
        if n > 1 or (r0 == 0 and r1 == Sq):
            assert (r0, r1, k0, k1) == (0, Sq, 0, Sk)
        else:
            assert r0 % 128 == 0
            assert k1 == (r1 + Sk - Sq if causal else Sk)
            assert k1 == Sk or k1 % 128 == 0
        for u in range(u0, u0 + n):
            covered.setdefault(u, []).append((r0, r1))
            assert k0 == keys.get(u, 0), "keys copied in order, once"
            keys[u] = k1
    assert sorted(covered) == list(range(units))
    for u, spans in covered.items():
        assert spans[0][0] == 0 and spans[-1][1] == Sq
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
        assert keys[u] == Sk
    order = [(u0, r0) for (u0, n, r0, r1, k0, k1) in plan]
    assert order == sorted(order)
    return plan


def test_host_buffer_plan(lib):
    # explicit chunk counts: whole units only
    plan = host_plan_checks(3, 6, 3, 300, 700, 64, True, 4)
    assert [p[1] for p in plan] == [2, 2, 2, 3] and all((p[2], p[3]) == (0, 300) for p in plan)
    assert [p[1] for p in host_plan_checks(2, 8, 4, 520, 520, 128, True, 3)] == [2, 3, 3]
    # automatic: the 32K workload, 4 units; the first and last unit in halving row pieces
    plan = host_plan_checks(1, 28, 4, 32768, 32768, 128, True, 0)
    assert [(p[0], p[2], p[3]) for p in plan] == [
        (0, 0, 4096), (0, 4096, 8192), (0, 8192, 16384), (0, 16384, 32768), (1, 0, 32768), (2, 0, 32768),
        (3, 0, 16384), (3, 16384, 24576), (3, 24576, 28672), (3, 28672, 32768)]
    # one unit cut at both ends; Sk > Sq by whole blocks; not causal with a ragged Sk
    assert len(host_plan_checks(1, 64, 1, 2048, 2048, 128, True, 0)) == 6
    assert len(host_plan_checks(1, 64, 1, 2048, 2048 + 256, 128, True, 0)) == 6
    assert len(host_plan_checks(1, 64, 1, 2048, 2000, 64, False, 0)) == 6
    # causal offsets that are not whole blocks, or rows that see no key: no row pieces
    assert len(host_plan_checks(1, 64, 1, 2048, 2048 + 100, 128, True, 0)) == 1
    assert len(host_plan_checks(1, 64, 1, 2048, 1024, 128, True, 0)) == 1
    # small problems stay one piece
    assert len(host_plan_checks(1, 8, 1, 300, 300, 128, True, 0)) == 1
    assert len(host_plan_checks(8, 28, 4, 1, 4096, 128, True, 0)) == 1
    for shape in [(4, 32, 8, 8192, 8192, 128, True), (2, 5, 5, 9216, 9216, 64, False), (3, 48, 3, 4096, 4224, 64, True)]:
        host_plan_checks(*shape, 0)
        host_plan_checks(*shape, 5)


def test_host_buffer_plan_properties(lib):
    """Random shapes, masks and chunk requests: every plan covers each (unit, query row)
    once, copies each key once and in order, keeps row pieces tile- and block-aligned, and
    the staging size holds at least the whole problem."""
    hypothesis = pytest.importorskip("hypothesis")
    st = hypothesis.strategies

    @hypothesis.settings(max_examples=300, deadline=None, derandomize=True)
    @hypothesis.given(B=st.integers(1, 6), Hkv=st.integers(1, 8), g=st.sampled_from([1, 2, 4, 7, 8, 16, 64]),
                      Sq=st.integers(1, 40000), dk=st.integers(-2000, 3000), D=st.sampled_from([64, 128]),
                      causal=st.booleans(), chunks=st.integers(0, 70))
    def check(B, Hkv, g, Sq, dk, D, causal, chunks):
        Sk = max(1, Sq + dk)
        plan = host_plan_checks(B, Hkv * g, Hkv, Sq, Sk, D, causal, chunks)
        units = B * Hkv
        assert len(plan) >= min(max(chunks, 1), units, 64) if chunks else len(plan) >= 1
        nbytes = lib.pasa_attn_fwd_host_device_bytes(B, Hkv * g, Hkv, Sq, Sk, D, int(causal), 0, chunks)
        problem = 2 * B * Hkv * g * Sq * D * 2 + 2 * units * Sk * D * 2 + B * Hkv * g * Sq * 4
        assert nbytes >= problem and nbytes % 256 == 0

    check()


def call_fused(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, Hq=2, Hkv=1, Sq=64, Sk=64, D=128,
               causal=0, mode=0, ks_out=None, m_out=None):
    P = ctypes.c_void_p
    return lib.pasa_attn_fwd_fused(P(q), P(k), P(v), P(o), P(lse), B, Hq, Hkv, Sq, Sk, D, causal, 0.0, mode,
                                   P(ks_out) if ks_out is not None else None,
                                   P(m_out) if m_out is not None else None, None)


def test_fused_argument_errors(lib):
    # the fused-shift entry point: D = 128 and the shifted modes only, checked before any launch
    assert call_fused(lib, q=0) == -1
    assert call_fused(lib, v=0) == -1
    assert call_fused(lib, B=0) == -2
    assert call_fused(lib, Hq=3, Hkv=2) == -2
    assert call_fused(lib, D=64) == -3
    for mode in (2, 3, 5, 6, 7):
        assert call_fused(lib, mode=mode) == -3, mode
    assert call_fused(lib, k=FAKE_MIS) == -4
    assert call_fused(lib, lse=FAKE_MIS) == -4
    assert call_fused(lib, ks_out=FAKE_MIS) == -4
    assert call_fused(lib, m_out=FAKE_MIS) == -4


def test_exp2_selftest_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.pasa_selftest_exp2(None, P(FAKE), P(FAKE), 16, None) == -1
    assert lib.pasa_selftest_exp2(P(FAKE), P(FAKE), None, 16, None) == -1
    assert lib.pasa_selftest_exp2(P(FAKE), P(FAKE), P(FAKE), 0, None) == -2
