"""Host-side checks of the C ABI: the library loads, exports every entry point
include/fa.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import exact_io_aware_35_gb300 as fa
    from exact_io_aware_35_gb300 import build as fa_build
    fa_build.build()
    return fa.load_library()


def declared_entry_points():
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for n in ("fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_get_device_error",
              "fa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import exact_io_aware_35_gb300 as fa
    for name in declared_entry_points():
        assert hasattr(lib, name), name
    assert set(declared_entry_points()) <= set(fa.EXPORTS)


def test_status_strings(lib):
    import exact_io_aware_35_gb300 as fa
    assert fa.status_string(0) == "FA_OK"
    assert fa.status_string(4) == "FA_ERR_DEVICE_TIMEOUT"
    assert fa.status_string(99) == "FA_ERR_UNKNOWN"


def _up256(x):
    return (x + 255) // 256 * 256


def test_workspace_size(lib):
    # D (4 bytes per query row and head), fp16 copies of q, k, v, dout, 512 bytes of scales
    def bwd(B, H, Hkv, N, d):
        return (_up256(4 * B * H * N) + 2 * _up256(2 * B * N * H * d) +
                2 * _up256(2 * B * N * Hkv * d) + 512)
    assert lib.fa_bwd_workspace_size(2, 3, 1, 5, 64) == bwd(2, 3, 1, 5, 64) == 11008
    assert lib.fa_bwd_workspace_size(4, 32, 8, 8192, 128) == bwd(4, 32, 8, 8192, 128)
    assert lib.fa_bwd_workspace_size(0, 1, 1, 1, 64) == 0
    assert lib.fa_bwd_workspace_size(1, 1, 1, 1, 96) == 0     # unsupported d
    assert lib.fa_bwd_workspace_size(1, 6, 4, 1, 64) == 0     # Hq % Hkv != 0



def _fwd(lib, ptr=16, B=1, H=1, Hkv=1, N=128, d=64, causal=0, scale=0.125):
    return lib.fa_fwd(ptr, ptr, ptr, ptr, ptr, B, H, Hkv, N, d, causal,
                      ctypes.c_float(scale), None)


def _bwd(lib, ptr=256, B=1, H=1, Hkv=1, N=128, d=64, scale=0.125, ws=256, o_lo=None):
    return lib.fa_bwd(ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ptr, ws, o_lo, B, H, Hkv, N, d,
                      0, ctypes.c_float(scale), None)


def test_invalid_arguments_rejected_on_host(lib):
    import exact_io_aware_35_gb300 as fa
    assert _fwd(lib, ptr=0) == fa.FA_ERR_INVALID_ARG          # null
    assert _fwd(lib, ptr=8) == fa.FA_ERR_INVALID_ARG          # not 16-byte aligned
    assert _fwd(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, B=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, H=6, Hkv=4) == fa.FA_ERR_INVALID_ARG     # Hq % Hkv != 0
    assert _fwd(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, d=256) == fa.FA_ERR_UNSUPPORTED
    assert _bwd(lib, ws=0) == fa.FA_ERR_INVALID_ARG
    assert _bwd(lib, ws=272) == fa.FA_ERR_INVALID_ARG         # workspace not 256-aligned
    assert _bwd(lib, o_lo=8) == fa.FA_ERR_INVALID_ARG         # o_lo misaligned
    assert _bwd(lib, d=80) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_train(16, 16, 16, 16, 8, 16, None, 1, 1, 1, 128, 64, 0,
                            ctypes.c_float(0.125), None) == fa.FA_ERR_INVALID_ARG  # o_lo
    assert lib.fa_fwd_train(16, 16, 16, 16, 16, 16, 272, 1, 1, 1, 128, 64, 0,
                            ctypes.c_float(0.125), None) == fa.FA_ERR_INVALID_ARG  # workspace
    for stages in (0, 32, -1):
        assert lib.fa_bwd_stage(stages, 256, 256, 256, 256, 256, 256, 256, 256, 256, 256, None,
                                1, 1, 1, 128, 64, 0, ctypes.c_float(0.125),
                                None) == fa.FA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch

    import exact_io_aware_35_gb300 as fa
    q = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q)


def test_binding_refuses_tensors_on_another_device():
    # every wrapper checks that each tensor sits on q's device before it
    # passes raw pointers to the library
    import torch

    import exact_io_aware_35_gb300 as fa
    a = torch.zeros(2)
    fa._on_device(a.device, k=a, v=None)
    with pytest.raises(ValueError, match="k is on cpu"):
        fa._on_device(torch.device("cuda", 0), k=a)


def test_splitkv_plan_and_workspace(lib):
    import exact_io_aware_35_gb300 as fa
    # one split: no workspace
    assert lib.fa_fwd_splitkv_num_splits(1, 8, 2, 1, 100, 128, 0, 1) == 1
    assert lib.fa_fwd_splitkv_workspace_size(1, 8, 2, 1, 100, 128, 0, 1) == 0
    # requested splits are clamped to the 128-key blocks and never left empty
    assert lib.fa_fwd_splitkv_num_splits(1, 8, 2, 1, 1000, 128, 0, 50) == 8
    assert lib.fa_fwd_splitkv_num_splits(1, 8, 2, 1, 1000, 128, 0, 3) == 3
    assert lib.fa_fwd_splitkv_num_splits(1, 8, 2, 1, 1000, 128, 0, 5) == 4  # 2 blocks each
    # fp32 O_s and lse_s per (split, batch, head, query), each rounded to 256
    n = 3 * 2 * 8 * 5
    assert lib.fa_fwd_splitkv_workspace_size(2, 8, 2, 5, 1000, 64, 1, 3) == \
        _up256(n * 64 * 4) + _up256(n * 4)
    # the library's choice: the count with the least waves x (blocks per split + 3)
    # on 152 SMs, one CTA each (units = batch x kv heads x query tiles)
    def cost(units, nblk, s2):
        bps = -(-nblk // s2)
        ctas = units * -(-nblk // bps)
        return -(-ctas // 152) * (bps + 3)
    for (B, H, Hkv, Nq, Nk) in ((8, 32, 8, 1, 32768), (1, 16, 1, 1, 131072), (2, 8, 1, 40, 5000)):
        s = lib.fa_fwd_splitkv_num_splits(B, H, Hkv, Nq, Nk, 128, 1, 0)
        g = H // Hkv
        units = B * Hkv * -(-Nq // (128 // g))
        nblk = -(-Nk // 128)
        assert cost(units, nblk, s) == min(cost(units, nblk, x) for x in range(1, nblk + 1))
        assert fa.fa_fwd_splitkv_num_splits(B, H, Hkv, Nq, Nk, 128, True) == s
    # invalid sizes
    assert lib.fa_fwd_splitkv_num_splits(1, 8, 2, 10, 5, 128, 1, 0) == 0   # causal Nq > Nk
    assert lib.fa_fwd_splitkv_num_splits(1, 6, 4, 1, 5, 128, 0, 0) == 0    # Hq % Hkv
    assert lib.fa_fwd_splitkv_num_splits(1, 256, 1, 1, 5, 128, 0, 0) == 0  # g > 128
    assert lib.fa_fwd_splitkv_workspace_size(1, 8, 2, 1, 100, 96, 0, 0) == 0


def test_splitkv_invalid_arguments_rejected_on_host(lib):
    import exact_io_aware_35_gb300 as fa

    def call(ptr=256, ws=256, B=1, H=8, Hkv=2, Nq=1, Nk=1000, d=128, causal=0, scale=0.1,
             splits=4):
        return lib.fa_fwd_splitkv(ptr, ptr, ptr, ptr, ptr, ws, B, H, Hkv, Nq, Nk, d, causal,
                                  ctypes.c_float(scale), splits, None)
    assert call(ptr=0) == fa.FA_ERR_INVALID_ARG
    assert call(ptr=8) == fa.FA_ERR_INVALID_ARG
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG          # several splits need a workspace
    assert call(ws=272) == fa.FA_ERR_INVALID_ARG        # not 256-aligned
    assert call(Nq=2000, causal=1) == fa.FA_ERR_INVALID_ARG
    assert call(Nk=0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(H=256, Hkv=1) == fa.FA_ERR_UNSUPPORTED


def test_blocksparse_invalid_arguments_rejected_on_host(lib):
    import exact_io_aware_35_gb300 as fa

    def call(ptr=256, mask=256, N=1000, d=128, H=4, Hkv=2, scale=0.1):
        return lib.fa_fwd_blocksparse(ptr, ptr, ptr, ptr, ptr, mask, 1, H, Hkv, N, d, 0,
                                      ctypes.c_float(scale), None)
    assert call(mask=None) == fa.FA_ERR_INVALID_ARG
    assert call(ptr=8) == fa.FA_ERR_INVALID_ARG
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    assert call(H=6, Hkv=4) == fa.FA_ERR_INVALID_ARG
    assert call(scale=-1.0) == fa.FA_ERR_INVALID_ARG
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    # mask rows longer than the 7,168 blocks a thread block keeps in shared memory
    assert call(N=7168 * 128 + 1) == fa.FA_ERR_UNSUPPORTED


def test_fp8_workspace_and_invalid_arguments(lib):
    import exact_io_aware_35_gb300 as fa
    B, H, Hkv, N = 2, 4, 2, 300
    nb, ldv = 3, 304
    want = (_up256(B * N * H * 128) + _up256(B * N * Hkv * 128) + _up256(B * Hkv * 128 * ldv) +
            _up256(B * H * nb * 4) + _up256(B * Hkv * nb * 4) + 2 * _up256(B * Hkv * 4))
    assert lib.fa_fwd_fp8_workspace_size(B, H, Hkv, N, 128) == want
    assert lib.fa_fwd_fp8_workspace_size(B, H, Hkv, N, 64) == 0

    def call(ptr=256, ws=256, d=128, flags=1, N=300, scale=0.1):
        return lib.fa_fwd_fp8(ptr, ptr, ptr, ptr, ptr, ws, 1, 4, 2, N, d, 1,
                              ctypes.c_float(scale), flags, None)
    assert call(d=64) == fa.FA_ERR_UNSUPPORTED
    assert call(ws=0) == fa.FA_ERR_INVALID_ARG
    assert call(ws=272) == fa.FA_ERR_INVALID_ARG
    assert call(flags=8) == fa.FA_ERR_INVALID_ARG
    assert call(flags=6) == fa.FA_ERR_INVALID_ARG   # quantise only and attend only
    assert call(ptr=8) == fa.FA_ERR_INVALID_ARG
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
