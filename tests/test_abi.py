"""The C ABI library loads and exports every entry point include/*.h
declares; argument checks answer on the host before any launch.  CPU only:
the calls below never reach a kernel (they fail validation or are empty)."""
import ctypes
import glob
import os
import re

import pytest
import torch

from conftest import ROOT

import nvfp4_w4a4_decode_gb300 as nv
from nvfp4_w4a4_decode_gb300 import build as nvbuild


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(nvfp4_\w+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    nvbuild.build()
    return nv.library()


def test_header_declares_entry_points():
    names = declared_functions()
    for want in ("nvfp4_pack_weight", "nvfp4_quantize_act", "nvfp4_gemm_smallm",
                 "nvfp4_global_scale", "nvfp4_status_string", "nvfp4_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(nv.SIGNATURES)


def test_status_strings(lib):
    for code, name in nv.STATUS.items():
        assert lib.nvfp4_status_string(code).decode() == name
    assert lib.nvfp4_status_string(99).decode() == "NVFP4_ERR_UNKNOWN"
    assert b"sm_103a" in lib.nvfp4_version()


FAKE = 1 << 20  # a non-null, 256-byte aligned value never dereferenced


def test_gemm_rejects_bad_arguments(lib):
    g = lib.nvfp4_gemm_smallm
    ok_args = [FAKE] * 7
    assert g(*ok_args, 9, 16, 32, None) == 2        # M > 8: unsupported
    assert g(*ok_args, 1, 16, 24, None) == 1        # K not a multiple of 16
    assert g(*ok_args, -1, 16, 32, None) == 1
    assert g(*ok_args, 1, -16, 32, None) == 1
    bad = list(ok_args)
    bad[3] = None                                   # null weight codes
    assert g(*bad, 1, 16, 32, None) == 1
    bad = list(ok_args)
    bad[0] = FAKE + 4                               # misaligned activation codes
    assert g(*bad, 1, 16, 32, None) == 1
    assert g(*ok_args, 0, 16, 32, None) == 0        # empty batch: nothing to do
    assert g(*ok_args, 2, 0, 32, None) == 0         # empty output


def test_quantize_and_pack_reject_bad_arguments(lib):
    q = lib.nvfp4_quantize_act
    assert q(FAKE, 1, 20, FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE + 8, 1, 32, FAKE, FAKE, FAKE, None) == 1    # X not 16-byte aligned
    assert q(None, 1, 32, FAKE, FAKE, FAKE, None) == 1
    assert q(FAKE, 0, 32, FAKE, FAKE, FAKE, None) == 0        # empty
    p = lib.nvfp4_pack_weight
    assert p(FAKE, 4, 40, FAKE, FAKE, FAKE, None) == 1
    assert p(FAKE, 4, 32, FAKE, FAKE, None, None) == 1
    s = lib.nvfp4_global_scale
    assert s(FAKE, -1, FAKE, None) == 1
    assert s(FAKE, 4, None, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(nv, "_lib", None)
    with pytest.raises(ImportError):
        nv.library(str(tmp_path / "missing.so"))


def test_gemm_select_host_only(lib):
    """Kernel selection is host logic: which kernel each shape gets."""
    AUTO, GENERIC, GEMV = nv.KERNEL_AUTO, nv.KERNEL_GENERIC, nv.KERNEL_GEMV
    for k in (2048, 4096, 5120, 6144, 8192, 12288, 25600, 10240):
        assert nv.gemm_select(1, 100, k) == GEMV, k
        assert nv.gemm_select(2, 100, k, GEMV) == GEMV, k
    for m, k in ((1, 384), (1, 16), (2, 4112), (8, 4112), (3, 48)):
        assert nv.gemm_select(m, 100, k) == GENERIC, (m, k)
    assert nv.gemm_select(3, 10, 4096, GEMV) == -2
    assert nv.gemm_select(1, 10, 512, GEMV) == -2
    assert nv.gemm_select(9, 10, 4096) == -2
    assert nv.gemm_select(1, 10, 24) == -1
    assert nv.gemm_select(1, 10, 4096, 77) == -2
    MMA = nv.KERNEL_MMA
    for m in range(1, 9):
        for k in (1024, 2048, 4096, 5120, 8192, 12288, 25600):
            assert nv.gemm_select(m, 100, k, MMA) == MMA, (m, k)
        # M >= 2: split-K in one chunk (K <= 32768 / M) or, where a device
        # allows it, in its cluster form; else the TMA-fed or register kernel
        assert nv.gemm_select(m, 100, 4096) == (GEMV if m == 1 else nv.KERNEL_SPLITK)
        assert nv.gemm_select(m, 100, 12288) in ((GEMV,) if m == 1 else (nv.KERNEL_SPLITK,) if m == 2
                                                 else (nv.KERNEL_SPLITK, MMA, nv.KERNEL_TMA))
    assert nv.gemm_select(1, 10, 384, MMA) == -2          # too few 128-ranges
    assert nv.gemm_select(4, 10, 256 * 37, MMA) == -2     # 74 ranges: no split fits
    # 37 sub-items of 256 at M = 4: two unequal chunks, so split-K where a
    # device runs its cluster form, else the generic kernel
    assert nv.gemm_select(4, 10, 256 * 37) == (nv.KERNEL_SPLITK if torch.cuda.is_available()
                                                else GENERIC)


def test_ex_options_validated(lib):
    ok = [FAKE] * 7
    assert lib.nvfp4_gemm_smallm_ex(*ok, 1, 16, 32, 0x200, None) == 1     # unknown flag
    assert lib.nvfp4_gemm_smallm_ex(*ok, 3, 16, 4096, 2, None) == 2       # GEMV with M = 3
    assert lib.nvfp4_quantize_act_ex(FAKE, 1, 32, FAKE, FAKE, FAKE, 1, None) == 1


def test_linear_rejects_bad_arguments(lib):
    f = lib.nvfp4_linear
    # x, m, n, k, x_g, w_q, w_s, w_g, y, x_q, x_s, options, stream
    assert f(FAKE, 9, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 2
    assert f(FAKE, 1, 16, 40, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 1
    assert f(FAKE + 4, 1, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 1
    assert f(FAKE, 1, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 0, None) == 1
    assert f(FAKE, 1, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0x4000, None) == 1
    assert f(FAKE, 0, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None) == 0


def test_dynamic_quantize_rejects_bad_arguments(lib):
    q = lib.nvfp4_quantize_act_dynamic
    assert q(FAKE, 1, 20, FAKE, FAKE, FAKE, None) == 1       # K not a multiple of 16
    assert q(FAKE, 1, 32, None, FAKE, FAKE, None) == 1       # no x_g output
    assert q(FAKE + 4, 1, 32, FAKE, FAKE, FAKE, None) == 1   # X misaligned


def test_workspace_entry_points_host_only(lib):
    """Workspace size and checks of the _ws entry points answer on the host."""
    SPLITK = nv.KERNEL_SPLITK
    assert lib.nvfp4_gemm_workspace_size(1, 100, 4096, nv.KERNEL_GEMV) == 0
    assert lib.nvfp4_gemm_workspace_size(8, 6144, 4096, SPLITK) >= 0
    assert lib.nvfp4_gemm_workspace_size(8, 6144, 12288, SPLITK) >= 0   # workspace or cluster
    assert lib.nvfp4_gemm_workspace_size(8, 512, 40960, SPLITK) > 0     # > 8 chunks: workspace
    assert lib.nvfp4_gemm_workspace_size(9, 100, 4096, SPLITK) == -2
    assert lib.nvfp4_gemm_workspace_size(1, 100, 40, SPLITK) == -1
    assert lib.nvfp4_gemm_workspace_size(1, 100, 4000, SPLITK) == -2   # K % 256 != 0
    assert nv.gemm_select(3, 100, 4096, SPLITK) == SPLITK    # one chunk: no workspace needed
    for m, n, k in ((4, 6144, 4096), (8, 4096, 12288), (3, 5120, 25600)):
        need = lib.nvfp4_gemm_workspace_size(m, n, k, nv.KERNEL_AUTO)
        assert need == lib.nvfp4_gemm_workspace_size(m, n, k, SPLITK)
        assert nv.gemm_select(m, n, k, nv.KERNEL_AUTO, need) == SPLITK     # offered: taken
    assert lib.nvfp4_gemm_workspace_size(1, 6144, 4096, nv.KERNEL_AUTO) == 0   # gemv
    assert nv.gemm_select(1, 6144, 4096, nv.KERNEL_AUTO, 1 << 30) == nv.KERNEL_GEMV
    if not torch.cuda.is_available():   # M = 8, K > 4096: a workspace or a device's clusters
        assert nv.gemm_select(8, 100, 8192, SPLITK) == -2
    assert nv.gemm_select(2, 100, 12288, SPLITK) == SPLITK   # M = 2: K up to 16384 in one chunk
    ok = [FAKE] * 7
    g = lib.nvfp4_gemm_smallm_ws
    assert g(*ok, 1, 16, 256, SPLITK, None, 64, None) == 1           # bytes without a pointer
    assert g(*ok, 1, 16, 256, SPLITK, FAKE + 8, 64, None) == 1       # misaligned workspace
    assert g(*ok, 9, 16, 256, SPLITK, FAKE, 64, None) == 2
    assert g(*ok, 0, 16, 256, SPLITK, FAKE, 64, None) == 0           # empty: nothing to do
    f = lib.nvfp4_linear_ws
    assert f(FAKE, 1, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None, 8, None) == 1
    assert f(FAKE, 0, 16, 32, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, 8, None) == 0


def test_read_probe_rejects_bad_arguments(lib):
    f = lib.nvfp4_read_probe
    assert f(FAKE, 17, FAKE, None) == 1          # not a multiple of 16
    assert f(FAKE, -16, FAKE, None) == 1
    assert f(FAKE + 8, 32, FAKE, None) == 1      # buffer not 16-byte aligned
    assert f(None, 32, FAKE, None) == 1
    assert f(FAKE, 32, None, None) == 1          # no sink
    assert f(FAKE, 32, FAKE + 4, None) == 1      # sink not 8-byte aligned


def test_splitk_planner_properties_host_only(lib):
    """For many shapes: the workspace the split-K plan asks for is accepted
    for that plan; without a workspace and without a device (so without the
    cluster form) a plan exists exactly when K fits one CTA's activation
    fragments (2 M bytes per element, 64 KB); K not a multiple of 256 and M
    outside 1..8 are refused."""
    import random
    rnd = random.Random(5)
    SPLITK = nv.KERNEL_SPLITK
    for _ in range(300):
        m = rnd.randint(1, 8)
        k = 256 * rnd.randint(1, 160)
        n = rnd.randint(1, 70000)
        need = lib.nvfp4_gemm_workspace_size(m, n, k, SPLITK)
        assert need >= 0
        assert lib.nvfp4_gemm_select_ws(m, n, k, SPLITK, need) == SPLITK
        one_chunk = k <= (65536 // (2 * m)) // 256 * 256
        nows = lib.nvfp4_gemm_select_ws(m, n, k, SPLITK, 0) == SPLITK
        assert nows == one_chunk or (nows and torch.cuda.is_available()), (m, n, k)
        if one_chunk:
            assert need == 0 or need >= 1024 * ((n + 15) // 16)   # 2+ partials of 512 B per tile
    for m, k in ((1, 4000), (9, 4096), (0, 4096)):
        assert lib.nvfp4_gemm_select_ws(m, 100, k, SPLITK, 1 << 30) < 0


def _chain_arr(**over):
    fields = dict(x=FAKE, x_g=FAKE, x_q=FAKE, x_s=FAKE, w_q=FAKE, w_s=FAKE, w_g=FAKE, y=FAKE,
                  n=64, k=4096)
    fields.update(over)
    arr = (nv.ChainLinear * 1)(nv.ChainLinear(**fields))
    return ctypes.cast(arr, ctypes.c_void_p), arr


def test_chain_rejects_before_launch(lib):
    """Every refusal of the multi-linear entry points returns before a launch."""
    f = lib.nvfp4_linear_chain
    p, _keep = _chain_arr()
    assert f(p, 1, 3, nv.KERNEL_GEMV, None) == 2            # CUDA-core stream: M of 1 or 2
    assert f(p, 1, 33, nv.KERNEL_AUTO, None) == 2           # tensor cores: M up to 32
    assert f(p, 1, 1, nv.KERNEL_SPLITK, None) == 2          # no chain on this kernel
    assert f(p, 1, 1, 0x10000, None) == 1                   # unknown flag
    assert f(p, -1, 1, 0, None) == 1
    assert f(p, 0, 1, 0, None) == 0                         # nothing to do
    assert f(None, 0, 1, 0, None) == 0
    assert f(p, 1, 0, 0, None) == 0
    for over, want in ((dict(k=4100), 1),                   # K not a multiple of 16
                       (dict(k=4112), 2),                   # nor of 256 (tensor cores)
                       (dict(n=-1), 1),
                       (dict(x_q=FAKE + 16), 1),            # codes 32-byte aligned
                       (dict(w_s=FAKE + 4), 1),             # tensor cores: scales 16-byte aligned
                       (dict(x=None), 1),                   # the quantiser reads x
                       (dict(y=None), 1)):
        q, _k = _chain_arr(**over)
        assert f(q, 1, 1, 0, None) == want, over
    q, _k = _chain_arr(k=2560)                               # K % 1024 != 0: not on the
                                                             # CUDA-core stream
    assert f(q, 1, 1, nv.KERNEL_GEMV, None) == 2
    assert lib.nvfp4_linear_chain_ws(p, 1, 1, 0, FAKE + 8, 16, None) == 1   # workspace alignment
    assert lib.nvfp4_linear_chain_ws(p, 1, 1, 0, None, 16, None) == 1       # size without memory


def test_chain_queries(lib):
    assert lib.nvfp4_chain_workspace_size(1, nv.KERNEL_GEMV) == 0
    assert lib.nvfp4_chain_workspace_size(1, nv.KERNEL_AUTO) >= 1024
    assert lib.nvfp4_chain_workspace_size(3, nv.KERNEL_GEMV) == -2
    assert lib.nvfp4_chain_workspace_size(33, nv.KERNEL_AUTO) == -2
    assert lib.nvfp4_chain_workspace_size(0, 0) == -1
    assert lib.nvfp4_chain_supported(1, 4096, 4096) == 1
    assert lib.nvfp4_chain_supported(32, 4096, 256) == 1
    assert lib.nvfp4_chain_supported(1, 4096, 4112) == 0
    assert lib.nvfp4_chain_supported(33, 4096, 4096) == 0
    assert lib.nvfp4_gemm_select(9, 4, 256, nv.KERNEL_TC) == nv.KERNEL_TC
    assert lib.nvfp4_gemm_select(9, 4, 256, nv.KERNEL_AUTO) == -2
    assert lib.nvfp4_gemm_select(33, 4, 256, nv.KERNEL_TC) == -2
    assert lib.nvfp4_gemm_select(4, 4, 272, nv.KERNEL_TC) == -2
