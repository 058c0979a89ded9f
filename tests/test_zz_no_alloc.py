"""The allocation-free GEMM entry point (nvfp4_gemm_smallm_static): the
split-K kernel on the library's static scratch array.  Two calls in a row give
the same bits as the workspace entry point with a freshly zeroed workspace of
the size it asks for (same plan, same fixed reduction order); a shape whose
scratch exceeds the array is refused without a launch.  Collected last (file
name), and passes alone or after the other tests.  Marked gpu."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import GEMM_TOL, gemm_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_w4a4_decode_gb300 as nvmod
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nvbuild.build()
    oracle.build()
    nvmod.library()
    return nvmod


def operands(nv, m, n, k, seed):
    x = synthetic.activations(m, k, seed=seed)
    w = synthetic.weights(n, k, 0.02, seed=seed + 1)
    xd = torch.from_numpy(x).cuda()
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(torch.from_numpy(w).cuda())
    xq, xs = nv.quantize_act(xd, xg)
    return (xq, xs, xg, wq, ws, wg), x, w


# a few tiles, the 8B qkv at M = 8, the 8B down at M = 1, the 32B down at
# M = 4 (K of 1 to 25600 / 256 chunks, whatever the plan picks), a shape whose
# plan keeps K in one chunk (the scratch is not touched), and K = 40960 at
# M = 8 (more chunks than one cluster holds: the partials go through the
# scratch)
SHAPES = [(3, 300, 4096), (8, 6144, 4096), (1, 4096, 12288), (4, 5120, 25600), (2, 40000, 1024),
          (8, 512, 40960)]


@pytest.mark.parametrize("m,n,k", SHAPES)
def test_static_twice_equals_workspace_entry_point(nv, m, n, k):
    ops, x, w = operands(nv, m, n, k, seed=7 * m + k)
    need = nv.gemm_workspace_size(m, n, k, nv.KERNEL_SPLITK)
    assert need <= nv.library().nvfp4_gemm_static_scratch_bytes()
    fresh = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    ref = nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK, workspace=fresh if need else None)
    y1 = nv.gemm_smallm_static(*ops)
    y2 = nv.gemm_smallm_static(*ops, pdl=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y1.cpu().numpy(), ref.cpu().numpy())
    np.testing.assert_array_equal(y2.cpu().numpy(), ref.cpu().numpy())
    if n <= 1024:  # and against the oracle's FP64 result
        gx = oracle.global_scale(x)
        oxq, oxs = oracle.quantize(x, gx)
        owq, ows, ogw = oracle.pack_weight(w)
        assert gemm_error(y1.cpu().numpy(), oracle.gemm(oxq, oxs, gx, owq, ows, ogw)) <= GEMM_TOL


def test_static_refuses_scratch_beyond_its_size(nv):
    m, n, k = 8, 200_000, 8192
    need = nv.gemm_workspace_size(m, n, k, nv.KERNEL_SPLITK)
    assert need > nv.library().nvfp4_gemm_static_scratch_bytes()
    q = torch.zeros(16, dtype=torch.uint8, device="cuda")      # never read: refused first
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    y = torch.full((4,), 7.0, device="cuda")
    st = nv.library().nvfp4_gemm_smallm_static(
        q.data_ptr(), q.data_ptr(), g.data_ptr(), q.data_ptr(), q.data_ptr(), g.data_ptr(),
        y.data_ptr(), m, n, k, nv.KERNEL_SPLITK, torch.cuda.current_stream().cuda_stream)
    assert st == 2
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 7.0).all()


def test_static_allocates_no_device_memory(nv):
    """Free device memory (cudaMemGetInfo, which sees every allocation on the
    device, not only torch's) is unchanged by repeated calls once the first
    call has looked up the scratch address; the shape here needs the scratch
    (its split-K plan cuts K into more chunks than one cluster holds)."""
    m, n, k = 8, 512, 40960
    assert nv.gemm_workspace_size(m, n, k, nv.KERNEL_SPLITK) > 0
    ops, _, _ = operands(nv, m, n, k, seed=11)
    y = torch.empty((m, n), device="cuda")
    lib = nv.library()
    st = torch.cuda.current_stream().cuda_stream

    def call():
        xq, xs, xg, wq, ws, wg = ops
        return lib.nvfp4_gemm_smallm_static(
            xq.data_ptr(), xs.data_ptr(), xg.data_ptr(), wq.data_ptr(), ws.data_ptr(),
            wg.data_ptr(), y.data_ptr(), m, n, k, nv.KERNEL_SPLITK, st)

    assert call() == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(20):
        assert call() == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
