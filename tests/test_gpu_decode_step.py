"""The decode step exactly as the benchmark times it, against the oracle.

``bench.DecodeStack`` builds the step: layers of the four 8B-shaped linears
(full size, distinct weights per layer), replayed as one CUDA graph with
programmatic dependent launch, in both of its forms --
* ``launches``: one nvfp4_linear call per linear, one (x_q, x_s) pair per
  linear shape shared by all layers, one workspace shared by all calls (the
  next linear's quantiser overwrites the codes the previous layer's GEMM of
  that shape read, which is safe only through the launches' ordering);
* ``chain``: all linears as one nvfp4_linear_chain call (the tensor-core
  kernel, the library's choice, at M up to 32, on the row-major packed
  weights or on a tile-major repack; the CUDA-core stream by request at
  M <= 2).
The step is replayed twice after its outputs are poisoned; then every
layer's tensor scales and codes are compared bit for bit with the oracle's
(for the shared buffers: the last layer's), and sampled rows of every Y (all
M columns) with the oracle's FP64 result from its own quantisation.  Here at
3 layers instead of the step's 36.  Marked gpu."""
import numpy as np
import pytest
import torch

import bench
import oracle
from helpers import GEMM_TOL, sampled_error

pytestmark = pytest.mark.gpu

GEMM_TOL_BF16 = GEMM_TOL + 2.0 ** -8 * (1 + GEMM_TOL)
LAYERS = 3


@pytest.fixture(scope="module")
def nv():
    import nvfp4_w4a4_decode_gb300 as nvmod
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nvbuild.build()
    oracle.build()
    nvmod.library()
    return nvmod


def host_f32(t):
    if t.dtype == torch.bfloat16:
        return oracle.bf16_to_f32(t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


# (mode, M, BF16 I/O, engine of the chain: library's choice or the tensor cores)
CASES = [("launches", 1, False, "auto"), ("launches", 8, False, "auto"),
         ("launches", 1, True, "auto"), ("launches", 8, True, "auto"),
         ("chain", 1, False, "auto"), ("chain", 2, False, "auto"), ("chain", 1, True, "auto"),
         ("chain", 8, False, "auto"), ("chain", 8, True, "auto"), ("chain", 32, False, "auto"),
         ("chain", 1, False, "tiled"), ("chain", 8, True, "tiled"),
         ("chain", 1, False, "gemv"), ("chain", 2, True, "gemv")]


@pytest.mark.parametrize("mode,m,bf16,engine", CASES,
                         ids=[f"{c[0]}-{c[3]}-m{c[1]}-{'bf16' if c[2] else 'fp32'}" for c in CASES])
def test_decode_step_graph_matches_oracle(nv, mode, m, bf16, engine):
    stack = bench.DecodeStack(nv, torch, m=m, layers=LAYERS, pdl=True, fused=False, bf16=bf16,
                              mode=mode,
                              chain_kernel=nv.KERNEL_GEMV if engine == "gemv" else nv.KERNEL_AUTO,
                              tiled=engine == "tiled")
    g = stack.capture(stack.step)
    stack.y_flat.fill_(float("nan"))
    for l in range(LAYERS):
        for j in range(4):
            stack.codes(l, j)[0].fill_(0xEE)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    rng = np.random.default_rng(m)
    tol = GEMM_TOL_BF16 if bf16 else GEMM_TOL
    for l in range(LAYERS):
        for j, lin in enumerate(stack.lins):
            x = host_f32(stack.x[l][j])
            gx = oracle.global_scale(x)
            assert np.float32(stack.xg[l][j].item()) == gx
            oxq, oxs = oracle.quantize(x, gx)
            if mode == "chain" or l == LAYERS - 1:
                xq, xs = stack.codes(l, j)
                np.testing.assert_array_equal(xq.cpu().numpy(), oxq)
                np.testing.assert_array_equal(xs.cpu().numpy(), oxs)
            w = stack.weight_fp32(l, j).cpu().numpy()
            gw = oracle.global_scale(w)
            assert np.float32(stack.w[l][j][2].item()) == gw
            rows = np.unique(np.concatenate([[0, lin.n - 1], rng.integers(0, lin.n, 30)]))
            owq, ows = oracle.quantize(w[rows], gw)
            del w
            ref = oracle.gemm(oxq, oxs, gx, owq, ows, gw)            # [m, len(rows)]
            y = host_f32(stack.y[l][j])
            assert not np.isnan(y).any()
            row_rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
            err = sampled_error(y[:, rows], ref, row_rms)
            assert err <= tol, (l, lin.name, err)
    del stack, g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("m", [1, 8])
def test_overlapped_end_to_end_buffers(nv, m):
    """The benchmark's end-to-end loop in chain mode alternates two device
    buffer sets (two graphs of the same chain call): the second set's step
    gives the same bits as the first on the same inputs, and the loop itself
    (host copies on their own streams, overlapping the neighbouring steps)
    runs and leaves the first set's outputs unchanged."""
    from types import SimpleNamespace
    stack = bench.DecodeStack(nv, torch, m=m, layers=2, pdl=True, fused=False, mode="chain",
                              tiled=True)
    g = stack.capture(stack.step)
    g.replay()
    torch.cuda.synchronize()
    ref = stack.y_flat.clone()
    x2, y2, ch2 = stack.second_buffers()
    assert torch.equal(x2, stack.x_flat)
    y2.fill_(float("nan"))
    ch2.run(pdl=True)
    torch.cuda.synchronize()
    assert torch.equal(y2, ref)
    res = bench.run_e2e(torch, stack, g, SimpleNamespace(warmup=3, steps=6), 1)
    assert res["ms_per_step"] > 0 and res["h2d_bytes_per_step"] == stack.x_flat.numel() * 4
    torch.cuda.synchronize()
    assert torch.equal(stack.y_flat, ref)
    assert nv.device_status() == 0
