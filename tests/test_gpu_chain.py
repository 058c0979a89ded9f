"""GPU parity of the multi-linear entry points (nvfp4_linear_chain,
nvfp4_gemm_chain) on the CUDA-core stream (NVFP4_KERNEL_GEMV; the
tensor-core engine is covered in test_gpu_tc.py): every linear's activation
codes bit-exact with the
oracle's, every Y equal bit for bit to the single-linear CUDA-core kernel
(NVFP4_KERNEL_GEMV) on the same codes and within GEMM_TOL of the oracle's FP64
result.  Lists cover every compiled CTA width (rows of K <= 8192 / 12288 /
16384 / 32768), ragged row counts (n = 1, fewer rows than a group, a partial
last group), CTAs that own no rows, more linears than one launch takes, BF16
in and out, and replay in a CUDA graph.  Marked gpu."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import GEMM_TOL, gemm_error

pytestmark = pytest.mark.gpu

GEMM_TOL_BF16 = GEMM_TOL + 2.0 ** -8 * (1 + GEMM_TOL)


@pytest.fixture(scope="module")
def nv():
    import nvfp4_w4a4_decode_gb300 as nvmod
    from nvfp4_w4a4_decode_gb300 import build as nvbuild
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    nvbuild.build()
    oracle.build()
    nvmod.library()
    return nvmod


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def make_linears(nv, m, shapes, seed, x_bf16=False, y_bf16=False):
    """Host operands and device tensors of a list of linears; X, W seeded per
    linear, the GPU packs W and calibrates gX itself."""
    out = []
    for i, (n, k) in enumerate(shapes):
        x32 = synthetic.activations(m, k, seed=seed + 2 * i)
        w = synthetic.weights(n, k, 0.02, seed=seed + 2 * i + 1)
        if x_bf16:
            bits = oracle.f32_to_bf16(x32)
            x_host = oracle.bf16_to_f32(bits)
            xd = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
        else:
            x_host = x32
            xd = dev(x32)
        xg = nv.global_scale(dev(x_host))
        wq, ws, wg = nv.pack_weight(dev(w))
        xq = torch.full((m, k // 2), 0xAB, dtype=torch.uint8, device="cuda")
        xs = torch.full((m, k // 16), 0xAB, dtype=torch.uint8, device="cuda")
        y = torch.full((m, n), float("nan"), device="cuda",
                       dtype=torch.bfloat16 if y_bf16 else torch.float32)
        out.append({"x_host": x_host, "w": w, "xd": xd, "xg": xg, "codes": (xq, xs),
                    "packed": (wq, ws, wg), "y": y, "n": n, "k": k})
    return out


def chain_of(nv, lins):
    """The chain on the CUDA-core stream (the engine these tests cover)."""
    return nv.Chain([(L["xd"], L["xg"], L["codes"], L["packed"], L["y"]) for L in lins],
                    kernel=nv.KERNEL_GEMV)


def check_against_oracle_and_gemv(nv, lins, m, y_bf16=False):
    for L in lins:
        gx = oracle.global_scale(L["x_host"])
        assert np.float32(L["xg"].item()) == gx
        oxq, oxs = oracle.quantize(L["x_host"], gx)
        xq, xs = L["codes"]
        np.testing.assert_array_equal(xq.cpu().numpy(), oxq)
        np.testing.assert_array_equal(xs.cpu().numpy(), oxs)
        wq, ws, wg = L["packed"]
        y_gemv = nv.gemm_smallm(xq, xs, L["xg"], wq, ws, wg, kernel=nv.KERNEL_GEMV,
                                out_dtype=torch.bfloat16 if y_bf16 else torch.float32)
        torch.cuda.synchronize()
        if y_bf16:
            np.testing.assert_array_equal(bf16_bits(L["y"]), bf16_bits(y_gemv))
            y = oracle.bf16_to_f32(bf16_bits(L["y"]))
        else:
            np.testing.assert_array_equal(L["y"].cpu().numpy(), y_gemv.cpu().numpy())
            y = L["y"].cpu().numpy()
        owq, ows, ogw = oracle.pack_weight(L["w"])
        ref = oracle.gemm(oxq, oxs, gx, owq, ows, ogw)
        assert gemm_error(y, ref) <= (GEMM_TOL_BF16 if y_bf16 else GEMM_TOL)


# (n, k) lists: one per compiled CTA width; ragged and tiny row counts
CHAINS = {
    "k4096": [(300, 4096), (1, 4096), (5, 1024), (4096, 4096), (77, 2048), (1000, 8192)],
    "k12288": [(700, 4096), (3, 12288), (1500, 4096), (400, 12288), (2, 1024), (6144, 4096)],
    "k16384": [(33, 16384), (100, 4096), (1, 16384), (257, 1024)],
    "k32768": [(17, 32768), (100, 25600), (64, 5120), (3, 1024), (90, 8192)],
}


@pytest.mark.parametrize("name", sorted(CHAINS))
@pytest.mark.parametrize("m", [1, 2])
def test_linear_chain_matches_gemv_and_oracle(nv, name, m):
    lins = make_linears(nv, m, CHAINS[name], seed=100 * m + len(name))
    ch = chain_of(nv, lins)
    ch.run()
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(nv, lins, m)


@pytest.mark.parametrize("m", [1, 2])
def test_gemm_chain_reads_given_codes(nv, m):
    """nvfp4_gemm_chain uses the codes already in x_q / x_s (written here by
    the stand-alone quantiser) and never reads x."""
    lins = make_linears(nv, m, CHAINS["k12288"], seed=7 + m)
    for L in lins:
        nv.quantize_act(L["xd"], L["xg"], out=L["codes"])
        L["xd"].fill_(float("nan"))     # would poison the codes if it were read
    ch = chain_of(nv, lins)
    ch.gemm_only(pdl=True)
    torch.cuda.synchronize()
    for L in lins:
        L["xd"].copy_(dev(L["x_host"]))
    check_against_oracle_and_gemv(nv, lins, m)


@pytest.mark.parametrize("m", [1, 2])
def test_linear_chain_bf16_in_and_out(nv, m):
    lins = make_linears(nv, m, CHAINS["k12288"], seed=31 + m, x_bf16=True, y_bf16=True)
    ch = chain_of(nv, lins)
    ch.run(pdl=True)
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(nv, lins, m, y_bf16=True)


def test_linear_chain_longer_than_one_launch(nv):
    """300 linears: two launch pairs; small shapes so that the oracle is quick."""
    shapes = [(3 + (i * 37) % 200, 1024 * (1 + i % 3)) for i in range(300)]
    lins = make_linears(nv, 1, shapes, seed=900)
    ch = chain_of(nv, lins)
    ch.run(pdl=True)
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(nv, lins, 1)


def test_linear_chain_fewer_rows_than_ctas(nv):
    """Three one-row linears: most CTAs own no group."""
    lins = make_linears(nv, 1, [(1, 4096), (1, 1024), (1, 12288)], seed=5)
    chain_of(nv, lins).run()
    torch.cuda.synchronize()
    check_against_oracle_and_gemv(nv, lins, 1)


def test_linear_chain_graph_replay(nv):
    """Captured in a CUDA graph with PDL and replayed twice: equal to the eager
    call bit for bit."""
    lins = make_linears(nv, 1, CHAINS["k12288"], seed=44)
    ch = chain_of(nv, lins)
    ch.run()
    torch.cuda.synchronize()
    eager = [L["y"].cpu().numpy().copy() for L in lins]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ch.run(pdl=True)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ch.run(pdl=True)
    for L in lins:
        L["y"].fill_(float("nan"))
        L["codes"][0].fill_(0xCD)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for L, e in zip(lins, eager):
        np.testing.assert_array_equal(L["y"].cpu().numpy(), e)


def test_linear_chain_full_size_8b_layer(nv):
    """The four 8B-shaped linears of one decode layer at M = 1 in one chain,
    full size: sampled rows against the oracle, all rows against the
    single-linear kernel."""
    lins = make_linears(nv, 1, [(l.n, l.k) for l in synthetic.LINEARS_8B], seed=321)
    chain_of(nv, lins).run(pdl=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    for L in lins:
        gx = oracle.global_scale(L["x_host"])
        oxq, oxs = oracle.quantize(L["x_host"], gx)
        np.testing.assert_array_equal(L["codes"][0].cpu().numpy(), oxq)
        wq, ws, wg = L["packed"]
        y_gemv = nv.gemm_smallm(*L["codes"], L["xg"], wq, ws, wg, kernel=nv.KERNEL_GEMV)
        y = L["y"].cpu().numpy()
        np.testing.assert_array_equal(y, y_gemv.cpu().numpy())
        rows = np.unique(np.concatenate([[0, L["n"] - 1], rng.integers(0, L["n"], 62)]))
        gw = oracle.global_scale(L["w"])
        owq, ows = oracle.quantize(L["w"][rows], gw)
        ref = oracle.gemm(oxq, oxs, gx, owq, ows, gw)   # [1, sampled rows]
        assert gemm_error(y[:, rows], ref) <= GEMM_TOL


def _raw_chain(nv, descs, m, options=0):
    arr = (nv.ChainLinear * len(descs))(*descs)
    return nv.library().nvfp4_linear_chain(ctypes.cast(arr, ctypes.c_void_p), len(descs), m,
                                           options | nv.KERNEL_GEMV,
                                           torch.cuda.current_stream().cuda_stream)


def test_linear_chain_refusals_launch_nothing(nv):
    lins = make_linears(nv, 1, [(64, 4096), (32, 1024)], seed=3)
    descs = []
    for L in lins:
        xq, xs = L["codes"]
        wq, ws, wg = L["packed"]
        descs.append(nv.ChainLinear(L["xd"].data_ptr(), L["xg"].data_ptr(), xq.data_ptr(),
                                    xs.data_ptr(), wq.data_ptr(), ws.data_ptr(), wg.data_ptr(),
                                    L["y"].data_ptr(), L["n"], L["k"]))
    assert _raw_chain(nv, descs, 3) == 2                     # M = 3: not the CUDA-core stream
    assert _raw_chain(nv, descs, 9) == 2
    bad = nv.ChainLinear(*[getattr(descs[1], f) for f, _ in nv.ChainLinear._fields_])
    bad.k = 512                                              # K not a multiple of 1024
    assert _raw_chain(nv, [descs[0], bad], 1) == 2
    bad.k = 1024
    bad.w_q = descs[1].w_q + 16                              # misaligned codes
    assert _raw_chain(nv, [descs[0], bad], 1) == 1
    bad.w_q = descs[1].w_q
    bad.y = 0                                                # null output
    assert _raw_chain(nv, [descs[0], bad], 1) == 1
    assert _raw_chain(nv, descs, 1, options=0x10000) == 1    # unknown option
    assert nv.library().nvfp4_linear_chain(                   # a kernel no chain runs on
        ctypes.cast((nv.ChainLinear * 2)(*descs), ctypes.c_void_p), 2, 1, nv.KERNEL_SPLITK,
        torch.cuda.current_stream().cuda_stream) == 2
    torch.cuda.synchronize()
    for L in lins:                                           # nothing was launched
        assert np.isnan(L["y"].cpu().numpy()).all()
        assert (L["codes"][0].cpu().numpy() == 0xAB).all()
    zero = nv.ChainLinear(*[getattr(descs[1], f) for f, _ in nv.ChainLinear._fields_])
    zero.n = 0                                               # an empty linear is skipped
    assert _raw_chain(nv, [zero], 1) == 0
    torch.cuda.synchronize()
    assert (lins[1]["codes"][0].cpu().numpy() == 0xAB).all()
