"""GPU parity of the small-M W4A4 GEMM against the oracle's FP64 result.

Operands are quantised by each side independently (the quantisers are
bit-exact, tested separately), then Y from the C ABI is compared with the
oracle's FP64 Y computed from the oracle's own bytes.  Tolerance: GEMM_TOL on
max |y - ref| / max(|ref|, row rms).  Marked gpu."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from helpers import GEMM_TOL, gemm_error, sampled_error

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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def run_both(nv, x, w):
    """(y_gpu, y_oracle, oracle operands) for one linear."""
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    y = nv.gemm_smallm(xq, xs, xg, wq, ws, wg)
    return host(y), ref


SMALL = [(1, 256, 512), (1, 1, 16), (2, 3, 32), (3, 17, 48), (5, 33, 272), (8, 64, 256),
         (4, 100, 4112), (7, 129, 1024), (8, 1000, 4096), (6, 31, 12288 + 16)]


@pytest.mark.parametrize("m,n,k", SMALL)
def test_gemm_small_shapes(nv, m, n, k):
    x = synthetic.activations(m, k, seed=m * 1000 + k)
    w = synthetic.weights(n, k, 0.02, seed=n * 1000 + k)
    y, ref = run_both(nv, x, w)
    assert gemm_error(y, ref) <= GEMM_TOL


@pytest.mark.parametrize("m", range(1, 9))
def test_gemm_every_m_tiles_and_tail(nv, m):
    """Several row tiles plus a ragged row tail, K spanning several tiles."""
    n, k = 16 * 37 + 5, 4096 + 256
    x = synthetic.activations(m, k, seed=m)
    w = synthetic.weights(n, k, 0.02, seed=77)
    y, ref = run_both(nv, x, w)
    assert gemm_error(y, ref) <= GEMM_TOL


def test_gemm_decades_of_scales(nv):
    """Block scales over many decades (subnormal to saturated E4M3)."""
    m, n, k = 4, 96, 2048
    x = synthetic.log_uniform_blocks(m, k, seed=3)
    w = synthetic.log_uniform_blocks(n, k, seed=4)
    y, ref = run_both(nv, x, w)
    assert gemm_error(y, ref) <= GEMM_TOL


def test_gemm_zero_operands(nv):
    m, n, k = 3, 40, 512
    x = np.zeros((m, k), np.float32)
    w = synthetic.weights(n, k, 0.02, seed=5)
    y, ref = run_both(nv, x, w)
    assert not ref.any() and not y.any()
    x = synthetic.activations(m, k, seed=6)
    w[:] = 0
    y, ref = run_both(nv, x, w)
    assert not y.any()


def test_gemm_k_zero_writes_zeros(nv):
    y = torch.full((2, 5), 7.0, device="cuda")
    e8 = torch.empty((2, 0), dtype=torch.uint8, device="cuda")
    w8 = torch.empty((5, 0), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    nv.gemm_smallm(e8, e8, g, w8, w8, g, out=y)
    assert not host(y).any()


def test_gemm_empty_m_leaves_output(nv):
    y = torch.full((0, 5), 7.0, device="cuda")
    xq = torch.empty((0, 16), dtype=torch.uint8, device="cuda")
    xs = torch.empty((0, 2), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((5, 16), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((5, 2), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    nv.gemm_smallm(xq, xs, g, wq, ws, g, out=y)


def test_gemm_m9_unsupported(nv):
    xq = torch.zeros((9, 16), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((9, 2), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((4, 16), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((4, 2), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.gemm_smallm(xq, xs, g, wq, ws, g)
    assert e.value.status == 2


def test_gemm_deterministic_and_no_overrun(nv):
    m, n, k = 8, 24576 // 8, 4096
    x = synthetic.activations(m, k, seed=8)
    w = synthetic.weights(n, k, 0.02, seed=9)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    canary = torch.full((m * n + 1024,), 123.0, device="cuda")
    y1 = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, out=canary[: m * n].view(m, n))
    a = host(y1).copy()
    y2 = nv.gemm_smallm(xq, xs, xg, wq, ws, wg)
    np.testing.assert_array_equal(a, host(y2))
    assert np.all(host(canary[m * n:]) == 123.0)


def full_size_case(nv, m, n, k, std, seed, samples=64):
    """Full-size linear: whole GPU path (the library's choice of kernel and
    the split-K tensor-core kernel, in the launch configuration the benchmark
    uses); the oracle evaluates ``samples`` output rows n (all m) from its own
    quantisation of those rows.  Returns the larger of the two errors."""
    w = synthetic.weights(n, k, std, seed=seed)
    x = synthetic.activations(m, k, seed=seed + 1)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    ys = [host(nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=kern)).copy()
          for kern in (nv.KERNEL_AUTO, nv.KERNEL_SPLITK)]
    del wq, ws
    gx = oracle.global_scale(x)
    gw = oracle.global_scale(w)
    oxq, oxs = oracle.quantize(x, gx)
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, samples - 2)]))
    owq, ows = oracle.quantize(w[rows], gw)
    ref = oracle.gemm(oxq, oxs, gx, owq, ows, gw)        # [m, len(rows)]
    # the row rms of the full output is estimated from the GPU-independent
    # sampled reference
    row_rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    err = max(sampled_error(y[:, rows], ref, row_rms) for y in ys)
    torch.cuda.empty_cache()
    return err


@pytest.mark.parametrize("m", synthetic.M_SWEEP_8B)
@pytest.mark.parametrize("lin", synthetic.LINEARS_8B, ids=lambda l: l.name)
def test_gemm_full_size_8b(nv, lin, m):
    err = full_size_case(nv, m, lin.n, lin.k, synthetic.WEIGHT_STD_8B, seed=lin.n + lin.k)
    assert err <= GEMM_TOL


@pytest.mark.parametrize("m", synthetic.M_SWEEP_32B)
@pytest.mark.parametrize("lin", synthetic.LINEARS_32B, ids=lambda l: l.name)
def test_gemm_full_size_32b(nv, lin, m):
    err = full_size_case(nv, m, lin.n, lin.k, synthetic.WEIGHT_STD_32B, seed=lin.n + 3 * lin.k)
    assert err <= GEMM_TOL


# ---- each kernel through the C ABI --------------------------------------------

# K values cover one and two chunks per thread, 1..4 rows per group, CTAs
# ending in a partial warp (K = 17408, 25600), and row counts that leave the
# last group and the last CTA partial.
GEMV_SHAPES = [(1, 16 * 9 + 3, 2048), (2, 40, 4096), (1, 1, 5120), (2, 333, 6144),
               (1, 70, 8192), (2, 64, 12288), (1, 20, 25600), (2, 5, 10240), (1, 17, 16384),
               (1, 1000, 1024), (2, 77, 3072), (1, 9, 17408), (2, 3, 32768), (2, 2000, 4096)]


@pytest.mark.parametrize("m,n,k", GEMV_SHAPES)
@pytest.mark.parametrize("pdl", [False, True])
def test_gemv_kernel(nv, m, n, k, pdl):
    assert nv.gemm_select(m, n, k, nv.KERNEL_GEMV) == nv.KERNEL_GEMV
    x = synthetic.activations(m, k, seed=k + m)
    w = synthetic.weights(n, k, 0.02, seed=n + k)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg, pdl=pdl)
    y = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_GEMV, pdl=pdl)
    assert gemm_error(host(y), ref) <= GEMM_TOL
    yg = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_GENERIC)
    assert gemm_error(host(yg), ref) <= GEMM_TOL


def test_gemv_rejects_unsupported(nv):
    xq = torch.zeros((3, 2048), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((3, 256), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((4, 2048), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    g = torch.ones(1, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.gemm_smallm(xq, xs, g, wq, ws, g, kernel=nv.KERNEL_GEMV)   # M = 3
    assert e.value.status == 2
    small = [torch.zeros(shape, dtype=torch.uint8, device="cuda")
             for shape in ((1, 8), (1, 1), (4, 8), (4, 1))]
    with pytest.raises(nv.Nvfp4Error):
        nv.gemm_smallm(small[0], small[1], g, small[2], small[3], g,
                       kernel=nv.KERNEL_GEMV)                          # K = 16


def test_pdl_chain_in_graph(nv):
    """quantize -> GEMM pairs with programmatic dependent launch, captured in
    a CUDA graph and replayed, equal the plain launches bit for bit."""
    lin = synthetic.LINEARS_8B
    xs_, ws_, refs = [], [], []
    for j, l in enumerate(lin):
        x = dev(synthetic.activations(1, l.k, seed=50 + j))
        w = nv.pack_weight(dev(synthetic.weights(l.n, l.k, 0.02, seed=60 + j)))
        xs_.append((x, nv.global_scale(x)))
        ws_.append(w)
    outs = [torch.empty((1, l.n), device="cuda") for l in lin]
    plain = []
    for j in range(4):
        xq, xsc = nv.quantize_act(*xs_[j])
        plain.append(nv.gemm_smallm(xq, xsc, xs_[j][1], *ws_[j]))
    bufs = [(torch.empty((1, l.k // 2), dtype=torch.uint8, device="cuda"),
             torch.empty((1, l.k // 16), dtype=torch.uint8, device="cuda")) for l in lin]

    def step():
        for j in range(4):
            nv.quantize_act(*xs_[j], out=bufs[j], pdl=True)
            nv.gemm_smallm(*bufs[j], xs_[j][1], *ws_[j], out=outs[j], pdl=True)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for j in range(4):
        np.testing.assert_array_equal(host(outs[j]), host(plain[j]))


# Tensor-core kernel: every M, K values that take 1..5 cluster ranks and
# 1, 2 or 4 ranges per warp, row counts below one tile, odd tile counts and a
# ragged last tile.
MMA_SHAPES = [(1024, 37), (2048, 5), (4096, 16 * 37 + 5), (5120, 300), (8192, 33),
              (12288, 64), (25600, 21), (6144, 17 * 16)]


@pytest.mark.parametrize("k,n", MMA_SHAPES)
@pytest.mark.parametrize("m", [1, 2, 3, 5, 8])
def test_mma_kernel(nv, m, n, k):
    assert nv.gemm_select(m, n, k, nv.KERNEL_MMA) == nv.KERNEL_MMA
    x = synthetic.activations(m, k, seed=k + 7 * m)
    w = synthetic.weights(n, k, 0.02, seed=n + 3 * k)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    y = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_MMA)
    assert gemm_error(host(y), ref) <= GEMM_TOL
    y2 = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_MMA, pdl=True)
    np.testing.assert_array_equal(host(y2), host(y))


def test_mma_decades_of_scales(nv):
    """Extreme block scales stay exact in the folded FP16 operands."""
    m, n, k = 8, 96, 4096
    x = synthetic.log_uniform_blocks(m, k, seed=13)
    w = synthetic.log_uniform_blocks(n, k, seed=14)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    y = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_MMA)
    assert gemm_error(host(y), ref) <= GEMM_TOL


# TMA-fed tensor-core kernel: every M, one to five cluster ranks, 2..4 ring
# stages, fewer rows than a tile, a ragged last tile, more tiles than ring
# stages per CTA.
TMA_SHAPES = [(512, 37), (1024, 5), (2048, 16 * 70 + 5), (4096, 16 * 37 + 5), (5120, 300),
              (6144, 17 * 16), (8192, 33), (12288, 64), (25600, 21), (4096, 40000)]


@pytest.mark.parametrize("k,n", TMA_SHAPES)
@pytest.mark.parametrize("m", [1, 2, 4, 8])
def test_tma_kernel(nv, m, n, k):
    assert nv.gemm_select(m, n, k, nv.KERNEL_TMA) == nv.KERNEL_TMA
    x = synthetic.activations(m, k, seed=k + 11 * m)
    w = synthetic.weights(n, k, 0.02, seed=n + 5 * k)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    y = host(nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_TMA))
    if n <= 4096:
        ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
        assert gemm_error(y, ref) <= GEMM_TOL
    else:  # many tiles: check a sample of rows (first, last, random)
        rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n).integers(0, n, 62)]))
        ref = oracle.gemm(xq_o, xs_o, gx, wq_o[rows], ws_o[rows], gw)
        rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
        assert sampled_error(y[:, rows], ref, rms) <= GEMM_TOL
    y2 = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_TMA, pdl=True)
    np.testing.assert_array_equal(host(y2), y)
    assert nv.device_status() == 0


def test_tma_bounded_wait_times_out_and_recovers(nv):
    """The test hook makes the first stage wait for bytes that never come:
    the bounded wait runs out, the kernel records the timeout and returns,
    and the context stays usable for a normal launch afterwards."""
    m, n, k = 1, 32, 4096
    x = synthetic.activations(m, k, seed=1)
    w = synthetic.weights(n, k, 0.02, seed=2)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    assert nv.device_status() == 0
    nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_TMA, test_wait_timeout=True)
    assert nv.device_status(clear=True) & nv.DEVICE_WAIT_TIMEOUT
    assert nv.device_status() == 0
    y = host(nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_TMA))
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    assert gemm_error(y, oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)) <= GEMM_TOL
    assert nv.device_status() == 0


# Split-K tensor-core kernel: every M; K of one chunk and of 3..100 chunks,
# including chunk lengths that are not powers of two (1280, 1536) and 17
# chunks of 256 (K = 4352); fewer rows than a tile, ragged last tiles, more
# tiles than warps.
SPLITK_SHAPES = [(256, 5), (512, 37), (1280, 16 * 70 + 5), (4096, 16 * 37 + 5), (4352, 33),
                 (5120, 300), (8192, 33), (12288, 64), (25600, 21), (4096, 40000),
                 (12288, 16 * 300 + 9)]


def splitk_case(nv, m, n, k, seed):
    x = synthetic.activations(m, k, seed=seed)
    w = synthetic.weights(n, k, 0.02, seed=seed + 1)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    return (xq, xs, xg, wq, ws, wg), (xq_o, xs_o, gx, wq_o, ws_o, gw)


def check_rows(y, oracle_ops, n):
    xq_o, xs_o, gx, wq_o, ws_o, gw = oracle_ops
    if n <= 4096:
        ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
        return gemm_error(y, ref)
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n).integers(0, n, 62)]))
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o[rows], ws_o[rows], gw)
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    return sampled_error(y[:, rows], ref, rms)


@pytest.mark.parametrize("k,n", SPLITK_SHAPES)
@pytest.mark.parametrize("m", range(1, 9))
def test_splitk_kernel(nv, m, n, k):
    ops, oops = splitk_case(nv, m, n, k, seed=k + 13 * m + n)
    wsp = nv.workspace(m, n, k, nv.KERNEL_SPLITK)
    assert (wsp is None) == (nv.gemm_workspace_size(m, n, k, nv.KERNEL_SPLITK) == 0)
    y = host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK, workspace=wsp)).copy()
    assert check_rows(y, oops, n) <= GEMM_TOL
    # same workspace again (its counters were reset), with PDL: same bytes
    y2 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK, pdl=True, workspace=wsp)
    np.testing.assert_array_equal(host(y2), y)
    if nv.gemm_select(m, n, k, nv.KERNEL_SPLITK) == nv.KERNEL_SPLITK:
        # without a workspace: K in one chunk, or the cluster form
        y3 = host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK, workspace=False))
        assert check_rows(y3, oops, n) <= GEMM_TOL


# Shapes whose K takes several chunks at that M, so that a call without a
# workspace runs the cluster form (partials summed through distributed shared
# memory): the 8B down at M = 8, the 32B down at M = 4 and M = 8 (100
# sub-items of 256: unequal chunks), a ragged N at M = 3, a 4-tile N, a
# 2500-tile N, M = 2 with K = 32768, M = 7, and 37 sub-items (a prime) at M = 8.
CLUSTER_SHAPES = [(8, 4096, 12288), (4, 5120, 25600), (8, 5120, 25600), (3, 16 * 37 + 5, 16384),
                  (8, 64, 8192), (6, 40000, 8192), (2, 2048, 32768), (7, 1000, 10240),
                  (8, 1000, 256 * 37)]


def gemm_raw(nv, ops, m, n, k, options, ws=None, entry="ws"):
    """One call through the C ABI: nvfp4_gemm_smallm_ws with the given
    workspace tensor (None: no workspace), or the plain nvfp4_gemm_smallm."""
    lib = nv.library()
    y = torch.full((m, n), float("nan"), device="cuda")
    ptrs = [t.data_ptr() for t in ops[:6]]
    st = torch.cuda.current_stream().cuda_stream
    if entry == "plain":
        status = lib.nvfp4_gemm_smallm(*ptrs, y.data_ptr(), m, n, k, st)
    else:
        status = lib.nvfp4_gemm_smallm_ws(*ptrs, y.data_ptr(), m, n, k, options,
                                          ws.data_ptr() if ws is not None else None,
                                          ws.numel() if ws is not None else 0, st)
    return status, y


@pytest.mark.parametrize("m,n,k", CLUSTER_SHAPES)
def test_splitk_cluster_form_without_workspace(nv, m, n, k):
    """Without a workspace (or with one too small for any split) the split-K
    kernel still takes a K of several chunks, in its cluster form: results
    within the tolerance of the oracle's FP64 sum, the same bits on every
    call (fixed chunk order), with PDL, with a too-small workspace, and
    through the plain boundary call, which selects it."""
    assert m * k * 2 > 65536                      # more than one chunk
    assert nv.gemm_select(m, n, k, nv.KERNEL_SPLITK) == nv.KERNEL_SPLITK
    assert nv.gemm_select(m, n, k) == nv.KERNEL_SPLITK
    ops, oops = splitk_case(nv, m, n, k, seed=3 * m + n + k)
    SPLITK = nv.KERNEL_SPLITK
    st, y = gemm_raw(nv, ops, m, n, k, SPLITK)
    assert st == 0
    yh = host(y).copy()
    assert check_rows(yh, oops, n) <= GEMM_TOL
    st, y2 = gemm_raw(nv, ops, m, n, k, SPLITK | nv.FLAG_PDL)
    assert st == 0
    np.testing.assert_array_equal(host(y2), yh)
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")   # too small for any split
    st, y3 = gemm_raw(nv, ops, m, n, k, SPLITK, ws=small)
    assert st == 0
    np.testing.assert_array_equal(host(y3), yh)
    st, y4 = gemm_raw(nv, ops, m, n, k, 0, entry="plain")
    assert st == 0
    np.testing.assert_array_equal(host(y4), yh)
    # with the workspace the plan asks for (if any): the same plan when that
    # is a cluster plan, else the workspace form, within the tolerance
    yw = host(nv.gemm_smallm(*ops, kernel=SPLITK))
    if nv.gemm_workspace_size(m, n, k, SPLITK) == 0:
        np.testing.assert_array_equal(yw, yh)
    assert check_rows(yw, oops, n) <= GEMM_TOL
    assert nv.device_status() == 0


def test_splitk_cluster_form_in_a_graph(nv):
    """The cluster form replayed from a CUDA graph, twice: same bits as the
    eager call."""
    m, n, k = 8, 4096, 12288
    ops, oops = splitk_case(nv, m, n, k, seed=17)
    st, y = gemm_raw(nv, ops, m, n, k, nv.KERNEL_SPLITK)
    assert st == 0
    ref = host(y).copy()
    assert check_rows(ref, oops, n) <= GEMM_TOL
    yg = torch.empty((m, n), device="cuda")
    lib = nv.library()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            assert lib.nvfp4_gemm_smallm_ws(*[t.data_ptr() for t in ops[:6]], yg.data_ptr(), m,
                                            n, k, nv.KERNEL_SPLITK | nv.FLAG_PDL, None, 0,
                                            s.cuda_stream) == 0
    for _ in range(2):
        yg.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        np.testing.assert_array_equal(host(yg), ref)


def test_splitk_workspace_shared_across_shapes(nv):
    """One workspace, sized for the largest, serves a sequence of shapes and
    orders (every call leaves its counters at zero); results equal those of
    fresh workspaces.  K = 40960 at M = 8 needs more chunks than one cluster
    holds, so its partials go through the workspace."""
    shapes = [(8, 6144, 4096), (8, 512, 40960), (1, 4096, 12288), (4, 5120, 25600),
              (8, 512, 40960), (8, 6144, 4096)]
    assert nv.gemm_workspace_size(8, 512, 40960, nv.KERNEL_SPLITK) > 0
    cases = [splitk_case(nv, m, n, k, seed=40 + i)[0] for i, (m, n, k) in enumerate(shapes)]
    size = max(nv.gemm_workspace_size(m, n, k, nv.KERNEL_SPLITK) for m, n, k in shapes)
    shared = torch.zeros(size, dtype=torch.uint8, device="cuda")
    got = [host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK, workspace=shared)).copy()
           for ops in cases]
    for ops, g in zip(cases, got):
        np.testing.assert_array_equal(host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK)), g)


def test_splitk_decades_of_scales(nv):
    """Extreme block scales stay exact in the folded FP16 operands (weights and
    activations drawn block by block over many decades)."""
    m, n, k = 8, 96, 8192
    x = synthetic.log_uniform_blocks(m, k, seed=23)
    w = synthetic.log_uniform_blocks(n, k, seed=24)
    gx = oracle.global_scale(x)
    xq_o, xs_o = oracle.quantize(x, gx)
    wq_o, ws_o, gw = oracle.pack_weight(w)
    ref = oracle.gemm(xq_o, xs_o, gx, wq_o, ws_o, gw)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq, xs = nv.quantize_act(xd, xg)
    y = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_SPLITK)
    assert gemm_error(host(y), ref) <= GEMM_TOL


def test_splitk_graph_chain_with_pdl(nv):
    """The four 8B linears at M = 8 as split-K calls with PDL, captured in a
    graph on one shared workspace, replay to the eager results."""
    lin = synthetic.LINEARS_8B
    cases = [splitk_case(nv, 8, l.n, l.k, seed=90 + j)[0] for j, l in enumerate(lin)]
    size = max(nv.gemm_workspace_size(8, l.n, l.k, nv.KERNEL_SPLITK) for l in lin)
    shared = torch.zeros(size, dtype=torch.uint8, device="cuda")
    outs = [torch.empty((8, l.n), device="cuda") for l in lin]
    eager = [host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK)).copy() for ops in cases]

    def step():
        for j, ops in enumerate(cases):
            nv.gemm_smallm(*ops, out=outs[j], kernel=nv.KERNEL_SPLITK, pdl=True, workspace=shared)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    for j in range(4):
        np.testing.assert_array_equal(host(outs[j]), eager[j])


# ---- BF16 output -----------------------------------------------------------------

# Tolerance of a BF16 output against the oracle's FP64 result: the FP32 result
# is within GEMM_TOL (relative to max(|ref|, row rms)), and rounding it to BF16
# (8 significant bits: for |y| in [2^e, 2^(e+1)) the spacing is 2^(e-7), so
# round to nearest moves y by at most 2^(e-8) <= 2^-8 |y|) adds at most
# 2^-8 |y|, with |y| <= (1 + GEMM_TOL) max(|ref|, rms).
GEMM_TOL_BF16 = GEMM_TOL + 2.0 ** -8 * (1 + GEMM_TOL)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("kernel,m,n,k", [("generic", 3, 100, 4112), ("gemv", 1, 333, 4096),
                                          ("gemv", 2, 64, 12288), ("splitk", 1, 300, 4096),
                                          ("splitk", 8, 16 * 37 + 5, 4096),
                                          ("splitk", 4, 200, 25600), ("mma", 5, 300, 5120),
                                          ("tma", 8, 16 * 70 + 5, 2048)])
def test_bf16_output_is_rounded_fp32_output(nv, kernel, m, n, k):
    """Y in BF16 is the same kernel's FP32 Y rounded to nearest even (bit for
    bit, the oracle's rounding), and within GEMM_TOL_BF16 of the FP64 result."""
    kid = {"generic": nv.KERNEL_GENERIC, "gemv": nv.KERNEL_GEMV, "splitk": nv.KERNEL_SPLITK,
           "mma": nv.KERNEL_MMA, "tma": nv.KERNEL_TMA}[kernel]
    ops, oops = splitk_case(nv, m, n, k, seed=k + 17 * m + n)
    wsp = nv.workspace(m, n, k, kid) if kid == nv.KERNEL_SPLITK else None
    y32 = host(nv.gemm_smallm(*ops, kernel=kid, workspace=wsp)).copy()
    y16 = nv.gemm_smallm(*ops, kernel=kid, workspace=wsp, out_dtype=torch.bfloat16)
    assert y16.dtype == torch.bfloat16
    np.testing.assert_array_equal(bf16_bits(y16), oracle.f32_to_bf16(y32))
    yw = oracle.bf16_to_f32(bf16_bits(y16))
    assert check_rows(yw, oops, n) <= GEMM_TOL_BF16


def test_bf16_static_entry_point(nv):
    m, n, k = 8, 6144, 4096
    ops, _ = splitk_case(nv, m, n, k, seed=77)
    y32 = host(nv.gemm_smallm(*ops, kernel=nv.KERNEL_SPLITK)).copy()
    y16 = nv.gemm_smallm_static(*ops, out_dtype=torch.bfloat16)
    np.testing.assert_array_equal(bf16_bits(y16), oracle.f32_to_bf16(y32))


@pytest.mark.parametrize("m,n,k", [(1, 256, 1024), (2, 1000, 4096), (4, 96, 4096), (8, 50, 12288)])
@pytest.mark.parametrize("fused", [False, True])
def test_linear_bf16_in_and_out(nv, m, n, k, fused):
    """BF16 X in, BF16 Y out through nvfp4_linear equals BF16 quantise +
    GEMM with BF16 output (the fused form falls back to two launches)."""
    x32 = synthetic.activations(m, k, seed=5 * k + m)
    bits = oracle.f32_to_bf16(x32)
    xb = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    xg = nv.global_scale(torch.from_numpy(oracle.bf16_to_f32(bits)).cuda())
    w = synthetic.weights(n, k, 0.02, seed=7 * n + k)
    wq, ws, wg = nv.pack_weight(dev(w))
    wsp = nv.workspace(m, n, k)
    y = nv.linear(xb, xg, wq, ws, wg, fused=fused, workspace=wsp, out_dtype=torch.bfloat16)
    xq, xs = nv.quantize_act(xb, xg)
    y2 = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, workspace=wsp, out_dtype=torch.bfloat16)
    np.testing.assert_array_equal(bf16_bits(y), bf16_bits(y2))
    gx = np.float32(host(xg)[0])
    oxq, oxs = oracle.quantize(oracle.bf16_to_f32(bits), gx)
    np.testing.assert_array_equal(host(xq), oxq)
    owq, ows, ogw = oracle.pack_weight(w)
    ref = oracle.gemm(oxq, oxs, gx, owq, ows, ogw)
    assert gemm_error(oracle.bf16_to_f32(bf16_bits(y)), ref) <= GEMM_TOL_BF16


# ---- fused quantise + GEMM (nvfp4_linear) --------------------------------------

LINEAR_SHAPES = [(1, 256, 1024), (2, 1000, 4096), (1, 16 * 37 + 5, 4096), (2, 77, 12288),
                 (1, 20, 25600), (1, 64, 8192), (4, 96, 4096), (8, 50, 4096), (3, 40, 512)]


@pytest.mark.parametrize("m,n,k", LINEAR_SHAPES)
@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("fused", [False, True])
def test_linear_matches_two_step_and_oracle(nv, m, n, k, pdl, fused):
    """The fused kernel writes the same activation bytes as the quantiser and
    the same Y as quantise + GEMM; both within tolerance of the oracle."""
    x = synthetic.activations(m, k, seed=3 * k + m)
    w = synthetic.weights(n, k, 0.02, seed=5 * n + k)
    xd = dev(x)
    xg = nv.global_scale(xd)
    wq, ws, wg = nv.pack_weight(dev(w))
    xq = torch.full((m, k // 2), 0xAB, dtype=torch.uint8, device="cuda")
    xs = torch.full((m, k // 16), 0xAB, dtype=torch.uint8, device="cuda")
    y = nv.linear(xd, xg, wq, ws, wg, x_out=(xq, xs), pdl=pdl, fused=fused)
    xq2, xs2 = nv.quantize_act(xd, xg)
    y2 = nv.gemm_smallm(xq2, xs2, xg, wq, ws, wg)
    np.testing.assert_array_equal(host(xq), host(xq2))
    np.testing.assert_array_equal(host(xs), host(xs2))
    np.testing.assert_array_equal(host(y), host(y2))
    gx = oracle.global_scale(x)
    oxq, oxs = oracle.quantize(x, gx)
    owq, ows, ogw = oracle.pack_weight(w)
    np.testing.assert_array_equal(host(xq), oxq)
    assert gemm_error(host(y), oracle.gemm(oxq, oxs, gx, owq, ows, ogw)) <= GEMM_TOL


def test_linear_pdl_graph_step(nv):
    """A captured decode-style chain of fused linears equals eager launches."""
    lin = synthetic.LINEARS_8B
    ins, ws_, outs, bufs = [], [], [], []
    for j, l in enumerate(lin):
        x = dev(synthetic.activations(1, l.k, seed=70 + j))
        ins.append((x, nv.global_scale(x)))
        ws_.append(nv.pack_weight(dev(synthetic.weights(l.n, l.k, 0.02, seed=80 + j))))
        outs.append(torch.empty((1, l.n), device="cuda"))
        bufs.append((torch.empty((1, l.k // 2), dtype=torch.uint8, device="cuda"),
                     torch.empty((1, l.k // 16), dtype=torch.uint8, device="cuda")))
    eager = [host(nv.linear(ins[j][0], ins[j][1], *ws_[j])).copy() for j in range(4)]

    def step():
        for j in range(4):
            nv.linear(ins[j][0], ins[j][1], *ws_[j], out=outs[j], x_out=bufs[j], pdl=True,
                      fused=(j % 2 == 0))

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    g.replay()
    for j in range(4):
        np.testing.assert_array_equal(host(outs[j]), eager[j])
