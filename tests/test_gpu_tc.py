"""GPU parity of the fifth-generation tensor-core kernel (NVFP4_KERNEL_TC:
tcgen05.mma kind::mxf4nvf4, swap-AB, TMA weight stream) against the oracle.

Single linears through nvfp4_gemm_smallm_ex for M from 1 to 32 (both MMA
widths, 16 and 32, and their edges), row counts below one 128-row tile,
exactly one, one plus one row and ragged; K from one 256-element stage to
25600; lists of linears through nvfp4_linear_chain with this kernel
(activation codes bit-exact with the oracle's, Y within GEMM_TOL of its FP64
result), BF16 in and out, decades of block scales, replay in a CUDA graph,
and the refusals.  Marked gpu."""
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


def oracle_y(x, w):
    gx = oracle.global_scale(x)
    oxq, oxs = oracle.quantize(x, gx)
    owq, ows, ogw = oracle.pack_weight(w)
    return oracle.gemm(oxq, oxs, gx, owq, ows, ogw), (oxq, oxs, gx)


def gpu_operands(nv, x, w):
    xd = dev(x)
    xg = nv.global_scale(xd)
    xq, xs = nv.quantize_act(xd, xg)
    wq, ws, wg = nv.pack_weight(dev(w))
    return xq, xs, xg, wq, ws, wg


M_VALUES = [1, 2, 3, 5, 8, 9, 12, 15, 16, 17, 24, 31, 32]


@pytest.mark.parametrize("m", M_VALUES)
def test_tc_every_m_class(nv, m):
    """Several tiles and a ragged last one, K of 17 stages."""
    n, k = 128 * 3 + 37, 256 * 17
    x = synthetic.activations(m, k, seed=11 * m)
    w = synthetic.weights(n, k, 0.02, seed=7 + m)
    ref, _ = oracle_y(x, w)
    y = nv.gemm_smallm(*gpu_operands(nv, x, w), kernel=nv.KERNEL_TC)
    torch.cuda.synchronize()
    assert gemm_error(y.cpu().numpy(), ref) <= GEMM_TOL


TC_SHAPES = [(1, 1, 256), (3, 127, 512), (8, 128, 4096), (16, 129, 1024), (32, 1, 256),
             (4, 4096, 4096), (8, 300, 12288), (2, 77, 25600), (32, 255, 8192), (20, 640, 5120)]


@pytest.mark.parametrize("m,n,k", TC_SHAPES)
@pytest.mark.parametrize("pdl", [False, True])
def test_tc_shapes(nv, m, n, k, pdl):
    x = synthetic.activations(m, k, seed=m + k)
    w = synthetic.weights(n, k, 0.02, seed=n + 3 * k)
    ref, _ = oracle_y(x, w)
    ops = gpu_operands(nv, x, w)
    y = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC, pdl=pdl)
    torch.cuda.synchronize()
    assert gemm_error(y.cpu().numpy(), ref) <= GEMM_TOL
    y2 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC)          # deterministic
    np.testing.assert_array_equal(y2.cpu().numpy(), y.cpu().numpy())


def test_tc_decades_of_scales(nv):
    """Block scales over many decades (E4M3 subnormal to saturated) on both
    sides: the tensor core applies them as given."""
    m, n, k = 8, 200, 2048
    x = synthetic.log_uniform_blocks(m, k, seed=21)
    w = synthetic.log_uniform_blocks(n, k, seed=22)
    ref, _ = oracle_y(x, w)
    y = nv.gemm_smallm(*gpu_operands(nv, x, w), kernel=nv.KERNEL_TC)
    torch.cuda.synchronize()
    assert gemm_error(y.cpu().numpy(), ref) <= GEMM_TOL


def test_tc_bf16_output(nv):
    m, n, k = 12, 333, 4096
    x = synthetic.activations(m, k, seed=31)
    w = synthetic.weights(n, k, 0.02, seed=32)
    ref, _ = oracle_y(x, w)
    ops = gpu_operands(nv, x, w)
    y32 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC)
    y16 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bf16_bits(y16), oracle.f32_to_bf16(y32.cpu().numpy()))
    assert gemm_error(oracle.bf16_to_f32(bf16_bits(y16)), ref) <= GEMM_TOL_BF16


def make_chain(nv, m, shapes, seed, x_bf16=False, y_bf16=False):
    lins = []
    for i, (n, k) in enumerate(shapes):
        x32 = synthetic.activations(m, k, seed=seed + 2 * i)
        w = synthetic.weights(n, k, 0.02, seed=seed + 2 * i + 1)
        if x_bf16:
            bits = oracle.f32_to_bf16(x32)
            xh = oracle.bf16_to_f32(bits)
            xd = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
        else:
            xh, xd = x32, dev(x32)
        xg = nv.global_scale(dev(xh))
        codes = (torch.full((m, k // 2), 0xAB, dtype=torch.uint8, device="cuda"),
                 torch.full((m, k // 16), 0xAB, dtype=torch.uint8, device="cuda"))
        y = torch.full((m, n), float("nan"), device="cuda",
                       dtype=torch.bfloat16 if y_bf16 else torch.float32)
        lins.append({"xh": xh, "w": w, "entry": (xd, xg, codes, nv.pack_weight(dev(w)), y)})
    return lins


def check_chain(lins, y_bf16=False):
    for L in lins:
        ref, (oxq, oxs, gx) = oracle_y(L["xh"], L["w"])
        xd, xg, (xq, xs), _, y = L["entry"]
        assert np.float32(xg.item()) == gx
        np.testing.assert_array_equal(xq.cpu().numpy(), oxq)
        np.testing.assert_array_equal(xs.cpu().numpy(), oxs)
        yy = oracle.bf16_to_f32(bf16_bits(y)) if y_bf16 else y.cpu().numpy()
        assert gemm_error(yy, ref) <= (GEMM_TOL_BF16 if y_bf16 else GEMM_TOL)


CHAIN_SHAPES = [(300, 4096), (1, 256), (129, 12288), (1000, 1024), (128, 5120), (70, 2048)]


@pytest.mark.parametrize("m", [1, 4, 8, 13, 32])
def test_tc_chain_matches_oracle(nv, m):
    lins = make_chain(nv, m, CHAIN_SHAPES, seed=40 + m)
    ch = nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC)
    ch.run(pdl=True)
    torch.cuda.synchronize()
    check_chain(lins)


def test_tc_chain_bf16_in_and_out(nv):
    lins = make_chain(nv, 8, CHAIN_SHAPES, seed=77, x_bf16=True, y_bf16=True)
    nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC).run()
    torch.cuda.synchronize()
    check_chain(lins, y_bf16=True)


def test_tc_chain_more_than_one_launch(nv):
    """200 small linears: two launch pairs of at most 160."""
    shapes = [(1 + (i * 53) % 300, 256 * (1 + i % 5)) for i in range(200)]
    lins = make_chain(nv, 3, shapes, seed=500)
    nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC).run(pdl=True)
    torch.cuda.synchronize()
    check_chain(lins)


def test_tc_chain_graph_replay_and_status(nv):
    lins = make_chain(nv, 8, CHAIN_SHAPES, seed=90)
    ch = nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC)
    nv.device_status(clear=True)
    ch.run()
    torch.cuda.synchronize()
    eager = [L["entry"][4].cpu().numpy().copy() for L in lins]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ch.run(pdl=True)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ch.run(pdl=True)
    for L in lins:
        L["entry"][4].fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for L, e in zip(lins, eager):
        np.testing.assert_array_equal(L["entry"][4].cpu().numpy(), e)
    assert nv.device_status(clear=True) == 0          # no wait ran out


def test_tc_full_size_8b_layer_m8(nv):
    """The four 8B-shaped linears at M = 8, full size, one chain: sampled rows
    against the oracle."""
    m = 8
    lins = make_chain(nv, m, [(l.n, l.k) for l in synthetic.LINEARS_8B], seed=123)
    nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC).run(pdl=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for L in lins:
        gx = oracle.global_scale(L["xh"])
        oxq, oxs = oracle.quantize(L["xh"], gx)
        np.testing.assert_array_equal(L["entry"][2][0].cpu().numpy(), oxq)
        n = L["w"].shape[0]
        rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 62)]))
        gw = oracle.global_scale(L["w"])
        owq, ows = oracle.quantize(L["w"][rows], gw)
        ref = oracle.gemm(oxq, oxs, gx, owq, ows, gw)
        y = L["entry"][4].cpu().numpy()[:, rows]
        assert gemm_error(y, ref) <= GEMM_TOL


def test_tc_refusals(nv):
    g = torch.ones(1, device="cuda")
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    y = torch.full((40, 4), 7.0, device="cuda")
    lib = nv.library()
    st = torch.cuda.current_stream().cuda_stream

    def call(m, n, k, opts):
        return lib.nvfp4_gemm_smallm_ex(z.data_ptr(), z.data_ptr(), g.data_ptr(), z.data_ptr(),
                                        z.data_ptr(), g.data_ptr(), y.data_ptr(), m, n, k, opts, st)
    assert call(9, 4, 256, nv.KERNEL_AUTO) == 2       # M > 8 only on request
    assert call(33, 4, 256, nv.KERNEL_TC) == 2        # the kernel's limit
    assert call(4, 4, 128, nv.KERNEL_TC) == 2         # K below one stage
    assert call(4, 4, 272, nv.KERNEL_TC) == 2         # K not a multiple of 256
    assert nv.gemm_select(9, 4, 256, nv.KERNEL_TC) == nv.KERNEL_TC
    assert nv.gemm_select(9, 4, 256, nv.KERNEL_AUTO) == -2
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 7.0).all()              # nothing launched


# ---- equal stage shares through a workspace (tiles cut between CTAs) ----------

@pytest.mark.parametrize("m,n,k", [(8, 300, 25600), (1, 1, 25600), (32, 130, 12288),
                                   (4, 4096, 4096), (2, 129, 256)])
def test_tc_split_tiles_deterministic(nv, m, n, k):
    """Few tiles of many stages: every tile is cut between many CTAs (up to
    about 50 partials per tile); the last to arrive sums them in stage order,
    so repeated calls on one workspace give the same bits, and the counters
    are left at zero (a second shape on the same workspace is right too)."""
    x = synthetic.activations(m, k, seed=3 * m + k)
    w = synthetic.weights(n, k, 0.02, seed=n + k)
    ref, _ = oracle_y(x, w)
    ops = gpu_operands(nv, x, w)
    wsp = nv.workspace(m, n, k, nv.KERNEL_TC)
    assert wsp is not None and wsp.numel() == nv.library().nvfp4_chain_workspace_size(m, 0)
    y1 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC, workspace=wsp)
    y2 = nv.gemm_smallm(*ops, kernel=nv.KERNEL_TC, workspace=wsp, pdl=True)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y1.cpu().numpy(), y2.cpu().numpy())
    assert gemm_error(y1.cpu().numpy(), ref) <= GEMM_TOL
    assert not wsp[:1024].any().item()                     # counters back at zero
    x2 = synthetic.activations(3, 1024, seed=5)
    w2 = synthetic.weights(70, 1024, 0.02, seed=6)
    ref2, _ = oracle_y(x2, w2)
    y3 = nv.gemm_smallm(*gpu_operands(nv, x2, w2), kernel=nv.KERNEL_TC, workspace=wsp)
    torch.cuda.synchronize()
    assert gemm_error(y3.cpu().numpy(), ref2) <= GEMM_TOL


def test_tc_without_workspace_tile_shares(nv):
    """The C entry point without a workspace: CTA shares end on tile
    boundaries (no partial sums); same bits as the reduction-free case of a
    chain with a workspace is not required, only the oracle's bound."""
    m, n, k = 8, 1000, 12288
    x = synthetic.activations(m, k, seed=41)
    w = synthetic.weights(n, k, 0.02, seed=42)
    ref, _ = oracle_y(x, w)
    xq, xs, xg, wq, ws, wg = gpu_operands(nv, x, w)
    y = torch.full((m, n), float("nan"), device="cuda")
    st = nv.library().nvfp4_gemm_smallm_ex(
        xq.data_ptr(), xs.data_ptr(), xg.data_ptr(), wq.data_ptr(), ws.data_ptr(), wg.data_ptr(),
        y.data_ptr(), m, n, k, nv.KERNEL_TC, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert gemm_error(y.cpu().numpy(), ref) <= GEMM_TOL


@pytest.mark.parametrize("m", [1, 8])
def test_tc_chain_without_workspace(nv, m):
    lins = make_chain(nv, m, CHAIN_SHAPES, seed=60 + m)
    nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC, workspace=False).run(pdl=True)
    torch.cuda.synchronize()
    check_chain(lins)


# ---- tile-major weights (nvfp4_tile_weight, NVFP4_FLAG_W_TILED) ----------------

def tile_reference(wq, ws, n, k):
    """The tile-major layout written out from its definition (include/nvfp4.h):
    blocks (tile, stage) of 128 rows; row r's chunk c of the stage at chunk
    c XOR (r mod 8); scales 16 bytes a row; rows past n zero."""
    tiles, nst = (n + 127) // 128, k // 256
    rows = tiles * 128
    q = np.zeros((rows, k // 2), np.uint8)
    q[:n] = wq
    s = np.zeros((rows, k // 16), np.uint8)
    s[:n] = ws
    q5 = q.reshape(tiles, 128, nst, 8, 16).transpose(0, 2, 1, 3, 4)   # [t][st][r][c][16]
    tq = np.empty_like(q5)
    for r in range(128):
        for c in range(8):
            tq[:, :, r, c ^ (r & 7)] = q5[:, :, r, c]
    ts = s.reshape(tiles, 128, nst, 16).transpose(0, 2, 1, 3)           # [t][st][r][16]
    return tq.reshape(-1), np.ascontiguousarray(ts).reshape(-1)


@pytest.mark.parametrize("n,k", [(300, 4096), (128, 256), (1, 12288), (129, 512)])
def test_tile_weight_layout(nv, n, k):
    w = synthetic.weights(n, k, 0.02, seed=n + k)
    owq, ows, _ = oracle.pack_weight(w)
    wq, ws, wg = nv.pack_weight(dev(w))
    tw = nv.tile_weight(wq, ws, wg)
    torch.cuda.synchronize()
    rq, rs = tile_reference(owq, ows, n, k)
    np.testing.assert_array_equal(tw.t_q.cpu().numpy(), rq)
    np.testing.assert_array_equal(tw.t_s.cpu().numpy(), rs)


@pytest.mark.parametrize("m,n,k", [(1, 300, 4096), (8, 129, 12288), (32, 640, 5120), (3, 1, 256),
                                   (12, 700, 1024)])
def test_tc_tiled_weights_same_bits(nv, m, n, k):
    """Tile-major weights stay within the oracle's bound, and give the same bits
    as the row-major ones where the same operands reach the same MMAs: every
    row when no tile goes to the stream warps (M > 8, or a single tile); at
    M <= 8 the stream warps' rows are summed on mma.sync in another FP32 order,
    the tcgen05 rows stay the same bits."""
    x = synthetic.activations(m, k, seed=2 * m + k)
    w = synthetic.weights(n, k, 0.02, seed=3 * n + k)
    ref, _ = oracle_y(x, w)
    xq, xs, xg, wq, ws, wg = gpu_operands(nv, x, w)
    y_row = nv.gemm_smallm(xq, xs, xg, wq, ws, wg, kernel=nv.KERNEL_TC)
    tw = nv.tile_weight(wq, ws, wg)
    y_tile = nv.gemm_smallm(xq, xs, xg, tw, None, None)
    torch.cuda.synchronize()
    yt, yr = y_tile.cpu().numpy(), y_row.cpu().numpy()
    if m > 8 or n <= 128:
        np.testing.assert_array_equal(yt, yr)
    else:
        np.testing.assert_array_equal(yt[:, :128], yr[:, :128])   # the first tile: tcgen05
    assert gemm_error(yt, ref) <= GEMM_TOL
    assert gemm_error(yr, ref) <= GEMM_TOL


@pytest.mark.parametrize("m", [1, 8])
def test_tc_chain_tiled_weights(nv, m):
    lins = make_chain(nv, m, CHAIN_SHAPES, seed=70 + m)
    nv.Chain([L["entry"] for L in lins], kernel=nv.KERNEL_TC).run()
    torch.cuda.synchronize()
    rows = [L["entry"][4].cpu().numpy().copy() for L in lins]
    tiled = []
    for L in lins:
        xd, xg, codes, (wq, ws, wg), y = L["entry"]
        y.fill_(float("nan"))
        tiled.append((xd, xg, codes, nv.tile_weight(wq, ws, wg), y))
    ch = nv.Chain(tiled)
    assert ch.tiled
    ch.run(pdl=True)
    torch.cuda.synchronize()
    # (the row-major chain's bits are not expected: with part of the tiles on
    # the stream warps the tcgen05 stages are shared out differently)
    for L, r in zip(lins, rows):
        assert gemm_error(r, oracle_y(L["xh"], L["w"])[0]) <= GEMM_TOL
    check_chain(lins)


# linears whose last tiles go to the stream warps at every M <= 8 (three or
# more tiles), ragged N, one-tile linears that keep all rows on tcgen05, and K
# from one stage (256) to 48 stages
STREAM_SHAPES = [(300, 4096), (640, 256), (1000, 12288), (128, 512), (5 * 128 + 7, 1024),
                 (3 * 128, 2048)]


@pytest.mark.parametrize("m", list(range(1, 9)) + [9, 16])
def test_tc_stream_warps_match_oracle(nv, m):
    """Tile-major chains at every M <= 8 (and at M = 9, 16, where every tile
    stays on the tcgen05 MMAs), where the last tiles of every linear
    run on the stream warps (mma.sync beside the tcgen05 MMAs): codes and
    outputs against the oracle, the same bits on a second run and from a CUDA
    graph, and the device status word clear."""
    lins = make_chain(nv, m, STREAM_SHAPES, seed=90 + m)
    entries = []
    for L in lins:
        xd, xg, codes, (wq, ws, wg), y = L["entry"]
        entries.append((xd, xg, codes, nv.tile_weight(wq, ws, wg), y))
    ch = nv.Chain(entries)
    assert ch.tiled
    ch.run(pdl=True)
    torch.cuda.synchronize()
    check_chain(lins)
    first = [L["entry"][4].cpu().numpy().copy() for L in lins]
    for L in lins:
        L["entry"][4].fill_(float("nan"))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            ch.run(pdl=True)
    g.replay()
    torch.cuda.synchronize()
    for L, f in zip(lins, first):
        np.testing.assert_array_equal(L["entry"][4].cpu().numpy(), f)
    assert nv.device_status() == 0


def test_tiled_flag_refusals(nv):
    lib = nv.library()
    g = torch.ones(1, device="cuda")
    z = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    y = torch.full((2, 4), 7.0, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    args = (z.data_ptr(), z.data_ptr(), g.data_ptr(), z.data_ptr(), z.data_ptr(), g.data_ptr(),
            y.data_ptr(), 2, 4, 256)
    assert lib.nvfp4_gemm_smallm_ex(*args, nv.KERNEL_SPLITK | nv.FLAG_W_TILED, st) == 1
    assert lib.nvfp4_gemm_smallm_ex(*args, nv.KERNEL_AUTO | nv.FLAG_W_TILED, st) == 1
    assert lib.nvfp4_tile_weight(z.data_ptr(), z.data_ptr(), 4, 272, z.data_ptr(),
                                 z.data_ptr(), st) == 1
    assert lib.nvfp4_tiled_weight_bytes(300, 4096, None) == 384 * 2048
    torch.cuda.synchronize()
    assert (y.cpu().numpy() == 7.0).all()
