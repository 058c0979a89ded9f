"""GPU parity of the quantisation kernels: tensor scale, activation
quantisation and weight packing are bit-exact with the oracle (every byte has
one correct value).  Marked gpu; the CUDA side runs through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synthetic

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


@pytest.mark.parametrize("count", [0, 1, 3, 4, 17, 4096, 1 << 20, (1 << 20) + 5])
def test_global_scale_bit_exact(nv, count):
    t = synthetic.activations(1, max(count, 1), seed=count)[0, :count].copy()
    g = host(nv.global_scale(dev(t)))[0]
    assert np.float32(g) == oracle.global_scale(t)


@pytest.mark.parametrize("m", [1, 3, 8])
@pytest.mark.parametrize("k", [16, 48, 512, 4096, 12288, 25600])
@pytest.mark.parametrize("dist", ["outliers", "decades"])
def test_quantize_act_bit_exact(nv, m, k, dist):
    if dist == "outliers":
        x = synthetic.activations(m, k, seed=100 + k + m)
    else:
        x = synthetic.log_uniform_blocks(m, k, seed=200 + k + m)
    gx = oracle.global_scale(x)
    oq, os_ = oracle.quantize(x, gx)
    xq, xs = nv.quantize_act(dev(x), dev(np.array([gx], np.float32)))
    np.testing.assert_array_equal(host(xq), oq)
    np.testing.assert_array_equal(host(xs), os_)


def test_quantize_static_scale_saturates(nv):
    """A static activation scale that is too small saturates block scales at
    448 and codes at 6, identically on both sides."""
    x = synthetic.activations(2, 256, seed=7)
    gx = np.float32(oracle.global_scale(x) / 50)
    oq, os_ = oracle.quantize(x, gx)
    assert (os_ == 0x7E).any()
    xq, xs = nv.quantize_act(dev(x), dev(np.array([gx], np.float32)))
    np.testing.assert_array_equal(host(xq), oq)
    np.testing.assert_array_equal(host(xs), os_)


def test_quantize_every_e4m3_tie_and_e2m1_tie(nv):
    """Block maxima at every E4M3 midpoint (and one FP32 ulp either side), and
    elements at every E2M1 midpoint with S == 1, against the oracle."""
    g = np.float32(0.25)                      # 6 g = 1.5
    codes = np.arange(0, 0x7E)
    vals = np.array([oracle.e4m3_value(c) for c in range(0, 0x7F)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    targets = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                              np.nextafter(mids, np.float32(1e9)), vals.astype(np.float32)])
    bmax = (targets.astype(np.float64) * 1.5).astype(np.float32)
    # bmax / 1.5 must reproduce the target in FP32 for the tie to be exact;
    # keep the rows where it does (most of them) and test all rows anyway.
    rows = bmax.size
    x = np.zeros((rows, 16), np.float32)
    x[:, 0] = bmax
    x[:, 1] = -bmax / 3
    x[:, 2:] = np.linspace(-1, 1, 14, dtype=np.float32) * bmax[:, None] / 7
    oq, os_ = oracle.quantize(x, g)
    xq, xs = nv.quantize_act(dev(x), dev(np.array([g], np.float32)))
    np.testing.assert_array_equal(host(xs), os_)
    np.testing.assert_array_equal(host(xq), oq)
    assert len(set(os_.ravel())) > 100 and codes.size == 0x7E
    # E2M1 ties: bmax 6 and g 0.25 give s = 4 exactly and S = 1.
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    x = np.zeros((2, 16), np.float32)
    x[0, 0] = 6.0
    x[0, 1:8] = ties
    x[0, 8:15] = -ties
    x[1, 0] = -6.0
    x[1, 1:8] = np.nextafter(ties, np.float32(0))
    x[1, 8:15] = np.nextafter(ties, np.float32(9))
    oq, os_ = oracle.quantize(x, g)
    xq, xs = nv.quantize_act(dev(x), dev(np.array([g], np.float32)))
    np.testing.assert_array_equal(host(xs), os_)
    np.testing.assert_array_equal(host(xq), oq)


def test_quantize_zeros_and_signed_zeros(nv):
    x = np.zeros((3, 64), np.float32)
    x[1, 5] = -0.0
    x[2, :16] = 1.0
    x[2, 16:32] = -0.0
    x[2, 33] = -1e-30          # rounds to a zero code, keeps its sign
    for gx in (np.float32(0.0), oracle.global_scale(x)):
        oq, os_ = oracle.quantize(x, gx)
        xq, xs = nv.quantize_act(dev(x), dev(np.array([gx], np.float32)))
        np.testing.assert_array_equal(host(xq), oq)
        np.testing.assert_array_equal(host(xs), os_)


@pytest.mark.parametrize("n,k", [(1, 16), (256, 512), (1000, 48), (300, 4096)])
def test_pack_weight_bit_exact(nv, n, k):
    w = synthetic.weights(n, k, 0.02, seed=n + k)
    oq, os_, og = oracle.pack_weight(w)
    wq, ws, wg = nv.pack_weight(dev(w))
    assert np.float32(host(wg)[0]) == og
    np.testing.assert_array_equal(host(wq), oq)
    np.testing.assert_array_equal(host(ws), os_)


@pytest.mark.parametrize("shape", [(l.n, l.k, "8B") for l in synthetic.LINEARS_8B]
                         + [(l.n, l.k, "32B") for l in synthetic.LINEARS_32B])
def test_pack_weight_full_size_sampled_rows(nv, shape):
    """Full-size layers: the tensor scale over the whole tensor, and the codes
    and scales of 48 sampled rows (first, last, random)."""
    n, k, fam = shape
    std = synthetic.WEIGHT_STD_8B if fam == "8B" else synthetic.WEIGHT_STD_32B
    w = synthetic.weights(n, k, std, seed=n * 7 + k)
    wq, ws, wg = nv.pack_weight(dev(w))
    og = oracle.global_scale(w)
    assert np.float32(host(wg)[0]) == og
    rng = np.random.default_rng(n + k)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 46)]))
    oq, os_ = oracle.quantize(w[rows], og)
    idx = torch.from_numpy(rows).cuda()
    np.testing.assert_array_equal(host(wq.index_select(0, idx)), oq)
    np.testing.assert_array_equal(host(ws.index_select(0, idx)), os_)
    del wq, ws
    torch.cuda.empty_cache()


def test_pack_weight_empty(nv):
    w = torch.empty((0, 32), dtype=torch.float32, device="cuda")
    wq, ws, wg = nv.pack_weight(w)
    assert wq.shape == (0, 16) and host(wg)[0] == 0.0


def test_quantize_codes_at_every_threshold_for_many_scales(nv):
    """The quantisers divide by one reciprocal per block with an FMA
    correction; elements placed on, and a few ulps around, every E2M1
    decision threshold for many block scales give the oracle's codes (which
    come from IEEE division)."""
    rng = np.random.default_rng(42)
    thresholds = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    rows = []
    for _ in range(400):
        S = np.float32(np.exp2(rng.uniform(-30, 30)))
        g = np.float32(S / 448.0)          # block scale code saturates near 448
        base = np.float32(6.0) * S         # block max: code 7, scale exact-ish
        vals = [base]
        for th in thresholds:
            c = np.float32(th) * S
            vals.append(c)
            for k in (1, 2, 3):
                vals.append(np.nextafter(c, np.float32(0), dtype=np.float32) if k == 1 else
                            np.float32(c) * np.float32(1 - k * 2.0 ** -23))
                vals.append(np.nextafter(c, np.float32(1e30), dtype=np.float32) if k == 1 else
                            np.float32(c) * np.float32(1 + k * 2.0 ** -23))
        vals = np.array(vals, np.float32)
        vals = np.concatenate([vals, -vals])
        pad = (-len(vals)) % 16
        vals = np.concatenate([vals, np.zeros(pad, np.float32)])
        blk = vals.reshape(-1, 16)
        blk[:, 0] = base                    # every block keeps the same max
        rows.append((blk.reshape(1, -1), g))
    for x, g in rows:
        oq, os_ = oracle.quantize(x, g)
        xq, xs = nv.quantize_act(dev(x), dev(np.array([g], np.float32)))
        np.testing.assert_array_equal(host(xs), os_)
        np.testing.assert_array_equal(host(xq), oq)


@pytest.mark.parametrize("m,k", [(1, 4096), (3, 12288), (8, 512), (2, 48)])
def test_quantize_dynamic_scale_bit_exact(nv, m, k):
    """Dynamic tensor scale: x_g = amax/2688 from this X, then the codes."""
    x = synthetic.activations(m, k, seed=900 + m + k)
    gx = oracle.global_scale(x)
    oq, os_ = oracle.quantize(x, gx)
    xq, xs, xg = nv.quantize_act_dynamic(dev(x))
    assert np.float32(host(xg)[0]) == gx
    np.testing.assert_array_equal(host(xq), oq)
    np.testing.assert_array_equal(host(xs), os_)


def bf16_tensor(bits: np.ndarray) -> torch.Tensor:
    """A CUDA bfloat16 tensor holding these BF16 bit patterns."""
    return torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("m,k", [(1, 4096), (3, 12288), (8, 512), (2, 48), (5, 25600)])
def test_quantize_act_bf16_input_bit_exact(nv, m, k):
    """BF16 activations: the codes and scales equal the oracle's for the
    FP32 values those BF16 numbers are (widening is exact)."""
    x32 = synthetic.activations(m, k, seed=1000 + m + k)
    bits = oracle.f32_to_bf16(x32)
    xw = oracle.bf16_to_f32(bits)
    gx = oracle.global_scale(xw)
    oq, os_ = oracle.quantize(xw, gx)
    xq, xs = nv.quantize_act(bf16_tensor(bits), dev(np.array([gx], np.float32)))
    np.testing.assert_array_equal(host(xq), oq)
    np.testing.assert_array_equal(host(xs), os_)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("m,k", [(1, 16), (3, 16 * 37), (1, 4096), (8, 12288), (2, 25600)])
def test_quantize_act_pdl_chain_bit_exact(nv, m, k, bf16):
    """The programmatic-dependent-launch form (it prefetches X into L2 before
    waiting on X's producer), launched right after a kernel that writes X:
    the codes are those of the X that kernel wrote, equal to the oracle's."""
    x = synthetic.activations(m, k, seed=3000 + m + k)
    stale = np.full_like(x, 1e4)           # what X holds before the producer runs
    if bf16:
        bits = oracle.f32_to_bf16(x)
        xv = oracle.bf16_to_f32(bits)
        xd = bf16_tensor(oracle.f32_to_bf16(stale))
        src = bf16_tensor(bits)
    else:
        xv = x
        xd = dev(stale)
        src = dev(x)
    gx = oracle.global_scale(xv)
    oq, os_ = oracle.quantize(xv, gx)
    g = dev(np.array([gx], np.float32))
    torch.cuda.synchronize()
    for _ in range(3):
        xd.zero_()
        xd.add_(src)                        # the producer of X: a kernel on the same stream
        xq, xs = nv.quantize_act(xd, g, pdl=True)
        np.testing.assert_array_equal(host(xq), oq)
        np.testing.assert_array_equal(host(xs), os_)
        xd.fill_(1e4)
