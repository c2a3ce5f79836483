"""The FP8 weight cache across micro-batches ("FP8 低精度训练：Transformer
Engine 简析" §三.3: a TE module skips the weight cast while a cached FP8 copy
exists).

The weight is cast once (is_first_microbatch=True) together with its decode
factor fl32(1/scale).  The scale update that follows may move the slot's
scale_inv on; the later micro-batches (is_first_microbatch=False) must still
decode the kept codes with the factor they were cast at.  The tests make the
update move the weight's scale (the weight grows 4x after the history was
seeded), so a decode with the slot's new scale_inv would be off by 4."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import check_gemm, gpu, host

pytestmark = pytest.mark.gpu


def _all(m, n):
    a, b = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    return a.ravel(), b.ravel()


@pytest.mark.parametrize("scale", [1.0, 0.75, 3.0, 448.0 / 0.02, 2.0 ** -60, 2.0 ** 100, 1.0 / 3.0])
def test_cast_writes_the_decode_factor(scale):
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    x = wl.normal((64, 128), 1.0, wl.generator(80, "sinv"), torch.bfloat16).to(dev)
    sc = torch.tensor([scale], dtype=torch.float32, device=dev)
    q = torch.empty((64, 128), dtype=torch.uint8, device=dev)
    sinv = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
    fd.fp8_cast_amax_transpose(x, fd.E4M3, sc, out=q, scale_inv_out=sinv)
    torch.cuda.synchronize()
    want = np.float32(1.0) / np.float32(scale)  # fl32(1/scale), IEEE division
    assert sinv.cpu().numpy()[0].tobytes() == want.tobytes()
    assert np.array_equal(q.cpu().numpy(), oracle.quantize(0, host(x.cpu()), np.float32(scale)))


def test_linear_weight_cache_keeps_the_decode_factor():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import GRAD, IN, WEIGHT, Fp8Linear, make_state
    dev = gpu()
    M, K, N = 384, 512, 768
    seed = 81
    x = wl.normal((M, K), 1.0, wl.generator(seed, "X"), torch.bfloat16)
    dy = wl.normal((M, N), 1e-3, wl.generator(seed, "dY"), torch.bfloat16)
    wa = wl.normal((N, K), 0.02, wl.generator(seed, "W"), torch.bfloat16)
    wb = (wa.float() * 4).to(torch.bfloat16)  # exact: a power of two
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=4)
    state = make_state(recipe, 1, device=dev)
    xd, dyd = x.to(dev), dy.to(dev)
    lin = Fp8Linear(state, 0, wa.to(dev), None, M)
    lin.seed_forward(xd)       # weight history seeded with amax(wa)
    lin.seed_backward(dyd)
    lin.w = wb.to(dev)          # the optimizer moved the weight
    s0 = state.read()

    # micro-batch 1: cast and keep
    y1 = lin.forward(xd, is_first_microbatch=True).clone()
    dx1, dw1, _ = (t.clone() if t is not None else None for t in lin.backward(dyd))
    qw1, qwT1 = lin.qw.clone(), lin.qwT.clone()
    torch.cuda.synchronize()
    snap = lin.wcache.scale_inv.cpu().numpy()[0]
    assert snap.tobytes() == s0["scale_inv"][WEIGHT].tobytes()
    assert np.array_equal(qw1.cpu().numpy(), oracle.quantize(0, host(wb), s0["scale"][WEIGHT]))
    state.update(0)
    torch.cuda.synchronize()
    s1 = state.read()
    # the update moved the weight's scale (amax(wb) = 4 amax(wa) entered the window)
    assert s1["scale_inv"][WEIGHT] == np.float32(4) * s0["scale_inv"][WEIGHT]
    # and left the input and gradient scales alone (same tensors as at seeding)
    assert s1["scale"][IN] == s0["scale"][IN] and s1["scale"][GRAD] == s0["scale"][GRAD]

    # micro-batch 2: no weight cast; the kept codes decode with the kept factor
    y2 = lin.forward(xd, is_first_microbatch=False).clone()
    dx2, dw2, _ = (t.clone() if t is not None else None for t in lin.backward(dyd))
    torch.cuda.synchronize()
    s2 = state.read()
    assert s2["amax"][WEIGHT] == 0.0  # the skipped cast recorded nothing
    assert torch.equal(lin.qw, qw1) and torch.equal(lin.qwT, qwT1)  # a cast at the new scale would differ
    assert torch.equal(y2, y1) and torch.equal(dx2, dx1) and torch.equal(dw2, dw1)
    ms, ns = _all(M, N)
    ref, absr = oracle.gemm_elems(lin.qx.cpu().numpy(), 0, qw1.cpu().numpy(), 0, s1["scale_inv"][IN], snap, None,
                                  ms, ns)
    check_gemm(y2, ref, absr, what="forward with the cached weight")

    # an uncached call recasts at the new scale and drops the cache
    y3 = lin.forward(xd, is_first_microbatch=None)
    torch.cuda.synchronize()
    assert np.array_equal(lin.qw.cpu().numpy(), oracle.quantize(0, host(wb), s1["scale"][WEIGHT]))
    ref3, absr3 = oracle.gemm_elems(lin.qx.cpu().numpy(), 0, lin.qw.cpu().numpy(), 0, s1["scale_inv"][IN],
                                    s1["scale_inv"][WEIGHT], None, ms, ns)
    check_gemm(y3, ref3, absr3, what="forward after the cache was dropped")
    with pytest.raises(RuntimeError):
        lin.forward(xd, is_first_microbatch=False)


def test_lnmlp_weight_cache_skips_the_weight_casts():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.lnmlp import FC1_W, FC2_IN, FC2_W, Fp8LayerNormMLP, make_state
    dev = gpu()
    M, H, F = 256, 512, 1024
    seed = 82
    g = wl.generator(seed, "p")
    gamma = (1.0 + wl.normal((H,), 0.1, g)).to(torch.bfloat16).to(dev)
    beta = torch.zeros(H, dtype=torch.bfloat16, device=dev)
    w1 = wl.normal((F, H), 0.02, g, torch.bfloat16).to(dev)
    w2 = wl.normal((H, F), 0.02, g, torch.bfloat16).to(dev)
    b1 = torch.zeros(F, dtype=torch.bfloat16, device=dev)
    b2 = torch.zeros(H, dtype=torch.bfloat16, device=dev)
    x = wl.normal((M, H), 1.0, g, torch.bfloat16).to(dev)
    dy = wl.normal((M, H), 1e-3, g, torch.bfloat16).to(dev)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=4)
    state = make_state(recipe, 1, device=dev)
    blk = Fp8LayerNormMLP(state, 0, gamma, beta, w1, b1, w2, b2, M)
    blk.forward(x, seed=True)
    blk.backward(x, dy, seed=True)
    state.update(0)
    blk.w2 = (w2.float() * 4).to(torch.bfloat16)  # the optimizer moved W2
    blk.forward(x, is_first_microbatch=True)
    blk.backward(x, dy)
    torch.cuda.synchronize()
    s0 = state.read()
    snap1, snap2 = blk.w1cache.scale_inv.cpu().numpy()[0], blk.w2cache.scale_inv.cpu().numpy()[0]
    assert snap1.tobytes() == s0["scale_inv"][FC1_W].tobytes()
    assert snap2.tobytes() == s0["scale_inv"][FC2_W].tobytes()
    q1, q2 = blk.qw1.clone(), blk.qw2.clone()
    state.update(1)
    torch.cuda.synchronize()
    s1 = state.read()
    assert s1["scale_inv"][FC2_W] == np.float32(4) * snap2  # W2's slot moved on
    blk.forward(x, is_first_microbatch=False)
    blk.backward(x, dy)
    torch.cuda.synchronize()
    s2 = state.read()
    assert s2["amax"][FC1_W] == 0.0 and s2["amax"][FC2_W] == 0.0
    assert torch.equal(blk.qw1, q1) and torch.equal(blk.qw2, q2)
    ms, ns = _all(M, H)
    ref, absr = oracle.gemm_elems(blk.q_g.cpu().numpy(), 0, q2.cpu().numpy(), 0, s1["scale_inv"][FC2_IN], snap2,
                                  host(b2.cpu()), ms, ns)
    check_gemm(blk.y, ref, absr, what="fc2 with the cached W2")
