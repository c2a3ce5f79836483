"""End-to-end te.Linear steps under delayed scaling vs the oracle.

linear_fwd:    2048 tokens, 768 -> 3072, fp32 X and W, E4M3 recipe, history 16
               seeded with the first step's amax; forward only; checked in full.
linear_hybrid: same layer, HYBRID (E5M2 gradients), 10 steps with a scale update
               each step, fresh X and dY (0.1 % outliers x1000) every step;
               every cast, amax, scale and GEMM output checked in full.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import check_gemm, gpu, host

pytestmark = pytest.mark.gpu

M, K, N = 2048, 768, 3072


def _all(m, n):
    a, b = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    return a.ravel(), b.ravel()


def test_linear_fwd_e4m3():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    seed = wl.SEEDS["linear_fwd"]
    x = wl.normal((M, K), 1.0, wl.generator(seed, "X"))
    w = wl.normal((N, K), 0.02, wl.generator(seed, "W"))
    b = torch.zeros(N, dtype=torch.float32)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_E4M3, amax_history_len=16)
    state = make_state(recipe, 1, device=dev)
    lin = Fp8Linear(state, 0, w.to(dev), b.to(dev), M, training=False)
    xd = x.to(dev)
    lin.seed_forward(xd)
    lin.forward(xd)
    torch.cuda.synchronize()
    got = state.read()

    ost = oracle.ScalingState([0, 0, 0], hist_len=16)
    xs, ws = host(x), host(w)
    ost.record_amax(0, oracle.amax(xs))
    ost.record_amax(1, oracle.amax(ws))
    ost.seed()
    assert np.array_equal(got["scale"][:2], ost.scale[:2])
    assert np.array_equal(got["scale_inv"][:2], ost.scale_inv[:2])
    assert np.array_equal(got["hist"][:2], ost.hist[:2])
    qx = oracle.quantize(0, xs, ost.scale[0])
    qw = oracle.quantize(0, ws, ost.scale[1])
    assert np.array_equal(lin.qx.cpu().numpy(), qx)
    assert np.array_equal(lin.qw.cpu().numpy(), qw)
    assert got["amax"][0] == oracle.amax(xs) and got["amax"][1] == oracle.amax(ws)
    ms, ns = _all(M, N)
    ref, absr = oracle.gemm_elems(qx, 0, qw, 0, ost.scale_inv[0], ost.scale_inv[1], host(b), ms, ns)
    check_gemm(lin.y, ref, absr, what="forward")


def test_linear_hybrid_ten_steps():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    seed = wl.SEEDS["linear_hybrid"]
    w = wl.normal((N, K), 0.02, wl.generator(seed, "W"))
    b = torch.zeros(N, dtype=torch.float32)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=16)
    state = make_state(recipe, 1, device=dev)
    lin = Fp8Linear(state, 0, w.to(dev), b.to(dev), M)
    ost = oracle.ScalingState([0, 0, 1], hist_len=16)
    ws = host(w)
    for step in range(10):
        x = wl.normal((M, K), 1.0, wl.generator(seed, "X", step))
        gdy = wl.generator(seed, "dY", step)
        dy = wl.with_outliers(wl.normal((M, N), 1e-3, gdy, torch.bfloat16), 0.001, 1000.0, gdy)
        xd, dyd = x.to(dev), dy.to(dev)
        xs, dys = host(x), host(dy)
        if step == 0:
            lin.seed_forward(xd)
            ost.record_amax(0, oracle.amax(xs))
            ost.record_amax(1, oracle.amax(ws))
        lin.forward(xd)
        if step == 0:
            lin.seed_backward(dyd)
            ost.record_amax(2, oracle.amax(dys))
            ost.seed()
        lin.backward(dyd)
        torch.cuda.synchronize()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale), step
        qx, qw, qdy = (oracle.quantize(0, xs, ost.scale[0]), oracle.quantize(0, ws, ost.scale[1]),
                       oracle.quantize(1, dys, ost.scale[2]))
        assert np.array_equal(lin.qx.cpu().numpy(), qx), step
        assert np.array_equal(lin.qxT.cpu().numpy(), qx.T), step
        assert np.array_equal(lin.qw.cpu().numpy(), qw), step
        assert np.array_equal(lin.qwT.cpu().numpy(), qw.T), step
        assert np.array_equal(lin.qdy.cpu().numpy(), qdy), step
        assert np.array_equal(lin.qdyT.cpu().numpy(), qdy.T), step
        for i, t in enumerate((xs, ws, dys)):
            ost.record_amax(i, oracle.amax(t))
        assert np.array_equal(got["amax"], ost.amax_cur), step
        si = ost.scale_inv
        ms, ns = _all(M, N)
        ref, absr = oracle.gemm_elems(qx, 0, qw, 0, si[0], si[1], host(b), ms, ns)
        check_gemm(lin.y, ref, absr, what="forward step %d" % step)
        ms, ks = _all(M, K)
        ref, absr = oracle.gemm_elems(qdy, 1, np.ascontiguousarray(qw.T), 0, si[2], si[1], None, ms, ks)
        check_gemm(lin.dx, ref, absr, what="dgrad step %d" % step)
        ns, ks = _all(N, K)
        ref, absr = oracle.gemm_elems(np.ascontiguousarray(qdy.T), 1, np.ascontiguousarray(qx.T), 0, si[2], si[0],
                                      None, ns, ks)
        check_gemm(lin.dw, ref, absr, what="wgrad step %d" % step)
        s, sabs = oracle.colsum(dys)
        assert np.all(np.abs(lin.db.cpu().numpy().astype(np.float64) - s) <= M * 2.0 ** -24 * sabs + 1e-30)
        state.update(step)
        ost.update(step)
        torch.cuda.synchronize()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale) and np.array_equal(got["hist"], ost.hist), step


def test_linear_current_scaling_two_steps():
    """Just-in-time (current) scaling, the alternative TE-brief §三.1 contrasts with
    delayed scaling: every cast of a step uses FP8_MAX/amax of that step's own tensor.
    The second step's tensors are 4x the first's, so a scale carried over from the
    previous step would give different codes."""
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    M2, K2, N2 = 384, 512, 640
    g = wl.generator(91, "current-linear")
    w = wl.normal((N2, K2), 0.02, g, torch.bfloat16)
    b = torch.zeros(N2, dtype=torch.bfloat16)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=1)
    state = make_state(recipe, 1, device=dev)
    lin = Fp8Linear(state, 0, w.to(dev), b.to(dev), M2, scaling="current")
    ws = host(w)
    for step, f in enumerate((1.0, 4.0)):
        x = (wl.normal((M2, K2), 1.0, g) * f).to(torch.bfloat16)
        dy = (wl.normal((M2, N2), 1e-3, g) * f).to(torch.bfloat16)
        lin.forward(x.to(dev))
        lin.backward(dy.to(dev))
        torch.cuda.synchronize()
        xs, dys = host(x), host(dy)
        ost = oracle.ScalingState([0, 0, 1], hist_len=1)
        for i, t in enumerate((xs, ws, dys)):
            ost.record_amax(i, oracle.amax(t))
        ost.seed()  # this step's own amaxes give this step's scales
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale), step
        assert np.array_equal(got["scale_inv"], ost.scale_inv), step
        qx, qw, qdy = (oracle.quantize(0, xs, ost.scale[0]), oracle.quantize(0, ws, ost.scale[1]),
                       oracle.quantize(1, dys, ost.scale[2]))
        assert np.array_equal(lin.qx.cpu().numpy(), qx), step
        assert np.array_equal(lin.qxT.cpu().numpy(), qx.T), step
        assert np.array_equal(lin.qw.cpu().numpy(), qw), step
        assert np.array_equal(lin.qdy.cpu().numpy(), qdy), step
        assert np.array_equal(lin.qdyT.cpu().numpy(), qdy.T), step
        si = ost.scale_inv
        ms, ns = _all(M2, N2)
        ref, absr = oracle.gemm_elems(qx, 0, qw, 0, si[0], si[1], host(b), ms, ns)
        check_gemm(lin.y, ref, absr, what="forward step %d" % step)
        ms, ks = _all(M2, K2)
        ref, absr = oracle.gemm_elems(qdy, 1, np.ascontiguousarray(qw.T), 0, si[2], si[1], None, ms, ks)
        check_gemm(lin.dx, ref, absr, what="dgrad step %d" % step)
        ns, ks = _all(N2, K2)
        ref, absr = oracle.gemm_elems(np.ascontiguousarray(qdy.T), 1, np.ascontiguousarray(qx.T), 0, si[2], si[0],
                                      None, ns, ks)
        check_gemm(lin.dw, ref, absr, what="wgrad step %d" % step)
        s, sabs = oracle.colsum(dys)
        assert np.all(np.abs(lin.db.cpu().numpy().astype(np.float64) - s) <= M2 * 2.0 ** -24 * sabs + 1e-30)
    with pytest.raises(RuntimeError):
        lin.forward(x.to(dev), is_first_microbatch=True)
