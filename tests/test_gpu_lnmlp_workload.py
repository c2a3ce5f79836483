"""The LayerNormMLP workload at full size (16384 tokens, 4096 -> 16384 -> 4096,
HYBRID, history 16) through the step sequencing of lnmlp.py, vs the oracle.

All 20 steps of the workload: the seeded first step, then 19 delayed steps,
so the 16-entry amax history ring wraps (step 16 overwrites the seeded entry
0, and the window max over the last 16 amaxes decides the scale from then
on; "FP8 低精度训练：Transformer Engine 简析" §三.1).  Checked after every step:
every slot's recorded amax (the oracle's amax of the GPU's own pre-cast
tensors), then after the update every slot's scale, scale_inv, history and
position, all bit-exact.  On steps 0, 1, 16 and 19 also: the FP8 codes of
every cast bit-exact on sampled rows of both orientations, every GEMM and the
activations on sampled elements within their bounds, dbias/dgamma/dbeta in
full."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import as_f64, check_gemm, gpu, host, sample_elems

pytestmark = pytest.mark.gpu

M, H, F = 16384, 4096, 16384


def _rows(rng, n, k=24):
    return np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)]))


def _check_codes(fmt, pre_bits, scale, q, qT, rng, what):
    """q = enc(fl32(pre*scale)) on sampled rows of q and of q^T."""
    R, C = pre_bits.shape
    rows = _rows(rng, R)
    qh = q[torch.from_numpy(rows).to(q.device)].cpu().numpy()
    assert np.array_equal(qh, oracle.quantize(fmt, pre_bits[rows], scale)), what
    cols = _rows(rng, C)
    qth = qT[torch.from_numpy(cols).to(q.device)].cpu().numpy()
    assert np.array_equal(qth, oracle.quantize(fmt, np.ascontiguousarray(pre_bits[:, cols].T), scale)), what + "^T"


def test_ln_mlp_twenty_steps():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.lnmlp import Fp8LayerNormMLP, make_state
    dev = gpu()
    seed = wl.SEEDS["ln_mlp"]
    gamma = (1.0 + wl.normal((H,), 0.1, wl.generator(seed, "gamma"))).to(torch.bfloat16)
    beta = torch.zeros(H, dtype=torch.bfloat16)
    w1 = wl.normal((F, H), 0.02, wl.generator(seed, "W1"), torch.bfloat16)
    w2 = wl.normal((H, F), 0.02, wl.generator(seed, "W2"), torch.bfloat16)
    b1 = torch.zeros(F, dtype=torch.bfloat16)
    b2 = torch.zeros(H, dtype=torch.bfloat16)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=16)
    state = make_state(recipe, 1, device=dev)
    blk = Fp8LayerNormMLP(state, 0, gamma.to(dev), beta.to(dev), w1.to(dev), b1.to(dev), w2.to(dev), b2.to(dev), M,
                          keep_activations=True)
    ost = oracle.ScalingState([0, 0, 1, 0, 0, 1], hist_len=16)
    rng = np.random.default_rng(0)
    gb, bb, w1b, w2b = host(gamma), host(beta), host(w1), host(w2)
    w_amax = (oracle.amax(w1b), oracle.amax(w2b))
    for step in range(20):
        full = step in (0, 1, 16, 19)
        x = wl.normal((M, H), 1.0, wl.generator(seed, "x", step), torch.bfloat16)
        dy = wl.normal((M, H), 1e-3, wl.generator(seed, "dY", step), torch.bfloat16)
        xd, dyd = x.to(dev), dy.to(dev)
        first = step == 0
        blk.forward(xd, seed=first)
        blk.backward(xd, dyd, seed=first)
        torch.cuda.synchronize()
        xb, dyb = host(x), host(dy)
        y_ln, g_act, dh = host(blk.y_ln), host(blk.g), host(blk.dh)
        # --- amaxes recorded by this step's casts (from the GPU's own pre-cast tensors)
        amaxes = [oracle.amax(y_ln), w_amax[0], oracle.amax(dh), oracle.amax(g_act), w_amax[1], oracle.amax(dyb)]
        if first:  # seeding used the same tensors
            for i, a in enumerate(amaxes):
                ost.record_amax(i, a)
            ost.seed()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale), step
        for i, a in enumerate(amaxes):
            ost.record_amax(i, a)
        assert np.array_equal(got["amax"], ost.amax_cur), (step, got["amax"], ost.amax_cur)
        sc, si = ost.scale, ost.scale_inv
        if full:
            _full_checks(blk, step, xb, dyb, y_ln, g_act, dh, w1b, w2b, gb, bb, b1, b2, sc, si, rng)
        # --- the delayed update
        state.update(step)
        ost.update(step)
        torch.cuda.synchronize()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale) and np.array_equal(got["scale_inv"], ost.scale_inv), step
        assert np.array_equal(got["hist"], ost.hist) and np.array_equal(got["pos"], ost.pos), step
    assert np.all(ost.pos == 20 % 16)  # the ring wrapped


def _full_checks(blk, step, xb, dyb, y_ln, g_act, dh, w1b, w2b, gb, bb, b1, b2, sc, si, rng):
    """Codes, activations, GEMMs, bias gradients and the LayerNorm of one step."""
    # --- LayerNorm forward values on sampled rows, then the casts
    rows = _rows(rng, M)
    yr, _, _ = oracle.layernorm_fwd(xb[rows], gb, bb, 1e-5)
    yg = as_f64(blk.y_ln)[rows]
    assert np.all(np.abs(yg - yr) <= 2.0 ** -7 * np.abs(yr) + 2.0 ** -14)
    _check_codes(0, y_ln, sc[0], blk.q_ln, blk.q_lnT, rng, "q_ln")
    _check_codes(0, w1b, sc[1], blk.qw1, blk.qw1T, rng, "qW1")
    _check_codes(0, g_act, sc[3], blk.q_g, blk.q_gT, rng, "q_g")
    _check_codes(0, w2b, sc[4], blk.qw2, blk.qw2T, rng, "qW2")
    _check_codes(1, dyb, sc[5], blk.qdy, blk.qdyT, rng, "qdY")
    _check_codes(1, dh, sc[2], blk.qdh, blk.qdhT, rng, "qdh")
    # --- activations on sampled rows
    h = host(blk.h)
    gr = oracle.gelu(np.ascontiguousarray(h[rows]))
    ga = as_f64(blk.g)[rows]
    assert np.all(np.abs(ga - gr) <= 2.0 ** -7 * np.abs(gr) + 2.0 ** -21 * np.abs(as_f64(blk.h)[rows]))
    dgb = host(blk.dg)
    dhr = oracle.dgelu(np.ascontiguousarray(dgb[rows]), np.ascontiguousarray(h[rows]))
    dha = as_f64(blk.dh)[rows]
    assert np.all(np.abs(dha - dhr) <= 2.0 ** -7 * np.abs(dhr) + 2.0 ** -21 * np.abs(as_f64(blk.dg)[rows]))
    # --- GEMMs on sampled elements (operands: the GPU's bit-exact codes)
    qln, qw1, qg, qw2 = (blk.q_ln.cpu().numpy(), blk.qw1.cpu().numpy(), blk.q_g.cpu().numpy(),
                         blk.qw2.cpu().numpy())
    qdy, qdh = blk.qdy.cpu().numpy(), blk.qdh.cpu().numpy()
    gemms = [
        ("fc1", blk.h, qln, 0, qw1, 0, si[0], si[1], host(b1)),
        ("fc2", blk.y, qg, 0, qw2, 0, si[3], si[4], host(b2)),
        ("fc2 dgrad", blk.dg, qdy, 1, np.ascontiguousarray(qw2.T), 0, si[5], si[4], None),
        ("fc2 wgrad", blk.dw2, np.ascontiguousarray(qdy.T), 1, np.ascontiguousarray(qg.T), 0, si[5], si[3], None),
        ("fc1 dgrad", blk.dln, qdh, 1, np.ascontiguousarray(qw1.T), 0, si[2], si[1], None),
        ("fc1 wgrad", blk.dw1, np.ascontiguousarray(qdh.T), 1, np.ascontiguousarray(qln.T), 0, si[2], si[0], None),
    ]
    for name, D, A, af, B, bf, sa, sb, bias in gemms:
        ms, ns = sample_elems(D.shape[0], D.shape[1], rng, n=1024)
        ref, absr = oracle.gemm_elems(A, af, B, bf, sa, sb, bias, ms, ns)
        check_gemm(D, ref, absr, ms, ns, what="%s step %d" % (name, step))
    # --- bias gradients in full
    for db, src, n in ((blk.db2, dyb, M), (blk.db1, dh, M)):
        s, sabs = oracle.colsum(src)
        assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - s) <= n * 2.0 ** -24 * sabs + 1e-30)
    # --- LayerNorm backward: dx on sampled rows, dgamma/dbeta in full, from the GPU's saved statistics
    mu, rs = blk.mu.cpu().numpy().astype(np.float64), blk.rs.cpu().numpy().astype(np.float64)
    dlnb = host(blk.dln)
    rdx, rdg, rdb, adx, adg, adb = oracle.layernorm_bwd(dlnb, xb, gb, mu, rs)
    dxg = as_f64(blk.dx)
    assert np.all(np.abs(dxg[rows] - rdx[rows]) <= 2.0 ** -7 * np.abs(rdx[rows]) + 2.0 ** -16 * adx[rows])
    assert np.all(np.abs(blk.dgamma.cpu().numpy() - rdg) <= (M + 8) * 2.0 ** -22 * adg + 1e-30)
    assert np.all(np.abs(blk.dbeta.cpu().numpy() - rdb) <= M * 2.0 ** -24 * adb + 1e-30)


def test_ln_mlp_current_scaling_step():
    """Just-in-time (current) scaling variant: each cast uses FP8_MAX/amax of the
    tensor it casts, from this step; codes bit-exact, GEMMs within bound."""
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.lnmlp import Fp8LayerNormMLP, make_state
    dev = gpu()
    Ms, Hs, Fs = 512, 256, 1024
    g = wl.generator(60, "current")
    gamma = (1.0 + wl.normal((Hs,), 0.1, g)).to(torch.bfloat16)
    beta = torch.zeros(Hs, dtype=torch.bfloat16)
    w1 = wl.normal((Fs, Hs), 0.02, g, torch.bfloat16)
    w2 = wl.normal((Hs, Fs), 0.02, g, torch.bfloat16)
    b1, b2 = torch.zeros(Fs, dtype=torch.bfloat16), torch.zeros(Hs, dtype=torch.bfloat16)
    x = wl.normal((Ms, Hs), 1.0, g, torch.bfloat16)
    dy = wl.normal((Ms, Hs), 1e-3, g, torch.bfloat16)
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=16)
    state = make_state(recipe, 1, device=dev)
    blk = Fp8LayerNormMLP(state, 0, gamma.to(dev), beta.to(dev), w1.to(dev), b1.to(dev), w2.to(dev), b2.to(dev), Ms,
                          scaling="current")
    xd = x.to(dev)
    blk.forward(xd)
    blk.backward(xd, dy.to(dev))
    torch.cuda.synchronize()
    got = state.read()
    pre = [host(blk.y_ln), host(w1), host(blk.dh), host(blk.g), host(w2), host(dy)]
    ost = oracle.ScalingState([0, 0, 1, 0, 0, 1], hist_len=16)
    for i, t in enumerate(pre):
        ost.record_amax(i, oracle.amax(t))
    ost.seed()  # the current scale of every tensor
    assert np.array_equal(got["scale"], ost.scale)
    sc, si = ost.scale, ost.scale_inv
    qs = [(blk.q_ln, blk.q_lnT, 0), (blk.qw1, blk.qw1T, 0), (blk.qdh, blk.qdhT, 1), (blk.q_g, blk.q_gT, 0),
          (blk.qw2, blk.qw2T, 0), (blk.qdy, blk.qdyT, 1)]
    for i, (q, qT, fmt) in enumerate(qs):
        ref = oracle.quantize(fmt, pre[i], sc[i])
        assert np.array_equal(q.cpu().numpy(), ref), i
        assert np.array_equal(qT.cpu().numpy(), ref.T), i
    rng = np.random.default_rng(3)
    qln, qw1, qg, qw2 = (blk.q_ln.cpu().numpy(), blk.qw1.cpu().numpy(), blk.q_g.cpu().numpy(), blk.qw2.cpu().numpy())
    qdy, qdh = blk.qdy.cpu().numpy(), blk.qdh.cpu().numpy()
    for name, D, A, af, B, bf, sa, sb in (
            ("fc1", blk.h, qln, 0, qw1, 0, si[0], si[1]),
            ("fc2", blk.y, qg, 0, qw2, 0, si[3], si[4]),
            ("fc2 dgrad", blk.dg, qdy, 1, np.ascontiguousarray(qw2.T), 0, si[5], si[4]),
            ("fc1 wgrad", blk.dw1, np.ascontiguousarray(qdh.T), 1, np.ascontiguousarray(qln.T), 0, si[2], si[0])):
        ms, ns = sample_elems(D.shape[0], D.shape[1], rng, n=1024)
        ref, absr = oracle.gemm_elems(A, af, B, bf, sa, sb, None, ms, ns)
        check_gemm(D, ref, absr, ms, ns, what=name)
