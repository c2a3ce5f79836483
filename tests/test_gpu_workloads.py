"""Full-size workloads through the step sequencing the benchmark times, vs the
oracle on sampled outputs.

llama_proj: 8192 tokens; QKV 4096->12288, out 4096->4096, up 4096->11008,
            down 11008->4096; X Student-t(3) x 0.5, W ~N(0,0.02), dY ~N(0,1e-3);
            HYBRID, margin 0, history 1024; two steps (seeded + delayed).
mx_mlp:     16384 tokens, 8192 -> 28672 -> 8192 MXFP8; X with per-channel
            factors log-uniform in [1e-3, 1e2], W ~N(0,0.02), dY ~N(0,1);
            the up projection's bf16 output feeds the down projection."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import check_gemm, gpu, host, sample_elems

pytestmark = pytest.mark.gpu


def _rows(rng, n, k=16):
    return np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)]))


def _codes_ok(fmt, pre_bits, scale, q, qT, rng):
    rows = _rows(rng, pre_bits.shape[0])
    assert np.array_equal(q[torch.from_numpy(rows).to(q.device)].cpu().numpy(),
                          oracle.quantize(fmt, pre_bits[rows], scale))
    cols = _rows(rng, pre_bits.shape[1])
    assert np.array_equal(qT[torch.from_numpy(cols).to(q.device)].cpu().numpy(),
                          oracle.quantize(fmt, np.ascontiguousarray(pre_bits[:, cols].T), scale))


def test_llama_projections_two_steps():
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    seed = wl.SEEDS["llama_proj"]
    M = 8192
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=1024)
    L = len(wl.LLAMA_PROJ)
    state = make_state(recipe, L, device=dev)
    ws = [wl.normal((n, k), 0.02, wl.generator(seed, "W/" + name), torch.bfloat16) for name, k, n in wl.LLAMA_PROJ]
    bs = [torch.zeros(n, dtype=torch.bfloat16) for _, _, n in wl.LLAMA_PROJ]
    layers = [Fp8Linear(state, i, ws[i].to(dev), bs[i].to(dev), M) for i in range(L)]
    ost = oracle.ScalingState([0, 0, 1] * L, hist_len=1024)
    rng = np.random.default_rng(1)
    for step in range(2):
        xs = [wl.student_t3((M, k), 0.5, wl.generator(seed, "X/" + name, step)) for name, k, _ in wl.LLAMA_PROJ]
        dys = [wl.normal((M, n), 1e-3, wl.generator(seed, "dY/" + name, step), torch.bfloat16)
               for name, _, n in wl.LLAMA_PROJ]
        xd = [x.to(dev) for x in xs]
        dyd = [d.to(dev) for d in dys]
        if step == 0:
            for lin, x in zip(layers, xd):
                lin.seed_forward(x)
        for lin, x in zip(layers, xd):
            lin.forward(x)
        if step == 0:
            for lin, d in zip(layers, dyd):
                lin.seed_backward(d)
        for lin, d in zip(layers, dyd):
            lin.backward(d)
        torch.cuda.synchronize()
        am = []
        for i in range(L):
            am += [oracle.amax(host(xs[i])), oracle.amax(host(ws[i])), oracle.amax(host(dys[i]))]
        if step == 0:
            for i, a in enumerate(am):
                ost.record_amax(i, a)
            ost.seed()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale)
        for i, a in enumerate(am):
            ost.record_amax(i, a)
        assert np.array_equal(got["amax"], ost.amax_cur)
        sc, si = ost.scale, ost.scale_inv
        for i, lin in enumerate(layers):
            b = 3 * i
            xb, wb, dyb = host(xs[i]), host(ws[i]), host(dys[i])
            _codes_ok(0, xb, sc[b], lin.qx, lin.qxT, rng)
            _codes_ok(0, wb, sc[b + 1], lin.qw, lin.qwT, rng)
            _codes_ok(1, dyb, sc[b + 2], lin.qdy, lin.qdyT, rng)
            qx, qw, qdy = lin.qx.cpu().numpy(), lin.qw.cpu().numpy(), lin.qdy.cpu().numpy()
            for name, D, A, af, B, bf, sa, sb, bias in (
                    ("fwd", lin.y, qx, 0, qw, 0, si[b], si[b + 1], host(bs[i])),
                    ("dgrad", lin.dx, qdy, 1, np.ascontiguousarray(qw.T), 0, si[b + 2], si[b + 1], None),
                    ("wgrad", lin.dw, np.ascontiguousarray(qdy.T), 1, np.ascontiguousarray(qx.T), 0, si[b + 2],
                     si[b], None)):
                ms, ns = sample_elems(D.shape[0], D.shape[1], rng, n=1024)
                ref, absr = oracle.gemm_elems(A, af, B, bf, sa, sb, bias, ms, ns)
                check_gemm(D, ref, absr, ms, ns, what="%s %s step %d" % (wl.LLAMA_PROJ[i][0], name, step))
            s, sabs = oracle.colsum(dyb)
            assert np.all(np.abs(lin.db.cpu().numpy().astype(np.float64) - s) <= M * 2.0 ** -24 * sabs + 1e-30)
        state.update(step)
        ost.update(step)
        torch.cuda.synchronize()
        got = state.read()
        assert np.array_equal(got["scale"], ost.scale) and np.array_equal(got["hist"], ost.hist)


def test_mx_mlp_step():
    from fp8_delayed_scaling_gb300.mxlinear import MxLinear
    from test_gpu_mx import tiled_to_plain
    dev = gpu()
    seed = wl.SEEDS["mx_mlp"]
    M, H, F = 16384, 8192, 28672
    x = wl.channel_scaled_normal(M, H, wl.generator(seed, "X"))
    w1 = wl.normal((F, H), 0.02, wl.generator(seed, "W1"), torch.bfloat16)
    w2 = wl.normal((H, F), 0.02, wl.generator(seed, "W2"), torch.bfloat16)
    dy = wl.normal((M, H), 1.0, wl.generator(seed, "dY"), torch.bfloat16)
    # zero biases, as in the te.Linear example (bias=True): their gradients come from the
    # column sums fused into the quantisation of dY and of dh
    up = MxLinear(w1.to(dev), torch.zeros(F, dtype=torch.bfloat16, device=dev), M)
    down = MxLinear(w2.to(dev), torch.zeros(H, dtype=torch.bfloat16, device=dev), M)
    hid = up.forward(x.to(dev))
    down.forward(hid)
    dh, _, _ = down.backward(dy.to(dev))
    up.backward(dh)
    torch.cuda.synchronize()
    rng = np.random.default_rng(2)
    for lin, src in ((down, dy), (up, dh)):  # bias gradients in full
        s, sabs = oracle.colsum(host(src))
        assert np.all(np.abs(lin.db.cpu().numpy().astype(np.float64) - s) <= M * 2.0 ** -24 * sabs + 1e-30)
    # quantisation of every operand: sampled rows of both orientations, bit-exact
    for mxt, src in ((up.mx_x, x), (up.mx_w, w1), (down.mx_x, hid), (down.mx_w, w2), (down.mx_dy, dy),
                     (up.mx_dy, dh)):
        sb = host(src)
        R, C = sb.shape
        rows = _rows(rng, R, 8)
        q, s = oracle.mx_quantize_rows(np.ascontiguousarray(sb[rows]))
        assert np.array_equal(mxt.row_q[torch.from_numpy(rows).to(dev)].cpu().numpy(), q)
        assert np.array_equal(tiled_to_plain(mxt.row_s.cpu().numpy(), R, C // 32)[rows], s)
        blk = rng.integers(0, R // 32)
        cols = _rows(rng, C, 8)
        qc, scc = oracle.mx_quantize_cols(np.ascontiguousarray(sb[32 * blk:32 * blk + 32][:, cols]))
        assert np.array_equal(mxt.col_q[torch.from_numpy(cols).to(dev)][:, 32 * blk:32 * blk + 32].cpu().numpy(), qc)
        assert np.array_equal(tiled_to_plain(mxt.col_s.cpu().numpy(), C, R // 32)[cols][:, blk:blk + 1], scc)
    # every GEMM on sampled outputs, from the GPU's (bit-exact) operands
    for name, lin, D, A, As, B, Bs, m, n, k in (
            ("up fwd", up, up.y, up.mx_x.row_q, up.mx_x.row_s, up.mx_w.row_q, up.mx_w.row_s, M, F, H),
            ("down fwd", down, down.y, down.mx_x.row_q, down.mx_x.row_s, down.mx_w.row_q, down.mx_w.row_s, M, H, F),
            ("down dgrad", down, down.dx, down.mx_dy.row_q, down.mx_dy.row_s, down.mx_w.col_q, down.mx_w.col_s,
             M, F, H),
            ("down wgrad", down, down.dw, down.mx_dy.col_q, down.mx_dy.col_s, down.mx_x.col_q, down.mx_x.col_s,
             H, F, M),
            ("up dgrad", up, up.dx, up.mx_dy.row_q, up.mx_dy.row_s, up.mx_w.col_q, up.mx_w.col_s, M, H, F),
            ("up wgrad", up, up.dw, up.mx_dy.col_q, up.mx_dy.col_s, up.mx_x.col_q, up.mx_x.col_s, F, H, M)):
        ms, ns = sample_elems(m, n, rng, n=512)
        um, un = np.unique(ms), np.unique(ns)
        Ah = A[torch.from_numpy(um).to(dev)].cpu().numpy()
        Bh = B[torch.from_numpy(un).to(dev)].cpu().numpy()
        Asp = tiled_to_plain(As.cpu().numpy(), m, k // 32)[um]
        Bsp = tiled_to_plain(Bs.cpu().numpy(), n, k // 32)[un]
        ref, absr = oracle.mx_gemm_elems(Ah, Asp, Bh, Bsp, None, np.searchsorted(um, ms), np.searchsorted(un, ns))
        check_gemm(D, ref, absr, ms, ns, what=name)
