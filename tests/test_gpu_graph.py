"""StepGraph: te.Linear steps replayed from CUDA graphs (one per residue of the step
counter modulo the recipe's interval) give, step by step, the eager steps' outputs and
scaling state bit for bit, with new inputs copied into the captured buffers each step."""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu

M, K, N = 256, 384, 512
STEPS = 7


def _setup(dev):
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    recipe = fd.Recipe(margin=1, interval=2, fp8_format=fd.FORMAT_HYBRID, amax_history_len=4)
    state = make_state(recipe, 1, device=dev)
    w = wl.normal((N, K), 0.02, wl.generator(92, "W"), torch.bfloat16).to(dev)
    b = torch.zeros(N, dtype=torch.bfloat16, device=dev)
    lin = Fp8Linear(state, 0, w, b, M)
    x = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dy = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    return state, lin, x, dy


def _inputs(i):
    x = wl.normal((M, K), 1.0 + 2 * i, wl.generator(92, "X", i), torch.bfloat16)
    dy = wl.normal((M, N), 1e-3 * (1 + i), wl.generator(92, "dY", i), torch.bfloat16)
    return x, dy


def test_graph_replay_matches_eager_steps():
    from fp8_delayed_scaling_gb300.graph import StepGraph
    dev = gpu()
    outs = {}
    for mode in ("eager", "graph"):
        state, lin, x, dy = _setup(dev)
        x0, dy0 = _inputs(0)
        x.copy_(x0)
        dy.copy_(dy0)
        lin.seed_forward(x)
        lin.seed_backward(dy)

        def step(n):
            lin.forward(x)
            lin.backward(dy)
            state.update(n)

        res = []
        if mode == "eager":
            for i in range(STEPS):
                xi, dyi = _inputs(i)
                x.copy_(xi)
                dy.copy_(dyi)
                step(i)
                res.append([t.clone() for t in (lin.y, lin.dx, lin.dw, lin.db)] + [state.buf.clone()])
        else:
            g = StepGraph(step, interval=2, warmup=1)  # runs step 0 eagerly
            res.append([t.clone() for t in (lin.y, lin.dx, lin.dw, lin.db)] + [state.buf.clone()])
            for i in range(1, STEPS):
                xi, dyi = _inputs(i)
                x.copy_(xi)
                dy.copy_(dyi)
                g.replay(i)
                res.append([t.clone() for t in (lin.y, lin.dx, lin.dw, lin.db)] + [state.buf.clone()])
        torch.cuda.synchronize()
        outs[mode] = res
    for i in range(STEPS):
        for a, b in zip(outs["eager"][i], outs["graph"][i]):
            assert torch.equal(a, b), "step %d" % i
    # the scales moved during the run (the test exercises both graphs' updates)
    s0 = outs["eager"][0][-1].cpu().numpy()
    s6 = outs["eager"][-1][-1].cpu().numpy()
    assert not np.array_equal(s0, s6)
