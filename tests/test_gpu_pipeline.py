"""HostStepPipeline: steps over pinned host inputs/outputs with the copies on their own
streams give, step by step, exactly the host outputs of plain in-order steps."""
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu

M, K, N = 256, 384, 512


def _layer(dev):
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    recipe = fd.Recipe(margin=0, interval=1, fp8_format=fd.FORMAT_HYBRID, amax_history_len=4)
    state = make_state(recipe, 1, device=dev)
    w = wl.normal((N, K), 0.02, wl.generator(91, "W"), torch.bfloat16).to(dev)
    b = torch.zeros(N, dtype=torch.bfloat16, device=dev)
    lin = Fp8Linear(state, 0, w, b, M)
    x0 = wl.normal((M, K), 1.0, wl.generator(91, "X0"), torch.bfloat16).to(dev)
    dy0 = wl.normal((M, N), 1e-3, wl.generator(91, "dY0"), torch.bfloat16).to(dev)
    lin.seed_forward(x0)
    lin.seed_backward(dy0)
    return state, lin, x0, dy0


def test_pipelined_steps_match_in_order_steps():
    from fp8_delayed_scaling_gb300.pipeline import HostStepPipeline
    dev = gpu()
    steps = 5
    # distinct host inputs per step (growing scale, so every step's scales move)
    hx = [wl.normal((M, K), 1.0 + 3 * i, wl.generator(91, "X", i), torch.bfloat16).pin_memory() for i in range(steps)]
    hdy = [wl.normal((M, N), 1e-3 * (1 + i), wl.generator(91, "dY", i), torch.bfloat16).pin_memory()
           for i in range(steps)]

    # in order: copy in, step, copy out, wait
    state, lin, x, dy = _layer(dev)
    ref = []
    for i in range(steps):
        x.copy_(hx[i])
        dy.copy_(hdy[i])
        lin.forward(x)
        lin.backward(dy)
        state.update(i)
        ref.append([t.cpu() for t in (lin.dx, lin.dw, lin.db, lin.y)])

    # pipelined
    state, lin, x, dy = _layer(dev)
    outs = [[torch.empty_like(t, device="cpu").pin_memory() for t in (lin.dx, lin.dw, lin.db, lin.y)]
            for _ in range(steps)]
    pipe = HostStepPipeline([x, dy], [lin.dx, lin.dw, lin.db, lin.y])
    count = [0]

    def step(ins):
        lin.forward(ins[0])
        lin.backward(ins[1])
        state.update(count[0])
        count[0] += 1

    pipe.run(steps, step, lambda i: [hx[i], hdy[i]], lambda i: outs[i])
    torch.cuda.synchronize()
    for i in range(steps):
        for a, b in zip(outs[i], ref[i]):
            assert torch.equal(a, b), "step %d" % i


def test_pipelined_steps_with_two_output_sets_match_in_order_steps():
    """out_sets=True: each step writes its products straight into output set i%2 (no
    snapshot copy); step i+2 waits for the host copy of step i's set."""
    from fp8_delayed_scaling_gb300.pipeline import HostStepPipeline
    dev = gpu()
    steps = 5
    hx = [wl.normal((M, K), 1.0 + 3 * i, wl.generator(92, "X", i), torch.bfloat16).pin_memory() for i in range(steps)]
    hdy = [wl.normal((M, N), 1e-3 * (1 + i), wl.generator(92, "dY", i), torch.bfloat16).pin_memory()
           for i in range(steps)]
    names = ("dx", "dw", "db", "y")

    state, lin, x, dy = _layer(dev)
    ref = []
    for i in range(steps):
        x.copy_(hx[i])
        dy.copy_(hdy[i])
        lin.forward(x)
        lin.backward(dy)
        state.update(i)
        ref.append([getattr(lin, n).cpu() for n in names])

    state, lin, x, dy = _layer(dev)
    outs = [[torch.empty_like(getattr(lin, n), device="cpu").pin_memory() for n in names] for _ in range(steps)]
    pipe = HostStepPipeline([x, dy], [getattr(lin, n) for n in names], out_sets=True)
    assert pipe.out_sets[0][0] is not pipe.out_sets[1][0]
    count = [0]

    def step(ins, outs_dev):
        for n, t in zip(names, outs_dev):
            setattr(lin, n, t)
        lin.forward(ins[0])
        lin.backward(ins[1])
        state.update(count[0])
        count[0] += 1

    pipe.run(steps, step, lambda i: [hx[i], hdy[i]], lambda i: outs[i])
    torch.cuda.synchronize()
    for i in range(steps):
        for n, a, b in zip(names, outs[i], ref[i]):
            assert torch.equal(a, b), "step %d %s" % (i, n)
