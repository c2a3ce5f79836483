"""fp8_autocast around te.Linear steps: the exit's update is the same launch a
manual step loop makes, so the state evolves bit for bit alike."""
import numpy as np
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu


def _run(use_autocast):
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    M, K, N = 256, 384, 512
    recipe = fd.Recipe(margin=1, interval=2, fp8_format=fd.FORMAT_HYBRID, amax_history_len=4)
    state = make_state(recipe, 1, device=dev)
    w = wl.normal((N, K), 0.02, wl.generator(90, "W"), torch.bfloat16).to(dev)
    lin = Fp8Linear(state, 0, w, None, M)
    ys = []
    for step in range(5):
        x = wl.normal((M, K), 1.0 + step, wl.generator(90, "X", step), torch.bfloat16).to(dev)
        dy = wl.normal((M, N), 1e-3, wl.generator(90, "dY", step), torch.bfloat16).to(dev)
        if step == 0:
            lin.seed_forward(x)
            lin.seed_backward(dy)
        if use_autocast:
            with fd.fp8_autocast(state):
                ys.append(lin.forward(x).clone())
                lin.backward(dy)
        else:
            ys.append(lin.forward(x).clone())
            lin.backward(dy)
            state.update(step)
    torch.cuda.synchronize()
    return state.buf.cpu().numpy(), [y.cpu() for y in ys]


def test_autocast_matches_manual_updates():
    a, ya = _run(True)
    b, yb = _run(False)
    assert np.array_equal(a, b)
    assert all(torch.equal(p, q) for p, q in zip(ya, yb))
