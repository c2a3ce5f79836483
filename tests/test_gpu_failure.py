"""Failure detection without a GPU fault: bounded waits report a timeout
through a device status word and leave the context usable; bad arguments fail
on the host before any launch; checkpoint/resume of the scaling state."""
import pytest
import torch

import workloads as wl
from helpers import gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    st = torch.full((4,), 12345, dtype=torch.int32, device=dev)
    fd.fp8dl_wait_selftest(20_000_000, False, st)  # ~10 ms at GB300 clocks; nothing completes the phase
    torch.cuda.synchronize()
    assert st[0].item() == fd.ERR_TIMEOUT
    st.fill_(12345)
    fd.fp8dl_wait_selftest(20_000_000, True, st)  # positive control: the phase completes
    torch.cuda.synchronize()
    assert st[0].item() == fd.OK
    # the context still runs real work afterwards
    x = torch.ones((32, 32), dtype=torch.bfloat16, device=dev)
    amax = torch.zeros(1, dtype=torch.float32, device=dev)
    fd.fp8_cast_amax_transpose(x, fd.E4M3, None, amax=amax)
    torch.cuda.synchronize()
    assert amax.item() == 1.0


def test_invalid_calls_fail_before_launch():
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    x = torch.zeros((24, 32), dtype=torch.bfloat16, device=dev)  # 24 rows: not a multiple of 16
    with pytest.raises(fd.FP8DLError) as e:
        fd.fp8_cast_amax_transpose(x, fd.E4M3, None, amax=torch.zeros(1, device=dev))
    assert e.value.status == fd.ERR_SHAPE
    a = torch.zeros((32, 40), dtype=torch.uint8, device=dev)  # K = 40: not a multiple of 16
    d = torch.zeros((32, 32), dtype=torch.bfloat16, device=dev)
    one = torch.ones(1, device=dev)
    with pytest.raises(fd.FP8DLError) as e:
        fd.fp8_gemm(a, fd.E4M3, a.clone(), fd.E4M3, one, one, d)
    assert e.value.status == fd.ERR_SHAPE
    torch.cuda.synchronize()


def test_checkpoint_resume_is_bit_identical():
    """Save the scaling state block at step k, restore it into a fresh state and
    continue: scales and histories match an uninterrupted run exactly."""
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.linear import Fp8Linear, make_state
    dev = gpu()
    M, K, N = 256, 512, 768
    recipe = fd.Recipe(margin=1, interval=2, fp8_format=fd.FORMAT_HYBRID, amax_history_len=5)
    w = wl.normal((N, K), 0.02, wl.generator(8, "ckpt-W"), torch.bfloat16).to(dev)
    xs = [wl.student_t3((M, K), 0.5, wl.generator(8, "ckpt-X", t)).to(dev) for t in range(8)]
    dys = [wl.normal((M, N), 1e-3, wl.generator(8, "ckpt-dY", t), torch.bfloat16).to(dev) for t in range(8)]

    def run(state, lin, lo, hi):
        for t in range(lo, hi):
            if t == 0:
                lin.seed_forward(xs[t])
            lin.forward(xs[t])
            if t == 0:
                lin.seed_backward(dys[t])
            lin.backward(dys[t])
            state.update(t)

    sa = make_state(recipe, 1, device=dev)
    la = Fp8Linear(sa, 0, w, None, M)
    run(sa, la, 0, 8)
    sb = make_state(recipe, 1, device=dev)
    lb = Fp8Linear(sb, 0, w, None, M)
    run(sb, lb, 0, 4)
    torch.cuda.synchronize()
    saved = sb.buf.cpu().clone()  # the checkpoint: plain bytes
    sc = make_state(recipe, 1, device=dev)
    sc.buf.copy_(saved.to(dev))
    lc = Fp8Linear(sc, 0, w, None, M)
    run(sc, lc, 4, 8)
    torch.cuda.synchronize()
    assert torch.equal(sa.buf.cpu(), sc.buf.cpu())
    assert torch.equal(la.qdy.cpu(), lc.qdy.cpu()) and torch.equal(la.dw.cpu(), lc.dw.cpu())
