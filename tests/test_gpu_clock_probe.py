"""fp8dl_clock_probe: one record per CTA (SM id, cycle counter, global timer), and two
probes around GPU work give a plausible mean SM clock."""
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_clock_probe_records_and_mean_clock():
    import bench
    import fp8_delayed_scaling_gb300 as fd
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    stream = torch.cuda.current_stream()
    n0 = fd.fp8dl_kernel_launches()
    cyc = bench.CycleClock(dev, stream)
    a = torch.randn(4096, 4096, device=dev, dtype=torch.bfloat16)
    cyc.mark(0)
    for _ in range(50):  # tens of milliseconds of work on every SM
        a = torch.tanh(a @ a * 0.01)
    cyc.mark(1)
    torch.cuda.synchronize()
    assert fd.fp8dl_kernel_launches() - n0 == 2
    for k in range(2):
        rec = cyc.buf[k].view(-1, 3).cpu()
        assert (rec[:, 0] >= 0).all() and (rec[:, 0] < sms).all()  # SM ids
        assert (rec[:, 1] > 0).all() and (rec[:, 2] > 0).all()
    t0, t1 = cyc.buf[0].view(-1, 3)[:, 2].max().item(), cyc.buf[1].view(-1, 3)[:, 2].min().item()
    assert t1 > t0  # the second probe ran after the first
    mhz, n_sm = cyc.mhz()
    assert n_sm >= sms // 2
    assert 200 < mhz < 2300
