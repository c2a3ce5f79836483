"""Concurrent first use: the library's per-device set-up (device check, function
attributes, occupancy of the cluster kernels, the static scratch address) runs
once under a lock while several host threads make their first calls together, on
one stream (the allocation-free cast's shared scratch needs that).
Runs in a fresh process so that the set-up has not happened yet; every thread's
results must equal a serial rerun bit for bit (the kernels are deterministic)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r'''
import threading, torch
import fp8_delayed_scaling_gb300 as fd
dev = torch.device("cuda", 0)
torch.cuda.set_device(dev)
T, R, C = 8, 256, 4096
g = torch.Generator().manual_seed(7)
xs = [torch.randn(R, C, generator=g).to(torch.bfloat16).to(dev) for _ in range(T)]
gam = torch.ones(C, dtype=torch.bfloat16, device=dev)
bet = torch.zeros(C, dtype=torch.bfloat16, device=dev)
sc = torch.ones(1, device=dev)

def work(i, out):
    torch.cuda.set_device(dev)
    x = xs[i]
    q = torch.empty(R, C, dtype=torch.uint8, device=dev)
    qt = torch.empty(C, R, dtype=torch.uint8, device=dev)
    mu = torch.empty(R, device=dev); rs = torch.empty(R, device=dev)
    fd.fp8_layernorm_cast(x, gam, bet, 1e-5, fd.E4M3, sc, mu, rs, out=q, out_t=qt)
    D = torch.empty(R, R, dtype=torch.bfloat16, device=dev)
    fd.fp8_gemm(q, fd.E4M3, q[:R], fd.E4M3, sc, sc, D)
    rq = torch.empty(R, C, dtype=torch.uint8, device=dev)
    rsf = torch.empty(fd._lib.mxfp8_scale_bytes(R, C), dtype=torch.uint8, device=dev)
    fd.mxfp8_quantize(x, rq, rsf)
    cq = torch.empty(R, C, dtype=torch.uint8, device=dev)
    db = torch.empty(C, device=dev)
    fd.fp8_cast_amax_transpose_noalloc(x, fd.E5M2, sc, out=cq, dbias=db)
    torch.cuda.synchronize()
    out[i] = [t.cpu() for t in (q, qt, mu, rs, D, rq, rsf, cq, db)]

first = [None] * T
barrier = threading.Barrier(T)
def run(i):
    barrier.wait()
    work(i, first)
ts = [threading.Thread(target=run, args=(i,)) for i in range(T)]
for t in ts: t.start()
for t in ts: t.join()
again = [None] * T
for i in range(T):
    work(i, again)
names = ["q", "q_t", "mu", "rsigma", "gemm", "mx codes", "mx scales", "cast codes", "dbias"]
for i in range(T):
    assert first[i] is not None, i
    for name, a, b in zip(names, first[i], again[i]):
        assert torch.equal(a, b), (i, name)
print("threads ok")
'''


def test_concurrent_first_calls_from_host_threads():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", SCRIPT], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
