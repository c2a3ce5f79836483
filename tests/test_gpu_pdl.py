"""Programmatic dependent launch changes no output bit: the te.Linear workload (2048 x 768 ->
3072, fwd + bwd, three steps; every call short enough to launch programmatically) in two
processes, FP8DL_PDL=0 and FP8DL_PDL=1, gives identical outputs and scaling state."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CODE = r"""
import sys, torch
import bench
dev = torch.device("cuda", 0)
model = bench.Model(bench.WORKLOADS["linear_hybrid"], dev, 1)
for _ in range(3):
    model.step()
torch.cuda.synchronize()
torch.save([t.detach().cpu() for t in model.outputs()] + [model.state.buf.cpu()], sys.argv[1])
"""


def test_programmatic_launch_changes_no_bit(tmp_path):
    res = []
    for pdl in ("0", "1"):
        f = str(tmp_path / ("out%s.pt" % pdl))
        env = dict(os.environ, FP8DL_PDL=pdl)
        r = subprocess.run([sys.executable, "-c", CODE, f], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        res.append(torch.load(f))
    assert len(res[0]) == len(res[1]) > 1
    for a, b in zip(*res):
        assert a.dtype == b.dtype and torch.equal(a, b)
