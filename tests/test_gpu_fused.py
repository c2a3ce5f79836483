"""The fused fc1 epilogue (fp8_gemm_gelu_cast): GEMM + bias -> bf16 H, GELU,
FP8 cast with amax and transposed codes in one kernel.  Checked bit for bit
against the unfused path (fp8_gemm then fp8_gelu_cast, itself checked against
the oracle), and against the oracle directly."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import as_f64, check_gemm, gpu, host

pytestmark = pytest.mark.gpu


def _codes(rng, shape):
    tab = oracle.decode_table(0)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c]) and abs(tab[c]) <= 8], np.uint8)
    return ok[rng.integers(0, ok.size, shape)]


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (512, 1024, 256), (384, 768, 1040), (2048, 4096, 1024),
                                   (128, 256, 64), (272, 528, 256)])
def test_fused_gelu_epilogue_matches_unfused_and_oracle(M, N, K):
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    rng = np.random.default_rng(M + N + K)
    A = torch.from_numpy(_codes(rng, (M, K))).to(dev)
    B = torch.from_numpy(_codes(rng, (N, K))).to(dev)
    sa = torch.tensor([0.05], device=dev)
    sb = torch.tensor([0.03], device=dev)
    bias = wl.normal((N,), 0.5, wl.generator(70, "fbias/%d" % N), torch.bfloat16).to(dev)
    qs = torch.tensor([37.0], device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    H1, H2 = (torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev) for _ in range(2))
    q1, q2 = torch.full((M, N), 0xAA, **u8), torch.full((M, N), 0xAA, **u8)
    t1, t2 = torch.full((N, M), 0xAA, **u8), torch.full((N, M), 0xAA, **u8)
    a1, a2 = torch.zeros(1, device=dev), torch.zeros(1, device=dev)
    g1, g2 = (torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(2))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fd.fp8_gemm_gelu_cast(A, fd.E4M3, B, fd.E4M3, sa, sb, H1, fd.E4M3, qs, q1, t1, a1, bias=bias, g=g1, dev_status=st)
    fd.fp8_gemm(A, fd.E4M3, B, fd.E4M3, sa, sb, H2, bias=bias)
    fd.fp8_gelu_cast(H2, fd.E4M3, qs, out=q2, out_t=t2, amax=a2, g=g2)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(H1, H2)
    assert torch.equal(g1, g2)
    assert torch.equal(q1, q2) and torch.equal(t1, t2)
    assert a1.item() == a2.item()
    # against the oracle: the GEMM within bound, GELU within bound, codes bit-exact from g
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ms, ns = ms.ravel(), ns.ravel()
    if ms.size > 200000:
        sel = rng.choice(ms.size, 200000, replace=False)
        ms, ns = ms[sel], ns[sel]
    ref, absr = oracle.gemm_elems(A.cpu().numpy(), 0, B.cpu().numpy(), 0, 0.05, 0.03, host(bias), ms, ns)
    check_gemm(H1, ref, absr, ms, ns, what="fused H")
    hb = host(H1)
    gr = oracle.gelu(hb)
    assert np.all(np.abs(as_f64(g1) - gr) <= 2.0 ** -7 * np.abs(gr) + 2.0 ** -21 * np.abs(as_f64(H1)))
    gb = host(g1)
    qo = oracle.quantize(0, gb, 37.0)
    assert np.array_equal(q1.cpu().numpy(), qo) and np.array_equal(t1.cpu().numpy(), qo.T)
    assert a1.item() == oracle.amax(gb)
