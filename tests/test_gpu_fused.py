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
                                   (128, 256, 64), (272, 528, 256), (4096, 2576, 8208)])
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


def _codes_fmt(rng, fmt, shape, lim=8.0):
    tab = oracle.decode_table(fmt)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c]) and abs(tab[c]) <= lim], np.uint8)
    return ok[rng.integers(0, ok.size, shape)]


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (384, 768, 1040), (2048, 4096, 1024), (128, 256, 64),
                                   (272, 528, 256), (48, 80, 32), (4096, 2576, 8208)])
def test_fused_dgelu_epilogue_matches_unfused_and_oracle(M, N, K, monkeypatch):
    """fp8_gemm_dgelu_cast (fc2 dgrad with dGELU + E5M2 cast + amax + db1 in its epilogue)
    against fp8_gemm + fp8_dgelu_cast on the same pair kernel, and against the oracle."""
    import fp8_delayed_scaling_gb300 as fd
    monkeypatch.setenv("FP8DL_GEMM_VARIANT", "2sm")  # the unfused GEMM on the fused one's kernel
    dev = gpu()
    rng = np.random.default_rng(3 * M + 5 * N + K)
    A = torch.from_numpy(_codes_fmt(rng, 1, (M, K))).to(dev)  # qdY, E5M2
    B = torch.from_numpy(_codes_fmt(rng, 0, (N, K))).to(dev)  # qW2^T, E4M3
    h = wl.normal((M, N), 2.0, wl.generator(71, "fh/%d/%d" % (M, N)), torch.bfloat16)
    hd = h.to(dev)
    sa = torch.tensor([0.05], device=dev)
    sb = torch.tensor([0.03], device=dev)
    qs = torch.tensor([1024.0], device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    bf = dict(dtype=torch.bfloat16, device=dev)
    ws_f = torch.empty(fd.fp8_gemm_dgelu_workspace_size(M, N), **u8)
    ws_u = torch.empty(fd.fp8_cast_workspace_size(M, N), **u8)
    dg1, dg2 = torch.full((M, N), float("nan"), **bf), torch.full((M, N), float("nan"), **bf)
    dh1, dh2 = torch.empty((M, N), **bf), torch.empty((M, N), **bf)
    q1, q2, q3 = (torch.full((M, N), 0xAA, **u8) for _ in range(3))
    t1, t2, t3 = (torch.full((N, M), 0xAA, **u8) for _ in range(3))
    a1, a2, a3 = (torch.zeros(1, device=dev) for _ in range(3))
    db1, db2, db3 = (torch.full((N,), float("nan"), device=dev) for _ in range(3))
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fd.fp8_gemm_dgelu_cast(A, fd.E5M2, B, fd.E4M3, sa, sb, hd, fd.E5M2, qs, q1, t1, a1, dbias=db1, workspace=ws_f,
                           dg=dg1, dh=dh1, dev_status=st)
    fd.fp8_gemm(A, fd.E5M2, B, fd.E4M3, sa, sb, dg2)
    fd.fp8_dgelu_cast(dg2, hd, fd.E5M2, qs, out=q2, out_t=t2, amax=a2, dbias=db2, workspace=ws_u, dh=dh2)
    # the production form: neither dg nor dh leaves the chip
    fd.fp8_gemm_dgelu_cast(A, fd.E5M2, B, fd.E4M3, sa, sb, hd, fd.E5M2, qs, q3, t3, a3, dbias=db3, workspace=ws_f)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert torch.equal(dg1, dg2) and torch.equal(dh1, dh2)
    assert torch.equal(q1, q2) and torch.equal(t1, t2) and a1.item() == a2.item()
    assert torch.equal(q3, q1) and torch.equal(t3, t1) and a3.item() == a1.item()
    assert torch.equal(db3, db1)  # a fixed summation order
    dhb = host(dh1)
    s, sabs = oracle.colsum(dhb)
    for db in (db1, db2):
        assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - s) <= M * 2.0 ** -24 * sabs + 1e-30)
    # against the oracle: the GEMM within bound, dGELU within bound, codes bit-exact from dh
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ms, ns = ms.ravel(), ns.ravel()
    if ms.size > 200000:
        sel = rng.choice(ms.size, 200000, replace=False)
        ms, ns = ms[sel], ns[sel]
    ref, absr = oracle.gemm_elems(A.cpu().numpy(), 1, B.cpu().numpy(), 0, 0.05, 0.03, None, ms, ns)
    check_gemm(dg1, ref, absr, ms, ns, what="fused dg")
    dr = oracle.dgelu(host(dg1), host(h))
    assert np.all(np.abs(as_f64(dh1) - dr) <= 2.0 ** -7 * np.abs(dr) + 2.0 ** -21 * np.abs(as_f64(dg1)))
    qo = oracle.quantize(1, dhb, 1024.0)
    assert np.array_equal(q1.cpu().numpy(), qo) and np.array_equal(t1.cpu().numpy(), qo.T)
    assert a1.item() == oracle.amax(dhb)


@pytest.mark.parametrize("M,N,K", [(256, 512, 128), (384, 1024, 256)])
def test_epilogue_16_byte_aligned_outputs(M, N, K, monkeypatch):
    """Outputs whose base is 16- but not 32-byte aligned take the 16-byte store path of the
    pair epilogue; their contents equal those written through 32-byte aligned outputs."""
    import fp8_delayed_scaling_gb300 as fd
    monkeypatch.setenv("FP8DL_GEMM_VARIANT", "2sm")
    dev = gpu()
    rng = np.random.default_rng(7 * M + N + K)
    A = torch.from_numpy(_codes(rng, (M, K))).to(dev)
    B = torch.from_numpy(_codes(rng, (N, K))).to(dev)
    sa = torch.tensor([0.05], device=dev)
    sb = torch.tensor([0.03], device=dev)
    bias = wl.normal((N,), 0.5, wl.generator(72, "abias/%d" % N), torch.bfloat16).to(dev)
    qs = torch.tensor([37.0], device=dev)
    u8 = dict(dtype=torch.uint8, device=dev)

    def outputs(offset):
        hb = torch.full((M * N + 16,), float("nan"), dtype=torch.bfloat16, device=dev)
        qb = torch.full((M * N + 32,), 0xAA, **u8)
        H = hb[offset // 2: offset // 2 + M * N].view(M, N)
        q = qb[offset: offset + M * N].view(M, N)
        assert H.data_ptr() % 32 == offset and q.data_ptr() % 32 == offset
        return H, q, torch.full((N, M), 0xAA, **u8), torch.zeros(1, device=dev)

    res = []
    for offset in (0, 16):
        H, q, t, a = outputs(offset)
        fd.fp8_gemm_gelu_cast(A, fd.E4M3, B, fd.E4M3, sa, sb, H, fd.E4M3, qs, q, t, a, bias=bias)
        D = outputs(offset)[0]
        fd.fp8_gemm(A, fd.E4M3, B, fd.E4M3, sa, sb, D, bias=bias)
        res.append((H, q, t, a, D))
    torch.cuda.synchronize()
    (H0, q0, t0, a0, D0), (H1, q1, t1, a1, D1) = res
    assert not torch.isnan(H0.float()).any() and not torch.isnan(D0.float()).any()
    assert torch.equal(H0, H1) and torch.equal(q0, q1) and torch.equal(t0, t1) and a0.item() == a1.item()
    assert torch.equal(D0, D1)


def test_fused_epilogues_independent_of_tile_order(monkeypatch):
    """The fused GELU and dGELU GEMMs write the same bits under any tile order and group
    size: every output element, code, bias-gradient partial and the amax (a max) depend
    only on their own tile."""
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    M, N, K = 1040, 784, 512
    rng = np.random.default_rng(11)
    A = torch.from_numpy(_codes(rng, (M, K))).to(dev)
    B = torch.from_numpy(_codes(rng, (N, K))).to(dev)
    sa = torch.tensor([0.05], device=dev)
    sb = torch.tensor([0.03], device=dev)
    qs = torch.tensor([37.0], device=dev)
    h = wl.normal((M, N), 2.0, wl.generator(73, "oh"), torch.bfloat16).to(dev)
    u8 = dict(dtype=torch.uint8, device=dev)
    ws = torch.empty(fd.fp8_gemm_dgelu_workspace_size(M, N), **u8)
    res = []
    for order, group in (("", ""), ("n", "3"), ("m", "1")):
        monkeypatch.setenv("FP8DL_GEMM_RASTER", order)
        monkeypatch.setenv("FP8DL_GEMM_GROUP", group)
        H = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        q, qt = torch.empty((M, N), **u8), torch.empty((N, M), **u8)
        a = torch.zeros(1, device=dev)
        fd.fp8_gemm_gelu_cast(A, fd.E4M3, B, fd.E4M3, sa, sb, H, fd.E4M3, qs, q, qt, a)
        q2, qt2 = torch.empty((M, N), **u8), torch.empty((N, M), **u8)
        a2 = torch.zeros(1, device=dev)
        db = torch.empty(N, device=dev)
        fd.fp8_gemm_dgelu_cast(A, fd.E4M3, B, fd.E4M3, sa, sb, h, fd.E5M2, qs, q2, qt2, a2, dbias=db, workspace=ws)
        torch.cuda.synchronize()
        res.append((H, q, qt, a, q2, qt2, a2, db))
    for other in res[1:]:
        for x, y in zip(res[0], other):
            assert torch.equal(x, y)
