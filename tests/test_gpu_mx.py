"""GPU parity of MXFP8 quantisation (bit-exact codes and E8M0 scales) and of the
block-scaled GEMM (error bound per element) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import check_gemm, gpu, host, sample_elems

pytestmark = pytest.mark.gpu


def sf_index(R, NB):
    """Byte offsets of S[r][b] in the tiled scale layout of include/fp8dl.h."""
    kg = (NB + 3) // 4
    r = np.arange(R, dtype=np.int64)[:, None]
    b = np.arange(NB, dtype=np.int64)[None, :]
    return ((r >> 7) * kg + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)


def tiled_to_plain(buf, R, NB):
    return np.asarray(buf)[sf_index(R, NB)]


def plain_to_tiled(S, R, NB):
    import fp8_delayed_scaling_gb300 as fd
    out = np.full(fd._lib.mxfp8_scale_bytes(R, 32 * NB), 127, np.uint8)
    out[sf_index(R, NB)] = S
    return out


def _quantize(x, dev):
    import fp8_delayed_scaling_gb300 as fd
    R, C = x.shape
    rq = torch.full((R, C), 0xAA, dtype=torch.uint8, device=dev)
    cq = torch.full((C, R), 0xAA, dtype=torch.uint8, device=dev)
    rs = torch.full((fd._lib.mxfp8_scale_bytes(R, C),), 0xAA, dtype=torch.uint8, device=dev)
    cs = torch.full((fd._lib.mxfp8_scale_bytes(C, R),), 0xAA, dtype=torch.uint8, device=dev)
    fd.mxfp8_quantize(x.to(dev), rq, rs, cq, cs)
    torch.cuda.synchronize()
    return rq, rs, cq, cs


@pytest.mark.parametrize("shape", [(32, 32), (64, 96), (128, 256), (160, 288), (512, 1024), (96, 800)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_quantize_parity(shape, dtype):
    dev = gpu()
    R, C = shape
    g = wl.generator(41, "mxq/%s/%s" % (shape, dtype))
    x = wl.channel_scaled_normal(R, C, g).to(dtype)
    rq, rs, cq, cs = _quantize(x, dev)
    xs = host(x)
    q, s = oracle.mx_quantize_rows(xs)
    qc, sc = oracle.mx_quantize_cols(xs)
    assert np.array_equal(rq.cpu().numpy(), q)
    assert np.array_equal(tiled_to_plain(rs.cpu().numpy(), R, C // 32), s)
    assert np.array_equal(cq.cpu().numpy(), qc)
    assert np.array_equal(tiled_to_plain(cs.cpu().numpy(), C, R // 32), sc)
    # padding entries of the tiled layout are 127
    for buf, rr, nb in ((rs, R, C // 32), (cs, C, R // 32)):
        b = buf.cpu().numpy()
        mask = np.ones(b.size, bool)
        mask[sf_index(rr, nb).ravel()] = False
        assert np.all(b[mask] == 127)


@pytest.mark.parametrize("shape", [(32, 32), (160, 288), (512, 1024), (96, 800), (384, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_mx_quantize_dbias(shape, dtype):
    """Column sums fused into the quantisation: within rows * 2^-24 * sum|x| of the oracle's
    fp64 sums (partial 128-row tiles included), the same bits on a second call, and the codes
    and scales unchanged by the extra output."""
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    R, C = shape
    g = wl.generator(42, "mxq-dbias/%s/%s" % (shape, dtype))
    x = (wl.channel_scaled_normal(R, C, g) * 1e-2).to(dtype)
    xd = x.to(dev)
    rq0, rs0, cq0, cs0 = _quantize(x, dev)
    ws = torch.full((fd.fp8_cast_workspace_size(R, C),), 0xFF, dtype=torch.uint8, device=dev)  # NaN-filled scratch
    res = []
    for outs in (("row", "col"), ("row",), ("col",), ("row", "col")):
        rq = torch.empty((R, C), dtype=torch.uint8, device=dev) if "row" in outs else None
        rs = torch.empty((fd._lib.mxfp8_scale_bytes(R, C),), dtype=torch.uint8, device=dev) if "row" in outs else None
        cq = torch.empty((C, R), dtype=torch.uint8, device=dev) if "col" in outs else None
        cs = torch.empty((fd._lib.mxfp8_scale_bytes(C, R),), dtype=torch.uint8, device=dev) if "col" in outs else None
        db = torch.full((C,), float("nan"), dtype=torch.float32, device=dev)
        fd.mxfp8_quantize(xd, rq, rs, cq, cs, dbias=db, workspace=ws)
        torch.cuda.synchronize()
        if rq is not None:
            assert torch.equal(rq, rq0) and torch.equal(rs, rs0)
        if cq is not None:
            assert torch.equal(cq, cq0) and torch.equal(cs, cs0)
        res.append(db.cpu().numpy())
    s, sabs = oracle.colsum(host(x))
    for d in res:
        assert np.array_equal(d, res[0])  # a fixed summation order
    assert np.all(np.abs(res[0].astype(np.float64) - s) <= R * 2.0 ** -24 * sabs + 1e-30)


def test_mx_quantize_special_blocks():
    """Blocks of zeros, powers of two, 448*2^k and values just above it, subnormals."""
    dev = gpu()
    R, C = 32, 256
    x = np.zeros((R, C), np.float32)
    x[1, :32] = 1.0
    x[2, :32] = 448.0 * 8
    x[3, :32] = np.float32(448.0 * 8) * np.float32(1 + 2 ** -23)
    x[4, :32] = 1e-40
    x[5, 32:64] = np.linspace(-3, 3, 32)
    x[6, :] = (2.0 ** np.arange(-128, 128, dtype=np.float64)).astype(np.float32)  # finite: 2^-128 .. 2^127
    x[7, :] = -np.abs(x[6, :])
    xt = torch.from_numpy(x)
    rq, rs, cq, cs = _quantize(xt, dev)
    q, s = oracle.mx_quantize_rows(x)
    assert np.array_equal(rq.cpu().numpy(), q)
    assert np.array_equal(tiled_to_plain(rs.cpu().numpy(), R, C // 32), s)
    qc, sc = oracle.mx_quantize_cols(x)
    assert np.array_equal(cq.cpu().numpy(), qc)
    assert np.array_equal(tiled_to_plain(cs.cpu().numpy(), C, R // 32), sc)


def _mx_gemm(A, As, B, Bs, dev, bias=None, d_dtype=torch.bfloat16):
    import fp8_delayed_scaling_gb300 as fd
    M, K = A.shape
    N = B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=d_dtype, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    fd.mxfp8_gemm(torch.from_numpy(A).to(dev), torch.from_numpy(plain_to_tiled(As, M, K // 32)).to(dev),
                  torch.from_numpy(B).to(dev), torch.from_numpy(plain_to_tiled(Bs, N, K // 32)).to(dev), D,
                  bias=bias, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    return D


def _codes(rng, shape):
    tab = oracle.decode_table(0)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c])], np.uint8)
    return ok[rng.integers(0, ok.size, shape)]


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (32, 32, 32), (96, 160, 64), (256, 512, 384), (160, 288, 96),
                                   (384, 768, 1024), (1024, 2048, 512), (288, 544, 320), (640, 416, 2080)])
def test_mx_gemm_parity(M, N, K):
    dev = gpu()
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    As = rng.integers(118, 136, (M, K // 32)).astype(np.uint8)
    Bs = rng.integers(118, 136, (N, K // 32)).astype(np.uint8)
    D = _mx_gemm(A, As, B, Bs, dev)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, absr = oracle.mx_gemm_elems(A, As, B, Bs, None, ms.ravel(), ns.ravel())
    check_gemm(D, ref, absr, ms.ravel(), ns.ravel(), what="mx gemm")


def test_mx_gemm_alternating_k_order(monkeypatch):
    """With K > 8192 and at least two waves of tiles every other tile of a CTA sums its k-blocks (and their
    block scales) last to first: within the oracle's bound on sampled elements, the same bits
    on a repeated call, and different rounding from the first-to-last order
    (FP8DL_GEMM_SNAKE=0), which meets the bound too."""
    dev = gpu()
    M, N, K = 4096, 2560, 8224  # 32 x 10 = 320 tiles of 128 x 256 (over two waves of 152 CTAs), K > 8192
    rng = np.random.default_rng(23)
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    As = rng.integers(118, 136, (M, K // 32)).astype(np.uint8)
    Bs = rng.integers(118, 136, (N, K // 32)).astype(np.uint8)
    D1 = _mx_gemm(A, As, B, Bs, dev)
    D2 = _mx_gemm(A, As, B, Bs, dev)
    monkeypatch.setenv("FP8DL_GEMM_SNAKE", "0")
    D0 = _mx_gemm(A, As, B, Bs, dev)
    assert torch.equal(D1, D2)
    assert not torch.equal(D1, D0)
    ms, ns = sample_elems(M, N, np.random.default_rng(8), n=4096)
    ref, absr = oracle.mx_gemm_elems(A, As, B, Bs, None, ms, ns)
    check_gemm(D1, ref, absr, ms, ns, what="mx alternating K order")
    check_gemm(D0, ref, absr, ms, ns, what="mx first-to-last K order")


@pytest.mark.parametrize("d_dtype", [torch.bfloat16, torch.float32])
def test_mx_gemm_bias_and_fp32_out(d_dtype):
    dev = gpu()
    rng = np.random.default_rng(4)
    M, N, K = 256, 544, 256
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    As = rng.integers(110, 140, (M, K // 32)).astype(np.uint8)
    Bs = rng.integers(110, 140, (N, K // 32)).astype(np.uint8)
    bias = wl.normal((N,), 2.0, wl.generator(3, "mxbias"), torch.bfloat16)
    D = _mx_gemm(A, As, B, Bs, dev, bias=bias.to(dev), d_dtype=d_dtype)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    ref, absr = oracle.mx_gemm_elems(A, As, B, Bs, host(bias), ms.ravel(), ns.ravel())
    check_gemm(D, ref, absr, ms.ravel(), ns.ravel(), what="mx gemm bias")


def test_mx_linear_step_sampled():
    """MXFP8 linear fwd, dgrad and wgrad from the GPU's own quantisations of
    channel-scaled X, W and dY (the MX MLP distributions), sampled outputs."""
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    M, K, N = 2048, 1024, 1536
    seed = wl.SEEDS["mx_mlp"]
    x = wl.channel_scaled_normal(M, K, wl.generator(seed, "X-small"))
    w = wl.normal((N, K), 0.02, wl.generator(seed, "W-small"), torch.bfloat16)
    dy = wl.normal((M, N), 1.0, wl.generator(seed, "dY-small"), torch.bfloat16)
    xq, xs, xcq, xcs = _quantize(x, dev)
    wq, ws, wcq, wcs = _quantize(w, dev)
    dq, ds, dcq, dcs = _quantize(dy, dev)
    rng = np.random.default_rng(1)
    cases = [  # (A, A_s, B, B_s, M, N, K)
        ("fwd", xq, xs, wq, ws, M, N, K),
        ("dgrad", dq, ds, wcq, wcs, M, K, N),
        ("wgrad", dcq, dcs, xcq, xcs, N, K, M),
    ]
    for name, A, As, B, Bs, m, n, k in cases:
        D = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        fd.mxfp8_gemm(A, As, B, Bs, D)
        torch.cuda.synchronize()
        ms, ns = sample_elems(m, n, rng, n=2048)
        Ah, Bh = A.cpu().numpy(), B.cpu().numpy()
        ref, absr = oracle.mx_gemm_elems(Ah, tiled_to_plain(As.cpu().numpy(), m, k // 32), Bh,
                                         tiled_to_plain(Bs.cpu().numpy(), n, k // 32), None, ms, ns)
        check_gemm(D, ref, absr, ms, ns, what="mx " + name)


def test_mx_linear_weight_cache():
    """MxLinear over micro-batches: is_first_microbatch=True quantises the weight and keeps it,
    False reuses it with no weight quantisation (its launches are saved) and gives the same bits
    as quantising again; False with nothing cached raises before any launch."""
    import fp8_delayed_scaling_gb300 as fd
    from fp8_delayed_scaling_gb300.mxlinear import MxLinear
    dev = gpu()
    M, K, N = 512, 1024, 768
    seed = wl.SEEDS["mx_mlp"]
    w = wl.normal((N, K), 0.02, wl.generator(seed, "W-cache"), torch.bfloat16).to(dev)
    x1 = wl.channel_scaled_normal(M, K, wl.generator(seed, "X1-cache")).to(dev)
    x2 = wl.channel_scaled_normal(M, K, wl.generator(seed, "X2-cache")).to(dev)
    lin = MxLinear(w, None, M)
    with pytest.raises(RuntimeError):
        lin.forward(x1, is_first_microbatch=False)
    fresh = MxLinear(w, None, M)
    lin.forward(x1, is_first_microbatch=True)
    torch.cuda.synchronize()
    n0 = fd.fp8dl_kernel_launches()
    y2 = lin.forward(x2, is_first_microbatch=False).clone()
    n1 = fd.fp8dl_kernel_launches()
    y2_ref = fresh.forward(x2).clone()
    n2 = fd.fp8dl_kernel_launches()
    torch.cuda.synchronize()
    n3 = fd.fp8dl_kernel_launches()
    fresh.mx_w.quantize(w)  # what one quantisation of the weight launches
    n4 = fd.fp8dl_kernel_launches()
    torch.cuda.synchronize()
    assert torch.equal(y2, y2_ref)
    assert n4 - n3 >= 1 and (n2 - n1) - (n1 - n0) == n4 - n3
    dx, dw, _ = lin.backward(torch.ones((M, N), dtype=torch.bfloat16, device=dev))
    dx_ref, dw_ref, _ = fresh.backward(torch.ones((M, N), dtype=torch.bfloat16, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref)
