"""Sizes past 2^31 elements: the casts, the MX quantisation and both GEMMs index with
64-bit offsets.  Inputs are a seeded host tile repeated on the device, so every sampled
output row or column has an oracle value from the tile; samples include the rows beyond
2^31 / cols and the last row and column."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from helpers import ABS, REL, gpu, host, sample_elems

pytestmark = pytest.mark.gpu

TILE, REPS, C = 4096, 16, 40960  # 65536 x 40960 = 2.68e9 elements
R = TILE * REPS


def _sf_offsets(rows, NB):
    """Byte offsets of S[r][b] (b = 0..NB-1) in the tiled scale layout, for the given rows only."""
    kg = (NB + 3) // 4
    r = np.asarray(rows, dtype=np.int64)[:, None]
    b = np.arange(NB, dtype=np.int64)[None, :]
    return ((r >> 7) * kg + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3)


def _rows(rng):
    edge = (1 << 31) // C  # the first row whose elements lie past 2^31
    return np.unique(np.concatenate([[0, 1, edge - 1, edge, edge + 1, R - 1], rng.integers(0, R, 6)]))


def _tile(seed):
    return wl.normal((TILE, C), 1.0, wl.generator(seed, "large"), torch.bfloat16)


def test_cast_amax_transpose_dbias_past_2_31_elements():
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    tile = _tile(93)
    th = host(tile)
    x = tile.to(dev).repeat(REPS, 1)
    amax0 = oracle.amax(th)
    scale = np.float32(448.0) / np.float32(amax0)
    q = torch.empty((R, C), dtype=torch.uint8, device=dev)
    qt = torch.empty((C, R), dtype=torch.uint8, device=dev)
    am = torch.zeros(1, device=dev)
    db = torch.empty(C, device=dev)
    ws = torch.empty(fd.fp8_cast_workspace_size(R, C), dtype=torch.uint8, device=dev)
    fd.fp8_cast_amax_transpose(x, fd.E4M3, torch.tensor([scale], device=dev), out=q, out_t=qt, amax=am, dbias=db,
                               workspace=ws)
    torch.cuda.synchronize()
    assert am.item() == amax0
    rng = np.random.default_rng(3)
    rows = _rows(rng)
    qo = oracle.quantize(0, th[rows % TILE], scale)
    assert np.array_equal(q[torch.from_numpy(rows).to(dev)].cpu().numpy(), qo)
    cols = np.unique(np.concatenate([[0, C - 1], rng.integers(0, C, 6)]))
    qto = oracle.quantize(0, np.ascontiguousarray(th[:, cols].T), scale)  # [cols x TILE]
    got = qt[torch.from_numpy(cols).to(dev)].cpu().numpy()
    assert np.array_equal(got, np.tile(qto, (1, REPS)))
    s, sabs = oracle.colsum(th)
    assert np.all(np.abs(db.cpu().numpy().astype(np.float64) - REPS * s) <= R * 2.0 ** -24 * REPS * sabs + 1e-30)
    del x, q, qt, ws
    torch.cuda.empty_cache()


def test_mx_quantize_past_2_31_elements():
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    tile = _tile(94)
    th = host(tile)
    x = tile.to(dev).repeat(REPS, 1)
    rq = torch.empty((R, C), dtype=torch.uint8, device=dev)
    cq = torch.empty((C, R), dtype=torch.uint8, device=dev)
    rs = torch.empty(fd._lib.mxfp8_scale_bytes(R, C), dtype=torch.uint8, device=dev)
    cs = torch.empty(fd._lib.mxfp8_scale_bytes(C, R), dtype=torch.uint8, device=dev)
    fd.mxfp8_quantize(x, rq, rs, cq, cs)
    torch.cuda.synchronize()
    rng = np.random.default_rng(4)
    rows = _rows(rng)
    qo, so = oracle.mx_quantize_rows(th[rows % TILE])
    assert np.array_equal(rq[torch.from_numpy(rows).to(dev)].cpu().numpy(), qo)
    rs_h = rs.cpu().numpy()
    assert np.array_equal(rs_h[_sf_offsets(rows, C // 32)], so)
    cols = np.unique(np.concatenate([[0, C - 1], rng.integers(0, C, 4)]))
    qc, sc = oracle.mx_quantize_rows(np.ascontiguousarray(th[:, cols].T))  # [cols x TILE], [cols x TILE/32]
    assert np.array_equal(cq[torch.from_numpy(cols).to(dev)].cpu().numpy(), np.tile(qc, (1, REPS)))
    cs_h = cs.cpu().numpy()
    assert np.array_equal(cs_h[_sf_offsets(cols, R // 32)], np.tile(sc, (1, REPS)))
    del x, rq, cq
    torch.cuda.empty_cache()


def _codes(rng, shape):
    tab = oracle.decode_table(0)
    ok = np.array([c for c in range(256) if np.isfinite(tab[c])], np.uint8)
    return ok[rng.integers(0, ok.size, shape)]


@pytest.mark.parametrize("mx", [False, True])
def test_gemm_past_2_31_outputs(mx):
    import fp8_delayed_scaling_gb300 as fd
    dev = gpu()
    M, N, K = R, C, 64
    rng = np.random.default_rng(5 + int(mx))
    A, B = _codes(rng, (M, K)), _codes(rng, (N, K))
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if mx:
        As = rng.integers(118, 136, (M, K // 32)).astype(np.uint8)
        Bs = rng.integers(118, 136, (N, K // 32)).astype(np.uint8)
        Ast = np.full(fd._lib.mxfp8_scale_bytes(M, K), 127, np.uint8)
        Ast[_sf_offsets(np.arange(M), K // 32)] = As
        Bst = np.full(fd._lib.mxfp8_scale_bytes(N, K), 127, np.uint8)
        Bst[_sf_offsets(np.arange(N), K // 32)] = Bs
        fd.mxfp8_gemm(torch.from_numpy(A).to(dev), torch.from_numpy(Ast).to(dev), torch.from_numpy(B).to(dev),
                      torch.from_numpy(Bst).to(dev), D)
    else:
        one = torch.tensor([0.125], device=dev)
        fd.fp8_gemm(torch.from_numpy(A).to(dev), fd.E4M3, torch.from_numpy(B).to(dev), fd.E4M3, one, one, D)
    torch.cuda.synchronize()
    ms, ns = sample_elems(M, N, rng, n=4096)
    edge = (1 << 31) // N
    ms = np.concatenate([ms, np.full(N, edge), np.full(N, R - 1)])
    ns = np.concatenate([ns, np.arange(N), np.arange(N)])
    if mx:
        ref, absr = oracle.mx_gemm_elems(A, As, B, Bs, None, ms, ns)
    else:
        ref, absr = oracle.gemm_elems(A, 0, B, 0, 0.125, 0.125, None, ms, ns)
    got = D[torch.from_numpy(ms).to(dev), torch.from_numpy(ns).to(dev)].float().cpu().numpy().astype(np.float64)
    bad = np.nonzero(~(np.abs(got - ref) <= REL * np.abs(ref) + ABS * absr))[0]
    assert bad.size == 0, ("large gemm", bad[:3], got[bad[:3]], ref[bad[:3]])
    del D
    torch.cuda.empty_cache()
