"""Shared test helpers: device setup, host copies, and the GEMM error bound."""
import numpy as np
import pytest
import torch

# GEMM tolerance per output element (fp32 accumulation on the tensor cores,
# then one rounding to the output type): |D - ref| <= 2^-7 |ref| + 2^-20 sum|a_i b_i|.
REL = 2.0 ** -7
ABS = 2.0 ** -20


def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fp8_delayed_scaling_gb300 as fd
    if not fd.fp8dl_device_supported(torch.cuda.current_device()):
        pytest.skip("not an sm_103 GPU")
    return torch.device("cuda", torch.cuda.current_device())


def host(t: torch.Tensor) -> np.ndarray:
    """CPU numpy copy; bf16 becomes its uint16 bit patterns (the oracle's bf16 input)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def check_gemm(D: torch.Tensor, ref: np.ndarray, absr: np.ndarray, ms=None, ns=None, what="gemm"):
    """D (device, [M,N]) against oracle values at (ms, ns) (all elements if None)."""
    d = as_f64(D)
    got = d.ravel() if ms is None else d[ms, ns]
    err = np.abs(got - ref)
    bound = REL * np.abs(ref) + ABS * absr
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, "%s: %d/%d elements out of bound, first %s: got %r ref %r bound %r" % (
        what, bad.size, err.size, bad[:3], got[bad[:3]], ref[bad[:3]], bound[bad[:3]])
    return float(np.max(err / np.maximum(bound, 1e-300)))


def sample_elems(M, N, rng, n=4096, tile_m=128, tile_n=256):
    """Seeded output sample: full first/last row and column, tile edges, random rest."""
    ms, ns = [], []
    for m in (0, M - 1):
        ms += [m] * N
        ns += list(range(N))
    for n in (0, N - 1):
        ms += list(range(M))
        ns += [n] * M
    edges_m = sorted({v for k in range(0, M, tile_m) for v in (k, min(k + tile_m - 1, M - 1))})
    edges_n = sorted({v for k in range(0, N, tile_n) for v in (k, min(k + tile_n - 1, N - 1))})
    for m in edges_m[:64]:
        for n in edges_n[:64]:
            ms.append(m)
            ns.append(n)
    ms += list(rng.integers(0, M, n))
    ns += list(rng.integers(0, N, n))
    ms, ns = np.array(ms, np.int64), np.array(ns, np.int64)
    if ms.size > 4 * n + 4 * (M + N):
        keep = rng.choice(ms.size, 4 * n, replace=False)
        ms, ns = ms[keep], ns[keep]
    return ms, ns
