"""The bench's work accounting, against figures worked out by hand for each workload:
GEMM FLOPs per step (2·M·N·K for each of the forward, dgrad and wgrad products) and
the algorithmic HBM bytes of the LayerNormMLP step's HBM-bound kernels."""
import bench


def _flops(name):
    return bench.step_flops(bench.WORKLOADS[name])


def test_step_flops_match_hand_counts():
    # te.Linear 2048 tokens, 768 -> 3072: 9.66 GFLOP per product, three products
    assert _flops("linear_hybrid") == 3 * 2 * 2048 * 768 * 3072 == 28_991_029_248
    assert _flops("linear_fwd") == 2 * 2048 * 768 * 3072
    # Llama-7B projections, 8192 tokens: QKV 4096x12288, out 4096x4096, up 4096x11008,
    # down 11008x4096 -> 2.577 TFLOP forward, 7.73 TFLOP with dgrad and wgrad
    fwd = 2 * 8192 * (4096 * 12288 + 4096 * 4096 + 4096 * 11008 + 11008 * 4096)
    assert abs(fwd - 2.577e12) < 1e9
    assert _flops("llama_proj") == 3 * fwd
    # LayerNormMLP 16384 tokens, 4096 -> 16384 -> 4096: 13.19 TFLOP per step
    assert _flops("ln_mlp") == 3 * 2 * 16384 * 2 * (4096 * 16384) == 13_194_139_533_312
    # MXFP8 MLP 16384 tokens, 8192 -> 28672 -> 8192: 46.18 TFLOP per step
    assert abs(_flops("mx_mlp") - 46.18e12) < 0.01e12


def test_ln_mlp_hbm_bytes_match_hand_counts():
    M, H, F = 16384, 4096, 16384
    b = bench.hbm_bytes(bench.WORKLOADS["ln_mlp"], fused=True)
    # W1 [F x H] and W2 [H x F]: read 2 B, write codes and transposed codes (1 + 1 B);
    # dY [M x H]: the same plus 4 B per column of bias gradient
    assert b["cast"] == 2 * F * H * 4 + M * H * 4 + 4 * H == 805_322_752
    # LayerNorm forward + cast: 2 B read, 1 + 1 B written; backward: dy and x read, dx written
    assert b["norm_act"] == M * H * 4 + M * H * 6 == 671_088_640
    # unfused, the GELU cast (2 B read, 2 B written) and the dGELU cast (dg and h read,
    # codes written, bias gradient) are HBM passes of their own
    u = bench.hbm_bytes(bench.WORKLOADS["ln_mlp_separate"], fused=False)
    assert u["norm_act"] - b["norm_act"] == M * F * 4 + M * F * 6 + 4 * F


def test_gemm_traffic_is_keyed_to_the_kernel_code(tmp_path, monkeypatch):
    """The DRAM traffic the bench line prints for a workload's GEMMs comes from an ncu capture
    of specific kernel code: the key ignores comments, follows any code change (the line then
    prints null), and matches the sources as committed (a GEMM change needs a new capture)."""
    src = "int f(int x) {  // doubles\n    return 2 * x; /* a comment */\n}\n"
    same = "int f(int x) {  // twice x\n\n    return 2 * x; /* another */\n}\n"
    other = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench.source_code(src) == bench.source_code(same)
    assert bench.source_code(src) != bench.source_code(other)
    for name in ("ln_mlp", "mx_mlp"):
        traffic, note = bench.gemm_traffic(name)
        assert traffic is not None, "%s: %s (capture the GEMM traffic again)" % (name, note)
        assert note.startswith("ncu capture: ")
    (tmp_path / "k.cu").write_text(src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = dict(bench.GEMM_TRAFFIC["ln_mlp"], sources=("k.cu",), src_sha256=bench.source_sha(("k.cu",)))
    monkeypatch.setitem(bench.GEMM_TRAFFIC, "ln_mlp", entry)
    assert bench.gemm_traffic("ln_mlp")[0] == entry["bytes"]
    (tmp_path / "k.cu").write_text(same)
    assert bench.gemm_traffic("ln_mlp")[0] == entry["bytes"]
    (tmp_path / "k.cu").write_text(other)
    assert bench.gemm_traffic("ln_mlp") == (None, "the GEMM kernels changed since the capture")
