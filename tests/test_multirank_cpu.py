"""Data parallelism across ranks, host side (CPU, gloo, world size 2).

Each replica runs the path on its own token slice; the one exchange delayed
scaling needs is a MAX all-reduce of the per-slot amaxes before the update
("FP8 低精度训练：Transformer Engine 简析" §三.3: at autocast exit the amaxes
of the processes in fp8_group are reduced).  Two gloo ranks each take the
oracle amax of their half of the tokens; after all_reduce(MAX) both hold the
single-process amax of the whole batch, so their scale updates agree with it
bit for bit.  The benchmark's max-over-ranks timing uses the same reduce."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import workloads as wl


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _tensors():
    x = wl.student_t3((512, 256), 0.5, wl.generator(6, "dp-x"))
    w = wl.normal((384, 256), 0.02, wl.generator(6, "dp-w"), torch.bfloat16)
    dy = wl.with_outliers(wl.normal((512, 384), 1e-3, wl.generator(6, "dp-dy"), torch.bfloat16), 0.001, 1000.0,
                          wl.generator(6, "dp-dy-out"))
    return x, w, dy


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x, w, dy = _tensors()
    rows = x.shape[0] // world
    xs = wl.bf16_bits(x[rank * rows:(rank + 1) * rows])
    dys = wl.bf16_bits(dy[rank * rows:(rank + 1) * rows])
    local = torch.tensor([float(oracle.amax(xs)), float(oracle.amax(wl.bf16_bits(w))), float(oracle.amax(dys))],
                         dtype=torch.float32)
    dist.all_reduce(local, op=dist.ReduceOp.MAX)
    st = oracle.ScalingState([0, 0, 1], hist_len=16)
    for i in range(3):
        st.record_amax(i, local[i].item())
    st.update(0)
    t = torch.tensor([1.5 + rank], dtype=torch.float64)  # per-rank step time: the job time is the max
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    q.put((rank, st.scale.copy(), st.scale_inv.copy(), t.item()))
    dist.destroy_process_group()


def test_amax_max_allreduce_matches_single_process():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x, w, dy = _tensors()
    ref = oracle.ScalingState([0, 0, 1], hist_len=16)
    for i, t in enumerate((x, w, dy)):
        ref.record_amax(i, oracle.amax(wl.bf16_bits(t)))
    ref.update(0)
    for rank, scale, scale_inv, tmax in res:
        assert np.array_equal(scale, ref.scale) and np.array_equal(scale_inv, ref.scale_inv)
        assert tmax == 2.5


class _HostState:
    """A scaling-state block in host memory with the library's slot layout; update() is
    recorded instead of launched (the reduce under test runs before it)."""

    def __init__(self, n_slots, hist_len=16):
        import fp8_delayed_scaling_gb300 as fd
        self.n_slots = n_slots
        self.stride = fd.fp8dl_slot_stride(hist_len)
        self.buf = torch.zeros(n_slots * self.stride, dtype=torch.uint8)
        self.updates = []

    def update(self, step, stream=None):
        self.updates.append((step, self.amaxes().tolist()))

    def amaxes(self):
        from fp8_delayed_scaling_gb300.autocast import amax_view
        return amax_view(self.buf, self.n_slots, self.stride).clone()


def _autocast_worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from fp8_delayed_scaling_gb300.autocast import amax_view, fp8_autocast
    st = _HostState(3)
    rows = st.buf.view(3, st.stride)
    rows[:, 12:].fill_(7)  # bytes other than the amaxes must survive the reduce
    for step in range(2):
        with fp8_autocast(st, group=dist.group.WORLD):
            amax_view(st.buf, 3, st.stride).copy_(torch.tensor([1.0 + rank, 5.0 - rank, 0.25 * (step + 1)]))
    untouched = bool((rows[:, 12:] == 7).all())
    q.put((rank, st.updates, untouched))
    dist.destroy_process_group()


def test_autocast_exit_reduces_amax_over_the_group_then_updates():
    """fp8_autocast(group=...) exit: MAX all-reduce of the amax fields in place, then one update."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_autocast_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, updates, untouched in res:
        assert untouched
        assert updates == [(0, [2.0, 5.0, 0.25]), (1, [2.0, 5.0, 0.5])]
