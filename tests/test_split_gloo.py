"""The multi-rank M-split of one activation, on CPU with gloo (world size 2):
each rank owns a slice of the token rows, computes the amax of its modulated
rows, the ranks all-reduce(MAX) that one float -- the only exchange the path
needs -- and each rank quantises its rows with the resulting global scale.
The gathered codes and block scales must equal the single-rank quantisation
of the whole tensor bit for bit.  (Oracle arithmetic on each rank.)"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _rank_main(rank, world, port, bounds, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import workloads as W
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = W.make_inputs("attn_out", M=bounds[-1])
        lo, hi = bounds[rank], bounds[rank + 1]
        seg = list(np.clip(d["seg_off"], lo, hi) - lo)
        m = oracle.modulate(d["x"][lo:hi], d["shift"], d["scale"], seg)
        amax = torch.tensor([oracle.amax(m)], dtype=torch.float32)
        dist.all_reduce(amax, op=dist.ReduceOp.MAX)
        gs = oracle.global_scale(float(amax.item()))
        codes, sf, g = oracle.quantize(d["x"][lo:hi], d["shift"], d["scale"], seg, gscale=gs)
        out = [None] * world
        dist.all_gather_object(out, (codes, sf, g))
        if rank == 0:
            q.put(out)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 256, 520], [0, 301, 520]])
def test_two_rank_m_split_is_bit_identical(orc, bounds):
    import workloads as W
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 2000) + bounds[1] % 7
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, bounds, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = q.get(timeout=300)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    d = W.make_inputs("attn_out", M=bounds[-1])
    rc, rsf, rg = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    K = d["K"]
    for r, (codes, sf, g) in enumerate(out):
        lo, hi = bounds[r], bounds[r + 1]
        assert g == rg
        assert np.array_equal(codes, rc[lo:hi])
        for row in range(hi - lo):
            idx = [orc.sf_offset(row, c, K) for c in range(K // 16)]
            ref = [orc.sf_offset(lo + row, c, K) for c in range(K // 16)]
            assert np.array_equal(sf[idx], rsf[ref])
