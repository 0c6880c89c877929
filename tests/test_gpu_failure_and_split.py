"""Failure detection (bounded device waits report a timeout instead of
hanging) and the multi-device M-split of one activation (per-shard amax ->
max -> global scale -> per-shard quantisation), emulated shard by shard on one
GPU: kernels of different shards never wait on one another."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import assert_quant_equal, dev_bf16, dev_f32, gpu_quantize  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def test_timeout_is_reported_and_context_survives(orc):
    import audio_dit_gb300 as A
    ws = A.alloc_workspace(128, 256, 256, 0)
    A.h3fp4_selftest_timeout(ws, 2_000_000)  # 2 ms limit, nothing ever arrives
    with pytest.raises(A.H3FP4Error) as e:
        A.h3fp4_check(ws)
    assert e.value.status == 5
    A.h3fp4_check(ws)  # the status word was cleared
    # the context is intact: a normal quantisation still matches the oracle
    d = W.make_inputs("tiny", M=64)
    assert_quant_equal(gpu_quantize(d["x"]), orc.quantize(d["x"]), "after timeout")


def _shard_quantize(d, bounds):
    import audio_dit_gb300 as A
    K = d["K"]
    ws = A.alloc_workspace(d["M"], 0, K, A.A_PREQUANT)
    shards = []
    amaxes = []
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        x = dev_bf16(d["x"][lo:hi])
        seg = np.clip(d["seg_off"], lo, hi) - lo
        am = torch.empty(1, dtype=torch.float32, device="cuda")
        A.h3fp4_act_amax(x, am, ws, shift=dev_f32(d["shift"]), scale=dev_f32(d["scale"]), seg_off=list(seg))
        shards.append((x, list(seg)))
        amaxes.append(am)
    amax = torch.stack(amaxes).max().reshape(1)          # the exchange step: all-reduce(MAX)
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    A.h3fp4_gscale_from_amax(amax, gs)
    out = []
    for x, seg in shards:
        codes, sf, g = A.alloc_nvfp4(x.shape[0], K)
        g.copy_(gs)
        A.h3fp4_quantize_act(x, codes, sf, g, ws, shift=dev_f32(d["shift"]), scale=dev_f32(d["scale"]),
                             seg_off=seg, gscale_given=True)
        out.append((codes.cpu().numpy(), sf.cpu().numpy(), float(g.item())))
    A.h3fp4_check(ws)
    return out


@pytest.mark.parametrize("bounds", [[0, 256, 512, 700], [0, 300, 301, 700]])
def test_m_split_matches_single_device(orc, bounds):
    d = W.make_inputs("attn_out", M=700)
    ref_codes, ref_sf, ref_gs = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    parts = _shard_quantize(d, bounds)
    K = d["K"]
    for (lo, hi), (codes, sf, gs) in zip(zip(bounds[:-1], bounds[1:]), parts):
        assert gs == ref_gs
        assert np.array_equal(codes, ref_codes[lo:hi])
        for r in range(hi - lo):
            for c in range(0, K // 16, 37):
                assert sf[orc.sf_offset(r, c, K)] == ref_sf[orc.sf_offset(lo + r, c, K)]
