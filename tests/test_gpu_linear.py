"""GPU parity of the fused NVFP4 linear against the oracle.

Every output must satisfy |out - ref| <= 2^-8 |ref| + 1e-5 |g| sum_k |a_k w_k|
(g = 1 without gate), ref being the float64 oracle on the oracle's own
quantisation of the same seeded inputs; the activation/weight codes and block
scales the GPU uses are the ones the quantiser tests prove bit-exact.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import (Guarded, LinearCase, assert_quant_equal, check_outputs, host_u16,  # noqa: E402
                          oracle_operands, sample_points, tile_points)


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def _full_compare(orc, d, case=None, **kw):
    case = case or LinearCase(d)
    out = host_u16(case.run(**kw))
    a, w = oracle_operands(orc, d)
    assert_quant_equal(case.weight_quant_host(), w, "weight")
    ref, bound = orc.linear_full(a, w, d["M"], d["N"], d["K"], bias=d["bias"], gate=d["gate"],
                                 resid=d["resid"], seg_off=d["seg_off"])
    return check_outputs(out, ref, bound, f"{d['workload'].name} M={d['M']}")


def test_tiny_full(orc):
    _full_compare(orc, W.make_inputs("tiny"))


@pytest.mark.parametrize("name,M", [("qkv", 300), ("fc1", 129), ("fc2", 200), ("attn_out", 300)])
def test_reduced_rows_all_outputs(orc, name, M):
    _full_compare(orc, W.make_inputs(name, M=M))


@pytest.mark.parametrize("name", ["qkv", "fc1", "fc2", "attn_out"])
def test_full_size_every_tile(orc, name):
    """Full size, as the bench runs it: every epilogue warp of every 256 x 256
    pair tile (both CTAs, all four lane quarters, both column halves; every
    round of the persistent loop and the partial last wave) contributes one
    point, plus random points and the segment edges."""
    d = W.make_inputs(name)
    case = LinearCase(d)
    out = host_u16(case.run())
    a, w = oracle_operands(orc, d)
    pts = np.concatenate([tile_points(d["M"], d["N"], seed=sum(name.encode())),
                          sample_points(d["M"], d["N"], 500, seed=sum(name.encode()), seg_off=d["seg_off"])])
    ref, bound = orc.linear_points(a, w, d["M"], d["N"], d["K"], pts, bias=d["bias"], gate=d["gate"],
                                   resid=d["resid"], seg_off=d["seg_off"])
    check_outputs(out[pts[:, 0], pts[:, 1]], ref, bound, f"{name} full size")


def _custom(M, N, K, seed, gated=True, mod=True, nseg=1):
    rng = np.random.default_rng(seed)
    seg = np.linspace(0, M, nseg + 1).round().astype(np.int64)
    wl = W.Workload(f"custom_{M}x{N}x{K}", M, K, N, seed, mod, gated, nseg > 1, "custom shape")
    d = dict(workload=wl, M=M, N=N, K=K, seg_off=seg)
    d["x"] = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    d["w"] = W.to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * 0.02)
    d["bias"] = W.to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * 0.01)
    d["shift"] = (rng.standard_normal((nseg, K), dtype=np.float32) * 0.1) if mod else None
    d["scale"] = (rng.standard_normal((nseg, K), dtype=np.float32) * 0.1) if mod else None
    d["gate"] = rng.uniform(0, 1, (nseg, N)).astype(np.float32) if gated else None
    d["resid"] = W.to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32)) if gated else None
    return d


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (130, 1000, 320), (64, 1096, 576), (300, 8, 256),
                                   (257, 392, 1024), (40, 2056, 128)])
def test_ragged_shapes(orc, M, N, K):
    """M, N and K tails: N not a multiple of the 256-wide tile (and an odd
    number of 128-row scale tiles), K not a multiple of the 256-deep stage."""
    _full_compare(orc, _custom(M, N, K, seed=M + N + K, nseg=3 if M > 3 else 1))


SHORT_SEGMENTS = [[0, 5, 11, 20, 37, 38, 200],
                  [0, 3, 3, 4, 40, 41, 100, 163, 200]]  # the most segments, one empty, one a single row


@pytest.mark.parametrize("seg", SHORT_SEGMENTS)
def test_segments_shorter_than_a_warp_block(orc, seg):
    """Segments of a few rows, so that one epilogue warp's 32 rows span three
    or more segments: with the gated epilogue over a short K loop the kernel
    stages the gate of the block's first and last segments in shared memory
    and reads the others from global memory."""
    d = _custom(200, 520, 256, seed=77, nseg=1)
    seg = np.array(seg, np.int64)
    nseg = len(seg) - 1
    rng = np.random.default_rng(78)
    d["seg_off"] = seg
    d["workload"] = W.Workload("custom_short_segments", 200, 256, 520, 77, True, True, True, "short segments")
    d["shift"] = rng.standard_normal((nseg, 256), dtype=np.float32) * 0.1
    d["scale"] = rng.standard_normal((nseg, 256), dtype=np.float32) * 0.1
    d["gate"] = rng.uniform(0, 1, (nseg, 520)).astype(np.float32)
    _full_compare(orc, d)


def test_no_bias_no_prologue(orc):
    d = _custom(200, 512, 512, seed=5, gated=False, mod=False)
    case = LinearCase(d, use_bias=False)
    out = host_u16(case.run())
    a, w = oracle_operands(orc, d)
    ref, bound = orc.linear_full(a, w, 200, 512, 512)
    check_outputs(out, ref, bound, "no bias")


def test_prequant_and_given_scale_match_fused(orc):
    """A_PREQUANT (codes from h3fp4_quantize_act) and GSCALE_GIVEN reproduce the
    fused call bit for bit (same codes, same GEMM)."""
    import audio_dit_gb300 as A
    d = W.make_inputs("attn_out", M=384)
    case = LinearCase(d)
    fused = case.run().clone()
    codes, sf, gs = A.alloc_nvfp4(d["M"], d["K"])
    A.h3fp4_quantize_act(case.x, codes, sf, gs, case.ws, shift=case.shift, scale=case.scale,
                         seg_off=case.seg_off)
    out2 = torch.empty_like(fused)
    A.h3fp4_linear(codes, *case.wq, out2, case.ws, a_sf=sf, a_gscale=gs, gate=case.gate, resid=case.resid,
                   bias=case.bias, seg_off=case.seg_off)
    out3 = torch.empty_like(fused)
    A.h3fp4_linear(case.x, *case.wq, out3, case.ws, a_gscale=gs, gscale_given=True, shift=case.shift,
                   scale=case.scale, gate=case.gate, resid=case.resid, bias=case.bias, seg_off=case.seg_off)
    A.h3fp4_check(case.ws)
    assert torch.equal(fused.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(fused.view(torch.int16), out3.view(torch.int16))


@pytest.mark.parametrize("M", [1024, 4096, 65536, 946, 37810])
def test_m_sweep_sampled(orc, M):
    d = W.m_sweep_inputs(M)
    case = LinearCase(d)
    out = host_u16(case.run())
    a, w = oracle_operands(orc, d)
    pts = np.concatenate([tile_points(M, d["N"], seed=M), sample_points(M, d["N"], 300, seed=M)])
    ref, bound = orc.linear_points(a, w, M, d["N"], d["K"], pts, bias=d["bias"], gate=d["gate"],
                                   resid=d["resid"], seg_off=d["seg_off"])
    check_outputs(out[pts[:, 0], pts[:, 1]], ref, bound, f"sweep M={M}")


def test_repeat_is_deterministic():
    d = W.make_inputs("fc2", M=512)
    case = LinearCase(d)
    o1 = case.run().clone()
    o2 = case.run().clone()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_guard_regions_detect_a_stray_write():
    """The canary check used by every linear/quantise test fires on a write
    just past a buffer (made here by torch, not by the library)."""
    g = Guarded((3, 100), torch.bfloat16)
    g.check("clean")
    g.raw[g.raw.numel() - 1] = 0
    with pytest.raises(AssertionError):
        g.check("planted")
