"""The quantise-once producer inside the GEMM (H3FP4_FUSED_QUANT): the GEMM
kernel's packer warps quantise the activation tile by tile while the same
kernel consumes the tiles behind ready flags.

It must leave exactly the bytes of the two-kernel path -- codes, block scales
(padding rows included), global scale -- and exactly its output, on ragged M
(a last m-tile of a few rows, an odd number of m-tiles), a K that ends in a
partial 256-column stage, two and three segments with the prologue, the gated
residual epilogue, with the computed and with a given global scale.  At full
size the fused output is checked against the oracle at one point per
epilogue warp of every pair tile.  A packer that publishes nothing makes the
GEMM's waits run out: the status word reports it and the context stays usable.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import (LinearCase, check_outputs, dev_bf16, host_u16, oracle_operands,  # noqa: E402
                          sample_points, tile_points)

# Workspace layout of the activation (h3fp4_api.cu / h3fp4_internal.h): codes
# at byte 16896, block scales after them at the next 256-byte boundary.
WS_ACT_GSCALE = 256 + 4 * 4096
WS_ACT_CODES = WS_ACT_GSCALE + 256


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def _act_region(ws, M, K):
    import audio_dit_gb300 as A
    codes = M * K // 2
    sf0 = WS_ACT_CODES + (codes + 255) // 256 * 256
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    return (raw[WS_ACT_CODES:WS_ACT_CODES + codes].copy(), raw[sf0:sf0 + A.h3fp4_sf_bytes(M, K)].copy(),
            raw[WS_ACT_GSCALE:WS_ACT_GSCALE + 4].copy())


def _custom(M, N, K, seed, nseg):
    rng = np.random.default_rng(seed)
    seg = np.linspace(0, M, nseg + 1).round().astype(np.int64)
    wl = W.Workload(f"custom_{M}x{N}x{K}", M, K, N, seed, True, True, nseg > 1, "custom shape")
    d = dict(workload=wl, M=M, N=N, K=K, seg_off=seg)
    d["x"] = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    d["w"] = W.to_bf16_bits(rng.standard_normal((N, K), dtype=np.float32) * 0.02)
    d["bias"] = W.to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * 0.01)
    d["shift"] = rng.standard_normal((nseg, K), dtype=np.float32) * 0.1
    d["scale"] = rng.standard_normal((nseg, K), dtype=np.float32) * 0.1
    d["gate"] = rng.uniform(0, 1, (nseg, N)).astype(np.float32)
    d["resid"] = W.to_bf16_bits(rng.standard_normal((M, N), dtype=np.float32))
    return d


CASES = [("qkv", 300), ("fc1", 520), ("fc2", 260), ("attn_out", 600), ("tiny", 256)]
CUSTOM = [(130, 1000, 320, 3), (257, 392, 1024, 2), (40, 2056, 128, 1), (1, 256, 64, 1)]


def _pair(d):
    """Two-kernel path, then the fused path, on one LinearCase (same workspace)."""
    import audio_dit_gb300 as A
    case = LinearCase(d)
    ref = case.run().clone()
    reg_ref = _act_region(case._gws.t, d["M"], d["K"])
    out = case.run(fused=True).clone()
    reg = _act_region(case._gws.t, d["M"], d["K"])
    A.h3fp4_check(case.ws)
    return case, ref, out, reg_ref, reg


def _assert_same(ref, out, reg_ref, reg, what):
    names = ("codes", "block scales", "global scale")
    for a, b, n in zip(reg_ref, reg, names):
        if not np.array_equal(a, b):
            bad = np.nonzero(a != b)[0]
            raise AssertionError(f"{what}: {bad.size} {n} bytes differ, first at {bad[:5]}")
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16)), f"{what}: outputs differ"


@pytest.mark.parametrize("name,M", CASES)
def test_fused_matches_two_kernel_path(name, M):
    d = W.make_inputs(name, M=M)
    _, ref, out, reg_ref, reg = _pair(d)
    _assert_same(ref, out, reg_ref, reg, f"{name} M={M}")


@pytest.mark.parametrize("M,N,K,nseg", CUSTOM)
def test_fused_ragged_shapes(M, N, K, nseg):
    d = _custom(M, N, K, seed=M + N + K, nseg=nseg)
    _, ref, out, reg_ref, reg = _pair(d)
    _assert_same(ref, out, reg_ref, reg, f"{M}x{N}x{K}")


@pytest.mark.parametrize("seg", [[0, 5, 11, 20, 37, 38, 200], [0, 3, 3, 4, 40, 41, 100, 163, 200]])
def test_fused_segments_shorter_than_a_tile(seg):
    """Segments of a few rows (up to the most the boundary accepts, one empty):
    the packer switches modulation constants inside a 32-row X tile (and
    within a thread's rows)."""
    d = _custom(200, 520, 256, seed=79, nseg=1)
    seg = np.array(seg, np.int64)
    rng = np.random.default_rng(80)
    d["seg_off"] = seg
    d["shift"] = rng.standard_normal((len(seg) - 1, 256), dtype=np.float32) * 0.1
    d["scale"] = rng.standard_normal((len(seg) - 1, 256), dtype=np.float32) * 0.1
    d["gate"] = rng.uniform(0, 1, (len(seg) - 1, 520)).astype(np.float32)
    _, ref, out, reg_ref, reg = _pair(d)
    _assert_same(ref, out, reg_ref, reg, "short segments")


@pytest.mark.parametrize("name,M", [("fc1", 520), ("attn_out", 600)])
def test_fused_given_scale(name, M):
    """With the caller's global scale the GEMM kernel is the only launch."""
    import audio_dit_gb300 as A
    d = W.make_inputs(name, M=M)
    case = LinearCase(d)
    gs = torch.tensor([0.0371], dtype=torch.float32, device="cuda")
    ref = case.run(a_gscale=gs, gscale_given=True).clone()
    reg_ref = _act_region(case._gws.t, M, d["K"])
    out = case.run(a_gscale=gs, gscale_given=True, fused=True).clone()
    reg = _act_region(case._gws.t, M, d["K"])
    A.h3fp4_check(case.ws)
    _assert_same(ref, out, reg_ref, reg, f"{name} given")


def test_fused_new_inputs_are_not_served_stale_tiles():
    """A second fused call with different X on the same workspace reads the
    new tiles (the flags of the first call do not count for the second)."""
    d1 = W.make_inputs("fc2", M=260)
    case = LinearCase(d1)
    case.run(fused=True)
    x2 = W.to_bf16_bits(np.random.default_rng(99).standard_normal((260, d1["K"]), dtype=np.float32))
    case.x = dev_bf16(x2)
    ref = case.run().clone()
    out = case.run(fused=True).clone()
    assert torch.equal(ref.view(torch.int16), out.view(torch.int16))
    out2 = case.run(fused=True).clone()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("name", ["qkv", "fc1", "fc2", "attn_out"])
def test_fused_full_size(orc, name):
    """Full size, fused: bit-identical to the two-kernel output everywhere, and
    within the oracle's bound at one point per epilogue warp of every pair
    tile plus random points and the segment edges."""
    d = W.make_inputs(name)
    case = LinearCase(d)
    ref = host_u16(case.run().clone())
    out = host_u16(case.run(fused=True))
    assert np.array_equal(ref, out), f"{name}: {int((ref != out).sum())} outputs differ from the two-kernel path"
    a, w = oracle_operands(orc, d)
    pts = np.concatenate([tile_points(d["M"], d["N"], seed=7 + sum(name.encode())),
                          sample_points(d["M"], d["N"], 300, seed=sum(name.encode()), seg_off=d["seg_off"])])
    refo, bound = orc.linear_points(a, w, d["M"], d["N"], d["K"], pts, bias=d["bias"], gate=d["gate"],
                                    resid=d["resid"], seg_off=d["seg_off"])
    check_outputs(out[pts[:, 0], pts[:, 1]], refo, bound, f"{name} fused full size")


def test_fused_rejects_unsupported():
    import audio_dit_gb300 as A
    d = W.make_inputs("tiny", M=64)
    case = LinearCase(d)
    with pytest.raises(A.H3FP4Error):
        A.h3fp4_linear(case.x, *case.wq, torch.empty((64, d["N"] // 2), dtype=torch.bfloat16, device="cuda"),
                       case.ws, swiglu=True, fused=True)


def test_pack_flag_timeout_is_reported_and_context_survives():
    import audio_dit_gb300 as A
    ws = A.alloc_workspace(128, 256, 256, 0)
    x = dev_bf16(W.to_bf16_bits(np.random.default_rng(3).standard_normal((128, 256), dtype=np.float32)))
    gs = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    A.h3fp4_selftest_pack_timeout(x, gs, ws, 2_000_000)  # 2 ms limit, no tile is ever published
    with pytest.raises(A.H3FP4Error) as e:
        A.h3fp4_check(ws)
    assert e.value.status == 5
    A.h3fp4_check(ws)  # cleared
    # the context is intact: a fused linear still matches the two-kernel path
    d = W.make_inputs("tiny", M=256)
    _, ref, out, reg_ref, reg = _pair(d)
    _assert_same(ref, out, reg_ref, reg, "after the pack timeout")


def test_fused_refuses_stream_capture():
    """The flags carry a call number fixed at launch, so a fused call may not be
    captured into a graph: it is refused on the host, and the capture ends
    cleanly (nothing was launched into it)."""
    import audio_dit_gb300 as A
    d = W.make_inputs("tiny", M=256)
    case = LinearCase(d)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            with pytest.raises(A.H3FP4Error) as e:
                A.h3fp4_linear(case.x, *case.wq, case.out, case.ws, bias=case.bias, fused=True)
            assert e.value.status == 1
        finally:
            g.capture_end()
    torch.cuda.synchronize()
    _, ref, out, reg_ref, reg = _pair(d)   # the context is intact
    _assert_same(ref, out, reg_ref, reg, "after the refused capture")
