"""GPU parity of the SwiGLU producer epilogue and the output amax.

SwiGLU: the epilogue's h = bf16(silu(g) * u) must equal the oracle's SwiGLU of
the plain epilogue's own bf16 output (same inputs, same GPU), element by element:
every element within one bf16 ulp and at least 99.9 % bit-identical (the GPU
evaluates silu in fp32 from the hardware's approximate 2^x and 1/x, within
3.4e-6 relative of the exact value for |g| < 88, the oracle in float64; they can
round a value lying that close to a bf16 midpoint differently).  The plain output
itself is held to the float64 oracle by test_gpu_linear.

Output amax: the stored value must be exactly max |out| of the bf16 output, and
quantising `out` with the global scale derived from it must give the same codes,
block scales and global scale as the two-pass quantisation of `out`.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import (Guarded, LinearCase, assert_quant_equal, gpu_quantize, host_u16,  # noqa: E402
                          oracle_operands)


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def _ulp_diff(a_u16, b_u16):
    """Distance in bf16 steps between two arrays of finite bf16 bit patterns."""
    def key(x):
        x = x.astype(np.int64)
        return np.where(x & 0x8000, -(x & 0x7FFF), x & 0x7FFF)
    return np.abs(key(a_u16) - key(b_u16))


def _run_pair(d, rows=None):
    """Plain linear [M, N] and SwiGLU linear [M, N/2] (both with out_amax) on one case."""
    import audio_dit_gb300 as A
    case = LinearCase(d)
    y = case.run(out_amax=True).clone()
    amax_plain = A.h3fp4_ws_out_amax(case.ws).clone()
    gh = Guarded((d["M"], d["N"] // 2), torch.bfloat16)
    h = gh.t
    A.h3fp4_linear(case.x, *case.wq, h, case.ws, shift=case.shift, scale=case.scale, bias=case.bias,
                   swiglu=True, out_amax=True)
    A.h3fp4_check(case.ws)
    case.check_guards([gh])
    amax_h = A.h3fp4_ws_out_amax(case.ws).clone()
    torch.cuda.synchronize()
    return case, y, h, amax_plain, amax_h


def _check_swiglu(orc, y, h, rows=None):
    yh = host_u16(y if rows is None else y[rows])
    hh = host_u16(h if rows is None else h[rows])
    ref = orc.swiglu_rows(yh)
    d = _ulp_diff(hh, ref)
    assert d.max() <= 1, f"{int((d > 1).sum())} SwiGLU outputs more than one bf16 step off"
    exact = float((d == 0).mean())
    print(f"SwiGLU bit-identical fraction {exact:.6f} over {d.size} outputs")
    assert exact >= 0.999, f"only {exact:.5f} of SwiGLU outputs bit-identical"
    return exact


def _check_amax(t, amax):
    want = t.float().abs().max()
    assert torch.equal(amax.cpu().view(torch.int32), want.cpu().reshape(1).view(torch.int32)), \
        (float(amax), float(want))


@pytest.mark.parametrize("M,N,K", [(300, 512, 512), (1000, 1024, 3072), (129, 256, 64)])
def test_swiglu_matches_plain_epilogue(orc, M, N, K):
    d = W.swiglu_fc1_inputs(M, N, K)
    _, y, h, amax_plain, amax_h = _run_pair(d)
    _check_swiglu(orc, y, h)
    _check_amax(y, amax_plain)
    _check_amax(h, amax_h)


def test_swiglu_extreme_gate_values(orc):
    """Gate values over [-120, 120] (set through the gate rows' bias), where
    e^-g alone would overflow fp32 below g = -88.7 and sigmoid(g) is subnormal:
    h stays within one bf16 step of the oracle's SwiGLU of the plain output."""
    d = W.swiglu_fc1_inputs(256, 512, 128)
    b = d["bias"].copy()
    for t in range(d["N"] // 256):
        b[256 * t:256 * t + 128] = W.to_bf16_bits(np.linspace(-120.0, 120.0, 128, dtype=np.float32)
                                                  + np.float32(t))
    d["bias"] = b
    _, y, h, _, amax_h = _run_pair(d)
    g = W.bf16_bits_to_f32(host_u16(y)[:, :128])
    assert g.min() < -100 and g.max() > 100 and ((g > -104) & (g < -87)).any()
    _check_swiglu(orc, y, h)
    _check_amax(h, amax_h)


# Largest |silu'(g)| over all real g (about 1.0998, near g = 2.4).
SILU_LIPSCHITZ = 1.1


def swiglu_end_to_end_bound(silu_yg, bg, yu, bu, h_true):
    """Tolerance for h = bf16(silu(g) * u) computed from GPU FC1 values g, u
    that lie within bg, bu of the oracle's float64 FC1 outputs yg, yu (the
    linear's own bound, bf16 rounding of g and u included):
      |silu(g) u - silu(yg) yu| <= (|silu(yg)| + L bg) bu + L bg |yu|,  L = max|silu'|,
    then h's own rounding to bf16 (half a step, <= 2^-8 relative) and the fp32
    evaluation of silu of the value reached: the approximate 2^x and 1/x and the
    rounding of the argument -|g| log2 e leave < 3.4e-6 < 2^-17 relative for
    |g| < 88 (the first term dominates beyond)."""
    first = (np.abs(silu_yg) + SILU_LIPSCHITZ * bg) * bu + SILU_LIPSCHITZ * bg * np.abs(yu)
    return first + (2.0 ** -8 + 2.0 ** -17) * (np.abs(h_true) + first)


def test_swiglu_full_size_end_to_end(orc):
    """FC1 with the SwiGLU producer at its full size (X [32768, 3072] with the
    prologue, W [24576, 3072]) -> h [32768, 12288], against the oracle end to
    end: the float64 oracle FC1 outputs of the gate and up columns, silu(g) * u
    of those in float64, and the derived bound above.  Rows: one per 256-row
    pair tile of M (alternating the CTA of the pair and the lane quarter) plus
    the edges, every h column of each."""
    d = W.swiglu_fc1_inputs(32768)
    M, N = d["M"], d["N"]
    _, y, h, _, amax_h = _run_pair(d)
    _check_amax(h, amax_h)
    rng = np.random.default_rng(11)
    t = np.arange((M + 255) // 256)
    rows = np.unique(np.concatenate([256 * t + 128 * (t % 2) + 32 * ((t // 2) % 4) + rng.integers(0, 32, t.size),
                                     [0, 127, 128, 255, 256, M - 1]]))
    rows = rows[rows < M]
    H = N // 2
    j = np.arange(H)
    gcol = 256 * (j // 128) + j % 128
    rr = np.repeat(rows, H)
    pts_g = np.stack([rr, np.tile(gcol, rows.size)], axis=1).astype(np.int64)
    pts_u = pts_g + np.array([0, 128], np.int64)
    a, w = oracle_operands(orc, d)
    yg, bg = orc.linear_points(a, w, M, N, d["K"], pts_g, bias=d["bias"])
    yu, bu = orc.linear_points(a, w, M, N, d["K"], pts_u, bias=d["bias"])
    h_true = orc.silu_mul_f64(yg, yu)
    bound = swiglu_end_to_end_bound(orc.silu_mul_f64(yg, np.ones_like(yg)), bg, yu, bu, h_true)
    got = W.bf16_bits_to_f32(host_u16(h)[rows].ravel()).astype(np.float64)
    err = np.abs(got - h_true)
    ratio = float(np.max(err / np.maximum(bound, 1e-300)))
    print(f"SwiGLU end to end: {got.size} outputs over {rows.size} rows, max err/bound {ratio:.3f}")
    assert (err <= bound).all(), (f"{int((err > bound).sum())} h outside the end-to-end bound; "
                                  f"max err/bound {ratio:.3g}")


def test_swiglu_full_size_sampled_rows(orc):
    """FC1 at its full size -> h: sampled rows (tile and pair edges included)
    against the oracle's SwiGLU of the GPU's own plain FC1 output (one bf16
    step, 99.9 % bit-identical)."""
    d = W.swiglu_fc1_inputs(32768)
    _, y, h, _, amax_h = _run_pair(d)
    rng = np.random.default_rng(11)
    rows = np.unique(np.concatenate([rng.integers(0, 32768, 48), [0, 127, 128, 255, 256, 32767]]))
    _check_swiglu(orc, y, h, torch.from_numpy(rows).cuda())
    _check_amax(h, amax_h)


def test_swiglu_chain_into_fc2_quantisation(orc):
    """h quantised with the scale from the producer's amax equals the two-pass
    quantisation of h (GPU and oracle), and the FC2 linear accepts it."""
    import audio_dit_gb300 as A
    d = W.swiglu_fc1_inputs(384, 512, 512)
    case, _, h, _, amax_h = _run_pair(d)
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    A.h3fp4_gscale_from_amax(amax_h, gs)
    hb = host_u16(h)
    one_pass = gpu_quantize(hb, gscale=float(gs.cpu()[0]))
    two_pass = gpu_quantize(hb)
    assert_quant_equal(one_pass, two_pass, "one pass (producer amax) vs two passes")
    assert_quant_equal(one_pass, orc.quantize(hb), "one pass vs oracle")
    # the FC2 linear consuming h with the caller-given global scale
    w2 = W.to_bf16_bits(np.random.default_rng(5).standard_normal((256, 256), dtype=np.float32) * np.float32(0.01))
    from _gpu_helpers import dev_bf16
    wq = A.alloc_nvfp4(256, 256)
    ws2 = A.alloc_workspace(384, 256, 256, 0)
    A.h3fp4_quantize_weight(dev_bf16(w2), *wq, ws2)
    out_given = torch.empty((384, 256), dtype=torch.bfloat16, device="cuda")
    out_amax = torch.empty_like(out_given)
    A.h3fp4_linear(h, *wq, out_given, ws2, a_gscale=gs, gscale_given=True)
    A.h3fp4_linear(h, *wq, out_amax, ws2)
    A.h3fp4_check(ws2)
    assert torch.equal(out_given.view(torch.int16), out_amax.view(torch.int16))


def test_out_amax_with_gate_residual_and_segments():
    """The output amax of the gated epilogue (two segments, residual) is exactly
    max |out| of the stored bf16 output, including a ragged last tile."""
    import audio_dit_gb300 as A
    d = W.make_inputs("attn_out", M=333)
    case = LinearCase(d)
    out = case.run(out_amax=True)
    torch.cuda.synchronize()
    _check_amax(out, A.h3fp4_ws_out_amax(case.ws).clone())


def _nvfp4_out_case(orc, M, N, K, check_oracle=True):
    """FC1 SwiGLU writing h as NVFP4 under the scale of its own amax, against
    the quantiser (GPU and oracle) applied to the bf16 h of the plain SwiGLU
    epilogue, and FC2 on those codes against FC2 on h with the same scale."""
    import audio_dit_gb300 as A
    from _gpu_helpers import check_guards, dev_bf16, guarded_nvfp4
    d = W.swiglu_fc1_inputs(M, N, K)
    case, _, h, _, amax_h = _run_pair(d)
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    A.h3fp4_gscale_from_amax(amax_h, gs)
    gq = guarded_nvfp4(M, N // 2)
    codes, sf = gq[0].t, gq[1].t
    A.h3fp4_linear_swiglu_nvfp4(case.x, *case.wq, codes, sf, gs, case.ws, shift=case.shift, scale=case.scale,
                                bias=case.bias)
    A.h3fp4_check(case.ws)
    check_guards(gq[:2], "h NVFP4")
    case.check_guards()
    hb = host_u16(h)
    got = (codes.cpu().numpy(), sf.cpu().numpy(), float(gs.cpu()[0]))
    assert_quant_equal(got, gpu_quantize(hb, gscale=got[2]), "h NVFP4 vs GPU quantiser")
    if check_oracle:
        assert_quant_equal(got, orc.quantize(hb, gscale=got[2]), "h NVFP4 vs oracle quantiser")
    # FC2 on the emitted codes == FC2 on h with the same global scale
    rng = np.random.default_rng(M + N)
    N2 = 256
    w2 = W.to_bf16_bits(rng.standard_normal((N2, N // 2), dtype=np.float32) * np.float32(0.01))
    wq2 = A.alloc_nvfp4(N2, N // 2)
    ws2 = A.alloc_workspace(M, N2, N // 2, 0)
    A.h3fp4_quantize_weight(dev_bf16(w2), *wq2, ws2)
    o_codes = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    o_h = torch.empty_like(o_codes)
    A.h3fp4_linear(codes, *wq2, o_codes, ws2, a_sf=sf, a_gscale=gs)
    A.h3fp4_linear(h, *wq2, o_h, ws2, a_gscale=gs, gscale_given=True)
    A.h3fp4_check(ws2)
    assert torch.equal(o_codes.view(torch.int16), o_h.view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(300, 512, 512), (1000, 1024, 3072), (129, 256, 64), (385, 768, 320)])
def test_swiglu_nvfp4_output(orc, M, N, K):
    _nvfp4_out_case(orc, M, N, K)


def test_swiglu_nvfp4_output_full_size(orc):
    """FC1 at full size (X [32768, 3072], W [24576, 3072]): h [32768, 12288]
    emitted as NVFP4 equals the quantiser's bytes for the bf16 h."""
    _nvfp4_out_case(orc, 32768, 24576, 3072)
