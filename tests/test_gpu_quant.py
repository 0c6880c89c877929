"""GPU parity of the NVFP4 quantiser against the oracle: codes, block scales
and global scales must be bit-exact (modulation prologue, segments, padding,
caller-given scale, edge shapes, exhaustive convert domains)."""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import assert_quant_equal, gpu_quantize  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


@pytest.mark.parametrize("name,M", [("tiny", None), ("qkv", 300), ("fc1", 1000), ("fc2", 257), ("attn_out", 700)])
def test_act_quant_reduced(orc, name, M):
    d = W.make_inputs(name, M=M)
    ref = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    gpu = gpu_quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    assert_quant_equal(gpu, ref, f"{name} M={d['M']}")


@pytest.mark.parametrize("name", ["qkv", "fc1", "fc2", "attn_out"])
def test_act_quant_full_size(orc, name):
    d = W.make_inputs(name)
    ref = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    gpu = gpu_quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    assert_quant_equal(gpu, ref, f"{name} full")


@pytest.mark.parametrize("name", ["tiny", "qkv", "fc1", "fc2", "attn_out"])
def test_weight_quant(orc, name):
    d = W.make_inputs(name, M=8)
    ref = orc.quantize(d["w"])
    gpu = gpu_quantize(d["w"], weight=True)
    assert_quant_equal(gpu, ref, f"{name} weight")


def test_gscale_given(orc):
    d = W.make_inputs("attn_out", M=333)
    for gs in [1.0, 0.0123, 3.5e-3]:
        ref = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"], gscale=gs)
        gpu = gpu_quantize(d["x"], d["shift"], d["scale"], d["seg_off"], gscale=gs)
        assert_quant_equal(gpu, ref, f"given {gs}")


def test_max_segments_with_empty_and_single_row_segments(orc):
    """The largest segment table the boundary accepts, with an empty segment
    and a one-row segment: every row takes its own segment's vectors, and the
    empty segment's vectors are never used."""
    import audio_dit_gb300 as A
    M, K = 200, 1024
    seg = np.array([0, 3, 3, 4, 40, 41, 100, 163, 200], np.int64)
    nseg = len(seg) - 1
    assert nseg == A.MAX_SEGMENTS
    rng = np.random.default_rng(201)
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    shift = rng.standard_normal((nseg, K), dtype=np.float32) * 0.1
    scale = rng.standard_normal((nseg, K), dtype=np.float32) * 0.1
    shift[1] = 1e6  # the empty segment: using it for any row would show
    ref = orc.quantize(x, shift, scale, seg)
    gpu = gpu_quantize(x, shift, scale, seg)
    assert_quant_equal(gpu, ref, f"{nseg} segments")


@pytest.mark.parametrize("M,K", [(1, 64), (7, 128), (127, 3072), (128, 64), (129, 512), (946, 3072), (5, 12288)])
def test_edge_rows(orc, M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = W.to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))
    assert_quant_equal(gpu_quantize(x), orc.quantize(x), f"M={M} K={K}")


def test_special_values(orc):
    K = 256
    x = np.zeros((6, K), np.float32)
    x[1, 17] = 1000.0                       # single outlier
    x[2] = -0.0                             # negative zeros
    x[3, :16] = 1e-38                       # tiny normal values
    x[4, ::2] = 2.0 ** -130                 # subnormal bf16 values
    x[5] = np.linspace(-3, 3, K)
    xb = W.to_bf16_bits(x)
    xb[2] = 0x8000
    assert_quant_equal(gpu_quantize(xb), orc.quantize(xb), "special")
    z = np.zeros((130, 64), np.uint16)
    assert_quant_equal(gpu_quantize(z), orc.quantize(z), "all zero")


def test_e2m1_convert_every_bf16_in_range(orc):
    """With s = 1 and a block maximum of 6 the block scale is exactly 1, so the
    codes are e2m1(m) for every bf16 m in [-6, 6] -- all such values, ties
    included, through the kernel's convert."""
    bits = np.arange(0, 0x10000, dtype=np.uint32).astype(np.uint16)
    f = W.bf16_bits_to_f32(bits)
    vals = bits[np.isfinite(f) & (np.abs(f) <= 6.0)]
    vals = np.concatenate([vals, np.full((-len(vals)) % 15, 0, np.uint16)])
    blocks = vals.reshape(-1, 15)
    six = np.full((len(blocks), 1), W.to_bf16_bits(np.array([6.0], np.float32))[0], np.uint16)
    rows = np.concatenate([blocks, six], axis=1).reshape(-1)
    K = 1024
    rows = np.concatenate([rows, np.zeros((-len(rows)) % K, np.uint16)]).reshape(-1, K)
    assert_quant_equal(gpu_quantize(rows, gscale=1.0), orc.quantize(rows, gscale=1.0), "e2m1 domain")


def test_e4m3_convert_grid_and_ties(orc):
    """Block maxima 6*v for every E4M3 value v and every midpoint between
    neighbours make the scale input exactly v (s = 1): grid points, ties to
    even and saturation through the kernel's convert."""
    grid = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    mids = (grid[:-1] + grid[1:]) / 2
    v = np.concatenate([grid, mids, [464.0, 480.0, 1024.0]])
    bmax = (6 * v).astype(np.float32)
    assert np.all(W.bf16_bits_to_f32(W.to_bf16_bits(bmax)) == bmax)  # exact in bf16
    blocks = np.zeros((len(bmax), 16), np.float32)
    blocks[:, 0] = bmax
    blocks[:, 1] = -bmax / 3
    blocks[:, 5] = bmax / 7
    xb = W.to_bf16_bits(blocks).reshape(-1)
    K = 512
    xb = np.concatenate([xb, np.zeros((-len(xb)) % K, np.uint16)]).reshape(-1, K)
    assert_quant_equal(gpu_quantize(xb, gscale=1.0), orc.quantize(xb, gscale=1.0), "e4m3 domain")
