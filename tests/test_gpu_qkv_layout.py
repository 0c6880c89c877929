"""QKV output consumed as strided NHD views (GPU).

The QKV projection writes [M, 3*H*D] row-major; attention reads Q, K and V as
strided [M, H, D] views of it (token stride 3*H*D, head stride D), with no copy.
Each view must equal, bit for bit, the output of the same linear restricted to
that projection's weight rows: the GEMM computes every output column the same
way wherever it sits in the N dimension.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from _gpu_helpers import dev_bf16, dev_f32  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


def test_qkv_strided_nhd_views_match_per_projection_outputs():
    import audio_dit_gb300 as A
    d = W.make_inputs("qkv", M=700)
    M, K, N = d["M"], d["K"], d["N"]
    H, D = 24, 128
    assert N == 3 * H * D
    x, w, bias = dev_bf16(d["x"]), dev_bf16(d["w"]), dev_bf16(d["bias"])
    shift, scale = dev_f32(d["shift"]), dev_f32(d["scale"])
    # one global weight scale shared by the three slices: quantise W once, slice codes and scales
    wq = A.alloc_nvfp4(N, K)
    ws = A.alloc_workspace(max(M, N), N, K, 0)
    A.h3fp4_quantize_weight(w, *wq, ws)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    A.h3fp4_linear(x, *wq, out, ws, shift=shift, scale=scale, bias=bias)
    qkv = out.view(M, 3, H, D)
    sf_rows = A.h3fp4_sf_bytes(H * D, K)   # scale bytes of 3072 rows (a multiple of 128)
    for t in range(3):
        rows = slice(t * H * D, (t + 1) * H * D)
        codes = wq[0][rows].contiguous()
        sf = wq[1][t * sf_rows:(t + 1) * sf_rows].contiguous()
        part = torch.empty(M, H * D, dtype=torch.bfloat16, device="cuda")
        A.h3fp4_linear(x, codes, sf, wq[2], part, ws, shift=shift, scale=scale, bias=bias[rows].contiguous())
        A.h3fp4_check(ws)
        view = qkv[:, t]                       # [M, H, D], strides (N, D, 1)
        assert view.stride() == (N, D, 1)
        assert torch.equal(view.reshape(M, H * D).view(torch.int16), part.view(torch.int16)), t
