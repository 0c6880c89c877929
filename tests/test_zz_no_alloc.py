"""GPU test of h3fp4_quantize_act_noalloc, the quantiser entry point for
callers that may not allocate device memory (it keeps its amax scratch in a
static device array of the library instead of a caller workspace).

Its codes, block scales and global scale must equal those of
h3fp4_quantize_act -- bit for bit, the quantiser's tolerance -- on two calls in
a row (the second call reuses the scratch the first one left behind).  This
file is collected last so that a run stopping at its first failure has already
run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module")
def A():
    from audio_dit_gb300 import build
    build.build()
    import audio_dit_gb300
    audio_dit_gb300.load_library()
    return audio_dit_gb300


def _dev_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def _dev_f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


@pytest.mark.parametrize("name,M,given", [("attn_out", 700, False), ("fc2", 257, False), ("qkv", 300, True)])
def test_noalloc_matches_workspace_quantiser_twice(A, name, M, given):
    d = W.make_inputs(name, M=M)
    K = d["K"]
    x = _dev_bf16(d["x"])
    shift, scale = _dev_f32(d["shift"]), _dev_f32(d["scale"])
    seg = [int(v) for v in d["seg_off"]]
    ref = A.alloc_nvfp4(M, K)
    ws = A.alloc_workspace(M, 0, K, A.A_PREQUANT)
    if given:
        ref[2].fill_(0.0123)
    A.h3fp4_quantize_act(x, *ref, ws, shift=shift, scale=scale, seg_off=seg, gscale_given=given)
    A.h3fp4_check(ws)
    for call in range(2):
        codes = torch.full_like(ref[0], 0xA5)
        sf = torch.full_like(ref[1], 0x5A)
        gs = torch.full_like(ref[2], -1.0)
        if given:
            gs.fill_(0.0123)
        A.h3fp4_quantize_act_noalloc(x, codes, sf, gs, shift=shift, scale=scale, seg_off=seg, gscale_given=given)
        torch.cuda.synchronize()
        assert torch.equal(codes, ref[0]), f"codes differ on call {call}"
        assert torch.equal(sf, ref[1]), f"block scales differ on call {call}"
        assert torch.equal(gs, ref[2]), f"global scale differs on call {call}"


def test_noalloc_rejects_oversized_k(A):
    lib = A.load_library()
    dummy = 4096
    # K beyond the static scratch's reach (4096 partials x 1024 columns)
    assert lib.h3fp4_quantize_act_noalloc(dummy, 1, 4096 * 1024 + 64, None, None, None, 1, dummy, dummy, dummy,
                                          0, None) == 2
