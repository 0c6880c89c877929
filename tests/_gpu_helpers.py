"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
on seeded workload inputs and compare with the CPU oracle."""
import numpy as np
import torch

import workloads as W


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def dev_f32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host_u16(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def gpu_quantize(x_u16, shift=None, scale=None, seg_off=None, gscale=None, weight=False):
    """Quantise on the GPU through the C ABI; returns numpy (codes, sf, gscale)."""
    import audio_dit_gb300 as A
    rows, K = x_u16.shape
    x = dev_bf16(x_u16)
    codes, sf, gs = A.alloc_nvfp4(rows, K)
    ws = A.alloc_workspace(rows, 0, K, A.A_PREQUANT)
    if weight:
        A.h3fp4_quantize_weight(x, codes, sf, gs, ws)
    else:
        if gscale is not None:
            gs.fill_(gscale)
        A.h3fp4_quantize_act(x, codes, sf, gs, ws, shift=dev_f32(shift), scale=dev_f32(scale),
                             seg_off=None if seg_off is None else list(seg_off),
                             gscale_given=gscale is not None)
    A.h3fp4_check(ws)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), sf.cpu().numpy(), float(gs.cpu().numpy()[0])


def assert_quant_equal(gpu, ref, what=""):
    gc, gsf, ggs = gpu
    rc, rsf, rgs = ref
    assert np.float32(ggs).tobytes() == np.float32(rgs).tobytes(), f"{what}: global scale {ggs!r} vs {rgs!r}"
    if not np.array_equal(gsf, rsf):
        bad = np.nonzero(gsf != rsf)[0]
        raise AssertionError(f"{what}: {bad.size} block-scale bytes differ, first at {bad[:5]}: "
                             f"gpu {gsf[bad[:5]]} oracle {rsf[bad[:5]]}")
    if not np.array_equal(gc, rc):
        bad = np.argwhere(gc != rc)
        raise AssertionError(f"{what}: {len(bad)} code bytes differ, first at {bad[:5].tolist()}: "
                             f"gpu {gc[tuple(bad[:5].T)]} oracle {rc[tuple(bad[:5].T)]}")


class LinearCase:
    """Device buffers for one linear problem built from a workload dict."""

    def __init__(self, d, use_bias=True):
        import audio_dit_gb300 as A
        self.d = d
        self.M, self.N, self.K = d["M"], d["N"], d["K"]
        self.x = dev_bf16(d["x"])
        self.w = dev_bf16(d["w"])
        self.shift = dev_f32(d["shift"])
        self.scale = dev_f32(d["scale"])
        self.gate = dev_f32(d["gate"])
        self.resid = None if d["resid"] is None else dev_bf16(d["resid"])
        self.bias = dev_bf16(d["bias"]) if use_bias else None
        self.seg_off = [int(v) for v in d["seg_off"]]
        self.wq = A.alloc_nvfp4(self.N, self.K)
        self.ws = A.alloc_workspace(max(self.M, self.N), self.N, self.K, 0)
        A.h3fp4_quantize_weight(self.w, *self.wq, self.ws)
        self.out = torch.empty((self.M, self.N), dtype=torch.bfloat16, device="cuda")

    def run(self, **kw):
        import audio_dit_gb300 as A
        A.h3fp4_linear(self.x, *self.wq, self.out, self.ws, shift=self.shift, scale=self.scale,
                       gate=self.gate, resid=self.resid, bias=self.bias, seg_off=self.seg_off, **kw)
        A.h3fp4_check(self.ws)
        return self.out

    def weight_quant_host(self):
        c, s, g = self.wq
        torch.cuda.synchronize()
        return c.cpu().numpy(), s.cpu().numpy(), float(g.cpu().numpy()[0])


def oracle_operands(orc, d):
    a = orc.quantize(d["x"], d["shift"], d["scale"], d["seg_off"])
    w = orc.quantize(d["w"])
    return a, w


def check_outputs(out_bf16: np.ndarray, ref: np.ndarray, bound: np.ndarray, what=""):
    got = W.bf16_bits_to_f32(out_bf16).astype(np.float64)
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad) if bad.ndim > 1 else np.nonzero(bad)[0]
        i0 = tuple(idx[0]) if bad.ndim > 1 else idx[0]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outputs outside tolerance; first {i0}: "
                             f"gpu {got[i0]!r} oracle {ref[i0]!r} bound {bound[i0]!r}; "
                             f"max err/bound {float(np.max(err / np.maximum(bound, 1e-300))):.3g}")
    return float(np.max(err / np.maximum(bound, 1e-300)))


def sample_points(M, N, n, seed, seg_off=None):
    rng = np.random.default_rng(seed)
    pts = np.stack([rng.integers(0, M, n), rng.integers(0, N, n)], axis=1)
    edges = [(0, 0), (M - 1, N - 1), (M - 1, 0), (0, N - 1), (M // 2, N // 2)]
    if seg_off is not None and len(seg_off) > 2:
        for b in seg_off[1:-1]:
            edges += [(b - 1, 7), (b, 7), (b, N - 1)]
    return np.concatenate([pts, np.array(edges, np.int64)]).astype(np.int64)
