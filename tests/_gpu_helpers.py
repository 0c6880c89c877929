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


GUARD_BYTES = 4096
CANARY = 0xA5


class Guarded:
    """A device buffer between two canary-filled guard regions (a host-side
    substitute for a memory checker): after a call, `check` fails if any byte
    before or after the buffer, or in its padding up to a 256-byte multiple,
    changed.  `t` is the buffer itself (zero-filled or left at the canary)."""

    def __init__(self, shape, dtype, zero=False):
        itemsize = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape)) * itemsize
        padded = (self.n + 255) // 256 * 256
        self.raw = torch.full((GUARD_BYTES + padded + GUARD_BYTES,), CANARY, dtype=torch.uint8, device="cuda")
        inner = self.raw[GUARD_BYTES:GUARD_BYTES + self.n]
        if zero:
            inner.zero_()
        self.t = inner.view(dtype).view(*shape)

    def check(self, what=""):
        torch.cuda.synchronize()
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.n:]
        for part, name in ((head, "before"), (tail, "after")):
            bad = torch.nonzero(part != CANARY)
            if bad.numel():
                raise AssertionError(f"{what}: {bad.numel()} guard bytes {name} the buffer were written "
                                     f"(first at offset {int(bad[0])})")


def guarded_nvfp4(rows, K):
    """Guarded (codes, sf, gscale) buffers: the layout of audio_dit_gb300.alloc_nvfp4."""
    import audio_dit_gb300 as A
    return [Guarded((rows, K // 2), torch.uint8), Guarded((A.h3fp4_sf_bytes(rows, K),), torch.uint8),
            Guarded((1,), torch.float32)]


def guarded_workspace(M, N, K, flags=0):
    import audio_dit_gb300 as A
    return Guarded((A.h3fp4_workspace_bytes(M, N, K, flags),), torch.uint8, zero=True)


def check_guards(bufs, what=""):
    for i, b in enumerate(bufs):
        b.check(f"{what} buffer {i}")


def gpu_quantize(x_u16, shift=None, scale=None, seg_off=None, gscale=None, weight=False):
    """Quantise on the GPU through the C ABI; returns numpy (codes, sf, gscale).
    Every output buffer and the workspace sit between canary guards, checked
    after the call."""
    import audio_dit_gb300 as A
    rows, K = x_u16.shape
    x = dev_bf16(x_u16)
    g = guarded_nvfp4(rows, K)
    gws = guarded_workspace(rows, 0, K, A.A_PREQUANT)
    codes, sf, gs = (b.t for b in g)
    ws = gws.t
    if weight:
        A.h3fp4_quantize_weight(x, codes, sf, gs, ws)
    else:
        if gscale is not None:
            gs.fill_(gscale)
        A.h3fp4_quantize_act(x, codes, sf, gs, ws, shift=dev_f32(shift), scale=dev_f32(scale),
                             seg_off=None if seg_off is None else list(seg_off),
                             gscale_given=gscale is not None)
    A.h3fp4_check(ws)
    check_guards(g + [gws], "quantise")
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
        # weight NVFP4 buffers, workspace and output between canary guards
        self._gwq = guarded_nvfp4(self.N, self.K)
        self.wq = tuple(b.t for b in self._gwq)
        self._gws = guarded_workspace(max(self.M, self.N), self.N, self.K, 0)
        self.ws = self._gws.t
        A.h3fp4_quantize_weight(self.w, *self.wq, self.ws)
        self._gout = Guarded((self.M, self.N), torch.bfloat16)
        self.out = self._gout.t
        self.check_guards()

    def check_guards(self, extra=()):
        check_guards(self._gwq + [self._gws, self._gout] + list(extra), f"linear {self.M}x{self.N}x{self.K}")

    def run(self, **kw):
        import audio_dit_gb300 as A
        A.h3fp4_linear(self.x, *self.wq, self.out, self.ws, shift=self.shift, scale=self.scale,
                       gate=self.gate, resid=self.resid, bias=self.bias, seg_off=self.seg_off, **kw)
        A.h3fp4_check(self.ws)
        self.check_guards()
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


def tile_points(M, N, seed, BM=128, BN=256):
    """Stratified output points: in every 256 x 256 pair tile of the GEMM's
    persistent schedule, one random point for each (CTA of the pair, 32-row
    lane quarter, 128-column half) -- every epilogue warp of every tile of
    every round, the partial last wave included; points past M or N are
    dropped (ragged tiles keep the ones inside)."""
    rng = np.random.default_rng(seed)
    pm, nt = (M + 2 * BM - 1) // (2 * BM), (N + BN - 1) // BN
    mp, n0 = np.meshgrid(np.arange(pm), np.arange(nt), indexing="ij")
    mp, n0 = mp.ravel(), n0.ravel()
    pts = []
    for r in range(2):
        for q in range(4):
            for h in range(2):
                row = mp * 2 * BM + r * BM + 32 * q + rng.integers(0, 32, mp.size)
                col = n0 * BN + 128 * h + rng.integers(0, 128, mp.size)
                pts.append(np.stack([row, col], axis=1))
    pts = np.concatenate(pts).astype(np.int64)
    return pts[(pts[:, 0] < M) & (pts[:, 1] < N)]
