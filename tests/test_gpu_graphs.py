"""CUDA-graph shape buckets over a block's four projections (GPU).

A block's QKV (with AdaLN prologue), attention-output (two segments, gate and
residual), FC1 with the SwiGLU producer and its amax, and FC2 on h with the
derived global scale are captured once per token count and replayed.  Every
replayed output must be bit-identical to the eager calls on the same inputs,
also after new inputs are written into the captured buffers.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)


@pytest.fixture(scope="module", autouse=True)
def built():
    from audio_dit_gb300 import build
    build.build()


class Block:
    MAX_M = 640
    K, NQKV, NATT, N1, N2 = 3072, 9216, 3072, 1024, 3072

    def __init__(self, seed=0):
        import audio_dit_gb300 as A
        self.A = A
        g = torch.Generator(device="cuda").manual_seed(seed)
        rn = lambda *s, std=1.0: (torch.randn(*s, generator=g, device="cuda") * std)
        K, M = self.K, self.MAX_M
        self.w = {}
        for name, (n, k, std) in {"qkv": (self.NQKV, K, 0.02), "att": (self.NATT, K, 0.02),
                                  "fc1": (self.N1, K, 0.02), "fc2": (self.N2, self.N1 // 2, 0.01)}.items():
            wq = A.alloc_nvfp4(n, k)
            ws = A.alloc_workspace(n, 0, k, A.A_PREQUANT)
            A.h3fp4_quantize_weight(rn(n, k, std=std).bfloat16(), *wq, ws)
            self.w[name] = wq
        self.bias = {n: rn(c, std=0.01).bfloat16() for n, c in
                     [("qkv", self.NQKV), ("att", self.NATT), ("fc1", self.N1), ("fc2", self.N2)]}
        self.shift, self.scale = rn(1, K, std=0.1), rn(1, K, std=0.1)
        self.seg_shift, self.seg_scale = rn(2, K, std=0.1), rn(2, K, std=0.1)
        self.gate_att = torch.rand(2, self.NATT, generator=g, device="cuda")
        self.gate_fc2 = torch.rand(1, self.N2, generator=g, device="cuda")
        self.x = {n: torch.empty(M, K, dtype=torch.bfloat16, device="cuda") for n in ("qkv", "att", "fc1")}
        self.resid_att = torch.empty(M, self.NATT, dtype=torch.bfloat16, device="cuda")
        self.resid_fc2 = torch.empty(M, self.N2, dtype=torch.bfloat16, device="cuda")
        self.out = {"qkv": torch.empty(M, self.NQKV, dtype=torch.bfloat16, device="cuda"),
                    "att": torch.empty(M, self.NATT, dtype=torch.bfloat16, device="cuda"),
                    "h": torch.empty(M, self.N1 // 2, dtype=torch.bfloat16, device="cuda"),
                    "fc2": torch.empty(M, self.N2, dtype=torch.bfloat16, device="cuda")}
        self.ws = {n: A.alloc_workspace(M, 0, k, 0) for n, k in
                   [("qkv", K), ("att", K), ("fc1", K), ("fc2", self.N1 // 2)]}
        self.gs2 = torch.empty(1, dtype=torch.float32, device="cuda")
        self.fill(seed + 1)

    def fill(self, seed):
        g = torch.Generator(device="cuda").manual_seed(seed)
        for t in list(self.x.values()) + [self.resid_att, self.resid_fc2]:
            t.copy_(torch.randn(t.shape, generator=g, device="cuda"))

    def issue(self, M):
        A, K = self.A, self.K
        A.h3fp4_linear(self.x["qkv"][:M], *self.w["qkv"], self.out["qkv"][:M], self.ws["qkv"],
                       shift=self.shift, scale=self.scale, bias=self.bias["qkv"])
        seg = [0, M - 128, M]
        A.h3fp4_linear(self.x["att"][:M], *self.w["att"], self.out["att"][:M], self.ws["att"],
                       shift=self.seg_shift, scale=self.seg_scale, gate=self.gate_att,
                       resid=self.resid_att[:M], bias=self.bias["att"], seg_off=seg)
        A.h3fp4_linear(self.x["fc1"][:M], *self.w["fc1"], self.out["h"][:M], self.ws["fc1"],
                       shift=self.shift, scale=self.scale, bias=self.bias["fc1"], swiglu=True, out_amax=True)
        A.h3fp4_gscale_from_amax(A.h3fp4_ws_out_amax(self.ws["fc1"]), self.gs2)
        A.h3fp4_linear(self.out["h"][:M], *self.w["fc2"], self.out["fc2"][:M], self.ws["fc2"],
                       a_gscale=self.gs2, gscale_given=True, gate=self.gate_fc2, resid=self.resid_fc2[:M],
                       bias=self.bias["fc2"])

    def snapshot(self, M):
        torch.cuda.synchronize()
        return {k: v[:M].clone() for k, v in self.out.items()}

    def check(self):
        for ws in self.ws.values():
            self.A.h3fp4_check(ws)


def _same(a, b):
    for k in a:
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k


def test_graph_buckets_replay_bit_identical():
    from audio_dit_gb300.graphs import GraphBuckets
    blk = Block()
    buckets = GraphBuckets(blk.issue)
    for M in (256, 640):
        blk.issue(M)
        eager = blk.snapshot(M)
        for k in blk.out.values():
            k.zero_()
        buckets.run(M)
        _same(eager, blk.snapshot(M))
        blk.check()
    assert len(buckets) == 2 and 256 in buckets
    # new inputs written into the captured buffers
    blk.fill(99)
    blk.issue(256)
    eager = blk.snapshot(256)
    for k in blk.out.values():
        k.zero_()
    buckets.run(256)
    _same(eager, blk.snapshot(256))
    buckets.run(256)                 # a second replay of the same bucket
    _same(eager, blk.snapshot(256))
    blk.check()
