"""Seeded synthetic inputs for the causal (GQA) long-sequence attention workloads.

This module holds shapes, seeds and value distributions only. It contains none of the
attention arithmetic: the fp64 oracle (``oracle/``) and the CUDA path
(``context_parallelism_gb300``) both draw their inputs from here and share nothing else.

Recipe (the same for every workload):
  * tensors are token-major: q and dO ``[B, S, Hq, D]``, k and v ``[B, S, Hkv, D]``;
  * they are drawn in the order q, k, v, dO from ONE ``torch.Generator`` seeded with
    ``Workload.seed``, as standard normals in fp32, multiplied by ``std`` and rounded
    to bf16 (round-to-nearest-even, torch's ``.to(torch.bfloat16)``);
  * a "peaky" workload then draws a permutation of the S token positions from the same
    generator and multiplies every entry of K at the first ``floor(peaky_frac * S)``
    positions by ``peaky_scale`` (8 is a power of two, so the scaling is exact in bf16);
  * small workloads are drawn on the CPU, large ones (>= 1 GiB of q) on the GPU
    (``gen_device``). The oracle reads back exactly the bf16 bytes the GPU path consumes.

The pages measure no public dataset; these tensors stand in for the activations of a
Llama3-8B-shaped (Hq=32, Hkv=8, D=128) and a 32B-class (Hq=64, Hkv=8, D=128) attention
layer. No weights are involved.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    Hq: int
    Hkv: int
    D: int
    head_chunk: int
    seq_trunk: int
    seed: int
    std: float = 1.0
    peaky_frac: float = 0.0
    peaky_scale: float = 8.0
    kv_on_host: bool = False
    causal: bool = True
    gen_device: str = "cpu"

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops_fwd(self) -> float:
        """Causal FLOP convention of the FlashAttention benchmarks: QK^T and PV, each
        2*B*Hq*S*S*D, halved by the causal mask; non-causal doubles it."""
        f = 4.0 * self.B * self.Hq * self.D * self.S * self.S
        return f / 2.0 if self.causal else f

    def flops_bwd(self) -> float:
        return 2.5 * self.flops_fwd()


# The five workloads: (1) small MHA check, (2) Llama3-8B-shaped S=8K,
# (3) Llama3-8B-shaped S=128K, (4) S=1M with K/V resident in pinned host memory,
# (5) 32B-class S=256K with 1% of K rows scaled x8.
WORKLOADS = {
    "mha_s512_d64": Workload("mha_s512_d64", B=1, S=512, Hq=4, Hkv=4, D=64,
                             head_chunk=4, seq_trunk=512, seed=0),
    "llama8b_s8k": Workload("llama8b_s8k", B=1, S=8192, Hq=32, Hkv=8, D=128,
                            head_chunk=8, seq_trunk=8192, seed=1),
    "llama8b_s128k": Workload("llama8b_s128k", B=1, S=131072, Hq=32, Hkv=8, D=128,
                              head_chunk=8, seq_trunk=131072, seed=2, gen_device="cuda"),
    "llama8b_s1m_hostkv": Workload("llama8b_s1m_hostkv", B=1, S=1048576, Hq=32, Hkv=8,
                                   D=128, head_chunk=4, seq_trunk=65536, seed=3, std=0.5,
                                   kv_on_host=True, gen_device="cuda"),
    "gqa32b_s256k_peaky": Workload("gqa32b_s256k_peaky", B=1, S=262144, Hq=64, Hkv=8,
                                   D=128, head_chunk=8, seq_trunk=32768, seed=4,
                                   peaky_frac=0.01, gen_device="cuda"),
}

WORKLOAD_ORDER = ["mha_s512_d64", "llama8b_s8k", "llama8b_s128k",
                  "llama8b_s1m_hostkv", "gqa32b_s256k_peaky"]


def _normal_bf16(shape, gen, device, std):
    # Drawn in fp32 then rounded: the same recipe on CPU and GPU. Large tensors are drawn
    # in slabs along the leading token axis to bound the fp32 temporary.
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1, shape[-1])
    rows = flat.shape[0]
    slab = max(1, (1 << 27) // shape[-1])
    for r0 in range(0, rows, slab):
        r1 = min(rows, r0 + slab)
        t = torch.randn((r1 - r0, shape[-1]), generator=gen, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        flat[r0:r1].copy_(t)
    return out


def make_inputs(w: Workload, device: str | None = None):
    """Return (q, k, v, dout) as bf16 torch tensors on ``device`` (default: w.gen_device)."""
    dev = device or w.gen_device
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    q = _normal_bf16((w.B, w.S, w.Hq, w.D), gen, dev, w.std)
    k = _normal_bf16((w.B, w.S, w.Hkv, w.D), gen, dev, w.std)
    v = _normal_bf16((w.B, w.S, w.Hkv, w.D), gen, dev, w.std)
    do = _normal_bf16((w.B, w.S, w.Hq, w.D), gen, dev, w.std)
    if w.peaky_frac > 0.0:
        n = int(math.floor(w.peaky_frac * w.S))
        rows = torch.randperm(w.S, generator=gen, device=dev)[:n]
        k[:, rows] = (k[:, rows].float() * w.peaky_scale).to(torch.bfloat16)
    return q, k, v, do


def peaky_rows(w: Workload, device: str | None = None):
    """The token positions whose K rows ``make_inputs`` scales (empty if not peaky)."""
    if w.peaky_frac <= 0.0:
        return torch.empty(0, dtype=torch.long)
    dev = device or w.gen_device
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    for shape in ((w.B, w.S, w.Hq, w.D), (w.B, w.S, w.Hkv, w.D),
                  (w.B, w.S, w.Hkv, w.D), (w.B, w.S, w.Hq, w.D)):
        _normal_bf16(shape, gen, dev, w.std)
    n = int(math.floor(w.peaky_frac * w.S))
    return torch.randperm(w.S, generator=gen, device=dev)[:n].cpu()


def random_small(B, S, Hq, Hkv, D, seed, dtype=torch.float64, std=1.0):
    """Small fp64 (default) CPU tensors for oracle self-tests: (q, k, v, dout)."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((B, S, Hq, D), generator=gen, dtype=torch.float64) * std
    k = torch.randn((B, S, Hkv, D), generator=gen, dtype=torch.float64) * std
    v = torch.randn((B, S, Hkv, D), generator=gen, dtype=torch.float64) * std
    do = torch.randn((B, S, Hq, D), generator=gen, dtype=torch.float64) * std
    return q.to(dtype), k.to(dtype), v.to(dtype), do.to(dtype)


def sample_rows(S: int, seq_trunk: int, n: int, seed: int):
    """Seeded query-row sample for large-S parity checks: always includes the tile and
    trunk edges {0, 1, 127, 128, T-1, T, S/2, S-1} (those < S), then uniform draws."""
    fixed = {0, 1, 127, 128, seq_trunk - 1, seq_trunk, S // 2, S - 1}
    fixed = sorted(i for i in fixed if 0 <= i < S)
    gen = torch.Generator().manual_seed(seed)
    extra = torch.randint(0, S, (max(0, n - len(fixed)),), generator=gen).tolist()
    return sorted(set(fixed) | set(extra))


# ---- sequence-tiled loss (readout + cross-entropy) ----------------------------------------

@dataclass(frozen=True)
class LossWorkload:
    """A language-model readout + token-level cross-entropy problem.

    Recipe: from ONE ``torch.Generator`` seeded with ``seed``, in this order: h [S, Dm] as
    standard normals (fp32, rounded to bf16; the scale of a normalised final hidden state),
    w [V, Dm] as normals of std ``w_std / sqrt(Dm)`` rounded to bf16 (logits of std about
    ``w_std``), target [S] uniform in [0, V), then a Bernoulli(``ignore_frac``) mask that sets
    the target of masked tokens to -1 (ignored: padding). The upstream gradient is the mean
    over the counted tokens, 1 / #(target >= 0), for every counted token.
    Shapes stand in for a Llama3-8B-shaped model (Dm 4096, vocabulary 128256); no weights
    are involved."""
    name: str
    S: int
    Dm: int
    V: int
    seq_tile: int
    seed: int
    w_std: float = 2.0
    ignore_frac: float = 1.0 / 16
    gen_device: str = "cpu"

    def flops_fwd(self) -> float:
        """The readout GEMM, 2 S V Dm (the merge and the epilogues are not counted)."""
        return 2.0 * self.S * self.V * self.Dm

    def flops_bwd(self) -> float:
        """Recomputed logits, dh = dlogits w and dw = dlogits^T h: three GEMMs."""
        return 3.0 * self.flops_fwd()

    def with_(self, **kw) -> "LossWorkload":
        return dataclasses.replace(self, **kw)


LOSS_WORKLOADS = {
    "readout_small": LossWorkload("readout_small", S=1000, Dm=256, V=1088, seq_tile=256,
                                  seed=20),
    "llama8b_readout_s128k": LossWorkload("llama8b_readout_s128k", S=131072, Dm=4096,
                                          V=128256, seq_tile=8192, seed=21,
                                          gen_device="cuda"),
}


def make_loss_inputs(lw: LossWorkload, device: str | None = None):
    """Return (h bf16 [S, Dm], w bf16 [V, Dm], target int64 [S], dloss float32 [S])."""
    dev = device or lw.gen_device
    gen = torch.Generator(device=dev)
    gen.manual_seed(lw.seed)
    h = _normal_bf16((lw.S, lw.Dm), gen, dev, 1.0)
    w = _normal_bf16((lw.V, lw.Dm), gen, dev, lw.w_std / math.sqrt(lw.Dm))
    target = torch.randint(0, lw.V, (lw.S,), generator=gen, device=dev, dtype=torch.int64)
    if lw.ignore_frac > 0.0:
        drop = torch.rand((lw.S,), generator=gen, device=dev) < lw.ignore_frac
        target[drop] = -1
    n = int((target >= 0).sum().item())
    dloss = torch.full((lw.S,), 1.0 / max(1, n), dtype=torch.float32, device=dev)
    return h, w, target, dloss


# ---- sequence-tiled gated MLP ---------------------------------------------------------------

@dataclass(frozen=True)
class MlpWorkload:
    """A gated (SwiGLU) MLP over S tokens.

    Recipe: from ONE ``torch.Generator`` seeded with ``seed``, in this order, each drawn as
    fp32 normals and rounded to bf16: x [S, Dm] with std 1 (a normalised hidden state),
    w_gu [2F, Dm] (gate rows, then up rows) with std 1/sqrt(Dm), w_d [Dm, F] with std
    1/sqrt(F), and the upstream gradient dy [S, Dm] with std 1. Shapes stand in for a
    Llama3-8B-shaped MLP (Dm 4096, F 14336); no weights are involved."""
    name: str
    S: int
    Dm: int
    F: int
    seq_tile: int
    seed: int
    gen_device: str = "cpu"

    def flops_fwd(self) -> float:
        """Gate/up projection 4 S Dm F plus down projection 2 S Dm F."""
        return 6.0 * self.S * self.Dm * self.F

    def flops_bwd(self) -> float:
        """Gate/up recompute 4, da 2, dWd 2, dWgu 4, dx 4 (units of S Dm F)."""
        return 16.0 * self.S * self.Dm * self.F

    def with_(self, **kw) -> "MlpWorkload":
        return dataclasses.replace(self, **kw)


MLP_WORKLOADS = {
    "mlp_small": MlpWorkload("mlp_small", S=1000, Dm=256, F=384, seq_tile=256, seed=30),
    "llama8b_mlp_s128k": MlpWorkload("llama8b_mlp_s128k", S=131072, Dm=4096, F=14336,
                                     seq_tile=8192, seed=31, gen_device="cuda"),
}


def make_mlp_inputs(mw: MlpWorkload, device: str | None = None):
    """Return (x, w_gu, w_d, dy), all bf16."""
    dev = device or mw.gen_device
    gen = torch.Generator(device=dev)
    gen.manual_seed(mw.seed)
    x = _normal_bf16((mw.S, mw.Dm), gen, dev, 1.0)
    w_gu = _normal_bf16((2 * mw.F, mw.Dm), gen, dev, 1.0 / math.sqrt(mw.Dm))
    w_d = _normal_bf16((mw.Dm, mw.F), gen, dev, 1.0 / math.sqrt(mw.F))
    dy = _normal_bf16((mw.S, mw.Dm), gen, dev, 1.0)
    return x, w_gu, w_d, dy
