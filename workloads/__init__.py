"""Seeded synthetic inputs for the verification pass.

This module is shared by the tests (which feed the same bytes to the oracle and
to the CUDA library) and by ``bench.py``. It holds none of the verification
arithmetic: it only draws logits, draft tokens and uniforms with the shapes and
value distributions of the workloads below.

Synthetic traffic stands in for the pages' serving workloads and datasets,
which are not available here. Recipe (per workload, seed ``s``):

* ``zt`` target logits ``[B, K+1, V]``: i.i.d. normal with the workload's sigma,
  optionally a spike added at one uniformly drawn token of every row, or a
  per-row temperature ``T ~ U(lo, hi)`` dividing the row; rows of sequences
  ``b >= B/2`` may use a second recipe (the FLy workload).
* ``zd`` draft logits ``[B, K, V]`` = target rows ``0..K-1`` plus i.i.d. normal
  noise. Both are rounded once to the storage dtype (round-to-nearest-even for
  bf16).
* ``x`` draft tokens ``[B, K]``: a draw from softmax of the stored draft row via
  the Gumbel-max identity (argmax of logits plus Gumbel noise), or the draft
  row's argmax for greedy drafting.
* ``u`` uniforms ``[B, K+1]`` in ``[0, 1)`` from a second generator seeded ``s+1``.
* ``inv_temp`` (workloads with a sampling temperature only) ``[B]`` float32:
  a per-sequence inverse temperature, log-uniform on ``[lo, hi]``, from a
  third generator seeded ``s+2``; the drafts are then drawn from the softmax
  of the stored draft row times it (the distribution the draft samples from
  at that temperature).

All values come from ``torch.Generator(device)`` seeded with ``s`` (Philox on
CUDA, mt19937 on CPU), so a given (workload, seed, device) always yields the
same bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    dtype: str                 # "bf16" | "f32"
    mode: str                  # "stochastic" | "greedy" | "fly"
    sigma_t: float = 3.0       # target logit std
    sigma_d: float = 1.0       # draft noise std
    spike: float = 0.0         # added at one random token per target row
    temp_range: Optional[tuple] = None   # per-row temperature U(lo, hi)
    # second recipe for sequences b >= B/2 (FLy workload): (sigma, spike)
    upper_half: Optional[tuple] = None
    # sampling inverse temperature per sequence, log-uniform on (lo, hi)
    inv_temp_range: Optional[tuple] = None
    draft_tokens: str = "sample"         # "sample" (x ~ q) | "argmax"
    fly_theta: float = 0.3
    fly_window: int = 6
    with_confidence: bool = False
    estimator_lr: float = 0.05

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logit_bytes(self, with_draft: Optional[bool] = None) -> int:
        """Bytes of logits one verification call reads once."""
        if with_draft is None:
            with_draft = self.mode == "stochastic" or self.with_confidence
        rows = (self.K + 1) + (self.K if with_draft else 0)
        return self.B * rows * self.V * self.elem_bytes


TINY = Workload("tiny_B4_K4_V1024_f32", B=4, K=4, V=1024, dtype="f32", mode="stochastic",
                sigma_t=3.0, sigma_d=1.0)
LLAMA3_VOCAB = Workload("llama3vocab_B64_K5_V128256_bf16", B=64, K=5, V=128256, dtype="bf16",
                        mode="stochastic", sigma_t=2.5, sigma_d=0.8, spike=12.0)
ESTIMATOR = Workload("estimator_B256_K8_V128256_bf16", B=256, K=8, V=128256, dtype="bf16",
                     mode="stochastic", sigma_t=3.0, sigma_d=1.0, temp_range=(0.5, 2.0),
                     with_confidence=True, estimator_lr=0.05)
FLY = Workload("fly_B128_K15_V152064_bf16", B=128, K=15, V=152064, dtype="bf16", mode="fly",
               sigma_t=0.5, sigma_d=1.5, upper_half=(4.0, 15.0), draft_tokens="argmax",
               fly_theta=0.3, fly_window=6)


def sweep():
    """The throughput sweep: B x K x V x dtype, stochastic mode."""
    out = []
    for dt in ("bf16", "f32"):
        for V in (32000, 128256, 152064):
            for K in (4, 8):
                for B in (32, 128, 512, 1024):
                    out.append(Workload(f"sweep_B{B}_K{K}_V{V}_{dt}", B=B, K=K, V=V, dtype=dt,
                                        mode="stochastic", sigma_t=3.0, sigma_d=1.0))
    return out


WORKLOADS = {w.name: w for w in (TINY, LLAMA3_VOCAB, ESTIMATOR, FLY)}


def _torch_dtype(w: Workload):
    return torch.bfloat16 if w.dtype == "bf16" else torch.float32


@torch.no_grad()
def make_inputs(w: Workload, seed: int, device="cpu", chunk_rows: int = 1 << 14):
    """Draw (zt, zd, x, u) for workload ``w`` on ``device``.

    Generation runs in chunks of whole sequences so that temporaries stay small
    for the multi-GB workloads.
    """
    device = torch.device(device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    gu = torch.Generator(device=device)
    gu.manual_seed(seed + 1)
    B, K, V = w.B, w.K, w.V
    dt = _torch_dtype(w)
    zt = torch.empty((B, K + 1, V), dtype=dt, device=device)
    zd = torch.empty((B, K, V), dtype=dt, device=device)
    x = torch.empty((B, K), dtype=torch.int32, device=device)
    s_inv = None
    if w.inv_temp_range is not None:
        gs = torch.Generator(device=device)
        gs.manual_seed(seed + 2)
        lo, hi = (float(v) for v in w.inv_temp_range)
        r = torch.rand((B,), generator=gs, device=device, dtype=torch.float64)
        s_inv = torch.exp(math.log(lo) + (math.log(hi) - math.log(lo)) * r).to(torch.float32)
    seqs_per_chunk = max(1, chunk_rows // (2 * K + 1))
    for b0 in range(0, B, seqs_per_chunk):
        b1 = min(B, b0 + seqs_per_chunk)
        n = b1 - b0
        t = torch.randn((n, K + 1, V), generator=g, device=device, dtype=torch.float32)
        sig = torch.full((n, 1, 1), w.sigma_t, device=device)
        spike = torch.full((n, 1, 1), w.spike, device=device)
        if w.upper_half is not None:
            upper = (torch.arange(b0, b1, device=device) >= B // 2).view(n, 1, 1)
            sig = torch.where(upper, torch.full_like(sig, w.upper_half[0]), sig)
            spike = torch.where(upper, torch.full_like(spike, w.upper_half[1]), spike)
        t.mul_(sig)
        if w.temp_range is not None:
            lo, hi = w.temp_range
            T = lo + (hi - lo) * torch.rand((n, K + 1, 1), generator=g, device=device)
            t.div_(T)
        pos = torch.randint(0, V, (n, K + 1, 1), generator=g, device=device)
        if w.spike != 0.0 or w.upper_half is not None:
            t.scatter_add_(2, pos, spike.expand(n, K + 1, 1).contiguous())
        zt[b0:b1] = t.to(dt)
        d = t[:, :K] + w.sigma_d * torch.randn((n, K, V), generator=g, device=device)
        zd[b0:b1] = d.to(dt)
        del t
        dq = zd[b0:b1].float()
        if s_inv is not None:
            dq = dq * s_inv[b0:b1].view(n, 1, 1)
        if w.draft_tokens == "argmax":
            x[b0:b1] = dq.argmax(dim=-1).to(torch.int32)
        else:
            # Gumbel-max: argmax(z + G), G = -log(-log U), is a draw from softmax(z)
            gum = torch.rand((n, K, V), generator=g, device=device)
            gum = -torch.log(-torch.log(gum))
            x[b0:b1] = (dq + gum).argmax(dim=-1).to(torch.int32)
            del gum
        del d, dq
    u = torch.rand((B, K + 1), generator=gu, device=device, dtype=torch.float32)
    out = dict(zt=zt, zd=zd, x=x, u=u)
    if s_inv is not None:
        out["inv_temp"] = s_inv
    return out


def to_numpy_logits(z: torch.Tensor):
    """CPU numpy view of logits: float32 as is, bf16 as raw uint16 bits."""
    z = z.detach().cpu().contiguous()
    if z.dtype == torch.bfloat16:
        return z.view(torch.int16).numpy().view("uint16")
    return z.numpy()
