"""Seeded synthetic chain inputs drawn directly on a CUDA device (torch), for the large
benchmark configurations whose host generation would take minutes.

The recipes are those of ``workloads.synthetic`` (same distributions, same drafting rule, same
uniforms), drawn with torch's device generator instead of numpy, so the values differ from the
host generators' while the workload is the same. Like the host generators this module draws
inputs only: it holds none of the verify step's arithmetic. bf16 logits are rounded from fp32
to nearest even (torch's conversion), as the host generators do.
"""

from __future__ import annotations

import torch

from .synthetic import BF16


def device_chain(B: int, gamma: int, V: int, dtype: int, temperature: float,
                 target_sigma: float, draft_sigma: float, zipf_s: float = 0.0, seed: int = 0,
                 device="cuda", block_bytes: int = 1 << 29):
    """Chain inputs on `device`: target ~ N(0, target_sigma^2) - zipf_s * ln(k + 1) over token
    id k, draft = target + N(0, draft_sigma^2), both stored as bf16 (dtype == BF16) or fp32;
    draft tokens by the Gumbel-max trick on the stored draft logits at the given temperature
    (argmax at T = 0); uniforms (2k + 1) / 2^24. Generated in blocks of batch rows so that the
    fp32 temporaries stay below block_bytes. Returns (target, draft, tokens int32, uniforms fp32)
    device tensors of shapes [B, gamma+1, V], [B, gamma, V], [B, gamma], [B, gamma+1]."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    tdt = torch.bfloat16 if dtype == BF16 else torch.float32
    tgt = torch.empty((B, gamma + 1, V), dtype=tdt, device=device)
    drf = torch.empty((B, gamma, V), dtype=tdt, device=device)
    tok = torch.empty((B, gamma), dtype=torch.int32, device=device)
    prior = None
    if zipf_s:
        ids = torch.arange(1, V + 1, dtype=torch.float64, device=device)
        prior = (-zipf_s * torch.log(ids)).float()
    nb = max(1, block_bytes // (4 * (2 * gamma + 1) * V))
    for b0 in range(0, B, nb):
        b1 = min(B, b0 + nb)
        t = torch.randn((b1 - b0, gamma + 1, V), generator=g, device=device) * target_sigma
        if prior is not None:
            t += prior
        tgt[b0:b1] = t.to(tdt)
        if gamma:
            d = t[:, :gamma] + torch.randn((b1 - b0, gamma, V), generator=g,
                                           device=device) * draft_sigma
            drf[b0:b1] = d.to(tdt)
            dq = drf[b0:b1].float()
            if temperature > 0:
                u = torch.rand(dq.shape, generator=g, device=device).clamp_min_(1e-30)
                dq = dq / temperature - torch.log(-torch.log(u))
            tok[b0:b1] = torch.argmax(dq, dim=-1).to(torch.int32)
        del t
    k = torch.randint(0, 1 << 23, (B, gamma + 1), generator=g, device=device)
    uni = ((2 * k + 1).to(torch.float64) / float(1 << 24)).to(torch.float32)
    return tgt, drf, tok, uni


def logits_bytes(B: int, rows: int, V: int, dtype: int) -> int:
    return B * rows * V * (2 if dtype == BF16 else 4)


__all__ = ["device_chain", "logits_bytes"]
