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

from .synthetic import BF16, lmhead_grid_scales


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


def device_lmhead_grid(B: int, gamma: int, V: int, Ht: int, Hd: int, temperature: float,
                       target_sigma: float = 3.0, draft_sigma: float = 1.0, seed: int = 0,
                       device="cuda", block_rows: int = 512):
    """workloads.synthetic.lmhead_grid's recipe drawn on `device`: integer-grid hidden states
    (a / 8) and LM heads (c / 64) in bf16, the drafter sharing the first min(Ht, Hd) hidden
    components with the target and perturbing its head there. Draft tokens are the drafter's
    own samples: the Gumbel-max trick on its logits, which are formed here with a plain torch
    matrix product (the drafter's last layer, upstream of verification), block_rows rows at a
    time. Returns (hidden_t, head_t, hidden_d, head_d, tokens [B, gamma] int32, uniforms
    [B, gamma+1] fp32) device tensors."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    sc = lmhead_grid_scales(Ht, Hd, target_sigma, draft_sigma)
    s = sc["shared"]
    Mt, Md = B * (gamma + 1), B * gamma
    bf = torch.bfloat16

    def ints(shape, m):
        return torch.randint(-m, m + 1, shape, generator=g, device=device, dtype=torch.int32)

    hidden_t = (ints((Mt, Ht), 4).float() / 8).to(bf)
    head_t = torch.empty((V, Ht), dtype=bf, device=device)
    head_t[:, :s] = (ints((V, s), sc["m_shared"]).float() / 64).to(bf)
    if Ht > s:
        head_t[:, s:] = (ints((V, Ht - s), sc["m_target_only"]).float() / 64).to(bf)
    rows_t = (torch.arange(B, device=device)[:, None] * (gamma + 1) +
              torch.arange(gamma, device=device)[None, :]).reshape(-1)
    hidden_d = torch.empty((Md, Hd), dtype=bf, device=device)
    hidden_d[:, :s] = hidden_t[rows_t, :s]
    if Hd > s:
        hidden_d[:, s:] = (ints((Md, Hd - s), 4).float() / 8).to(bf)
    head_d = torch.empty((V, Hd), dtype=bf, device=device)
    head_d[:, :s] = (head_t[:, :s].float() + ints((V, s), sc["m_delta"]).float() / 64).to(bf)
    if Hd > s:
        head_d[:, s:] = (ints((V, Hd - s), sc["m_draft_only"]).float() / 64).to(bf)
    tok = torch.empty(Md, dtype=torch.int32, device=device)
    wd = head_d.float()
    for r0 in range(0, Md, block_rows):
        r1 = min(Md, r0 + block_rows)
        lg = hidden_d[r0:r1].float() @ wd.T
        if temperature > 0:
            u = torch.rand(lg.shape, generator=g, device=device).clamp_min_(1e-30)
            lg = lg / temperature - torch.log(-torch.log(u))
        tok[r0:r1] = torch.argmax(lg, dim=-1).to(torch.int32)
    del wd
    k = torch.randint(0, 1 << 23, (B, gamma + 1), generator=g, device=device)
    uni = ((2 * k + 1).to(torch.float64) / float(1 << 24)).to(torch.float32)
    return hidden_t, head_t, hidden_d, head_d, tok.view(B, gamma), uni


def logits_bytes(B: int, rows: int, V: int, dtype: int) -> int:
    return B * rows * V * (2 if dtype == BF16 else 4)


__all__ = ["device_chain", "device_lmhead_grid", "logits_bytes"]
