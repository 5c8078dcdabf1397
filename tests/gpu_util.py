"""Helpers of the GPU parity tests: host arrays to device tensors, calls through the C ABI,
comparison with the oracle."""

import numpy as np
import torch

from workloads import BF16

MARGIN = 1e-5   # draws closer than this (relative) to a decision or CDF boundary are flagged


def dev(a: np.ndarray, offset_elems: int = 0) -> torch.Tensor:
    """Copy a host array to cuda:0 (uint16 arrays become bfloat16). With offset_elems > 0 the
    tensor is a view starting that many elements into a larger allocation, so its base address
    is deliberately not 16-byte aligned."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    if offset_elems:
        flat = t.reshape(-1)
        big = torch.empty(flat.numel() + offset_elems, dtype=flat.dtype, device="cuda")
        big[offset_elems:].copy_(flat)
        t = big[offset_elems:].view(t.shape)
    else:
        t = t.to("cuda")
    return t.view(torch.bfloat16) if a.dtype == np.uint16 else t


def run_chain(ci, offset_elems=0, workspace=None):
    import speculative_decoding_verification_78_gb300 as sv
    tgt = dev(ci.target, offset_elems)
    drf = dev(ci.draft, offset_elems) if ci.draft.size else None
    tok = dev(ci.tokens) if ci.tokens.size else None
    uni = dev(ci.uniforms)
    acc, out, st = sv.verify_chain(tgt, drf, tok, uni, ci.temperature, workspace=workspace)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), int(st.item())


def run_tree(ti, offset_elems=0):
    import speculative_decoding_verification_78_gb300 as sv
    acc, path, out, st = sv.verify_tree(dev(ti.target, offset_elems), dev(ti.parents),
                                        dev(ti.tokens))
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), int(st.item())


def compare_chain(orc, ci, gpu, rows=None):
    """Exact match on every batch row whose oracle margin is >= MARGIN. Rows below it
    (near-boundary draws) are counted and reported; their GPU outputs must still be a valid
    step: n in [0, gamma], the accepted prefix equal to the drafts, one token in [0, V), then
    -1. Returns (flagged, flagged_and_different, oracle accept_len)."""
    acc, out, _ = gpu
    tgt, drf, tok, uni = ci.target, ci.draft, ci.tokens, ci.uniforms
    if rows is not None:
        tgt, drf, tok, uni = tgt[rows], drf[rows], tok[rows], uni[rows]
        acc, out = acc[rows], out[rows]
    oa, oo, om, rc = orc.verify_chain(tgt, drf if drf.size else None, ci.dtype, tok, uni,
                                      ci.temperature)
    ok = om >= MARGIN
    diff = (acc != oa) | np.any(out != oo, axis=1)
    bad = np.nonzero(ok & diff)[0]
    assert bad.size == 0, (f"{ci.name}: {bad.size} rows differ, e.g. row {bad[:5]}: "
                           f"gpu {acc[bad[:3]]} {out[bad[:3]]} oracle {oa[bad[:3]]} "
                           f"{oo[bad[:3]]} margins {om[bad[:3]]}")
    g = ci.gamma
    for b in np.nonzero(~ok)[0]:
        n = int(acc[b])
        assert 0 <= n <= g
        assert np.array_equal(out[b, :n], tok[b, :n])
        assert 0 <= out[b, n] < ci.V and np.all(out[b, n + 1:] == -1)
    flagged = int((~ok).sum())
    fdiff = int((~ok & diff).sum())
    report(ci.name, rows=len(ok), flagged=flagged, flagged_and_different=fdiff)
    return flagged, fdiff, oa


def report(name, **kw):
    """Appends one JSON line per comparison to the file named by SPEC_PARITY_REPORT, when that
    variable is set (the counts of near-boundary draws are part of the result)."""
    import json
    import os
    path = os.environ.get("SPEC_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(name=name, **kw)) + "\n")


def to_np_logits(t: torch.Tensor, dtype: int) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == BF16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
