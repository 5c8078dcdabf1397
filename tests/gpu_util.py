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
    """Checks a GPU chain result against the oracle draw by draw.

    The oracle's detail evaluates every position of every batch row (decision, and the draw the
    step would make if it stopped there). With n the GPU's accept length:
      - every decision the GPU took (accept x_i for i < n, reject x_n when n < gamma) must be the
        oracle's, unless that decision's margin is below MARGIN (then either is correct);
      - the accepted prefix equals the drafts, entries after position n are -1;
      - the emitted token equals the oracle's draw at position n, unless that draw's margin is
        below MARGIN: then it must lie in the draw's band (the tokens whose CDF cell comes within
        MARGIN * P of u * S) and have p_n > 0 (for a correction also p_n >= (1 - MARGIN) q_n,
        i.e. a residual that fp32 rounding can make positive).
    So accept_len is compared exactly unless the deciding draw is itself near a boundary.
    Invalid rows must match exactly (-1 everywhere). Returns (flagged draws on the oracle's
    path, of those the ones where the GPU differs, oracle accept_len)."""
    acc, out, _ = gpu
    tgt, drf, tok, uni = ci.target, ci.draft, ci.tokens, ci.uniforms
    if rows is not None:
        tgt, drf, tok, uni = tgt[rows], drf[rows], tok[rows], uni[rows]
        acc, out = acc[rows], out[rows]
    g, T = ci.gamma, ci.temperature
    dr = drf if drf.size and T > 0 else None
    oa, oo, _, _ = orc.verify_chain(tgt, dr, ci.dtype, tok, uni, T)
    d = orc.verify_chain_detail(tgt, dr, ci.dtype, tok, uni, T, band=MARGIN)
    n_dec = n_draw = f_dec = f_draw = f_diff = 0
    bad = []
    for b in range(len(acc)):
        n, no = int(acc[b]), int(oa[b])
        if no < 0 or d["tok"][b, 0] < 0:          # invalid row: exact
            if n != -1 or np.any(out[b] != -1):
                bad.append((b, "invalid row not reported"))
            continue
        # the oracle's path: its decisions and its draw, flagged when near a boundary
        path_dec = range(min(no + 1, g))
        n_dec += len(path_dec)
        n_draw += 1
        fl_dec = [i for i in path_dec if d["dmargin"][b, i] < MARGIN]
        fl_draw = d["cmargin"][b, no] < MARGIN
        f_dec += len(fl_dec)
        f_draw += int(fl_draw)
        if not 0 <= n <= g:
            bad.append((b, f"accept_len {n}"))
            continue
        ok = True
        for i in range(min(n + 1, g)):        # the decisions the GPU took
            gpu_accepts = i < n
            if gpu_accepts != bool(d["accept"][b, i]) and d["dmargin"][b, i] >= MARGIN:
                bad.append((b, f"decision {i}: gpu n={n}, oracle n={no}, "
                               f"margin {d['dmargin'][b, i]:.3g}"))
                ok = False
                break
        if not ok:
            continue
        if not np.array_equal(out[b, :n], tok[b, :n]) or np.any(out[b, n + 1:] != -1):
            bad.append((b, "prefix or padding"))
            continue
        t = int(out[b, n])
        if d["cmargin"][b, n] >= MARGIN:
            if t != d["tok"][b, n]:
                bad.append((b, f"token {t} != {d['tok'][b, n]} at n={n}, "
                               f"margin {d['cmargin'][b, n]:.3g}"))
        elif not (d["lo"][b, n] <= t <= d["hi"][b, n] and _drawable(orc, ci, tgt, dr, b, n, t)):
            bad.append((b, f"token {t} outside band [{d['lo'][b, n]}, {d['hi'][b, n]}] at n={n}"))
        # a row that passed and still differs from the oracle's path has a flagged draw on it
        f_diff += int(n != no or t != int(oo[b, n]))
    assert not bad, f"{ci.name}: {len(bad)} rows fail, e.g. {bad[:4]}"
    report(ci.name, rows=len(acc), decisions=n_dec, draws=n_draw, flagged_decisions=f_dec,
           flagged_draws=f_draw, flagged_and_different=f_diff, outside_band=0)
    return f_dec + f_draw, f_diff, oa


def _drawable(orc, ci, tgt, dr, b, n, t):
    """The emitted token has p_n(t) > 0 and, for a correction (n < gamma), a residual that
    rounding can make positive: p_n(t) >= (1 - MARGIN) q_n(t)."""
    T = ci.temperature
    p, _ = orc.probs(tgt[b, n:n + 1], ci.dtype, T)
    if p[0, t] <= 0:
        return False
    if n < ci.gamma and dr is not None:
        q, _ = orc.probs(dr[b, n:n + 1], ci.dtype, T)
        return p[0, t] >= (1 - MARGIN) * q[0, t]
    return True


def compare_sample(orc, lg, dtype, u, T, tok):
    """spec_sample against the oracle, draw by draw (a sample is a chain step with no drafts:
    its one draw is the bonus draw): the token must equal the oracle's unless the draw's margin
    is below MARGIN, and then lie in the draw's band with p > 0. Returns the flagged count."""
    want, mg, rc = orc.sample(lg, dtype, u, T)
    rows, V = lg.shape
    d = orc.verify_chain_detail(lg.reshape(rows, 1, V), None, dtype,
                                np.zeros((rows, 0), np.int32), u.reshape(rows, 1), T,
                                band=MARGIN)
    np.testing.assert_array_equal(d["tok"][:, 0], want)
    p, _ = orc.probs(lg, dtype, T)
    flagged = 0
    for r in range(rows):
        if want[r] < 0 or mg[r] >= MARGIN:
            assert tok[r] == want[r], (r, tok[r], want[r], mg[r])
        else:
            flagged += 1
            assert d["lo"][r, 0] <= tok[r] <= d["hi"][r, 0] and p[r, tok[r]] > 0, \
                (r, tok[r], d["lo"][r, 0], d["hi"][r, 0])
    report("sample", rows=rows, draws=rows, flagged_draws=flagged, outside_band=0)
    return flagged


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


def run_tree_sample(ti, draft, uniforms, T, offset_elems=0):
    import speculative_decoding_verification_78_gb300 as sv
    acc, path, out, st = sv.verify_tree_sample(dev(ti.target, offset_elems),
                                               dev(draft, offset_elems), dev(ti.parents),
                                               dev(ti.tokens), dev(uniforms), T)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), path.cpu().numpy(), out.cpu().numpy(), int(st.item())


def compare_tree_sample(orc, ti, draft, uniforms, T, gpu, name="tree_sample"):
    """Stochastic tree verification against the oracle. A tree whose walk has no decision within
    MARGIN of its boundary must take the oracle's path exactly; its final token must be the
    oracle's unless the draw's margin is below MARGIN, and then lie in the oracle's band for it.
    A tree with a near-boundary decision may take another path: it must still be a valid walk
    (each path node the previous one's child, the tokens of the path, a final token of positive
    target probability at the last node). Invalid trees must match exactly. Returns (trees with
    a flagged decision, trees with a flagged draw, trees different from the oracle)."""
    acc, path, out, _ = gpu
    d = orc.verify_tree_sample_detail(ti.target, draft, ti.dtype, ti.parents, ti.tokens,
                                      uniforms, T, band=MARGIN)
    oa, op, oo = d["accept_len"], d["path_nodes"], d["out_tokens"]
    f_dec = f_draw = diff = 0
    bad = []
    for b in range(len(acc)):
        if oa[b] < 0:
            if acc[b] != -1 or np.any(out[b] != -1) or np.any(path[b] != -1):
                bad.append((b, "invalid tree not reported"))
            continue
        n = int(acc[b])
        same = (n == oa[b] and np.array_equal(path[b], op[b]) and np.array_equal(out[b], oo[b]))
        diff += int(not same)
        if d["dmargin"][b] >= MARGIN:
            if n != oa[b] or not np.array_equal(path[b], op[b]) or \
                    not np.array_equal(out[b, :n], oo[b, :n]) or np.any(out[b, n + 1:] != -1):
                bad.append((b, f"path differs: gpu {path[b, :n + 1]} oracle {op[b, :oa[b] + 1]}"))
                continue
            t = int(out[b, n])
            if d["cmargin"][b] >= MARGIN:
                if t != oo[b, n]:
                    bad.append((b, f"token {t} != {oo[b, n]}, margin {d['cmargin'][b]:.3g}"))
            else:
                f_draw += 1
                if not d["lo"][b] <= t <= d["hi"][b]:
                    bad.append((b, f"token {t} outside [{d['lo'][b]}, {d['hi'][b]}]"))
            continue
        f_dec += 1   # a near-boundary decision: any valid walk
        if not 0 <= n < ti.N or path[b, 0] != 0 or np.any(path[b, n + 1:] != -1):
            bad.append((b, "invalid walk"))
            continue
        ok = all(ti.parents[b, path[b, i]] == path[b, i - 1] and out[b, i - 1] == ti.tokens[b, path[b, i]]
                 for i in range(1, n + 1))
        p_last, _ = orc.probs(ti.target[b, path[b, n]:path[b, n] + 1], ti.dtype, T)
        t = int(out[b, n])
        if not (ok and 0 <= t < ti.V and p_last[0, t] > 0 and np.all(out[b, n + 1:] == -1)):
            bad.append((b, "invalid walk"))
    assert not bad, f"{name}: {len(bad)} trees fail, e.g. {bad[:4]}"
    report(name, trees=len(acc), flagged_decisions=f_dec, flagged_draws=f_draw,
           different=diff, outside_band=0)
    return f_dec, f_draw, diff
