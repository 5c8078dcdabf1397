"""Loads the hand-derived fixtures under tests/golden/ as numpy arrays."""

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f32(x, shape_hint=None):
    def conv(v):
        if isinstance(v, list):
            return [conv(e) for e in v]
        return float(v)
    a = np.asarray(conv(x), dtype=np.float32)
    if shape_hint is not None:
        a = a.reshape(shape_hint)
    return a


def chain_cases():
    with open(os.path.join(GOLDEN, "chain_cases.json")) as f:
        data = json.load(f)
    out = []
    for c in data["cases"]:
        V, g = c["V"], c["gamma"]
        tgt = _f32(c["target"])
        B = tgt.shape[0]
        drf = _f32(c["draft"], (B, g, V))
        out.append(dict(
            name=c["name"], T=float(c["T"]), V=V, gamma=g, target=tgt.reshape(B, g + 1, V),
            draft=drf, tokens=np.asarray(c["tokens"], dtype=np.int32).reshape(B, g),
            uniforms=np.asarray(c["uniforms"], dtype=np.float32).reshape(B, g + 1),
            accept_len=np.asarray(c["accept_len"], dtype=np.int32),
            out_tokens=np.asarray(c["out_tokens"], dtype=np.int32).reshape(B, g + 1)))
    return out


def tree_cases():
    with open(os.path.join(GOLDEN, "tree_cases.json")) as f:
        data = json.load(f)
    out = []
    for c in data["cases"]:
        tgt = _f32(c["target"])
        out.append(dict(
            name=c["name"], V=c["V"], target=tgt,
            parents=np.asarray(c["parents"], dtype=np.int32),
            tokens=np.asarray(c["tokens"], dtype=np.int32),
            accept_len=np.asarray(c["accept_len"], dtype=np.int32),
            path_nodes=np.asarray(c["path_nodes"], dtype=np.int32),
            out_tokens=np.asarray(c["out_tokens"], dtype=np.int32)))
    return out


def _rational(v):
    """'a/b' -> a/b as a float ('1/ln2' -> 1/ln 2); numbers pass through."""
    import math
    from fractions import Fraction
    if isinstance(v, str):
        if v == "1/ln2":
            return 1.0 / math.log(2.0)
        if v == "inf":
            return math.inf
        return float(Fraction(v))
    return float(v)


def margin_cases():
    """The boundary-margin fixtures: inputs as for chain_cases, plus the per-position
    expectations of the oracle's detail (accept, dmargin, tok, cmargin, lo, hi)."""
    with open(os.path.join(GOLDEN, "margin_cases.json")) as f:
        data = json.load(f)
    out = []
    for c in data["cases"]:
        V, g = c["V"], c["gamma"]
        tgt = _f32(c["target"])
        B = tgt.shape[0]
        rat = lambda x: np.asarray([[_rational(v) for v in row] for row in x], np.float64)
        out.append(dict(
            name=c["name"], T=_rational(c["T"]), V=V, gamma=g, band=float(data["band"]),
            target=tgt.reshape(B, g + 1, V), draft=_f32(c["draft"], (B, g, V)),
            tokens=np.asarray(c["tokens"], dtype=np.int32).reshape(B, g),
            uniforms=rat(c["uniforms"]).astype(np.float32),
            accept=np.asarray(c["accept"], dtype=np.int32), dmargin=rat(c["dmargin"]),
            tok=np.asarray(c["tok"], dtype=np.int32), cmargin=rat(c["cmargin"]),
            lo=np.asarray(c["lo"], dtype=np.int32), hi=np.asarray(c["hi"], dtype=np.int32),
            accept_len=np.asarray(c["accept_len"], dtype=np.int32),
            out_tokens=np.asarray(c["out_tokens"], dtype=np.int32).reshape(B, g + 1)))
    return out


def tree_sample_cases():
    """The stochastic tree-verification fixtures (one tree per case, B = 1)."""
    with open(os.path.join(GOLDEN, "tree_sample_cases.json")) as f:
        data = json.load(f)
    out = []
    for c in data["cases"]:
        V = c["V"]
        N = len(c["parents"])
        out.append(dict(
            name=c["name"], T=_rational(c["T"]), V=V,
            target=_f32(c["target"], (1, N, V)), draft=_f32(c["draft"], (1, N, V)),
            parents=np.asarray(c["parents"], dtype=np.int32).reshape(1, N),
            tokens=np.asarray(c["tokens"], dtype=np.int32).reshape(1, N),
            uniforms=np.asarray(c["uniforms"], dtype=np.float32).reshape(1, N),
            accept_len=np.asarray([c["accept_len"]], dtype=np.int32),
            path_nodes=np.asarray(c["path_nodes"], dtype=np.int32).reshape(1, N),
            out_tokens=np.asarray(c["out_tokens"], dtype=np.int32).reshape(1, N),
            margin=_rational(c["margin"])))
    return out
