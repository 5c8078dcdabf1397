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
