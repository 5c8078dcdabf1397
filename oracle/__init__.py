"""CPU oracle of the speculative-decoding verify step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference arm
may import this package. The product path (the CUDA library and its binding) never does, and
this package imports nothing from it.

The arithmetic lives in ``spec_oracle.c`` (plain single-threaded C in double precision); this
module only compiles it with gcc and marshals numpy arrays through ctypes. The one exception is
the LM-head product of ``lm_head_logits``, a float64 numpy matrix product (a library routine)
whose results the C code rounds to bf16.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libspec_oracle.so")
_lock = threading.Lock()
_lib = None

F32 = 0
BF16 = 1

# error codes of spec_oracle.c
OK, ERR_ROW, ERR_TOKEN, ERR_PARENT, ERR_ARG, ERR_MEM = 0, -1, -2, -3, -4, -5


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into libspec_oracle.so (no fast-math, no FMA contraction, so
    the same doubles come out on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i64, dbl, i32 = ctypes.c_void_p, ctypes.c_long, ctypes.c_double, ctypes.c_int
            lib.oracle_probs.argtypes = [vp, i32, i64, i64, dbl, vp]
            lib.oracle_argmax.argtypes = [vp, i32, i64, i64, vp]
            lib.oracle_verify_chain.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, dbl, vp,
                                                vp, vp]
            lib.oracle_verify_chain_detail.argtypes = [vp, vp, i32, vp, vp, i64, i64, i64, dbl,
                                                       dbl, vp, vp, vp, vp, vp, vp]
            lib.oracle_verify_tree.argtypes = [vp, i32, vp, vp, i64, i64, i64, vp, vp, vp]
            lib.oracle_verify_tree_sample.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64, i64,
                                                      dbl, vp, vp, vp, vp]
            lib.oracle_verify_tree_sample_detail.argtypes = [vp, vp, i32, vp, vp, vp, i64, i64,
                                                             i64, dbl, dbl, vp, vp, vp, vp, vp,
                                                             vp, vp]
            lib.oracle_sample.argtypes = [vp, i32, i64, i64, dbl, vp, vp, vp]
            lib.oracle_topk.argtypes = [vp, i32, i64, i64, i64, vp]
            lib.oracle_tree_mask.argtypes = [vp, i64, i64, vp]
            lib.oracle_round_bf16.argtypes = [vp, i64, vp]
            for f in (lib.oracle_probs, lib.oracle_argmax, lib.oracle_verify_chain,
                      lib.oracle_verify_chain_detail,
                      lib.oracle_verify_tree, lib.oracle_verify_tree_sample,
                      lib.oracle_verify_tree_sample_detail,
                      lib.oracle_sample, lib.oracle_topk,
                      lib.oracle_tree_mask, lib.oracle_round_bf16):
                f.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _logits(a: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint16 if dtype == BF16 else np.float32
    if a.dtype != want:
        raise TypeError(f"logits dtype {a.dtype} does not match dtype flag {dtype}")
    return np.ascontiguousarray(a)


def probs(logits: np.ndarray, dtype: int, temperature: float):
    """[..., V] logits -> float64 probabilities (NaN rows for invalid rows), return code."""
    lg = _logits(logits, dtype)
    V = lg.shape[-1]
    rows = lg.size // V
    out = np.empty(lg.shape, dtype=np.float64)
    rc = _load().oracle_probs(_ptr(lg), dtype, rows, V, float(temperature), _ptr(out))
    return out, rc


def argmax(logits: np.ndarray, dtype: int):
    lg = _logits(logits, dtype)
    V = lg.shape[-1]
    rows = lg.size // V
    out = np.empty(lg.shape[:-1], dtype=np.int32)
    rc = _load().oracle_argmax(_ptr(lg), dtype, rows, V, _ptr(out))
    return out, rc


def verify_chain(target, draft, dtype, tokens, uniforms, temperature):
    """Returns (accept_len [B], out_tokens [B, gamma+1], margin [B], rc)."""
    tg = _logits(target, dtype)
    B, g1, V = tg.shape
    gamma = g1 - 1
    if draft is None:
        dr = None
    else:
        dr = _logits(draft, dtype)
        assert dr.shape == (B, gamma, V)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, gamma)
    uni = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, gamma + 1)
    acc = np.empty(B, dtype=np.int32)
    out = np.empty((B, gamma + 1), dtype=np.int32)
    mg = np.empty(B, dtype=np.float64)
    dptr = _ptr(dr) if dr is not None and dr.size else None
    rc = _load().oracle_verify_chain(_ptr(tg), dptr, dtype, _ptr(tok), _ptr(uni), B, gamma, V,
                                     float(temperature), _ptr(acc), _ptr(out), _ptr(mg))
    return acc, out, mg, rc


def verify_chain_detail(target, draft, dtype, tokens, uniforms, temperature, band=1e-5):
    """Every position of every batch row, as if the step had reached it (see
    oracle_verify_chain_detail). Returns a dict of numpy arrays: accept [B, gamma] (0/1),
    dmargin [B, gamma], tok / cmargin / lo / hi [B, gamma+1], and rc."""
    tg = _logits(target, dtype)
    B, g1, V = tg.shape
    gamma = g1 - 1
    dr = None if draft is None else _logits(draft, dtype)
    if dr is not None:
        assert dr.shape == (B, gamma, V)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, gamma)
    uni = (None if uniforms is None else
           np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, gamma + 1))
    out = dict(accept=np.empty((B, gamma), np.int32), dmargin=np.empty((B, gamma), np.float64),
               tok=np.empty((B, g1), np.int32), cmargin=np.empty((B, g1), np.float64),
               lo=np.empty((B, g1), np.int32), hi=np.empty((B, g1), np.int32))
    dptr = _ptr(dr) if dr is not None and dr.size else None
    rc = _load().oracle_verify_chain_detail(
        _ptr(tg), dptr, dtype, _ptr(tok), _ptr(uni), B, gamma, V, float(temperature),
        float(band), _ptr(out["accept"]), _ptr(out["dmargin"]), _ptr(out["tok"]),
        _ptr(out["cmargin"]), _ptr(out["lo"]), _ptr(out["hi"]))
    out["rc"] = rc
    return out


def verify_tree(target, dtype, parents, tokens):
    """Returns (accept_len [B], path_nodes [B, N], out_tokens [B, N], rc)."""
    tg = _logits(target, dtype)
    B, N, V = tg.shape
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    acc = np.empty(B, dtype=np.int32)
    path = np.empty((B, N), dtype=np.int32)
    out = np.empty((B, N), dtype=np.int32)
    rc = _load().oracle_verify_tree(_ptr(tg), dtype, _ptr(par), _ptr(tok), B, N, V, _ptr(acc),
                                    _ptr(path), _ptr(out))
    return acc, path, out, rc


def verify_tree_sample(target, draft, dtype, parents, tokens, uniforms, temperature):
    """Stochastic tree verify (see oracle_verify_tree_sample). uniforms [B, N]: u[b,0] the final
    draw, u[b,i] node i's acceptance test. Returns (accept_len [B], path_nodes [B, N],
    out_tokens [B, N], margin [B], rc)."""
    tg = _logits(target, dtype)
    B, N, V = tg.shape
    dr = _logits(draft, dtype) if draft is not None else tg
    assert dr.shape == (B, N, V)
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    uni = (np.zeros((B, N), np.float32) if uniforms is None else
           np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, N))
    acc = np.empty(B, dtype=np.int32)
    path = np.empty((B, N), dtype=np.int32)
    out = np.empty((B, N), dtype=np.int32)
    mg = np.empty(B, dtype=np.float64)
    rc = _load().oracle_verify_tree_sample(_ptr(tg), _ptr(dr), dtype, _ptr(par), _ptr(tok),
                                           _ptr(uni), B, N, V, float(temperature), _ptr(acc),
                                           _ptr(path), _ptr(out), _ptr(mg))
    return acc, path, out, mg, rc


def verify_tree_sample_detail(target, draft, dtype, parents, tokens, uniforms, temperature,
                              band=1e-5):
    """The walk with its margins apart: a dict of accept_len, path_nodes, out_tokens, dmargin
    (smallest decision margin), cmargin (the final draw's), lo / hi (the draw's band), rc."""
    tg = _logits(target, dtype)
    B, N, V = tg.shape
    dr = _logits(draft, dtype) if draft is not None else tg
    par = np.ascontiguousarray(parents, dtype=np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, dtype=np.int32).reshape(B, N)
    uni = (np.zeros((B, N), np.float32) if uniforms is None else
           np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, N))
    o = dict(accept_len=np.empty(B, np.int32), path_nodes=np.empty((B, N), np.int32),
             out_tokens=np.empty((B, N), np.int32), dmargin=np.empty(B, np.float64),
             cmargin=np.empty(B, np.float64), lo=np.empty(B, np.int32), hi=np.empty(B, np.int32))
    o["rc"] = _load().oracle_verify_tree_sample_detail(
        _ptr(tg), _ptr(dr), dtype, _ptr(par), _ptr(tok), _ptr(uni), B, N, V, float(temperature),
        float(band), _ptr(o["accept_len"]), _ptr(o["path_nodes"]), _ptr(o["out_tokens"]),
        _ptr(o["dmargin"]), _ptr(o["cmargin"]), _ptr(o["lo"]), _ptr(o["hi"]))
    return o


def sample(logits, dtype, uniforms, temperature):
    """[rows, V] logits -> (tokens [rows] int32, margin [rows] float64, rc)."""
    lg = _logits(logits, dtype)
    V = lg.shape[-1]
    rows = lg.size // V
    uni = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(rows)
    out = np.empty(rows, dtype=np.int32)
    mg = np.empty(rows, dtype=np.float64)
    rc = _load().oracle_sample(_ptr(lg), dtype, rows, V, float(temperature), _ptr(uni),
                               _ptr(out), _ptr(mg))
    return out, mg, rc


def topk(logits, dtype, k):
    """[rows, V] logits -> (indices [rows, k] int32, rc)."""
    lg = _logits(logits, dtype)
    V = lg.shape[-1]
    rows = lg.size // V
    out = np.empty((rows, k), dtype=np.int32)
    rc = _load().oracle_topk(_ptr(lg), dtype, rows, V, int(k), _ptr(out))
    return out, rc


def tree_mask(parents):
    """[B, N] parents -> (words [B, N, ceil(N/32)] uint32, rc)."""
    par = np.ascontiguousarray(parents, dtype=np.int32)
    B, N = par.shape
    W = (N + 31) // 32
    out = np.empty((B, N, W), dtype=np.uint32)
    rc = _load().oracle_tree_mask(_ptr(par), B, N, _ptr(out))
    return out, rc


def round_bf16(x):
    """float64 array -> bf16 bit patterns (uint16) of the nearest bf16 values, ties to even,
    rounded once, straight from double."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    rc = _load().oracle_round_bf16(_ptr(v), v.size, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_round_bf16: {rc}")
    return out


def _widen_bf16(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def lm_head_logits(hidden, head):
    """LM-head logits of the fused producer ("Fast Inference from Transformers via Speculative
    Decoding", pith.science review, "The pith": the target scores every drafted position in
    one parallel pass, whose last layer maps each position's final hidden state to a logit
    per vocabulary token).

    hidden [M, H] and head [V, H] bf16 bit patterns -> (logits [M, V] as bf16 bit patterns,
    the same logits in float64 before rounding): logits[m, v] = sum_k hidden[m, k] head[v, k],
    each product and sum in float64 (a numpy matrix product), then rounded once to bf16."""
    h = _widen_bf16(hidden)
    w = _widen_bf16(head)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise ValueError(f"lm_head_logits: shapes {h.shape} and {w.shape}")
    exact = h @ w.T
    return round_bf16(exact), exact
