"""The C ABI without a GPU: the library loads, exports every symbol include/spec_verify.h
declares, sizes workspaces, and rejects bad arguments on the host before touching CUDA."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_78_gb300 import build as b
    b.build()
    import speculative_decoding_verification_78_gb300 as sv
    return sv.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    import speculative_decoding_verification_78_gb300 as sv
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"
    assert sorted(sv.EXPORTS) == names


def test_status_strings(lib):
    import speculative_decoding_verification_78_gb300 as sv
    for code in (sv.SPEC_OK, sv.SPEC_ERR_NULL, sv.SPEC_ERR_SHAPE, sv.SPEC_ERR_TEMP,
                 sv.SPEC_ERR_DTYPE, sv.SPEC_ERR_WORKSPACE, sv.SPEC_ERR_ALIGN, sv.SPEC_ERR_LAUNCH,
                 sv.SPEC_ERR_NONFINITE, sv.SPEC_ERR_TOKEN, sv.SPEC_ERR_PARENT,
                 sv.SPEC_ERR_TIMEOUT, sv.SPEC_ERR_CHECK):
        assert sv.spec_status_string(code) != "unknown status"
    assert sv.spec_status_string(12345) == "unknown status"


def test_launch_failure_reports_cuda_error(lib):
    """With arguments that pass every host check, a call on a machine without a usable device
    fails at launch; the CUDA error behind it is kept for the caller."""
    import torch
    import speculative_decoding_verification_78_gb300 as sv
    if torch.cuda.is_available():
        pytest.skip("a device is present: the launch would run")
    need = sv.spec_workspace_bytes(4, 7, 1000, 1)
    assert _chain(lib, wsb=need) == sv.SPEC_ERR_LAUNCH
    ce = sv.spec_last_cuda_error()
    assert ce != 0
    assert sv.spec_cuda_error_string(ce)
    err = sv.SpecError(sv.SPEC_ERR_LAUNCH, "spec_verify_chain")
    assert f"CUDA error {ce}" in str(err)


def test_workspace_bytes(lib):
    import speculative_decoding_verification_78_gb300 as sv
    a = sv.spec_workspace_bytes(64, 11, 32000, sv.SPEC_BF16)
    b = sv.spec_workspace_bytes(64, 11, 32000, sv.SPEC_F32)
    assert 0 < a < b                      # bf16 rows are half as many units
    assert a % 256 == 0
    assert sv.spec_workspace_bytes(64, 11, 0, sv.SPEC_BF16) == 0
    assert sv.spec_workspace_bytes(64, 11, sv.SPEC_MAX_V + 1, sv.SPEC_BF16) == 0
    assert sv.spec_workspace_bytes(64, 11, 100, 7) == 0
    # grows with the batch and the rows per batch row
    assert sv.spec_workspace_bytes(128, 11, 32000, 1) > a
    assert sv.spec_workspace_bytes(64, 21, 32000, 1) > a


FAKE = 0x100000          # a 256-byte aligned fake device address: never dereferenced here


def _chain(lib, **kw):
    a = dict(t=FAKE, d=FAKE, dtype=1, tok=FAKE, uni=FAKE, B=4, g=3, V=1000, T=1.0, acc=FAKE,
             out=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.spec_verify_chain(vp(a["t"]), vp(a["d"]), a["dtype"], vp(a["tok"]), vp(a["uni"]),
                                 a["B"], a["g"], a["V"], a["T"], vp(a["acc"]), vp(a["out"]),
                                 vp(a["st"]), vp(a["ws"]), a["wsb"], None)


def test_chain_host_validation(lib):
    import speculative_decoding_verification_78_gb300 as sv
    assert _chain(lib, dtype=3) == sv.SPEC_ERR_DTYPE
    assert _chain(lib, V=0) == sv.SPEC_ERR_SHAPE
    assert _chain(lib, V=sv.SPEC_MAX_V + 1) == sv.SPEC_ERR_SHAPE
    assert _chain(lib, g=-1) == sv.SPEC_ERR_SHAPE
    assert _chain(lib, g=sv.SPEC_MAX_GAMMA + 1) == sv.SPEC_ERR_SHAPE
    assert _chain(lib, B=-1) == sv.SPEC_ERR_SHAPE
    assert _chain(lib, T=-1.0) == sv.SPEC_ERR_TEMP
    assert _chain(lib, T=float("nan")) == sv.SPEC_ERR_TEMP
    assert _chain(lib, T=float("inf")) == sv.SPEC_ERR_TEMP
    assert _chain(lib, T=1e-40) == sv.SPEC_ERR_TEMP        # below FLT_MIN
    assert _chain(lib, t=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, d=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, uni=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, tok=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, st=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, ws=0) == sv.SPEC_ERR_NULL
    assert _chain(lib, t=FAKE + 1) == sv.SPEC_ERR_ALIGN     # bf16 needs 2-byte alignment
    assert _chain(lib, dtype=0, t=FAKE + 2) == sv.SPEC_ERR_ALIGN
    assert _chain(lib, ws=FAKE + 8) == sv.SPEC_ERR_ALIGN
    assert _chain(lib, acc=FAKE + 2) == sv.SPEC_ERR_ALIGN
    need = sv.spec_workspace_bytes(4, 7, 1000, 1)
    assert _chain(lib, wsb=need - 1) == sv.SPEC_ERR_WORKSPACE
    # empty batch: nothing to do, nothing launched
    assert _chain(lib, B=0) == sv.SPEC_OK
    # greedy needs neither draft logits nor uniforms; gamma = 0 needs no tokens
    assert _chain(lib, T=0.0, d=0, uni=0, wsb=need - 1) == sv.SPEC_ERR_WORKSPACE
    assert _chain(lib, g=0, tok=0, d=0, wsb=8) == sv.SPEC_ERR_WORKSPACE


def test_tree_and_probs_host_validation(lib):
    import speculative_decoding_verification_78_gb300 as sv
    vp = ctypes.c_void_p

    def tree(**kw):
        a = dict(t=FAKE, dtype=1, par=FAKE, tok=FAKE, B=2, N=64, V=1000, acc=FAKE, path=FAKE,
                 out=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.spec_verify_tree(vp(a["t"]), a["dtype"], vp(a["par"]), vp(a["tok"]), a["B"],
                                    a["N"], a["V"], vp(a["acc"]), vp(a["path"]), vp(a["out"]),
                                    vp(a["st"]), vp(a["ws"]), a["wsb"], None)

    assert tree(N=0) == sv.SPEC_ERR_SHAPE
    assert tree(N=sv.SPEC_MAX_NODES + 1) == sv.SPEC_ERR_SHAPE
    assert tree(par=0) == sv.SPEC_ERR_NULL
    assert tree(path=0) == sv.SPEC_ERR_NULL
    assert tree(dtype=-1) == sv.SPEC_ERR_DTYPE
    assert tree(tok=FAKE + 2) == sv.SPEC_ERR_ALIGN
    assert tree(wsb=100) == sv.SPEC_ERR_WORKSPACE
    assert tree(B=0) == sv.SPEC_OK

    def pr(**kw):
        a = dict(t=FAKE, dtype=0, rows=3, V=100, T=1.0, out=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.spec_probs(vp(a["t"]), a["dtype"], a["rows"], a["V"], a["T"], vp(a["out"]),
                              vp(a["st"]), vp(a["ws"]), a["wsb"], None)

    assert pr(V=0) == sv.SPEC_ERR_SHAPE
    assert pr(rows=-2) == sv.SPEC_ERR_SHAPE
    assert pr(T=-0.5) == sv.SPEC_ERR_TEMP
    assert pr(out=0) == sv.SPEC_ERR_NULL
    assert pr(out=FAKE + 1) == sv.SPEC_ERR_ALIGN
    assert pr(wsb=16) == sv.SPEC_ERR_WORKSPACE
    assert pr(rows=0) == sv.SPEC_OK


def test_lmhead_host_validation(lib):
    """spec_verify_chain_lmhead rejects bad shapes, temperatures, pointers, alignment and short
    workspaces on the host, before any CUDA call."""
    import speculative_decoding_verification_78_gb300 as sv
    vp = ctypes.c_void_p

    def lm(**kw):
        a = dict(ht=FAKE, wt=FAKE, Ht=256, hd=FAKE, wd=FAKE, Hd=128, tok=FAKE, uni=FAKE, B=4,
                 g=3, V=1024, T=1.0, lt=FAKE, ld=FAKE, acc=FAKE, out=FAKE, st=FAKE, ws=FAKE,
                 wsb=1 << 30)
        a.update(kw)
        return lib.spec_verify_chain_lmhead(
            vp(a["ht"]), vp(a["wt"]), a["Ht"], vp(a["hd"]), vp(a["wd"]), a["Hd"], vp(a["tok"]),
            vp(a["uni"]), a["B"], a["g"], a["V"], a["T"], vp(a["lt"]), vp(a["ld"]),
            vp(a["acc"]), vp(a["out"]), vp(a["st"]), vp(a["ws"]), a["wsb"], None)

    assert lm(V=1000) == sv.SPEC_ERR_SHAPE                 # not a multiple of 256
    assert lm(V=0) == sv.SPEC_ERR_SHAPE
    assert lm(V=sv.SPEC_LMHEAD_MAX_V + 256) == sv.SPEC_ERR_SHAPE
    assert lm(Ht=100) == sv.SPEC_ERR_SHAPE                 # not a multiple of 64
    assert lm(Hd=0) == sv.SPEC_ERR_SHAPE
    assert lm(g=0) == sv.SPEC_ERR_SHAPE                    # nothing to verify
    assert lm(g=sv.SPEC_MAX_GAMMA + 1) == sv.SPEC_ERR_SHAPE
    assert lm(B=-1) == sv.SPEC_ERR_SHAPE
    assert lm(T=0.0) == sv.SPEC_ERR_TEMP                   # greedy: spec_verify_chain
    assert lm(T=float("nan")) == sv.SPEC_ERR_TEMP
    for k in ("ht", "wt", "hd", "wd", "tok", "uni", "lt", "ld", "acc", "out", "st", "ws"):
        assert lm(**{k: 0}) == sv.SPEC_ERR_NULL, k
    for k in ("ht", "wt", "hd", "wd", "lt", "ld", "ws"):
        assert lm(**{k: FAKE + 8}) == sv.SPEC_ERR_ALIGN, k   # 16-byte alignment
    assert lm(tok=FAKE + 2) == sv.SPEC_ERR_ALIGN
    need = sv.spec_lmhead_workspace_bytes(4, 3, 1024)
    assert need > 0 and need % 256 == 0
    assert lm(wsb=need - 1) == sv.SPEC_ERR_WORKSPACE
    assert lm(B=0) == sv.SPEC_OK
    assert sv.spec_lmhead_workspace_bytes(4, 3, 1000) == 0
    assert sv.spec_lmhead_workspace_bytes(4, 0, 1024) == 0
    # one partial per 256-column tile: more than the verify step's own workspace
    assert need > sv.spec_workspace_bytes(4, 3, 1024, sv.SPEC_BF16)


def test_selftest_bounded_wait_host_validation(lib):
    """The bounded-wait self-check rejects a NULL or misaligned status and a limit outside
    1e-6 .. 10 s on the host, before any CUDA call."""
    import speculative_decoding_verification_78_gb300 as sv
    vp = ctypes.c_void_p
    f = lib.spec_selftest_bounded_wait
    assert f(None, 0.01, None) == sv.SPEC_ERR_NULL
    assert f(vp(FAKE + 2), 0.01, None) == sv.SPEC_ERR_ALIGN
    for bad in (0.0, -1.0, 1e-7, 10.5, float("nan"), float("inf")):
        assert f(vp(FAKE), bad, None) == sv.SPEC_ERR_SHAPE, bad


def test_helpers_host_validation(lib):
    """spec_sample, spec_topk, spec_tree_mask and spec_verify_chain_static reject bad arguments
    on the host, before anything is enqueued (the fake device addresses are never touched)."""
    import speculative_decoding_verification_78_gb300 as sv
    vp = ctypes.c_void_p

    def sample(**kw):
        a = dict(t=FAKE, dtype=1, rows=5, V=1000, T=1.0, uni=FAKE, out=FAKE, st=FAKE, ws=FAKE,
                 wsb=1 << 30)
        a.update(kw)
        return lib.spec_sample(vp(a["t"]), a["dtype"], a["rows"], a["V"], a["T"], vp(a["uni"]),
                               vp(a["out"]), vp(a["st"]), vp(a["ws"]), a["wsb"], None)

    assert sample(dtype=2) == sv.SPEC_ERR_DTYPE
    assert sample(V=0) == sv.SPEC_ERR_SHAPE
    assert sample(rows=-1) == sv.SPEC_ERR_SHAPE
    assert sample(T=float("nan")) == sv.SPEC_ERR_TEMP
    assert sample(uni=0) == sv.SPEC_ERR_NULL
    assert sample(ws=0) == sv.SPEC_ERR_NULL
    assert sample(t=FAKE + 1) == sv.SPEC_ERR_ALIGN
    assert sample(uni=FAKE + 2) == sv.SPEC_ERR_ALIGN
    assert sample(wsb=8) == sv.SPEC_ERR_WORKSPACE
    assert sample(rows=0) == sv.SPEC_OK
    # greedy sampling needs no uniforms
    assert sample(T=0.0, uni=0, wsb=8) == sv.SPEC_ERR_WORKSPACE

    def topk(**kw):
        a = dict(t=FAKE, dtype=0, rows=5, V=1000, k=4, out=FAKE, st=FAKE, ws=FAKE, wsb=1 << 30)
        a.update(kw)
        return lib.spec_topk(vp(a["t"]), a["dtype"], a["rows"], a["V"], a["k"], vp(a["out"]),
                             vp(a["st"]), vp(a["ws"]), a["wsb"], None)

    assert topk(dtype=5) == sv.SPEC_ERR_DTYPE
    assert topk(k=0) == sv.SPEC_ERR_SHAPE
    assert topk(k=sv.SPEC_MAX_TOPK + 1) == sv.SPEC_ERR_SHAPE
    assert topk(V=3, k=4) == sv.SPEC_ERR_SHAPE           # k > V
    assert topk(out=0) == sv.SPEC_ERR_NULL
    assert topk(t=FAKE + 2) == sv.SPEC_ERR_ALIGN          # fp32 rows need 4-byte alignment
    assert topk(wsb=64) == sv.SPEC_ERR_WORKSPACE
    assert topk(rows=0) == sv.SPEC_OK

    def mask(**kw):
        a = dict(par=FAKE, B=3, N=64, out=FAKE, st=FAKE)
        a.update(kw)
        return lib.spec_tree_mask(vp(a["par"]), a["B"], a["N"], vp(a["out"]), vp(a["st"]), None)

    assert mask(N=0) == sv.SPEC_ERR_SHAPE
    assert mask(N=sv.SPEC_MAX_NODES + 1) == sv.SPEC_ERR_SHAPE
    assert mask(B=-1) == sv.SPEC_ERR_SHAPE
    assert mask(out=0) == sv.SPEC_ERR_NULL
    assert mask(par=FAKE + 2) == sv.SPEC_ERR_ALIGN
    assert mask(B=0) == sv.SPEC_OK

    def static(**kw):
        a = dict(t=FAKE, d=FAKE, dtype=1, tok=FAKE, uni=FAKE, B=4, g=3, V=1000, T=1.0, acc=FAKE,
                 out=FAKE, st=FAKE)
        a.update(kw)
        return lib.spec_verify_chain_static(vp(a["t"]), vp(a["d"]), a["dtype"], vp(a["tok"]),
                                            vp(a["uni"]), a["B"], a["g"], a["V"], a["T"],
                                            vp(a["acc"]), vp(a["out"]), vp(a["st"]), None)

    assert static(dtype=9) == sv.SPEC_ERR_DTYPE
    assert static(g=-1) == sv.SPEC_ERR_SHAPE
    assert static(T=-2.0) == sv.SPEC_ERR_TEMP
    assert static(acc=0) == sv.SPEC_ERR_NULL
    # more scratch than the library's static array holds
    assert static(B=4096, g=8, V=128256) == sv.SPEC_ERR_WORKSPACE
    assert static(B=0) == sv.SPEC_OK


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import speculative_decoding_verification_78_gb300._binding as bnd
    monkeypatch.setattr(bnd, "_lib", None)
    monkeypatch.setattr(bnd, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        bnd.load_library()


def test_launch_shape_host_validation(lib):
    import speculative_decoding_verification_78_gb300 as sv
    k, g, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    ref = (ctypes.byref(k), ctypes.byref(g), ctypes.byref(c))
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 4, 11, 1000, sv.SPEC_F32, 1.0, *ref) == 0
    assert k.value in (1, 2) and g.value >= 1 and c.value >= 1
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 4, 11, 1000, sv.SPEC_F32, 1.0,
                                 None, None, None) == sv.SPEC_ERR_NULL
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 4, 10, 1000, sv.SPEC_F32, 1.0,
                                 *ref) == sv.SPEC_ERR_SHAPE          # rows_per_b must be odd
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 4, 11, 1000, 7, 1.0,
                                 *ref) == sv.SPEC_ERR_DTYPE
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 4, 11, 1000, sv.SPEC_F32, -1.0,
                                 *ref) == sv.SPEC_ERR_TEMP
    assert lib.spec_launch_shape(sv.SPEC_CALL_TREE, 4, sv.SPEC_MAX_NODES + 1, 1000, sv.SPEC_F32,
                                 0.0, *ref) == sv.SPEC_ERR_SHAPE
    assert lib.spec_launch_shape(sv.SPEC_CALL_PROBS, 4, 2, 1000, sv.SPEC_F32, 1.0,
                                 *ref) == sv.SPEC_ERR_SHAPE
    assert lib.spec_launch_shape(sv.SPEC_CALL_PROBS, 4, 1, 1000, sv.SPEC_BF16, 0.0, *ref) == 0
    assert (k.value, g.value, c.value) == (1, 4, 1)      # rows held in registers, one CTA each
    assert lib.spec_launch_shape(sv.SPEC_CALL_PROBS, 4, 1, 70001, sv.SPEC_F32, 1.0, *ref) == 0
    assert (k.value, g.value, c.value) == (1, 20, 5)     # a cluster of 5 CTAs per row
    assert lib.spec_launch_shape(sv.SPEC_CALL_PROBS, 4, 1, 200000, sv.SPEC_F32, 1.0, *ref) == 0
    assert k.value == 2                                  # too long: stream kernel + write pass
    assert lib.spec_launch_shape(9, 4, 1, 1000, sv.SPEC_F32, 1.0, *ref) == sv.SPEC_ERR_SHAPE
    # sampling (a chain without drafts) over multi-unit rows: one warp per row, four per CTA
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 37, 1, 32000, sv.SPEC_BF16, 1.0, *ref) == 0
    assert (k.value, g.value, c.value) == (2, 10, 1)
    # single-unit rows: the one-warp chain finisher, four warps per CTA
    assert lib.spec_launch_shape(sv.SPEC_CALL_CHAIN, 37, 9, 1000, sv.SPEC_F32, 1.0, *ref) == 0
    assert (k.value, g.value, c.value) == (2, 10, 1)


def test_binding_checks_chain_operands(lib):
    """The binding refuses operands whose size or dtype does not match (B, gamma, V) before any
    pointer reaches the library: a short draft tensor would be read past its end, int64 tokens
    or fp64 uniforms would be read as other values. CPU tensors suffice: nothing is launched."""
    import torch
    import speculative_decoding_verification_78_gb300 as sv
    B, g, V = 3, 2, 10
    tgt = torch.zeros((B, g + 1, V), dtype=torch.float32)
    ok = dict(draft_logits=torch.zeros((B, g, V), dtype=torch.float32),
              draft_tokens=torch.zeros((B, g), dtype=torch.int32),
              uniforms=torch.full((B, g + 1), 0.5, dtype=torch.float32),
              accept_len=torch.zeros(B, dtype=torch.int32),
              out_tokens=torch.zeros((B, g + 1), dtype=torch.int32),
              status=torch.zeros(1, dtype=torch.int32))
    bad = [("draft_logits", torch.zeros((B, g - 1, V), dtype=torch.float32), ValueError),
           ("draft_logits", torch.zeros((B, g, V), dtype=torch.bfloat16), TypeError),
           ("draft_tokens", torch.zeros((B, g), dtype=torch.int64), TypeError),
           ("draft_tokens", torch.zeros((B, g + 1), dtype=torch.int32), ValueError),
           ("uniforms", torch.zeros((B, g + 1), dtype=torch.float64), TypeError),
           ("uniforms", torch.zeros((B, g), dtype=torch.float32), ValueError),
           ("accept_len", torch.zeros(B + 1, dtype=torch.int32), ValueError),
           ("out_tokens", torch.zeros((B, g + 1), dtype=torch.int64), TypeError),
           ("status", torch.zeros(2, dtype=torch.int32), ValueError)]
    for name, t, exc in bad:
        args = dict(ok, **{name: t})
        with pytest.raises(exc):
            sv.spec_verify_chain(tgt, args["draft_logits"], args["draft_tokens"],
                                 args["uniforms"], 1.0, args["accept_len"], args["out_tokens"],
                                 args["status"], torch.zeros(16, dtype=torch.uint8))
        with pytest.raises(exc):
            sv.spec_verify_chain_static(tgt, args["draft_logits"], args["draft_tokens"],
                                        args["uniforms"], 1.0, args["accept_len"],
                                        args["out_tokens"], args["status"])
    with pytest.raises(ValueError):
        sv.spec_verify_chain(torch.zeros((B, V), dtype=torch.float32), None, None, None, 0.0,
                             ok["accept_len"], ok["out_tokens"], ok["status"], None)
    # well-formed operands get past the checks (then refused as host tensors by _ptr)
    with pytest.raises(ValueError, match="device tensor"):
        sv.spec_verify_chain(tgt, ok["draft_logits"], ok["draft_tokens"], ok["uniforms"], 1.0,
                             ok["accept_len"], ok["out_tokens"], ok["status"],
                             torch.zeros(16, dtype=torch.uint8))
