"""GPU parity of spec_verify_chain_lmhead: the LM-head GEMMs on the tensor cores with the
softmax reduction in their epilogue, followed by chain verification of the stored logits.

- Integer-grid inputs (workloads.lmhead_grid): every logit is exact in fp32 whatever the
  summation order, so the stored bf16 logits must equal the oracle's correctly rounded ones bit
  for bit, and the verification outputs must match the oracle's chain verification of those
  logits draw by draw (the same per-draw rule as spec_verify_chain's parity).
- Gaussian bf16 inputs: the stored logits lie within the fp32-accumulation bound of the exact
  products, rounded once to bf16.
- Invalid rows (a token outside [0, V), a NaN hidden state) report -1 as in spec_verify_chain.
- The full-size configuration (B=256, gamma=8, V=128256, hidden 4096 / 2048), in the launch
  configuration the benchmark times: sampled logit rows bit-exact, sampled batch rows against
  the oracle.
"""

import numpy as np
import pytest
import torch

from gpu_util import MARGIN, compare_chain, dev
from workloads import (BF16, ChainInputs, bf16_to_f32, f32_to_bf16, gumbel_draft_tokens,
                       lmhead_grid)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verification_78_gb300 as sv
    sv.load_library()


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(hidden_t, head_t, hidden_d, head_d, tokens, uniforms, T):
    import speculative_decoding_verification_78_gb300 as sv
    acc, out, st, lt, ld = sv.verify_chain_lmhead(dev(hidden_t), dev(head_t), dev(hidden_d),
                                                  dev(head_d), dev(tokens), dev(uniforms), T)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), int(st.item()), _bits(lt), _bits(ld)


def _oracle_case(orc, li, seed):
    """The oracle's logits of a grid workload and the drafter's tokens drawn from them."""
    lt, _ = orc.lm_head_logits(li.hidden_t, li.head_t)
    ld, _ = orc.lm_head_logits(li.hidden_d, li.head_d)
    B, g, V = li.B, li.gamma, li.V
    tok = gumbel_draft_tokens(np.random.default_rng(seed), bf16_to_f32(ld).reshape(B, g, V),
                              li.temperature)
    ci = ChainInputs(li.name, lt.reshape(B, g + 1, V), ld.reshape(B, g, V), BF16,
                     tok.astype(np.int32), li.uniforms, li.temperature)
    return ci, lt, ld


# B, gamma, V, Ht, Hd, T: ragged row tiles on both GEMMs and a K ring that wraps (640 / 64 = 10
# blocks over 4 stages); one 256-column half per row (the warp-level finisher) and a one-block K;
# a drafter wider than the target and a last column tile with one half (V / 256 = 9); row tiles
# that end exactly on a tile boundary; gamma at its largest; the largest vocabulary; more tiles
# than clusters with a drafter 16 times narrower (48 target and 32 drafter tiles: the clusters
# one target tile short take every drafter tile, some of them two)
SHAPES = [(30, 5, 4096, 640, 256, 1.0), (1, 1, 256, 64, 64, 0.7), (9, 8, 2304, 128, 320, 1.3),
          (128, 3, 1024, 256, 128, 1.0), (4, 32, 512, 64, 128, 1.0),
          (2, 2, 1 << 19, 64, 64, 0.3),   # the largest vocabulary the call accepts, low T
          (128, 4, 8192, 1024, 64, 1.0),
          (8, 3, 1024, 128, 64, 0.01), (8, 3, 1024, 128, 64, 100.0)]   # extreme temperatures


@pytest.mark.parametrize("B,gamma,V,Ht,Hd,T", SHAPES)
def test_lmhead_grid_exact(orc, B, gamma, V, Ht, Hd, T):
    li = lmhead_grid(seed=B + 7 * gamma, B=B, gamma=gamma, V=V, Ht=Ht, Hd=Hd, temperature=T)
    ci, lt_ref, ld_ref = _oracle_case(orc, li, seed=B)
    acc, out, st, lt, ld = _run(li.hidden_t, li.head_t, li.hidden_d, li.head_d, ci.tokens,
                                ci.uniforms, T)
    assert st == 0
    np.testing.assert_array_equal(lt, lt_ref)
    np.testing.assert_array_equal(ld, ld_ref)
    flagged, differ, oacc = compare_chain(orc, ci, (acc, out, st))
    assert differ <= flagged
    if B >= 30:
        assert 0 < oacc.mean() < gamma     # the grid's drafter is accepted part of the time


def test_lmhead_gaussian_within_accumulation_bound(orc):
    """Inputs off the grid: each stored logit is the exact dot product, summed in fp32 in some
    order and rounded once to bf16. Bound: |stored - exact| <= ulp_bf16(|exact| + e) + e with
    e = H * 2^-23 * sum_k |h_k w_k| (a generous bound on any fp32 summation order); nearly all
    logits equal the correctly rounded exact value."""
    rng = np.random.default_rng(31)
    B, g, V, Ht, Hd = 12, 4, 2048, 512, 192
    ht = f32_to_bf16(rng.standard_normal((B * (g + 1), Ht)).astype(np.float32))
    wt = f32_to_bf16((rng.standard_normal((V, Ht)) * 3 / np.sqrt(Ht)).astype(np.float32))
    hd = f32_to_bf16(rng.standard_normal((B * g, Hd)).astype(np.float32))
    wd = f32_to_bf16((rng.standard_normal((V, Hd)) * 3 / np.sqrt(Hd)).astype(np.float32))
    tok = rng.integers(0, V, (B, g)).astype(np.int32)
    u = np.full((B, g + 1), 0.5, np.float32)
    acc, out, st, lt, ld = _run(ht, wt, hd, wd, tok, u, 1.0)
    assert st == 0
    for h, w, got in ((ht, wt, lt), (hd, wd, ld)):
        bits, exact = orc.lm_head_logits(h, w)
        absdot = np.abs(bf16_to_f32(h).astype(np.float64)) @ np.abs(
            bf16_to_f32(w).astype(np.float64)).T
        e = h.shape[1] * 2.0 ** -23 * absdot
        mag = np.abs(exact) + e
        ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 2.0 ** -126))) - 7)
        err = np.abs(bf16_to_f32(got).astype(np.float64) - exact)
        assert np.all(err <= ulp + e), float(np.max(err - ulp - e))
        assert np.mean(got == bits) > 0.99


def test_lmhead_invalid_rows(orc):
    B, g, V, Ht, Hd = 8, 3, 1024, 128, 128
    li = lmhead_grid(seed=3, B=B, gamma=g, V=V, Ht=Ht, Hd=Hd)
    ci, lt_ref, ld_ref = _oracle_case(orc, li, seed=4)
    ci.tokens[1, 2] = V                 # a token outside the vocabulary
    ci.tokens[5, 0] = -1
    hidden_t = li.hidden_t.copy()
    hidden_t[3 * (g + 1) + 1, 7] = 0x7FC0   # NaN in one target position of batch row 3
    acc, out, st, lt, ld = _run(hidden_t, li.head_t, li.hidden_d, li.head_d, ci.tokens,
                                ci.uniforms, 1.0)
    assert st < 0
    for b in (1, 3, 5):
        assert acc[b] == -1 and np.all(out[b] == -1)
    ok = [b for b in range(B) if b not in (1, 3, 5)]
    compare_chain(orc, ci, (acc, out, st), rows=np.array(ok))


def test_lmhead_full_size(orc):
    """B=256, gamma=8, V=128256, target hidden 4096, drafter hidden 2048 (LLaMA-3-like vocabulary
    and widths), integer-grid inputs drawn on the device: 48 sampled logit rows of each GEMM
    bit-exact against the oracle, 6 sampled batch rows verified against the oracle draw by
    draw."""
    import speculative_decoding_verification_78_gb300 as sv
    from workloads.device import device_lmhead_grid
    B, g, V, Ht, Hd, T = 256, 8, 128256, 4096, 2048, 0.7
    ht, wt, hd, wd, tok, uni = device_lmhead_grid(B, g, V, Ht, Hd, T, seed=5)
    acc, out, st, lt, ld = sv.verify_chain_lmhead(ht, wt, hd, wd, tok, uni, T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rng = np.random.default_rng(12)
    h_t, w_t, h_d, w_d = _bits(ht), _bits(wt), _bits(hd), _bits(wd)
    for h, w, got in ((h_t, w_t, lt), (h_d, w_d, ld)):
        rows = np.sort(rng.choice(h.shape[0], 48, replace=False))
        want, _ = orc.lm_head_logits(h[rows], w)
        np.testing.assert_array_equal(_bits(got[torch.as_tensor(rows, device=got.device)]), want)
    sel = np.sort(rng.choice(B, 6, replace=False))
    rt = (sel[:, None] * (g + 1) + np.arange(g + 1)[None, :]).reshape(-1)
    rd = (sel[:, None] * g + np.arange(g)[None, :]).reshape(-1)
    lt_ref, _ = orc.lm_head_logits(h_t[rt], w_t)
    ld_ref, _ = orc.lm_head_logits(h_d[rd], w_d)
    ci = ChainInputs("lmhead_full_sampled", lt_ref.reshape(len(sel), g + 1, V),
                     ld_ref.reshape(len(sel), g, V), BF16, tok.cpu().numpy()[sel],
                     uni.cpu().numpy()[sel], T)
    compare_chain(orc, ci, (acc.cpu().numpy()[sel], out.cpu().numpy()[sel], 0))


def test_lmhead_after_large_tree_sample_on_one_stream():
    """The GEMM (193 KB of shared memory per CTA) launched right after the stochastic-tree
    finisher at its largest shared-memory size (N = 1024 nodes, V = 600064: the limit raised past
    the default), and the other way round, on one stream: every call launches and succeeds."""
    import speculative_decoding_verification_78_gb300 as sv
    from workloads import tree_shape
    rng = np.random.default_rng(41)
    B, N, V = 1, 1024, 600064
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    tgt = (torch.randn((B, N, V), generator=g, device="cuda") * 2).to(torch.bfloat16)
    drf = (tgt.float() + torch.randn((B, N, V), generator=g, device="cuda")).to(torch.bfloat16)
    par = torch.from_numpy(tree_shape(rng, N, branching=(4, 4, 4, 4, 4, 4))[None]).cuda()
    tok = torch.randint(0, V, (B, N), generator=g, device="cuda", dtype=torch.int32)
    uni = torch.rand((B, N), generator=g, device="cuda").clamp_(1e-6, 1 - 1e-6)
    li = lmhead_grid(seed=2, B=8, gamma=3, V=1024, Ht=128, Hd=64)
    toks = torch.from_numpy(rng.integers(0, 1024, (8, 3)).astype(np.int32)).cuda()
    unis = torch.from_numpy(li.uniforms).cuda()
    for _ in range(2):
        acc, path, out, st = sv.verify_tree_sample(tgt, drf, par, tok, uni, 1.0)
        r = sv.verify_chain_lmhead(dev(li.hidden_t), dev(li.head_t), dev(li.hidden_d),
                                   dev(li.head_d), toks, unis, 1.0)
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and int(acc[0].item()) >= 0
        assert int(r[2].item()) == 0


def test_bounded_waits_give_up_and_report(orc):
    """The kernel's waits end: waiting (through the GEMM's own wait routines) on barriers nothing
    arrives on gives up after the limit, writes SPEC_ERR_TIMEOUT, and the kernel returns; the
    context stays usable (an LM-head call right after succeeds and matches the oracle's logits)."""
    import time
    import speculative_decoding_verification_78_gb300 as sv
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert sv.spec_selftest_bounded_wait(st, 0.02) == sv.SPEC_OK
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == sv.SPEC_ERR_TIMEOUT
    assert 0.02 <= dt < 5.0, dt      # two waits of 20 ms in the even CTA
    li = lmhead_grid(seed=9, B=4, gamma=2, V=512, Ht=128, Hd=64)
    tok = np.random.default_rng(9).integers(0, 512, (4, 2)).astype(np.int32)
    acc, out, st2, lt, ld = _run(li.hidden_t, li.head_t, li.hidden_d, li.head_d, tok,
                                 li.uniforms, 1.0)
    assert st2 == 0
    np.testing.assert_array_equal(lt, orc.lm_head_logits(li.hidden_t, li.head_t)[0])
    np.testing.assert_array_equal(ld, orc.lm_head_logits(li.hidden_d, li.head_d)[0])

