"""Seeded synthetic workloads for the speculative-decoding verify step.

This module draws inputs only: logits, draft tokens, uniforms and candidate trees, as plain
host (numpy) arrays. It holds none of the verify step's arithmetic (no softmax, no acceptance
test, no residual, no inverse CDF); both the CUDA library and the CPU oracle consume the
arrays it returns, so the two sides share data and nothing else.

Workloads (shapes and value distributions follow the workloads the pages evaluate on: a
LLaMA/Vicuna-sized vocabulary of 32000, two larger modern vocabularies, greedy tree drafting
as in Falcon's semi-autoregressive drafter, and a tiny fp32 case):

* ``chain_tiny``      B=1000 independent steps (B=1 each, batched), gamma=4, V=1000, fp32,
                      target ~ N(0, 2^2), draft = target + N(0, 0.5^2), T=1.
* ``chain_32k``       B=64, gamma=5, V=32000, bf16, target ~ N(0, 3^2) with 50 distinct
                      "peaked" ids per (row, position) raised by +8, draft = target + N(0, 1), T=1.
* ``chain_128k``      B=256, gamma=8, V=128256, bf16, target ~ N(0, 3^2) - 1.1 ln(k+1)
                      (a Zipf(1.1) log-prior over token id k), draft = target + N(0, sigma^2)
                      with sigma in {0.25, 1, 4}, T=0.7.
* ``tree_32k``        B=32 rows of a 64-node candidate tree, V=32000, bf16, greedy (T=0).
* ``sweep_152k``      B in {1,16,128,1024} x gamma in {3,7}, V=152064, fp32, target ~ N(0, 2^2),
                      draft = target + N(0, 0.5^2), T=1.

Draft tokens are drawn the way a drafter samples from its own distribution: the Gumbel-max
trick on the draft logits at the verify temperature (argmax of the draft logits at T=0).
This is drafter-side input generation, not part of the verify step.

Uniforms are ``(2k+1) / 2^24`` for k uniform in [0, 2^23): exactly representable in fp32 and
strictly inside (0, 1).

bf16 logits are produced from fp32 by round-to-nearest-even and returned as uint16 bit
patterns; ``bf16_to_f32`` widens them exactly.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = 0
BF16 = 1

__all__ = [
    "F32", "BF16", "ChainInputs", "TreeInputs", "f32_to_bf16", "bf16_to_f32", "as_f32",
    "make_uniforms", "gumbel_draft_tokens", "chain_tiny", "chain_32k", "chain_128k",
    "tree_32k", "tree_sample_32k", "sweep_152k", "tree_shape", "WORKLOADS", "LmHeadInputs",
    "lmhead_grid", "lmhead_grid_scales",
]


# --------------------------------------------------------------------------- encoding

def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even. Inputs are finite
    or +-inf; NaN is never generated here."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def as_f32(arr: np.ndarray, dtype: int) -> np.ndarray:
    """The fp32 values a logits array stands for (bf16 arrays are widened exactly)."""
    return bf16_to_f32(arr) if dtype == BF16 else np.asarray(arr, dtype=np.float32)


def _encode(x: np.ndarray, dtype: int) -> np.ndarray:
    return f32_to_bf16(x) if dtype == BF16 else np.ascontiguousarray(x, dtype=np.float32)


# --------------------------------------------------------------------------- containers

@dataclass
class ChainInputs:
    """Inputs of one batched chain verify call (host arrays).

    target   [B, gamma+1, V]  float32, or uint16 bf16 bit patterns
    draft    [B, gamma, V]    same dtype as target
    tokens   [B, gamma]       int32 draft tokens x_i
    uniforms [B, gamma+1]     float32 in (0,1): u_0..u_{gamma-1} acceptance tests, u_gamma the
                              one uniform of the correction / bonus draw
    """
    name: str
    target: np.ndarray
    draft: np.ndarray
    dtype: int
    tokens: np.ndarray
    uniforms: np.ndarray
    temperature: float
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def gamma(self) -> int:
        return self.target.shape[1] - 1

    @property
    def V(self) -> int:
        return self.target.shape[2]

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


@dataclass
class TreeInputs:
    """Inputs of one batched greedy tree verify call (host arrays).

    target   [B, N, V]  target logits at every tree node (bf16 bits or fp32)
    parents  [B, N]     int32, parents[b,0] = -1, 0 <= parents[b,i] < i
    tokens   [B, N]     int32 node tokens (node 0 is the committed root; its token is unused)
    """
    name: str
    target: np.ndarray
    dtype: int
    parents: np.ndarray
    tokens: np.ndarray
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.target.shape[0]

    @property
    def N(self) -> int:
        return self.target.shape[1]

    @property
    def V(self) -> int:
        return self.target.shape[2]

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


# --------------------------------------------------------------------------- primitives

def _rngs(seed: int, n: int):
    ss = np.random.SeedSequence(seed)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(n)]


def make_uniforms(rng: np.random.Generator, shape) -> np.ndarray:
    k = rng.integers(0, 1 << 23, size=shape, dtype=np.int64)
    return ((2 * k + 1).astype(np.float64) / float(1 << 24)).astype(np.float32)


def gumbel_draft_tokens(rng: np.random.Generator, draft_f32: np.ndarray, temperature: float,
                        block_rows: int = 256) -> np.ndarray:
    """Drafter-side sampling of one token per draft row: x = argmax_k(d[k]/T + G_k) with
    G_k iid standard Gumbel (the Gumbel-max trick), or argmax_k d[k] at T = 0.

    draft_f32: [..., V] fp32 values of the draft logits. Returns int32 [...]."""
    lead = draft_f32.shape[:-1]
    V = draft_f32.shape[-1]
    flat = draft_f32.reshape(-1, V)
    out = np.empty(flat.shape[0], dtype=np.int32)
    for r0 in range(0, flat.shape[0], block_rows):
        blk = flat[r0:r0 + block_rows].astype(np.float32)
        if temperature > 0:
            g = rng.random(blk.shape, dtype=np.float32)
            np.maximum(g, np.float32(1e-30), out=g)
            g = -np.log(-np.log(g))
            blk = blk / np.float32(temperature) + g
        out[r0:r0 + block_rows] = np.argmax(blk, axis=1)
    return out.reshape(lead)


def _normal(rng, shape, sigma):
    return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)


# --------------------------------------------------------------------------- chain workloads

def _chain_from_f32(name, rng_tok, target_f32, draft_f32, dtype, uniforms, temperature, meta):
    target = _encode(target_f32, dtype)
    draft = _encode(draft_f32, dtype)
    tokens = gumbel_draft_tokens(rng_tok, as_f32(draft, dtype), temperature)
    return ChainInputs(name, target, draft, dtype, tokens.astype(np.int32), uniforms,
                       float(temperature), meta)


def chain_tiny(seed: int = 1, B: int = 1000, gamma: int = 4, V: int = 1000) -> ChainInputs:
    """1000 independent B=1 steps, batched: gamma=4, V=1000, fp32, N(0,2^2) target, draft
    noise N(0, 0.5^2), T=1."""
    r_t, r_d, r_tok, r_u = _rngs(seed, 4)
    tgt = _normal(r_t, (B, gamma + 1, V), 2.0)
    drf = tgt[:, :gamma] + _normal(r_d, (B, gamma, V), 0.5)
    u = make_uniforms(r_u, (B, gamma + 1))
    return _chain_from_f32(f"chain_tiny_B{B}_g{gamma}_V{V}_f32", r_tok, tgt, drf, F32, u, 1.0,
                           {"target_sigma": 2.0, "draft_sigma": 0.5})


def chain_32k(seed: int = 2, B: int = 64, gamma: int = 5, V: int = 32000,
              dtype: int = BF16, temperature: float = 1.0, peaked: int = 50,
              boost: float = 8.0) -> ChainInputs:
    """LLaMA-sized vocabulary: N(0,3^2) target with `peaked` distinct ids per (row, position)
    raised by `boost`; draft = target + N(0,1); bf16; T=1."""
    r_t, r_p, r_d, r_tok, r_u = _rngs(seed, 5)
    tgt = _normal(r_t, (B, gamma + 1, V), 3.0)
    npk = min(peaked, V)
    for b in range(B):
        for i in range(gamma + 1):
            ids = r_p.choice(V, size=npk, replace=False)
            tgt[b, i, ids] += np.float32(boost)
    drf = tgt[:, :gamma] + _normal(r_d, (B, gamma, V), 1.0)
    u = make_uniforms(r_u, (B, gamma + 1))
    return _chain_from_f32(f"chain_32k_B{B}_g{gamma}_V{V}", r_tok, tgt, drf, dtype, u,
                           temperature, {"target_sigma": 3.0, "peaked": npk, "boost": boost,
                                         "draft_sigma": 1.0})


def chain_128k(seed: int = 3, sigma: float = 1.0, B: int = 256, gamma: int = 8,
               V: int = 128256, dtype: int = BF16, temperature: float = 0.7,
               block: int = 16) -> ChainInputs:
    """Large vocabulary: N(0,3^2) - 1.1 ln(k+1) target (Zipf(1.1) log-prior over ids),
    draft = target + N(0, sigma^2), bf16, T=0.7. Generated in blocks of batch rows to bound
    host memory."""
    r_t, r_d, r_tok, r_u = _rngs(seed * 1000 + int(round(sigma * 100)), 4)
    prior = (-1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    esz = 2 if dtype == BF16 else 4
    edt = np.uint16 if dtype == BF16 else np.float32
    target = np.empty((B, gamma + 1, V), dtype=edt)
    draft = np.empty((B, gamma, V), dtype=edt)
    tokens = np.empty((B, gamma), dtype=np.int32)
    for b0 in range(0, B, block):
        b1 = min(B, b0 + block)
        t = _normal(r_t, (b1 - b0, gamma + 1, V), 3.0) + prior
        d = t[:, :gamma] + _normal(r_d, (b1 - b0, gamma, V), sigma)
        target[b0:b1] = _encode(t, dtype)
        draft[b0:b1] = _encode(d, dtype)
        tokens[b0:b1] = gumbel_draft_tokens(r_tok, as_f32(draft[b0:b1], dtype), temperature)
    u = make_uniforms(r_u, (B, gamma + 1))
    del esz
    return ChainInputs(f"chain_128k_B{B}_g{gamma}_V{V}_s{sigma}", target, draft, dtype, tokens,
                       u, float(temperature), {"target_sigma": 3.0, "zipf_s": 1.1,
                                               "draft_sigma": sigma})


def sweep_152k(seed: int = 5, B: int = 1, gamma: int = 3, V: int = 152064,
               block: int = 16) -> ChainInputs:
    """Batch/length sweep point: fp32, N(0,2^2) target, draft noise N(0,0.5^2), T=1."""
    r_t, r_d, r_tok, r_u = _rngs(seed * 100000 + B * 10 + gamma, 4)
    target = np.empty((B, gamma + 1, V), dtype=np.float32)
    draft = np.empty((B, gamma, V), dtype=np.float32)
    tokens = np.empty((B, gamma), dtype=np.int32)
    for b0 in range(0, B, block):
        b1 = min(B, b0 + block)
        t = _normal(r_t, (b1 - b0, gamma + 1, V), 2.0)
        target[b0:b1] = t
        draft[b0:b1] = t[:, :gamma] + _normal(r_d, (b1 - b0, gamma, V), 0.5)
        tokens[b0:b1] = gumbel_draft_tokens(r_tok, draft[b0:b1], 1.0)
    u = make_uniforms(r_u, (B, gamma + 1))
    return ChainInputs(f"sweep_152k_B{B}_g{gamma}_V{V}", target, draft, F32, tokens, u, 1.0,
                       {"target_sigma": 2.0, "draft_sigma": 0.5})


# --------------------------------------------------------------------------- tree workload

TREE_BRANCHING = (4, 3, 2, 2, 1, 1)


@dataclass
class LmHeadInputs:
    """Inputs of one fused LM-head + chain verify call (host arrays, bf16 bit patterns).

    hidden_t [B*(gamma+1), Ht]  final hidden states of the target at the gamma+1 positions
    head_t   [V, Ht]            the target's LM head
    hidden_d [B*gamma, Hd]      the drafter's final hidden states at its gamma positions
    head_d   [V, Hd]            the drafter's LM head
    uniforms [B, gamma+1]       float32, as for ChainInputs
    (the draft tokens come from the drafter's own distribution, which needs its logits: the
    caller draws them)
    """
    name: str
    B: int
    gamma: int
    hidden_t: np.ndarray
    head_t: np.ndarray
    hidden_d: np.ndarray
    head_d: np.ndarray
    uniforms: np.ndarray
    temperature: float
    meta: dict = field(default_factory=dict)

    @property
    def V(self) -> int:
        return self.head_t.shape[0]


def lmhead_grid_scales(Ht: int, Hd: int, target_sigma: float = 3.0,
                       draft_sigma: float = 1.0) -> dict:
    """Integer ranges of the LM-head recipe (see lmhead_grid): hidden entries a / 8 with a
    uniform on [-4, 4]; head entries c / 64 with c uniform on [-m, m], m chosen per block of
    columns so that the logits have the requested spread. s = min(Ht, Hd) columns are shared by
    the two models; the rest belong to one model only."""
    s = min(Ht, Hd)
    var_h = 20.0 / 3.0 / 64.0                      # variance of a / 8, a uniform on [-4, 4]

    def m_for(var_logit, cols):
        if cols <= 0:
            return 0
        var_c = var_logit / (cols * var_h)          # variance of c / 64
        return int(min(63, max(1, round(64.0 * np.sqrt(3.0 * var_c)))))

    half = 0.5 * draft_sigma ** 2
    return {"shared": s, "m_shared": m_for(target_sigma ** 2, s),
            "m_target_only": m_for(half, Ht - s), "m_delta": m_for(half, s),
            "m_draft_only": m_for(half, Hd - s)}


def lmhead_grid(seed: int = 8, B: int = 30, gamma: int = 5, V: int = 4096, Ht: int = 640,
                Hd: int = 256, temperature: float = 1.0, target_sigma: float = 3.0,
                draft_sigma: float = 1.0) -> LmHeadInputs:
    """LM-head workload on an integer grid: every hidden entry is a / 8 and every head entry
    c / 64 with small integers a, c, so each logit is an integer multiple of 2^-9 below 2^15 in
    magnitude: every partial sum of its dot product is exact in fp32, in any order, and the
    stored bf16 logit is the correctly rounded exact value whichever way a kernel sums.

    Structure (a drafter that resembles the target): the first s = min(Ht, Hd) hidden
    components of a drafted position are the target's at that position, and the drafter's head
    on them is the target's plus a small integer perturbation; the remaining components are
    each model's own. The target logits spread about N(0, target_sigma^2) (a sum of many small
    products), the draft logits differ from them by about N(0, draft_sigma^2)."""
    r_h, r_w, r_d, r_u = _rngs(seed, 4)
    sc = lmhead_grid_scales(Ht, Hd, target_sigma, draft_sigma)
    s = sc["shared"]
    Mt, Md = B * (gamma + 1), B * gamma

    def ints(rng, shape, m):
        return rng.integers(-m, m + 1, size=shape).astype(np.float32)

    ht = ints(r_h, (Mt, Ht), 4) / 8
    wt = np.empty((V, Ht), np.float32)
    wt[:, :s] = ints(r_w, (V, s), sc["m_shared"]) / 64
    if Ht > s:
        wt[:, s:] = ints(r_w, (V, Ht - s), sc["m_target_only"]) / 64
    rows_t = (np.arange(B)[:, None] * (gamma + 1) + np.arange(gamma)[None, :]).reshape(-1)
    hd = np.empty((Md, Hd), np.float32)
    hd[:, :s] = ht[rows_t, :s]
    if Hd > s:
        hd[:, s:] = ints(r_d, (Md, Hd - s), 4) / 8
    wd = np.empty((V, Hd), np.float32)
    wd[:, :s] = wt[:, :s] + ints(r_d, (V, s), sc["m_delta"]) / 64
    if Hd > s:
        wd[:, s:] = ints(r_d, (V, Hd - s), sc["m_draft_only"]) / 64
    u = make_uniforms(r_u, (B, gamma + 1))
    return LmHeadInputs(f"lmhead_grid_B{B}_g{gamma}_V{V}_Ht{Ht}_Hd{Hd}", B, gamma,
                        f32_to_bf16(ht), f32_to_bf16(wt), f32_to_bf16(hd), f32_to_bf16(wd), u,
                        float(temperature), dict(sc, target_sigma=target_sigma,
                                                 draft_sigma=draft_sigma))


def tree_shape(rng: np.random.Generator, n_nodes: int = 64,
               branching=TREE_BRANCHING) -> np.ndarray:
    """Parents of an n_nodes candidate tree cut from the full tree with the given per-depth
    branching (root at depth 0).

    Falcon's decoding tree gives deeper and wider branches to higher-probability tokens. Here a
    child's sibling rank stands in for its probability rank, and a node's priority is the sum
    of sibling ranks on its root path. The root and the n_nodes-1 lowest-priority nodes are
    kept (ties: shallower first, then a seeded random order), which keeps every kept node's
    parent. Kept nodes are renumbered breadth-first, so parents[i] < i and parents[0] = -1."""
    # full tree, breadth first: (depth, parent_full, rank, priority)
    nodes = [(0, -1, 0, 0)]
    frontier = [0]
    for d, br in enumerate(branching):
        nxt = []
        for p in frontier:
            for r in range(br):
                nodes.append((d + 1, p, r, nodes[p][3] + r))
                nxt.append(len(nodes) - 1)
        frontier = nxt
    n_full = len(nodes)
    n_keep = min(n_nodes, n_full)
    rnd = rng.random(n_full)
    order = sorted(range(1, n_full), key=lambda i: (nodes[i][3], nodes[i][0], rnd[i]))
    keep = [0] + order[: n_keep - 1]
    keep_set = set(keep)
    assert all(nodes[i][1] in keep_set for i in keep if i != 0), "cut is not prefix-closed"
    # renumber breadth first: by depth, then parent's new index, then sibling rank
    new_index = {0: 0}
    by_depth = sorted(keep[1:], key=lambda i: nodes[i][0])
    parents = [-1]
    depth = 1
    while len(new_index) < n_keep:
        level = [i for i in by_depth if nodes[i][0] == depth]
        level.sort(key=lambda i: (new_index[nodes[i][1]], nodes[i][2]))
        for i in level:
            new_index[i] = len(parents)
            parents.append(new_index[nodes[i][1]])
        depth += 1
    return np.asarray(parents, dtype=np.int32)


def tree_32k(seed: int = 4, B: int = 32, N: int = 64, V: int = 32000, dtype: int = BF16,
             p_follow: float = 0.7, peaked: int = 50, tie_offsets=()) -> TreeInputs:
    """Greedy tree verify workload.

    Node logits: N(0,3^2) clipped to +-12 plus +8 on 50 distinct ids, and one designated id
    (the first of the 50) set to 24, strictly above every other logit of that node. The
    designated id is therefore the node's greedy (argmax) token by construction, so this
    module never has to compute an argmax. A node's token is its parent's designated id with
    probability p_follow, otherwise a uniform id in [0, V).

    tie_offsets (positive, increasing): the ids designated + offset get the same value 24, so
    the node's maximum is held by several ids (bf16 ties, e.g. in the same 16-byte vector, the
    same 4 KB unit and later units). The designated id is drawn below V - max(tie_offsets) and is
    the lowest of the tied ids by construction, i.e. still the node's lowest-index argmax."""
    r_shape, r_t, r_p, r_tok = _rngs(seed, 4)
    target_f = np.empty((B, N, V), dtype=np.float32)
    designated = np.empty((B, N), dtype=np.int64)
    parents = np.empty((B, N), dtype=np.int32)
    tokens = np.empty((B, N), dtype=np.int32)
    npk = min(peaked, V)
    for b in range(B):
        parents[b] = tree_shape(r_shape, N)
        t = np.clip(_normal(r_t, (N, V), 3.0), -12.0, 12.0)
        for j in range(N):
            ids = r_p.choice(V, size=npk, replace=False)
            t[j, ids] += np.float32(8.0)
            if tie_offsets:
                d = int(r_p.integers(0, V - int(tie_offsets[-1])))
                for off in (0,) + tuple(tie_offsets):
                    t[j, d + int(off)] = np.float32(24.0)
                designated[b, j] = d
            else:
                t[j, ids[0]] = np.float32(24.0)
                designated[b, j] = ids[0]
        target_f[b] = t
        follow = r_tok.random(N) < p_follow
        rand_tok = r_tok.integers(0, V, size=N)
        for i in range(N):
            if i == 0:
                tokens[b, i] = 0
            else:
                tokens[b, i] = designated[b, parents[b, i]] if follow[i] else rand_tok[i]
    return TreeInputs(f"tree_32k_B{B}_N{N}_V{V}", _encode(target_f, dtype), dtype, parents,
                      tokens, {"p_follow": p_follow, "branching": TREE_BRANCHING,
                               "designated": designated})


def tree_sample_32k(seed: int = 6, B: int = 32, N: int = 64, V: int = 32000, dtype: int = BF16,
                    temperature: float = 1.0, draft_sigma: float = 1.0,
                    peaked: int = 50) -> TreeInputs:
    """Stochastic tree verify workload: configuration 4's trees and target logits (N(0,3^2)
    clipped to +-12, plus 8 on 50 distinct ids per node), a draft row per node (target + N(0,
    draft_sigma^2)), and every node's token drafted from the draft distribution at its parent
    (the Gumbel-max trick at the temperature), so that the children of a node are independent
    draws from it. Uniforms [B, N]: [b, 0] the final draw, [b, i] node i's acceptance test.
    meta["draft"] holds the draft logits (same dtype), meta["uniforms"] the uniforms."""
    r_shape, r_t, r_p, r_d, r_tok, r_u = _rngs(seed, 6)
    target_f = np.empty((B, N, V), dtype=np.float32)
    parents = np.empty((B, N), dtype=np.int32)
    npk = min(peaked, V)
    for b in range(B):
        parents[b] = tree_shape(r_shape, N)
        t = np.clip(_normal(r_t, (N, V), 3.0), -12.0, 12.0)
        for j in range(N):
            ids = r_p.choice(V, size=npk, replace=False)
            t[j, ids] += np.float32(8.0)
        target_f[b] = t
    draft_f = target_f + _normal(r_d, (B, N, V), draft_sigma)
    target = _encode(target_f, dtype)
    draft = _encode(draft_f, dtype)
    dq = as_f32(draft, dtype)
    tokens = np.zeros((B, N), dtype=np.int32)
    for b in range(B):
        # node i's token: one draw from the draft distribution at its parent
        draws = gumbel_draft_tokens(r_tok, dq[b, np.maximum(parents[b], 0)], temperature)
        tokens[b, 1:] = draws[1:]
    u = make_uniforms(r_u, (B, N))
    return TreeInputs(f"tree_sample_B{B}_N{N}_V{V}", target, dtype, parents, tokens,
                      {"draft": draft, "uniforms": u, "temperature": float(temperature),
                       "draft_sigma": draft_sigma, "branching": TREE_BRANCHING})


WORKLOADS = {
    "chain_tiny": chain_tiny,
    "chain_32k": chain_32k,
    "chain_128k": chain_128k,
    "tree_32k": tree_32k,
    "tree_sample_32k": tree_sample_32k,
    "sweep_152k": sweep_152k,
}
