"""Benchmark of the verify step on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  chain verify  B=64, gamma=5, V=32000, bf16, T=1   (softmax statistics, acceptance ballot,
                                                     correction/bonus draw, emit)
  tree verify   B=32 trees of 64 nodes, V=32000, bf16, greedy (argmax, path, bonus)
  probs         the chain's 384 target rows -> fp32 probabilities, T=1
Metric: verified positions per second (chain positions B*(gamma+1) plus tree nodes B*N), and
achieved HBM GB/s against the measured copy bandwidth.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream, max over ranks.
The launches are captured once in CUDA graphs, exactly as the C entry points enqueue them, so
the timed region measures the GPU work rather than Python's launch rate. The K timed steps run
as K // 16 blocks: 16 chain calls, then 16 tree calls, then 16 probs calls (one graph each,
CUDA events between them, which give the per-call durations over the whole timed region), and
the K % 16 remaining steps as whole-step graphs. Inputs rotate over 6 copies, so a buffer is
read again only after more than the L2 size (129 MB) of other traffic.
`e2e` repeats the step through the same C entry points with inputs in pinned host memory:
host-to-device copies of the step's inputs and device-to-host copies of all its outputs are
inside the timed region.

--impl reference times the CPU oracle (test infrastructure, single-threaded C, fp64) on a
bounded row sample of the same workload each step.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified positions/sec and achieved HBM GB/s (% of GB300 peak) on 1 GPU"
UNIT = "positions/s"
L2_BYTES = 129e6
ROT = 6
BLOCK = 16
KINDS = ("chain", "tree", "probs")
WORKLOAD = ("verify step: chain B=64 gamma=5 V=32000 bf16 T=1 + tree B=32 N=64 V=32000 bf16 "
            "greedy + probs 384x32000 bf16->fp32 T=1")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=500)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-helpers", action="store_true")
    ap.add_argument("--seed-offset", type=int, default=0)
    return ap.parse_args()


# ------------------------------------------------------------------ distributed plumbing

def dist_init(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if _cuda_ok() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def _cuda_ok():
    import torch
    return torch.cuda.is_available()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cpu"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world, device="cpu"):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ workload

def make_inputs(seed_offset=0):
    from workloads import chain_32k, tree_32k
    ci = chain_32k(seed=2 + 100 * seed_offset)
    ti = tree_32k(seed=4 + 100 * seed_offset)
    return ci, ti


def config_for(world):
    """The JSON line's config: the workload, its batch over all replicas, and how L2 reuse is
    avoided between timed steps."""
    return {"workload": WORKLOAD, "global_batch": world * (64 + 32),
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": f"inputs rotated over {ROT} copies (> L2 size of traffic between reuses)",
            "order": f"timed steps run as blocks of {BLOCK} calls of each kind"}


def step_bytes(ci, ti):
    """Algorithmic bytes of one step per kernel: every logit read once, small int/fp32 arrays
    read or written once, the probabilities written once."""
    B, g, V = ci.B, ci.gamma, ci.V
    chain = (ci.target.nbytes + ci.draft.nbytes + ci.tokens.nbytes + ci.uniforms.nbytes
             + 4 * B + 4 * B * (g + 1))
    tree = ti.target.nbytes + ti.parents.nbytes + ti.tokens.nbytes + 4 * ti.B * (2 * ti.N + 1)
    probs = ci.target.nbytes + 4 * ci.target.size
    return {"chain": chain, "tree": tree, "probs": probs}


def launch_shapes(ci, ti):
    """Per call of the step: the kernels it launches (from the library's own launch plan)."""
    import speculative_decoding_verification_78_gb300 as sv
    out = {}
    for kind, code, B, rows, V, T, mode in (
            ("chain", sv.SPEC_CALL_CHAIN, ci.B, 2 * ci.gamma + 1, ci.V, ci.temperature,
             "chain-sample"),
            ("tree", sv.SPEC_CALL_TREE, ti.B, ti.N, ti.V, 0.0, "tree"),
            ("probs", sv.SPEC_CALL_PROBS, ci.B * (ci.gamma + 1), 1, ci.V, 1.0, "probs")):
        k, grid, cluster = sv.spec_launch_shape(code, B, rows, V, sv.SPEC_BF16, T)
        shape = f"{grid} CTAs" + (f", clusters of {cluster}" if cluster > 1 else "")
        if k == 1:
            names = f"probs_resident<bf16> ({shape})"
        else:
            fin = {"chain-sample": "finish_chain_sample<bf16>", "tree": "finish_cta<bf16, tree>",
                   "probs": "finish_probs<bf16>"}[mode]
            names = f"stream_kernel<bf16, {mode}> + {fin} ({shape})"
        out[kind] = {"launches": k, "kernels": names}
    return out


def positions(ci, ti):
    return ci.B * (ci.gamma + 1) + ti.B * ti.N


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash():
    """Hash of the sources that define the kernels and their launches (the C ABI's host checks
    and the static-scratch entry point do not change what a kernel reads or writes)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_78_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cuh") or f == "spec_launch.h" or f.startswith("spec_kernels_"):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """dram read+write bytes per launch of `kernel` from the committed ncu summary, if it was
    taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != kernel_source_hash():
            return None
        return d["per_launch_bytes"].get(kernel)
    except Exception:
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        self.path = tempfile.mktemp(suffix=".csv")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm

class Runner:
    """Pre-marshalled C calls of one step on device buffers (copy `k` of each input)."""

    def __init__(self, ci, ti, device):
        import torch
        import speculative_decoding_verification_78_gb300 as sv
        from speculative_decoding_verification_78_gb300._binding import load_library
        self.torch, self.sv = torch, sv
        self.lib = load_library()
        self.ci, self.ti = ci, ti
        dev = device

        def d(a):
            a = np.ascontiguousarray(a)
            if a.dtype == np.uint16:
                return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
            return torch.from_numpy(a).to(dev)

        self.d = d
        self.copies = []
        for _ in range(ROT):
            self.copies.append(dict(ct=d(ci.target), cd=d(ci.draft), tt=d(ti.target)))
        B, g, V = ci.B, ci.gamma, ci.V
        # per input copy: the small inputs and all outputs too, so that copies can overlap
        for c in self.copies:
            c.update(tok=d(ci.tokens), uni=d(ci.uniforms), par=d(ti.parents),
                     ttok=d(ti.tokens),
                     acc=torch.empty(B, dtype=torch.int32, device=dev),
                     out=torch.empty((B, g + 1), dtype=torch.int32, device=dev),
                     tacc=torch.empty(ti.B, dtype=torch.int32, device=dev),
                     tpath=torch.empty((ti.B, ti.N), dtype=torch.int32, device=dev),
                     tout=torch.empty((ti.B, ti.N), dtype=torch.int32, device=dev),
                     probs=torch.empty(ci.target.shape, dtype=torch.float32, device=dev))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        rows = B * (g + 1)
        # one workspace per copy and call: calls of different steps may overlap in e2e
        self.ws_c = [sv.new_workspace(B, 2 * g + 1, V, sv.SPEC_BF16, dev) for _ in range(ROT)]
        self.ws_t = [sv.new_workspace(ti.B, ti.N, ti.V, sv.SPEC_BF16, dev) for _ in range(ROT)]
        self.ws_p = [sv.new_workspace(rows, 1, V, sv.SPEC_BF16, dev) for _ in range(ROT)]
        self.stream = torch.cuda.Stream(dev)
        vp = ctypes.c_void_p
        sp = vp(self.stream.cuda_stream)
        self.args = []
        for k in range(ROT):
            c = self.copies[k]
            # probs reads the target rows of the chain call just made on the same copy
            chain = (vp(c["ct"].data_ptr()), vp(c["cd"].data_ptr()), sv.SPEC_BF16,
                     vp(c["tok"].data_ptr()), vp(c["uni"].data_ptr()), B, g, V,
                     ctypes.c_float(ci.temperature), vp(c["acc"].data_ptr()),
                     vp(c["out"].data_ptr()), vp(self.status.data_ptr()),
                     vp(self.ws_c[k].data_ptr()), self.ws_c[k].numel(), sp)
            tree = (vp(c["tt"].data_ptr()), sv.SPEC_BF16, vp(c["par"].data_ptr()),
                    vp(c["ttok"].data_ptr()), ti.B, ti.N, ti.V, vp(c["tacc"].data_ptr()),
                    vp(c["tpath"].data_ptr()), vp(c["tout"].data_ptr()),
                    vp(self.status.data_ptr()), vp(self.ws_t[k].data_ptr()),
                    self.ws_t[k].numel(), sp)
            probs = (vp(c["ct"].data_ptr()), sv.SPEC_BF16, rows, V, ctypes.c_float(1.0),
                     vp(c["probs"].data_ptr()), vp(self.status.data_ptr()),
                     vp(self.ws_p[k].data_ptr()), self.ws_p[k].numel(), sp)
            self.args.append((chain, tree, probs))

    def call(self, kind, k):
        chain, tree, probs = self.args[k]
        lib = self.lib
        if kind == "chain":
            rc = lib.spec_verify_chain(*chain)
        elif kind == "tree":
            rc = lib.spec_verify_tree(*tree)
        else:
            rc = lib.spec_probs(*probs)
        if rc:
            raise RuntimeError(f"{kind} call failed: {rc}")

    def capture(self):
        """CUDA graphs, captured once, holding the launches exactly as the C entry points
        enqueue them: per input copy k, a whole step (chain, tree and probs calls); and per kind
        of call, BLOCK consecutive calls of that kind over copies 0, 1, ... (mod ROT)."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            for k in range(ROT):
                for kind in KINDS:
                    self.call(kind, k)
        torch.cuda.synchronize()
        self.step_graphs, self.block_graphs = {}, {}
        for k in range(ROT):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for kind in KINDS:
                    self.call(kind, k)
            self.step_graphs[k] = g
        for kind in KINDS:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                for j in range(BLOCK):
                    self.call(kind, j % ROT)
            self.block_graphs[kind] = g
        torch.cuda.synchronize()

    def step(self, i):
        self.step_graphs[i % ROT].replay()


def run_ours(args, rank, world, local):
    import torch
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    ci, ti = make_inputs(args.seed_offset + rank)
    r = Runner(ci, ti, device)
    K = args.steps
    r.capture()
    with torch.cuda.stream(r.stream):
        for i in range(args.warmup):
            r.step(i)
    torch.cuda.synchronize()
    assert int(r.status.item()) == 0, "device-side error in warm-up"

    # K steps of work: K // BLOCK blocks, each the block graph of every kind of call (BLOCK
    # chain calls, then BLOCK tree calls, then BLOCK probs calls, with CUDA events between
    # them), then the K % BLOCK remaining steps as whole-step graphs
    nblk, rem = divmod(K, BLOCK)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KINDS) + 1)]
           for _ in range(nblk)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    host0 = time.perf_counter()
    with torch.cuda.stream(r.stream):
        t0.record(r.stream)
        for b in range(nblk):
            for j, kind in enumerate(KINDS):
                evs[b][j].record(r.stream)
                r.block_graphs[kind].replay()
            evs[b][len(KINDS)].record(r.stream)
        for i in range(rem):
            r.step(i)
        t1.record(r.stream)
    host_issue = time.perf_counter() - host0
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed = t0.elapsed_time(t1) * 1e-3
    elapsed = max_over_ranks(elapsed, world, device)
    assert int(r.status.item()) == 0, "device-side error in timed steps"

    per_kernel = {kind: [e[j].elapsed_time(e[j + 1]) * 1e-3 / BLOCK for e in evs]
                  for j, kind in enumerate(KINDS)}
    if args.steps < BLOCK:
        raise SystemExit(f"--steps must be at least {BLOCK} (one block of each call)")
    avg = {k: float(np.mean(v)) for k, v in per_kernel.items()}
    nbytes = step_bytes(ci, ti)
    peak, peak_kind = measured_peak()
    rows = {}
    for k in ("chain", "tree", "probs"):
        gbs = nbytes[k] / avg[k] / 1e9
        rows[k] = {"us_per_launch": avg[k] * 1e6, "algorithmic_bytes": nbytes[k],
                   "GBps": gbs, "frac_of_peak": gbs / peak}
    rows["chain"]["verified_positions"] = ci.B * (ci.gamma + 1)
    rows["tree"]["verified_positions"] = ti.B * ti.N
    dom = max(("chain", "tree", "probs"), key=lambda k: avg[k])
    shapes = launch_shapes(ci, ti)
    kname = shapes[dom]["kernels"]
    pos_total = sum_over_ranks(positions(ci, ti) * K, world, device)
    value = pos_total / elapsed
    step_total_bytes = sum(nbytes.values())
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": elapsed / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_for(world), positions_per_step=positions(ci, ti) * world),
        "achieved_GBps": step_total_bytes * world * K / elapsed / 1e9 / world,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": rows[dom]["GBps"],
                     "peak": peak, "unit": "GB/s", "frac": rows[dom]["GBps"] / peak,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs copy)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": ncu_traffic(dom), "algorithmic_bytes": nbytes[dom]},
        "rows": rows,
        "gpu_launches": sum(v["launches"] for v in shapes.values()) * K,
        "launch_shapes": shapes,
        "clocks": clk,
        "host_issue_us_per_step": host_issue / K * 1e6,
        "emitted_tokens_per_step": int((r.copies[0]["acc"].cpu().numpy() + 1).sum()),
    }
    out["e2e"] = e2e(r, ci, ti, args.e2e_steps, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(ci, ti, budget_s=10.0)
    if not args.no_helpers:
        out["helpers"] = helpers(ci, ti, device, peak, with_oracle=(rank == 0 and world == 1
                                                                      and not args.no_cpu_baseline))
    return out


def helpers(ci, ti, device, peak, with_oracle):
    """The drafter-side helpers on the same data, outside the step: spec_sample of the chain's
    320 draft rows, spec_topk (k = 4) of the same rows, spec_tree_mask of the 32 trees. Each is
    timed as one CUDA graph of 32 back-to-back calls over 6 rotated input copies (CUDA events
    around it); the oracle's time per call comes from a bounded sample of rows."""
    import torch
    import speculative_decoding_verification_78_gb300 as sv
    from speculative_decoding_verification_78_gb300 import _binding as B_
    V = ci.V
    drafts = torch.from_numpy(ci.draft.reshape(-1, V).view(np.int16)).to(device) \
        .view(torch.bfloat16)
    rows = drafts.shape[0]
    copies = [drafts.clone() for _ in range(ROT)]
    rng = np.random.default_rng(7)
    from workloads import make_uniforms
    u_h = make_uniforms(rng, (rows,))
    u = torch.from_numpy(u_h).to(device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    tok = torch.empty(rows, dtype=torch.int32, device=device)
    idx = torch.empty((rows, 4), dtype=torch.int32, device=device)
    par = torch.from_numpy(ti.parents).to(device)
    mask = torch.empty((ti.B, ti.N, (ti.N + 31) // 32), dtype=torch.int32, device=device)
    ws = sv.new_workspace(rows, 1, V, sv.SPEC_BF16, device)
    ws4 = sv.new_workspace(rows, 4, V, sv.SPEC_BF16, device)
    stream = torch.cuda.Stream(device)
    calls = {
        "sample": (lambda k: B_.spec_sample(copies[k % ROT], ci.temperature, u, tok, st, ws,
                                            stream), rows * V * 2 + rows * 8),
        "topk": (lambda k: B_.spec_topk(copies[k % ROT], 4, idx, st, ws4, stream),
                 rows * V * 2 + rows * 16),
        "tree_mask": (lambda k: B_.spec_tree_mask(par, mask, st, stream),
                      ti.B * ti.N * 4 + ti.B * ti.N * ((ti.N + 31) // 32) * 4),
    }
    res = {}
    for name, (fn, nbytes) in calls.items():
        with torch.cuda.stream(stream):
            for k in range(ROT):
                if fn(k):
                    raise RuntimeError(f"{name} call failed")
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(32):
                fn(k)
        ts = []
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3 / 32)
        t = float(np.median(ts))
        res[name] = {"us_per_call": t * 1e6, "algorithmic_bytes": nbytes,
                     "GBps": nbytes / t / 1e9, "frac_of_peak": nbytes / t / 1e9 / peak}
    assert int(st.item()) == 0, "device-side error in the helpers"
    res["shapes"] = {"sample": f"{rows} x {V} bf16, T = {ci.temperature}",
                     "topk": f"{rows} x {V} bf16, k = 4", "tree_mask": f"{ti.B} x {ti.N}"}
    if with_oracle:
        import oracle
        from workloads import BF16
        dh = ci.draft.reshape(-1, V)
        t0 = time.perf_counter()
        oracle.sample(dh[:32], BF16, u_h[:32], ci.temperature)
        res["sample"]["oracle_us_per_call"] = (time.perf_counter() - t0) / 32 * rows * 1e6
        t0 = time.perf_counter()
        oracle.topk(dh[:8], BF16, 4)
        res["topk"]["oracle_us_per_call"] = (time.perf_counter() - t0) / 8 * rows * 1e6
        t0 = time.perf_counter()
        oracle.tree_mask(ti.parents)
        res["tree_mask"]["oracle_us_per_call"] = (time.perf_counter() - t0) * 1e6
        res["oracle_sample"] = "32 / 8 / 32 rows or trees timed on one host core, scaled"
    return res


def e2e(r, ci, ti, steps, world, device):
    """The step through the same C entry points with HOST inputs: every step copies its inputs
    from pinned host memory to the device and all its outputs back, inside the timed region.
    Three streams pipeline consecutive steps: host-to-device copies of step i+1 and
    device-to-host copies of step i-1 overlap the kernels of step i (each step uses its own
    device copy of inputs, outputs and workspaces, ROT of them in rotation)."""
    import torch
    pin = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
                     if a.dtype == np.uint16 else torch.from_numpy(a)).pin_memory()
    host_in = dict(ct=pin(ci.target), cd=pin(ci.draft), tt=pin(ti.target), tok=pin(ci.tokens),
                   uni=pin(ci.uniforms), par=pin(ti.parents), ttok=pin(ti.tokens))
    c0 = r.copies[0]
    host_out = {k: torch.empty_like(c0[k], device="cpu").pin_memory()
                for k in ("acc", "out", "tacc", "tpath", "tout", "probs")}
    bi = sum(t.numel() * t.element_size() for t in host_in.values())
    bo = sum(t.numel() * t.element_size() for t in host_out.values())
    h2d, d2h, ks = torch.cuda.Stream(), torch.cuda.Stream(), r.stream
    ev_in = [torch.cuda.Event() for _ in range(ROT)]
    ev_k = [torch.cuda.Event() for _ in range(ROT)]
    ev_out = [torch.cuda.Event() for _ in range(ROT)]
    lib = r.lib

    def one(i):
        k = i % ROT
        c = r.copies[k]
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_k[k])           # the previous user of copy k has read its inputs
            for name, t in host_in.items():
                c[name].copy_(t, non_blocking=True)
            ev_in[k].record(h2d)
        ks.wait_event(ev_in[k])
        ks.wait_event(ev_out[k])              # its previous outputs have been copied out
        chain, tree, probs = r.args[k]
        rc = lib.spec_verify_chain(*chain) | lib.spec_verify_tree(*tree) | \
            lib.spec_probs(*probs)
        if rc:
            raise RuntimeError(f"verify call failed: {rc}")
        ev_k[k].record(ks)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_k[k])
            for name, t in host_out.items():
                t.copy_(c[name], non_blocking=True)
            ev_out[k].record(d2h)

    for i in range(2 * ROT):
        one(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d)
    for i in range(steps):
        one(i)
    t1.record(d2h)
    torch.cuda.synchronize()
    el = max_over_ranks(t0.elapsed_time(t1) * 1e-3, world, device)
    pos = sum_over_ranks(positions(ci, ti) * steps, world, device)
    return {"value": pos / el, "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": steps, "ms_per_step": el / steps * 1e3,
            "pipelined": "h2d / kernels / d2h on three streams, consecutive steps overlap"}


# ------------------------------------------------------------------ the oracle

def oracle_step(ci, ti, crow, trow, prow):
    """One bounded sample of the step on the CPU oracle: chain rows crow, tree rows trow, probs
    rows prow (numpy index arrays). Returns the positions verified."""
    import oracle
    from workloads import BF16
    oracle.verify_chain(ci.target[crow], ci.draft[crow], BF16, ci.tokens[crow],
                        ci.uniforms[crow], ci.temperature)
    oracle.verify_tree(ti.target[trow], BF16, ti.parents[trow], ti.tokens[trow])
    flat = ci.target.reshape(-1, ci.V)
    oracle.probs(flat[prow], BF16, 1.0)
    return len(crow) * (ci.gamma + 1) + len(trow) * ti.N


def cpu_baseline(ci, ti, budget_s=10.0):
    """The oracle as it stands, single-threaded, on whole steps of the same workload, repeated
    until about budget_s seconds of CPU work."""
    crow, trow = np.arange(ci.B), np.arange(ti.B)
    prow = np.arange(ci.B * (ci.gamma + 1))
    pos, n = 0, 0
    t0 = time.perf_counter()
    while True:
        pos += oracle_step(ci, ti, crow, trow, prow)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": pos / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} full steps of the same workload (chain 64 rows, tree 32 rows, probs "
                      f"384 rows) in {el:.1f} s on one host core, fp64 C oracle"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    ci, ti = make_inputs(args.seed_offset)
    # size each step's row sample so that warm-up + timed steps take about 2 minutes
    full = time.perf_counter()
    oracle_step(ci, ti, np.arange(4), np.arange(2), np.arange(24))
    t_small = time.perf_counter() - full          # 1/16 of a full step
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    frac = min(1.0, per_step_budget / (16 * t_small))
    nc = max(1, int(round(ci.B * frac)))
    nt = max(1, int(round(ti.B * frac)))
    npb = max(1, int(round(ci.B * (ci.gamma + 1) * frac)))

    def rows(i):
        return ((np.arange(nc) + i * nc) % ci.B, (np.arange(nt) + i * nt) % ti.B,
                (np.arange(npb) + i * npb) % (ci.B * (ci.gamma + 1)))

    for i in range(args.warmup):
        oracle_step(ci, ti, *rows(i))
    pos = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        pos += oracle_step(ci, ti, *rows(i + args.warmup))
    el = time.perf_counter() - t0
    value = pos / el
    sample = (f"each step: {nc}/{ci.B} chain rows, {nt}/{ti.B} tree rows, {npb}/"
              f"{ci.B * (ci.gamma + 1)} probs rows of the same workload, one host core")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(config_for(1), positions_per_step=positions(ci, ti)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out))
        return
    rank, world, local = dist_init(args.gpus)
    out = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
