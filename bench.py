"""Benchmark of the speculative-decoding verify step on GB300.

Headline (the JSON line's `value`): the largest single-GPU configuration of the workload list,
chain verification of B=256 steps of gamma=8 drafts over V=128256 bf16 logits at T=0.7 (target
N(0, 3^2) plus a Zipf(1.1) log-prior over token ids, draft noise sigma=1). One step = one
spec_verify_chain call over that batch: softmax statistics of all 256 x 17 rows, the
acceptance ballot, the correction / bonus draw and the emitted tokens (two kernels: the stream
kernel over every logit, then the finishing kernel). Metric: verified positions per second,
B * (gamma + 1) per step, and achieved HBM GB/s against the measured copy bandwidth.

Timing: W untimed warm-up steps, then exactly K steps between a barrier and
torch.cuda.synchronize() on both sides, CUDA events on the launching stream, max over ranks.
Each call reads 1.116 GB of logits, more than the L2 size (129 MB), so no input is served from
L2 between steps (two input copies alternate all the same).

`rows`: every configuration of the workload list (and the probability and drafter-side
helpers), each timed independently of --steps: one CUDA graph of at least 10 back-to-back calls
over enough rotated input copies that a buffer is read again only after more than three L2
sizes of other traffic, replayed until at least 50 calls are timed; CUDA events around each
replay; the median per-call time over the replays.

`e2e`: the headline step through the same C entry point with inputs in pinned host memory;
host-to-device copies of the step's inputs and device-to-host copies of its outputs are inside
the timed region (three streams pipeline consecutive steps).

`cpu_baseline` / --impl reference: the CPU oracle (test infrastructure: single-threaded C,
fp64) timed on a bounded sample of the headline's batch rows; the same sample's GPU outputs are
checked against the oracle (the parity tests' per-draw rule) and the result reported.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import platform
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
MARGIN = 1e-5
WORKLOAD = ("chain verify B=256 gamma=8 V=128256 bf16 T=0.7 (target N(0,3^2) - 1.1 ln(k+1), "
            "draft noise sigma=1): workload configuration 3")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--rows", default="all",
                    help="'all', 'none', or a comma list of row names (see ROW_NAMES)")
    ap.add_argument("--min-calls", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-helpers", action="store_true")
    ap.add_argument("--seed-offset", type=int, default=0)
    return ap.parse_args(argv)


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


# ------------------------------------------------------------------ the headline workload

def headline_inputs(seed_offset=0):
    from workloads import chain_128k
    return chain_128k(sigma=1.0) if seed_offset == 0 else chain_128k(seed=3 + 100 * seed_offset,
                                                                    sigma=1.0)


def config_for(world):
    """The JSON line's config: the workload, its batch over all replicas, and how L2 reuse is
    avoided between timed steps."""
    return {"workload": WORKLOAD, "global_batch": world * 256,
            "parallelism": f"replicas{world}" if world > 1 else "single",
            "l2": "each step reads 1.116 GB of logits (> L2 size); two input copies alternate"}


def chain_bytes(B, gamma, V, esz, greedy=False):
    """Algorithmic bytes of a chain call: every logit read once (target rows, and the draft rows
    unless greedy), drafts and uniforms read once, accept_len and out_tokens written once."""
    rows = (gamma + 1) + (0 if greedy else gamma)
    return B * rows * V * esz + 4 * B * gamma + (0 if greedy else 4 * B * (gamma + 1)) + \
        4 * B + 4 * B * (gamma + 1)


def tree_bytes(B, N, V, esz):
    return B * N * V * esz + 8 * B * N + 4 * B * (2 * N + 1)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def measured_tensor_peaks():
    """Dense bf16 tensor throughput (TFLOP/s) of this GPU model from MEASURED_PEAKS.json: the
    burst figure (a cuBLAS GEMM timed alone) and the sustained one (back to back for seconds
    under the power cap); the fallback figures when the file is absent."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"burst": float(d["bf16_tflops"]),
                "sustained": float(d.get("bf16_tflops_sustained", 0.0)) or None,
                "source": "measured (MEASURED_PEAKS.json, cuBLAS bf16 GEMM)"}
    except Exception:
        return {"burst": 1900.0, "sustained": 1700.0, "source": "fallback"}


def kernel_source_hash():
    """Hash of the sources that define the verify kernels and their launches (the C ABI's host
    checks, the static-scratch entry point and the LM-head GEMM's tensor-core helpers do not
    change what those kernels read or write)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_78_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if (f.endswith(".cuh") and f != "spec_tc.cuh") or f == "spec_launch.h" or \
                f.startswith("spec_kernels_"):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(key):
    """dram read+write bytes per call of `key` from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != kernel_source_hash():
            return None
        return d["per_call_bytes"].get(key)
    except Exception:
        return None


def host_info():
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return {"cpu_model": model, "nproc": os.cpu_count(), "machine": platform.machine()}


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
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ calls

class ChainCall:
    """Pre-marshalled spec_verify_chain calls over `ncopies` device copies of one chain input
    (target, draft, tokens, uniforms), each copy with its own outputs and workspace."""

    def __init__(self, lib, sv, inputs, dtype, T, stream, ncopies, device):
        import torch
        tgt, drf, tok, uni = inputs
        B, g1, V = tgt.shape
        self.B, self.gamma, self.V, self.T, self.dtype = B, g1 - 1, V, T, dtype
        self.lib, self.stream = lib, stream
        greedy = T == 0
        vp = ctypes.c_void_p
        sp = vp(stream.cuda_stream)
        self.copies, self.args = [], []
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        for k in range(ncopies):
            c = dict(tgt=tgt if k == 0 else tgt.clone(),
                     drf=drf if (k == 0 or greedy) else drf.clone(), tok=tok, uni=uni,
                     acc=torch.empty(B, dtype=torch.int32, device=device),
                     out=torch.empty((B, g1), dtype=torch.int32, device=device),
                     ws=sv.new_workspace(B, 2 * (g1 - 1) + 1, V, dtype, device))
            self.copies.append(c)
            self.args.append((vp(c["tgt"].data_ptr()),
                              None if greedy or not c["drf"].numel() else vp(c["drf"].data_ptr()),
                              dtype, vp(tok.data_ptr()) if tok.numel() else None,
                              vp(uni.data_ptr()), B, g1 - 1, V, ctypes.c_float(T),
                              vp(c["acc"].data_ptr()), vp(c["out"].data_ptr()),
                              vp(self.status.data_ptr()), vp(c["ws"].data_ptr()),
                              c["ws"].numel(), sp))
        # the copies were made on the current stream; the calls run on `stream`
        torch.cuda.synchronize()

    def __call__(self, k):
        rc = self.lib.spec_verify_chain(*self.args[k % len(self.args)])
        if rc:
            raise RuntimeError(f"spec_verify_chain failed: {rc}")


def copies_for(nbytes):
    """Input copies to rotate over so that a buffer is read again only after more than three
    L2 sizes of other traffic."""
    return max(1, min(128, math.ceil(3 * L2_BYTES / max(1, nbytes)) + 1))


def time_calls(call, ncopies, stream, min_calls=50):
    """Median per-call time (seconds) of `call(k)` over copies k = 0, 1, ...: a CUDA graph of
    L = max(10, ncopies) consecutive calls, replayed until at least min_calls calls were timed,
    CUDA events around each replay on the launching stream. Returns (median, min, max, calls)."""
    import torch
    L = max(10, ncopies)
    with torch.cuda.stream(stream):
        for k in range(ncopies):
            call(k)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for j in range(L):
            call(j % ncopies)
    reps = max(5, math.ceil(min_calls / L))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    with torch.cuda.stream(stream):
        g.replay()                                   # warm
        for e0, e1 in evs:
            e0.record(stream)
            g.replay()
            e1.record(stream)
    torch.cuda.synchronize()
    per = [e0.elapsed_time(e1) * 1e-3 / L for e0, e1 in evs]
    del g
    return statistics.median(per), min(per), max(per), reps * L


# ------------------------------------------------------------------ the per-configuration rows

ROW_NAMES = ("cfg1_chain_tiny", "cfg2_chain_32k", "cfg3_sigma0.25", "cfg3_sigma1", "cfg3_sigma4",
             "cfg4_tree_32k", "cfg5_B1_g3", "cfg5_B1_g7", "cfg5_B16_g3", "cfg5_B16_g7",
             "cfg5_B128_g3", "cfg5_B128_g7", "cfg5_B1024_g3", "cfg5_B1024_g7", "probs_32k",
             "tree_sample_32k", "lmhead_cfg2", "lmhead_cfg3")

# fused LM-head rows: (batch, gamma, V, target hidden size, drafter hidden size, temperature)
LMHEAD_SHAPES = {"lmhead_cfg2": (64, 5, 32000, 4096, 1024, 1.0),
                 "lmhead_cfg3": (256, 8, 128256, 4096, 2048, 0.7)}


def _dev(a, device):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def row_inputs(name, device):
    """(description, chain inputs as device tensors (target, draft, tokens, uniforms), dtype,
    temperature) of a chain row; tree and probs rows are handled by their own callers. The
    large configurations are drawn on the device (workloads.device), the others on the host
    (workloads.synthetic, the generators the parity tests use)."""
    from workloads import BF16, F32, chain_32k, chain_tiny, sweep_152k
    from workloads.device import device_chain
    if name == "cfg1_chain_tiny":
        ci = chain_tiny()
        return ("1000 x 4 x 1000 fp32, T=1 (1000 independent steps, one call)",
                tuple(_dev(a, device) for a in (ci.target, ci.draft, ci.tokens, ci.uniforms)),
                F32, 1.0)
    if name == "cfg2_chain_32k":
        ci = chain_32k()
        return ("64 x 5 x 32000 bf16, T=1",
                tuple(_dev(a, device) for a in (ci.target, ci.draft, ci.tokens, ci.uniforms)),
                BF16, 1.0)
    if name.startswith("cfg3_sigma"):
        sigma = float(name[len("cfg3_sigma"):])
        return (f"256 x 8 x 128256 bf16, T=0.7, sigma={sigma} (drawn on the device)",
                device_chain(256, 8, 128256, BF16, 0.7, 3.0, sigma, zipf_s=1.1,
                             seed=300 + int(100 * sigma), device=device), BF16, 0.7)
    if name.startswith("cfg5_"):
        B, g = (int(x[1:]) for x in name[len("cfg5_"):].split("_"))
        if B <= 16:
            ci = sweep_152k(B=B, gamma=g)
            return (f"{B} x {g} x 152064 fp32, T=1",
                    tuple(_dev(a, device) for a in (ci.target, ci.draft, ci.tokens,
                                                    ci.uniforms)), F32, 1.0)
        return (f"{B} x {g} x 152064 fp32, T=1 (drawn on the device)",
                device_chain(B, g, 152064, F32, 1.0, 2.0, 0.5, seed=500 + 10 * B + g,
                             device=device), F32, 1.0)
    raise KeyError(name)


def lmhead_row(name, lib, sv, device, stream, min_calls):
    """Chain verification with its logits produced by the LM heads: the fused path
    (spec_verify_chain_lmhead: tcgen05 GEMMs whose epilogue emits the softmax partials, then the
    chain finisher) against the unfused one (two cuBLAS bf16 GEMMs through torch.matmul writing
    the logits, then spec_verify_chain reading them), and the two cuBLAS GEMMs alone. Integer-grid
    inputs drawn on the device; the heads (about 1.5 GB at V=128256) exceed L2 many times over,
    so every call reads them from HBM."""
    import torch
    from workloads.device import device_lmhead_grid
    B, g, V, Ht, Hd, T = LMHEAD_SHAPES[name]
    ht, wt, hd, wd, tok, uni = device_lmhead_grid(B, g, V, Ht, Hd, T, seed=900, device=device)
    Mt, Md = B * (g + 1), B * g
    lt = torch.empty((Mt, V), dtype=torch.bfloat16, device=device)
    ld = torch.empty((Md, V), dtype=torch.bfloat16, device=device)
    lt2, ld2 = torch.empty_like(lt), torch.empty_like(ld)
    acc = torch.empty(B, dtype=torch.int32, device=device)
    out = torch.empty((B, g + 1), dtype=torch.int32, device=device)
    acc2, out2 = torch.empty_like(acc), torch.empty_like(out)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    ws = torch.empty(sv.spec_lmhead_workspace_bytes(B, g, V), dtype=torch.uint8, device=device)
    ws2 = sv.new_workspace(B, 2 * g + 1, V, sv.SPEC_BF16, device)
    vp = ctypes.c_void_p
    sp = vp(stream.cuda_stream)
    fused_args = (vp(ht.data_ptr()), vp(wt.data_ptr()), Ht, vp(hd.data_ptr()), vp(wd.data_ptr()),
                  Hd, vp(tok.data_ptr()), vp(uni.data_ptr()), B, g, V, ctypes.c_float(T),
                  vp(lt.data_ptr()), vp(ld.data_ptr()), vp(acc.data_ptr()), vp(out.data_ptr()),
                  vp(st.data_ptr()), vp(ws.data_ptr()), ws.numel(), sp)
    verify_args = (vp(lt2.data_ptr()), vp(ld2.data_ptr()), sv.SPEC_BF16, vp(tok.data_ptr()),
                   vp(uni.data_ptr()), B, g, V, ctypes.c_float(T), vp(acc2.data_ptr()),
                   vp(out2.data_ptr()), vp(st.data_ptr()), vp(ws2.data_ptr()), ws2.numel(), sp)
    torch.cuda.synchronize()

    def fused(k):
        rc = lib.spec_verify_chain_lmhead(*fused_args)
        if rc:
            raise RuntimeError(f"spec_verify_chain_lmhead failed: {rc}")

    def gemms(k):
        torch.matmul(ht, wt.T, out=lt2)
        torch.matmul(hd, wd.T, out=ld2)

    def unfused(k):
        gemms(k)
        rc = lib.spec_verify_chain(*verify_args)
        if rc:
            raise RuntimeError(f"spec_verify_chain failed: {rc}")

    flops = 2.0 * (Mt * Ht + Md * Hd) * V
    peaks = measured_tensor_peaks()
    res = {"shape": (f"B={B} gamma={g} V={V} bf16, target hidden {Ht}, drafter hidden {Hd}, "
                     f"T={T}; integer-grid hidden states and heads drawn on the device"),
           "gemm_flops_per_call": flops,
           "tensor_peak_TFLOPs": peaks}
    for arm, fn in (("fused", fused), ("cublas_gemms_plus_verify", unfused),
                    ("cublas_gemms_only", gemms)):
        med, lo, hi, n = time_calls(fn, 1, stream, min_calls)
        tf = flops / med / 1e12
        res[arm] = {"us_median": med * 1e6, "us_min": lo * 1e6, "us_max": hi * 1e6,
                    "calls_timed": n, "TFLOPs": tf,
                    "frac_of_burst_peak": tf / peaks["burst"] if peaks["burst"] else None,
                    "frac_of_sustained_peak": (tf / peaks["sustained"] if peaks["sustained"]
                                               else None)}
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"{name}: device-side error {int(st.item())}")
    res["fused_logits_equal_cublas"] = bool(torch.equal(lt, lt2) and torch.equal(ld, ld2))
    res["verified_positions_per_call"] = B * (g + 1)
    res["positions_per_s_fused"] = B * (g + 1) / (res["fused"]["us_median"] * 1e-6)
    res["step_stats"] = accept_stats(acc.cpu().numpy(), g)
    return res


def measure_rows(names, lib, sv, device, stream, peak, min_calls):
    import torch
    from workloads import BF16, chain_32k, tree_32k
    rows = {}
    for name in names:
        torch.cuda.nvtx.range_push(f"row {name}")
        if name in LMHEAD_SHAPES:
            rows[name] = lmhead_row(name, lib, sv, device, stream, min_calls)
            torch.cuda.nvtx.range_pop()
            torch.cuda.empty_cache()
            continue
        if name == "cfg4_tree_32k":
            ti = tree_32k()
            nbytes = tree_bytes(ti.B, ti.N, ti.V, 2)
            nc = copies_for(ti.target.nbytes)
            tt = [_dev(ti.target, device) for _ in range(nc)]
            par, tok = _dev(ti.parents, device), _dev(ti.tokens, device)
            acc = torch.empty(ti.B, dtype=torch.int32, device=device)
            path = torch.empty((ti.B, ti.N), dtype=torch.int32, device=device)
            out = torch.empty((ti.B, ti.N), dtype=torch.int32, device=device)
            st = torch.zeros(1, dtype=torch.int32, device=device)
            ws = sv.new_workspace(ti.B, ti.N, ti.V, BF16, device)
            vp = ctypes.c_void_p
            args = [(vp(t.data_ptr()), BF16, vp(par.data_ptr()), vp(tok.data_ptr()), ti.B, ti.N,
                     ti.V, vp(acc.data_ptr()), vp(path.data_ptr()), vp(out.data_ptr()),
                     vp(st.data_ptr()), vp(ws.data_ptr()), ws.numel(),
                     vp(stream.cuda_stream)) for t in tt]
            call = lambda k: lib.spec_verify_tree(*args[k % nc])
            desc, pos = "32 trees x 64 nodes x 32000 bf16, greedy", ti.B * ti.N
            torch.cuda.synchronize()
        elif name == "tree_sample_32k":
            from workloads import tree_sample_32k
            ti = tree_sample_32k()
            # target and draft logits, parents, tokens, uniforms, outputs: each once
            nbytes = (2 * ti.B * ti.N * ti.V * 2 + 8 * ti.B * ti.N + 4 * ti.B * ti.N
                      + 4 * ti.B * (2 * ti.N + 1))
            nc = copies_for(ti.target.nbytes + ti.meta["draft"].nbytes)
            tt = [_dev(ti.target, device) for _ in range(nc)]
            dd = [_dev(ti.meta["draft"], device) for _ in range(nc)]
            par, tok = _dev(ti.parents, device), _dev(ti.tokens, device)
            uu = _dev(ti.meta["uniforms"], device)
            acc = torch.empty(ti.B, dtype=torch.int32, device=device)
            path = torch.empty((ti.B, ti.N), dtype=torch.int32, device=device)
            out = torch.empty((ti.B, ti.N), dtype=torch.int32, device=device)
            st = torch.zeros(1, dtype=torch.int32, device=device)
            ws = sv.new_workspace(ti.B, 2 * ti.N, ti.V, BF16, device)
            vp = ctypes.c_void_p
            args = [(vp(tt[k].data_ptr()), vp(dd[k].data_ptr()), BF16, vp(par.data_ptr()),
                     vp(tok.data_ptr()), vp(uu.data_ptr()), ti.B, ti.N, ti.V,
                     ctypes.c_float(1.0), vp(acc.data_ptr()), vp(path.data_ptr()),
                     vp(out.data_ptr()), vp(st.data_ptr()), vp(ws.data_ptr()), ws.numel(),
                     vp(stream.cuda_stream)) for k in range(nc)]
            call = lambda k: lib.spec_verify_tree_sample(*args[k % nc])
            desc = "32 trees x 64 nodes x 32000 bf16, sampled drafts, T=1 (stochastic walk)"
            pos = ti.B * ti.N
            torch.cuda.synchronize()
        elif name == "probs_32k":
            ci = chain_32k()
            x = ci.target.reshape(-1, ci.V)
            nbytes = x.nbytes + 4 * x.size
            nc = copies_for(nbytes)
            xs = [_dev(x, device) for _ in range(nc)]
            outs = [torch.empty(x.shape, dtype=torch.float32, device=device) for _ in range(nc)]
            st = torch.zeros(1, dtype=torch.int32, device=device)
            ws = sv.new_workspace(x.shape[0], 1, ci.V, BF16, device)
            vp = ctypes.c_void_p
            args = [(vp(xs[k].data_ptr()), BF16, x.shape[0], ci.V, ctypes.c_float(1.0),
                     vp(outs[k].data_ptr()), vp(st.data_ptr()), vp(ws.data_ptr()), ws.numel(),
                     vp(stream.cuda_stream)) for k in range(nc)]
            call = lambda k: lib.spec_probs(*args[k % nc])
            desc, pos = "384 x 32000 bf16 -> fp32 probabilities, T=1", 0
            torch.cuda.synchronize()
        else:
            desc, inputs, dtype, T = row_inputs(name, device)
            B, g1, V = inputs[0].shape
            esz = 2 if dtype == BF16 else 4
            nbytes = chain_bytes(B, g1 - 1, V, esz, greedy=(T == 0))
            nc = copies_for(nbytes)
            call = ChainCall(lib, sv, inputs, dtype, T, stream, nc, device)
            st = call.status
            pos = B * g1
        med, lo, hi, n = time_calls(call, nc, stream, min_calls)
        torch.cuda.synchronize()
        if int(st.item()) != 0:
            raise RuntimeError(f"{name}: device-side error {int(st.item())}")
        gbs = nbytes / med / 1e9
        rows[name] = {"shape": desc, "calls_timed": n, "input_copies": nc,
                      "us_median": med * 1e6, "us_min": lo * 1e6, "us_max": hi * 1e6,
                      "algorithmic_bytes": nbytes, "GBps": gbs, "frac_of_peak": gbs / peak}
        if pos:
            rows[name]["verified_positions_per_call"] = pos
            rows[name]["positions_per_s"] = pos / med
        torch.cuda.nvtx.range_pop()
        del call
        torch.cuda.empty_cache()
    return rows


def helpers(device, peak, stream, min_calls):
    """The drafter-side helpers on configuration 2's data: spec_sample of its 320 draft rows,
    spec_topk (k = 4) of the same rows, spec_tree_mask of configuration 4's 32 trees."""
    import torch
    import speculative_decoding_verification_78_gb300 as sv
    from speculative_decoding_verification_78_gb300 import _binding as B_
    from workloads import chain_32k, make_uniforms, tree_32k
    ci, ti = chain_32k(), tree_32k()
    V = ci.V
    drafts = _dev(ci.draft.reshape(-1, V), device)
    rows = drafts.shape[0]
    nc = copies_for(drafts.numel() * 2)
    copies = [drafts.clone() for _ in range(nc)]
    u = torch.from_numpy(make_uniforms(np.random.default_rng(7), (rows,))).to(device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    tok = torch.empty(rows, dtype=torch.int32, device=device)
    idx = torch.empty((rows, 4), dtype=torch.int32, device=device)
    par = _dev(ti.parents, device)
    mask = torch.empty((ti.B, ti.N, (ti.N + 31) // 32), dtype=torch.int32, device=device)
    ws = sv.new_workspace(rows, 1, V, sv.SPEC_BF16, device)
    ws4 = sv.new_workspace(rows, 4, V, sv.SPEC_BF16, device)
    torch.cuda.synchronize()   # inputs made on the current stream, calls on `stream`
    calls = {
        "sample": (lambda k: B_.spec_sample(copies[k % nc], ci.temperature, u, tok, st, ws,
                                            stream), rows * V * 2 + rows * 8, nc),
        "topk": (lambda k: B_.spec_topk(copies[k % nc], 4, idx, st, ws4, stream),
                 rows * V * 2 + rows * 16, nc),
        "tree_mask": (lambda k: B_.spec_tree_mask(par, mask, st, stream),
                      ti.B * ti.N * 4 + ti.B * ti.N * ((ti.N + 31) // 32) * 4, 1),
    }
    res = {}
    for name, (fn, nbytes, ncop) in calls.items():
        med, lo, hi, n = time_calls(fn, ncop, stream, min_calls)
        res[name] = {"us_median": med * 1e6, "calls_timed": n, "algorithmic_bytes": nbytes,
                     "GBps": nbytes / med / 1e9, "frac_of_peak": nbytes / med / 1e9 / peak}
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "device-side error in the helpers"
    res["shapes"] = {"sample": f"{rows} x {V} bf16, T = {ci.temperature}",
                     "topk": f"{rows} x {V} bf16, k = 4", "tree_mask": f"{ti.B} x {ti.N}"}
    return res


# ------------------------------------------------------------------ our arm

def accept_stats(acc, gamma):
    acc = acc[acc >= 0].astype(np.float64)
    decisions = np.minimum(acc + 1, gamma).sum()
    return {"mean_accept_len": float(acc.mean()),
            "acceptance_rate": float(acc.sum() / decisions) if decisions else None,
            "emitted_tokens_per_step": int((acc + 1).sum())}


def run_ours(args, rank, world, local):
    import torch
    import speculative_decoding_verification_78_gb300 as sv
    from speculative_decoding_verification_78_gb300._binding import load_library
    from workloads import BF16
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    lib = load_library()
    ci = headline_inputs(args.seed_offset + rank)
    stream = torch.cuda.Stream(device)
    inputs = tuple(_dev(a, device) for a in (ci.target, ci.draft, ci.tokens, ci.uniforms))
    head = ChainCall(lib, sv, inputs, BF16, ci.temperature, stream, 2, device)
    K, W = args.steps, args.warmup
    if K < 1 or W < 0:
        raise SystemExit("--steps must be >= 1 and --warmup >= 0")
    peak, peak_kind = measured_peak()

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for i in range(W):
            head(i)
    torch.cuda.synchronize()
    assert int(head.status.item()) == 0, "device-side error in warm-up"
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed steps")
    with torch.cuda.stream(stream):
        t0.record(stream)
        for i in range(K):
            head(i)
        t1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    elapsed = t0.elapsed_time(t1) * 1e-3
    elapsed = max_over_ranks(elapsed, world, device)
    assert int(head.status.item()) == 0, "device-side error in timed steps"

    B, g = ci.B, ci.gamma
    per_call = elapsed / K
    nbytes = chain_bytes(B, g, ci.V, 2)
    achieved = nbytes / per_call / 1e9
    pos_total = sum_over_ranks(B * (g + 1) * K, world, device)
    acc0 = head.copies[0]["acc"].cpu().numpy()
    out0 = head.copies[0]["out"].cpu().numpy()
    k_, grid, cluster = sv.spec_launch_shape(sv.SPEC_CALL_CHAIN, B, 2 * g + 1, ci.V, BF16,
                                             ci.temperature)
    kname = (f"stream_kernel<bf16, chain-sample> + finish_chain_sample<bf16> ({grid} CTAs, "
             f"clusters of {cluster})")
    out = {
        "metric": METRIC, "value": pos_total / elapsed, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": elapsed / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": dict(config_for(world), positions_per_step=B * (g + 1) * world),
        "achieved_GBps": achieved,
        "roofline": {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": (f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)"
                                     if peak_kind == "measured" else "fallback 6.8 TB/s"),
                     "traffic": ncu_traffic("cfg3_sigma1"), "algorithmic_bytes": nbytes,
                     "duration": "average call over the K timed steps (CUDA events)"},
        "gpu_launches": k_ * K,
        "launches_per_step": k_,
        "step_stats": accept_stats(acc0, g),
    }
    names = ([] if args.rows == "none" else list(ROW_NAMES) if args.rows == "all"
             else [n for n in args.rows.split(",") if n])
    if names:
        out["rows"] = measure_rows(names, lib, sv, device, stream, peak, args.min_calls)
    if not args.no_helpers:
        out["helpers"] = helpers(device, peak, stream, args.min_calls)
    out["clocks"] = clocks.stop()
    out["clocks"]["window"] = "warm-up, timed steps and the rows (sampled every 50 ms)"
    if args.e2e_steps > 0:
        out["e2e"] = e2e(lib, ci, head, args.e2e_steps, world, device)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(ci, acc0, out0, budget_s=10.0)
    return out


def e2e(lib, ci, head, steps, world, device):
    """The headline step through the same C entry point with HOST inputs: every step copies its
    inputs from pinned host memory to the device and its outputs back, inside the timed region.
    Three streams pipeline consecutive steps: the host-to-device copies of step i+1 and the
    device-to-host copies of step i-1 overlap the kernels of step i (two device copies of
    inputs, outputs and workspace in rotation)."""
    import torch

    def pin(a):
        a = np.ascontiguousarray(a)
        t = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
             else torch.from_numpy(a))
        return t.pin_memory()

    host_in = dict(tgt=pin(ci.target), drf=pin(ci.draft))
    small = dict(tok=pin(ci.tokens), uni=pin(ci.uniforms))
    c0 = head.copies[0]
    host_out = {k: torch.empty_like(c0[k], device="cpu").pin_memory() for k in ("acc", "out")}
    bi = sum(t.numel() * t.element_size() for t in list(host_in.values()) + list(small.values()))
    bo = sum(t.numel() * t.element_size() for t in host_out.values())
    n = len(head.copies)
    # per copy: its own small inputs too (the headline's copies share tokens and uniforms)
    dsmall = [dict(tok=torch.empty_like(c0["tok"]), uni=torch.empty_like(c0["uni"]))
              for _ in range(n)]
    vp = ctypes.c_void_p
    args = []
    for k, c in enumerate(head.copies):
        a = list(head.args[k])
        a[3] = vp(dsmall[k]["tok"].data_ptr())
        a[4] = vp(dsmall[k]["uni"].data_ptr())
        args.append(tuple(a))
    h2d, d2h, ks = torch.cuda.Stream(), torch.cuda.Stream(), head.stream
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_k = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]

    def one(i):
        k = i % n
        c = head.copies[k]
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_k[k])           # the previous user of copy k has read its inputs
            c["tgt"].copy_(host_in["tgt"], non_blocking=True)
            c["drf"].copy_(host_in["drf"], non_blocking=True)
            dsmall[k]["tok"].copy_(small["tok"], non_blocking=True)
            dsmall[k]["uni"].copy_(small["uni"], non_blocking=True)
            ev_in[k].record(h2d)
        ks.wait_event(ev_in[k])
        ks.wait_event(ev_out[k])              # its previous outputs have been copied out
        rc = lib.spec_verify_chain(*args[k])
        if rc:
            raise RuntimeError(f"verify call failed: {rc}")
        ev_k[k].record(ks)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_k[k])
            for name, t in host_out.items():
                t.copy_(c[name], non_blocking=True)
            ev_out[k].record(d2h)

    for i in range(2 * n):
        one(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(h2d)
    for i in range(steps):
        one(i)
    t1.record(d2h)
    torch.cuda.synchronize()
    el = max_over_ranks(t0.elapsed_time(t1) * 1e-3, world, device)
    pos = sum_over_ranks(ci.B * (ci.gamma + 1) * steps, world, device)
    return {"value": pos / el, "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": steps, "ms_per_step": el / steps * 1e3,
            "pipelined": "h2d / kernels / d2h on three streams, consecutive steps overlap"}


# ------------------------------------------------------------------ the oracle

def oracle_rows(ci, rows):
    """The CPU oracle (single-threaded C, fp64) on batch rows `rows` of the headline input.
    Returns the positions verified."""
    import oracle
    from workloads import BF16
    oracle.verify_chain(ci.target[rows], ci.draft[rows], BF16, ci.tokens[rows],
                        ci.uniforms[rows], ci.temperature)
    return len(rows) * (ci.gamma + 1)


def parity_sample(ci, rows, acc, out):
    """The GPU outputs of batch rows `rows` against the oracle, draw by draw: decisions and
    tokens must be the oracle's, except draws within MARGIN of a boundary, whose outcome must
    lie in the oracle's band. Returns counts."""
    import oracle
    from workloads import BF16
    d = oracle.verify_chain_detail(ci.target[rows], ci.draft[rows], BF16, ci.tokens[rows],
                                   ci.uniforms[rows], ci.temperature, band=MARGIN)
    g = ci.gamma
    exact = flagged = bad = 0
    for j, b in enumerate(rows):
        acc_o = g
        for i in range(g):
            if not d["accept"][j, i]:
                acc_o = i
                break
        n = int(acc[b])
        fl = any(d["dmargin"][j, i] < MARGIN for i in range(min(acc_o + 1, g))) or \
            d["cmargin"][j, acc_o] < MARGIN
        flagged += int(fl)
        same = n == acc_o and int(out[b, n]) == int(d["tok"][j, n]) and \
            np.array_equal(out[b, :n], ci.tokens[b, :n])
        exact += int(same)
        if not same:
            ok = 0 <= n <= g and all(
                (i < n) == bool(d["accept"][j, i]) or d["dmargin"][j, i] < MARGIN
                for i in range(min(n + 1, g)))
            t = int(out[b, n]) if 0 <= n <= g else -1
            ok = ok and (d["tok"][j, n] == t or (d["cmargin"][j, n] < MARGIN and
                                                 d["lo"][j, n] <= t <= d["hi"][j, n]))
            bad += int(not ok)
    return {"rows": len(rows), "equal_to_oracle": exact, "rows_with_flagged_draws": flagged,
            "outside_rule": bad}


def cpu_baseline(ci, acc, out, budget_s=10.0):
    """The oracle as it stands, single-threaded, on rows of the headline batch (8 at a time,
    cycling through the batch) until about budget_s seconds of CPU work; then the GPU outputs of
    the rows it covered are checked against the oracle."""
    rows_done, pos, n = [], 0, 0
    t0 = time.perf_counter()
    while True:
        rows = (np.arange(8) + 8 * n) % ci.B
        pos += oracle_rows(ci, rows)
        rows_done.extend(rows.tolist())
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    chk = sorted(set(rows_done))[:64]
    res = {"value": pos / el, "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{len(rows_done)} batch rows ({n} calls of 8 rows) of the headline batch "
                     f"in {el:.1f} s on one host core, fp64 C oracle",
           "host": host_info()}
    res["parity_sample"] = parity_sample(ci, np.asarray(chk), acc, out)
    return res


def run_reference(args, rank, world):
    if rank != 0:
        return None
    ci = headline_inputs(args.seed_offset)
    t = time.perf_counter()
    oracle_rows(ci, np.arange(2))
    per_row = (time.perf_counter() - t) / 2
    # size each step's row sample so that warm-up + timed steps take about two minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    nr = int(max(1, min(ci.B, round(budget / per_row))))

    def rows(i):
        return (np.arange(nr) + i * nr) % ci.B

    for i in range(args.warmup):
        oracle_rows(ci, rows(i))
    pos = 0
    t0 = time.perf_counter()
    for i in range(args.steps):
        pos += oracle_rows(ci, rows(i + args.warmup))
    el = time.perf_counter() - t0
    value = pos / el
    sample = (f"each step: {nr} of the {ci.B} batch rows of the headline batch, one host core, "
              f"fp64 C oracle")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(config_for(1), positions_per_step=nr * (ci.gamma + 1)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "host": host_info()},
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
