#!/usr/bin/env python
"""Benchmark of the W12 tree-verify pass on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
best-first tree build from a drafter lattice, every W12 linear of the layer,
the W12 LM head with per-row argmax, and greedy acceptance.  The headline
metric is the effective W12 weight-stream bandwidth of the step (W12 bytes
read per step / step time, GB/s), reported with the step time in
microseconds and as a fraction of the HBM roofline.

Default workload: 64 stacked 27B-like decoder layers (QKV 5120->7168, O
5120->5120, gate/up 5120->34816, down 17408->5120; 4 distinct weight sets,
each layer streaming its own copy) + LM head 5120x151936 in W12 (32.9 GB
resident), one request, a 32-row tree from a top-16 x 16-position lattice.
After the headline, the same step is timed at 1, 8, 32, 64, 128 and 192
rows (one request) and at 192 rows from 24 requests, each next to dense BF16
cuBLAS on the same shapes.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--rows R] [--impl reference]

Multi-GPU (torchrun): the pass has no exchange step at this scope, so N GPUs
run N independent replicas (weak scaling); value = all ranks' bytes / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify-step µs and W12 weight-stream HBM GB/s (% of GB300 peak) vs tree rows"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

DESCRIPTIONS = {
    "tiny": "1 linear 512->1024 + head 512x4096 (1% x64 outliers, 1% zeros), 8-row chain over 8 positions",
    "single_27b": "one 27B-like layer (QKV 5120->7168, O 5120->5120, gate/up 5120->34816, down 17408->5120) "
                  "+ LM head 5120x151936, W12; 1 request, 32-node tree from top-16 x 16 positions",
    "batched_27b": "same shapes; 24 requests sharing a 192-node budget, 16/12/8 positions",
    "b4_tree": "4B-like layer (2560->3584, 2560->2560, 2560->19456, 9728->2560) + head 2560x151936; "
               "32 requests, 256-node budget, trees",
    "b4_chain": "4B-like layer + head; 32 requests, 256-node budget, chains",
    "full_depth_27b": "64 stacked 27B-like layers (QKV 5120->7168, O 5120->5120, gate/up 5120->34816, "
                      "down 17408->5120) + LM head 5120x151936, W12 (32.9 GB resident); 1 request, "
                      "32-node tree from top-16 x 16 positions",
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# replicas: one process per GPU, no exchange on the data path
# ---------------------------------------------------------------------------

def replica_env():
    """(world, rank, local_rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_replicas(world: int, backend: str):
    """Process group for the barrier and the max over ranks only (None at N=1)."""
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend)
    return dist


def max_over_ranks(value: float, dist, device) -> float:
    """The slowest rank's figure (every rank gets it)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_step: float, ms_per_step: float) -> float:
    """Weak scaling: every replica streams its own copy of the step's bytes."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("k_gemm.cu", "k_gemm_tc.cu", "w12_device.cuh", "w12_abi.cpp"):
        with open(os.path.join(ROOT, "speculative_decoding_tree_w12_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(gemms):
    """DRAM bytes (read + written) of a step's GEMM launches from a committed
    ncu capture, if it was taken on the current kernel source: `gemms` lists
    the step's launches as (n, k, rows); every one must have a captured
    launch of the same shape and rows (stacked layers reuse one layer's
    capture: same kernel, shape and rows, so the same traffic)."""
    p = os.path.join(ROOT, "profiles", "w12_gemm_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != kernel_source_hash():
            return None
        per = {(l["n"], l["k"], l["rows"]): l["dram_read_bytes"] + l["dram_write_bytes"] for l in d["launches"]}
        return int(sum(per[g] for g in gemms))
    except Exception:
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = tempfile.mktemp(prefix="w12clk", suffix=".csv")
        self.gpu = gpu_index

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

class Workload:
    def __init__(self, name, rows, device, seed=0, share=None, one_request=False, variant=None):
        """`share`: another Workload of the same name whose packed device
        weights are reused (only the tree, its rows and the activations are
        rebuilt for the new node budget).  `one_request`: a single request
        drafting 16 positions (the rows of one best-first tree).  `variant`:
        other request/lattice fields of the workload replaced."""
        import torch
        import speculative_decoding_tree_w12_gb300 as w12
        from speculative_decoding_tree_w12_gb300 import synth

        self.w12, self.torch, self.synth = w12, torch, synth
        w = synth.WORKLOADS[name]
        if one_request:
            w = synth.scaled(w, n_req=1, positions=(16,))
        if variant:
            w = synth.scaled(w, **variant)
        if rows:
            w = synth.scaled(w, budget=int(rows))
        self.wl, self.name, self.device = w, name, device
        t0 = time.time()
        self.lat = synth.lattice(w, seed)
        if share is not None:
            self.lin_bits, self.lin, self.lin_hp = share.lin_bits, share.lin, share.lin_hp
            self.head_bits, self.head_hp, self.head = share.head_bits, share.head_hp, share.head
            self.head_n2 = share.head_n2
            self._rows(seed)
            return
        # weights: generate, pack on the host (library packer, self-checked), upload
        self.lin_bits, self.lin = [], []
        distinct = {}
        for layer in range(w.layers):
            for i, (n, k) in enumerate(w.linears):
                # stacked layers reuse 4 distinct weight sets (each layer still
                # streams its own copy from HBM)
                key = (layer % 4, i)
                if key not in distinct:
                    bits = synth.weights(n, k, seed, synth.STREAM_LINEAR + 100 * (layer % 4) + i,
                                         w.outlier_frac, w.zero_frac)
                    distinct[key] = (bits, w12.w12_pack(bits))
                    if layer == 0:
                        self.lin_bits.append(bits)
                bits, hp = distinct[key]
                self.lin.append(w12.DeviceWeight(hp, device))
        self.head_bits = synth.weights(w.vocab, w.hidden, seed, synth.STREAM_HEAD, w.outlier_frac, w.zero_frac)
        self.head_hp = w12.w12_pack(self.head_bits)
        self.head = w12.DeviceWeight(self.head_hp, device)
        self.lin_hp = [distinct[(0, i)][1] for i in range(len(w.linears))]
        log(f"[bench] weights generated and packed in {time.time() - t0:.1f}s")
        self._rows(seed)

    def _rows(self, seed):
        torch, w12, synth, w, device = self.torch, self.w12, self.synth, self.wl, self.device
        # tree (GPU), then the toy target's hidden rows for that tree
        self.dlat = w12.DeviceLattice(self.lat, device)
        max_n = max(n for n, _ in w.linears)
        self.ws = w12.Workspace(min(w.budget, 256), max_n, w.vocab, w.n_req, device)
        self.tree = w12.w12_tree_build(self.dlat, w.budget, self.ws)
        torch.cuda.synchronize()
        self.R = self.tree.R
        th = self.tree.host()
        if getattr(self, "head_n2", None) is None:
            self.head_n2 = synth.head_norms(self.head_bits)
        self.h_bits = synth.hidden_rows(th["req"], th["parent"], th["token"], self.lat.truth, self.head_bits, seed,
                                        head_norm2=self.head_n2)
        self.x_bits = [synth.activations(self.R, k, seed, synth.STREAM_X + i) for i, (n, k) in enumerate(w.linears)]
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
        self.h = dev(self.h_bits)
        xs_layer = [dev(x) for x in self.x_bits]
        self.xs = [xs_layer[j % len(w.linears)] for j in range(len(self.lin))]
        self.ys = [torch.empty((self.R, dw.n), dtype=torch.bfloat16, device=device) for dw in self.lin]
        self.argmax = torch.empty(self.R, dtype=torch.int32, device=device)
        self.acc_tok = torch.empty((w.n_req, w.p_max + 1), dtype=torch.int32, device=device)
        self.acc_len = torch.empty(w.n_req, dtype=torch.int32, device=device)
        self.step_args = w12.VerifyStep(self.lin, self.xs, self.ys, self.head, self.h, self.argmax)

    # bytes ---------------------------------------------------------------
    def w12_bytes(self):
        return sum(d.nbytes for d in self.lin) + self.head.nbytes

    def launch_bytes(self, launches_per_weight):
        """Algorithmic bytes of each GEMM launch of a step, in launch order:
        W12 record/base/escape bytes + activations in + outputs out (a weight
        split into row slices is streamed once per slice)."""
        R = self.R
        out = []
        slices = launches_per_weight
        for d in self.lin:
            for s in range(slices):
                r = R if slices == 1 else min(64, R - 64 * s)
                out.append(d.nbytes + r * d.k * 2 + r * d.n * 2)
        for s in range(slices):
            r = R if slices == 1 else min(64, R - 64 * s)
            out.append(self.head.nbytes + r * self.head.k * 2 + r * (self.head.n // 128) * 8)
        return out

    def gpu_launches_per_step(self, launches_per_weight):
        return 1 + launches_per_weight * (len(self.lin) + 1) + 2

    def gemm_shapes(self):
        """The step's GEMM launches as (n, k, rows), one row slice per launch
        where the library splits a weight into slices of 64 rows."""
        return [(d.n, d.k, self.R) for d in self.lin] + [(self.head.n, self.head.k, self.R)]

    # the step ------------------------------------------------------------
    def step(self):
        w, w12 = self.wl, self.w12
        w12.w12_tree_build(self.dlat, w.budget, self.ws, self.tree)
        w12.w12_verify_step(self.step_args, self.tree, w.n_req, w.p_max, self.ws, self.acc_tok, self.acc_len)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------

def oracle_sample_runner(wk: Workload, frac: float, nthreads: int = 0):
    """A callable that runs the oracle over the first `frac` of every weight's
    output channels (multiples of 128, all rows): W12 decode (oracle unpack),
    FP64 GEMM for the linears, FP64 logits + argmax for the head, then the
    tree build and acceptance.  The linears are one layer's: stacked layers
    repeat the same shapes, so bytes per second carry over.  `nthreads`: the
    oracle's worker threads (0: one per core).  Returns (callable, sampled W12
    bytes, text)."""
    import oracle
    jobs = []
    total = 0
    w = wk.wl
    for bits, x in zip(wk.lin_bits, wk.x_bits):
        n = max(128, int(bits.shape[0] * frac) // 128 * 128)
        p = oracle.w12_pack(bits[:n])
        jobs.append(("lin", p, x))
        total += p.bytes
    nh = max(128, int(wk.head_bits.shape[0] * frac) // 128 * 128)
    ph = oracle.w12_pack(wk.head_bits[:nh])
    jobs.append(("head", ph, wk.h_bits))
    total += ph.bytes

    def run():
        for kind, p, x in jobs:
            wdec = oracle.w12_unpack(p)
            if kind == "lin":
                oracle.gemm_f64(x, wdec, nthreads=nthreads)
            else:
                am, _, _ = oracle.head_argmax(x, wdec, nthreads=nthreads)
        t = oracle.tree_build(wk.lat, w.budget)
        oracle.tree_accept(t, np.resize(am, t.R), w.n_req, w.p_max)

    text = (f"first {frac:.4f} of the output channels of one layer's linears and of the LM head "
            f"({total / 1e6:.1f} MB of W12), all {wk.R} rows; decode + FP64 GEMM/argmax + tree build + accept")
    return run, total, text


def cpu_baseline(wk: Workload, target_s=10.0):
    import oracle
    oracle.build()
    run, b0, _ = oracle_sample_runner(wk, 1.0 / 64)
    t = time.time()
    run()
    dt = max(time.time() - t, 1e-3)
    frac = min(1.0, (1.0 / 64) * target_s / dt)
    run, b, text = oracle_sample_runner(wk, frac)
    t = time.time()
    n = 0
    while True:                      # whole passes until about target_s of CPU work
        run()
        n += 1
        dt = time.time() - t
        if dt >= 0.8 * target_s or n >= 8:
            break
    cores = os.cpu_count() or 1
    out = {"value": n * b / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": f"{text}; {n} pass(es)", "seconds": round(dt, 2)}
    # the same oracle on one core, over a quarter of that sample
    run1, b1, text1 = oracle_sample_runner(wk, max(1.0 / 512, frac / 4), nthreads=1)
    t = time.time()
    run1()
    dt1 = max(time.time() - t, 1e-3)
    out["one_core"] = {"value": b1 / dt1 / 1e9, "unit": "GB/s", "cores": 1, "sample": f"{text1}; 1 pass",
                       "seconds": round(dt1, 2)}
    return out


# ---------------------------------------------------------------------------
# the reference arm: the oracle timed as it stands
# ---------------------------------------------------------------------------

def run_reference(args):
    _, rank, _ = replica_env()
    if rank != 0:
        return 0
    from speculative_decoding_tree_w12_gb300 import synth
    import oracle
    oracle.build()

    class HostOnly:
        pass

    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = synth.scaled(w, budget=args.rows)
    wk = HostOnly()
    wk.wl = w
    wk.lat = synth.lattice(w, 0)
    frac = 1.0 / 32
    # sampled weights only (the reference arm never touches the GPU)
    wk.lin_bits = []
    for i, (n, k) in enumerate(w.linears):
        nn = max(128, int(n * frac) // 128 * 128)
        wk.lin_bits.append(synth.weights(n, k, 0, synth.STREAM_LINEAR + i, w.outlier_frac, w.zero_frac)[:nn])
    t = oracle.tree_build(wk.lat, w.budget)
    wk.R = t.R
    wk.head_bits = synth.weights(w.vocab, w.hidden, 0, synth.STREAM_HEAD, w.outlier_frac, w.zero_frac)
    wk.h_bits = synth.hidden_rows(t.req, t.parent, t.token, wk.lat.truth, wk.head_bits, 0)
    nh = max(128, int(w.vocab * frac) // 128 * 128)
    wk.head_bits = wk.head_bits[:nh]
    wk.x_bits = [synth.activations(t.R, k, 0, synth.STREAM_X + i) for i, (n, k) in enumerate(w.linears)]
    run, nbytes, text = oracle_sample_runner(wk, 1.0)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.time()
        run()
        times.append(time.time() - t0)
    total = sum(times)
    value = nbytes * args.steps / total / 1e9
    cores = os.cpu_count() or 1
    text = text.replace("first 1.0000 of the output channels", f"first {frac:.4f} of the output channels")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}", "rows": int(t.R),
                       "sample": f"each step: the oracle over the first {frac:.4f} of the output channels of one "
                                 "layer's linears and of the LM head (stacked layers repeat the same shapes), all "
                                 "rows, plus tree build and acceptance; GB/s of the sampled W12 bytes",
                       "same_config": False},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": text},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# quick pass (view planes only)
# ---------------------------------------------------------------------------

def quick_pass(wk: "Workload", K: int, W: int):
    """The same step read through the quick pass (w12_verify_step_q: the 8 KB
    view plane of every record, low mantissa bits at the midpoint):
    graph-timed pass (tree build, every linear, the head, the argmax
    reduction and acceptance, as the exact step), the head launch alone, and
    the top-1 agreement of the quick argmax with the exact one on the step's
    rows."""
    import torch
    w12 = wk.w12
    qs = [torch.empty_like(y) for y in wk.ys]
    qam = torch.empty_like(wk.argmax)
    qstep_args = w12.VerifyStep(wk.lin, wk.xs, qs, wk.head, wk.h, qam)
    qtok, qlen = torch.empty_like(wk.acc_tok), torch.empty_like(wk.acc_len)

    def qstep():
        w12.w12_tree_build(wk.dlat, wk.wl.budget, wk.ws, wk.tree)
        w12.w12_verify_step_q(qstep_args, wk.tree, wk.wl.n_req, wk.wl.p_max, wk.ws, qtok, qlen)

    def timed(fn):
        for _ in range(W):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fn()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    ms_step = timed(qstep)
    ms_head = timed(lambda: w12.w12_lmhead_argmax(wk.head, wk.h, wk.ws, argmax=qam, quick=True))
    if wk.ws.status() != 0:
        raise RuntimeError(f"device status {w12.status_str(wk.ws.status())}")
    view = lambda d: d.nbytes - d.rec.numel() // 3    # the view plane is 8 of every 12 KB
    qbytes = sum(view(d) for d in wk.lin) + view(wk.head)
    wk.step()
    torch.cuda.synchronize()
    agree = float((qam == wk.argmax).float().mean().item())
    return {"step_us": round(1e3 * ms_step, 2), "w12_view_bytes_per_step": int(qbytes),
            "gbs": round(qbytes / (ms_step * 1e-3) / 1e9, 1),
            "head_us": round(1e3 * ms_head, 2), "head_gbs": round(view(wk.head) / (ms_head * 1e-3) / 1e9, 1),
            "top1_agreement": round(agree, 4), "rows": int(wk.R)}


def certified_head(wk: "Workload", K: int, W: int):
    """The LM head through the certified head (quick-pass logits of every
    token, per-row Cauchy-Schwarz bound, exact FP64 rescoring of the
    survivors): graph-timed launch sequence, survivor counts, and the top-1
    agreement with the exact head's argmax on the step's rows."""
    import torch
    w12 = wk.w12
    norms = w12.w12_head_cert_norms(wk.head)
    cws = w12.CertWorkspace(wk.R, wk.head.n)
    cam = torch.empty_like(wk.argmax)
    surv = torch.empty(wk.R, dtype=torch.int32, device=wk.argmax.device)
    fn = lambda: w12.w12_lmhead_argmax_certified(wk.head, norms, wk.h, wk.ws, cws, argmax=cam, survivors=surv)
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    if wk.ws.status() != 0:
        raise RuntimeError(f"device status {w12.status_str(wk.ws.status())}")
    wk.step()
    torch.cuda.synchronize()
    n = surv.cpu().numpy()
    return {"head_us": round(1e3 * ms, 2), "survivors_mean": round(float(n.mean()), 2),
            "survivors_max": int(n.max()), "top1_agreement": round(float((cam == wk.argmax).float().mean().item()), 4),
            "rows": int(wk.R)}


def tlv_cycle(wk: "Workload", K: int, W: int, seed: int = 0):
    """One TLV cycle (explainer 4.3) on the step's first tree: the Q pass
    (w12_verify_step_q: every linear and the head on the view planes, then
    acceptance, giving the commit chain), the chain lengths read back to the
    host (w12_tlv_chain), the fresh subtree from the chain ends
    (w12_tree_build on a second synthetic lattice standing in for the
    drafter's second draft, prepared once: the inputs repeat every cycle),
    the splice (w12_tlv_splice) and the exact pass over the combined tree
    (w12_verify_step).  Eager launches with one host synchronisation per
    cycle (the chain lengths), timed with CUDA events; per-stage times from
    events around each stage.  Accepted tokens per exact pass are reported
    for the toy target of the synthetic rows, next to a single exact pass
    over the first tree: a property of the synthetic inputs, not of a model."""
    import torch
    w12, synth, w = wk.w12, wk.synth, wk.wl
    dev = wk.argmax.device
    n_req, p1 = w.n_req, w.p_max
    p2 = p1
    p_comb = p1 + 1 + p2
    i32 = torch.int32
    c_tok = torch.empty((n_req, p1 + 1), dtype=i32, device=dev)
    c_len = torch.empty(n_req, dtype=i32, device=dev)
    c_node = torch.empty(n_req, dtype=i32, device=dev)
    c_len_host = torch.empty(n_req, dtype=i32, pin_memory=True)
    q_args = w12.VerifyStep(wk.lin, wk.xs, [torch.empty_like(y) for y in wk.ys], wk.head, wk.h,
                            torch.empty_like(wk.argmax))
    row_off = wk.tree.req_row_off.cpu().numpy()
    # the second draft: rooted at each chain end, offered the rest of the true
    # continuation where the chain follows it
    w12.w12_verify_step_q(q_args, wk.tree, n_req, p1, wk.ws, c_tok, c_len, c_node)
    torch.cuda.synchronize()
    m, sub = w12.w12_tlv_chain(c_len.cpu().numpy(), row_off, w.budget)
    g = np.random.default_rng(seed + 977)
    truth_long = np.concatenate([wk.lat.truth, g.integers(0, w.vocab, size=(n_req, p2 + 1)).astype(np.int32)], 1)
    ct = c_tok.cpu().numpy()
    truth2 = g.integers(0, w.vocab, size=(n_req, p2 + 1)).astype(np.int32)
    root2 = np.asarray(wk.lat.root_tok, np.int32).copy()
    for q in range(n_req):
        mq = int(m[q])
        if mq:
            root2[q] = int(ct[q][mq - 1])
        if np.array_equal(ct[q][:mq], truth_long[q, :mq]):
            truth2[q] = truth_long[q, mq:mq + p2 + 1]
    lat2 = synth.lattice(synth.scaled(w, positions=(p2,)), seed + 101, truth=truth2, root_tok=root2)
    dlat2 = w12.DeviceLattice(lat2, dev)
    t2 = w12.DeviceTree(w.budget, n_req, dev)
    comb = w12.DeviceTree(w.budget, n_req, dev)
    w12.w12_tree_build(dlat2, sub, wk.ws, tree=t2)
    w12.w12_tlv_splice(wk.tree, c_tok, c_len, c_node, m, t2, wk.ws, out=comb)
    torch.cuda.synchronize()
    th = comb.host()
    Rc = comb.R
    hc = synth.hidden_rows(th["req"], th["parent"], th["token"], truth_long, wk.head_bits, seed,
                           head_norm2=wk.head_n2)
    tobf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    xc_layer = [tobf(synth.activations(Rc, k, seed, synth.STREAM_X + i)) for i, (n, k) in enumerate(w.linears)]
    xc = [xc_layer[j % len(w.linears)] for j in range(len(wk.lin))]
    yc = [torch.empty((Rc, dw.n), dtype=torch.bfloat16, device=dev) for dw in wk.lin]
    step_c = w12.VerifyStep(wk.lin, xc, yc, wk.head, tobf(hc), torch.empty(Rc, dtype=i32, device=dev))
    e_tok = torch.empty((n_req, p_comb + 1), dtype=i32, device=dev)
    e_len = torch.empty(n_req, dtype=i32, device=dev)
    e_node = torch.empty(n_req, dtype=i32, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def cycle(events):
        if events:
            events[0].record()
        w12.w12_verify_step_q(q_args, wk.tree, n_req, p1, wk.ws, c_tok, c_len, c_node)
        c_len_host.copy_(c_len, non_blocking=True)
        if events:
            events[1].record()
        torch.cuda.current_stream().synchronize()
        mm, sb = w12.w12_tlv_chain(c_len_host.numpy(), row_off, w.budget)
        w12.w12_tree_build(dlat2, sb, wk.ws, tree=t2)
        w12.w12_tlv_splice(wk.tree, c_tok, c_len, c_node, mm, t2, wk.ws, out=comb)
        if events:
            events[2].record()
        w12.w12_verify_step(step_c, comb, n_req, p_comb, wk.ws, e_tok, e_len, e_node)
        if events:
            events[3].record()

    for _ in range(W):
        cycle(None)
    torch.cuda.synchronize()
    q_ms = ops_ms = ex_ms = 0.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        cycle(ev)
        torch.cuda.synchronize()
        q_ms += ev[0].elapsed_time(ev[1])
        ops_ms += ev[1].elapsed_time(ev[2])
        ex_ms += ev[2].elapsed_time(ev[3])
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    if wk.ws.status() != 0:
        raise RuntimeError(f"device status {w12.status_str(wk.ws.status())}")
    wk.step()
    torch.cuda.synchronize()
    return {"cycle_us": round(1e3 * ms, 2), "q_pass_us": round(1e3 * q_ms / K, 2),
            "chain_subtree_splice_us": round(1e3 * ops_ms / K, 2), "exact_pass_us": round(1e3 * ex_ms / K, 2),
            "rows_q": int(wk.R), "rows_exact": int(Rc), "committed_chain_tokens": int(m.sum()),
            "synthetic_tokens_per_exact_pass": round(float(e_len.float().mean().item()), 3),
            "synthetic_tokens_single_pass": round(float(wk.acc_len.float().mean().item()), 3),
            "timing": "eager launches, one host sync per cycle for the chain lengths, CUDA events"}


GDN_LAYERS, GDN_HEADS, GDN_DIM = 48, 32, 128


def gdn_stack(wk: "Workload", K: int, W: int, seed: int = 0):
    """Recurrent-layer tree verification over the step's tree (explainer
    4.2): 48 Gated DeltaNet layers of 32 heads of 128 (synthetic committed
    states and q/k/v/gates, 4 distinct input sets, each layer with its own
    device copy), one launch per layer as a real stack would need, captured
    in a CUDA graph.  Times the WY kernel, the path-walk kernel, the
    commit replay of one accepted row per request, the WY kernel writing its
    vectors u, and the commit from those vectors (one pass over the states);
    bytes are the states read (and written by the commits) plus q/k/v/gates
    in and outputs out."""
    import torch
    w12, synth = wk.w12, wk.synth
    dev = wk.argmax.device
    n_req, R = wk.wl.n_req, wk.R
    tobf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    base = [synth.gdn_inputs(R, n_req, GDN_HEADS, GDN_DIM, seed=seed + i) for i in range(4)]
    layers = []
    for l in range(GDN_LAYERS):
        x = base[l % 4]
        layers.append(w12.GdnLayer(torch.from_numpy(x.S0).to(dev), tobf(x.q), tobf(x.k), tobf(x.v),
                                   torch.from_numpy(x.alpha).to(dev), torch.from_numpy(x.beta).to(dev)))
    outs = [torch.empty((R, GDN_HEADS, GDN_DIM), dtype=torch.float32, device=dev) for _ in range(GDN_LAYERS)]
    states = [torch.empty_like(L.S0) for L in layers]
    acc = (wk.tree.req_row_off[1:] - 1).contiguous()   # each request's last row: its deepest branch
    ws = w12.Workspace(1, 0, 0, n_req, dev)

    def run(method):
        for L, o in zip(layers, outs):
            w12.w12_gdn_tree_verify(L, wk.tree, n_req, ws, method, out=o)

    def commit():
        for L, st in zip(layers, states):
            w12.w12_gdn_commit(L, wk.tree, n_req, acc, ws, state=st)

    us = [torch.empty((R, GDN_HEADS, GDN_DIM), dtype=torch.float32, device=dev) for _ in range(GDN_LAYERS)]

    def run_wy_u():
        for L, o, u in zip(layers, outs, us):
            w12.w12_gdn_wy_verify(L, wk.tree, n_req, ws, out=o, u=u)

    def commit_wy():
        for L, st, u in zip(layers, states, us):
            w12.w12_gdn_wy_commit(L, wk.tree, n_req, acc, u, ws, state=st)

    def timed(fn):
        for _ in range(W):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fn()
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / K

    ms_wy = timed(lambda: run(w12.W12_GDN_WY))
    ms_path = timed(lambda: run(w12.W12_GDN_PATH))
    ms_commit = timed(commit)
    ms_wy_u = timed(run_wy_u)
    ms_commit_wy = timed(commit_wy)
    if ws.status() != 0:
        raise RuntimeError(f"device status {w12.status_str(ws.status())}")
    state_b = n_req * GDN_HEADS * GDN_DIM * GDN_DIM * 4
    io_b = R * GDN_HEADS * (3 * GDN_DIM * 2 + 2 * 4) + R * GDN_HEADS * GDN_DIM * 4
    verify_bytes = GDN_LAYERS * (state_b + io_b)
    commit_bytes = GDN_LAYERS * (2 * state_b + R * GDN_HEADS * (2 * GDN_DIM * 2 + 2 * 4))
    return {"layers": GDN_LAYERS, "heads": GDN_HEADS, "head_dim": GDN_DIM, "rows": int(R), "requests": int(n_req),
            "wy_us": round(1e3 * ms_wy, 2), "path_us": round(1e3 * ms_path, 2), "commit_us": round(1e3 * ms_commit, 2),
            "wy_with_u_us": round(1e3 * ms_wy_u, 2), "commit_wy_us": round(1e3 * ms_commit_wy, 2),
            "verify_bytes": int(verify_bytes), "wy_gbs": round(verify_bytes / (ms_wy * 1e-3) / 1e9, 1),
            "commit_gbs": round(commit_bytes / (ms_commit * 1e-3) / 1e9, 1),
            "commit_wy_gbs": round(commit_bytes / (ms_commit_wy * 1e-3) / 1e9, 1),
            "timing": "CUDA graph of the 48 per-layer launches, CUDA events",
            "inputs": "synthetic: N(0, 0.05) states, unit-norm q/k, N(0, 1) v, gates U[0.85, 1), strengths U[0.05, 0.95]"}


def gdn_batched(wk: "Workload", K: int, W: int):
    """The same 48-layer recurrent stack over the batched_27b tree (24
    requests drafting 16/12/8 positions, 192 rows): the WY form runs on the
    tensor-memory kernel there, on the sliced kernel for one request."""
    import types
    w12, synth = wk.w12, wk.synth
    dev = wk.argmax.device
    w = synth.WORKLOADS["batched_27b"]
    ws = w12.Workspace(w.budget, 0, 0, w.n_req, dev)
    tree = w12.w12_tree_build(w12.DeviceLattice(synth.lattice(w, 0), dev), w.budget, ws)
    sub = types.SimpleNamespace(w12=w12, synth=synth, argmax=wk.argmax, wl=w, R=tree.R, tree=tree)
    return gdn_stack(sub, K, W)


# ---------------------------------------------------------------------------
# step time vs tree rows
# ---------------------------------------------------------------------------

class CublasRef:
    """Context for the W12 step: dense BF16 torch.matmul (cuBLAS) over the
    same GEMM shapes, every stacked layer with dense weights of its own (so no
    layer is served from L2), then the LM head's logits and their argmax,
    captured in one CUDA graph.  Weights are N(0, 0.02) BF16."""

    def __init__(self, wk: "Workload"):
        import torch
        self.torch, self.device = torch, wk.device
        g = torch.Generator(device=wk.device)
        g.manual_seed(1234)
        bf = torch.bfloat16
        self.lin = [(torch.randn((d.n, d.k), generator=g, device=wk.device, dtype=torch.float32) * 0.02).to(bf)
                    for d in wk.lin]
        self.head = (torch.randn((wk.head.n, wk.head.k), generator=g, device=wk.device,
                                 dtype=torch.float32) * 0.02).to(bf)
        self.bytes = sum(2 * w.numel() for w in self.lin) + 2 * self.head.numel()

    def time_us(self, R: int, K: int, W: int) -> float:
        torch = self.torch
        xs = {}
        for w in self.lin:
            if w.shape[1] not in xs:
                xs[w.shape[1]] = torch.randn((R, w.shape[1]), device=self.device, dtype=torch.bfloat16)
        h = torch.randn((R, self.head.shape[1]), device=self.device, dtype=torch.bfloat16)

        def step():
            for w in self.lin:
                torch.matmul(xs[w.shape[1]], w.t())
            torch.argmax(torch.matmul(h, self.head.t()).float(), dim=1)

        g = _graph_of(step)
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        del g
        return 1e3 * e0.elapsed_time(e1) / K

    def free(self):
        self.lin, self.head = [], None
        self.torch.cuda.empty_cache()


def parse_sweep(spec: str):
    """'1,8,32,b192' -> [(1, False), (8, False), (32, False), (192, True)]:
    node budgets of one request's tree, or ('b' prefix) of 24 requests drafting
    16/12/8 positions sharing the budget."""
    out = []
    for v in spec.split(","):
        v = v.strip()
        if v:
            out.append((int(v[1:]), True) if v.startswith("b") else (int(v), False))
    return out


def rows_sweep(base: "Workload", points, K: int, W: int, device, cublas=None, peak=None):
    """Step time and W12 GB/s of the graph-captured step at each node budget,
    reusing the packed weights of `base` (only the tree, its rows and the
    activations change), with dense cuBLAS BF16 on the same shapes and rows
    beside it.  Same timing rules as the headline number."""
    import torch
    out = []
    for b, batched in points:
        variant = dict(n_req=24, positions=(16, 12, 8)) if batched else None
        wk = Workload(base.name, int(b), device, share=base, one_request=not batched, variant=variant)
        for _ in range(W):
            wk.step()
        torch.cuda.synchronize()
        g = _graph_of(wk.step)
        for _ in range(W):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / K
        if wk.ws.status() != 0:
            raise RuntimeError(f"device status {wk.w12.status_str(wk.ws.status())} at budget {b}")
        gbs = wk.w12_bytes() / (ms * 1e-3) / 1e9
        e = {"rows": int(wk.R), "requests": int(wk.wl.n_req), "step_us": round(1e3 * ms, 2), "w12_gbs": round(gbs, 1),
             "pct_of_8tbs": round(100 * gbs / NOMINAL_HBM_GBS, 2)}
        if peak:
            e["pct_of_measured_hbm"] = round(100 * gbs / peak, 2)
        del g
        if cublas is not None:
            cu = cublas.time_us(int(wk.R), K, W)
            e["cublas_bf16_us"] = round(cu, 2)
            e["w12_speedup_vs_cublas"] = round(cu / (1e3 * ms), 3)
        out.append(e)
        del wk
    return out


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--workload", default="full_depth_27b")
    ap.add_argument("--rows", type=int, default=0, help="override the node budget (tree rows)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cublas", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--rows-sweep", default=None,
                    help="comma-separated node budgets timed after the headline, each of one request's tree, "
                         "or with a 'b' prefix of 24 requests' trees (default: 1,8,32,64,128,192,b192 for "
                         "single-request workloads, none otherwise; 'none' to skip)")
    ap.add_argument("--extras", default="all", choices=["all", "none"],
                    help="the measurements after the headline and its end-to-end pass (quick pass, certified "
                         "head, TLV cycle, recurrent-layer stack): all, or none for a launch list of the step alone")
    ap.add_argument("--gemm", default="auto", choices=["auto", "tcgen05", "warp_mma"],
                    help="GEMM kernel: the library's choice by row count, or one forced")
    ap.add_argument("--chain", default="auto", choices=["auto", "on", "off"],
                    help="verify step as one persistent GEMM-chain launch (on), one launch per GEMM (off), "
                         "or the library's choice")
    args = ap.parse_args()
    if args.warmup < 3:
        log("[bench] warmup raised to 3")
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = replica_env()
    if world > 1:
        torch.cuda.set_device(local)
    dist = init_replicas(world, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    from speculative_decoding_tree_w12_gb300 import build as w12build
    if rank == 0 or world == 1:
        w12build.build()
    if dist:
        dist.barrier()
    import speculative_decoding_tree_w12_gb300 as w12
    w12.debug_set({"auto": 0, "tcgen05": 2, "warp_mma": 4}[args.gemm] | {"auto": 0, "on": 16, "off": 8}[args.chain], 0)

    wk = Workload(args.workload, args.rows, device)
    W, K = args.warmup, args.steps
    for _ in range(W):
        wk.step()
    torch.cuda.synchronize()
    st = wk.ws.status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {w12.status_str(st)}")
    ref_tok = wk.acc_tok.clone()
    ref_len = wk.acc_len.clone()

    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            wk.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph):
            wk.step()
        for _ in range(W):
            graph.replay()
        torch.cuda.synchronize()

    run = graph.replay if graph is not None else wk.step

    # ------------------------------------------------------------ timed region
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(K):
        run()
    e1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clocks = clk.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / K, dist, device)
    st = wk.ws.status()
    if st != 0 or not torch.equal(wk.acc_tok, ref_tok) or not torch.equal(wk.acc_len, ref_len):
        raise RuntimeError(f"timed steps diverged from the warm-up result (status {w12.status_str(st)})")

    w12_bytes = wk.w12_bytes()
    value = whole_job_gbs(world, w12_bytes, ms)

    # ------------------------------------------------ per-launch roofline pass
    w12.profile(True)
    per_launch = None
    tb_ms = []
    for _ in range(K):
        w12.w12_tree_build(wk.dlat, wk.wl.budget, wk.ws, wk.tree)
        w12.w12_verify_step(wk.step_args, wk.tree, wk.wl.n_req, wk.wl.p_max, wk.ws, wk.acc_tok, wk.acc_len)
        lt = np.asarray(w12.profile_read())
        torch.cuda.synchronize()
        per_launch = lt if per_launch is None else per_launch + lt
    # tree build alone: back-to-back launches between the events, so that the
    # host's launch latency is not counted
    for _ in range(max(1, K // 10)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w12.w12_tree_build(wk.dlat, wk.wl.budget, wk.ws, wk.tree)
        a.record()
        for _ in range(10):
            w12.w12_tree_build(wk.dlat, wk.wl.budget, wk.ws, wk.tree)
        b.record()
        torch.cuda.synchronize()
        tb_ms.append(a.elapsed_time(b) / 10)
    w12.profile(False)
    per_launch = per_launch / K
    n_gemm = len(per_launch) - 2                     # then the argmax reduction and acceptance
    n_weights = len(wk.lin) + 1
    chain = n_gemm < n_weights                       # the whole GEMM chain in one or two launches
    per_weight = 1 if chain else n_gemm // n_weights
    lb = wk.launch_bytes(per_weight)
    gemm_ms = per_launch[:n_gemm]
    gemm_bytes = float(sum(lb))
    achieved = gemm_bytes / (float(gemm_ms.sum()) * 1e-3) / 1e9
    if chain:
        lb = [gemm_bytes]
    peak, peak_kind = load_peaks()
    traffic = None if chain or per_weight != 1 else committed_traffic(wk.gemm_shapes())
    kernels = {
        "tree_build_us": 1e3 * float(np.mean(tb_ms)),
        "argmax_stage2_us": 1e3 * float(per_launch[n_gemm]),
        "accept_us": 1e3 * float(per_launch[n_gemm + 1]),
    }
    n_lin = len(wk.wl.linears)
    if chain:
        kernels["w12_gemm_chain_us"] = [round(1e3 * float(v), 2) for v in gemm_ms]
    elif per_weight == 1:
        # per linear of the layer (mean over the stacked layers) and the LM head
        names = ["qkv", "o", "gate_up", "down"] if n_lin == 4 else [f"linear{i}" for i in range(n_lin)]
        for i, nm in enumerate(names):
            sel = range(i, len(wk.lin), n_lin)
            t = float(np.mean([gemm_ms[j] for j in sel]))
            kernels[f"{nm}_us"] = round(1e3 * t, 2)
            kernels[f"{nm}_gbs"] = round(float(np.mean([lb[j] for j in sel])) / (t * 1e-3) / 1e9, 1)
        kernels["head_us"] = round(1e3 * float(gemm_ms[-1]), 2)
        kernels["head_gbs"] = round(lb[-1] / (float(gemm_ms[-1]) * 1e-3) / 1e9, 1)
        kernels["layer_us"] = round(1e3 * float(np.sum(gemm_ms[:-1])) / max(1, wk.wl.layers), 2)
    else:
        kernels["w12_gemm_us"] = [round(1e3 * float(v), 2) for v in gemm_ms]

    # ------------------------------------------------------------ end to end
    e2e = None
    try:
        e2e = measure_e2e(wk, K, w12_bytes, world, dist, device)
    except Exception as ex:  # reported, never hidden
        e2e = {"value": None, "unit": "GB/s", "error": str(ex)[:200]}

    # ------------------------------------------------------- cuBLAS context
    cublas, cref = None, None
    if not args.no_cublas and rank == 0:
        try:
            cref = CublasRef(wk)
            cu = cref.time_us(wk.R, max(10, min(K, 50)), W)
            cublas = {"us_per_step": round(cu, 2), "bf16_bytes": cref.bytes, "gbs": round(cref.bytes / (cu * 1e-6) / 1e9, 1),
                      "layers_per_step": wk.wl.layers, "w12_speedup": round(cu / (1e3 * ms), 3),
                      "note": "torch.matmul BF16 (cuBLAS), dense weights of the same shapes for every stacked layer, "
                              "LM head logits + argmax, one CUDA graph"}
        except Exception as ex:
            cublas = {"error": str(ex)[:200]}

    # ------------------------------------------------------- quick pass
    quick = None
    try:
        if args.extras == "all":
            quick = quick_pass(wk, K, W)
    except Exception as ex:  # reported, never hidden
        quick = {"error": str(ex)[:200]}

    # ------------------------------------------------- certified head
    cert = None
    try:
        if args.extras == "all":
            cert = certified_head(wk, K, W)
    except Exception as ex:  # reported, never hidden
        cert = {"error": str(ex)[:200]}

    # ------------------------------------------------------------ TLV cycle
    tlv = None
    try:
        if args.extras == "all":
            tlv = tlv_cycle(wk, max(10, min(K, 50)), W)
    except Exception as ex:  # reported, never hidden
        tlv = {"error": str(ex)[:200]}

    # ------------------------------------------- recurrent-layer verification
    gdn = gdn_b = None
    try:
        if args.extras == "all":
            gdn = gdn_stack(wk, max(10, min(K, 50)), W)
    except Exception as ex:  # reported, never hidden
        gdn = {"error": str(ex)[:200]}
    try:
        if args.extras == "all":
            gdn_b = gdn_batched(wk, max(10, min(K, 50)), W)
            if gdn and "wy_us" in gdn:
                # per layer, batched tree over the workload's tree
                gdn_b["wy_over_workload_tree"] = round(gdn_b["wy_us"] / gdn["wy_us"], 3)
    except Exception as ex:  # reported, never hidden
        gdn_b = {"error": str(ex)[:200]}

    # --------------------------------------------------- step time vs rows
    sweep = None
    spec = args.rows_sweep
    if spec is None:
        spec = "1,8,32,64,128,192,b192" if wk.wl.n_req == 1 else "none"
    if spec != "none":
        try:
            sweep = rows_sweep(wk, parse_sweep(spec), max(10, min(K, 50)), W, device, cublas=cref, peak=peak)
        except Exception as ex:  # reported, never hidden
            sweep = [{"error": str(ex)[:200]}]
    if cref is not None:
        cref.free()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wk)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}", "rows": wk.R,
                       "requests": wk.wl.n_req, "layers": wk.wl.layers, "w12_bytes_per_step": w12_bytes,
                       "l2": "inputs larger than L2 (W12 bytes per step vs 129 MB L2); no flush",
                       "timing": "CUDA-graph replays of the whole step, CUDA events" if graph else "eager launches",
                       "parallelism": "replicas" if world > 1 else "single GPU", "gemm_kernel": args.gemm,
                       "gemm_chain": args.chain},
            "step_us": round(1e3 * ms, 2),
            "pct_of_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
            "pct_of_measured_hbm": round(100 * value / world / peak, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": "k_w12_chain" if chain else "k_w12_gemm + k_w12_gemm_tc",
                         "peak_kind": peak_kind,
                         "note": "all W12 GEMM launches of a step (linears + LM head), serialised, algorithmic bytes "
                                 "(W12 + activations + outputs) / summed launch time; traffic: ncu DRAM bytes read + "
                                 "written of one layer's launches and the head at the same rows, times the layers"},
            "kernels": kernels,
            "e2e": e2e,
            "cublas_bf16": cublas,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "gpu_launches": K * (3 + n_gemm if chain else wk.gpu_launches_per_step(per_weight)),
            "rows_sweep": sweep,
            "quick_pass": quick,
            "certified_head": cert,
            "tlv_cycle": tlv,
            "gdn_tree": gdn,
            "gdn_tree_batched": gdn_b,
        }
        if sweep and all("step_us" in e for e in sweep):
            one = {e["rows"]: e["step_us"] for e in sweep if e["requests"] == 1}
            if 1 in one and 64 in one:
                line["rows_sweep_flatness"] = round(one[64] / one[1], 4)
                line["rows_sweep_flatness_note"] = "step time at 64 rows / at 1 row, one request's tree"
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def _graph_of(fn):
    """Capture fn() (CUDA work on the current stream) in a CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    return g


def measure_e2e(wk: Workload, K: int, w12_bytes: int, world: int = 1, dist=None, device=None):
    """Through the public API with host buffers: every step copies its inputs
    (the lattice, the activations of every linear and the hidden rows) in
    from pinned host memory, runs the pass (tree build + verify step) and
    reads the accepted tokens and lengths back, all inside the timed region.
    Two device input sets alternate, so the copies of step k+1 overlap the
    pass of step k (a serving loop's double buffering)."""
    import torch
    wkb = Workload(wk.name, wk.wl.budget, device, share=wk)       # second input set, same content
    sets = [wk, wkb]
    pin = lambda t: t.cpu().pin_memory()

    def inputs(w):
        dev = [w.dlat.root_tok, w.dlat.cand_tok, w.dlat.cand_logp, w.h]
        seen = set()
        for x in w.xs:
            if x.data_ptr() not in seen:
                seen.add(x.data_ptr())
                dev.append(x)
        return dev

    host = [pin(t) for t in inputs(wk)]
    dev_in = [inputs(w) for w in sets]
    out = [(torch.empty_like(w.acc_tok, device="cpu").pin_memory(),
            torch.empty_like(w.acc_len, device="cpu").pin_memory()) for w in sets]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out[0][0].numel() * 4 + out[0][1].numel() * 4
    graphs = [_graph_of(w.step) for w in sets]
    copy_s = torch.cuda.Stream()
    comp_s = torch.cuda.current_stream()
    copied = [torch.cuda.Event() for _ in sets]
    freed = [torch.cuda.Event() for _ in sets]

    def run(n):
        for w in freed:
            w.record(comp_s)
        for k in range(n):
            b = k & 1
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(freed[b])          # the pass that last read set b is done
                for h, d in zip(host, dev_in[b]):
                    d.copy_(h, non_blocking=True)
                copied[b].record(copy_s)
            comp_s.wait_event(copied[b])
            graphs[b].replay()
            out[b][0].copy_(sets[b].acc_tok, non_blocking=True)
            out[b][1].copy_(sets[b].acc_len, non_blocking=True)
            freed[b].record(comp_s)
        comp_s.wait_stream(copy_s)

    run(4)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp_s)
    run(K)
    e1.record(comp_s)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / K, dist, device)
    same = all(torch.equal(out[b][0], wk.acc_tok.cpu()) and torch.equal(out[b][1], wk.acc_len.cpu()) for b in (0, 1))
    if not same:
        raise RuntimeError("end-to-end steps diverged from the device-resident result")
    return {"value": round(whole_job_gbs(world, w12_bytes, ms), 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "inputs copied from pinned host memory and results read back every step; two device input "
                    "sets alternate so that step k+1's copies overlap step k's pass"}


if __name__ == "__main__":
    sys.exit(main())
