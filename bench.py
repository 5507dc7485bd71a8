"""Benchmark of the persistent KV-cache hot path on one GB300 (or N replicas).

A step is one pass of the whole path over one batch: device-side lengths,
the RoPE append of the new K/V row, and the split-KV GQA decode (with its
merge).  The default workload is the contiguous persistent-cache decode
(batch 32, 32 query / 8 KV heads, head_dim 128, capacity 8192, per-sequence
total length uniform in [512, 8192], bf16, RoPE theta 10000).  Inputs are
seeded synthetic tensors; the 570 MB the step reads exceed the 129 MB L2, so
no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload contig-decode|window-decode|scatter]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV append+GQA decode: achieved HBM GB/s (% of peak), decode steps/s"
FALLBACK_HBM_GBS = 6800.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------
# clocks during the run (nvidia-smi sampler)
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.index = str(device.index or 0)
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            self.index = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r[2] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in busy])), "sm_max_mhz": busy[0][1],
                "reasons": reasons, "samples": len(busy)}


# --------------------------------------------------------------------------
# multi-rank plumbing (one process per GPU; ranks are independent replicas)
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

class ContigDecode:
    """Contiguous persistent-cache GQA decode, one-token append then attention."""

    def __init__(self, dev, seed=0, with_kernels=True):
        import torch

        from persistent_kv_cache_gb300 import synth
        self.torch = torch
        w = self.w = synth.CONTIG_DECODE
        B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.kc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.vc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.T = synth.randint(w.total_lo, w.total_hi + 1, (B,), seed, 77).numpy()
        self.sk_host = torch.from_numpy((self.T - 1).astype(np.int32))
        self.q_host = synth.normal((B, Hq, 1, D), seed, 5)
        self.nk_host = synth.normal((B, Hkv, 1, D), seed, 3)
        self.nv_host = synth.normal((B, Hkv, 1, D), seed, 4)
        self.sk = self.sk_host.to(dev)
        self.q = self.q_host.to(dev)
        self.nk = self.nk_host.to(dev)
        self.nv = self.nv_host.to(dev)
        cos, sin = synth.rope_cache(C, D, w.theta)
        self.rope = (cos.to(dev), sin.to(dev))
        e = 2
        self.decode_bytes = int(self.T.sum()) * Hkv * D * 2 * e + 2 * B * Hq * D * e
        self.append_bytes = 2 * 2 * B * Hkv * D * e
        self.bytes_per_step = self.decode_bytes + self.append_bytes
        self.tokens_per_step = B
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = torch.empty(B, Hq, 1, D, dtype=bf, device=dev)
        self.ws = K.decode_workspace(self.out, self.kc)
        self.L = K.Lengths(B, dev)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches_per_step = 3 + (1 if K.kvc_gqa_decode_workspace_size(
            B, Hq, Hkv, C, D, K.KVC_BF16) > 256 else 0)

    def step(self, ev=None):
        K = self.K
        K.kvc_seq_lengths(self.sk, 1, self.w.capacity, 0, out=self.L, status=self.st)
        K.kvc_window_append(self.kc, self.vc, self.nk, self.nv, self.L, 0, rope=self.rope,
                            status=self.st)
        if ev is not None:
            ev[0].record()
        K.kvc_gqa_decode(self.out, self.q, self.kc, self.vc, self.L, rope=self.rope,
                         workspace=self.ws, status=self.st)
        if ev is not None:
            ev[1].record()

    # end-to-end: per step copy the inputs from pinned host memory and read
    # the result back, all inside the timed region
    def e2e_setup(self):
        torch = self.torch
        self.h_in = [t.pin_memory() for t in (self.sk_host, self.q_host, self.nk_host,
                                               self.nv_host)]
        self.d_in = [self.sk, self.q, self.nk, self.nv]
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.h2d = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h = self.h_out.numel() * self.h_out.element_size()

    def e2e_step(self):
        for h, d in zip(self.h_in, self.d_in):
            d.copy_(h, non_blocking=True)
        self.step()
        self.h_out.copy_(self.out, non_blocking=True)

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                "total_len": f"U[{w.total_lo},{w.total_hi}] after the append",
                "rope_theta": w.theta, "new_tokens": 1,
                "l2": "inputs larger than L2 (~570 MB of K/V read per step)",
                "bytes_per_step": self.bytes_per_step}

    # ---- CPU oracle on a bounded sample of the same workload ----
    def oracle_sample(self, rows):
        """Times the oracle's append + attention for the given batch rows;
        returns (seconds, algorithmic bytes of those rows)."""
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        torch = self.torch
        rows = list(rows)
        kc = synth.bits(self.kc[rows].cpu()).copy()
        vc = synth.bits(self.vc[rows].cpu()).copy()
        nk, nv = synth.bits(self.nk_host[rows]), synth.bits(self.nv_host[rows])
        q = synth.bits(self.q_host[rows])
        cos, sin = (t.cpu().numpy() for t in self.rope)
        sk = (self.T[rows] - 1).astype(np.int32)
        t0 = time.perf_counter()
        lens = oracle.seq_lengths(sk, 1, w.capacity, 0)
        oracle.window_append(kc, vc, nk, nv, lens, 0, cos, sin)
        oracle.gqa_attention(q, kc, vc, lens["cache_total"], lens["total_abs"], cos_cache=cos,
                             sin_cache=sin)
        dt = time.perf_counter() - t0
        e = 2
        nbytes = (int(self.T[rows].sum()) * w.kv_heads * w.head_dim * 2 * e
                  + 2 * len(rows) * w.q_heads * w.head_dim * e
                  + 2 * 2 * len(rows) * w.kv_heads * w.head_dim * e)
        return dt, nbytes


WORKLOADS = {"contig-decode": ContigDecode}


def kernel_traffic(kernel_file: str, key: str):
    """dram bytes per launch recorded from an ncu capture, or None when the
    kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[key]
        src = open(os.path.join(ROOT, "persistent_kv_cache_gb300", "csrc", kernel_file), "rb").read()
        if rec["source_sha256"] != hashlib.sha256(src).hexdigest():
            return None
        return rec["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[args.workload](dev, seed=rank)
    peak, peak_kind = load_peaks()

    with ClockSampler(dev) as clocks:
        for _ in range(args.warmup):
            wl.step()
        torch.cuda.synchronize()
        # device-timed steps, inputs resident in HBM
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for i in range(args.steps):
            wl.step(evs[i])
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = start.elapsed_time(end)
        dec_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        # end to end through the public API with host buffers
        wl.e2e_setup()
        for _ in range(args.warmup):
            wl.e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            wl.e2e_step()
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        barrier(world)
    status = int(wl.st.item())
    ms = max_over_ranks(ms, world, dev)
    e2e_s = max_over_ranks(e2e_s, world, dev)

    if rank != 0:
        return
    sec = ms / 1e3
    gbs = wl.bytes_per_step * args.steps * world / sec / 1e9
    e2e_gbs = wl.bytes_per_step * args.steps * world / e2e_s / 1e9
    achieved = wl.decode_bytes / (dec_ms / 1e3) / 1e9
    traffic = kernel_traffic("kvc_decode.cu", "decode_split_kernel")
    cpu = None
    if world == 1:
        dt, nb = wl.oracle_sample(range(wl.w.batch))
        cpu = {"value": nb / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"one full step ({wl.w.batch} batch rows: append + attention), "
                         f"{dt:.2f} s single-threaded C oracle"}
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": wl.config(),
        "pct_of_peak": 100.0 * gbs / peak,
        "decode_steps_per_s": args.steps * world / sec,
        "tokens_per_s": wl.tokens_per_step * args.steps * world / sec,
        "e2e": {"value": e2e_gbs, "unit": "GB/s", "h2d_bytes_per_step": wl.h2d,
                "d2h_bytes_per_step": wl.d2h,
                "steps_per_s": args.steps * world / e2e_s},
        "roofline": {"bound": "hbm", "kernel": "kvc_gqa_decode (split + merge launches)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes_per_launch": wl.decode_bytes,
                     "avg_launch_ms": dec_ms},
        "cpu_baseline": cpu,
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "device_status": status,
    }
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Setup, W + K device steps and nothing else: the command profiled by
    ncu (no end-to-end pass, no oracle timing)."""
    import torch
    dev = torch.device("cuda", 0)
    wl = WORKLOADS[args.workload](dev, seed=0)
    for _ in range(args.warmup + args.steps):
        wl.step()
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": args.workload, "steps": args.steps, "warmup": args.warmup,
                      "device_status": int(wl.st.item())}), flush=True)


def run_reference(args):
    """The oracle timed on the host cores, each step a bounded sample (two
    batch rows) of the same workload."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    torch.set_num_threads(1)
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    wl = WORKLOADS[args.workload](dev, seed=0, with_kernels=False)
    B = wl.w.batch
    for i in range(args.warmup):
        wl.oracle_sample([(2 * i) % B, (2 * i + 1) % B])
    total_t, total_b = 0.0, 0
    for i in range(args.steps):
        dt, nb = wl.oracle_sample([(2 * i) % B, (2 * i + 1) % B])
        total_t += dt
        total_b += nb
    v = total_b / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": wl.config(),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "two batch rows of the workload per step"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="contig-decode")
    ap.add_argument("--profile", action="store_true",
                    help="device steps only (the command run under ncu)")
    args = ap.parse_args()
    if args.profile:
        from persistent_kv_cache_gb300 import build as B
        B.build()
        run_profile(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        from persistent_kv_cache_gb300 import build as B
        B.build()
        run_ours(args)


if __name__ == "__main__":
    main()
