"""Benchmark of the persistent KV-cache hot path on one GB300 (or N replicas).

A step is one pass of the whole path over one batch.  Default workload: the
contiguous persistent-cache decode (batch 32, 32 query / 8 KV heads,
head_dim 128, capacity 8192, per-sequence total length uniform in
[512, 8192] after the append, bf16, RoPE theta 10000); one step = device-side
lengths + RoPE append of the new K/V row + split-KV GQA decode + merge, as
one kvc_decode_step call (two launches; --workload contig-decode-unfused:
the same as four separate launches).
The ~570 MB the step reads exceed the 129 MB L2, so no flush is needed.

Other workloads (--workload):
  window-decode   64 x 64/8 heads x 64, C = W = 128, T0 ~ U[1, 32768];
                  one step = lengths + in-place compaction/append + decode on
                  one of 16 replica caches in turn (268 MB > L2, "cold"), as
                  one fused kvc_window_decode_step launch
  window-decode-unfused  the same as three launches
  window-decode-drift    the same with the drifting layout, C = W + 16 = 144
                  (a block of 17 rows reclaimed every 17 steps; fused step)
  window-decode-ring     the same window as a ring of C = W = 128 slots
                  (token p in slot p mod C, nothing moves; fused step)
  window-prefill  8 x 16/8 heads x 256, C = W = 4096, P ~ U[0, 20000],
                  --chunk S in {64, 512, 2048}; one step = lengths + staging
                  seed/append + tcgen05 chunk attention + copy-back
  window-prefill-inplace  the same step with the stage held in the cache's
                  own rows (no seed copy; the copy-back is an in-place shift)
  window-prefill-hazard  the same step as one kvc_window_prefill_step call,
                  which stages only the rows whose eviction the chunk sees
  window-prefill-hazard-slack  the same with C = W + 64 (no row is staged)
  scatter         TensorScatter circular, (16, 8, 4096, 128) bf16, in place,
                  --chunk S in {1, 16, 64}; one step = one scatter call (the
                  line also reports the per-launch floor of a graph node)
  scatter-functional  the same into a separate present cache (the whole
                  128 MiB cache copied, HBM-bound)
  window-decode-hot   window-decode on one cache (16.8 MB, L2-resident)
  paged-decode    the contiguous decode workload held in 64-row pages of a
                  shuffled page pool (lengths + paged append + paged decode)
  paged-decode-int8  the same with every full page below a row's newest one
                  quantized to int8 (lengths + append + mixed-page decode)
  ring-decode-d256  one-token decode at head_dim 256: 8 x 16/8 heads held as
                  a ring of C = W = 4096 slots, T ~ U[1, 20000] (one
                  kvc_decode_step + merge)
  window-decode-d256  the same heads kept compacted (C = W = 4096): lengths +
                  in-place compaction by one row (cluster kernel) + split
                  decode + merge; the roofline kernel is the compaction

The default one-GPU run also times window-prefill at S = 2048 and S = 64,
window-decode, scatter-functional (S = 64), ring-decode-d256,
window-decode-d256, paged-decode-int8 and window-prefill-hazard (S = 64),
each as an
entry of the line's "secondary" list with its own roofline, clocks and CPU
baseline (--no-secondary leaves them out).  Before each timed region the
step graph is replayed for --soak seconds (default 1) so that the clock
record covers the GPU under that load.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload ...] [--chunk S] [--profile] [--soak SEC]
                       [--secondary | --no-secondary]
Prints one JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV append+GQA decode: achieved HBM GB/s (% of peak), decode steps/s"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# nominal GB300 figures: HBM3e bandwidth and dense bf16 tensor throughput
NOMINAL_GBS, NOMINAL_TFLOPS = 7900.0, 2250.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


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
        self.lines = []

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
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "samples_under_load": 0}
        loaded = [r for r in rows if r[2] > 0]
        busy = loaded or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in busy])), "sm_max_mhz": busy[0][1],
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "sm_mhz_min_under_load": min(r[0] for r in busy)}


# --------------------------------------------------------------------------
# multi-rank plumbing (one process per GPU; ranks are independent replicas)
# --------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float, world: int, device) -> float:
    """Largest value over all ranks (timings are reported as the slowest rank)."""
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

E2E_COPIES = {
    False: "every step copies its inputs in from pinned host memory and its result out, "
           "on the compute stream",
    True: "every step copies its inputs in from pinned host memory and its result out, "
          "on two copy streams with doubled device buffers, overlapped with the "
          "neighbouring steps' compute"}


class Workload:
    """Common end-to-end pass: per step, copy the step's inputs from pinned
    host memory, run the step through the public API, copy the result back;
    all inside the timed region.  With e2e_overlap the copies run on streams
    of their own and the device buffers are doubled, so that step i + 1's
    inputs travel while step i computes and step i's result travels while
    step i + 1 computes (events keep every buffer from being overwritten
    while in use); that costs about ten more host calls a step, so it is
    taken by the workloads whose step lasts clearly longer than their host
    side (about 90 us and up), and the others copy on the compute stream."""
    e = 2  # bytes per bf16 element
    e2e_overlap = False
    # False where the result read back is a view of state the next step
    # updates in place: that step then waits for the read-back
    out_double = True

    def e2e_setup(self):
        """The step's inputs travel as one pinned host buffer and one copy:
        every device input is re-pointed (in place, so the workload keeps
        using the same tensor objects) at its slice of the device buffer the
        step uses (one, or two taken in turn)."""
        torch = self.torch
        self._offs, n = [], 0
        for t in self.host_inputs:
            self._offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        self.h_pack = torch.empty(n, dtype=torch.uint8).pin_memory()
        dev = self.device_inputs[0].device
        for h, o in zip(self.host_inputs, self._offs):
            nb = h.numel() * h.element_size()
            self.h_pack[o:o + nb].copy_(h.contiguous().view(-1).view(torch.uint8))
        nbuf = 2 if self.e2e_overlap else 1
        self.d_packs = [torch.empty(n, dtype=torch.uint8, device=dev) for _ in range(nbuf)]
        for d in self.d_packs:
            d.copy_(self.h_pack)
        self._point_inputs(0)
        two = self.e2e_overlap and self.out_double
        self.outs = [self.out, torch.empty_like(self.out) if two else self.out]
        self.h_outs = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
                       for _ in range(nbuf)]
        if self.e2e_overlap:
            self.s_in, self.s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
            self.ev_in, self.ev_comp, self.ev_out = ([torch.cuda.Event() for _ in range(2)]
                                                     for _ in range(3))
        self._n = 0
        self.h2d = n
        self.d2h = self.h_outs[0].numel() * self.h_outs[0].element_size()

    def _point_inputs(self, k):
        for d, o in zip(self.device_inputs, self._offs):
            d.set_(self.d_packs[k].untyped_storage(), o // d.element_size(), d.shape, d.stride())

    def e2e_step(self, i):
        if not self.e2e_overlap:
            self.d_packs[0].copy_(self.h_pack, non_blocking=True)
            self.step(i)
            self.h_outs[0].copy_(self.out, non_blocking=True)
            return
        torch = self.torch
        k, first = self._n % 2, self._n < 2
        comp = torch.cuda.current_stream()
        with torch.cuda.stream(self.s_in):
            if not first:
                self.s_in.wait_event(self.ev_comp[k])   # step n - 2 is done with buffer k
            self.d_packs[k].copy_(self.h_pack, non_blocking=True)
            self.ev_in[k].record(self.s_in)
        comp.wait_event(self.ev_in[k])
        if self._n > 0:
            # the result buffer this step writes has been read back
            comp.wait_event(self.ev_out[k if self.out_double else 1 - k])
        self._point_inputs(k)
        self.out = self.outs[k]
        self.step(i)
        self.ev_comp[k].record(comp)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.ev_comp[k])
            self.h_outs[k].copy_(self.out, non_blocking=True)
            self.ev_out[k].record(self.s_out)
        self._n += 1


class ContigDecode(Workload):
    """Contiguous persistent-cache GQA decode, one-token append then attention.
    fused=True runs each step as one kvc_decode_step launch; otherwise as
    kvc_seq_lengths + kvc_window_append + kvc_gqa_decode (split + merge)."""
    e2e_overlap = True   # a step of about 93 us
    bound = "hbm"
    fused = True

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None):
        import torch
        self.roofline_kernel = ("kvc_decode_step (fused step + merge)" if self.fused
                                else "kvc_gqa_decode (split + merge launches)")
        self.traffic_key = ("kvc_decode.cu",
                            "decode_split_kernel_fused" if self.fused else "decode_split_kernel")

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
        sk_host = torch.from_numpy((self.T - 1).astype(np.int32))
        self.q_host = synth.normal((B, Hq, 1, D), seed, 5)
        self.nk_host = synth.normal((B, Hkv, 1, D), seed, 3)
        self.nv_host = synth.normal((B, Hkv, 1, D), seed, 4)
        self.host_inputs = [sk_host, self.q_host, self.nk_host, self.nv_host]
        self.device_inputs = [t.to(dev) for t in self.host_inputs]
        self.sk, self.q, self.nk, self.nv = self.device_inputs
        cos, sin = synth.rope_cache(C, D, w.theta)
        self.rope = (cos.to(dev), sin.to(dev))
        e = self.e
        self.kernel_bytes = int(self.T.sum()) * Hkv * D * 2 * e + 2 * B * Hq * D * e
        self.append_bytes = 2 * 2 * B * Hkv * D * e
        self.bytes_per_step = self.kernel_bytes + self.append_bytes
        if self.fused:
            self.kernel_bytes = self.bytes_per_step
        self.tokens_per_step = B
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = torch.empty(B, Hq, 1, D, dtype=bf, device=dev)
        self.L = K.Lengths(B, dev)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        merge = 1 if K.kvc_gqa_decode_workspace_size(B, Hq, Hkv, C, D, K.KVC_BF16) > 256 else 0
        if self.fused:
            self.ws = K.decode_step_workspace(self.out, self.kc)
            self.launches_per_step = 1 + merge
        else:
            self.ws = K.decode_workspace(self.out, self.kc)
            self.launches_per_step = 3 + (1 if K.kvc_gqa_decode_workspace_size(
                B, Hq, Hkv, C, D, K.KVC_BF16) > 256 else 0)

    def step(self, i):
        K = self.K
        if self.fused:
            K.kvc_decode_step(self.out, self.q, self.kc, self.vc, self.nk, self.nv, self.sk,
                              lengths=self.L, rope=self.rope, workspace=self.ws, status=self.st)
            return
        K.kvc_seq_lengths(self.sk, 1, self.w.capacity, 0, out=self.L, status=self.st)
        K.kvc_window_append(self.kc, self.vc, self.nk, self.nv, self.L, 0, rope=self.rope,
                            status=self.st)
        self.kernel(i)

    def kernel(self, i):
        if self.fused:
            self.step(i)
            return
        self.K.kvc_gqa_decode(self.out, self.q, self.kc, self.vc, self.L, rope=self.rope,
                              workspace=self.ws, status=self.st)

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                "total_len": f"U[{w.total_lo},{w.total_hi}] after the append",
                "rope_theta": w.theta, "new_tokens": 1, "fused_step": self.fused,
                "l2": "inputs larger than L2 (~570 MB of K/V read per step)",
                "bytes_per_step": self.bytes_per_step}

    def oracle_sample(self, rows, sync=None):
        """Times the oracle's lengths + append + attention for the given batch
        rows; returns (seconds, algorithmic bytes of those rows)."""
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)
        kc = synth.bits(self.kc[rows].cpu()).copy()
        vc = synth.bits(self.vc[rows].cpu()).copy()
        nk, nv = synth.bits(self.nk_host[rows]), synth.bits(self.nv_host[rows])
        q = synth.bits(self.q_host[rows])
        cos, sin = (t.cpu().numpy() for t in self.rope)
        sk = (self.T[rows] - 1).astype(np.int32)
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        lens = oracle.seq_lengths(sk, 1, w.capacity, 0)
        oracle.window_append(kc, vc, nk, nv, lens, 0, cos, sin)
        oracle.gqa_attention(q, kc, vc, lens["cache_total"], lens["total_abs"], cos_cache=cos,
                             sin_cache=sin)
        dt = time.perf_counter() - t0
        e = self.e
        nbytes = (int(self.T[rows].sum()) * w.kv_heads * w.head_dim * 2 * e
                  + 2 * len(rows) * w.q_heads * w.head_dim * e
                  + 2 * 2 * len(rows) * w.kv_heads * w.head_dim * e)
        return dt, nbytes

    def metric(self):
        return METRIC, "GB/s"


def _cache_lengths(policy, T, S, C, W):
    """Lp, E, L per row for the byte accounting (include/kvc.h, kvc_seq_lengths)."""
    T = np.asarray(T, dtype=np.int64)

    def end(t):
        gap = C - W + 1
        return np.where(t <= C, t, t - gap * ((t - C + gap - 1) // gap))
    if policy == 2:
        Lp, L = end(T - S), end(T)
        return Lp, Lp + S - L, L
    # windowed and ring share the counts (a ring overwrites instead of moving)
    Lp = np.minimum(T - S, C)
    E = np.maximum(0, Lp + S - C)
    return Lp, E, Lp - E + S


class WindowDecode(Workload):
    """Sliding-window cache decode with in-place compaction, cycling over 16
    replica caches (one per model layer, 268 MB in all).  fused=True runs each
    step as one kvc_window_decode_step launch; otherwise as kvc_seq_lengths +
    kvc_window_append + kvc_gqa_decode."""
    bound = "hbm"
    replicas = 16
    fused = True
    spec = "WINDOW_DECODE"

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None, max_steps=4096):
        self.roofline_kernel = ("kvc_window_decode_step (fused step)" if self.fused
                                else "kvc_gqa_decode (window decode)")
        # the kernel's DRAM traffic depends on the layout and on the replicas
        layout = self.spec.lower() + ("_hot" if self.replicas == 1 else "")
        self.traffic_key = ("kvc_decode.cu", ("window_step_kernel@" if self.fused
                                              else "decode_split_kernel_window@") + layout)
        import torch

        from persistent_kv_cache_gb300 import synth
        self.torch = torch
        w = self.w = getattr(synth, self.spec)
        self.policy = w.extra.get("policy", 1)
        B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
        R = self.replicas
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.kc = torch.randn(R, B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.vc = torch.randn(R, B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.T0 = synth.randint(w.total_lo, w.total_hi + 1, (B,), seed, 1).numpy()
        # step i runs replica i % R at its (i // R)-th token
        n_rounds = max_steps // R + 2
        sk = np.stack([self.T0 + r - 1 for r in range(n_rounds)]).astype(np.int32)
        self.sk_all = torch.from_numpy(sk).to(dev)
        self.q_host = synth.normal((B, Hq, 1, D), seed, 5)
        self.nk_host = synth.normal((B, Hkv, 1, D), seed, 3)
        self.nv_host = synth.normal((B, Hkv, 1, D), seed, 4)
        self.host_inputs = [self.q_host, self.nk_host, self.nv_host]
        self.device_inputs = [t.to(dev) for t in self.host_inputs]
        self.q, self.nk, self.nv = self.device_inputs
        cos, sin = synth.rope_cache(int(self.T0.max()) + n_rounds + 1, D, w.theta)
        self.rope = (cos.to(dev), sin.to(dev))
        e = self.e
        # Algorithmic bytes of one step, averaged over the rounds the run
        # cycles through: the old rows read once (all resident rows when they
        # move, else only those the window sees), the moved rows written back
        # E rows lower, the new K/V rows read and written, q read, out
        # written.  The unfused decode kernel alone reads the visible rows.
        W = w.window
        T = self.T0.astype(np.int64)[None, :] + 1 + np.arange(n_rounds)[:, None]
        Lp, E, L = _cache_lengths(self.policy, T, 1, C, W)
        moves = (E > 0) & (self.policy != 3)
        moved = np.where(moves, L - 1, 0)
        old = np.where(moves, L - 1, np.minimum(L, W) - 1)
        row = Hkv * D * 2 * e
        self.bytes_per_step = int(round(float((old + moved).sum(axis=1).mean()) * row
                                        + 2 * 2 * B * Hkv * D * e + 2 * B * Hq * D * e))
        attn = int(round(float(np.minimum(L, W).sum(axis=1).mean()) * row)) + 2 * B * Hq * D * e
        self.kernel_bytes = self.bytes_per_step if self.fused else attn
        self.tokens_per_step = B
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = torch.empty(B, Hq, 1, D, dtype=bf, device=dev)
        self.ws = K.decode_workspace(self.out, self.kc[0])
        self.L = K.Lengths(B, dev)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches_per_step = 1 if self.fused else 3

    def step(self, i):
        K, w, R = self.K, self.w, self.replicas
        r = i % R
        if self.fused:
            K.kvc_window_decode_step(self.out, self.q, self.kc[r], self.vc[r], self.nk, self.nv,
                                     self.sk_all[i // R], w.window, lengths=self.L,
                                     rope=self.rope, status=self.st, windowed=self.policy)
            return
        if self.policy == 3:
            raise ValueError("the ring workload runs as the fused step")
        K.kvc_seq_lengths(self.sk_all[i // R], 1, w.capacity, self.policy,
                          local_window_size=w.window, out=self.L, status=self.st)
        K.kvc_window_append(self.kc[r], self.vc[r], self.nk, self.nv, self.L, self.policy,
                            rope=self.rope, status=self.st)
        self.kernel(i)

    def kernel(self, i):
        if self.fused:
            self.step(i)
            return
        r = i % self.replicas
        self.K.kvc_gqa_decode(self.out, self.q, self.kc[r], self.vc[r], self.L,
                              local_window_size=self.w.window, rope=self.rope, workspace=self.ws,
                              status=self.st)

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                "window": w.window, "start_total": f"U[{w.total_lo},{w.total_hi}]",
                "replica_caches": self.replicas, "new_tokens": 1, "fused_step": self.fused,
                "layout": {1: "compact every step", 2: "drifting", 3: "ring"}[self.policy],
                "l2": ("16 replica caches cycled (268 MB > L2)" if self.replicas > 1
                       else "one cache, L2-resident (hot)"),
                "bytes_per_step": self.bytes_per_step}

    def oracle_sample(self, rows, sync=None):
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)
        kc = synth.bits(self.kc[0][rows].cpu()).copy()
        vc = synth.bits(self.vc[0][rows].cpu()).copy()
        cos, sin = (t.cpu().numpy() for t in self.rope)
        sk = (self.T0[rows]).astype(np.int32)  # the first step: T = T0 + 1
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        lens = oracle.seq_lengths(sk, 1, w.capacity, self.policy, w.window)
        if self.policy == 3:
            oracle.ring_append(kc, vc, synth.bits(self.nk_host[rows]),
                               synth.bits(self.nv_host[rows]), lens["past_abs"], cos, sin)
            oracle.ring_attention(synth.bits(self.q_host[rows]), kc, vc, lens["total_abs"],
                                  w.window, cos_cache=cos, sin_cache=sin)
        else:
            oracle.window_append(kc, vc, synth.bits(self.nk_host[rows]),
                                 synth.bits(self.nv_host[rows]), lens, 1, cos, sin)
            oracle.gqa_attention(synth.bits(self.q_host[rows]), kc, vc, lens["cache_total"],
                                 lens["total_abs"], window=w.window, cos_cache=cos,
                                 sin_cache=sin)
        dt = time.perf_counter() - t0
        return dt, self.bytes_per_step * len(rows) / w.batch

    def metric(self):
        return "window decode: achieved HBM GB/s, decode steps/s", "GB/s"


class WindowPrefill(Workload):
    """Windowed chunked prefill through the C + S staging cache."""
    e2e_overlap = True   # steps of 0.15 to 1 ms
    roofline_kernel = "kvc_gqa_prefill_chunk (tcgen05)"
    bound = "tensor"
    slack = 0  # rows of capacity beyond the window (C = W + slack)

    def __init__(self, dev, seed=0, with_kernels=True, chunk=2048):
        import torch

        from persistent_kv_cache_gb300 import synth
        self.torch = torch
        w = self.w = synth.WINDOW_PREFILL
        S = self.S = int(chunk or 2048)
        # the kernel's DRAM traffic depends on the chunk (grid and reuse)
        self.traffic_key = ("kvc_prefill.cu", f"prefill_tc_kernel@chunk{S}")
        B, Hq, Hkv, D, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.window
        C = self.C = w.capacity + self.slack
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.kc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.vc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.ks = torch.empty(B, Hkv, C + S, D, device=dev, dtype=bf)
        self.vs = torch.empty_like(self.ks)
        self.P = synth.randint(w.total_lo, w.total_hi + 1, (B,), seed, S).numpy()
        sk_host = torch.from_numpy((self.P + S - 1).astype(np.int32))
        self.q_host = synth.normal((B, Hq, S, D), seed, 5)
        self.nk_host = synth.normal((B, Hkv, S, D), seed, 3)
        self.nv_host = synth.normal((B, Hkv, S, D), seed, 4)
        self.host_inputs = [sk_host, self.q_host, self.nk_host, self.nv_host]
        self.device_inputs = [t.to(dev) for t in self.host_inputs]
        self.sk, self.q, self.nk, self.nv = self.device_inputs
        cos, sin = synth.rope_cache(int(self.P.max()) + S + 1, D, w.theta)
        self.rope = (cos.to(dev), sin.to(dev))
        e = self.e
        Lp = np.minimum(self.P, C)
        E = np.maximum(0, Lp + S - C)
        L = Lp - E + S
        i = np.arange(S)
        vis = np.minimum(Lp[:, None] + i[None, :] + 1, W)           # [B, S]
        self.flops = 4 * Hq * D * int(vis.sum())                     # QK^T and PV, visible
        qb = 128 // (Hq // Hkv)
        issued = 0
        for b in range(B):
            for q0 in range(0, S, qb):
                ql = min(S - 1, q0 + qb - 1)
                hi = Lp[b] + ql
                lo = max(0, Lp[b] + q0 - W + 1)
                issued += (hi - lo + 128) // 128
        self.issued_flops = int(issued) * Hkv * 4 * 128 * 128 * D
        self.stage_bytes = int(2 * Hkv * D * e * int((2 * Lp + 2 * L).sum()))  # seed + copy-back r+w
        self.kernel_bytes = 2 * B * Hq * S * D * e + 2 * Hkv * D * e * int((Lp + S).sum())
        self.bytes_per_step = self.stage_bytes + self.kernel_bytes + 2 * 2 * B * Hkv * S * D * e
        self.tokens_per_step = B * S
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = torch.empty(B, Hq, S, D, dtype=bf, device=dev)
        self.L = K.Lengths(B, dev)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        # the KV split's partials (small chunks only: the grid is under a wave)
        self.pws = K.prefill_workspace(self.out, self.ks, w.window)
        self.launches_per_step = 5 + (1 if self.pws is not None else 0)

    def step(self, i):
        K, w = self.K, self.w
        K.kvc_seq_lengths(self.sk, self.S, self.C, 1, local_window_size=w.window, out=self.L,
                          status=self.st)
        K.kvc_window_append(self.kc, self.vc, self.nk, self.nv, self.L, 1, K.KVC_APPEND,
                            self.ks, self.vs, rope=self.rope, status=self.st)
        self.kernel(i)
        K.kvc_window_append(self.kc, self.vc, None, None, self.L, 1, K.KVC_COPY_BACK, self.ks,
                            self.vs, rope=self.rope, status=self.st)

    def kernel(self, i):
        self.K.kvc_gqa_prefill_chunk(self.out, self.q, self.ks, self.vs, self.L,
                                     local_window_size=self.w.window, rope=self.rope,
                                     status=self.st, workspace=self.pws)

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": self.C,
                "window": w.window, "past_len": f"U[{w.total_lo},{w.total_hi}]",
                "chunk": self.S, "visible_flops_per_step": self.flops,
                "kv_split": (getattr(self, "pws", None) is not None
                             if hasattr(self, "K") else None),
                "issued_flops_per_step": self.issued_flops,
                "l2": "stage + cache ~1 GB per step > L2",
                "bytes_per_step": self.bytes_per_step}

    def oracle_sample(self, rows, sync=None):
        """One query of each sampled batch row (the chunk's last), all heads."""
        import oracle
        from persistent_kv_cache_gb300 import synth
        w, S = self.w, self.S
        rows = list(rows)
        kc = synth.bits(self.kc[rows].cpu()).copy()
        vc = synth.bits(self.vc[rows].cpu()).copy()
        cos, sin = (t.cpu().numpy() for t in self.rope)
        sk = (self.P[rows] + S - 1).astype(np.int32)
        ks = np.zeros((len(rows), w.kv_heads, self.C + S, w.head_dim), np.uint16)
        vs = np.zeros_like(ks)
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        lens = oracle.seq_lengths(sk, S, self.C, 1)
        oracle.window_append(kc, vc, synth.bits(self.nk_host[rows]),
                             synth.bits(self.nv_host[rows]), lens, 1, cos, sin, ks, vs)
        q = np.ascontiguousarray(synth.bits(self.q_host[rows])[:, :, S - 1:S])
        oracle.gqa_attention(q, ks, vs, (lens["cache_past"] + S).astype(np.int32),
                             lens["total_abs"], window=w.window, cos_cache=cos, sin_cache=sin)
        dt = time.perf_counter() - t0
        Lp = np.minimum(self.P[rows], self.C)
        fl = 4 * w.q_heads * w.head_dim * int(np.minimum(Lp + S, w.window).sum())
        return dt, fl

    def metric(self):
        return "windowed chunked prefill: tcgen05 TFLOP/s (visible), tokens/s", "TFLOP/s"


class WindowPrefillInplace(WindowPrefill):
    """The windowed chunked-prefill step with the stage held in the cache's
    own rows (kvc_window_append_inplace): the cache lives in rows [0, C) of
    a buffer of C + S rows per head, the new rows are written after it, the
    attention runs there, and the copy-back is an in-place shift (no seed
    copy)."""

    def __init__(self, dev, seed=0, with_kernels=True, chunk=2048):
        super().__init__(dev, seed=seed, with_kernels=with_kernels, chunk=chunk)
        import torch
        w, S, e = self.w, self.S, self.e
        B, Hkv, C, D = w.batch, w.kv_heads, w.capacity, w.head_dim
        self.rows_k = torch.empty(B, Hkv, C + S, D, device=dev, dtype=torch.bfloat16)
        self.rows_v = torch.empty_like(self.rows_k)
        self.rows_k[:, :, :C] = self.kc
        self.rows_v[:, :, :C] = self.vc
        del self.ks, self.vs
        Lp = np.minimum(self.P, C)
        E = np.maximum(0, Lp + S - C)
        L = Lp - E + S
        # the shift reads and writes L rows of every (K/V, head) where rows evict
        self.stage_bytes = int(2 * Hkv * D * e * int((2 * L * (E > 0)).sum()))
        self.bytes_per_step = self.stage_bytes + self.kernel_bytes + 2 * 2 * B * Hkv * S * D * e
        if with_kernels:
            self.launches_per_step = 4 + (1 if self.pws is not None else 0)

    def step(self, i):
        K, w = self.K, self.w
        K.kvc_seq_lengths(self.sk, self.S, w.capacity, 1, local_window_size=w.window, out=self.L,
                          status=self.st)
        K.kvc_window_append_inplace(self.rows_k, self.rows_v, self.nk, self.nv, self.L,
                                    w.capacity, 1, K.KVC_APPEND, rope=self.rope, status=self.st)
        self.kernel(i)
        K.kvc_window_append_inplace(self.rows_k, self.rows_v, None, None, self.L, w.capacity, 1,
                                    K.KVC_COPY_BACK, new_tokens=self.S, rope=self.rope,
                                    status=self.st)

    def kernel(self, i):
        self.K.kvc_gqa_prefill_chunk(self.out, self.q, self.rows_k, self.rows_v, self.L,
                                     local_window_size=self.w.window, rope=self.rope,
                                     status=self.st, workspace=self.pws)

    def config(self):
        c = super().config()
        c["workload"] = self.w.name + "-inplace-stage"
        c["l2"] = "cache + stage rows ~0.6 GB per step > L2"
        return c


class WindowPrefillHazard(WindowPrefill):
    """The windowed chunked-prefill step as one kvc_window_prefill_step call:
    only the batch rows whose eviction the chunk would see use the stage,
    and those only for their new rows and the 127 old rows below them (the
    attention reads older tiles from the cache, and the copy-back is one
    in-place move of the window plus the new rows); a row that evicts
    nothing (its cache not yet full) appends in place and its attention
    reads the cache.  The timed kernel is the whole call."""
    roofline_kernel = "kvc_window_prefill_step (the whole call)"

    def __init__(self, dev, seed=0, with_kernels=True, chunk=64):
        super().__init__(dev, seed=seed, with_kernels=with_kernels, chunk=chunk)
        w, S, e, C = self.w, self.S, self.e, self.C
        B, Hkv, D, W = w.batch, w.kv_heads, w.head_dim, w.window
        self.traffic_key = ("kvc_prefill.cu", f"window_prefill_step@c{C}-chunk{S}")
        Lp = np.minimum(self.P, C)
        E = np.maximum(0, Lp + S - C)
        L = Lp - E + S
        staged = (E > 0) & (E > Lp - W + 1)
        moved = (E > 0) & ~staged
        self.n_staged, self.n_moved = int(staged.sum()), int(moved.sum())
        # rows read + written: a staged row seeds the 127 old rows below its
        # new ones, moves its kept old rows down after the attention and
        # copies its kept new rows back; a row that moves in place moves its
        # Lp - E old rows
        kept_old = np.maximum(Lp - E, 0)
        kept_new = Lp + S - np.maximum(E, Lp)
        staged_rows = np.minimum(Lp, 127) + kept_old + kept_new
        self.stage_bytes = int(2 * Hkv * D * e * int((staged * 2 * staged_rows).sum() +
                                                      (moved * 2 * (Lp - E)).sum()))
        self.bytes_per_step = self.stage_bytes + self.kernel_bytes + 2 * 2 * B * Hkv * S * D * e
        self.kernel_bytes = self.bytes_per_step
        if with_kernels:
            self.launches_per_step = 6 + (1 if self.pws is not None else 0)

    def step(self, i):
        K, w = self.K, self.w
        K.kvc_seq_lengths(self.sk, self.S, self.C, 1, local_window_size=w.window, out=self.L,
                          status=self.st)
        self.kernel(i)

    def kernel(self, i):
        self.K.kvc_window_prefill_step(self.out, self.q, self.kc, self.vc, self.nk, self.nv,
                                       self.L, 1, self.w.window, self.ks, self.vs,
                                       rope=self.rope, status=self.st, workspace=self.pws)

    def config(self):
        c = super().config()
        c["workload"] = self.w.name + ("-hazard-staging" if not self.slack else
                                       f"-c{self.C}-hazard-staging")
        c["rows_staged"], c["rows_moved_in_place"] = self.n_staged, self.n_moved
        return c


class WindowPrefillHazardSlack(WindowPrefillHazard):
    """The same with C = W + 64: once a row's cache is full, a chunk of 64
    evicts 64 rows that none of its queries sees (64 <= Lp - W + 1), so no
    row needs the stage: the old rows move down in place and the attention
    reads the cache."""
    slack = 64


class Scatter(Workload):
    """TensorScatter circular on one (16, 8, 4096, 128) bf16 cache: in place,
    or (functional) into a separate present cache."""
    bound = "hbm"
    in_place = True
    out_double = False  # the result read back is a slice of present

    def __init__(self, dev, seed=0, with_kernels=True, chunk=64, max_steps=4096):
        import torch

        from persistent_kv_cache_gb300 import synth
        self.torch = torch
        self.roofline_kernel = ("kvc_tensor_scatter (in place)" if self.in_place
                                else "kvc_tensor_scatter (functional: one-pass scatter_copy_kernel)")
        # DRAM traffic per call depends on the number of update rows
        self.traffic_key = ("kvc_scatter.cu",
                            ("scatter_rows_kernel" if self.in_place else "scatter_functional")
                            + f"@chunk{int(chunk or 64)}")
        w = self.w = synth.SCATTER
        S = self.S = int(chunk or 64)
        shape = (w.batch, w.heads, w.max_seq, w.head_dim)
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        self.cache = torch.randn(*shape, generator=g, device=dev, dtype=torch.bfloat16)
        self.present = self.cache if self.in_place else torch.empty_like(self.cache)
        self.upd_host = synth.normal((w.batch, w.heads, S, w.head_dim), seed, 2)
        self.n_wi = max_steps + 64
        self.wi_all = synth.randint(0, w.max_seq, (self.n_wi, w.batch), seed, 3).to(dev)
        wi_host = synth.randint(0, w.max_seq, (w.batch,), seed, 4)
        self.host_inputs = [self.upd_host, wi_host]
        self.device_inputs = [t.to(dev) for t in self.host_inputs]
        self.upd, self.wi = self.device_inputs
        self.kernel_bytes = 2 * w.batch * w.heads * S * w.head_dim * self.e + 8 * w.batch
        if not self.in_place:
            # every present row written once, from past or from the update
            self.kernel_bytes = 2 * self.cache.numel() * self.e + 8 * w.batch
        self.bytes_per_step = self.kernel_bytes
        self.tokens_per_step = w.batch * S
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = self.present[:1, :1, :S]  # the e2e result read back: one slice
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        self.launches_per_step = 1

    def step(self, i):
        self.K.kvc_tensor_scatter(self.present, self.cache, self.upd, self.wi_all[i % self.n_wi],
                                  mode=self.K.KVC_CIRCULAR, status=self.st)

    def kernel(self, i):
        self.step(i)

    def extra_measure(self):
        """Per-launch floor of one graph node: the same call on a (1, 1, 16, 8)
        float32 cache with one update row, 256 nodes replayed as one graph."""
        if not self.in_place:
            return {}
        torch, K = self.torch, self.K
        dev = self.cache.device
        tiny = torch.zeros(1, 1, 16, 8, device=dev)
        upd = torch.ones(1, 1, 1, 8, device=dev)
        wi = torch.zeros(1, dtype=torch.int64, device=dev)
        n = 256
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(n):
                K.kvc_tensor_scatter(tiny, tiny, upd, wi, mode=K.KVC_CIRCULAR)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        return {"graph_node_floor_us": e0.elapsed_time(e1) * 1e3 / n}

    def config(self):
        w = self.w
        return {"workload": w.name + ("" if self.in_place else "-functional"),
                "shape": [w.batch, w.heads, w.max_seq, w.head_dim],
                "axis": -2, "mode": "circular", "update_len": self.S, "in_place": self.in_place,
                "l2": ("launch-bound; 128 MiB cache, updates touch 32 KiB x S per step"
                       if self.in_place else "past and present 128 MiB each (> L2)"),
                "bytes_per_step": self.bytes_per_step}

    def oracle_sample(self, rows, sync=None):
        import oracle
        from persistent_kv_cache_gb300 import synth
        cache = synth.bits(self.cache.cpu()).copy()
        upd = synth.bits(self.upd_host)
        wi = self.wi_all[0].cpu().numpy()
        n = 20 if self.in_place else 2
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        for _ in range(n):
            oracle.tensor_scatter(cache, upd, wi, mode=oracle.CIRCULAR,
                                  out=cache if self.in_place else None)
        return time.perf_counter() - t0, n * self.bytes_per_step

    def metric(self):
        if self.in_place:
            return "TensorScatter circular in place: GB/s of update bytes, steps/s", "GB/s"
        return "TensorScatter circular functional: GB/s (whole cache), steps/s", "GB/s"


class ScatterFunctional(Scatter):
    in_place = False


class WindowDecodeUnfused(WindowDecode):
    fused = False


class ContigDecodeUnfused(ContigDecode):
    fused = False


class PagedDecode(ContigDecode):
    """The contiguous decode workload in 64-row pages: K/V pools of
    B * C / 64 pages in a random order, a per-row page table; one step =
    kvc_seq_lengths + kvc_paged_append + kvc_gqa_decode_paged (+ merge)."""
    fused = False
    page_size = 64

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None):
        import torch
        super().__init__(dev, seed=seed, with_kernels=with_kernels, chunk=chunk)
        self.roofline_kernel = "kvc_gqa_decode_paged (split + merge launches)"
        self.traffic_key = ("kvc_decode.cu", "decode_split_kernel_paged")
        w = self.w
        B, Hkv, D, C = w.batch, w.kv_heads, w.head_dim, w.capacity
        P = self.page_size
        max_pages = C // P
        rng = np.random.default_rng(1000 + seed)
        self.table_host = rng.permutation(B * max_pages).reshape(B, max_pages).astype(np.int32)
        table = torch.from_numpy(self.table_host).to(dev)
        # the same rows as the contiguous caches, moved into the shuffled pages
        kp = torch.empty(B * max_pages, Hkv, P, D, dtype=self.kc.dtype, device=dev)
        vp = torch.empty_like(kp)
        idx = table.reshape(-1).long()
        kp[idx] = self.kc.reshape(B, Hkv, max_pages, P, D).transpose(1, 2).reshape(-1, Hkv, P, D)
        vp[idx] = self.vc.reshape(B, Hkv, max_pages, P, D).transpose(1, 2).reshape(-1, Hkv, P, D)
        self.kc, self.vc, self.table = kp, vp, table
        # (the workspace from the contiguous setup has the right size)

    def step(self, i):
        K = self.K
        K.kvc_seq_lengths(self.sk, 1, self.w.capacity, 0, out=self.L, status=self.st)
        K.kvc_paged_append(self.kc, self.vc, self.nk, self.nv, self.table, self.L,
                           rope=self.rope, status=self.st)
        self.kernel(i)

    def kernel(self, i):
        self.K.kvc_gqa_decode_paged(self.out, self.q, self.kc, self.vc, self.table, self.L,
                                    rope=self.rope, workspace=self.ws, status=self.st)

    def config(self):
        c = super().config()
        c.update({"workload": self.w.name + "-paged64", "page_size": self.page_size,
                  "pages": int(self.table_host.size), "page_order": "random permutation"})
        return c

    def oracle_sample(self, rows, sync=None):
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)[:2]
        P = self.page_size
        tab = self.table_host[rows]
        used = np.unique(tab)
        remap = {int(p): j for j, p in enumerate(used)}
        kp = synth.bits(self.kc[torch_index(used)].cpu()).copy()
        vp = synth.bits(self.vc[torch_index(used)].cpu()).copy()
        tab_local = np.vectorize(remap.get)(tab).astype(np.int32)
        nk, nv = synth.bits(self.nk_host[rows]), synth.bits(self.nv_host[rows])
        q = synth.bits(self.q_host[rows])
        cos, sin = (t.cpu().numpy() for t in self.rope)
        T = self.T[rows]
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        oracle.paged_append(kp, vp, tab_local, P, nk, nv, T - 1, cos, sin)
        oracle.paged_attention(q, kp, vp, tab_local, P, T, T, cos_cache=cos, sin_cache=sin)
        dt = time.perf_counter() - t0
        nbytes = (int(T.sum()) * w.kv_heads * w.head_dim * 2 * self.e
                  + 2 * len(rows) * w.q_heads * w.head_dim * self.e
                  + 2 * 2 * len(rows) * w.kv_heads * w.head_dim * self.e)
        return dt, nbytes


class PagedDecodeQ8(PagedDecode):
    """The paged decode workload with every full page below a row's newest
    one held as int8 (affine, scale 0.04, zero point 0 for K and V; the
    newest page, where the step appends, stays 16-bit): one step =
    kvc_seq_lengths + kvc_paged_append + kvc_gqa_decode_paged_q (+ merge)."""
    e2e_overlap = False  # a step of about 68 us: the plain loop is faster
    k_scale = v_scale = 0.04

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None):
        import torch
        super().__init__(dev, seed=seed, with_kernels=with_kernels, chunk=chunk)
        self.roofline_kernel = "kvc_gqa_decode_paged_q (split + merge launches)"
        self.traffic_key = ("kvc_decode.cu", "decode_split_kernel_paged_q")
        w, P, e = self.w, self.page_size, self.e
        B, Hq, Hkv, D = w.batch, w.q_heads, w.kv_heads, w.head_dim
        # the rows of each sequence that live in int8 pages (all pages before
        # the one holding row T - 1, which the step appends to)
        full = (self.T - 1) // P
        self.q8_rows = full * P
        n16 = self.T - self.q8_rows
        self.kernel_bytes = (int(self.q8_rows.sum()) * Hkv * D * 2
                             + int(n16.sum()) * Hkv * D * 2 * e + 2 * B * Hq * D * e)
        self.bytes_per_step = self.kernel_bytes + self.append_bytes
        src, dst = [], []
        self.qtab_host = self.table_host.copy()
        for b in range(B):
            for j in range(int(full[b])):
                src.append(int(self.table_host[b, j]))
                self.qtab_host[b, j] = 0x40000000 | len(dst)
                dst.append(len(dst))
        self.n_q_pages = max(1, len(dst))
        if not with_kernels:
            return
        K = self.K
        self.qk = torch.empty(self.n_q_pages, Hkv, P, D, dtype=torch.uint8, device=dev)
        self.qv = torch.empty_like(self.qk)
        self.qp = torch.zeros(self.n_q_pages, 4, dtype=torch.float32, device=dev)
        if src:
            K.kvc_quantize_pages(self.kc, self.vc, self.qk, self.qv,
                                 torch.tensor(src, dtype=torch.int32, device=dev),
                                 torch.tensor(dst, dtype=torch.int32, device=dev), self.qp,
                                 self.k_scale, 0, False, self.v_scale, 0, False, status=self.st)
        self.qtable = torch.from_numpy(self.qtab_host).to(dev)
        torch.cuda.synchronize()

    def kernel(self, i):
        self.K.kvc_gqa_decode_paged_q(self.out, self.q, self.kc, self.vc, self.qk, self.qv,
                                      self.qp, self.qtable, self.L, rope=self.rope,
                                      workspace=self.ws, status=self.st)

    def config(self):
        c = super().config()
        c.update({"workload": self.w.name + "-paged64-int8",
                  "int8_pages": int(self.n_q_pages), "int8_scale": self.k_scale,
                  "int8_rows_fraction": float(self.q8_rows.sum() / self.T.sum())})
        return c

    def oracle_sample(self, rows, sync=None):
        """The oracle's append + attention over the sampled rows, with their
        int8 pages quantized by the oracle from the same 16-bit pages (once,
        before the timed part: quantizing is not part of a step)."""
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)[:2]
        P = self.page_size
        kp = synth.bits(self.kc.cpu()).copy()
        vp = synth.bits(self.vc.cpu()).copy()
        tab16 = self.table_host[rows]
        T = self.T[rows]
        full = (T - 1) // P
        n_q = max(1, int(full.sum()))
        qk = np.zeros((n_q, w.kv_heads, P, w.head_dim), np.uint8)
        qv = np.zeros_like(qk)
        qp = np.zeros((n_q, 4), np.float32)
        tab = tab16.copy()
        n = 0
        for i in range(len(rows)):
            for j in range(int(full[i])):
                qk[n], zk = oracle.quantize_page(kp[tab16[i, j]], self.k_scale, 0)
                qv[n], zv = oracle.quantize_page(vp[tab16[i, j]], self.v_scale, 0)
                qp[n] = (self.k_scale, zk, self.v_scale, zv)
                tab[i, j] = oracle.PAGE_QUANT | n
                n += 1
        nk, nv = synth.bits(self.nk_host[rows]), synth.bits(self.nv_host[rows])
        q = synth.bits(self.q_host[rows])
        cos, sin = (t.cpu().numpy() for t in self.rope)
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        oracle.paged_append(kp, vp, tab16, P, nk, nv, T - 1, cos, sin)
        oracle.paged_attention_q(q, kp, vp, qk, qv, qp, tab, P, T, T, cos_cache=cos,
                                 sin_cache=sin)
        dt = time.perf_counter() - t0
        q8 = self.q8_rows[rows]
        nbytes = (int(q8.sum()) * w.kv_heads * w.head_dim * 2
                  + int((T - q8).sum()) * w.kv_heads * w.head_dim * 2 * self.e
                  + 2 * len(rows) * w.q_heads * w.head_dim * self.e
                  + 2 * 2 * len(rows) * w.kv_heads * w.head_dim * self.e)
        return dt, nbytes


def torch_index(a):
    import torch
    return torch.from_numpy(np.asarray(a, dtype=np.int64))


class WindowDecodeHot(WindowDecode):
    replicas = 1


class WindowDecodeDrift(WindowDecode):
    spec = "WINDOW_DECODE_DRIFT"


class WindowDecodeRing(WindowDecode):
    spec = "WINDOW_DECODE_RING"


class RingDecode256(Workload):
    """One-token decode at head_dim 256: the windowed-prefill workload's heads
    (8 x 16/8 heads, W = 4096) as a ring of C = 4096 slots, past lengths
    U[1, 20000]; one step = one kvc_decode_step (lengths, RoPE append of the
    new row, split decode) plus the split merge."""
    bound = "hbm"
    roofline_kernel = "kvc_decode_step, ring, head_dim 256 (split + merge)"
    traffic_key = ("kvc_decode.cu", "decode_split_kernel_fused@ring_d256")

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None):
        import torch

        from persistent_kv_cache_gb300 import synth
        self.torch = torch
        w = self.w = synth.WINDOW_DECODE_256
        B, Hq, Hkv, D, C, W = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity, w.window
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        bf = torch.bfloat16
        self.kc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.vc = torch.randn(B, Hkv, C, D, generator=g, device=dev, dtype=bf)
        self.T = synth.randint(w.total_lo, w.total_hi + 1, (B,), seed, 256).numpy()
        sk_host = torch.from_numpy((self.T - 1).astype(np.int32))
        self.q_host = synth.normal((B, Hq, 1, D), seed, 5)
        self.nk_host = synth.normal((B, Hkv, 1, D), seed, 3)
        self.nv_host = synth.normal((B, Hkv, 1, D), seed, 4)
        self.host_inputs = [sk_host, self.q_host, self.nk_host, self.nv_host]
        self.device_inputs = [t.to(dev) for t in self.host_inputs]
        self.sk, self.q, self.nk, self.nv = self.device_inputs
        cos, sin = synth.rope_cache(int(self.T.max()) + 1, D, w.theta)
        self.rope = (cos.to(dev), sin.to(dev))
        e = self.e
        # the visible rows (the newest min(T, C, W) positions) of K and V,
        # q read, out written, the new K/V row read and written
        vis = np.minimum(np.minimum(self.T, C), W)
        self.bytes_per_step = (int(vis.sum()) * Hkv * D * 2 * e + 2 * B * Hq * D * e
                               + 2 * 2 * B * Hkv * D * e)
        self.kernel_bytes = self.bytes_per_step
        self.tokens_per_step = B
        if not with_kernels:
            return
        from persistent_kv_cache_gb300 import kvc as K
        self.K = K
        self.out = torch.empty(B, Hq, 1, D, dtype=bf, device=dev)
        self.L = K.Lengths(B, dev)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = K.decode_step_workspace(self.out, self.kc)
        merge = 1 if K.kvc_gqa_decode_workspace_size(B, Hq, Hkv, C, D, K.KVC_BF16) > 256 else 0
        self.launches_per_step = 1 + merge

    def step(self, i):
        self.K.kvc_decode_step(self.out, self.q, self.kc, self.vc, self.nk, self.nv, self.sk,
                               self.w.window, lengths=self.L, rope=self.rope, workspace=self.ws,
                               status=self.st, windowed=self.K.KVC_RING)

    def kernel(self, i):
        self.step(i)

    def config(self):
        w = self.w
        return {"workload": w.name, "batch": w.batch, "q_heads": w.q_heads,
                "kv_heads": w.kv_heads, "head_dim": w.head_dim, "capacity": w.capacity,
                "window": w.window, "layout": "ring", "total_len": f"U[{w.total_lo},{w.total_hi}]",
                "rope_theta": w.theta, "new_tokens": 1, "fused_step": True,
                "l2": "inputs larger than L2 (~268 MB of K/V read per step)",
                "bytes_per_step": self.bytes_per_step}

    def oracle_sample(self, rows, sync=None):
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)
        kc = synth.bits(self.kc[rows].cpu()).copy()
        vc = synth.bits(self.vc[rows].cpu()).copy()
        cos, sin = (t.cpu().numpy() for t in self.rope)
        T = self.T[rows]
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        oracle.ring_append(kc, vc, synth.bits(self.nk_host[rows]), synth.bits(self.nv_host[rows]),
                           T - 1, cos, sin)
        oracle.ring_attention(synth.bits(self.q_host[rows]), kc, vc, T, w.window, cos_cache=cos,
                              sin_cache=sin)
        dt = time.perf_counter() - t0
        return dt, self.bytes_per_step * len(rows) / w.batch

    def metric(self):
        return "ring decode, head_dim 256: achieved HBM GB/s, decode steps/s", "GB/s"


class WindowDecode256(RingDecode256):
    """One-token steps on the windowed-prefill workload's cache kept
    compacted (C = W = 4096, head_dim 256, 8 x 16/8 heads, past lengths
    U[1, 20000]): lengths, the in-place compaction of the whole window by one
    row plus the RoPE append (a cluster of eight CTAs per slice), then the
    split decode and merge.  The roofline kernel is the compaction."""
    e2e_overlap = True   # a step of about 112 us
    roofline_kernel = "kvc_window_append, S = 1 (cluster compaction)"
    traffic_key = ("kvc_cache.cu", "compact_cluster_kernel@window_d256")

    def __init__(self, dev, seed=0, with_kernels=True, chunk=None):
        super().__init__(dev, seed=seed, with_kernels=with_kernels, chunk=chunk)
        w, e = self.w, self.e
        B, Hq, Hkv, D, C = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.capacity
        Lp, E, L = _cache_lengths(1, self.T, 1, C, w.window)
        row = Hkv * D * 2 * e
        # compaction: the Lp - E surviving rows read and written where rows
        # evict, the new row read and written; decode: the L visible rows,
        # q read and out written
        self.kernel_bytes = int((2 * (Lp - E) * (E > 0)).sum()) * row + 2 * B * row
        self.bytes_per_step = self.kernel_bytes + int(L.sum()) * row + 2 * B * Hq * D * e
        if with_kernels:
            self.ws = self.K.decode_workspace(self.out, self.kc)
            self.launches_per_step = 3 + (1 if self.ws.numel() > 256 else 0)

    def step(self, i):
        K, w = self.K, self.w
        K.kvc_seq_lengths(self.sk, 1, w.capacity, K.KVC_WINDOWED, local_window_size=w.window,
                          out=self.L, status=self.st)
        self.kernel(i)
        K.kvc_gqa_decode(self.out, self.q, self.kc, self.vc, self.L, local_window_size=w.window,
                         rope=self.rope, workspace=self.ws, status=self.st)

    def kernel(self, i):
        self.K.kvc_window_append(self.kc, self.vc, self.nk, self.nv, self.L, self.K.KVC_WINDOWED,
                                 rope=self.rope, status=self.st)

    def config(self):
        c = super().config()
        c.update({"workload": "window-decode-bf16-b8-h16kv8-d256-c4096-w4096",
                  "layout": "compact every step", "fused_step": False,
                  "l2": "~805 MB moved and read per step > L2"})
        return c

    def oracle_sample(self, rows, sync=None):
        import oracle
        from persistent_kv_cache_gb300 import synth
        w = self.w
        rows = list(rows)
        kc = synth.bits(self.kc[rows].cpu()).copy()
        vc = synth.bits(self.vc[rows].cpu()).copy()
        cos, sin = (t.cpu().numpy() for t in self.rope)
        sk = (self.T[rows] - 1).astype(np.int32)
        if sync is not None:
            sync()  # the threads of a parallel sample start together
        t0 = time.perf_counter()
        lens = oracle.seq_lengths(sk, 1, w.capacity, 1, w.window)
        oracle.window_append(kc, vc, synth.bits(self.nk_host[rows]),
                             synth.bits(self.nv_host[rows]), lens, 1, cos, sin)
        oracle.gqa_attention(synth.bits(self.q_host[rows]), kc, vc, lens["cache_total"],
                             lens["total_abs"], window=w.window, cos_cache=cos, sin_cache=sin)
        dt = time.perf_counter() - t0
        return dt, self.bytes_per_step * len(rows) / w.batch

    def metric(self):
        return "window decode, head_dim 256, C = W = 4096: achieved HBM GB/s, steps/s", "GB/s"


WORKLOADS = {"contig-decode": ContigDecode, "contig-decode-unfused": ContigDecodeUnfused,
             "ring-decode-d256": RingDecode256, "window-decode-d256": WindowDecode256,
             "paged-decode": PagedDecode,
             "window-decode": WindowDecode,
             "window-decode-unfused": WindowDecodeUnfused,
             "window-decode-drift": WindowDecodeDrift, "window-decode-ring": WindowDecodeRing,
             "window-decode-hot": WindowDecodeHot, "window-prefill": WindowPrefill,
             "window-prefill-inplace": WindowPrefillInplace,
             "window-prefill-hazard": WindowPrefillHazard,
             "window-prefill-hazard-slack": WindowPrefillHazardSlack,
             "paged-decode-int8": PagedDecodeQ8,
             "scatter-functional": ScatterFunctional,
             "scatter": Scatter}


def oracle_threads(wl, rows, threads, min_wall, max_wall):
    """The oracle over `rows` on `threads` host threads (rows dealt round
    robin, one chunk a thread; the oracle's C calls release the GIL), the
    threads starting their timed regions together.  Repeats until `min_wall`
    seconds of wall time (at most about `max_wall`); returns (wall seconds,
    units of work, repetitions, threads used)."""
    import threading
    from concurrent.futures import ThreadPoolExecutor
    rows = list(rows)
    chunks = [c for c in (rows[i::threads] for i in range(threads)) if c]
    n = len(chunks)
    wall = amount = 0.0
    reps = 0
    with ThreadPoolExecutor(max_workers=n) as ex:
        while wall < min_wall and (reps == 0 or wall + wall / reps < max_wall):
            bar = threading.Barrier(n)
            res = list(ex.map(lambda c: wl.oracle_sample(c, sync=bar.wait), chunks))
            wall += max(r[0] for r in res)
            amount += sum(r[1] for r in res)
            reps += 1
    return wall, amount, reps, n


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def source_digest(path):
    """sha256 of a CUDA source's code: comments removed and whitespace
    collapsed, so that an edit of comments alone keeps a capture valid."""
    text = open(path, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256(" ".join(text.split()).encode()).hexdigest()


def kernel_traffic(key):
    """DRAM bytes per launch recorded from an ncu capture, or None when the
    kernel's source code changed since."""
    kernel_file, name = key
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[name]
        src = os.path.join(ROOT, "persistent_kv_cache_gb300", "csrc", kernel_file)
        if rec["source_sha256"] != source_digest(src):
            return None
        return rec["dram_bytes_per_launch"]
    except (OSError, KeyError, ValueError):
        return None


# workloads whose per-step inputs are drawn for a fixed number of steps
_MAX_STEPS = ("window-decode", "window-decode-unfused", "window-decode-drift",
              "window-decode-ring", "window-decode-hot", "scatter", "scatter-functional")

# what the default one-GPU run also times, each as an entry of the line's
# "secondary" list: (workload, chunk)
SECONDARY = (("window-prefill", 2048), ("window-prefill", 64), ("window-decode", None),
             ("scatter-functional", 64), ("ring-decode-d256", None),
             ("window-decode-d256", None), ("paged-decode-int8", None),
             ("window-prefill-hazard", 64))


def make_workload(name, dev, seed, chunk, n_steps):
    kw = {"chunk": chunk}
    if name in _MAX_STEPS:
        kw["max_steps"] = n_steps
    return WORKLOADS[name](dev, seed=seed, **kw)


def time_workload(wl, args, world, dev, soak_s):
    """W eager warm-up steps; the K timed steps captured once as a CUDA graph
    (no host work in the timed region); the graph replayed for at least
    `soak_s` seconds so that the clock sampler sees the GPU under this load;
    then the K steps timed once (CUDA events, barrier and synchronize on both
    sides), the roofline kernel's K launches timed from a second graph, ten
    more replays for the spread, and the end-to-end pass."""
    import torch
    with ClockSampler(dev) as clocks:
        i = 0
        for _ in range(args.warmup):
            wl.step(i)
            i += 1
        torch.cuda.synchronize()
        step_graph, kern_graph = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph):
            for k in range(args.steps):
                wl.step(i + k)
        with torch.cuda.graph(kern_graph):
            for k in range(args.steps):
                wl.kernel(i + k)
        i += args.steps
        step_graph.replay()
        kern_graph.replay()
        torch.cuda.synchronize()
        t_soak = time.perf_counter()
        soak_replays = 0
        while time.perf_counter() - t_soak < soak_s:
            step_graph.replay()
            soak_replays += 1
            if soak_replays % 4 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        soak_wall = time.perf_counter() - t_soak
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        step_graph.replay()
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = start.elapsed_time(end)
        k0.record()
        kern_graph.replay()
        k1.record()
        torch.cuda.synchronize()
        kern_ms = k0.elapsed_time(k1) / args.steps
        # outside the timed region: the spread of the step time over ten more
        # replays of the same K-step graph (median and 10th percentile)
        reps = []
        for _ in range(10):
            start.record()
            step_graph.replay()
            end.record()
            torch.cuda.synchronize()
            reps.append(start.elapsed_time(end) / args.steps)
        reps.sort()
        replay_stats = {"replays": len(reps), "median_ms_per_step": reps[len(reps) // 2],
                        "p10_ms_per_step": reps[len(reps) // 10],
                        "soak_replays_before_timing": soak_replays, "soak_s": soak_wall}
        del step_graph, kern_graph
        wl.e2e_setup()
        for _ in range(args.warmup):
            wl.e2e_step(i)
            i += 1
        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            wl.e2e_step(i)
            i += 1
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        barrier(world)
        measured = wl.extra_measure() if hasattr(wl, "extra_measure") else {}
    return {"ms": ms, "kern_ms": kern_ms, "replay_stats": replay_stats, "e2e_s": e2e_s,
            "measured": measured, "clocks": clocks.summary(), "status": int(wl.st.item())}


def roofline_of(wl, args, world, ms, kern_ms, e2e_s, peaks, peak_kind):
    """(value, e2e value, roofline object, extra keys) of one timed workload."""
    sec = ms / 1e3
    if wl.bound == "tensor":
        value = wl.flops * args.steps * world / sec / 1e12
        e2e_value = wl.flops * args.steps * world / e2e_s / 1e12
        achieved = wl.flops / (kern_ms / 1e3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": f"{peak_kind} bf16 burst",
                "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                "issued_tflops": wl.issued_flops / (kern_ms / 1e3) / 1e12,
                "algorithmic_flops_per_launch": wl.flops}
        extra = {"stage_and_cache_gbs": wl.bytes_per_step * args.steps / sec / 1e9}
        # a chunk whose flops per algorithmic byte sit below the ridge point
        # of the two measured peaks is bound by HBM, not by the tensor pipe:
        # the roofline is then the bytes' (the tensor figures stay beside it)
        ai = wl.flops / wl.kernel_bytes
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        if ai < ridge:
            gbs = wl.kernel_bytes / (kern_ms / 1e3) / 1e9
            roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": gbs / peaks["hbm_gbs"], "peak_kind": peak_kind,
                    "algorithmic_bytes_per_launch": wl.kernel_bytes,
                    "flops_per_byte": ai, "ridge_flops_per_byte": ridge,
                    "tensor_achieved_tflops": achieved, "tensor_frac": achieved / peak,
                    "tensor_peak_kind": f"{peak_kind} bf16 burst",
                    "algorithmic_flops_per_launch": wl.flops}
    else:
        value = wl.bytes_per_step * args.steps * world / sec / 1e9
        e2e_value = wl.bytes_per_step * args.steps * world / e2e_s / 1e9
        achieved = wl.kernel_bytes / (kern_ms / 1e3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": wl.kernel_bytes}
        extra = {"pct_of_peak": 100.0 * value / peak}
    # the same fraction against the part's nominal figure (context only)
    roof["frac_of_nominal"] = roof["achieved"] / (NOMINAL_TFLOPS if roof["unit"] == "TFLOP/s"
                                                  else NOMINAL_GBS)
    roof.update({"kernel": wl.roofline_kernel, "traffic": kernel_traffic(wl.traffic_key),
                 "avg_launch_ms": kern_ms})
    return value, e2e_value, roof, extra


def cpu_baseline_of(wl, parallel=(5.0, 15.0), single=(10.0, 30.0)):
    """Bounded samples of the oracle over the workload's batch rows (at most
    32): on every host core (rows dealt over threads), and, when `single` is
    given, on one thread."""
    unit = wl.metric()[1]
    rows = range(min(wl.w.batch, 32))
    scale = 1e12 if wl.bound == "tensor" else 1e9
    pw, pa, preps, pn = oracle_threads(wl, rows, host_cores(), *parallel)
    cpu = {"value": pa / pw / scale, "unit": unit, "cores": pn, "kind": "oracle",
           "sample": f"{type(wl).__name__}.oracle_sample over {len(rows)} batch rows "
                     f"dealt over {pn} threads, {preps} repetitions, {pw:.1f} s wall; "
                     f"the C oracle as written"}
    if single is not None:
        sw, sa, sreps, _ = oracle_threads(wl, rows, 1, *single)
        cpu["single_thread"] = {"value": sa / sw / scale, "cores": 1,
                                "sample": f"the same rows on one thread, {sreps} "
                                          f"repetitions, {sw:.1f} s"}
    return cpu


def secondary_entry(name, chunk, args, dev, peaks, peak_kind):
    """One more workload timed the same way as the main line (one GPU)."""
    import torch
    n_steps = args.warmup * 2 + args.steps * 3 + 8
    wl = make_workload(name, dev, 0, chunk, n_steps)
    r = time_workload(wl, args, 1, dev, args.soak)
    value, e2e_value, roof, extra = roofline_of(wl, args, 1, r["ms"], r["kern_ms"], r["e2e_s"],
                                                peaks, peak_kind)
    metric, unit = wl.metric()
    sec = r["ms"] / 1e3
    entry = {"workload": name, "chunk": chunk, "metric": metric, "value": value, "unit": unit,
             "ms_per_step": r["ms"] / args.steps, "steps": args.steps,
             "higher_is_better": True, "config": wl.config(), **extra, **r["measured"],
             "steps_per_s": args.steps / sec,
             "tokens_per_s": wl.tokens_per_step * args.steps / sec,
             "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": wl.h2d,
                     "d2h_bytes_per_step": wl.d2h, "steps_per_s": args.steps / r["e2e_s"],
                     "copies": E2E_COPIES[wl.e2e_overlap]},
             "roofline": roof, "replay_stats": r["replay_stats"],
             "cpu_baseline": cpu_baseline_of(wl, parallel=(2.0, 6.0), single=None),
             "gpu_launches": wl.launches_per_step * args.steps, "clocks": r["clocks"],
             "device_status": r["status"]}
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    n_steps = args.warmup * 2 + args.steps * 3 + 8
    wl = make_workload(args.workload, dev, rank, args.chunk, n_steps)
    peaks, peak_kind = load_peaks()
    r = time_workload(wl, args, world, dev, args.soak)
    ms = max_over_ranks(r["ms"], world, dev)
    e2e_s = max_over_ranks(r["e2e_s"], world, dev)
    if rank != 0:
        return

    sec = ms / 1e3
    metric, unit = wl.metric()
    value, e2e_value, roof, extra = roofline_of(wl, args, world, ms, r["kern_ms"], e2e_s, peaks,
                                                peak_kind)
    cpu = cpu_baseline_of(wl) if world == 1 else None
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": wl.config(), **extra, **r["measured"],
        "steps_per_s": args.steps * world / sec,
        "tokens_per_s": wl.tokens_per_step * args.steps * world / sec,
        "e2e": {"value": e2e_value, "unit": unit, "h2d_bytes_per_step": wl.h2d,
                "d2h_bytes_per_step": wl.d2h, "steps_per_s": args.steps * world / e2e_s,
                "copies": E2E_COPIES[wl.e2e_overlap]},
        "roofline": roof,
        "replay_stats": r["replay_stats"],
        "cpu_baseline": cpu,
        "gpu_launches": wl.launches_per_step * args.steps,
        "clocks": r["clocks"],
        "device_status": r["status"],
    }
    if world == 1 and args.secondary:
        del wl
        torch.cuda.empty_cache()
        line["secondary"] = [secondary_entry(n, c, args, dev, peaks, peak_kind)
                             for n, c in SECONDARY if (n, c) != (args.workload, args.chunk)]
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Setup, W + K device steps and nothing else: the command profiled by
    ncu (no end-to-end pass, no oracle timing)."""
    import torch
    dev = torch.device("cuda", 0)
    kw = {"chunk": args.chunk}
    wl = WORKLOADS[args.workload](dev, seed=0, **kw)
    for i in range(args.warmup + args.steps):
        wl.step(i)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": args.workload, "steps": args.steps, "warmup": args.warmup,
                      "device_status": int(wl.st.item())}), flush=True)


def run_reference(args):
    """The oracle timed on the host cores, each step a bounded sample of the
    same workload: one batch row per host thread (rows dealt round robin over
    the steps), the threads running together."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    torch.set_num_threads(1)
    dev = torch.device("cuda") if torch.cuda.is_available() else torch.device("cpu")
    wl = WORKLOADS[args.workload](dev, seed=0, with_kernels=False, chunk=args.chunk)
    B = wl.w.batch
    cores = min(host_cores(), B)
    step_rows = lambda i: [(cores * i + j) % B for j in range(cores)]
    for i in range(args.warmup):
        oracle_threads(wl, step_rows(i), cores, 1e-9, float("inf"))
    total_t, total_amount = 0.0, 0
    for i in range(args.steps):
        dt, amount, _, used = oracle_threads(wl, step_rows(i), cores, 1e-9, float("inf"))
        total_t += dt
        total_amount += amount
    metric, unit = wl.metric()
    scale = 1e12 if wl.bound == "tensor" else 1e9
    v = total_amount / total_t / scale
    line = {
        "impl": "reference", "metric": metric, "value": v, "unit": unit, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": wl.config(),
        "cpu_baseline": {"value": v, "unit": unit, "cores": used, "kind": "oracle",
                         "sample": f"{cores} batch rows of the workload per step, one a "
                                   f"thread on {used} threads"},
        "e2e": {"value": v, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="contig-decode")
    ap.add_argument("--chunk", type=int, default=None,
                    help="new tokens per step (window-prefill: 64/512/2048; scatter: 1/16/64)")
    ap.add_argument("--profile", action="store_true",
                    help="device steps only (the command run under ncu)")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of replays of the step graph before the timed region, so "
                         "that the clock record covers the GPU under this load")
    ap.add_argument("--secondary", dest="secondary", action="store_true", default=None,
                    help="also time the other workloads (default on the one-GPU default run)")
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    args = ap.parse_args()
    if args.secondary is None:
        args.secondary = args.workload == "contig-decode" and args.chunk is None
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
