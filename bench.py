#!/usr/bin/env python
"""Benchmark of the Windowed-MTP draft-attention hot path on one GB300 per rank.

Workload (default): the million-token draft step of "Windowed-MTP: Removing
the Full-Context Draft-KV Tax at Million-Token Context" (§6 setup: B=1, 1M
context, 2 KV heads, head_dim 256, bf16 KV, n_sink 64, W 4032, d 7 = gamma 6
draft forwards) on seeded synthetic data: K/V ~ N(0,1) with 1% of K rows x4,
a seeded random permutation as the page table.

One timed step = one decode step's draft-attention phase for both arms:
  full arm     : full-context index build + 6 x (append + attention over the
                 whole table, 1,048,577.. keys; one fused launch per step)
  windowed arm : sink+window index build + 6 x (append + attention over
                 64 + 4032 keys; one fused launch per step)
The full arm is launched directly (its attention launches are each bracketed
by CUDA events for the roofline); the windowed arm, whose kernels take a few
microseconds, is replayed from a CUDA graph.  L2 is flushed (256 MiB write)
before each arm, outside the events.

Prints ONE JSON line (rank 0).  `value` is the windowed arm's microseconds
per decode step (lower is better); both arms' numbers are under "arms".
`--impl reference` times the fp64 CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "draft-attn μs/step and KV GB/s (% of HBM peak), windowed vs full, at 1M ctx"
UNIT = "us/step"
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "1m": dict(name="million-token draft step", B=1, S=1_048_576, H_q=16, H_kv=2, D=256,
               n_sink=64, W=4032, gamma=6, outlier_frac=0.01, seed=1002),
    "131k": dict(name="131K-context draft step", B=1, S=131_072, H_q=16, H_kv=2, D=256,
                 n_sink=64, W=4032, gamma=6, outlier_frac=0.0, seed=1001),
}


# ------------------------------------------------------------------ helpers
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def attn_bytes(L, n_q, H_q, H_kv, D, n_new=0):
    """Algorithmic bytes of one attention launch over a table row of L keys:
    K and V rows of every KV head (bf16), the int32 table, q (bf16), out and
    lse (fp32); with a fused append of n_new tokens, their K/V rows are read
    once more and written to the pool."""
    return (L * H_kv * D * 2 * 2 + 4 * L + n_q * H_q * D * 2 + n_q * H_q * (D + 1) * 4
            + n_new * H_kv * D * 2 * 2 * 2)


def source_hash():
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "speculative_decoding_draft_build_gb300", "csrc", "wmtp_attn.cu"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current attention source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_key)
        if ent and ent.get("source_hash") == source_hash():
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Polls SM clock and clock-event reasons through NVML (read-only) while
    the timed region runs; falls back to nvidia-smi."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []  # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._h = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0".encode()
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device_index), ctypes.byref(h)) != 0:
                    raise OSError("no NVML handle")
            self._nvml, self._h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            try:
                self._reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self._reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            self._nvml = None

    def _sample_nvml(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        ok1 = self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0
        ok2 = self._reasons_fn(self._h, ctypes.byref(rs)) == 0
        if ok1:
            self.samples.append((int(clk.value), int(rs.value) if ok2 else 0))

    def _run(self):
        while not self._stop.is_set():
            self._sample_nvml()
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
            self._sample_nvml()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        mhz = [s[0] for s in self.samples]
        mask = 0
        for _, m in self.samples:
            mask |= m
        reasons = [n for b, n in self.REASONS.items() if mask & b]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(mhz), "source": "nvml"}


class Dist:
    def __init__(self, n_gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, values):
        """Elementwise max of a list of floats over ranks."""
        if self.pg is None:
            return list(values)
        dev = torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")
        t = torch.tensor(values, dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return t.cpu().tolist()

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ workload
def packed(dev, parts):
    """One device byte buffer holding tensors of the given (dtype, shape) at
    256-byte aligned offsets, and the tensors as views into it (so that a set
    of inputs or outputs moves between host and device in one copy)."""
    offs, off = [], 0
    for dt, shape in parts:
        nbytes = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        offs.append((off, nbytes))
        off += (nbytes + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=dev)
    views = [buf[o:o + n].view(dt).view(shape) for (o, n), (dt, shape) in zip(offs, parts)]
    return buf, views


class Workload:
    """Inputs resident on the device; tables, outputs and workspaces preallocated."""

    def __init__(self, cfg, dev):
        from speculative_decoding_draft_build_gb300 import synth
        import speculative_decoding_draft_build_gb300 as wm
        self.cfg = cfg
        self.dev = dev
        B, S, H_q, H_kv, D, g = cfg["B"], cfg["S"], cfg["H_q"], cfg["H_kv"], cfg["D"], cfg["gamma"]
        seed = cfg["seed"]
        self.scale = 1.0 / math.sqrt(D)
        pool = B * (S + g)
        self.kp = synth.normal_bf16((pool, H_kv, D), seed, dev)
        if cfg["outlier_frac"] > 0:
            synth.scale_random_rows_(self.kp, cfg["outlier_frac"], 4.0, seed + 1)
        self.vp = synth.normal_bf16((pool, H_kv, D), seed + 2, dev)
        # the step's inputs from the host (new K/V, queries, lengths) in one
        # buffer, its windowed outputs in another: one copy each way per step
        # in the end-to-end leg
        bf = torch.bfloat16
        self.io_in, (self.kn, self.vn, self.q, self.seq) = packed(
            dev, [(bf, (g, B, H_kv, D)), (bf, (g, B, H_kv, D)), (bf, (g, B, 1, H_q, D)), (torch.int32, (B,))])
        self.kn.copy_(synth.normal_bf16((g, B, H_kv, D), seed + 3, dev))
        self.vn.copy_(synth.normal_bf16((g, B, H_kv, D), seed + 4, dev))
        self.q.copy_(synth.normal_bf16((g, B, 1, H_q, D), seed + 5, dev))
        self.seq.fill_(S)
        if cfg.get("identity"):
            # identity page table: request b's positions in consecutive slots
            self.rtt = torch.arange(pool, dtype=torch.int32, device=dev).view(B, S + g)
        else:
            self.rtt = synth.permutation(pool, seed + 6, dev).view(B, S + g)
        self.slots = torch.stack([self.rtt[:, S + j] for j in range(g)]).contiguous()  # [g, B]
        self.full_stride = S + g
        self.win_stride = cfg["n_sink"] + cfg["W"]
        self.tab_full = torch.empty((g, B, self.full_stride), dtype=torch.int32, device=dev)
        self.len_full = torch.empty((g, B), dtype=torch.int32, device=dev)
        self.tab_win = torch.empty((g, B, self.win_stride), dtype=torch.int32, device=dev)
        self.len_win = torch.empty((g, B), dtype=torch.int32, device=dev)
        self.io_out_full, (self.out_full, self.lse_full) = packed(
            dev, [(torch.float32, (g, B, 1, H_q, D)), (torch.float32, (g, B, 1, H_q))])
        self.io_out, (self.out_win, self.lse_win) = packed(
            dev, [(torch.float32, (g, B, 1, H_q, D)), (torch.float32, (g, B, 1, H_q))])
        self.ns_full = wm.attn_num_splits(B, 1, H_kv, S + g, dev)
        self.ns_win = wm.attn_num_splits(B, 1, H_kv, self.win_stride, dev)
        self.ws_full = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, self.ns_full), dev)
        self.ws_win = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, self.ns_win), dev)
        self.flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)

    # overlap=True: chained steps; steps after the first start their copies
    # while the step before finishes (overlap_hold=2: the previous step's key
    # and the step's own wait for it); step 0 follows the index build, which
    # writes its table, so it reads nothing early (-1) but, like every
    # chained step, releases the next step only after its own wait.
    def full_arm(self, events=None, attn_only=False, n_split=None, overlap=False):
        import speculative_decoding_draft_build_gb300 as wm
        c = self.cfg
        if not attn_only:
            wm.build_draft_indices(self.seq, c["gamma"], c["n_sink"], c["W"], c["gamma"] + 1,
                                   windowed=False, req_to_token=self.rtt, table=self.tab_full,
                                   lens=self.len_full)
        for j in range(c["gamma"]):
            if events is not None:
                events[j][0].record()
            wm.draft_decode_attn_append(self.kn[j], self.vn[j], self.slots[j],
                                        self.q[j], self.kp, self.vp, self.tab_full[j], self.len_full[j],
                                        self.scale, out=self.out_full[j], lse=self.lse_full[j],
                                        n_split=n_split or self.ns_full, workspace=self.ws_full,
                                        overlap_hold=(2 if j > 0 else -1) if overlap else None)
            if events is not None:
                events[j][1].record()

    def win_arm(self, events=None, attn_only=False, n_split=None, overlap=False):
        import speculative_decoding_draft_build_gb300 as wm
        c = self.cfg
        if not attn_only:
            wm.build_draft_indices(self.seq, c["gamma"], c["n_sink"], c["W"], c["gamma"] + 1,
                                   windowed=True, req_to_token=self.rtt, table=self.tab_win,
                                   lens=self.len_win)
        ws = self.ws_win
        if n_split is not None and n_split != self.ns_win:
            ws = self.workspace_for(n_split)
        for j in range(c["gamma"]):
            if events is not None:
                events[j][0].record()
            wm.draft_decode_attn_append(self.kn[j], self.vn[j], self.slots[j],
                                        self.q[j], self.kp, self.vp, self.tab_win[j], self.len_win[j],
                                        self.scale, out=self.out_win[j], lse=self.lse_win[j],
                                        n_split=n_split or self.ns_win, workspace=ws,
                                        overlap_hold=(2 if j > 0 else -1) if overlap else None)
            if events is not None:
                events[j][1].record()

    def workspace_for(self, n_split):
        import speculative_decoding_draft_build_gb300 as wm
        c = self.cfg
        key = ("ws", n_split)
        if key not in self.__dict__:
            self.__dict__[key] = wm.AttnWorkspace(
                wm.attn_workspace_bytes(c["B"], 1, c["H_q"], c["H_kv"], c["D"], n_split), self.dev)
        return self.__dict__[key]

    def bytes_full_attn(self, j):
        c = self.cfg
        return c["B"] * attn_bytes(c["S"] + j + 1, 1, c["H_q"], c["H_kv"], c["D"], n_new=1)

    def bytes_win_attn(self, j):
        c = self.cfg
        L = min(c["S"] + j + 1, c["n_sink"] + c["W"])
        return c["B"] * attn_bytes(L, 1, c["H_q"], c["H_kv"], c["D"], n_new=1)


def hold_gpu(us: float = 150.0):
    """Queue a spin kernel so the GPU is still busy when a timed call is
    enqueued: its start event then stamps the kernel, not the host time the
    Python binding spends preparing the launch (tens of microseconds)."""
    torch.cuda._sleep(int(us * 2100))  # cycles at about 2.1 GHz


def graph_of(fn, dev):
    """The launches `fn` makes, captured once in a CUDA graph (on a side
    stream; the current stream waits for the capture)."""
    cur = torch.cuda.current_stream(dev)
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(cur)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            fn()
    cur.wait_stream(cap)
    torch.cuda.synchronize(dev)
    return gr


def time_graph_samples(gr, flush, reps, dev, warm=3):
    """Microseconds of `reps` replays of `gr`, each bracketed by CUDA events on
    the current stream with L2 flushed (a 256 MiB write) just before it."""
    for _ in range(warm):
        gr.replay()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush.zero_()
        a.record()
        gr.replay()
        b.record()
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b) * 1e3)
    return ts


def time_graph(gr, flush, reps, dev):
    return statistics.median(time_graph_samples(gr, flush, reps, dev))


# ------------------------------------------------------------------ our arm
def run_ours(args, dist_ctx):
    import speculative_decoding_draft_build_gb300 as wm
    wm.build()
    wm.load()
    dev = torch.device("cuda", dist_ctx.local)
    torch.cuda.set_device(dev)
    cfg = WORKLOADS[args.workload]
    w = Workload(cfg, dev)
    g = cfg["gamma"]
    stream = torch.cuda.current_stream(dev)

    # warm-up (also sets kernel attributes before capture)
    for _ in range(max(args.warmup, 1)):
        w.full_arm()
        w.win_arm()
    torch.cuda.synchronize(dev)

    # windowed arm as a CUDA graph (its kernels take microseconds)
    graph = graph_of(w.win_arm, dev)
    # the same step as chained launches (bit-identical results)
    graph_chain = graph_of(lambda: w.win_arm(overlap=True), dev)
    for _ in range(max(args.warmup, 1)):
        graph.replay()
        graph_chain.replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    e_full = [[ev(), ev()] for _ in range(K)]
    e_win = [[ev(), ev()] for _ in range(K)]
    e_chain = [[ev(), ev()] for _ in range(K)]
    e_attn = [[[ev(), ev()] for _ in range(g)] for _ in range(K)]
    sampler = ClockSampler(dev.index)
    dist_ctx.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    t0 = time.perf_counter()
    for k in range(K):
        w.flush.zero_()
        e_full[k][0].record()
        w.full_arm(e_attn[k])
        e_full[k][1].record()
        w.flush.zero_()
        e_win[k][0].record()
        graph.replay()
        e_win[k][1].record()
        w.flush.zero_()
        e_chain[k][0].record()
        graph_chain.replay()
        e_chain[k][1].record()
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    dist_ctx.barrier()
    sampler.stop()

    full_ms = [a.elapsed_time(b) for a, b in e_full]
    win_ms = [a.elapsed_time(b) for a, b in e_win]
    chain_ms = [a.elapsed_time(b) for a, b in e_chain]
    attn_full_ms = [[e_attn[k][j][0].elapsed_time(e_attn[k][j][1]) for j in range(g)] for k in range(K)]
    # median over the launches: the first launch of a step can start after a
    # host-side gap (its Python call is prepared while the index build runs)
    full_attn_mean_ms = statistics.median(x for row in attn_full_ms for x in row)

    # windowed attention per launch: a graph of the six attention launches
    # alone (no index build), replayed with L2 flushed before each replay;
    # per launch = replay time / 6, so the six launches never sum to more
    # than the step they belong to
    win_attn_source = "graph of the six windowed attention launches alone (L2 flushed), replay time / 6"
    g_attn = graph_of(lambda: w.win_arm(attn_only=True), dev)
    win_attn_ms = [x / g * 1e-3 for x in time_graph_samples(g_attn, w.flush, K, dev)]
    win_attn_mean_ms = statistics.median(win_attn_ms)

    full_bytes = sum(w.bytes_full_attn(j) for j in range(g))
    win_bytes = sum(w.bytes_win_attn(j) for j in range(g))
    stats = [statistics.median(full_ms), statistics.median(win_ms), full_attn_mean_ms,
             win_attn_mean_ms, wall, statistics.median(chain_ms)]
    stats = dist_ctx.max(stats)
    full_step_ms, win_step_ms, full_attn_ms_max, win_attn_ms_max, wall_max, chain_step_ms = stats

    peak, peak_kind = hbm_peak()
    full_gbs = (full_bytes / g) / (full_attn_ms_max * 1e-3) / 1e9
    win_gbs = (win_bytes / g) / (win_attn_ms_max * 1e-3) / 1e9

    result = {
        "metric": METRIC,
        "value": round(win_step_ms * 1e3, 3),
        "unit": UNIT,
        "n_gpus": dist_ctx.world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(full_step_ms + win_step_ms, 4),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{cfg['name']}: B={cfg['B']}, S={cfg['S']}, H_q={cfg['H_q']}, "
                        f"H_kv={cfg['H_kv']}, D={cfg['D']}, n_sink={cfg['n_sink']}, W={cfg['W']}, "
                        f"gamma={g}, d={g + 1}, permuted page table"
                        + (f", {cfg['outlier_frac']:.0%} of K rows x4" if cfg["outlier_frac"] else ""),
            "B": cfg["B"], "S": cfg["S"], "gamma": g, "n_sink": cfg["n_sink"], "W": cfg["W"],
            "H_q": cfg["H_q"], "H_kv": cfg["H_kv"], "D": cfg["D"],
            "l2": "flushed before each arm (256 MiB write, outside the event brackets)",
            "parallelism": "replicas" if dist_ctx.world > 1 else "single GPU",
            "value_is": "windowed arm: index build + 6 x fused (append_kv + draft attention), us per decode step",
        },
        "arms": {
            "windowed": {
                "us_per_step": round(win_step_ms * 1e3, 3),
                "us_per_step_chained": round(chain_step_ms * 1e3, 3),
                "attn_us_per_launch": round(win_attn_ms_max * 1e3, 3),
                "attn_us_per_step": round(win_attn_ms_max * 1e3 * g, 3),
                "keys_per_launch": min(cfg["S"] + 1, cfg["n_sink"] + cfg["W"]),
                "kv_gbs": round(win_gbs, 1),
                "frac_of_hbm": round(win_gbs / peak, 4),
                "n_split": w.ns_win,
                "launch": "cuda graph",
                "attn_timing": win_attn_source,
            },
            "full": {
                "us_per_step": round(full_step_ms * 1e3, 3),
                "attn_us_per_launch": round(full_attn_ms_max * 1e3, 3),
                "attn_us_per_step": round(full_attn_ms_max * 1e3 * g, 3),
                "keys_per_launch": cfg["S"] + 1,
                "kv_gbs": round(full_gbs, 1),
                "frac_of_hbm": round(full_gbs / peak, 4),
                "n_split": w.ns_full,
                "launch": "direct, an event pair around each launch",
            },
        },
        "roofline": {
            "kernel": "split_decode_kernel<256> (full-context draft attention)",
            "bound": "hbm",
            "achieved": round(full_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(full_gbs / peak, 4),
            "peak_kind": peak_kind,
            "bytes_per_launch": int(full_bytes / g),
            "traffic": profiled_traffic("full_1m") if args.workload == "1m" else None,
        },
        "roofline_windowed": {
            "kernel": "split_decode_kernel<256> (windowed draft attention)",
            "bound": "hbm",
            "achieved": round(win_gbs, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(win_gbs / peak, 4),
            "peak_kind": peak_kind,
            "bytes_per_launch": int(win_bytes / g),
            "traffic": profiled_traffic("windowed_4096") if args.workload == "1m" else None,
        },
        # per timed iteration: the full arm, the windowed step and the same
        # step as chained launches, each an index build and g attention launches
        "gpu_launches": K * 3 * (1 + g),
        "clocks": sampler.summary(),
        "timed_region_s": round(wall_max, 4),
    }

    result["e2e"] = measure_e2e(w, args, dev)
    result["mass_diagnostics"] = measure_mass(w, dev)
    if args.workload == "1m" and not args.no_tree:
        result["tree"] = measure_tree(args, dev)
    if not args.no_extend:
        result["extend"] = measure_extend(w, args, dev)
    if not args.no_fp8:
        result["fp8"] = measure_fp8(w, args, dev)
    if not args.no_ring:
        result["ring"] = measure_ring(w, args, dev)
    if args.workload == "1m" and not args.no_configs:
        o = None
        if dist_ctx.rank == 0 and dist_ctx.world == 1 and not args.no_cpu_baseline:
            import oracle as o
            o.build()
        result["configs"] = measure_configs(args, dev, w, result, o)
    if dist_ctx.rank == 0 and dist_ctx.world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args)
    return result


# ------------------------------------------------------------------ the other configs
TINY = dict(name="tiny draft step", B=1, S=8192, H_q=8, H_kv=2, D=128, n_sink=64, W=1024, gamma=1,
            outlier_frac=0.0, seed=1000)


def measure_arms(w, args, dev, o=None):
    """Both arms of a workload, each replayed from a CUDA graph with L2
    flushed before every replay: the step (index build + gamma fused append +
    attention launches) and the gamma attention launches alone (per launch =
    replay / gamma).  With the oracle `o`, also its host time for one step of
    each arm (tables, appends and attention of every query head)."""
    g = w.cfg["gamma"]
    reps = max(5, min(args.steps, 30))
    peak, _ = hbm_peak()
    host = _oracle_inputs(w) if o is not None else None
    res = {}
    for name, arm, nbytes_fn, ns, keys in (
            ("full", w.full_arm, w.bytes_full_attn, w.ns_full, w.cfg["S"] + 1),
            ("windowed", w.win_arm, w.bytes_win_attn, w.ns_win,
             min(w.cfg["S"] + 1, w.cfg["n_sink"] + w.cfg["W"]))):
        arm()
        torch.cuda.synchronize(dev)
        t_step = time_graph(graph_of(arm, dev), w.flush, reps, dev)
        t_chain_step = time_graph(graph_of(lambda: arm(overlap=True), dev), w.flush, reps, dev)
        # per launch: each launch's own duration (no overlap), and the time
        # per launch of the chained launches
        t_attn = time_graph(graph_of(lambda: arm(attn_only=True), dev), w.flush, reps, dev) / g
        t_chain = time_graph(graph_of(lambda: arm(attn_only=True, overlap=True), dev), w.flush, reps, dev) / g
        nbytes = sum(nbytes_fn(j) for j in range(g)) / g
        gbs = nbytes / (t_attn * 1e-6) / 1e9
        res[name] = {"us_per_step": round(t_step, 3), "us_per_step_chained": round(t_chain_step, 3),
                     "attn_us_per_launch": round(t_attn, 3),
                     "attn_us_per_launch_chained": round(t_chain, 3),
                     "keys_per_launch": keys, "kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4),
                     "bytes_per_launch": int(nbytes), "n_split": ns}
        if o is not None:
            t = time.perf_counter()
            oracle_step(o, w, host, windowed=name == "windowed")
            res[name]["oracle_host_us_per_step"] = round((time.perf_counter() - t) * 1e6, 1)
    if o is not None:
        res["oracle_cores"] = o.num_threads()
    res["timing"] = ("CUDA graph replays, L2 flushed before each, median; *_chained: the same launches as "
                     "chained steps (steps 2-6 copy their keys while the step before finishes)")
    return res


class RingBatch:
    """Batched ring layout: B=6 requests at lengths uniform in [900K, 1M],
    H_q=16, H_kv=2, D=256, n_sink=64, W=4032, d=7; each request's draft KV
    lives in a ring of n_sink + W + d = 4103 slots at a seeded ring base
    inside a pool of 2 * B rings, filled from the kept prompt positions.  The
    same logical rows also sit un-ringed in a flat pool (every position of
    every request, ~12 GB, a seeded permutation as the page table)."""

    def __init__(self, dev, seed=1003):
        import speculative_decoding_draft_build_gb300 as wm
        from speculative_decoding_draft_build_gb300 import synth
        self.dev = dev
        B, g, n_sink, W, d = 6, 6, 64, 4032, 7
        H_q, H_kv, D = 16, 2, 256
        self.cfg = dict(B=B, gamma=g, n_sink=n_sink, W=W, d=d, H_q=H_q, H_kv=H_kv, D=D)
        self.R = R = n_sink + W + d
        self.S_list = synth.uniform_lengths(B, 900_000, 1_048_576, seed)
        ctx = [s + g for s in self.S_list]
        total = sum(ctx)
        self.flat_k = synth.normal_bf16((total, H_kv, D), seed + 1, dev)
        self.flat_v = synth.normal_bf16((total, H_kv, D), seed + 2, dev)
        perm = synth.permutation(total, seed + 3, dev)
        self.rtt = torch.zeros((B, max(ctx)), dtype=torch.int32, device=dev)
        off = 0
        for b in range(B):
            self.rtt[b, :ctx[b]] = perm[off:off + ctx[b]]
            off += ctx[b]
        self.ring_base = torch.tensor(synth.ring_bases(B, R, 2 * B, seed + 4), dtype=torch.int32, device=dev)
        self.ring_k = torch.zeros((2 * B * R, H_kv, D), dtype=torch.bfloat16, device=dev)
        self.ring_v = torch.zeros_like(self.ring_k)
        self.seq = torch.tensor(self.S_list, dtype=torch.int32, device=dev)
        pos, cnt = wm.prefill_keep_positions(self.seq, n_sink, W)
        live = torch.arange(pos.shape[1], device=dev).view(1, -1) < cnt.view(-1, 1).long()
        rows = torch.gather(self.rtt, 1, torch.where(live, pos, torch.zeros_like(pos)).long()).long()
        wm.ring_fill(self.flat_k[rows].contiguous(), self.flat_v[rows].contiguous(), self.seq, self.ring_base,
                     n_sink, W, d, self.ring_k, self.ring_v)
        self.kn = synth.normal_bf16((g, B, H_kv, D), seed + 5, dev)
        self.vn = synth.normal_bf16((g, B, H_kv, D), seed + 6, dev)
        self.q = synth.normal_bf16((g, B, 1, H_q, D), seed + 7, dev)
        req = torch.arange(B, dtype=torch.int32, device=dev)
        self.slots_ring = torch.stack([wm.ring_map(self.ring_base, (self.seq + j).to(torch.int32), req,
                                                   n_sink, W, d) for j in range(g)]).contiguous()
        self.slots_flat = torch.stack([self.rtt[req.long(), (self.seq + j).long()] for j in range(g)]).contiguous()
        self.stride = n_sink + W
        self.tab_ring = torch.empty((g, B, self.stride), dtype=torch.int32, device=dev)
        self.tab_flat = torch.empty_like(self.tab_ring)
        self.len_ring = torch.empty((g, B), dtype=torch.int32, device=dev)
        self.len_flat = torch.empty_like(self.len_ring)
        self.ns = wm.attn_num_splits(B, 1, H_kv, self.stride, dev)
        self.ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, self.ns), dev)
        self.out_ring = torch.empty((g, B, 1, H_q, D), dtype=torch.float32, device=dev)
        self.lse_ring = torch.empty((g, B, 1, H_q), dtype=torch.float32, device=dev)
        self.out_flat = torch.empty_like(self.out_ring)
        self.lse_flat = torch.empty_like(self.lse_ring)
        self.flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.scale = 1.0 / math.sqrt(D)
        torch.cuda.synchronize(dev)

    def ring_steps(self):
        """The ring layout without tables: each step's slots come from the
        ring rule in the kernel (its window arrives in TMA boxes), the step's
        own K/V appended in the same launch; chained steps (steps 2-6 copy
        their keys while the step before finishes)."""
        import speculative_decoding_draft_build_gb300 as wm
        c = self.cfg
        for j in range(c["gamma"]):
            wm.draft_decode_attn_ring(self.q[j], self.ring_k, self.ring_v, self.seq, self.ring_base, j, c["n_sink"],
                                      c["W"], c["d"], self.scale, k_new=self.kn[j], v_new=self.vn[j],
                                      out=self.out_ring[j], lse=self.lse_ring[j], n_split=self.ns, workspace=self.ws,
                                      overlap_hold=2 if j > 0 else -1)

    def arm(self, ring=True, attn_only=False):
        import speculative_decoding_draft_build_gb300 as wm
        c = self.cfg
        kp, vp = (self.ring_k, self.ring_v) if ring else (self.flat_k, self.flat_v)
        tab, ln = (self.tab_ring, self.len_ring) if ring else (self.tab_flat, self.len_flat)
        slots = self.slots_ring if ring else self.slots_flat
        out, lse = (self.out_ring, self.lse_ring) if ring else (self.out_flat, self.lse_flat)
        if not attn_only:
            src = dict(ring_base=self.ring_base) if ring else dict(req_to_token=self.rtt)
            wm.build_draft_indices(self.seq, c["gamma"], c["n_sink"], c["W"], c["d"], windowed=True,
                                   table=tab, lens=ln, **src)
        for j in range(c["gamma"]):
            wm.draft_decode_attn_append(self.kn[j], self.vn[j], slots[j], self.q[j], kp, vp, tab[j], ln[j],
                                        self.scale, out=out[j], lse=lse[j], n_split=self.ns, workspace=self.ws)

    def bytes_per_launch(self, j):
        c = self.cfg
        return sum(attn_bytes(min(S + j + 1, c["n_sink"] + c["W"]), 1, c["H_q"], c["H_kv"], c["D"], n_new=1)
                   for S in self.S_list)


def measure_ring_batch(args, dev, o=None):
    """The batched ring workload: gamma = 6 steps of fused append + windowed
    attention (index build in ring layout first), replayed from a CUDA graph
    with L2 flushed before each replay; the attention launches alone as a
    second graph; ring outputs compared bit for bit with the same steps on the
    un-ringed flat pool; the oracle's host time for one ring step."""
    rb = RingBatch(dev)
    g = rb.cfg["gamma"]
    reps = max(5, min(args.steps, 30))
    rb.ring_steps()
    rb.arm(ring=False)
    torch.cuda.synchronize(dev)
    same = bool(torch.equal(rb.out_ring, rb.out_flat) and torch.equal(rb.lse_ring, rb.lse_flat))
    rb.arm(ring=True)
    torch.cuda.synchronize(dev)
    same_tables = bool(torch.equal(rb.out_ring, rb.out_flat) and torch.equal(rb.lse_ring, rb.lse_flat))
    t_step = time_graph(graph_of(rb.ring_steps, dev), rb.flush, reps, dev)
    t_tab = time_graph(graph_of(lambda: rb.arm(ring=True), dev), rb.flush, reps, dev)
    t_flat = time_graph(graph_of(lambda: rb.arm(ring=False), dev), rb.flush, reps, dev)
    nbytes = sum(rb.bytes_per_launch(j) - 4 * rb.cfg["B"] * min(4096, rb.cfg["n_sink"] + rb.cfg["W"])
                 for j in range(g)) / g  # no table read
    peak, _ = hbm_peak()
    gbs = nbytes / (t_step / g * 1e-6) / 1e9
    res = {"workload": "B=6 requests, lengths uniform in [900K, 1M], H_q=16, H_kv=2, D=256, n_sink=64, "
                       "W=4032, d=7, ring of 4103 slots per request at seeded ring bases, gamma=6",
           "S": rb.S_list, "us_per_step": round(t_step, 3), "us_per_launch": round(t_step / g, 3),
           "kv_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peak, 4), "bytes_per_launch": int(nbytes),
           "n_split": rb.ns, "path": "table-free chained ring steps (slots from the ring rule, TMA boxes for runs of "
                                     "consecutive ring slots; steps 2-6 copy while the step before finishes), "
                                     "fused append",
           "ring_via_tables_us_per_step": round(t_tab, 3),
           "unringed_flat_pool_us_per_step": round(t_flat, 3),
           "ring_equals_unringed_bitwise": same and same_tables,
           "timing": "CUDA graph replays, L2 flushed before each, median; steps include the index build where "
                     "there are tables"}
    if o is not None:
        import numpy as np

        def bits(t):
            return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        c = rb.cfg
        kp, vp = bits(rb.ring_k), bits(rb.ring_v)
        kn, vn, q = bits(rb.kn), bits(rb.vn), bits(rb.q)
        seq, base, slots = rb.seq.cpu().numpy(), rb.ring_base.cpu().numpy(), rb.slots_ring.cpu().numpy()
        t = time.perf_counter()
        table, lens = o.build_draft_indices(seq, g, c["n_sink"], c["W"], c["d"], windowed=True, ring_base=base,
                                            stride=rb.stride)
        for j in range(g):
            o.append_kv(kn[j], vn[j], slots[j], kp, vp)
            o.draft_decode_attn(q[j], kp, vp, table[j], lens[j], rb.scale)
        res["oracle_host_us_per_step"] = round((time.perf_counter() - t) * 1e6, 1)
        res["oracle_cores"] = o.num_threads()
    del rb
    torch.cuda.empty_cache()
    return res


def measure_configs(args, dev, w3, result, o=None):
    """Every workload of the hot path's configuration table next to the
    million-token headline: the tiny step (S=8192, and S=1000 inside the
    window, where the windowed and full outputs must be bit-identical at the
    same split count), the 131K step (full vs windowed), the batched ring, and
    pointers to the million-token arms and the tree row measured above."""
    res = {}
    for key, cfg in (("1_tiny_S8192", TINY), ("1_tiny_S1000", dict(TINY, S=1000)),
                     ("2_131k", WORKLOADS["131k"])):
        w = Workload(cfg, dev)
        res[key] = measure_arms(w, args, dev, o)
        res[key]["workload"] = (f"{cfg['name']}: B={cfg['B']}, S={cfg['S']}, H_q={cfg['H_q']}, "
                                f"H_kv={cfg['H_kv']}, D={cfg['D']}, n_sink={cfg['n_sink']}, W={cfg['W']}, "
                                f"gamma={cfg['gamma']}, permuted page table")
        if cfg["S"] + 1 <= cfg["n_sink"] + cfg["W"]:
            w.full_arm()
            w.win_arm(n_split=w.ns_full)
            torch.cuda.synchronize(dev)
            res[key]["windowed_equals_full_bitwise"] = bool(
                torch.equal(w.out_win, w.out_full) and torch.equal(w.lse_win, w.lse_full))
        del w
        torch.cuda.empty_cache()
    res["3_1m"] = {"see": "arms, roofline, roofline_windowed (the headline workload)",
                   "windowed_us_per_step": result["arms"]["windowed"]["us_per_step"],
                   "full_us_per_step": result["arms"]["full"]["us_per_step"]}
    # the same 131K and 1M steps over an identity page table (each request's
    # positions in consecutive slots) instead of a permuted one
    for key, cfg, oo in (("2_131k_identity", dict(WORKLOADS["131k"], identity=True), o),
                         ("3_1m_identity", dict(WORKLOADS["1m"], identity=True), None)):
        w = Workload(cfg, dev)
        res[key] = measure_arms(w, args, dev, oo)
        res[key]["workload"] = (f"{cfg['name']}: B={cfg['B']}, S={cfg['S']}, H_q={cfg['H_q']}, "
                                f"H_kv={cfg['H_kv']}, D={cfg['D']}, n_sink={cfg['n_sink']}, W={cfg['W']}, "
                                f"gamma={cfg['gamma']}, identity page table"
                                + (f", {cfg['outlier_frac']:.0%} of K rows x4" if cfg["outlier_frac"] else ""))
        del w
        torch.cuda.empty_cache()
    res["4_ring_batch"] = measure_ring_batch(args, dev, o)
    if "tree" in result:
        res["5_tree"] = {"see": "tree (per window W)"}
    return res


def measure_mass(w, dev):
    """Attention-mass diagnostics (in-window mass, win_perturb, tail out-frac;
    App. C, Table 12) of the step's six draft queries: the far-key tables of
    the six steps, the attention over the far keys (the full-context split
    count), then one diagnostics launch over all query rows from the windowed
    arm's outputs and the far outputs, event-timed (median of 20).  The
    merged output of the two parts is compared with the full arm's output."""
    import speculative_decoding_draft_build_gb300 as wm
    c = w.cfg
    g = c["gamma"]
    tab_far, len_far = wm.build_far_indices(w.seq, g, c["n_sink"], c["W"], w.rtt, stride=w.full_stride)
    o_far = torch.empty_like(w.out_win)
    lse_far = torch.empty_like(w.lse_win)
    for j in range(g):
        wm.draft_decode_attn(w.q[j], w.kp, w.vp, tab_far[j], len_far[j], w.scale, out=o_far[j],
                             lse=lse_far[j], n_split=w.ns_full, workspace=w.ws_full)
    o_full = torch.empty_like(w.out_win)
    lse_full = torch.empty_like(w.lse_win)
    args = (w.out_win, w.lse_win, o_far, lse_far)
    for _ in range(3):
        res = wm.attn_mass_diagnostics(*args, o_full=o_full, lse_full=lse_full)
    ts = []
    for _ in range(20):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_gpu()
        a.record()
        res = wm.attn_mass_diagnostics(*args, o_full=o_full, lse_full=lse_full)
        b.record()
        torch.cuda.synchronize(dev)
        ts.append(a.elapsed_time(b) * 1e3)
    in_win, perturb, tail = (r.double().mean().item() for r in res)
    merged_err = (o_full - w.out_full).abs().max().item()
    return {"us_per_launch": round(statistics.median(ts), 2), "rows": int(w.lse_win.numel()),
            "mean_in_win": round(in_win, 6), "mean_win_perturb": round(perturb, 6),
            "mean_tail_out_frac": round(tail, 6),
            "merged_vs_full_arm_max_abs": float(f"{merged_err:.3e}"),
            "how": "windowed attention + attention over the far-key table (wmtp_build_far_indices), "
                   "combined per row (wmtp_attn_mass_diagnostics)",
            "note": "synthetic N(0,1) keys and values; the pages measure these on model activations"}


def measure_extend(w, args, dev):
    """Draft-extend pass on the bench's workload (the million-token one by
    default): the draft forward over n_new = 5 accepted tokens (positions
    S..S+4) in one launch, windowed and full-context.  Event-timed with L2 flushed before each launch; algorithmic
    bytes are the pass's unique bytes: K and V of every key of the union table
    once (every KV head), the table, q, out and lse.  `token_reads_gbs` counts
    instead each token's own key set (the tokens of a request share most of
    their keys).  `kernel` names the launch the library picks for the row."""
    import speculative_decoding_draft_build_gb300 as wm
    c = w.cfg
    B, S, H_q, H_kv, D = c["B"], c["S"], c["H_q"], c["H_kv"], c["D"]
    n = 5
    seq = torch.full((B,), S, dtype=torch.int32, device=dev)
    nn = torch.full((B,), n, dtype=torch.int32, device=dev)
    q = w.q[:n].permute(1, 0, 2, 3, 4).reshape(B, n, H_q, D).contiguous()
    out = torch.empty((B, n, H_q, D), dtype=torch.float32, device=dev)
    lse = torch.empty((B, n, H_q), dtype=torch.float32, device=dev)
    peak, _ = hbm_peak()
    reps = max(5, min(args.steps, 30))
    res = {"n_new": n, "B": B, "S": S,
           "timing": "CUDA events per launch, L2 flushed before each, median"}
    for windowed in (True, False):
        tab, ln = wm.build_extend_indices(seq, nn, c["n_sink"], c["W"], c["gamma"] + 1,
                                          windowed=windowed, req_to_token=w.rtt)
        ns = wm.extend_num_splits(B, n, H_kv, tab.shape[-1], dev)
        ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, n, H_q, H_kv, D, ns), dev)

        def call():
            wm.draft_extend_attn(q, w.kp, w.vp, tab, ln, seq, nn, c["n_sink"], c["W"], w.scale,
                                 windowed=windowed, out=out, lse=lse, n_split=ns, workspace=ws)
        for _ in range(3):
            call()
        ts = []
        for _ in range(reps):
            w.flush.zero_()
            hold_gpu()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e-3)
        t = statistics.median(ts)
        keys = sum(min(S + j + 1, c["n_sink"] + c["W"]) if windowed else S + j + 1 for j in range(n))
        L = int(ln.max().item())
        rest = 4 * L + n * H_q * (D * 2 + (D + 1) * 4)
        nbytes = B * (L * H_kv * D * 2 * 2 + rest)
        token_bytes = B * (keys * H_kv * D * 2 * 2 + rest)
        stride = tab.shape[-1]
        if 2 <= n <= 8 and ns <= 128 and stride >= 65536:
            kernel = f"tree_tc_kernel<{D}, false> (tcgen05, union table row, combined gather roles)"
        elif 2 <= n <= 8 and ns <= 128 and stride >= 1024 * ns:
            kernel = f"extend_kernel<{D}> (one K/V read for all tokens)"
        else:
            kernel = f"split_decode_kernel<{D}, extend> (CTAs per token)"
        res["windowed" if windowed else "full"] = {
            "kernel": kernel,
            "us_per_pass": round(t * 1e6, 2), "kv_gbs": round(nbytes / t / 1e9, 1),
            "frac_of_hbm": round(nbytes / t / 1e9 / peak, 4), "n_split": ns,
            "union_keys": L, "bytes_per_pass": int(nbytes),
            "token_reads_gbs": round(token_bytes / t / 1e9, 1)}
    return res


def measure_fp8(w, args, dev):
    """fp8 (E4M3) KV on the million-token workload ([WMTP] §6, "Robustness to
    KV-cache quantization"): the bf16 pools quantised once with per-KV-head
    scales (amax / 448), then for each of the 6 draft steps the quantising
    append of the step's K/V and the attention, full-context and windowed.
    Each launch event-timed with L2 flushed before it; algorithmic bytes are
    one byte per K/V element plus the table, q, out and lse."""
    import speculative_decoding_draft_build_gb300 as wm
    c = w.cfg
    B, S, H_q, H_kv, D, g = c["B"], c["S"], c["H_q"], c["H_kv"], c["D"], c["gamma"]
    n_slots = w.kp.shape[0]
    ks = (w.kp.abs().amax(dim=(0, 2)).float() / 448).contiguous()
    vs = (w.vp.abs().amax(dim=(0, 2)).float() / 448).contiguous()
    kp8 = torch.empty((n_slots, H_kv, D), dtype=torch.uint8, device=dev)
    vp8 = torch.empty_like(kp8)
    all_slots = torch.arange(n_slots, dtype=torch.int32, device=dev)
    wm.append_kv_fp8(w.kp, w.vp, all_slots, ks, vs, kp8, vp8)
    peak, _ = hbm_peak()
    reps = max(3, min(args.steps, 10))
    res = {"k_scale": [round(x, 6) for x in ks.tolist()], "v_scale": [round(x, 6) for x in vs.tolist()],
           "timing": "CUDA events per launch, L2 flushed before each, median over steps x reps"}
    for name, tab, ln, stride in (("full", w.tab_full, w.len_full, w.full_stride),
                                  ("windowed", w.tab_win, w.len_win, w.win_stride)):
        ns = wm.attn_num_splits(B, 1, H_kv, stride, dev, fp8=True)
        ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, ns), dev)
        out = torch.empty((B, 1, H_q, D), dtype=torch.float32, device=dev)
        lse = torch.empty((B, 1, H_q), dtype=torch.float32, device=dev)

        def attn(j):
            wm.draft_decode_attn_fp8(w.q[j], kp8, vp8, ks, vs, tab[j], ln[j], w.scale, out=out, lse=lse,
                                     n_split=ns, workspace=ws)

        def append(j):
            wm.append_kv_fp8(w.kn[j], w.vn[j], w.slots[j], ks, vs, kp8, vp8)
        for j in range(g):
            append(j)
            attn(j)
        t_attn, t_app, gbs = [], [], []
        for _ in range(reps):
            for j in range(g):
                ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
                w.flush.zero_()
                hold_gpu()
                ev[0].record()
                append(j)
                ev[1].record()
                w.flush.zero_()
                hold_gpu()
                ev[2].record()
                attn(j)
                ev[3].record()
                torch.cuda.synchronize(dev)
                ta = ev[2].elapsed_time(ev[3]) * 1e-3
                L = min(S + j + 1, c["n_sink"] + c["W"]) if name == "windowed" else S + j + 1
                nbytes = B * (L * H_kv * D * 2 + 4 * L + H_q * D * 2 + H_q * (D + 1) * 4)
                t_attn.append(ta)
                t_app.append(ev[0].elapsed_time(ev[1]) * 1e-3)
                gbs.append(nbytes / ta / 1e9)
        res[name] = {"attn_us_per_launch": round(statistics.median(t_attn) * 1e6, 2),
                     "append_us_per_launch": round(statistics.median(t_app) * 1e6, 2),
                     "kv_gbs": round(statistics.median(gbs), 1),
                     "frac_of_hbm": round(statistics.median(gbs) / peak, 4), "n_split": ns}
    full_bytes = B * (S + 1) * H_kv * D * 2 + 4 * B * (S + 1) + B * H_q * (D * 2 + (D + 1) * 4)
    res["roofline"] = {
        "kernel": "split_decode_kernel<256, fp8> (full-context draft attention over E4M3 pools)",
        "bound": "hbm", "achieved": res["full"]["kv_gbs"], "peak": peak, "unit": "GB/s",
        "frac": res["full"]["frac_of_hbm"], "bytes_per_launch": int(full_bytes),
        "traffic": profiled_traffic("fp8_full_1m") if args.workload == "1m" else None}
    del kp8, vp8
    return res


def measure_ring(w, args, dev):
    """Ring path without tables ([WMTP] App. A ring; §7 "Prefill
    sparsification and TTFT") on the million-token workload:
      prefill: the draft KV build of the prompt pruned to keep(S) (one ring
               fill of n_sink + W rows) against the unpruned build (all S + 6
               rows appended to a full-length pool), event-timed, L2 flushed;
      step:    6 implicit-table ring draft steps (fused append + attention,
               slots from the ring rule in the kernel, no index build)
               replayed from a CUDA graph, L2 flushed before each replay."""
    import speculative_decoding_draft_build_gb300 as wm
    c = w.cfg
    B, S, H_q, H_kv, D, g = c["B"], c["S"], c["H_q"], c["H_kv"], c["D"], c["gamma"]
    n_sink, W, d = c["n_sink"], c["W"], c["gamma"] + 1
    R = n_sink + W + d
    ring_base = (torch.arange(B, dtype=torch.int32, device=dev) * R).contiguous()
    ring_k = torch.zeros((B * R, H_kv, D), dtype=torch.bfloat16, device=dev)
    ring_v = torch.zeros_like(ring_k)
    pos, cnt = wm.prefill_keep_positions(w.seq, n_sink, W)
    live = torch.arange(pos.shape[1], device=dev).view(1, -1) < cnt.view(-1, 1).long()
    pos = torch.where(live, pos, torch.zeros_like(pos))
    rows = torch.gather(w.rtt, 1, pos.long()).long()  # pool rows of the kept prompt positions
    rows_k = w.kp[rows].contiguous()
    rows_v = w.vp[rows].contiguous()
    full_k = torch.empty_like(w.kp)
    full_v = torch.empty_like(w.vp)
    all_slots = torch.arange(w.kp.shape[0], dtype=torch.int32, device=dev)
    reps = max(3, min(args.steps, 10))

    def timed(fn):
        fn()
        ts = []
        for _ in range(reps):
            w.flush.zero_()
            hold_gpu()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e3)
        return statistics.median(ts)
    t_pruned = timed(lambda: wm.ring_fill(rows_k, rows_v, w.seq, ring_base, n_sink, W, d, ring_k, ring_v))
    t_full = timed(lambda: wm.append_kv(w.kp, w.vp, all_slots, full_k, full_v))
    del full_k, full_v
    ns = wm.attn_num_splits(B, 1, H_kv, n_sink + W, dev)
    ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, ns), dev)
    out = torch.empty((g, B, 1, H_q, D), dtype=torch.float32, device=dev)
    lse = torch.empty((g, B, 1, H_q), dtype=torch.float32, device=dev)

    def step():
        for j in range(g):
            wm.draft_decode_attn_ring(w.q[j], ring_k, ring_v, w.seq, ring_base, j, n_sink, W, d, w.scale,
                                      k_new=w.kn[j], v_new=w.vn[j], out=out[j], lse=lse[j], n_split=ns,
                                      workspace=ws, overlap_hold=2 if j > 0 else -1)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    cap = torch.cuda.Stream(dev)
    cur = torch.cuda.current_stream(dev)
    cap.wait_stream(cur)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            step()
    cur.wait_stream(cap)
    for _ in range(3):
        gr.replay()
    torch.cuda.synchronize(dev)
    t_step = timed(gr.replay)
    peak, _ = hbm_peak()
    step_bytes = sum(B * attn_bytes(min(S + j + 1, n_sink + W), 1, H_q, H_kv, D, n_new=1) - B * 4 *
                     min(S + j + 1, n_sink + W) for j in range(g))
    return {"ring_slots_per_request": R, "n_split": ns,
            "prefill_kv_build": {"pruned_us": round(t_pruned, 2), "unpruned_us": round(t_full, 2),
                                 "rows_pruned": int(B * min(S, n_sink + W)), "rows_unpruned": int(w.kp.shape[0]),
                                 "note": "the draft's prompt KV build only; the draft prompt pass itself "
                                         "(projections over the kept positions) needs the model"},
            "step": {"us_per_step": round(t_step, 3), "us_per_launch": round(t_step / g, 3),
                     "launches": g, "kv_gbs": round(step_bytes / (t_step * 1e-6) / 1e9, 1),
                     "frac_of_hbm": round(step_bytes / (t_step * 1e-6) / 1e9 / peak, 4),
                     "launch": "cuda graph, no index build, no table; chained steps (steps 2-6 copy while the step before finishes)"},
            "timing": "CUDA events, L2 flushed before each, median"}


def measure_tree(args, dev):
    """Tree-draft attention (k=4 branches x d=7, B=8 requests with contexts
    log-uniform in [32K, 1M], H_q=16, H_kv=2, D=256, n_sink=64) for each
    window W: event-timed launches with L2 flushed before each, algorithmic
    bytes (each ring key row once per KV head, q, out, lse) and useful flops
    (4*D per visible key per query row).  Means of the launches: the event
    clock's ticks are too coarse for a median."""
    import speculative_decoding_draft_build_gb300 as wm
    from speculative_decoding_draft_build_gb300 import synth
    B, k, d, H_q, H_kv, D, n_sink = 8, 4, 7, 16, 2, 256, 64
    S_list = synth.log_uniform_lengths(B, 32_768, 1_048_576, 5000)
    seq = torch.tensor(S_list, dtype=torch.int32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    peak_hbm, _ = hbm_peak()
    peak_tf = bf16_peak()
    res = {}
    reps = max(5, min(args.steps, 30))
    for W in (args.tree_w or (1024, 2048, 4096, 8192)):
        R = n_sink + W + d * k
        rb = torch.tensor(synth.ring_bases(B, R, B + 2, 5000 + W), dtype=torch.int32, device=dev)
        kp = synth.normal_bf16(((B + 2) * R, H_kv, D), 5001 + W, dev)
        vp = synth.normal_bf16(((B + 2) * R, H_kv, D), 5002 + W, dev)
        q = synth.normal_bf16((B, k * d, H_q, D), 5003 + W, dev)
        out = torch.empty((B, k * d, H_q, D), dtype=torch.float32, device=dev)
        lse = torch.empty((B, k * d, H_q), dtype=torch.float32, device=dev)
        ns = wm.tree_num_splits(B, H_q, H_kv, d, k, n_sink, W, dev)
        ws = wm.AttnWorkspace(wm.tree_workspace_bytes(B, H_q, H_kv, D, d, k, ns), dev)
        for _ in range(3):
            wm.tree_draft_attn(q, kp, vp, seq, rb, n_sink, W, d, k, 1 / 16, out=out, lse=lse,
                               n_split=ns, workspace=ws)
        ts = []
        for _ in range(reps):
            flush.zero_()
            hold_gpu()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            wm.tree_draft_attn(q, kp, vp, seq, rb, n_sink, W, d, k, 1 / 16, out=out, lse=lse,
                               n_split=ns, workspace=ws)
            b.record()
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b) * 1e-3)
        t = statistics.mean(ts)  # the event clock ticks in ~2 us steps: a mean resolves finer
        keys = n_sink + W - 1 + k * d  # key list per request (contexts exceed the window)
        nbytes = B * keys * H_kv * D * 2 * 2 + B * k * d * H_q * (D * 2 + (D + 1) * 4)
        flops = B * k * d * H_q * (n_sink + W) * 4 * D
        res[f"W={W}"] = {"us_per_launch": round(t * 1e6, 2), "kv_gbs": round(nbytes / t / 1e9, 1),
                         "frac_of_hbm": round(nbytes / t / 1e9 / peak_hbm, 4),
                         "tflops": round(flops / t / 1e12, 2),
                         "frac_of_bf16_peak": round(flops / t / 1e12 / peak_tf, 4),
                         "n_split": ns, "bytes_per_launch": int(nbytes), "flops_per_launch": int(flops)}
        del kp, vp
    return {"workload": "tree drafter: B=8, contexts log-uniform [32K, 1M], k=4, d=7 (28 nodes), "
                        "H_q=16, H_kv=2, D=256, n_sink=64, ring of n_sink+W+d*k slots",
            "timing": "CUDA events per launch, L2 flushed before each, mean", "windows": res,
            "kernel": "tree_tc_kernel<256, split> (tcgen05, TMEM accumulators); chunks of 16 tiles or more "
                      "take the instance with separate K and V gather warps", "bf16_peak_tflops": peak_tf}


def measure_e2e(w, args, dev):
    """Both arms through the Python binding with host buffers: every step
    copies its inputs (q, new K/V, seq_lens; one packed buffer) from pinned
    host memory, runs the arm, and reads its outputs (out, lse; one packed
    buffer) back; timed on the host around a stream synchronisation.
    `value` (windowed arm) and `full.value`: the whole step (copy in, index
    build, six fused launches, copy out) captured once in a CUDA graph and
    replayed per step, as a serving loop runs it; `eager_us`: the windowed
    step with direct calls from Python."""
    in_h = w.io_in.cpu().pin_memory()
    stream = torch.cuda.current_stream(dev)
    h2d = in_h.numel()

    def host_timed(fn, reps):
        for _ in range(max(args.warmup, 1)):
            fn()
        times = []
        for _ in range(reps):
            w.flush.zero_()  # L2 flushed before each step, outside the timed interval
            torch.cuda.synchronize(dev)
            t = time.perf_counter()
            fn()
            times.append(time.perf_counter() - t)
        return statistics.median(times)

    def graph_step(arm, io_out, out_h):
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap):
            with torch.cuda.graph(gr, stream=cap):
                w.io_in.copy_(in_h, non_blocking=True)
                arm()
                out_h.copy_(io_out, non_blocking=True)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)

        def run():
            gr.replay()
            stream.synchronize()
        return run

    out_h = torch.empty(w.io_out.shape, dtype=torch.uint8).pin_memory()

    def eager():
        w.io_in.copy_(in_h, non_blocking=True)
        w.win_arm()
        out_h.copy_(w.io_out, non_blocking=True)
        stream.synchronize()
    eager_s = host_timed(eager, args.steps)
    win_s = host_timed(graph_step(w.win_arm, w.io_out, out_h), args.steps)
    out_full_h = torch.empty(w.io_out_full.shape, dtype=torch.uint8).pin_memory()
    full_s = host_timed(graph_step(w.full_arm, w.io_out_full, out_full_h), max(3, min(args.steps, 10)))
    return {"value": round(win_s * 1e6, 3), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out_h.numel()),
            "eager_us": round(eager_s * 1e6, 3),
            "full": {"value": round(full_s * 1e6, 3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                     "d2h_bytes_per_step": int(out_full_h.numel())},
            "how": "each arm with pinned host I/O, host-timed (L2 flushed before each step, outside the "
                   "interval): one CUDA graph per step (packed copy in, index build, 6 fused launches, packed "
                   "copy out); value = windowed arm, full.value = full-context arm; eager_us = windowed arm by "
                   "direct calls"}


# ------------------------------------------------------------------ oracle legs
def _oracle_inputs(w):
    import numpy as np

    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return dict(kp=bits(w.kp), vp=bits(w.vp), kn=bits(w.kn), vn=bits(w.vn), q=bits(w.q),
                rtt=w.rtt.cpu().numpy(), slots=w.slots.cpu().numpy(), seq=w.seq.cpu().numpy())


def oracle_step(o, w, host, windowed=True, nthreads=None):
    """One decode step of either arm in the oracle: tables, then per draft step
    the append and the attention of every query head."""
    c = w.cfg
    g = c["gamma"]
    stride = c["n_sink"] + c["W"] if windowed else c["S"] + g
    table, lens = o.build_draft_indices(host["seq"], g, c["n_sink"], c["W"], g + 1, windowed=windowed,
                                        req_to_token=host["rtt"], stride=stride)
    for j in range(g):
        o.append_kv(host["kn"][j], host["vn"][j], host["slots"][j], host["kp"], host["vp"])
        o.draft_decode_attn(host["q"][j], host["kp"], host["vp"], table[j], lens[j], w.scale,
                            nthreads=nthreads)


def cpu_baseline(w, args):
    import oracle as o
    o.build()
    host = _oracle_inputs(w)
    t = time.perf_counter()
    oracle_step(o, w, host)
    first = time.perf_counter() - t
    reps = max(1, min(5, int(5.0 / max(first, 1e-3))))
    ts = [first]
    for _ in range(reps):
        t = time.perf_counter()
        oracle_step(o, w, host)
        ts.append(time.perf_counter() - t)
    win_us = statistics.median(ts) * 1e6
    t = time.perf_counter()
    oracle_step(o, w, host, nthreads=1)
    win_1t_us = (time.perf_counter() - t) * 1e6
    # full arm: one draft forward over the whole table, all query heads
    c = w.cfg
    g = c["gamma"]
    t = time.perf_counter()
    table, lens = o.build_draft_indices(host["seq"], 1, c["n_sink"], c["W"], g + 1, windowed=False,
                                        req_to_token=host["rtt"], stride=c["S"] + g)
    t_build = time.perf_counter() - t
    t = time.perf_counter()
    o.draft_decode_attn(host["q"][0], host["kp"], host["vp"], table[0], lens[0], w.scale)
    t_fwd = time.perf_counter() - t
    return {"value": round(win_us, 1), "unit": UNIT, "cores": o.num_threads(), "kind": "oracle",
            "sample": f"windowed decode step (gamma={g}, all {c['H_q']} heads) x{len(ts)}, median; "
                      f"full arm estimated from one full-context forward ({c['S'] + 1} keys, all heads) "
                      f"x{g} + one table build",
            "full_us_per_step_est": round((t_fwd * g + t_build * g) * 1e6, 1),
            "single_thread_us": round(win_1t_us, 1)}


def run_reference(args, dist_ctx):
    """The fp64 CPU oracle as the reference arm, timed on the host cores on
    the same workload; each step is one windowed decode step."""
    import oracle as o
    o.build()
    cfg = WORKLOADS[args.workload]
    dev = torch.device("cuda", dist_ctx.local) if torch.cuda.is_available() else torch.device("cpu")
    w = Workload.__new__(Workload)
    # inputs only (same seeds as our arm); no CUDA library involved
    from speculative_decoding_draft_build_gb300 import synth
    B, S, H_q, H_kv, D, g = cfg["B"], cfg["S"], cfg["H_q"], cfg["H_kv"], cfg["D"], cfg["gamma"]
    seed = cfg["seed"]
    w.cfg = cfg
    w.scale = 1.0 / math.sqrt(D)
    pool = B * (S + g)
    w.kp = synth.normal_bf16((pool, H_kv, D), seed, dev)
    if cfg["outlier_frac"] > 0:
        synth.scale_random_rows_(w.kp, cfg["outlier_frac"], 4.0, seed + 1)
    w.vp = synth.normal_bf16((pool, H_kv, D), seed + 2, dev)
    w.kn = synth.normal_bf16((g, B, H_kv, D), seed + 3, dev)
    w.vn = synth.normal_bf16((g, B, H_kv, D), seed + 4, dev)
    w.q = synth.normal_bf16((g, B, 1, H_q, D), seed + 5, dev)
    w.rtt = synth.permutation(pool, seed + 6, dev).view(B, S + g)
    w.seq = torch.full((B,), S, dtype=torch.int32, device=dev)
    w.slots = torch.stack([w.rtt[:, S + j] for j in range(g)]).contiguous()
    host = _oracle_inputs(w)
    for _ in range(args.warmup):
        oracle_step(o, w, host)
    ts = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle_step(o, w, host)
        ts.append(time.perf_counter() - t)
    wall = time.perf_counter() - t0
    val = statistics.median(ts) * 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": round(val, 1), "unit": UNIT,
        "n_gpus": dist_ctx.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(val / 1e3, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg['name']}: B={B}, S={S}, H_q={H_q}, H_kv={H_kv}, D={D}, "
                               f"n_sink={cfg['n_sink']}, W={cfg['W']}, gamma={g}, windowed arm",
                   "B": B, "S": S, "gamma": g},
        "cpu_baseline": {"kind": "oracle", "cores": o.num_threads(), "value": round(val, 1),
                         "unit": UNIT,
                         "sample": f"{args.steps} windowed decode steps (index build + {g} x "
                                   f"(append + attention, all {H_q} heads)), median"},
        "e2e": {"value": round(val, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "timed_region_s": round(wall, 3),
    }


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=sorted(WORKLOADS), default="1m")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-tree", action="store_true", help="skip the tree-drafter measurement")
    p.add_argument("--no-extend", action="store_true", help="skip the draft-extend measurement")
    p.add_argument("--no-fp8", action="store_true", help="skip the fp8-KV measurement")
    p.add_argument("--no-ring", action="store_true", help="skip the table-free ring measurement")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the tiny, 131K and batched-ring configurations")
    p.add_argument("--tree-only", action="store_true",
                   help="run only the tree-drafter measurement (a profiling driver; prints the tree object)")
    p.add_argument("--tree-w", type=int, action="append",
                   help="window(s) for the tree measurement (default 1024, 2048, 4096, 8192)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    dist_ctx = Dist(args.gpus)
    try:
        if args.impl == "reference":
            if dist_ctx.rank != 0:
                return 0
            res = run_reference(args, dist_ctx)
        elif args.tree_only:
            import speculative_decoding_draft_build_gb300 as wm
            wm.build()
            wm.load()
            dev = torch.device("cuda", dist_ctx.local)
            torch.cuda.set_device(dev)
            res = {"tree": measure_tree(args, dev)}
        else:
            res = run_ours(args, dist_ctx)
        if dist_ctx.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        dist_ctx.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
