#!/usr/bin/env python
"""Benchmark of SnapKV prefill-time KV-cache compression on GB300.

One step = the whole compression (scores, pooling, selection, emission) of
every layer of the workload, each layer with its own K/V, through the C ABI
on device-resident inputs: one snapkv_compress_layers call, which runs
consecutive layers on four streams (--layer-streams) so that a layer's
selection overlaps the next layers' scoring.  The metric is prompt tokens compressed per second per
layer, all heads: (prompt tokens x layers) / time.  The step is captured once
in a CUDA graph and the timed region replays it (every replay runs every
memset and kernel of every layer); the step issued directly
(`us_per_layer_eager`) and every layer through snapkv_compress on one stream
(`us_per_layer_single_calls`) are timed as well, and layer 0's outputs are
checked byte for byte against snapkv_compress's.

Default workload: a Llama-3-8B-shaped model at a 131072-token prompt, 32
layers (32 query / 8 KV heads, d = 128, bf16, W = 64, avg pooling k = 13,
C = 4096).  Each layer's K and V (537 MB) are far larger than L2, so no L2
flush is needed between iterations.

Also reported: the score kernel alone against the HBM roofline (CUDA events
on the launching stream) and, beside it, against its tensor-core and exp2
ceilings (two passes recompute the logits), the end-to-end figure through the host-buffer entry
point (host->device copies of the inputs and device->host copies of the
compressed cache inside the timed region), the oracle timed on host cores on
a bounded sample, SM clocks and throttle reasons sampled during the timed
region, and the number of library kernels launched in it; after the timed
region, decode steps over the full and the compressed cache, and decode steps
with Scissorhands eviction starting from the compressed cache.

`--impl reference` times the CPU oracle instead, on the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prompt tokens compressed/s per layer (all heads) and % of HBM roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="4", help="workload name (see synth.CONFIGS)")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-scissorhands", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--no-lse", action="store_true", help="skip the caller's-LSE step")
    ap.add_argument("--layer-streams", type=int, default=4,
                    help="streams snapkv_compress_layers overlaps consecutive layers on (1-4)")
    ap.add_argument("--eager", action="store_true",
                    help="time the calls issued one by one instead of the captured step")
    ap.add_argument("--case", choices=["decode", "scissorhands"], default=None,
                    help="run a small fixed case for a profiler and exit (no timing)")
    return ap.parse_args()


# ----------------------------------------------------------------- peaks ---

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    """SM clock and clock-event reasons sampled during a region (NVML)."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x20: "sync_boost", 0x40: "sw_thermal_slowdown",
               0x80: "hw_thermal_slowdown", 0x100: "hw_power_brake_slowdown",
               0x200: "display_clock_setting"}

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self._stop = threading.Event()
        self._th = None
        self._nvml = None
        self._h = None
        try:
            import torch
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit")
            h = ctypes.c_void_p()
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            if nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) != 0:
                if nv.nvmlDeviceGetHandleByIndex_v2(cuda_index, ctypes.byref(h)) != 0:
                    raise RuntimeError("nvml handle")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._h = nv, h
        except Exception:
            self._nvml = None

    def _loop(self):
        nv, h = self._nvml, self._h
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(mhz.value)
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._th = threading.Thread(target=self._loop, daemon=True)
            self._th.start()

    def stop(self):
        if self._th is not None:
            self._stop.set()
            self._th.join()

    def summary(self):
        if self._nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        reasons = [n for bit, n in self.REASONS.items() if self.reasons & bit]
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples)}


# ------------------------------------------------------------ workloads ---

def workload_bytes(cfg, seqlens, esz):
    """Algorithmic bytes of one layer: (score kernel, whole compression)."""
    H_q, H_kv, d, W, C = cfg["H_q"], cfg["H_kv"], cfg["d"], cfg["W"], cfg["C"]
    score = sum(L * H_kv * d * esz + W * H_q * d * esz for L in seqlens)
    gather = sum(4 * min(C, L) * H_kv * d * esz + 4 * min(C, L) * H_kv for L in seqlens)
    return score, score + gather


# exp2 per clock per SM of the special-function units, measured on GB300 (an
# in-bounds throughput probe, matching ncu's XU pipe counter)
MUFU_EX2_PER_CLK_SM = 32


def score_work(cfg, seqlens):
    """Tensor-core flops and exp2 count of one layer's two-pass scoring: per
    scored sequence (L > C) and KV head, pass 1 forms the W*g window rows'
    logits against all L keys and pass 2 against the P = L - W prefix keys;
    each logit is 2 d flops of bf16 MMA and one exp2."""
    Wp = cfg["W"] * cfg["H_q"] // cfg["H_kv"]
    keys = sum(L + (L - cfg["W"]) for L in seqlens if L > cfg["C"])
    return 2 * Wp * cfg["d"] * keys * cfg["H_kv"], Wp * keys * cfg["H_kv"]


def compute_peaks(sms: int):
    """(bf16 TFLOP/s, its kind, exp2 per second in 1e12, its kind)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mp = json.load(f)
        tc, tc_kind = float(mp["bf16_tflops"]), "measured (burst)"
        mhz = float(mp.get("sm_max_mhz", 2070.0))
    except Exception:
        tc, tc_kind, mhz = 1900.0, "fallback", 2070.0
    mufu = MUFU_EX2_PER_CLK_SM * sms * mhz * 1e6 / 1e12
    return tc, tc_kind, mufu, f"derived: {MUFU_EX2_PER_CLK_SM} ex2/clk/SM x {sms} SMs x {mhz:.0f} MHz"


def cpu_baseline(name, layers_total, nthreads=None, lay=None, min_seconds=10.0, max_layers=4,
                 keep_first=False):
    """Oracle on whole layers (all KV heads), layer 0 onwards, until about
    min_seconds of CPU time are spent (at most max_layers): a bounded sample.
    The oracle uses all host cores: (sequence, KV head) units in parallel, or
    one unit at a time with its window rows and keys spread over the cores
    when there are fewer units than cores.  keep_first: also return layer 0
    and the oracle's outputs for it (the bench's parity check)."""
    import oracle
    import synth

    cfg = synth.CONFIGS[name]
    nthreads = nthreads or (os.cpu_count() or 1)
    dt, tokens, done = 0.0, 0, 0
    first = None
    while done < max_layers and (done == 0 or dt < min_seconds):
        cur = lay if (lay is not None and done == 0) else synth.make_layer(name, done)
        t0 = time.perf_counter()
        out = oracle.compress(cur.q_win, cur.k, cur.v, cur.seqlens, cur.W, cfg["k_pool"],
                              cfg["pool"], cfg["C"], nthreads=nthreads)
        dt += time.perf_counter() - t0
        if keep_first and done == 0:
            first = (cur, out)
        tokens += int(sum(cur.seqlens))
        done += 1
        if lay is not None:
            break
    info = {"value": tokens / dt, "unit": UNIT, "cores": nthreads, "kind": "oracle",
            "host_cores": os.cpu_count(), "threads": nthreads,
            "sample": f"layers 0-{done - 1} of {layers_total}, all KV heads, "
                      f"{tokens} prompt tokens, fp64 C oracle on {nthreads} threads, {dt:.2f} s"}
    return (info, first) if keep_first else info


def single_thread_baseline(name="2"):
    """The oracle on one thread over one layer of a workload (tokens/s)."""
    import oracle
    import synth

    cfg = synth.CONFIGS[name]
    lay = synth.make_layer(name, 0)
    t0 = time.perf_counter()
    oracle.compress(lay.q_win, lay.k, lay.v, lay.seqlens, lay.W, cfg["k_pool"], cfg["pool"],
                    cfg["C"], nthreads=1)
    return int(sum(lay.seqlens)) / (time.perf_counter() - t0)


def parity_vs_oracle(S, torch, lay, ora, cfg, dev):
    """The library's compression of one numpy layer against the oracle's, by
    the agreement rule of the parity tests: raw and pooled scores within
    1e-7 + 1e-5 |oracle|; kept prefix sets equal outside the band of pooled
    scores within 1e-5 relative of the (C - W)-th best; every slot holds the
    bytes of its own index's K and V rows; the window block is exact."""
    import numpy as np

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if a.dtype == np.uint16 else t).to(dev)

    W, C, H_kv = lay.W, cfg["C"], lay.H_kv
    q, k, v = to_dev(lay.q_win), to_dev(lay.k), to_dev(lay.v)
    ok, ov, oi, ws = S.compress(q, k, v, lay.seqlens, W, cfg["k_pool"], cfg["pool"], C)
    shape = S.make_shape(lay.B, lay.H_q, H_kv, lay.d, q.dtype)
    raw, pooled = S.scores_from_workspace(ws, shape, lay.seqlens, W, C)
    torch.cuda.synchronize()
    raw, pooled = raw.cpu().numpy(), pooled.cpu().numpy()
    idx = oi.cpu().numpy()
    bits = lambda t: t.cpu().view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.cpu().numpy()
    okh, ovh = bits(ok), bits(ov)
    n = C - W
    off, units, band, decided, worst, ok_all = 0, 0, 0, 0, 0.0, True
    for b, L in enumerate(lay.seqlens):
        L = int(L)
        P = L - W
        for h in range(H_kv):
            gi = idx[b, h]
            if L > C:
                units += 1
                for got, want in ((raw[off + h * P: off + (h + 1) * P], ora["raw"][b][h]),
                                  (pooled[off + h * P: off + (h + 1) * P], ora["pooled"][b][h])):
                    err = np.abs(got - want)
                    ok_all &= bool(np.all(err <= 1e-7 + 1e-5 * np.abs(want)))
                    worst = max(worst, float(np.max(err / (1e-7 + 1e-5 * np.abs(want)))))
                po, tau = ora["pooled"][b][h], ora["tau"][b, h]
                band += int(np.count_nonzero(np.abs(po - tau) <= 1e-5 * tau))
                diff = set(gi[:n].tolist()) ^ set(ora["idx"][b, h, :n].tolist())
                decided += len(diff)
                ok_all &= all(abs(po[j] - tau) <= 1e-5 * tau for j in diff)
                ok_all &= gi[n:].tolist() == list(range(P, L))
            else:
                ok_all &= gi.tolist() == ora["idx"][b, h].tolist()
            rows = gi >= 0
            src = lay.offsets[b] + gi[rows]
            ok_all &= bool(np.array_equal(okh[b, rows, h], lay.k[src, h]))
            ok_all &= bool(np.array_equal(ovh[b, rows, h], lay.v[src, h]))
        if L > C:
            off += H_kv * P
    return {"layer": 0, "units": units, "pass": bool(ok_all),
            "max_score_error_over_tolerance": worst,
            "exemption_band_positions": band, "kept_by_one_side_in_band": decided,
            "rule": "scores 1e-7 + 1e-5 rel; sets equal outside the 1e-5 band; bytes by index"}


def workload_table(S, torch, dev, peak, names=("1", "2", "3", "5a", "5b"), reps=12,
                   layer_streams=4):
    """Every other workload of the pages' shapes through snapkv_compress (and
    snapkv_score alone), four layers in rotation so that inputs exceed L2:
    microseconds per layer through snapkv_compress_layers and through
    snapkv_compress per layer (calls captured in a CUDA graph and replayed, and
    the same calls issued directly), prompt tokens/s and the fraction of the
    HBM roofline of the algorithmic bytes."""
    import synth
    from synth.device import make_layer_device

    out = {}
    for name in names:
        cfg = synth.CONFIGS[name]
        W, C, kp, pool = cfg["W"], cfg["C"], cfg["k_pool"], cfg["pool"]
        layers = [make_layer_device(name, l, dev) for l in range(4)]
        seqlens = layers[0][3]
        B, H_q, H_kv, d = len(seqlens), cfg["H_q"], cfg["H_kv"], cfg["d"]
        dt = layers[0][1].dtype
        esz = 2 if cfg["dtype"] == "bf16" else 4
        shape = S.make_shape(B, H_q, H_kv, d, dt)
        ws = torch.empty(S.workspace_size(shape, seqlens, W, C), dtype=torch.uint8, device=dev)
        ok = torch.empty((B, C, H_kv, d), dtype=dt, device=dev)
        ov, oi = torch.empty_like(ok), torch.empty((B, H_kv, C), dtype=torch.int32, device=dev)

        def comp(i, st=None):
            q, k, v, _ = layers[i % 4]
            S.compress(q, k, v, seqlens, W, kp, pool, C, out_k=ok, out_v=ov, out_idx=oi,
                       workspace=ws, stream=st)

        wsl = torch.empty(S.workspace_size_layers(shape, seqlens, W, C, layer_streams),
                          dtype=torch.uint8, device=dev)
        lstreams = [torch.cuda.Stream() for _ in range(layer_streams)]
        levents = [torch.cuda.Event() for _ in range(layer_streams + 1)]
        louts = [(torch.empty_like(ok), torch.empty_like(ov), torch.empty_like(oi))
                 for _ in range(reps)]

        def comp_layers(i, st=None):
            # all reps layer compressions in one call (inputs rotating over
            # the four layers): the timed "calls" below are its layers
            if i % reps == 0:
                S.compress_layers([layers[j % 4][:3] for j in range(reps)], seqlens, W, kp, pool,
                                  C, louts, wsl, lstreams, levents, stream=st)

        def score(i, st=None):
            q, k, _, _ = layers[i % 4]
            S.score(q, k, seqlens, W, C, ws, stream=st)

        res = {"desc": cfg["desc"]}
        for tag, fn in (("compress", comp_layers), ("compress_single", comp), ("score", score)):
            for i in range(4):
                fn(i)
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for i in range(reps):
                fn(i)
            b.record()
            torch.cuda.synchronize()
            res[f"us_per_layer_{tag}_eager"] = 1e3 * a.elapsed_time(b) / reps
            # the same calls captured in a CUDA graph and replayed
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cap):
                with torch.cuda.graph(g, stream=cap):
                    for i in range(reps):
                        fn(i, cap)
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            a.record()
            for _ in range(3):
                g.replay()
            b.record()
            torch.cuda.synchronize()
            res[f"us_per_layer_{tag}"] = 1e3 * a.elapsed_time(b) / (3 * reps)
            del g
        assert S.get_status(ws) == S.OK and S.get_status(wsl) == S.OK
        score_bytes, compress_bytes = workload_bytes(cfg, seqlens, esz)
        us = res["us_per_layer_compress"]
        res["tokens_per_s"] = sum(seqlens) / (us / 1e6)
        res["frac_compress"] = compress_bytes / (us / 1e6) / 1e9 / peak
        res["frac_score"] = score_bytes / (res["us_per_layer_score"] / 1e6) / 1e9 / peak
        res["bytes_per_layer"] = compress_bytes
        out[name] = res
        del layers
    out["note"] = ("four layers in rotation, 12 layer compressions per timing: compress = "
                   f"one snapkv_compress_layers call over them ({layer_streams} layer streams), "
                   "compress_single = snapkv_compress per layer on one stream, score = "
                   "snapkv_score per layer; CUDA events around three replays of a CUDA graph "
                   "of the calls (us_per_layer_*) and around the calls issued directly "
                   "(*_eager); fractions of the measured HBM copy bandwidth for the "
                   "algorithmic bytes, from the graph timings")
    return out


def lse_input_step(S, torch, data, outs, wsl, seqlens, cfg, dev, ns, peak, compress_bytes):
    """The same step with the caller's window LSE (snapkv_compress_layers with
    lse_wins: pass 2 only, as when the prefill attention kernel returns its
    row LSE).  The LSE is computed once per layer in plain torch on the device
    (fp32 logits under the causal mask, torch.logsumexp), outside any timed
    region; the step is captured in a CUDA graph and replayed."""
    import math

    W, C, kp, pool = cfg["W"], cfg["C"], cfg["k_pool"], cfg["pool"]
    H_q, H_kv, d = cfg["H_q"], cfg["H_kv"], cfg["d"]
    g = H_q // H_kv
    B = len(seqlens)
    lses = []
    for q, k, _ in data:
        lse = torch.full((B, W, H_q), float("nan"), dtype=torch.float32, device=dev)
        row0 = 0
        for b, L in enumerate(seqlens):
            if L > C:
                P = L - W
                kb = k[row0:row0 + L].float()
                mask = torch.arange(L, device=dev)[None, :] > (P + torch.arange(W, device=dev))[:, None]
                for h in range(H_kv):
                    s = torch.einsum("igd,jd->igj", q[b, :, h * g:(h + 1) * g].float(),
                                     kb[:, h]) / math.sqrt(d)
                    s.masked_fill_(mask[:, None, :], float("-inf"))
                    lse[b, :, h * g:(h + 1) * g] = torch.logsumexp(s, dim=-1)
                    del s
            row0 += L
        lses.append(lse)
    streams = [torch.cuda.Stream() for _ in range(ns)]
    events = [torch.cuda.Event() for _ in range(ns + 1)]
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        S.compress_layers(data, seqlens, W, kp, pool, C, outs, wsl, streams, events, stream=cap,
                          lse_wins=lses)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            S.compress_layers(data, seqlens, W, kp, pool, C, outs, wsl, streams, events,
                              stream=cap, lse_wins=lses)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 5
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    assert S.get_status(wsl) == S.OK
    us = 1e3 * a.elapsed_time(b) / reps / len(data)
    return {"us_per_layer": us, "tokens_per_s": sum(seqlens) / (us / 1e6),
            "frac_compress": compress_bytes / (us / 1e6) / 1e9 / peak,
            "note": "the step with the caller's window LSE (pass 2 only), through "
                    f"snapkv_compress_layers ({ns} layer streams), captured in a CUDA graph; "
                    "the LSE comes from torch on the device, outside the timed region"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import synth

    name = args.workload
    cfg = synth.CONFIGS[name]
    layers = args.layers or cfg["layers"]
    lay = synth.make_layer(name, 0)
    for _ in range(args.warmup):
        cpu_baseline(name, layers, lay=lay)
    vals = []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        vals.append(cpu_baseline(name, layers, lay=lay))
    wall = time.perf_counter() - t0
    v = statistics.median(x["value"] for x in vals)
    seqlens = synth.config_seqlens(name)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{name}: {cfg['desc']}", "seqlens": seqlens if len(seqlens) <= 16
                   else len(seqlens), "layers": layers,
                   "step": "oracle on a bounded sample: one full layer, all KV heads"},
        "cpu_baseline": {"kind": "oracle", "cores": vals[0]["cores"],
                         "host_cores": vals[0]["host_cores"], "threads": vals[0]["threads"],
                         "sample": vals[0]["sample"], "value": v, "unit": UNIT},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.case:
        profile_case(args.case)
        return

    import torch
    import torch.distributed as dist

    import synth
    from synth.device import make_layer_device
    from prefill_kv_cache_gb300 import snapkv as S

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    S.load()

    name = args.workload
    cfg = synth.CONFIGS[name]
    layers = args.layers or cfg["layers"]
    W, C, kp, pool = cfg["W"], cfg["C"], cfg["k_pool"], cfg["pool"]
    esz = 2 if cfg["dtype"] == "bf16" else 4

    data = []
    for l in range(layers):
        q, k, v, seqlens = make_layer_device(name, l + 1000 * rank, dev)
        data.append((q, k, v))
    B = len(seqlens)
    H_q, H_kv, d = cfg["H_q"], cfg["H_kv"], cfg["d"]
    dt = data[0][1].dtype
    outs = [(torch.empty((B, C, H_kv, d), dtype=dt, device=dev),
             torch.empty((B, C, H_kv, d), dtype=dt, device=dev),
             torch.empty((B, H_kv, C), dtype=torch.int32, device=dev)) for _ in range(layers)]
    shape = S.make_shape(B, H_q, H_kv, d, dt)
    ws = torch.empty(S.workspace_size(shape, seqlens, W, C), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    lib = S.load()
    sl_arr = (ctypes.c_int32 * B)(*seqlens)
    pool_code = S.pool_code(pool)
    sh_ref = ctypes.byref(shape)
    ws_ptr, ws_len = ws.data_ptr(), ws.numel()
    st = stream.cuda_stream
    calls = [(q.data_ptr(), k.data_ptr(), v.data_ptr(), ok.data_ptr(), ov.data_ptr(), oi.data_ptr())
             for (q, k, v), (ok, ov, oi) in zip(data, outs)]

    def single_calls():
        """Every layer through snapkv_compress, one after another on one stream."""
        for qp, kp_, vp, okp, ovp, oip in calls:
            rc = lib.snapkv_compress(sh_ref, qp, kp_, vp, sl_arr, W, kp, pool_code, C, okp, ovp,
                                     oip, ws_ptr, ws_len, st)
            if rc:
                raise S.SnapKVError(rc, "snapkv_compress")

    # the step: all layers in one snapkv_compress_layers call (consecutive
    # layers on two streams, so that a layer's selection overlaps the next
    # layer's scoring)
    ns = args.layer_streams
    wsl = torch.empty(S.workspace_size_layers(shape, seqlens, W, C, ns), dtype=torch.uint8,
                      device=dev)
    layer_streams = [torch.cuda.Stream() for _ in range(ns)]
    layer_events = [torch.cuda.Event() for _ in range(ns + 1)]
    for e in layer_events:
        e.record(stream)
    arrs = [(ctypes.c_void_p * layers)(*[c[j] for c in calls]) for j in range(6)]
    ls_arr = (ctypes.c_void_p * ns)(*[x.cuda_stream for x in layer_streams])
    ev_arr = (ctypes.c_void_p * (ns + 1))(*[e.cuda_event for e in layer_events])

    def step():
        rc = lib.snapkv_compress_layers(sh_ref, layers, arrs[0], arrs[1], arrs[2], None, sl_arr, W, kp,
                                        pool_code, C, arrs[3], arrs[4], arrs[5], wsl.data_ptr(),
                                        wsl.numel(), st, ns, ls_arr, ev_arr)
        if rc:
            raise S.SnapKVError(rc, "snapkv_compress_layers")

    def barrier():
        if world > 1:
            dist.barrier()

    # every layer through snapkv_compress on one stream: warm-up, timing and
    # the reference outputs of layer 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max(3, args.warmup)):
        single_calls()
    torch.cuda.synchronize()
    assert S.get_status(ws) == S.OK
    e0.record(stream)
    for _ in range(max(1, args.steps // 2)):
        single_calls()
    e1.record(stream)
    torch.cuda.synchronize()
    single_ms = e0.elapsed_time(e1) / max(1, args.steps // 2)
    ref0 = [t.clone() for t in outs[0]]

    # the step issued directly
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert S.get_status(wsl) == S.OK
    e0.record(stream)
    for _ in range(max(1, args.steps // 2)):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / max(1, args.steps // 2)
    for a, b in zip(outs[0], ref0):
        assert torch.equal(a, b), "snapkv_compress_layers differs from snapkv_compress"

    # the same calls captured once (launches recorded at capture time)
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        n_cap = S.kernel_launches()
        with torch.cuda.stream(cap):
            st = cap.cuda_stream
            with torch.cuda.graph(graph, stream=cap):
                step()
            st = stream.cuda_stream
        per_step_launches = S.kernel_launches() - n_cap
        for t in outs[0]:
            t.zero_()
        for _ in range(max(3, args.warmup)):
            graph.replay()
        torch.cuda.synchronize()
        assert S.get_status(wsl) == S.OK
        for a, b in zip(outs[0], ref0):
            assert torch.equal(a, b), "a replayed layer differs from snapkv_compress's"

    sampler = ClockSampler(local_rank)
    barrier()
    torch.cuda.synchronize()
    n0 = S.kernel_launches()
    sampler.start()
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step()
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.stop()
    launches = (per_step_launches * args.steps if graph is not None
                else S.kernel_launches() - n0)
    assert S.get_status(wsl) == S.OK
    barrier()
    ms = replica_ms(e0.elapsed_time(e1) / args.steps, world, dev)
    value = replica_value(sum(seqlens) * layers, world, ms)

    # score kernel alone, per launch, on the launching stream
    score_ms = []
    for _ in range(2):
        for (q, k, _), _o in zip(data, outs):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rc = lib.snapkv_score(sh_ref, q.data_ptr(), k.data_ptr(), sl_arr, W, C, ws_ptr,
                                  ws_len, st)
            b.record(stream)
            if rc:
                raise S.SnapKVError(rc, "snapkv_score")
            score_ms.append((a, b))
    torch.cuda.synchronize()
    score_avg_ms = statistics.mean(a.elapsed_time(b) for a, b in score_ms[len(data):])
    score_bytes, compress_bytes = workload_bytes(cfg, seqlens, esz)
    peak, peak_kind = hbm_peak()
    achieved = score_bytes / (score_avg_ms / 1e3) / 1e9
    flops, exps = score_work(cfg, seqlens)
    tc_peak, tc_kind, mufu_peak, mufu_kind = compute_peaks(
        torch.cuda.get_device_properties(dev).multi_processor_count)
    tensor_cores = cfg["dtype"] == "bf16" and cfg["W"] * H_q // H_kv in (128, 256)
    compress_gbs = compress_bytes / (ms / layers / 1e3) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "score_kernel_traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                tinfo = json.load(f)
            if tinfo.get("workload") == name and tinfo.get("kernel_version") == S.load().snapkv_version():
                traffic = tinfo.get("bytes_per_launch")
        except Exception:
            traffic = None

    lse_input = None
    if not args.no_lse and cfg["dtype"] == "bf16":
        lse_input = lse_input_step(S, torch, data, outs, wsl, seqlens, cfg, dev, ns, peak,
                                   compress_bytes)

    decode = decode_step(S, torch, data, outs, seqlens, cfg, dev, stream, peak)
    sh_decode = None
    if not args.no_scissorhands:
        sh_decode = scissorhands_decode(torch, outs, seqlens, cfg, dev, stream, peak)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(S, torch, data, seqlens, cfg, shape, dev, stream, args, layers)

    workloads = None
    if rank == 0 and name == "4" and not args.no_workloads:
        workloads = workload_table(S, torch, dev, peak, layer_streams=ns)

    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, (lay0, ora0) = cpu_baseline(name, layers, keep_first=True)
        cpu["single_thread_cfg2_tokens_per_s"] = single_thread_baseline("2")
        parity = parity_vs_oracle(S, torch, lay0, ora0, cfg, dev)

    if rank == 0:
        clk = sampler.summary()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": cfg["dtype"], "data": "synthetic",
            "config": {
                "workload": f"{name}: {cfg['desc']}",
                "seqlens": seqlens if len(seqlens) <= 16 else len(seqlens),
                "layers": layers, "us_per_layer": 1e3 * ms / layers,
                "step": f"one snapkv_compress_layers call over all layers ({ns} layer streams)",
                "timing": "the step captured in a CUDA graph, replayed" if graph is not None
                          else "the step issued directly",
                "us_per_layer_eager": 1e3 * eager_ms / layers,
                "us_per_layer_single_calls": 1e3 * single_ms / layers,
                "l2": "inputs larger than L2 (each layer's K and V: "
                      f"{2 * sum(seqlens) * H_kv * d * esz / 1e6:.0f} MB)",
                "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            },
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": "score (snapkv_score)", "peak_kind": peak_kind,
                         "us_per_launch": 1e3 * score_avg_ms,
                         "bytes_per_launch": score_bytes},
            "roofline_compress": {"achieved": compress_gbs, "peak": peak, "unit": "GB/s",
                                  "frac": compress_gbs / peak, "bytes_per_layer": compress_bytes},
            # the same launch against its compute ceilings (two passes recompute the logits)
            "roofline_tensor": None if not tensor_cores else {
                "bound": "tensor", "achieved": flops / (score_avg_ms / 1e3) / 1e12,
                "peak": tc_peak, "unit": "TFLOP/s",
                "frac": flops / (score_avg_ms / 1e3) / 1e12 / tc_peak,
                "flops_per_launch": flops, "peak_kind": tc_kind},
            "roofline_mufu": {
                "bound": "alu", "achieved": exps / (score_avg_ms / 1e3) / 1e12,
                "peak": mufu_peak, "unit": "T exp2/s",
                "frac": exps / (score_avg_ms / 1e3) / 1e12 / mufu_peak,
                "exp2_per_launch": exps, "peak_kind": mufu_kind},
            "cpu_baseline": cpu,
            "parity": parity,
            "workloads": workloads,
            "lse_input": lse_input,
            "e2e": e2e,
            "decode": decode,
            "scissorhands": sh_decode,
            "gpu_launches": launches,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def profile_case(name: str) -> None:
    """Small fixed cases for ncu (a few hundred MB on the device, a handful of
    launches): 'decode' = four decode steps over one 131072-token Llama-3-8B
    layer cache; 'scissorhands' = 40 Scissorhands steps (budget 4096, r = 10,
    w = 400, batches of 2048) of one layer starting from a full cache, so the
    first step evicts."""
    import torch

    from prefill_kv_cache_gb300 import scissorhands as SH
    from prefill_kv_cache_gb300 import snapkv as S

    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    rnd = lambda *shape: torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    if name == "decode":
        L = 131072
        k, v, q = rnd(L, 8, 128), rnd(L, 8, 128), rnd(1, 32, 128)
        for _ in range(4):
            S.decode_attention(q, k, v, [L], S.CACHE_PACKED)
    else:
        c = SH.Cache(1, 32, 8, 128, torch.bfloat16, SH.Params(budget=4096))
        c.init([4096], [131072], rnd(1, 4096, 8, 128), rnd(1, 4096, 8, 128))
        q, kn, vn = rnd(1, 32, 128), rnd(1, 8, 128), rnd(1, 8, 128)
        for _ in range(40):
            c.step(q, kn, vn)
    torch.cuda.synchronize()
    print(f"case {name}: ok")


def replica_ms(ms_local: float, world: int, dev) -> float:
    """Step time of the whole job: the slowest replica's (max over ranks).
    The replicas share nothing on the data path: this reduction and the
    barriers around the timed region are the only collectives."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist

    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(tokens_per_step_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank compresses its own layers (weak
    scaling), all ranks' tokens over the slowest rank's time."""
    return tokens_per_step_per_rank * world / (ms / 1e3)


def decode_step(S, torch, data, outs, seqlens, cfg, dev, stream, peak, reps=5):
    """One decode step (one query token per sequence) through every layer,
    over the full prompt cache and over the compressed cache the timed
    compression just wrote (snapkv_decode_attention; the decode phase of the
    glossary's algorithm flow, step 4).  Each layer's cache is its own buffer,
    so the 32-layer sweep streams from HBM."""
    B = len(seqlens)
    H_q, H_kv, d, C = cfg["H_q"], cfg["H_kv"], cfg["d"], cfg["C"]
    dt = data[0][1].dtype
    gen = torch.Generator(device=dev)
    gen.manual_seed(77)
    qs = [torch.randn((B, H_q, d), generator=gen, device=dev).to(dt) for _ in data]
    lens_c = [min(int(L), C) for L in seqlens]
    shape = S.make_shape(B, H_q, H_kv, d, dt)
    ws = torch.empty(max(S.decode_workspace_size(shape, seqlens, S.CACHE_PACKED),
                         S.decode_workspace_size(shape, lens_c, S.CACHE_SLOTS, C)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, H_q, d), dtype=torch.float32, device=dev)

    def sweep(compressed, st):
        for q, (_, k, v), (ok, ov, _) in zip(qs, data, outs):
            if compressed:
                S.decode_attention(q, ok, ov, lens_c, S.CACHE_SLOTS, C, out=out, workspace=ws,
                                   stream=st)
            else:
                S.decode_attention(q, k, v, seqlens, S.CACHE_PACKED, out=out, workspace=ws,
                                   stream=st)

    # the sweep is captured in a CUDA graph, so host launch cost is not timed
    # (a decode step's per-layer kernels are short)
    res = {}
    cap = torch.cuda.Stream(device=dev)
    for tag, comp, rows in (("full", False, sum(seqlens)), ("compressed", True, sum(lens_c))):
        for _ in range(3):
            sweep(comp, stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            sweep(comp, cap)
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
        us = 1e3 * a.elapsed_time(b) / reps / len(data)
        nbytes = 2 * rows * H_kv * d * data[0][1].element_size()
        res[f"us_per_layer_{tag}"] = us
        res[f"gbs_{tag}"] = nbytes / us / 1e3
        res[f"frac_{tag}"] = nbytes / us / 1e3 / peak
    res["speedup"] = res["us_per_layer_full"] / res["us_per_layer_compressed"]
    res["note"] = ("one query token per sequence, all layers back to back in one CUDA graph; "
                   "K and V bytes read once per layer are the roofline bytes")
    return res


def scissorhands_decode(torch, outs, seqlens, cfg, dev, stream, peak):
    """Decode steps with Scissorhands eviction (scissorhands_step) through
    every layer, each layer's cache starting from the compressed cache the
    timed compression wrote, with the settings of the Scissorhands page:
    budget = C, r = 10, w = 400, batches of C / 2.  One step of all layers is
    captured in a CUDA graph; the state lives on the device, so each replay is
    the next decode step.  Timed: the first step (the cache starts full, so it
    evicts) and then one whole eviction period of C / 2 steps."""
    from prefill_kv_cache_gb300 import scissorhands as SH

    B = len(seqlens)
    H_q, H_kv, d, C = cfg["H_q"], cfg["H_kv"], cfg["d"], cfg["C"]
    dt = outs[0][0].dtype
    prm = SH.Params(budget=C, recent=10, history=400, evict=C // 2)
    caches = [SH.Cache(B, H_q, H_kv, d, dt, prm, device=dev) for _ in outs]
    gen = torch.Generator(device=dev)
    gen.manual_seed(78)
    qs, ks, vs = ([torch.randn((B, n, d), generator=gen, device=dev).to(dt) for _ in outs]
                  for n in (H_q, H_kv, H_kv))
    out = torch.empty((B, H_q, d), dtype=torch.float32, device=dev)
    lens_c = [min(int(L), C) for L in seqlens]

    def init():
        for c, (ok, ov, oi) in zip(caches, outs):
            c.init(lens_c, seqlens, ok, ov, oi, stream=stream)

    def sweep(st):
        for c, q, k, v in zip(caches, qs, ks, vs):
            c.step(q, k, v, out=out, stream=st)

    init()
    for _ in range(3):
        sweep(stream)
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        sweep(cap)
    init()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    period = prm.c().evict
    ev[0].record()
    graph.replay()
    ev[1].record()
    for _ in range(period):
        graph.replay()
    ev[2].record()
    torch.cuda.synchronize()
    layers = len(outs)
    n = list(lens_c)
    rows = []
    for t in range(period + 1):
        n = [x + 1 - (period if x + 1 > C else 0) for x in n]
        if t > 0:
            rows.append(sum(n))
    rows_mean = statistics.mean(rows)
    us_first = 1e3 * ev[0].elapsed_time(ev[1]) / layers
    us_mean = 1e3 * ev[1].elapsed_time(ev[2]) / period / layers
    nbytes = 2 * rows_mean * H_kv * d * outs[0][0].element_size()
    return {
        "budget": C, "recent": 10, "history": 400, "evict": period,
        "us_per_layer_step": us_mean, "us_per_layer_evicting_step": us_first,
        "rows_mean": rows_mean, "gbs": nbytes / us_mean / 1e3,
        "frac": nbytes / us_mean / 1e3 / peak,
        "note": ("mean over one eviction period (the last step evicts), all layers back to "
                 "back in one CUDA graph; the K and V bytes of the rows attended are the "
                 "roofline bytes"),
    }


def run_e2e(S, torch, data, seqlens, cfg, shape, dev, stream, args, layers):
    """Same metric through snapkv_compress_host_layers: pinned host in, pinned
    host out, every layer of a step in one call, each layer's upload
    overlapping the previous layer's compression (V stays on the host; the
    gather reads the kept rows in place)."""
    W, C, kp, pool = cfg["W"], cfg["C"], cfg["k_pool"], cfg["pool"]
    B = len(seqlens)
    H_kv, d = cfg["H_kv"], cfg["d"]
    dt = data[0][1].dtype
    host = []
    for layer in data:
        hl = []
        for x in layer:
            h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
            h.copy_(x)
            hl.append(h)
        host.append(tuple(hl))
    outs = [(torch.empty((B, C, H_kv, d), dtype=dt).pin_memory(),
             torch.empty((B, C, H_kv, d), dtype=dt).pin_memory(),
             torch.empty((B, H_kv, C), dtype=torch.int32).pin_memory()) for _ in range(layers)]
    staging = torch.empty(S.host_staging_size_layers(shape, seqlens, W, C), dtype=torch.uint8,
                          device=dev)
    copy_stream = torch.cuda.Stream(device=dev)
    events = [torch.cuda.Event() for _ in range(4)]

    def step():
        S.compress_host_layers(host, seqlens, W, kp, pool, C, outs, staging, stream,
                               copy_stream, events)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    sec = (time.perf_counter() - t0) / args.steps
    # q_win and K are copied whole; page-locked V is read in place by the
    # gather, so only the kept rows (C per sequence and KV head) cross the link
    kept_v = sum(min(int(L), C) for L in seqlens) * H_kv * d * host[0][2].element_size()
    h2d = sum(q.numel() * q.element_size() + k.numel() * k.element_size() + kept_v
              for q, k, _ in host)
    d2h = sum(sum(x.numel() * x.element_size() for x in o) for o in outs)
    # the host link alone: one layer's K, page-locked host -> device
    kh = host[0][1]
    kd = torch.empty(kh.shape, dtype=kh.dtype, device=dev)
    kd.copy_(kh, non_blocking=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        kd.copy_(kh, non_blocking=True)
    torch.cuda.synchronize()
    link = 3 * kh.numel() * kh.element_size() / (time.perf_counter() - t0) / 1e9
    return {"value": sum(seqlens) * layers / sec, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * sec,
            "h2d_gbs_effective": h2d / sec / 1e9, "h2d_link_gbs": link,
            "note": ("all layers of a step in one snapkv_compress_host_layers call; "
                     "h2d_link_gbs: a plain page-locked host-to-device copy of one layer's K, "
                     "the ceiling of the host link")}


if __name__ == "__main__":
    main()
