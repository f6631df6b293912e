#!/usr/bin/env python3
"""Benchmark of the fused LayerNorm -> modulate -> FP8 row path on GB300.

One step = one pass of the path over one batch: a single fp8q_nss_fp8 launch over the
Qwen-Image activation x bf16 [4608, 3072] (4096 image + 512 text tokens), emitting bf16 y
and E4M3 q. `value` is rows/s with inputs resident in HBM; `e2e` is the same metric through
the C ABI with pinned host buffers (host->device copy of x and device->host copy of y and q
inside every timed step). The other kernels of the path (scale-residual, bias_mul_add, the
FLUX.2 width-6144 LayerNorm and token-cat) are timed the same way and reported under
`kernels` with their own roofline figures.

Timing: W warm-up steps, then windows of exactly K steps replayed from CUDA graphs on one
stream, each timed with CUDA events recorded as nodes of those graphs (before the first and
after the last launch) and bracketed by a barrier and a device synchronisation; the headline
is the median window. The buffer sets rotate and together exceed 2x L2, so every launch reads
its inputs from HBM. SM clocks are sampled with nvidia-smi during the timed region. Under torchrun each rank runs the same workload on its own GPU (independent
replicas, weak scaling; the only collective is the timing barrier / max-reduce).

  python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused norm-modulate-FP8 rows/s and achieved HBM GB/s (% of GB300 peak)"
FALLBACK_HBM_GBS = 6800.0
GRAPH_CHUNK = 500


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, torch copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and blank-line or indentation differences (string
    literals are kept as they are; the sources' asm strings hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments excluded), which keys the committed ncu
    counters: a change to the code makes them stale, a change to a comment does not."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fp8_quant_row_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key: str):
    """dram bytes per launch from the committed ncu summary, only if the kernel sources are
    unchanged since it was captured."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
    except Exception:
        return None
    if d.get("source_hash") != kernel_source_hash():
        return None
    e = d.get("kernels", {}).get(kernel_key)
    return None if e is None else e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------------------------------
# clocks
# ------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.samples = []
        self.proc = None
        self.thread = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if uuid:
            cmd += ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception as e:  # nvidia-smi missing: report no samples
            log("clock sampler unavailable:", e)
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                self.samples.append((time.time(), float(parts[2]), float(parts[3]),
                                     parts[6], parts[7], parts[8], parts[9]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if not inside:
            inside, window = self.samples, "whole run (timed region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in inside:
            for name, v in zip(names, s[3:]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[1] for s in inside),
                "sm_max_mhz": max(s[2] for s in inside), "reasons": sorted(reasons),
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def dev_bf16(torch, a):
    import numpy as np
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def n_sets_for(bytes_per_set: int, l2: int) -> int:
    return max(2, math.ceil(2 * l2 / bytes_per_set) + 1)


class Case:
    """A kernel launch over rotating buffer sets: launch(i) runs on set i % n."""

    def __init__(self, name, launch, n_sets, alg_bytes, rows, ncu_key, describe):
        self.name, self.launch, self.n_sets = name, launch, n_sets
        self.alg_bytes, self.rows, self.ncu_key, self.describe = alg_bytes, rows, ncu_key, describe


def make_cases(torch, fq, lib, l2):
    import numpy as np
    import workloads as W

    cases = {}
    stream_handle = lambda: torch.cuda.current_stream().cuda_stream

    # main: nss_fp8 Qwen-Image
    c = W.CONFIGS["nss_qwen"]
    inp = W.config_inputs("nss_qwen")
    R, C = inp["x"].shape
    per_set = R * C * 5
    n = n_sets_for(per_set, l2)
    xs = [dev_bf16(torch, inp["x"]) for _ in range(n)]
    ys = [torch.empty(R, C, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    qs = [torch.empty(R, C, dtype=torch.uint8, device="cuda") for _ in range(n)]
    sc, sh = dev_bf16(torch, inp["scale"]), dev_bf16(torch, inp["shift"])
    s = torch.tensor([c["input_scale"]], dtype=torch.float32, device="cuda")
    ptrs = [(ys[i].data_ptr(), qs[i].data_ptr(), xs[i].data_ptr()) for i in range(n)]

    def nss_launch(i, ptrs=ptrs, sc=sc.data_ptr(), sh=sh.data_ptr(), s=s.data_ptr()):
        y, q, x = ptrs[i % len(ptrs)]
        st = lib.fp8q_nss_fp8(y, q, x, sc, sh, 0, s, R, C, 1e-6, stream_handle())
        if st:
            raise RuntimeError(f"fp8q_nss_fp8 status {st}")

    cases["nss_qwen"] = Case("nss_fp8", nss_launch, n, per_set, R, "nss_fp8_qwen",
                             f"nss_fp8 Qwen-Image x bf16 [{R},{C}] -> y bf16 + q e4m3, "
                             f"input_scale {c['input_scale']}")
    cases["nss_qwen"].keep = (xs, ys, qs, sc, sh, s, inp)
    return cases


def extra_cases(torch, lib, l2, only=None):
    """The per-kernel cases: all of them, or only the one named `only`."""
    import workloads as W

    sh_ = lambda: torch.cuda.current_stream().cuda_stream

    def scale_residual_qwen():
        c = W.CONFIGS["scale_residual_qwen"]
        inp = W.config_inputs("scale_residual_qwen")
        R, C = inp["x"].shape
        per = R * C * 9
        n = n_sets_for(per, l2)
        bufs = [dict(x=dev_bf16(torch, inp["x"]), r=dev_bf16(torch, inp["residual"]),
                     ro=torch.empty(R, C, dtype=torch.bfloat16, device="cuda"),
                     y=torch.empty(R, C, dtype=torch.bfloat16, device="cuda"),
                     q=torch.empty(R, C, dtype=torch.uint8, device="cuda")) for _ in range(n)]
        vec = {k: dev_bf16(torch, inp[k]) for k in ("bias", "gate", "scale", "shift")}
        s = torch.tensor([c["input_scale"]], dtype=torch.float32, device="cuda")

        def sr(i):
            b = bufs[i % len(bufs)]
            st = lib.fp8q_scale_residual_nss_fp8(
                b["ro"].data_ptr(), b["y"].data_ptr(), b["q"].data_ptr(), b["x"].data_ptr(),
                b["r"].data_ptr(), vec["bias"].data_ptr(), vec["gate"].data_ptr(),
                vec["scale"].data_ptr(), vec["shift"].data_ptr(), 0, s.data_ptr(), R, C, 1e-6,
                sh_())
            if st:
                raise RuntimeError(f"scale_residual status {st}")

        case = Case("scale_residual_nss_fp8", sr, n, per, R, "scale_residual_nss_fp8_qwen",
                    f"x, residual bf16 [{R},{C}] + bias -> residual_out, y, q")
        case.keep = (bufs, vec, s)
        return case

    def bias_mul_add_qwen():
        inp = W.config_inputs("bias_mul_add_qwen")
        R, C = inp["x"].shape
        per = R * C * 6
        n = n_sets_for(per, l2)
        bufs = [dict(x=dev_bf16(torch, inp["x"]), r=dev_bf16(torch, inp["residual"]),
                     y=torch.empty(R, C, dtype=torch.bfloat16, device="cuda")) for _ in range(n)]
        b, g = dev_bf16(torch, inp["bias"]), dev_bf16(torch, inp["gate"][0])

        def bma(i):
            d = bufs[i % len(bufs)]
            st = lib.fp8q_bias_mul_add(d["y"].data_ptr(), d["x"].data_ptr(), b.data_ptr(),
                                       g.data_ptr(), d["r"].data_ptr(), R, C, sh_())
            if st:
                raise RuntimeError(f"bias_mul_add status {st}")

        case = Case("bias_mul_add", bma, n, per, R, "bias_mul_add_qwen",
                    f"x, residual bf16 [{R},{C}] -> y bf16")
        case.keep = (bufs, b, g)
        return case

    def nss_tiny():
        c = W.CONFIGS["nss_tiny"]
        inp = W.config_inputs("nss_tiny")
        R, C = inp["x"].shape
        per = R * C * 5
        n = n_sets_for(per, l2)
        bufs = [dict(x=dev_bf16(torch, inp["x"]),
                     y=torch.empty(R, C, dtype=torch.bfloat16, device="cuda"),
                     q=torch.empty(R, C, dtype=torch.uint8, device="cuda")) for _ in range(n)]
        sc, shf = dev_bf16(torch, inp["scale"]), dev_bf16(torch, inp["shift"])
        s = torch.tensor([c["input_scale"]], dtype=torch.float32, device="cuda")

        def nt(i):
            d = bufs[i % len(bufs)]
            st = lib.fp8q_nss_fp8(d["y"].data_ptr(), d["q"].data_ptr(), d["x"].data_ptr(),
                                  sc.data_ptr(), shf.data_ptr(), 0, s.data_ptr(), R, C, 1e-6,
                                  sh_())
            if st:
                raise RuntimeError(f"nss tiny status {st}")

        case = Case("nss_fp8", nt, n, per, R, "nss_fp8_tiny",
                    f"x bf16 [{R},{C}], latency-bound ({R} rows over all SMs); {n} rotating "
                    f"buffer sets keep the inputs cold")
        case.keep = (bufs, sc, shf, s)
        return case

    def nss_flux():
        c = W.CONFIGS["nss_flux"]
        inp = W.config_inputs("nss_flux")
        R, C = inp["x"].shape
        per = R * C * 5
        n = n_sets_for(per, l2)
        bufs = [dict(x=dev_bf16(torch, inp["x"]),
                     y=torch.empty(R, C, dtype=torch.bfloat16, device="cuda"),
                     q=torch.empty(R, C, dtype=torch.uint8, device="cuda")) for _ in range(n)]
        sc, shf = dev_bf16(torch, inp["scale"]), dev_bf16(torch, inp["shift"])
        s = torch.tensor([c["input_scale"]], dtype=torch.float32, device="cuda")
        mr = c["mod_rows"]

        def nf(i):
            d = bufs[i % len(bufs)]
            st = lib.fp8q_nss_fp8(d["y"].data_ptr(), d["q"].data_ptr(), d["x"].data_ptr(),
                                  sc.data_ptr(), shf.data_ptr(), mr, s.data_ptr(), R, C, 1e-6,
                                  sh_())
            if st:
                raise RuntimeError(f"nss flux status {st}")

        case = Case("nss_fp8", nf, n, per, R, "nss_fp8_flux",
                    f"x bf16 [{R},{C}], scale/shift [2,{C}], mod_rows {mr}")
        case.keep = (bufs, sc, shf, s)
        return case

    def token_cat_flux():
        c = W.CONFIGS["token_cat_flux"]
        inp = W.config_inputs("token_cat_flux")
        R, A = inp["a"].shape
        M = inp["m"].shape[1]
        per = R * (A + M) * 3
        n = n_sets_for(per, l2)
        bufs = [dict(a=dev_bf16(torch, inp["a"]), m=dev_bf16(torch, inp["m"]),
                     q=torch.empty(R, A + M, dtype=torch.uint8, device="cuda")) for _ in range(n)]
        s = torch.tensor([c["input_scale"]], dtype=torch.float32, device="cuda")

        def tc(i):
            d = bufs[i % len(bufs)]
            st = lib.fp8q_token_cat_fp8(d["q"].data_ptr(), d["a"].data_ptr(), A,
                                        d["m"].data_ptr(), M, s.data_ptr(), R, sh_())
            if st:
                raise RuntimeError(f"token_cat status {st}")

        case = Case("token_cat_fp8", tc, n, per, R, "token_cat_fp8_flux",
                    f"a bf16 [{R},{A}] + m bf16 [{R},{M}] -> q e4m3 [{R},{A + M}]")
        case.keep = (bufs, s)
        return case

    def token_cat_nvfp4_flux(rows=None):
        c = W.CONFIGS["token_cat_nvfp4_flux"]
        inp = W.config_inputs("token_cat_nvfp4_flux", rows=rows)
        R, A = inp["a"].shape
        M = inp["m"].shape[1]
        K = (A + M) // 16
        sf_bytes = lib.fp8q_nvfp4_scale_bytes(R, A + M)
        per = R * (A + M) * 2 + R * (A + M) // 2 + sf_bytes
        n = n_sets_for(per, l2)
        bufs = [dict(a=dev_bf16(torch, inp["a"]), m=dev_bf16(torch, inp["m"]),
                     q=torch.empty(R, (A + M) // 2, dtype=torch.uint8, device="cuda"),
                     sf=torch.empty(sf_bytes, dtype=torch.uint8, device="cuda"))
                for _ in range(n)]
        s = torch.tensor([c["global_scale"]], dtype=torch.float32, device="cuda")

        def tc4(i):
            d = bufs[i % len(bufs)]
            st = lib.fp8q_token_cat_nvfp4(d["q"].data_ptr(), d["sf"].data_ptr(),
                                          d["a"].data_ptr(), A, d["m"].data_ptr(), M,
                                          s.data_ptr(), R, sh_())
            if st:
                raise RuntimeError(f"token_cat_nvfp4 status {st}")

        case = Case("token_cat_nvfp4", tc4, n, per, R,
                    "token_cat_nvfp4_flux" if rows is None else f"token_cat_nvfp4_flux_{rows}",
                    f"a bf16 [{R},{A}] + m bf16 [{R},{M}] -> q e2m1 [{R},{(A + M) // 2}] "
                    f"bytes + {K} e4m3 block scales per row (128x4 tiles), global scale "
                    f"{c['global_scale']}")
        case.keep = (bufs, s)
        return case

    def qkv(name):
        import fp8_quant_row_gb300._capi as capi
        c = W.CONFIGS[name]
        d = W.config_inputs(name)
        H = c["heads"]
        T = c["txt_tokens"] + c["img_tokens"]
        per = T * (3 * H * 128 * 2 * 2 + 128 * 4)
        n = n_sets_for(per, l2)
        sets = []
        for _ in range(n):
            streams, keep = [], []
            for key in ("txt", "img"):
                st = d[key]
                packed = dev_bf16(torch, st["packed"])
                wq, wk = dev_bf16(torch, st["wq"]), dev_bf16(torch, st["wk"])
                cs = torch.from_numpy(st["cos_sin"]).cuda()
                hd = H * 128
                streams.append(capi.QkvStream(packed.data_ptr(), packed.data_ptr() + hd * 2,
                                              packed.data_ptr() + 2 * hd * 2, packed.shape[1],
                                              packed.shape[0], wq.data_ptr(), wk.data_ptr(),
                                              cs.data_ptr(), st["eps"]))
                keep += [packed, wq, wk, cs]
            outs = [torch.empty(T, H, 128, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
            sets.append((streams, outs, keep))

        def run_qkv(i):
            streams, outs, _ = sets[i % len(sets)]
            st = lib.fp8q_qkv_epilogue(outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(),
                                       streams[0], streams[1], H, sh_())
            if st:
                raise RuntimeError(f"qkv_epilogue status {st}")

        case = Case("qkv_epilogue", run_qkv, n, per, T, f"qkv_epilogue_{name[4:]}",
                    f"packed QKV bf16 text [{c['txt_tokens']},{3 * H * 128}] + image "
                    f"[{c['img_tokens']},{3 * H * 128}], {H} heads x 128 -> joint q, k, v "
                    f"[{T},{H},128] (RMSNorm + interleaved RoPE on q, k)")
        case.keep = sets
        return case

    builders = {"nss_tiny": nss_tiny,
                "scale_residual_qwen": scale_residual_qwen, "bias_mul_add_qwen": bias_mul_add_qwen,
                "nss_flux": nss_flux, "token_cat_flux": token_cat_flux,
                "token_cat_nvfp4_flux": token_cat_nvfp4_flux,
                # the pages' token-cat microbenchmark token counts (latency end)
                "token_cat_nvfp4_flux_17": lambda: token_cat_nvfp4_flux(17),
                "token_cat_nvfp4_flux_512": lambda: token_cat_nvfp4_flux(512),
                "token_cat_nvfp4_flux_4096": lambda: token_cat_nvfp4_flux(4096),
                "qkv_qwen": lambda: qkv("qkv_qwen"), "qkv_flux": lambda: qkv("qkv_flux")}
    return {k: f for k, f in builders.items() if only is None or k == only}


def capture(torch, case: Case, count: int, start: int, ev_first=None, ev_last=None):
    """A graph of `count` launches; ev_first / ev_last (events created with external=True)
    are recorded as graph nodes before the first and after the last launch, so a window's
    time is the device time of exactly its launches, without the host's graph-launch latency
    in front of them."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        if ev_first is not None:
            ev_first.record()
        for i in range(count):
            case.launch(start + i)
        if ev_last is not None:
            ev_last.record()
    return g


def graph_events(torch):
    """Timing events that become event-record nodes when recorded during capture, or None
    where torch lacks them (then the events are recorded on the stream around the replay)."""
    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


def windows_needed(first_window_ms: float, repeats: int, min_region_s: float) -> int:
    """Windows to time: at least `repeats`, and enough that the timed region lasts about
    `min_region_s` (so that the clock sampler sees it), at most 2000."""
    per = max(first_window_ms / 1e3, 1e-6)
    return int(min(2000, max(repeats, math.ceil(min_region_s / per))))


def time_case(torch, case: Case, steps: int, warmup: int, use_graph=True, barrier=None,
              repeats: int = 1, min_region_s: float = 0.0, agree=None):
    """Times windows of exactly `steps` launches. Returns (window_ms list, t0_wall, t1_wall).
    The first window sets how many are timed (windows_needed); `agree` (max over ranks) makes
    every rank time the same number. Each window is bracketed by a barrier and a device
    synchronisation and timed with CUDA events on the launch stream."""
    for i in range(warmup):
        case.launch(i)
    torch.cuda.synchronize()
    graphs = []
    in_graph = graph_events(torch) if use_graph else None
    if use_graph:
        # chunks of GRAPH_CHUNK launches (the last one may be shorter); every chunk starts on
        # a set index that continues the rotation
        done = 0
        while done < steps:
            cnt = min(GRAPH_CHUNK, steps - done)
            first = in_graph[0] if in_graph and done == 0 else None
            last = in_graph[1] if in_graph and done + cnt >= steps else None
            graphs.append(capture(torch, case, cnt, warmup + done, first, last))
            done += cnt
        # one untimed replay to page everything in
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
    if in_graph:
        ev0, ev1 = in_graph
    else:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
    windows = []
    t0 = t1 = None
    while True:
        if barrier:
            barrier()
        torch.cuda.synchronize()
        if t0 is None:
            t0 = time.time()
        if not in_graph:
            ev0.record()
        if use_graph:
            for g in graphs:
                g.replay()
        else:
            for i in range(steps):
                case.launch(warmup + i)
        if not in_graph:
            ev1.record()
        torch.cuda.synchronize()
        t1 = time.time()
        windows.append(ev0.elapsed_time(ev1))
        if len(windows) == 1:
            target = windows_needed(windows[0], repeats, min_region_s)
            if agree is not None:
                target = agree(target)
        if len(windows) >= target:
            break
    if barrier:
        barrier()
    return windows, t0, t1


def e2e_measure(torch, lib, case: Case, steps: int):
    """Same metric through the C ABI with host buffers. Every step copies its x from pinned
    host memory to the device, runs the kernel and copies y and q back to pinned host memory.
    Steps alternate between two streams with their own device and host buffers, so step i+1's
    host-to-device copy overlaps step i's device-to-host copy (both copy directions run at
    once); the timed region spans all K steps on both streams (CUDA events)."""
    xs, ys, qs, sc, sh, s, inp = case.keep
    R, C = inp["x"].shape
    import numpy as np
    hx = torch.from_numpy(np.ascontiguousarray(inp["x"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    nb = 2
    hy = [torch.empty(R, C, dtype=torch.bfloat16).pin_memory() for _ in range(nb)]
    hq = [torch.empty(R, C, dtype=torch.uint8).pin_memory() for _ in range(nb)]
    dx, dy, dq = xs[:nb], ys[:nb], qs[:nb]
    streams = [torch.cuda.Stream() for _ in range(nb)]

    def step(i):
        b = i % nb
        st = streams[b]
        with torch.cuda.stream(st):
            dx[b].copy_(hx, non_blocking=True)
            status = lib.fp8q_nss_fp8(dy[b].data_ptr(), dq[b].data_ptr(), dx[b].data_ptr(),
                                      sc.data_ptr(), sh.data_ptr(), 0, s.data_ptr(), R, C, 1e-6,
                                      st.cuda_stream)
            if status:
                raise RuntimeError(f"status {status}")
            hy[b].copy_(dy[b], non_blocking=True)
            hq[b].copy_(dq[b], non_blocking=True)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(main)
    for st in streams:
        st.wait_event(ev0)
    for i in range(steps):
        step(i)
    for st in streams:
        done = torch.cuda.Event()
        done.record(st)
        main.wait_event(done)
    ev1.record(main)
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    return {"value": R * steps / (ms / 1e3), "unit": "rows/s", "steps": steps,
            "ms_per_step": ms / steps, "h2d_bytes_per_step": R * C * 2,
            "d2h_bytes_per_step": R * C * 3,
            "method": "pinned host buffers; torch copies + C-ABI launch; steps alternate between "
                      "two streams (double-buffered), so one step's H2D overlaps the previous "
                      "step's D2H; CUDA events around all steps"}


def host_cpu() -> str:
    """The host's CPU model and logical core count (lscpu where available)."""
    import platform
    import subprocess
    model = platform.processor() or platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    return f"{model}, {os.cpu_count()} logical cores, {platform.machine()}"


def cpu_baseline(sample_seconds: float = 10.0):
    """The oracle as it stands, single-threaded, on row chunks of the main workload."""
    import numpy as np
    import oracle
    import workloads as W

    c = W.CONFIGS["nss_qwen"]
    inp = W.config_inputs("nss_qwen", rows=256)
    rows_done, t0 = 0, time.perf_counter()
    while True:
        oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], c["input_scale"])
        rows_done += inp["x"].shape[0]
        el = time.perf_counter() - t0
        if el >= sample_seconds:
            break
    return {"value": rows_done / el, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"{rows_done} rows of the nss_fp8 Qwen-Image workload (256-row chunks, "
                      f"{el:.1f} s, single-threaded C oracle, fp64 statistics)"}


def _oracle_rows_for(seconds: float, seed: int):
    """Worker of cpu_baseline_all_cores: the single-threaded oracle on 256-row chunks for
    about `seconds`; returns (rows, elapsed)."""
    import oracle
    import workloads as W
    c = W.CONFIGS["nss_qwen"]
    inp = W.config_inputs("nss_qwen", rows=256, seed=seed)
    rows_done, t0 = 0, time.perf_counter()
    while True:
        oracle.nss_fp8(inp["x"], inp["scale"], inp["shift"], c["input_scale"])
        rows_done += inp["x"].shape[0]
        el = time.perf_counter() - t0
        if el >= seconds:
            return rows_done, el


def cpu_baseline_all_cores(sample_seconds: float = 10.0):
    """The same oracle, one process per host core (spawned), each on its own row chunks."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    t0 = time.perf_counter()
    with ctx.Pool(n) as pool:
        res = pool.starmap(_oracle_rows_for, [(sample_seconds, 100 + i) for i in range(n)])
    wall = time.perf_counter() - t0
    rows = sum(r for r, _ in res)
    el = max(e for _, e in res)
    return {"value": rows / el, "unit": "rows/s", "cores": n, "kind": "oracle",
            "host": host_cpu(),
            "sample": f"{rows} rows of the nss_fp8 Qwen-Image workload, {n} spawned processes "
                      f"x ~{sample_seconds:.0f} s of 256-row chunks (rate over the slowest "
                      f"process's time; {wall:.1f} s wall with start-up)"}


def roofline_entry(case: Case, ms_per_launch: float, peak: float, peak_src: str):
    achieved = case.alg_bytes / (ms_per_launch / 1e3) / 1e9
    traffic = ncu_traffic(case.ncu_key)
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": case.alg_bytes, "peak_source": peak_src,
            "kernel": case.name}


def max_over_ranks(ms: float, device: str = "cuda") -> float:
    """Slowest rank's elapsed time (the job finishes when the last replica does)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank processes rows_per_step rows per step."""
    return rows_per_step * steps * world / (max_ms / 1e3)


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)

    import fp8_quant_row_gb300 as fq
    fq.build()
    lib = fq._capi.lib()
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    peak, peak_src = peaks()

    cases = make_cases(torch, fq, lib, l2)
    main = cases["nss_qwen"]

    def barrier():
        if world > 1:
            dist.barrier()

    sampler = ClockSampler(getattr(props, "uuid", None) and str(props.uuid))
    try:
        windows, t0, t1 = time_case(torch, main, args.steps, args.warmup,
                                    use_graph=not args.no_graph, barrier=barrier,
                                    repeats=args.repeats, min_region_s=args.min_region_s,
                                    agree=lambda n: int(max_over_ranks(float(n), "cuda")))
    finally:
        sampler.stop()
    # headline: the median K-launch window, the slowest rank's median under torchrun
    ms = max_over_ranks(statistics.median(windows), "cuda")
    clocks = sampler.summary(t0, t1)
    ms_step = ms / args.steps
    value = job_rows_per_s(main.rows, args.steps, world, ms)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": main.describe, "rows": main.rows, "cols": 3072,
                   "l2": f"{main.n_sets} rotating buffer sets, "
                         f"{main.n_sets * main.alg_bytes / 2**20:.0f} MiB > 2x L2 "
                         f"({l2 / 2**20:.0f} MiB): inputs are cold in L2 at every launch",
                   "timing": "CUDA events recorded as nodes of the CUDA graphs that hold the K "
                             "launches (before the first, after the last), so a window is the "
                             "device time of exactly its K launches; the median window of "
                             "several, each bracketed by a barrier and device synchronisation"
                             if not args.no_graph else "CUDA events around K direct launches",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline_entry(main, ms_step, peak, peak_src),
        "gpu_launches": args.steps,
        "repeats": {"windows": len(windows), "launches_per_window": args.steps,
                    "ms_per_step_min": round(min(windows) / args.steps, 6),
                    "ms_per_step_median": round(statistics.median(windows) / args.steps, 6),
                    "ms_per_step_max": round(max(windows) / args.steps, 6),
                    "note": "value and ms_per_step are the median window (max over ranks)"},
        "clocks": clocks,
    }
    if rank == 0 and not args.skip_e2e:
        line["e2e"] = e2e_measure(torch, lib, main, max(3, min(args.steps, 200)))
    kernels = None
    if rank == 0 and not args.skip_kernels:
        # every other kernel of the path, the same way (200-launch windows, median of 5); the
        # workloads are described on stderr, the line keeps a compact table at its end
        kernels = {}
        for key, build_case in extra_cases(torch, lib, l2).items():
            case = build_case()
            kw, _, _ = time_case(torch, case, 200, 5, use_graph=not args.no_graph, repeats=5)
            per = statistics.median(kw) / 200
            rl = roofline_entry(case, per, peak, peak_src)
            kernels[key] = {"us": round(per * 1e3, 3), "frac": rl["frac"],
                            "gbs": rl["achieved"], "traffic": rl["traffic"]}
            log(f"kernel {key}: {case.name}: {case.describe}: {per * 1e3:.3f} us, "
                f"{rl['achieved']} GB/s, {rl['frac']} of {peak} GB/s ({peak_src})")
            del case
            torch.cuda.empty_cache()
    if rank == 0 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(args.cpu_seconds)
    if kernels is not None:
        # last key of the line, so that a reader of only the end of the output still sees it
        line["kernels"] = {"unit": "us per launch / fraction of measured HBM", **kernels}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ------------------------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    import workloads as W

    c = W.CONFIGS["nss_qwen"]
    full = W.config_inputs("nss_qwen")
    x, sc, sh = full["x"], full["scale"], full["shift"]
    # calibrate: rows per step so that the K timed steps take about a minute
    t0 = time.perf_counter()
    oracle.nss_fp8(x[:32], sc, sh, c["input_scale"])
    rate = 32 / max(time.perf_counter() - t0, 1e-6)
    rows_per_step = int(max(1, min(x.shape[0], rate * 60.0 / max(args.steps, 1))))
    for i in range(args.warmup):
        oracle.nss_fp8(x[:rows_per_step], sc, sh, c["input_scale"])
    t0 = time.perf_counter()
    for i in range(args.steps):
        r0 = (i * rows_per_step) % max(1, x.shape[0] - rows_per_step + 1)
        oracle.nss_fp8(x[r0:r0 + rows_per_step], sc, sh, c["input_scale"])
    el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"nss_fp8 Qwen-Image x bf16 [4608,3072], input_scale "
                               f"{c['input_scale']}; each step a {rows_per_step}-row sample",
                   "rows_per_step": rows_per_step},
        "cpu_baseline": {"value": round(value, 2), "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "host": host_cpu(),
                         "sample": f"{rows_per_step} rows per step x {args.steps} steps"},
        "e2e": {"value": round(value, 2), "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_only(args):
    """Launch one workload W + K times with no timing and no JSON (for ncu captures)."""
    import torch
    import fp8_quant_row_gb300 as fq
    torch.cuda.set_device(0)
    fq.build()
    lib = fq._capi.lib()
    l2 = int(getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 126 * 2 ** 20))
    if args.profile_only == "nss_qwen":
        case = make_cases(torch, fq, lib, l2)["nss_qwen"]
    else:
        case = extra_cases(torch, lib, l2, only=args.profile_only)[args.profile_only]()
    for i in range(args.warmup + args.steps):
        case.launch(i)
    torch.cuda.synchronize()
    log(f"profile-only {args.profile_only}: {args.warmup + args.steps} launches of {case.name}")


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-graph", action="store_true", help="launch directly instead of graphs")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-kernels", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--repeats", type=int, default=10,
                    help="timed windows of K launches (the headline is their median)")
    ap.add_argument("--min-region-s", type=float, default=0.3,
                    help="add windows until the timed region lasts this long (clock samples)")
    ap.add_argument("--profile-only", choices=("nss_qwen", "nss_tiny", "scale_residual_qwen",
                                               "token_cat_nvfp4_flux", "qkv_qwen", "qkv_flux",
                                               "bias_mul_add_qwen", "nss_flux", "token_cat_flux"),
                    help="only launch this workload (W+K launches, no timing): for ncu captures")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile_only:
        ap.error("--warmup must be >= 3")
    if args.profile_only:
        run_profile_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
