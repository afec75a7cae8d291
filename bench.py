#!/usr/bin/env python
"""Benchmark of the decode hot path on GB300: prints ONE JSON line.

Workload (one GPU): the q8_0 decode mat-vec of a 14336 x 4096 weight (32-element
int8 blocks with fp16 scales, quantized from N(0, 0.02) bf16) at batch 1, with the
activation x (length 4096, N(0,1)) quantized to q8_0 in front of it, and the
256-element superblock quantizer on x (length 4096) and on y (length 14336).

  token  = quantize_gemv_q8_0(W_{t mod 16}, x_t): one launch that quantizes x_t to q8_0
           (writing q and d out) and runs the mat-vec, PDL-linked to the previous
           token on the main stream; quantize_q8(x_t, 256) and quantize_q8(y_t, 256) on
           a side stream that forks after it (they overlap the next token's chain).
           The same step with the quantizer as its own launch (quantize_q8 ->
           gemv_q8_0) is timed too and reported as "two_launch_step".
  step   = a batch of 2048 tokens (distinct synthetic activations), captured once in
           a CUDA graph and replayed.  16 distinct weight copies (1.0 GB) rotate, so
           every GEMV streams weights that are not in the 129 MB L2.
  value  = algorithmic bytes of the step / step time (GB/s), summed over ranks.

The same line also reports: the fused quantize + GEMV kernel against the HBM roofline
(CUDA events over back-to-back launches on distinct weight copies), the GEMV alone, the
other hot-path calls on their configured shapes ("rows": prefill GEMM, KV dequant, decode
and prefill attention over the binary16 KV, each grouped MoE call and its quantizer), each as plain back-to-back launches,
PDL-linked, and where one copy fits in L2 also L2-hot (one copy repeated, labelled
"l2hot"), the end-to-end rate through the C ABI with host buffers, the CPU oracle on a
bounded sample (all host cores, rows cut over threads, and one core), the 27B-shaped
bf16 decode chain (64 layers x [QKV, O, gate/up, down] + lm_head, 257 PDL-linked
mat-vecs, 43.16 GB per token), the batch-1 bf16 4096 x 4096 GEMV, the MoE step
(quantize -> grouped gate_up -> quantize -> grouped down at T = 1, 16, 512), and last a
compact "key_numbers" summary.

--impl reference times the CPU oracle (the plain C restatement) on the same workload,
one token per step, its GEMV rows cut over the host cores.
--profile-case CASE runs one call a few times for a profiler (see profile_case).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
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

M, K = 14336, 4096
NCOPY = 16
TOKENS = 2048
NOMINAL_HBM_GBS = 8000.0
METRIC = "decode GEMV HBM GB/s and % of GB300 peak; Q8 quantizer us/call at batch 1"

# algorithmic bytes per token (read + write, each byte once)
B_Q32 = K * 4 + K + (K // 32) * 2                       # x in, q out, fp16 scales out
B_GEMV = M * K + M * (K // 32) * 2 + K + (K // 32) * 2 + M * 4
B_Q256_Y = M * 4 + M + (M // 256) * 4
B_Q256_X = K * 4 + K + (K // 256) * 4
B_TOKEN_2L = B_Q32 + B_GEMV + B_Q256_Y + B_Q256_X          # quantizer as its own launch
B_FUSED = B_GEMV - K - (K // 32) * 2 + K * 4 + K + (K // 32) * 2  # x in, q and d out, no re-read
B_TOKEN = B_FUSED + B_Q256_Y + B_Q256_X

WORKLOAD = "q8_0 decode GEMV 14336x4096 batch 1 + fused q8_0 quantizer n=4096 + superblock quantizer n=4096/14336"
CHAIN_LAYER = [(6144, 5120), (5120, 5120), (34816, 5120), (5120, 17408)]
CHAIN_HEAD = (152064, 5120)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def whole_job_rate(pg, torch, elapsed_s, units_per_rank, device="cpu"):
    """Whole-job rate over the ranks of process group pg (None: one process): the
    slowest rank's elapsed time (max over ranks) and the units of all ranks, so
    value = units_per_rank * world / max_elapsed.  Returns (value, max_elapsed)."""
    world = 1
    if pg is not None:
        world = pg.get_world_size()
        t = torch.tensor([elapsed_s], device=device, dtype=torch.float64)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        elapsed_s = float(t.item())
    return units_per_rank * world / elapsed_s, elapsed_s


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi samples (100 ms) taken while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.t0, self.t1 = t0, t1

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = [s for (t, s) in self.samples if self.t0 is not None and self.t0 - 0.05 <= t <= self.t1 + 0.05]
        parsed = []
        for r in rows:
            f = [v.strip() for v in r.split(",")]
            if len(f) < 7:
                continue
            try:
                parsed.append((float(f[0]), float(f[1]), f[3:7]))
            except ValueError:
                continue
        if not parsed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for (_, _, fl) in parsed for i, v in enumerate(fl) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(p[0] for p in parsed), "sm_max_mhz": max(p[1] for p in parsed),
                "reasons": reasons, "samples": len(parsed)}


# -------------------------------------------------------------- our arm ----
class Workload:
    def __init__(self, wsw, torch, dev):
        import weight_streaming_warp_gb300.synthetic as syn
        self.wsw, self.torch = wsw, torch
        g = torch.Generator(device=dev)
        g.manual_seed(0)
        self.Wq, self.Wd = [], []
        for c in range(NCOPY):
            Wf = torch.randn((M, K), generator=g, device=dev).mul_(0.02).to(torch.bfloat16).float()
            q, d = wsw.quantize_q8(Wf, 32)  # weights quantized once, by the library
            self.Wq.append(q)
            self.Wd.append(d)
            del Wf
        self.X = syn.normal(0, "bench_x", (TOKENS, K), device=dev)
        self.xq = torch.empty((TOKENS, K), dtype=torch.int8, device=dev)
        self.xd = torch.empty((TOKENS, K // 32), dtype=torch.float16, device=dev)
        self.Y = torch.empty((TOKENS, M), dtype=torch.float32, device=dev)
        self.yq = torch.empty((TOKENS, M), dtype=torch.int8, device=dev)
        self.ys = torch.empty((TOKENS, M // 256), dtype=torch.float32, device=dev)
        self.xq2 = torch.empty((TOKENS, K), dtype=torch.int8, device=dev)
        self.xs2 = torch.empty((TOKENS, K // 256), dtype=torch.float32, device=dev)
        self._bind()

    def _bind(self):
        """Raw C-ABI entry points and pre-computed pointers (per-token launches)."""
        L = self.wsw.load()
        self.L = L
        opts = self.wsw._COpts(0, 0, 1, 0)
        self.opts = opts
        self.popts = ctypes.byref(opts)
        self.ptr = dict(X=self.X.data_ptr(), xq=self.xq.data_ptr(), xd=self.xd.data_ptr(), Y=self.Y.data_ptr(),
                        yq=self.yq.data_ptr(), ys=self.ys.data_ptr(), xq2=self.xq2.data_ptr(),
                        xs2=self.xs2.data_ptr())
        self.wq = [w.data_ptr() for w in self.Wq]
        self.wd = [w.data_ptr() for w in self.Wd]

    def token(self, t, stream, side, rc, fused=True):
        L, p, o = self.L, self.ptr, self.popts
        x = p["X"] + t * K * 4
        xq, xd = p["xq"] + t * K, p["xd"] + t * (K // 32) * 2
        y = p["Y"] + t * M * 4
        if fused:
            rc |= L.wsw_quantize_gemv_q8_0(self.wq[t % NCOPY], self.wd[t % NCOPY], M, K, K, x, xq, xd, y,
                                           stream, o)
        else:
            rc |= L.wsw_quantize_q8(x, 1, K, K, 32, xq, xd, stream, o)
            rc |= L.wsw_gemv_q8_0(self.wq[t % NCOPY], self.wd[t % NCOPY], M, K, K, xq, xd, y, stream, o)
        if side is None:
            rc |= L.wsw_quantize_q8(y, 1, M, M, 256, p["yq"] + t * M, p["ys"] + t * (M // 256) * 4, stream, o)
            rc |= L.wsw_quantize_q8(x, 1, K, K, 256, p["xq2"] + t * K, p["xs2"] + t * (K // 256) * 4, stream, o)
        else:
            ev, s2 = side
            ev[t].record(self.torch.cuda.ExternalStream(stream.value))
            s2.wait_event(ev[t])
            sp = ctypes.c_void_p(s2.cuda_stream)
            rc |= L.wsw_quantize_q8(y, 1, M, M, 256, p["yq"] + t * M, p["ys"] + t * (M // 256) * 4, sp, o)
            rc |= L.wsw_quantize_q8(x, 1, K, K, 256, p["xq2"] + t * K, p["xs2"] + t * (K // 256) * 4, sp, o)
        return rc

    def step(self, stream, overlap=True, fused=True):
        """One batch of TOKENS decode tokens on `stream`; with overlap the
        superblock quantizations go to a side stream joined at the end."""
        torch = self.torch
        rc = 0
        side = None
        main = None
        if overlap:
            main = torch.cuda.ExternalStream(stream.value)
            if not hasattr(self, "_side"):
                self._side = torch.cuda.Stream()
                self._ev = [torch.cuda.Event() for _ in range(TOKENS)]
            side = (self._ev, self._side)
            self._side.wait_stream(main)
        for t in range(TOKENS):
            rc = self.token(t, stream, side, rc, fused)
        if side is not None:
            main.wait_stream(self._side)
        if rc:
            raise RuntimeError("a launch failed: %s" % self.wsw.status_string(rc))


def _graph(torch, fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(ctypes.c_void_p(s.cuda_stream))  # first use (per-device set-up) outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return g


def _time_graph(torch, g, reps):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1000.0 / reps


KERNEL_SOURCES = {"gemv_q8_0": ("gemv_q8_0.cu", "stream_gemv.cuh", "q8_dot.cuh", "q8_math.cuh", "common.cuh"),
                  "quantize_gemv_q8_0": ("gemv_q8_0.cu", "stream_gemv.cuh", "q8_dot.cuh", "q8_math.cuh",
                                         "common.cuh")}


def kernel_source_sha(name):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[name]:
        with open(os.path.join(ROOT, "weight_streaming_warp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic_record(name):
    """DRAM bytes per launch from the committed ncu summary (profiles/traffic.json),
    or None when the kernel's sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            r = json.load(f).get(name)
        if r and r.get("source_sha256") == kernel_source_sha(name):
            return r["bytes_per_launch"]
    except Exception:
        pass
    return None


def measure_gemv_kernel(torch, wl, fused=True):
    """The fused quantize + GEMV (or gemv_q8_0 alone): 256 back-to-back PDL launches
    over the 16 weight copies."""
    n = 256

    def fn(stream):
        rc = 0
        for i in range(n):
            t = i % 64
            if fused:
                rc |= wl.L.wsw_quantize_gemv_q8_0(wl.wq[i % NCOPY], wl.wd[i % NCOPY], M, K, K,
                                                  wl.ptr["X"] + t * K * 4, wl.ptr["xq"] + t * K,
                                                  wl.ptr["xd"] + t * (K // 32) * 2, wl.ptr["Y"] + t * M * 4,
                                                  stream, wl.popts)
            else:
                rc |= wl.L.wsw_gemv_q8_0(wl.wq[i % NCOPY], wl.wd[i % NCOPY], M, K, K, wl.ptr["xq"],
                                         wl.ptr["xd"], wl.ptr["Y"] + t * M * 4, stream, wl.popts)
        assert rc == 0

    g = _graph(torch, fn)
    _time_graph(torch, g, 3)
    times = [_time_graph(torch, g, 1) / n for _ in range(10)]
    return statistics.median(times), min(times), max(times)


def measure_quantizer(torch, wl):
    """Batch-1 quantizer calls back to back in a graph: us per call."""
    n = 1000
    out = {}
    for (name, length, block, src) in (("q8_0_n4096", K, 32, "X"), ("superblock_n4096", K, 256, "X"),
                                       ("superblock_n14336", M, 256, "Y")):
        qs = wl.xq if length == K else wl.yq
        sc = wl.xd if block == 32 else (wl.xs2 if length == K else wl.ys)

        def fn(stream, length=length, block=block, src=src, qs=qs, sc=sc):
            rc = 0
            for i in range(n):
                t = i % TOKENS
                rc |= wl.L.wsw_quantize_q8(wl.ptr[src] + t * length * 4, 1, length, length, block,
                                           qs.data_ptr() + t * length,
                                           sc.data_ptr() + t * (length // block) * sc.element_size(),
                                           stream, wl.popts)
            assert rc == 0

        g = _graph(torch, fn)
        _time_graph(torch, g, 2)
        out[name] = round(statistics.median(_time_graph(torch, g, 1) for _ in range(5)) / n * 1e6, 3)
    return out


def measure_chain(torch, wsw, dev):
    """27B-shaped dense decode chain, bf16 weights N(0, 0.02), one token per replay."""
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    shapes = [s for _ in range(64) for s in CHAIN_LAYER] + [CHAIN_HEAD]
    Ws, ys = [], []
    for (Mi, Ki) in shapes:
        Ws.append(torch.randn((Mi, Ki), generator=g, device=dev, dtype=torch.float32).mul_(0.02).to(torch.bfloat16))
        ys.append(torch.empty(Mi, dtype=torch.float32, device=dev))
    x0 = torch.randn(CHAIN_LAYER[0][1], generator=g, device=dev)
    links = []
    for i, (Mi, Ki) in enumerate(shapes):
        x = x0 if i == 0 else ys[i - 1][:Ki]
        links.append((Ws[i], Ki, x, 1.0 / (0.02 * math.sqrt(Ki)), ys[i]))
    nbytes = sum(Mi * Ki * 2 + Ki * 4 + Mi * 4 for (Mi, Ki) in shapes)
    res = {}
    graphs = {}
    # the library's chain (PDL), plain stream order, and PDL plus an L2 prefetch of each
    # next link's first loads by the finishing warps (off by default: it measured slower)
    arms = {"pdl": {"pdl": 1}, "no_pdl": {"pdl": 0}, "pdl_l2_prefetch_4": {"pdl": 1, "l2_prefetch_steps": 4}}
    for name, o in arms.items():
        graphs[name] = _graph(torch, lambda stream, o=o: wsw.gemv_bf16_chain(links, opts=o))
        _time_graph(torch, graphs[name], 2)
    t = {name: [] for name in arms}
    for rep in range(6):  # paired, alternating order
        for name in (list(arms) if rep % 2 == 0 else list(arms)[::-1]):
            t[name].append(_time_graph(torch, graphs[name], 1))
    for name in arms:
        med = statistics.median(t[name])
        res[name] = {"ms_per_token": round(med * 1e3, 4), "GBps": round(nbytes / med / 1e9, 1),
                     "tok_per_s": round(1.0 / med, 2),
                     "min_ms": round(min(t[name]) * 1e3, 4), "max_ms": round(max(t[name]) * 1e3, 4)}
    ok = all(bool(torch.isfinite(y).all()) for y in ys[-2:])
    del graphs, Ws, ys, links
    torch.cuda.empty_cache()
    res["bytes_per_token"] = nbytes
    res["launches_per_token"] = len(shapes)
    res["finite"] = ok
    return res


def _graph_rate(torch, fn, n, reps=5):
    """Median seconds per call of fn(stream) captured n times in one graph."""
    def body(stream):
        for _ in range(n):
            fn(stream)
    g = _graph(torch, body)
    _time_graph(torch, g, 2)
    return statistics.median(_time_graph(torch, g, 1) for _ in range(reps)) / n


def _rates(torch, make, n, hot=True):
    """Seconds per call of back-to-back calls in a graph: plain and PDL-linked, both
    rotating over copies larger than L2, and (hot) PDL-linked on one copy, L2-hot."""
    t = _graph_rate(torch, make(0, False), n)
    tp = _graph_rate(torch, make(1, False), n)
    th = _graph_rate(torch, make(1, True), n) if hot else None
    return t, tp, th


def _decode_attn_key(rows, peak):
    """us per call and fraction of the HBM peak of the decode attention rows (per-head
    layout, PDL-linked), for the key numbers; rows that are absent are left out."""
    out = {}
    for d in (32768, 65536):
        for gq in (1, 8):
            r = rows.get("attn_decode_d%d_g%d_per_head" % (d, gq))
            if r:
                out["d%d_g%d" % (d, gq)] = {"us": r["us_pdl"], "frac": round(r["GBps_pdl"] / peak, 4)}
    return out


def _entry(nbytes, t, tp, th=None, flops=None, **extra):
    """One bench row: us and GB/s (algorithmic bytes) per regime."""
    e = {"us": round(t * 1e6, 2), "GBps": round(nbytes / t / 1e9, 1),
         "us_pdl": round(tp * 1e6, 2), "GBps_pdl": round(nbytes / tp / 1e9, 1)}
    if flops:
        e["TFLOPs"] = round(flops / t / 1e12, 2)
        e["TFLOPs_pdl"] = round(flops / tp / 1e12, 2)
    if th is not None:
        e["us_l2hot"] = round(th * 1e6, 2)
        e["GBps_l2hot"] = round(nbytes / th / 1e9, 1)
        if flops:
            e["TFLOPs_l2hot"] = round(flops / th / 1e12, 2)
    e["bytes"] = nbytes
    e.update(extra)
    return e


def measure_config1(torch, wsw, dev):
    """The batch-1 bf16 decode GEMV, W 4096 x 4096 (33.6 MB): 32 rotating copies
    (1.07 GB) plain and PDL-linked, and one copy repeated (L2-hot)."""
    Mc, Kc, ncp = 4096, 4096, 32
    g = torch.Generator(device=dev)
    g.manual_seed(3)
    Ws = [torch.randn((Mc, Kc), generator=g, device=dev).mul_(0.02).to(torch.bfloat16) for _ in range(ncp)]
    X = torch.randn((64, Kc), generator=g, device=dev)
    Y = torch.empty((64, Mc), dtype=torch.float32, device=dev)
    it = [0]

    def make(pdl, hot):
        def fn(stream):
            i = it[0]
            it[0] += 1
            wsw.gemv_bf16(Ws[0 if hot else i % ncp], X[i % 64], out=Y[i % 64], opts={"pdl": pdl})
        return fn
    t, tp, th = _rates(torch, make, 256)
    nb = Mc * Kc * 2 + Kc * 4 + Mc * 4
    del Ws
    torch.cuda.empty_cache()
    return _entry(nb, t, tp, th, note="bf16 4096x4096; rotating copies 1.07 GB; l2hot = one copy repeated")


def measure_gemm(torch, wsw, dev, out):
    """Small-batch prefill GEMM, W 2560 x 10240 (packed and one-line padded rows)."""
    g = torch.Generator(device=dev)
    g.manual_seed(2)
    Mg, Kg = 2560, 10240
    Ws = [torch.randn((Mg, Kg), generator=g, device=dev).mul_(0.02).to(torch.bfloat16) for _ in range(12)]
    for ld in (Kg, Kg + 64):
        Wl = Ws if ld == Kg else [wsw.upload_padded(w, ld) for w in Ws]
        for N in (8, 128, 512):
            X = torch.randn((N, Kg), generator=g, device=dev).to(torch.bfloat16)
            Y = torch.empty((N, Mg), dtype=torch.float32, device=dev)
            it = [0]

            def make(pdl, hot, X=X, Y=Y, Wl=Wl):
                def fn(stream):
                    wsw.gemm_bf16(Wl[0 if hot else it[0] % len(Wl)], X, out=Y, opts={"pdl": pdl})
                    it[0] += 1
                return fn
            t, tp, th = _rates(torch, make, 24, hot=(ld == Kg))
            key = "gemm_bf16_N%d_%s" % (N, "packed" if ld == Kg else "padded")
            out[key] = _entry(Mg * Kg * 2 + N * Kg * 2 + N * Mg * 4, t, tp, th, flops=2.0 * N * Mg * Kg)
        del Wl
    del Ws
    torch.cuda.empty_cache()


def measure_dequant(torch, wsw, dev, out):
    """q8_0 KV cache dequant, 4 heads x 128, 8 rotating copies."""
    g = torch.Generator(device=dev)
    g.manual_seed(4)
    for depth in (32768, 65536):
        copies = 8
        qs = [torch.randint(-127, 128, (depth, 4, 128), dtype=torch.int8, device=dev, generator=g)
              for _ in range(copies)]
        ds = [torch.rand((depth, 4, 4), device=dev, generator=g).half() for _ in range(copies)]
        o = torch.empty((4, depth, 128), dtype=torch.float16, device=dev)
        it = [0]

        def make(pdl, hot, qs=qs, ds=ds, o=o):
            def fn(stream):
                i = 0 if hot else it[0] % copies
                wsw.dequant_q8_0_kv(qs[i], ds[i], out=o, opts={"pdl": pdl})
                it[0] += 1
            return fn
        t, tp, th = _rates(torch, make, 32)
        nb = depth * 4 * 128 * (1 + 2) + depth * 4 * 4 * 2
        out["dequant_kv_d%d" % depth] = _entry(nb, t, tp, th)
        del qs, ds
    torch.cuda.empty_cache()


def measure_attn_decode(torch, wsw, dev, out):
    """Decode attention over the binary16 KV (4 KV heads x 128; groups of 1 and 8
    query heads), reading the per-head scratch and the position-major cache; 4 copies
    of K and V rotate (268 MB and more)."""
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    for depth in (32768, 65536):
        copies = 4
        Ks = [torch.randn((4, depth, 128), generator=g, device=dev).half() for _ in range(copies)]
        Vs = [torch.randn((4, depth, 128), generator=g, device=dev).half() for _ in range(copies)]
        Kc = [t.permute(1, 0, 2).contiguous() for t in Ks]
        Vc = [t.permute(1, 0, 2).contiguous() for t in Vs]
        for group in (1, 8):
            qq = torch.randn((4, group, 128), generator=g, device=dev)
            o = torch.empty((4, group, 128), dtype=torch.float32, device=dev)
            ws = torch.zeros(wsw.attn_decode_workspace_bytes(depth, 4, group), dtype=torch.uint8, device=dev)
            for layout in ("per_head", "position_major"):
                it = [0]

                def make(pdl, hot, qq=qq, o=o, ws=ws, layout=layout, it=it):
                    def fn(stream):
                        i = 0 if hot else it[0] % copies
                        it[0] += 1
                        if layout == "per_head":
                            k, v = Ks[i], Vs[i]
                        else:
                            k, v = Kc[i].permute(1, 0, 2), Vc[i].permute(1, 0, 2)
                        wsw.attn_decode_f16(qq, k, v, out=o, ws=ws, opts={"pdl": pdl})
                    return fn
                t, tp, th = _rates(torch, make, 32, hot=(layout == "per_head"))
                nb = 2 * depth * 4 * 128 * 2 + 2 * 4 * group * 128 * 4
                out["attn_decode_d%d_g%d_%s" % (depth, group, layout)] = _entry(nb, t, tp, th)
        del Ks, Vs, Kc, Vc
    torch.cuda.empty_cache()


def attn_prefill_flops(depth, heads, group, nq, hd=128):
    """Tensor-core flops of the causal prefill pass: query i sees depth - nq + i + 1
    positions; per position 2 hd for q.K and 2 hd for P V."""
    visible = nq * (depth - nq) + nq * (nq + 1) // 2
    return 4 * hd * visible * heads * group


def measure_attn_prefill(torch, wsw, dev, out, peak_tf):
    """Causal prefill attention, 512 queries at the end of a binary16 cache of depth
    32768 / 65536, 4 KV heads x 128, 8 query heads per KV head; 4 copies of K and V
    rotate.  Also the page's pass as a whole: dequantize the q8_0 K and V once into the
    per-head scratch, then the prefill attention over it (three PDL-linked launches)."""
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    heads, group, nq = 4, 8, 512
    for depth in (32768, 65536):
        copies = 4
        Ks = [torch.randn((heads, depth, 128), generator=g, device=dev).half() for _ in range(copies)]
        Vs = [torch.randn((heads, depth, 128), generator=g, device=dev).half() for _ in range(copies)]
        Kc = [t.permute(1, 0, 2).contiguous() for t in Ks]
        Vc = [t.permute(1, 0, 2).contiguous() for t in Vs]
        q = torch.randn((heads, group, nq, 128), generator=g, device=dev).half()
        o = torch.empty((heads, group, nq, 128), dtype=torch.float32, device=dev)
        fl = attn_prefill_flops(depth, heads, group, nq)
        nb = 2 * depth * heads * 128 * 2 + q.numel() * 2 + o.numel() * 4
        for layout in ("per_head", "position_major"):
            it = [0]

            def make(pdl, hot, layout=layout, it=it):
                def fn(stream):
                    i = 0 if hot else it[0] % copies
                    it[0] += 1
                    if layout == "per_head":
                        k, v = Ks[i], Vs[i]
                    else:
                        k, v = Kc[i].permute(1, 0, 2), Vc[i].permute(1, 0, 2)
                    wsw.attn_prefill_f16(q, k, v, out=o, opts={"pdl": pdl})
                return fn
            t, tp, th = _rates(torch, make, 8, hot=(layout == "per_head"))
            e = _entry(nb, t, tp, th, flops=fl)
            e["frac_of_bf16_peak_pdl"] = round(fl / tp / 1e12 / peak_tf, 4)
            out["attn_prefill_d%d_%s" % (depth, layout)] = e
        del Kc, Vc
        # dequant once (K and V, q8_0 -> per-head binary16 scratch) + prefill attention
        kq = [torch.randint(-127, 128, (depth, heads, 128), dtype=torch.int8, device=dev, generator=g)
              for _ in range(2)]
        kd = [torch.rand((depth, heads, 4), device=dev, generator=g).half() for _ in range(2)]
        sk = torch.empty((heads, depth, 128), dtype=torch.float16, device=dev)
        sv = torch.empty((heads, depth, 128), dtype=torch.float16, device=dev)

        def make_pass(pdl, hot):
            def fn(stream):
                wsw.dequant_q8_0_kv(kq[0], kd[0], out=sk, opts={"pdl": pdl})
                wsw.dequant_q8_0_kv(kq[1], kd[1], out=sv, opts={"pdl": pdl})
                wsw.attn_prefill_f16(q, sk, sv, out=o, opts={"pdl": pdl})
            return fn
        t, tp, _ = _rates(torch, make_pass, 8, hot=False)
        out["dequant_then_prefill_d%d" % depth] = {"us": round(t * 1e6, 2), "us_pdl": round(tp * 1e6, 2),
                                                   "TFLOPs_pdl": round(fl / tp / 1e12, 1),
                                                   "scratch_bytes": 2 * sk.numel() * 2,
                                                   "calls": "dequant K, dequant V, attn_prefill"}
        # the same pass with a bounded scratch: one window of K and V at a time
        window = 4096 if depth == 32768 else 8192
        ws = torch.empty(wsw.attn_prefill_q8_0_workspace_bytes(depth, heads, group, nq, window), dtype=torch.uint8,
                         device=dev)

        def make_win(pdl, hot):
            def fn(stream):
                wsw.attn_prefill_q8_0(q, kq[0], kd[0], kq[1], kd[1], window, out=o, ws=ws, opts={"pdl": pdl})
            return fn
        t, tp, _ = _rates(torch, make_win, 4, hot=False)
        out["windowed_q8_0_prefill_d%d_w%d" % (depth, window)] = {
            "us": round(t * 1e6, 2), "us_pdl": round(tp * 1e6, 2), "TFLOPs_pdl": round(fl / tp / 1e12, 1),
            "frac_of_bf16_peak_pdl": round(fl / tp / 1e12 / peak_tf, 4), "workspace_bytes": ws.numel(),
            "calls": "per window: dequant K, dequant V, attention with the carried softmax state"}
        del Ks, Vs, kq, kd, sk, sv, ws
    torch.cuda.empty_cache()


MOE_E, MOE_H, MOE_F, MOE_TOPK = 128, 2048, 768, 8


def _moe_bytes(used, Mo, Kx, R):
    """Algorithmic bytes of one grouped call: the used experts' q8_0 rows once, the
    q8_0 activations, y."""
    return int(used * (Mo * Kx + Mo * Kx // 16) + R * (Kx + Kx // 16) + R * Mo * 4)


def _quant_bytes(R, n):
    return R * n * 4 + R * n + R * (n // 32) * 2


def measure_moe(torch, wsw, dev, out):
    """The MoE step of 128 experts, top-8, hidden 2048, expert FFN 768: per T the
    activations (R = 8 T rows, N(0,1)) are quantized per row (q8_0), the grouped
    gate_up mat-vec (1536 x 2048 per expert) runs, the down input (R x 768, N(0,1),
    standing in for the SwiGLU output) is quantized and the grouped down mat-vec
    (2048 x 768 per expert) runs.  Calls rotate over 8 routings and 2 copies of the
    expert weights (2 x 428 MB gate_up, 2 x 214 MB down), so the experts a call reads
    are not left in L2 by the call before.  Reports the whole step, each grouped call,
    and (T = 1 and 16, whose experts fit in L2) the same calls repeated on one routing
    and one copy (L2-hot)."""
    import weight_streaming_warp_gb300.synthetic as syn
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    E, H, F = MOE_E, MOE_H, MOE_F
    nw, nr = 2, 8

    def qweights(Mo, Kx):
        return [(torch.randint(-127, 128, (E, Mo, Kx), dtype=torch.int8, device=dev, generator=g),
                 (torch.rand((E, Mo, Kx // 32), device=dev, generator=g) * 1e-3).half()) for _ in range(nw)]
    Wg, Wdn = qweights(2 * F, H), qweights(H, F)
    steps = {}
    for T in (1, 16, 512):
        R = T * MOE_TOPK
        idss = [syn.routing(r, "bench_route%d" % T, T, E, MOE_TOPK).to(dev) for r in range(nr)]
        xs = [torch.randn((R, H), generator=g, device=dev) for _ in range(2)]
        hs = [torch.randn((R, F), generator=g, device=dev) for _ in range(2)]
        xq = torch.empty((R, H), dtype=torch.int8, device=dev)
        xd = torch.empty((R, H // 32), dtype=torch.float16, device=dev)
        hq = torch.empty((R, F), dtype=torch.int8, device=dev)
        hd = torch.empty((R, F // 32), dtype=torch.float16, device=dev)
        yg = torch.empty((R, 2 * F), dtype=torch.float32, device=dev)
        yd = torch.empty((R, H), dtype=torch.float32, device=dev)
        nws = max(wsw.moe_workspace_bytes(E, H, R), wsw.moe_workspace_bytes(E, F, R))
        ws = torch.empty(nws, dtype=torch.uint8, device=dev) if nws else False
        used = statistics.mean(len(set(ids.tolist())) for ids in idss)
        it = [0]

        def part(which, pdl, hot):
            def fn(stream):
                i = 0 if hot else it[0]
                it[0] += 1
                o = {"pdl": pdl}
                ids = idss[i % nr]
                if which in ("step", "quant_gate_up"):
                    wsw.quantize_q8(xs[i % 2], 32, out=(xq, xd), opts=o)
                if which in ("step", "gate_up"):
                    Wq, Wd = Wg[i % nw]
                    wsw.moe_gemv_q8_0(Wq, Wd, xq, xd, ids, out=yg, opts=o, ws=ws)
                if which in ("step", "quant_down"):
                    wsw.quantize_q8(hs[i % 2], 32, out=(hq, hd), opts=o)
                if which in ("step", "down"):
                    Wq, Wd = Wdn[i % nw]
                    wsw.moe_gemv_q8_0(Wq, Wd, hq, hd, ids, out=yd, opts=o, ws=ws)
            return fn
        n = 8 if T == 512 else 32
        hot = T <= 16
        b_qg, b_qd = _quant_bytes(R, H), _quant_bytes(R, F)
        b_g, b_d = _moe_bytes(used, 2 * F, H, R), _moe_bytes(used, H, F, R)
        t, tp, th = _rates(torch, lambda pdl, h: part("step", pdl, h), n, hot=hot)
        steps[T] = _entry(b_qg + b_g + b_qd + b_d, t, tp, th, experts_used=used,
                          calls="quantize_q8 gate_up input -> moe gate_up -> quantize_q8 down input -> moe down")
        parts = {}
        for name, nb in (("quant_gate_up", b_qg), ("gate_up", b_g), ("quant_down", b_qd), ("down", b_d)):
            tt, ttp, tth = _rates(torch, lambda pdl, h, name=name: part(name, pdl, h), n, hot=hot)
            parts[name] = _entry(nb, tt, ttp, tth)
        out["moe_gate_up_T%d" % T] = dict(parts["gate_up"], experts_used=used)
        out["moe_down_T%d" % T] = dict(parts["down"], experts_used=used)
        out["moe_quantize_T%d" % T] = {"gate_up_input_us_pdl": parts["quant_gate_up"]["us_pdl"],
                                       "down_input_us_pdl": parts["quant_down"]["us_pdl"],
                                       "gate_up_input_GBps_pdl": parts["quant_gate_up"]["GBps_pdl"],
                                       "down_input_GBps_pdl": parts["quant_down"]["GBps_pdl"]}
        del xs, hs, ws
    del Wg, Wdn
    torch.cuda.empty_cache()
    return steps


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1900.0


def measure_rows(torch, wsw, dev):
    """The other hot-path calls on their configured shapes (graph-amortised, inputs
    rotating over copies larger than L2 where a single copy would fit).  Each is timed
    as plain back-to-back launches ("us"), PDL-linked ones ("us_pdl") and, where one
    copy fits in the 129 MB L2, PDL-linked on one copy ("us_l2hot")."""
    out = {}
    measure_gemm(torch, wsw, dev, out)
    measure_dequant(torch, wsw, dev, out)
    measure_attn_decode(torch, wsw, dev, out)
    measure_attn_prefill(torch, wsw, dev, out, _bf16_peak())
    moe_steps = measure_moe(torch, wsw, dev, out)
    return out, moe_steps


def measure_e2e(torch, wl, dev, steps, step_graph=None):
    """End to end with host buffers, timed by the host clock: per step, copy the
    batch's activations from pinned host memory, run the step (the CUDA graph of the
    library's calls when step_graph is given, else every call launched eagerly from
    Python), and copy every token's y back to pinned host memory."""
    xh = wl.X.cpu().pin_memory()
    yh = torch.empty((TOKENS, M), dtype=torch.float32).pin_memory()
    s = torch.cuda.current_stream()
    stream = ctypes.c_void_p(s.cuda_stream)
    n = max(1, steps if step_graph is not None else min(steps, 3))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        wl.X.copy_(xh, non_blocking=True)
        if step_graph is not None:
            step_graph.replay()
        else:
            wl.step(stream, overlap=False)
        yh.copy_(wl.Y, non_blocking=True)
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / n
    return {"value": round(B_TOKEN * TOKENS / dt / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": TOKENS * K * 4, "d2h_bytes_per_step": TOKENS * M * 4,
            "ms_per_step": round(dt * 1e3, 3), "steps": n,
            "how": "step's CUDA graph of library calls" if step_graph is not None else "eager calls from Python"}


_CPU_INPUTS = None


def _cpu_inputs():
    """Host inputs of the CPU oracle: one q8_0 weight copy and 8 activations."""
    global _CPU_INPUTS
    if _CPU_INPUTS is None:
        import torch
        import oracle as orc
        import weight_streaming_warp_gb300.synthetic as syn
        W = syn.normal(0, "cpu_W", (M, K), 0.02, torch.bfloat16).float().numpy()
        Wq, Wd = orc.quantize_q8(W, 32)
        X = syn.normal(0, "cpu_x", (8, K)).numpy()
        _CPU_INPUTS = (Wq, Wd, X)
    return _CPU_INPUTS


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_oracle_tokens(n, threads=1):
    """Run n tokens of the workload through the oracle (quantize x, q8_0 GEMV over
    all 14336 rows, the two superblock quantizations); returns elapsed seconds.
    With threads > 1 the GEMV's rows are cut into `threads` contiguous ranges, each
    an oracle call on its own host thread (the C oracle runs without the GIL); the
    oracle's arithmetic per row is unchanged."""
    import numpy as np
    import oracle as orc
    Wq, Wd, X = _cpu_inputs()
    pool = None
    if threads > 1:
        import concurrent.futures as cf
        pool = cf.ThreadPoolExecutor(max_workers=threads)
        cuts = [M * i // threads for i in range(threads + 1)]
    t0 = time.perf_counter()
    for i in range(n):
        x = X[i % 8:i % 8 + 1]
        xq, xd = orc.quantize_q8(x, 32)
        if pool is None:
            y = orc.gemv_q8_0(Wq, Wd, xq[0], xd[0])
        else:
            parts = list(pool.map(lambda j: orc.gemv_q8_0(Wq[cuts[j]:cuts[j + 1]], Wd[cuts[j]:cuts[j + 1]],
                                                          xq[0], xd[0]), range(threads)))
            y = np.concatenate(parts)
        orc.quantize_q8(y.astype(np.float32)[None, :], 256)
        orc.quantize_q8(x, 256)
    el = time.perf_counter() - t0
    if pool is not None:
        pool.shutdown()
    return el


def cpu_oracle_rate(seconds=10.0, threads=1):
    """GB/s of the oracle over about `seconds` of host time (at least 2 tokens)."""
    _cpu_inputs()
    per = cpu_oracle_tokens(1, threads)
    n = max(2, int(seconds / max(per, 1e-6)))
    el = cpu_oracle_tokens(n, threads)
    return B_TOKEN * n / el / 1e9, n, el


def run_ours(args):
    import torch
    import weight_streaming_warp_gb300 as wsw
    from weight_streaming_warp_gb300 import build as wbuild

    rank, world, local = _dist()
    wbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    wl = Workload(wsw, torch, dev)
    step_graph = _graph(torch, wl.step)

    for _ in range(args.warmup):
        step_graph.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    e0.record()
    for _ in range(args.steps):
        step_graph.replay()
    e1.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if pg:
        pg.barrier()
    clocks.mark(t0, t1)
    clk = clocks.stop()
    value, elapsed = whole_job_rate(pg, torch, e0.elapsed_time(e1) / 1000.0,
                                    B_TOKEN * TOKENS * args.steps / 1e9, device=dev)
    step_s = elapsed / args.steps

    # the same step with the quantizer as its own launch
    two_graph = _graph(torch, lambda stream: wl.step(stream, fused=False))
    for _ in range(2):
        two_graph.replay()
    two_s = statistics.median(_time_graph(torch, two_graph, 1) for _ in range(5))
    del two_graph

    peak, peak_kind = _peaks()
    k_med, k_min, k_max = measure_gemv_kernel(torch, wl)
    achieved = B_FUSED / k_med / 1e9
    g_med, _, _ = measure_gemv_kernel(torch, wl, fused=False)
    quant = measure_quantizer(torch, wl)
    e2e = measure_e2e(torch, wl, dev, args.steps, step_graph)
    e2e_eager = measure_e2e(torch, wl, dev, args.steps)
    del step_graph
    chain = measure_chain(torch, wsw, dev) if rank == 0 else None
    config1 = measure_config1(torch, wsw, dev) if rank == 0 else None
    rows, moe_steps = measure_rows(torch, wsw, dev) if rank == 0 else (None, None)

    if pg:
        pg.barrier()
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    cores = host_cores()
    cpu1 = cpu_oracle_rate(seconds=8.0) if world == 1 else None
    cpuN = cpu_oracle_rate(seconds=8.0, threads=cores) if world == 1 else None
    if chain is not None:
        for arm in ("pdl", "no_pdl", "pdl_l2_prefetch_4"):
            chain[arm]["frac_of_measured"] = round(chain[arm]["GBps"] / peak, 4)
            chain[arm]["frac_of_nominal_8TBps"] = round(chain[arm]["GBps"] / NOMINAL_HBM_GBS, 4)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8",
        "data": "synthetic: seeded N(0,0.02) bf16 weights quantized to q8_0, N(0,1) activations",
        "config": {"workload": WORKLOAD,
                   "arithmetic": "int8 x int8 -> exact int32 block sums, fp32 scales and accumulation; "
                                 "fp32 quantizer",
                   "tokens_per_step": TOKENS, "bytes_per_token": B_TOKEN,
                   "weight_copies": NCOPY, "weight_bytes_per_copy": B_GEMV - K - (K // 32) * 2 - M * 4,
                   "l2": "inputs larger than L2: 16 rotating weight copies (1.0 GB) vs 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "timing": "CUDA events around K replays of a CUDA graph of one step"},
        "pct_of_measured_hbm_peak": round(100.0 * value / world / peak, 2),
        "pct_of_nominal_8TBps": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
        "roofline": {"kernel": "stream_gemv_kernel<Q8X> (quantize_gemv_q8_0)", "bound": "hbm",
                     "achieved": round(achieved, 1),
                     "peak": peak, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy)",
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_of_nominal_8TBps": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": _traffic_record("quantize_gemv_q8_0"),
                     "algorithmic_bytes_per_launch": B_FUSED,
                     "launch_us": {"median": round(k_med * 1e6, 3), "min": round(k_min * 1e6, 3),
                                   "max": round(k_max * 1e6, 3)}},
        "gemv_q8_0_alone": {"GBps": round(B_GEMV / g_med / 1e9, 1), "frac": round(B_GEMV / g_med / 1e9 / peak, 4),
                            "launch_us": round(g_med * 1e6, 3), "traffic": _traffic_record("gemv_q8_0"),
                            "algorithmic_bytes_per_launch": B_GEMV},
        "two_launch_step": {"GBps": round(B_TOKEN_2L * TOKENS / two_s / 1e9, 2),
                            "ms_per_step": round(two_s * 1e3, 4),
                            "note": "quantize_q8 -> gemv_q8_0 as two PDL-linked launches per token"},
        "rows": rows,
        "e2e": e2e,
        "e2e_eager": e2e_eager,
        "gpu_launches": 3 * TOKENS * args.steps,
        "clocks": clk,
        "cpu_baseline": None if cpuN is None else {
            "value": round(cpuN[0], 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d full tokens (quantize + 14336x4096 q8_0 GEMV rows cut over %d host threads + 2 "
                      "superblock quantizations) in %.1f s" % (cpuN[1], cores, cpuN[2]),
            "single_core": {"value": round(cpu1[0], 4), "cores": 1,
                            "sample": "%d full tokens in %.1f s" % (cpu1[1], cpu1[2])}},
        "chain_27b_bf16": chain,
        "config1_gemv_bf16_4096x4096": config1,
        "moe_step": None if moe_steps is None else {"T%d" % T: s for T, s in moe_steps.items()},
    }
    # The figures a reader needs first, last on the line.
    if rank == 0:
        key = {"fused_q8_0_gemv": {"GBps": round(achieved, 1), "frac_measured": round(achieved / peak, 4),
                                   "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4)},
               "gemv_q8_0_alone_frac": round(B_GEMV / g_med / 1e9 / peak, 4),
               "quantizer_us_per_call": quant}
        if chain is not None:
            c = chain["pdl"]
            key["chain_27b_bf16_pdl"] = {"GBps": c["GBps"], "tok_per_s": c["tok_per_s"],
                                         "frac_measured": c["frac_of_measured"],
                                         "frac_nominal": c["frac_of_nominal_8TBps"]}
        if config1 is not None:
            key["config1_gemv_bf16"] = {"GBps_pdl": config1["GBps_pdl"], "GBps": config1["GBps"],
                                        "frac_pdl": round(config1["GBps_pdl"] / peak, 4),
                                        "GBps_l2hot": config1["GBps_l2hot"]}
        if rows is not None:
            key["attn_prefill_TFLOPs_pdl"] = {
                "d%d" % d: rows["attn_prefill_d%d_per_head" % d]["TFLOPs_pdl"] for d in (32768, 65536)}
            key["attn_prefill_frac_of_bf16_peak"] = {
                "d%d" % d: rows["attn_prefill_d%d_per_head" % d]["frac_of_bf16_peak_pdl"] for d in (32768, 65536)}
            key["windowed_q8_0_prefill_TFLOPs_pdl"] = {
                "d32768_w4096": rows["windowed_q8_0_prefill_d32768_w4096"]["TFLOPs_pdl"],
                "d65536_w8192": rows["windowed_q8_0_prefill_d65536_w8192"]["TFLOPs_pdl"]}
            key["attn_decode_pdl"] = _decode_attn_key(rows, peak)
        if moe_steps is not None:
            key["config4_moe_step_us_pdl"] = {"T%d" % T: s["us_pdl"] for T, s in moe_steps.items()}
            key["config4_moe_step_GBps_pdl"] = {"T%d" % T: s["GBps_pdl"] for T, s in moe_steps.items()}
        if cpuN is not None:
            key["cpu_oracle_GBps"] = {"cores_%d" % cores: round(cpuN[0], 3), "cores_1": round(cpu1[0], 3)}
        line["key_numbers"] = key
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    import oracle
    oracle.lib()
    _cpu_inputs()
    cores = host_cores()
    cpu_oracle_tokens(args.warmup, cores)
    el = cpu_oracle_tokens(args.steps, cores)
    value = B_TOKEN * args.steps / el / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": WORKLOAD, "arithmetic": "fp64 oracle",
                                        "sample": "one token per step"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "one full token per step (all 14336 rows, cut over %d host threads)" % cores},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------- profile cases --
def profile_case(argv):
    """Run one hot-path call on its configured shape a few times, for a profiler:

        python bench.py --profile-case gemv_q8_0
        python bench.py --profile-case quantize_gemv_q8_0
        python bench.py --profile-case gemv_bf16 [M K]
        python bench.py --profile-case gemm_bf16 [N]
        python bench.py --profile-case dequant_kv [depth]
        python bench.py --profile-case moe [T [gate_up|down]]
        python bench.py --profile-case moe_repeat
        python bench.py --profile-case quantize [n block]
        python bench.py --profile-case attn_decode [depth group]
        python bench.py --profile-case attn_prefill [depth]

    Weights rotate over copies that together exceed the 129 MB L2, so every profiled
    launch streams its weights from HBM; the device holds at most a few GB.  Inputs
    are random (values do not change the work of these kernels)."""
    import torch
    import weight_streaming_warp_gb300 as wsw
    from weight_streaming_warp_gb300 import build as wbuild
    wbuild.build()
    what = argv[0] if argv else "gemv_q8_0"
    dev = "cuda"
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    launches = 6
    if what in ("gemv_q8_0", "quantize_gemv_q8_0"):
        nc = 4
        Wq = [torch.randint(-127, 128, (M, K), dtype=torch.int8, device=dev, generator=g) for _ in range(nc)]
        Wd = [(torch.rand((M, K // 32), device=dev, generator=g) * 1e-3).half() for _ in range(nc)]
        x = torch.randn((launches, K), device=dev, generator=g)
        xq = torch.empty(K, dtype=torch.int8, device=dev)
        xd = torch.empty(K // 32, dtype=torch.float16, device=dev)
        for i in range(launches):
            if what == "gemv_q8_0":
                wsw.gemv_q8_0(Wq[i % nc], Wd[i % nc], xq, xd)
            else:
                wsw.quantize_gemv_q8_0(Wq[i % nc], Wd[i % nc], x[i], x_out=(xq, xd))
    elif what == "gemv_bf16":
        Mi, Ki = (int(argv[1]), int(argv[2])) if len(argv) > 2 else (5120, 17408)
        nc = max(2, (512 << 20) // (Mi * Ki * 2) + 1)
        W = [torch.randn((Mi, Ki), device=dev, generator=g).to(torch.bfloat16) for _ in range(nc)]
        x = torch.randn(Ki, device=dev, generator=g)
        for i in range(launches):
            wsw.gemv_bf16(W[i % nc], x)
    elif what == "gemm_bf16":
        N = int(argv[1]) if len(argv) > 1 else 512
        Mg, Kg, nc = 2560, 10240, 4
        W = [torch.randn((Mg, Kg), device=dev, generator=g).mul_(0.02).to(torch.bfloat16) for _ in range(nc)]
        X = torch.randn((N, Kg), device=dev, generator=g).to(torch.bfloat16)
        for i in range(launches):
            wsw.gemm_bf16(W[i % nc], X)
    elif what == "dequant_kv":
        D = int(argv[1]) if len(argv) > 1 else 65536
        nc = 4
        q = [torch.randint(-127, 128, (D, 4, 128), dtype=torch.int8, device=dev, generator=g) for _ in range(nc)]
        d = [torch.rand((D, 4, 4), device=dev, generator=g).half() for _ in range(nc)]
        for i in range(launches):
            wsw.dequant_q8_0_kv(q[i % nc], d[i % nc])
    elif what == "moe":
        from weight_streaming_warp_gb300 import synthetic as syn
        T = int(argv[1]) if len(argv) > 1 else 16
        down = len(argv) > 2 and argv[2] == "down"
        E = MOE_E
        Mo, Kx = (MOE_H, MOE_F) if down else (2 * MOE_F, MOE_H)
        Wq = torch.randint(-127, 128, (E, Mo, Kx), dtype=torch.int8, device=dev, generator=g)
        Wd = (torch.rand((E, Mo, Kx // 32), device=dev, generator=g) * 1e-3).half()
        ids = syn.routing(0, "profile%d" % T, T, E, MOE_TOPK).to(dev)
        xq = torch.randint(-127, 128, (T * MOE_TOPK, Kx), dtype=torch.int8, device=dev, generator=g)
        xd = torch.rand((T * MOE_TOPK, Kx // 32), device=dev, generator=g).half()
        for _ in range(launches):
            wsw.moe_gemv_q8_0(Wq, Wd, xq, xd, ids)
    elif what == "moe_repeat":
        # the gathered form (16 routed rows) with each of 8 experts routed twice; two
        # weight copies alternate, so a call finds none of its experts in L2
        E, Mo, Kx = MOE_E, 2 * MOE_F, MOE_H
        W = [(torch.randint(-127, 128, (E, Mo, Kx), dtype=torch.int8, device=dev, generator=g),
              (torch.rand((E, Mo, Kx // 32), device=dev, generator=g) * 1e-3).half()) for _ in range(2)]
        ids = torch.tensor([3, 17, 3, 40, 17, 99, 40, 5, 99, 64, 5, 64, 120, 7, 120, 7], dtype=torch.int32,
                           device=dev)
        xq = torch.randint(-127, 128, (16, Kx), dtype=torch.int8, device=dev, generator=g)
        xd = torch.rand((16, Kx // 32), device=dev, generator=g).half()
        for i in range(launches):
            wsw.moe_gemv_q8_0(W[i % 2][0], W[i % 2][1], xq, xd, ids)
    elif what == "attn_decode":
        D = int(argv[1]) if len(argv) > 1 else 32768
        G = int(argv[2]) if len(argv) > 2 else 1
        nc = 3  # 3 x 67 MB of K and V at depth 32768
        Kt = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        Vt = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        q = torch.randn((4, G, 128), device=dev, generator=g)
        for i in range(launches):
            wsw.attn_decode_f16(q, Kt[i % nc], Vt[i % nc])
    elif what == "attn_prefill":
        D = int(argv[1]) if len(argv) > 1 else 32768
        nc = 3
        Kt = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        Vt = [torch.randn((4, D, 128), device=dev, generator=g).half() for _ in range(nc)]
        q = torch.randn((4, 8, 512, 128), device=dev, generator=g).half()
        for i in range(launches):
            wsw.attn_prefill_f16(q, Kt[i % nc], Vt[i % nc])
    elif what == "quantize":
        n = int(argv[1]) if len(argv) > 1 else 4096
        block = int(argv[2]) if len(argv) > 2 else 32
        X = torch.randn((64, n), device=dev, generator=g)
        for i in range(launches):
            wsw.quantize_q8(X[i], block)
    else:
        raise SystemExit("unknown profile case %r" % what)
    torch.cuda.synchronize()
    print("done", what)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--profile-case", nargs="+", metavar="CASE",
                    help="run one call a few times for a profiler (see profile_case) and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
