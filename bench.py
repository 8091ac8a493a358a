"""Benchmark of the NVFP4 hot path on GB300.

One step runs every stage of the path once on synthetic inputs shaped like
the pages' workloads, inputs resident in HBM:
  prefill  activation quantisation + W4A4 block-scaled GEMM of the fused
           qkv-style linear (M = 8192 tokens, N = 5120 + 1024 + 1024, K = 5120)
  decode   W4A16 GEMM at T = 1, 2, 4, 8, 16 on (N, K) = (8704, 5120) and
           (5120, 4352), each a CUDA graph over >= 2.5 GB of distinct weight
           copies so that every call reads its weight from HBM
  moe      the W4A4 MoE layer, E = 128, top-8, hidden 2048, intermediate 768,
           T = 4096 (align, permute+quantise, gate_up with SiLU*up and NVFP4
           requantisation, down with routing weight and top-k sum, bf16)
The L2 is flushed before each stage (a 256 MiB write, then a 256 MiB read so
that the write's dirty lines are written back before the stage); the flush is
outside the timed events.  `value` is the W4A4 prefill throughput in TFLOP/s (the
first clause of the metric); the decode GB/s and MoE TFLOP/s are reported in
their own objects.  Multi-GPU: replicas (each rank runs the same step on its
own GPU, weak scaling).

--impl reference times the CPU oracle (the only reference this path has) on
a bounded sample of the same prefill workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synthdata  # noqa: E402

METRIC = "W4A4 prefill TFLOP/s (frac of FP4 peak); W4A16 decode HBM GB/s at T=1..16"
PREFILL_M = 8192
MOE_T = 4096
MOE16_T = (1, 4, 16)
MOE16_BANKS = 8  # expert-bank copies, one per call of a CUDA graph (8 x 340 MB: cold experts)
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor ratio of GB300


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        try:
            lines = [ln.split(",") for ln in open(self.path).read().strip().splitlines() if ln.strip()]
        except Exception:
            return out
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for f in lines:
            f = [x.strip() for x in f]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), reasons=sorted(reasons), samples=len(sm))
        return out


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------

class Workload:
    def __init__(self, dev, nv):
        self.nv = nv
        self.dev = dev
        self.lib = nv.load_library()
        # prefill (fused qkv linear)
        pc = synthdata.prefill_case(PREFILL_M, seed=0, device=dev)
        self.pre_W = nv.quantize_weight(pc.w_parts)
        self.pre_x = pc.x
        self.pre_g = nv.nvfp4_compute_global(pc.x_calib)
        self.pre_alpha = nv.nvfp4_make_alpha(self.pre_g, self.pre_W.g)
        self.pre_codes, self.pre_sf = nv.nvfp4_quantize_act(self.pre_x, self.pre_g)
        self.pre_out = torch.empty(PREFILL_M, self.pre_W.N, dtype=torch.bfloat16, device=dev)
        self.pre_flops = 2.0 * PREFILL_M * self.pre_W.N * self.pre_W.K
        N, K, M = self.pre_W.N, self.pre_W.K, PREFILL_M
        self.pre_bytes = N * K // 2 + nv.nvfp4_scale_bytes(N, K) + M * K // 2 + nv.nvfp4_scale_bytes(M, K) + 2 * M * N
        self.quant_bytes = M * K * 2 + M * K // 2 + nv.nvfp4_scale_bytes(M, K)
        # decode
        self.decode = []
        for (N, K) in synthdata.DECODE_SHAPES:
            d = synthdata.decode_case(16, N, K, seed=1, device=dev)
            W = nv.quantize_weight(d.w_parts)
            alpha = nv.nvfp4_make_alpha(None, W.g)
            wbytes = N * K // 2 + nv.nvfp4_scale_bytes(N, K)
            ncopy = max(2, int(2.5e9 // wbytes) + 1)
            codes = [W.codes] + [W.codes.clone() for _ in range(ncopy - 1)]
            scales = [W.scales] + [W.scales.clone() for _ in range(ncopy - 1)]
            for T in synthdata.DECODE_TOKENS:
                x = d.x[:T].contiguous()
                out = torch.empty(T, N, dtype=torch.bfloat16, device=dev)
                wsb = nv.nvfp4_linear_w4a16_workspace(T, N, K)
                ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev)
                self.decode.append(dict(N=N, K=K, T=T, x=x, out=out, ws=ws, wsb=wsb, codes=codes, scales=scales,
                                        alpha=alpha, ncopy=ncopy, wbytes=wbytes,
                                        bytes=wbytes + 2 * T * K + 2 * T * N, graph=None,
                                        launches=1 + (1 if wsb > 0 else 0)))
        # MoE
        cfg = synthdata.MOE_SMALL
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        mc = synthdata.moe_case(MOE_T, E, H, I, topk, cfg["skewed"], seed=0, device=dev)
        self.moe_W = nv.quantize_moe_weights(lambda e: mc.w13(e), lambda e: mc.w2(e), E, H, I, dev)
        self.moe_g_a1 = nv.nvfp4_compute_global(mc.x_calib)
        self.moe_a13 = nv.nvfp4_make_alpha(self.moe_g_a1, self.moe_W.g13)
        self.moe_g_a2, _ = nv.nvfp4_moe_calibrate(mc.x_calib, self.moe_g_a1, self.moe_W.w13_codes,
                                                  self.moe_W.w13_sf, self.moe_a13, E, I)
        self.moe_a2 = nv.nvfp4_make_alpha(self.moe_g_a2, self.moe_W.g2)
        self.moe_x, self.moe_ids, self.moe_w = mc.x, mc.topk_ids, mc.topk_w
        self.moe_out = torch.empty(MOE_T, H, dtype=torch.bfloat16, device=dev)
        self.moe_ws = torch.empty(nv.nvfp4_moe_workspace(MOE_T, H, I, E, topk), dtype=torch.uint8, device=dev)
        self.moe_E, self.moe_I, self.moe_H, self.moe_topk = E, I, H, topk
        self.moe_flops = 2.0 * MOE_T * topk * 3 * H * I
        # algorithmic bytes of the layer: the touched experts' W13 and W2 (codes and
        # scales), x and out in bf16, and the NVFP4 intermediate written and read once
        used = int(torch.unique(mc.topk_ids).numel())
        ebytes = 2 * I * H // 2 + nv.nvfp4_scale_bytes(2 * I, H) + H * I // 2 + nv.nvfp4_scale_bytes(H, I)
        R = MOE_T * topk
        self.moe_bytes = used * ebytes + 2 * MOE_T * H * 2 + 2 * (R * I // 2 + nv.nvfp4_scale_bytes(R, I))
        # W4A16 MoE for small batches on the same expert banks (decode-sized T)
        self.moe16_a13 = nv.nvfp4_make_alpha(None, self.moe_W.g13)
        self.moe16_a2 = nv.nvfp4_make_alpha(None, self.moe_W.g2)
        ebytes = 2 * I * H // 2 + nv.nvfp4_scale_bytes(2 * I, H) + H * I // 2 + nv.nvfp4_scale_bytes(H, I)
        bank0 = (self.moe_W.w13_codes, self.moe_W.w13_sf, self.moe_W.w2_codes, self.moe_W.w2_sf)
        self.moe16_banks = [bank0] + [tuple(t.clone() for t in bank0) for _ in range(MOE16_BANKS - 1)]
        self.moe16 = []
        for T in MOE16_T:
            c = synthdata.moe_case(T, E, H, I, topk, cfg["skewed"], seed=T, device=dev)
            used = int(torch.unique(c.topk_ids).numel())
            self.moe16.append(dict(T=T, x=c.x, ids=c.topk_ids, w=c.topk_w, experts=used,
                                   out=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                                   ws=torch.empty(nv.nvfp4_moe_w4a16_workspace(T, H, I, E, topk), dtype=torch.uint8,
                                                  device=dev),
                                   bytes=used * ebytes + 2 * T * H * 2, graph=None))
        self.flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
        self.flush_src = torch.ones(64 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.flush_sink = torch.empty(1, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()

    def large_moe(self):
        """Weights and static globals of the E = 256 MoE (built on first use):
        (W, g_a1, alpha13, g_a2, alpha2)."""
        nv = self.nv
        cfg = synthdata.MOE_LARGE
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        mc = synthdata.moe_case(16, E, H, I, topk, cfg["skewed"], seed=0, device=self.dev)
        W = nv.quantize_moe_weights(lambda e: mc.w13(e), lambda e: mc.w2(e), E, H, I, self.dev)
        g1 = nv.nvfp4_compute_global(mc.x_calib)
        a13 = nv.nvfp4_make_alpha(g1, W.g13)
        g2, _ = nv.nvfp4_moe_calibrate(mc.x_calib, g1, W.w13_codes, W.w13_sf, a13, E, I)
        a2 = nv.nvfp4_make_alpha(g2, W.g2)
        return W, g1, a13, g2, a2

    # --- stages ------------------------------------------------------------
    def prefill(self):
        nv = self.nv
        nv.nvfp4_quantize_act(self.pre_x, self.pre_g, self.pre_codes, self.pre_sf)
        nv.nvfp4_linear_w4a4(self.pre_codes, self.pre_sf, self.pre_W.codes, self.pre_W.scales, self.pre_alpha,
                             self.pre_W.N, self.pre_W.K, out=self.pre_out)

    def quant_only(self):
        self.nv.nvfp4_quantize_act(self.pre_x, self.pre_g, self.pre_codes, self.pre_sf)

    def gemm_only(self):
        self.nv.nvfp4_linear_w4a4(self.pre_codes, self.pre_sf, self.pre_W.codes, self.pre_W.scales,
                                  self.pre_alpha, self.pre_W.N, self.pre_W.K, out=self.pre_out)

    def moe(self):
        self.nv.nvfp4_moe_w4a4(self.moe_x, self.moe_ids, self.moe_w, self.moe_g_a1, self.moe_W.w13_codes,
                               self.moe_W.w13_sf, self.moe_a13, self.moe_g_a2, self.moe_W.w2_codes,
                               self.moe_W.w2_sf, self.moe_a2, self.moe_E, self.moe_I, out=self.moe_out,
                               workspace=self.moe_ws)

    def moe16_call(self, c, j):
        w13c, w13s, w2c, w2s = self.moe16_banks[j]
        self.nv.nvfp4_moe_w4a16(c["x"], c["ids"], c["w"], w13c, w13s, self.moe16_a13, w2c, w2s, self.moe16_a2,
                                self.moe_E, self.moe_I, out=c["out"], workspace=c["ws"])

    def build_moe16_graphs(self):
        """One CUDA graph per T: a chain of MOE16_BANKS W4A16 MoE calls, call j
        on bank copy j (as the MoE layers of a decode step, each with its own
        experts), so every call reads its experts from HBM."""
        for c in self.moe16:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                self.moe16_call(c, 0)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(len(self.moe16_banks)):
                    self.moe16_call(c, j)
            c["graph"] = g
        torch.cuda.synchronize()

    def build_decode_graphs(self):
        lib = self.lib
        for d in self.decode:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())

            def call(j, d=d, stream=None):
                st = lib.nvfp4_linear_w4a16(
                    ctypes.c_void_p(d["x"].data_ptr()), d["T"], d["K"], ctypes.c_void_p(d["codes"][j].data_ptr()),
                    ctypes.c_void_p(d["scales"][j].data_ptr()), d["N"], d["K"], ctypes.c_void_p(d["alpha"].data_ptr()),
                    ctypes.c_void_p(d["out"].data_ptr()), d["N"], ctypes.c_void_p(d["ws"].data_ptr()),
                    d["ws"].numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
                if st != 0:
                    raise RuntimeError(f"nvfp4_linear_w4a16 status {st}")
            with torch.cuda.stream(s):
                call(0)
            torch.cuda.current_stream().wait_stream(s)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for j in range(d["ncopy"]):
                    call(j)
            d["graph"] = g
        torch.cuda.synchronize()

    def flush(self):
        # write 256 MiB (evicts everything), then read another 256 MiB: the
        # dirty lines of the write are written back here rather than during
        # the next timed stage, which starts with a cold and clean L2
        self.flush_buf.fill_(1)
        torch.sum(self.flush_src, dim=0, keepdim=True, out=self.flush_sink)

    def launches_per_step(self) -> int:
        # prefill (quantise + GEMM), GEMM alone, quantiser alone; the decode graphs;
        # the W4A4 MoE layer (align x3, quantise/permute, gate_up, down, finalize);
        # the W4A16 MoE graphs (gate_up, down, finalize per call)
        return (4 + sum(d["ncopy"] * d["launches"] for d in self.decode) + 7 +
                3 * len(self.moe16_banks) * len(self.moe16))


def _decode_kernel(T: int) -> str:
    """The decode GEMM instantiation a call with T tokens runs on these shapes:
    two k-groups below 4 tokens, three from 4; 16 tokens per MMA pass above 8."""
    return f"gemv_ring_kernel<{1 if T > 8 else 0}, {3 if T >= 4 else 2}>"


def _decode_kernel_rooflines(wl, decode: dict, hbm: float) -> dict:
    """Per decode instantiation: its share of the step's decode time (every
    graph replays its calls once per step) and its time-weighted bandwidth."""
    agg = {}
    for d in wl.decode:
        t = decode[f"T{d['T']}_{d['N']}x{d['K']}"]["us"] * 1e-6
        a = agg.setdefault(_decode_kernel(d["T"]), [0.0, 0.0])
        a[0] += d["ncopy"] * t
        a[1] += d["ncopy"] * d["bytes"]
    total = sum(v[0] for v in agg.values())
    return {k: {"share_of_decode_time": round(v[0] / total, 4), "gbs": round(v[1] / v[0] / 1e9, 1),
                "frac_hbm": round(v[1] / v[0] / 1e9 / hbm, 4)} for k, v in agg.items()}


def _profile_traffic(name: str):
    """DRAM bytes per launch recorded in profiles/<name> by an ncu capture, or
    None when the kernel source has changed since (its git blob hash differs
    from the one recorded with the capture) or the summary is missing."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
        src, blob = next(l.split()[1:3] for l in text.splitlines() if l.startswith("source-blob:"))
        nbytes = next(int(l.split()[1]) for l in text.splitlines() if l.startswith("dram-bytes-per-launch:"))
        data = open(os.path.join(ROOT, src), "rb").read()
        now = hashlib.sha1(b"blob %d\0" % len(data) + data).hexdigest()
        return nbytes if now == blob else None
    except (OSError, StopIteration, ValueError, IndexError):
        return None


def max_over_ranks(values, world: int, device="cpu"):
    """The slowest replica bounds the job: element-wise max of per-rank times
    over all ranks (any backend: NCCL on GPUs, gloo on CPU)."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def job_throughput(world: int, units_per_rank: float, seconds: float) -> float:
    """Weak scaling: every rank processes the same units; the job's rate is all
    ranks' units over the slowest rank's time."""
    return world * units_per_rank / seconds


def _timed(fn, stream):
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    return a, b


def _median_ms(fn, flush, reps, stream):
    """Median CUDA-event time of fn over reps runs, the L2 flushed before each
    (outside the events)."""
    ts = []
    for _ in range(reps):
        flush()
        a, b = _timed(fn, stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def _roof(flops, nbytes, seconds, hbm, fp4_peak):
    """Achieved rates and the roofline of one timed stage: the roofline time is
    the larger of its FP4 tensor time and its HBM time."""
    t_fp4 = flops / (fp4_peak * 1e12)
    t_hbm = nbytes / (hbm * 1e9)
    return {"tflops": round(flops / seconds / 1e12, 2), "gbs": round(nbytes / seconds / 1e9, 1),
            "frac_fp4_peak": round(flops / seconds / 1e12 / fp4_peak, 4),
            "bytes": int(nbytes), "roofline_us": round(max(t_fp4, t_hbm) * 1e6, 2),
            "bound": "tensor" if t_fp4 >= t_hbm else "hbm",
            "frac_roofline": round(max(t_fp4, t_hbm) / seconds, 4)}


def _moe_bytes(nv, ids, T, E, H, I, topk):
    """Algorithmic bytes of one MoE layer: the W13 and W2 codes and scales of the
    experts in use, x and out in bf16, the NVFP4 intermediate written and read once."""
    used = int(torch.unique(ids[(ids >= 0) & (ids < E)]).numel())
    ebytes = 2 * I * H // 2 + nv.nvfp4_scale_bytes(2 * I, H) + H * I // 2 + nv.nvfp4_scale_bytes(H, I)
    R = T * topk
    return used * ebytes + 2 * T * H * 2 + 2 * (R * I // 2 + nv.nvfp4_scale_bytes(R, I)), used


def sweep_configs(wl, nv, dev, hbm, fp4_peak, reps=5):
    """Every workload shape, timed stage by stage outside the step (each the
    median of `reps` runs, L2 flushed before each): the tiny W4A4 linear, the
    fused-qkv prefill at every M (quantise + GEMM, and the GEMM alone), the
    E = 128 MoE layer at every T and the E = 256 MoE layer at every T."""
    stream = torch.cuda.current_stream()
    flush = wl.flush
    out = {}
    # tiny W4A4 linear: M = 8, N = 256, K = 512
    tc = synthdata.tiny_linear(seed=0, device=dev)
    Wt = nv.quantize_weight(tc.w_parts)
    gt = nv.nvfp4_compute_global(tc.x_calib)
    at = nv.nvfp4_make_alpha(gt, Wt.g)
    ct, st = nv.nvfp4_quantize_act(tc.x, gt)
    ot = torch.empty(tc.x.shape[0], Wt.N, dtype=torch.bfloat16, device=dev)
    M, N, K = tc.x.shape[0], Wt.N, Wt.K

    def tiny():
        nv.nvfp4_quantize_act(tc.x, gt, ct, st)
        nv.nvfp4_linear_w4a4(ct, st, Wt.codes, Wt.scales, at, N, K, out=ot)
    t = _median_ms(tiny, flush, 4 * reps, stream) * 1e-3
    nb = N * K // 2 + nv.nvfp4_scale_bytes(N, K) + 2 * M * K + 2 * M * N
    out["tiny_w4a4_M8_N256_K512"] = dict(us=round(t * 1e6, 2), **_roof(2.0 * M * N * K, nb, t, hbm, fp4_peak))
    # prefill, fused qkv weight, every M: rows and scale atoms of the M = 8192
    # buffers are prefixes of the smaller problems
    pre = {}
    N, K = wl.pre_W.N, wl.pre_W.K
    for M in synthdata.PREFILL_M:
        x = wl.pre_x[:M]
        codes, sf = wl.pre_codes[:M], wl.pre_sf[:nv.nvfp4_scale_bytes(M, K)]
        o = wl.pre_out[:M]

        def quant_gemm(x=x, codes=codes, sf=sf, o=o):
            nv.nvfp4_quantize_act(x, wl.pre_g, codes, sf)
            nv.nvfp4_linear_w4a4(codes, sf, wl.pre_W.codes, wl.pre_W.scales, wl.pre_alpha, N, K, out=o)

        def gemm(codes=codes, sf=sf, o=o):
            nv.nvfp4_linear_w4a4(codes, sf, wl.pre_W.codes, wl.pre_W.scales, wl.pre_alpha, N, K, out=o)
        tq = _median_ms(quant_gemm, flush, reps, stream) * 1e-3
        tg = _median_ms(gemm, flush, reps, stream) * 1e-3
        fl = 2.0 * M * N * K
        b_gemm = N * K // 2 + nv.nvfp4_scale_bytes(N, K) + M * K // 2 + nv.nvfp4_scale_bytes(M, K) + 2 * M * N
        b_pre = N * K // 2 + nv.nvfp4_scale_bytes(N, K) + 2 * M * K + 2 * M * N
        pre[f"M{M}"] = {"quant_gemm_us": round(tq * 1e6, 2), "quant_gemm": _roof(fl, b_pre, tq, hbm, fp4_peak),
                        "gemm_us": round(tg * 1e6, 2), "gemm": _roof(fl, b_gemm, tg, hbm, fp4_peak)}
    out["prefill_fused_qkv_N7168_K5120"] = pre
    # small batches on the fused qkv weight: the W4A4 GEMM beside the W4A16
    # decode GEMM, each a CUDA graph over 16 weight copies (cold weights)
    small = {}
    copies16 = [(wl.pre_W.codes, wl.pre_W.scales)] + [(wl.pre_W.codes.clone(), wl.pre_W.scales.clone())
                                                      for _ in range(15)]
    alpha16 = nv.nvfp4_make_alpha(None, wl.pre_W.g)
    wbytes = N * K // 2 + nv.nvfp4_scale_bytes(N, K)

    def graph_us(call):
        s2 = torch.cuda.Stream()
        s2.wait_stream(stream)
        with torch.cuda.stream(s2):
            call(0)
        stream.wait_stream(s2)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(len(copies16)):
                call(j)
        return _median_ms(g.replay, flush, reps, stream) * 1e3 / len(copies16)

    for M in (1, 8, 16, 32, 48, 64, 128, 256):
        x = wl.pre_x[:M]
        codes, sf = nv.nvfp4_quantize_act(x, wl.pre_g)
        o = torch.empty(M, N, dtype=torch.bfloat16, device=dev)

        def w4a4(j, codes=codes, sf=sf, o=o):
            nv.nvfp4_linear_w4a4(codes, sf, copies16[j][0], copies16[j][1], wl.pre_alpha, N, K, out=o)
        entry = {"w4a4_gemm_us": round(graph_us(w4a4), 2)}
        entry["w4a4_gbs"] = round(wbytes / entry["w4a4_gemm_us"] / 1e3, 1)
        if M <= 16:
            ws = torch.empty(max(nv.nvfp4_linear_w4a16_workspace(M, N, K), 16), dtype=torch.uint8, device=dev)

            def w4a16(j, x=x, o=o, ws=ws):
                nv.nvfp4_linear_w4a16(x, copies16[j][0], copies16[j][1], alpha16, N, K, out=o, workspace=ws)
            entry["w4a16_us"] = round(graph_us(w4a16), 2)
        small[f"M{M}"] = entry
    out["small_batch_fused_qkv_N7168_K5120"] = small
    del copies16
    # a stack of 8 prefill layers (quantise + GEMM, M = 8192) on 8 distinct
    # weight copies in one CUDA graph: the activations of a layer and its
    # output meet the next layer's weights in L2
    M = synthdata.PREFILL_M[-1]
    copies = [(wl.pre_W.codes, wl.pre_W.scales)] + [(wl.pre_W.codes.clone(), wl.pre_W.scales.clone())
                                                    for _ in range(7)]

    def stack():
        for c, sc in copies:
            nv.nvfp4_quantize_act(wl.pre_x, wl.pre_g, wl.pre_codes, wl.pre_sf)
            nv.nvfp4_linear_w4a4(wl.pre_codes, wl.pre_sf, c, sc, wl.pre_alpha, N, K, out=wl.pre_out)
    s2 = torch.cuda.Stream()
    s2.wait_stream(stream)
    with torch.cuda.stream(s2):
        stack()
    stream.wait_stream(s2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        stack()
    t = _median_ms(g.replay, flush, reps, stream) * 1e-3 / len(copies)
    fl = 2.0 * M * N * K
    b_pre = N * K // 2 + nv.nvfp4_scale_bytes(N, K) + 2 * M * K + 2 * M * N
    out["prefill_stack_8_layers_M8192"] = dict(us_per_layer=round(t * 1e6, 2), **_roof(fl, b_pre, t, hbm, fp4_peak))
    del copies, g
    # MoE layers
    for name, cfg, W, g1, a13, g2, a2 in (
            ("moe_E128_H2048_I768", synthdata.MOE_SMALL, wl.moe_W, wl.moe_g_a1, wl.moe_a13, wl.moe_g_a2, wl.moe_a2),
            ("moe_E256_H7168_I2048", synthdata.MOE_LARGE) + wl.large_moe()):
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        res = {}
        ws = torch.empty(nv.nvfp4_moe_workspace(max(cfg["tokens"]), H, I, E, topk), dtype=torch.uint8, device=dev)
        for T in cfg["tokens"]:
            c = synthdata.moe_case(T, E, H, I, topk, cfg["skewed"], seed=0, device=dev)
            o = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

            def layer(c=c, o=o):
                nv.nvfp4_moe_w4a4(c.x, c.topk_ids, c.topk_w, g1, W.w13_codes, W.w13_sf, a13, g2, W.w2_codes,
                                  W.w2_sf, a2, E, I, out=o, workspace=ws)
            layer()
            t = _median_ms(layer, flush, reps, stream) * 1e-3
            nb, used = _moe_bytes(nv, c.topk_ids, T, E, H, I, topk)
            res[f"T{T}"] = dict(ms=round(t * 1e3, 4), experts_used=used,
                                **_roof(2.0 * T * topk * 3 * H * I, nb, t, hbm, fp4_peak))
            del c, o
        out[name] = res
        del ws
    torch.cuda.synchronize()
    return out


def run_ours(args, world, rank, local):
    import nvfp4_block_scaled_act_gb300 as nv
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = Workload(dev, nv)
    wl.build_decode_graphs()
    wl.build_moe16_graphs()
    stream = torch.cuda.current_stream()

    def step(record):
        wl.flush()
        ev_pre = _timed(wl.prefill, stream)
        wl.flush()
        ev_gemm = _timed(wl.gemm_only, stream)
        wl.flush()
        ev_quant = _timed(wl.quant_only, stream)
        dec = []
        for d in wl.decode:
            wl.flush()
            dec.append(_timed(d["graph"].replay, stream))
        wl.flush()
        ev_moe = _timed(wl.moe, stream)
        m16 = []
        for c in wl.moe16:
            wl.flush()
            m16.append(_timed(c["graph"].replay, stream))
        if record is not None:
            record.append((ev_pre, ev_gemm, dec, ev_moe, ev_quant, m16))

    for _ in range(args.warmup):
        step(None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    recs = []
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(recs)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        hbm, bf16, bf16_sus, peak_src = _peaks()
        configs = None if args.no_sweep else sweep_configs(wl, nv, dev, hbm, bf16 * FP4_OVER_BF16)
    if world > 1:
        torch.distributed.barrier()
    # device times
    ms = lambda ev: ev[0].elapsed_time(ev[1])  # noqa: E731
    pre_ms = [ms(r[0]) for r in recs]
    gemm_ms = [ms(r[1]) for r in recs]
    moe_ms = [ms(r[3]) for r in recs]
    dec_ms = [[ms(e) for e in r[2]] for r in recs]
    m16_ms = [[ms(e) for e in r[5]] for r in recs]
    step_ms = [p + g + sum(d) + m + sum(q) for p, g, d, m, q in zip(pre_ms, gemm_ms, dec_ms, moe_ms, m16_ms)]
    t_pre = statistics.median(pre_ms) * 1e-3
    t_gemm = statistics.median(gemm_ms) * 1e-3
    t_moe = statistics.median(moe_ms) * 1e-3
    t_quant = statistics.median([ms(r[4]) for r in recs]) * 1e-3
    per_step = sum(step_ms) / len(step_ms)
    t_pre, per_step = max_over_ranks([t_pre, per_step], world, dev)
    hbm, bf16, bf16_sus, peak_src = _peaks()
    fp4_peak = bf16 * FP4_OVER_BF16
    decode = {}
    for i, d in enumerate(wl.decode):
        t = statistics.median([x[i] for x in dec_ms]) * 1e-3 / d["ncopy"]
        decode[f"T{d['T']}_{d['N']}x{d['K']}"] = {
            "us": round(t * 1e6, 3), "gbs": round(d["bytes"] / t / 1e9, 1),
            "frac_hbm": round(d["bytes"] / t / 1e9 / hbm, 4)}
    moe16 = {}
    for i, c in enumerate(wl.moe16):
        t = statistics.median([x[i] for x in m16_ms]) * 1e-3 / len(wl.moe16_banks)
        moe16[f"T{c['T']}"] = {"us": round(t * 1e6, 2), "experts": c["experts"], "gbs": round(c["bytes"] / t / 1e9, 1),
                               "frac_hbm": round(c["bytes"] / t / 1e9 / hbm, 4)}
    head_key = f"T1_{synthdata.DECODE_SHAPES[0][0]}x{synthdata.DECODE_SHAPES[0][1]}"
    head = decode[head_key]
    head_bytes = next(d["bytes"] for d in wl.decode if d["T"] == 1 and (d["N"], d["K"]) == synthdata.DECODE_SHAPES[0])
    value = job_throughput(world, wl.pre_flops, t_pre) / 1e12
    gemm_tflops = wl.pre_flops / t_gemm / 1e12
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(per_step, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, ue4m3 block scales) -> fp32 accumulate",
        "data": "synthetic (seeded N(0,1) activations with 1% outlier channels x20, N(0,0.02) weights)",
        "config": {"workload": "fused qkv W4A4 prefill M=8192 N=5120+1024+1024 K=5120 (quant + GEMM)",
                   "decode": "W4A16 T=1..16 on 8704x5120 and 5120x4352, cold weights in CUDA graphs",
                   "moe": "W4A4 MoE E=128 top8 H=2048 I=768 T=4096",
                   "moe_w4a16": (f"W4A16 MoE E=128 top8 H=2048 I=768 T=1, 4, 16; per call of a CUDA graph of "
                                 f"{MOE16_BANKS} calls on distinct expert banks; bytes: the touched experts' weights"),
                   "l2": "flushed before every stage, outside the timed events: a 256 MiB write, then a 256 MiB read so the write's dirty lines drain before the stage",
                   "parallelism": f"replicas x{world}"},
        "prefill": {"ms": round(t_pre * 1e3, 4), "tflops": round(wl.pre_flops / t_pre / 1e12, 1),
                    "frac_fp4_peak": round(wl.pre_flops / t_pre / 1e12 / fp4_peak, 4)},
        "gemm_w4a4": {"ms": round(t_gemm * 1e3, 4), "tflops": round(gemm_tflops, 1),
                      "frac_fp4_peak": round(gemm_tflops / fp4_peak, 4)},
        "quant_act": {"us": round(t_quant * 1e6, 2), "gbs": round(wl.quant_bytes / t_quant / 1e9, 1),
                      "frac_hbm": round(wl.quant_bytes / t_quant / 1e9 / hbm, 4)},
        "decode": decode,
        "moe": {"ms": round(t_moe * 1e3, 4), "tflops": round(wl.moe_flops / t_moe / 1e12, 1),
                "frac_fp4_peak": round(wl.moe_flops / t_moe / 1e12 / fp4_peak, 4),
                # the layer's roofline time is the larger of its FP4 and HBM times
                "bytes": wl.moe_bytes,
                "roofline_us": round(max(wl.moe_flops / (fp4_peak * 1e12), wl.moe_bytes / (hbm * 1e9)) * 1e6, 1),
                "roofline_bound": "hbm" if wl.moe_bytes / (hbm * 1e9) > wl.moe_flops / (fp4_peak * 1e12) else "tensor",
                "frac_roofline": round(max(wl.moe_flops / (fp4_peak * 1e12), wl.moe_bytes / (hbm * 1e9)) / t_moe, 4)},
        "moe_w4a16": moe16,
        # every workload shape, timed after the step (see sweep_configs)
        "configs": configs,
        # the dominant kernel of the step (most of its device time, by the ncu
        # launch list of this command) is the decode GEMM; its roofline is
        # given for the headline decode call, T = 1 on 8704 x 5120, and per
        # instantiation below
        "roofline_decode_kernels": _decode_kernel_rooflines(wl, decode, hbm),
        "roofline": {"kernel": "gemv_ring_kernel<0, 2> (W4A16 decode, T=1, 8704x5120)", "bound": "hbm",
                     "achieved": round(head["gbs"], 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(head["gbs"] / hbm, 4),
                     "peak_source": f"{peak_src} copy bandwidth",
                     "algorithmic_bytes_per_launch": head_bytes, "launch_us": round(head["us"], 3),
                     "traffic": _profile_traffic("gemv_w4a16_T1_8704x5120.md")},
        "roofline_gemm": {"kernel": "gemm_pair_kernel (W4A4, M=8192, CTA pairs)", "bound": "tensor",
                          "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                          "frac": round(gemm_tflops / fp4_peak, 4),
                          "peak_source": f"{peak_src} bf16 burst {bf16} TFLOP/s x {FP4_OVER_BF16:g} (nominal FP4:BF16)",
                          "algorithmic_bytes": wl.pre_bytes,
                          "traffic": _profile_traffic("gemm_w4a4_M8192_N7168_K5120.md")},
        "gpu_launches": wl.launches_per_step() * args.steps,
        "wall_s_timed_region": round(wall, 3),
    }
    clk = clocks.summary()
    result["clocks"] = {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"]}
    # end to end through the public API: pinned host input -> device -> quant + GEMM -> host output
    result["e2e"] = e2e_prefill(wl, nv, dev, args)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def e2e_prefill(wl, nv, dev, args):
    """Prefill end to end through the public API, as a serving loop runs it:
    every step copies its activations in from pinned host memory, quantises
    them, runs the W4A4 GEMM and copies the bf16 result back to pinned host
    memory.  Copy-in, compute and copy-out run on three streams with two sets
    of device buffers, so step i+1's upload and step i-1's download overlap
    step i's compute; events keep each buffer from being reused before the
    step that reads it is done.  The timed region spans all steps, from the
    first upload to the last download."""
    M, N, K = PREFILL_M, wl.pre_W.N, wl.pre_W.K
    steps = max(args.steps, 1)
    x_host = wl.pre_x.cpu().pin_memory()
    out_host = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
    x_dev = [torch.empty_like(wl.pre_x) for _ in range(2)]
    out_dev = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        comp_done = [None] * n
        out_done = [None] * n
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # x_dev[b] has been quantised
                x_dev[b].copy_(x_host, non_blocking=True)
                h2d = torch.cuda.Event()
                h2d.record(s_in)
            with torch.cuda.stream(s_comp):
                s_comp.wait_event(h2d)
                if i >= 2:
                    s_comp.wait_event(out_done[i - 2])  # out_dev[b] has been copied out
                nv.nvfp4_quantize_act(x_dev[b], wl.pre_g, wl.pre_codes, wl.pre_sf)
                nv.nvfp4_linear_w4a4(wl.pre_codes, wl.pre_sf, wl.pre_W.codes, wl.pre_W.scales, wl.pre_alpha, N, K,
                                     out=out_dev[b])
                comp_done[i] = torch.cuda.Event()
                comp_done[i].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                out_host.copy_(out_dev[b], non_blocking=True)
                out_done[i] = torch.cuda.Event()
                out_done[i].record(s_out)
        return out_done[-1]

    run(max(args.warmup, 3)).synchronize()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    last = run(steps)
    s_out.wait_event(last)
    b.record(s_out)
    b.synchronize()
    t = a.elapsed_time(b) * 1e-3 / steps
    return {"value": round(wl.pre_flops / t / 1e12, 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
            "overlap": "copy-in / compute / copy-out on three streams, two buffer sets; time over all steps"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def _oracle_prefill_setup(rows):
    import oracle
    case = synthdata.prefill_case(rows, seed=0)
    wc, ws, g_w, _ = oracle.quantize_weight_parts(case.w_parts)
    g_a = oracle.global_scale(case.x_calib)
    return oracle, case, wc, ws, g_w, g_a


def cpu_baseline(seconds: float):
    """The oracle (as it stands) on a bounded sample of the prefill: quantise
    `rows` activation rows and run the W4A4 GEMM against the full fused weight."""
    ora, case, wc, ws, g_w, g_a = _oracle_prefill_setup(64)
    N, K = case.N, case.K
    threads = ora.threads()
    t0 = time.perf_counter()
    ac, asf = ora.quantize(case.x, g_a)
    ora.linear_w4a4(ac, asf, 64, wc, ws, N, K, ora.alpha_w4a4(g_a, g_w))
    t1 = time.perf_counter() - t0
    rows = int(max(64, min(PREFILL_M, 64 * seconds / max(t1, 1e-3))))
    rows = (rows // 64) * 64
    ora2, case2, wc2, ws2, g_w2, g_a2 = _oracle_prefill_setup(rows)
    t0 = time.perf_counter()
    ac, asf = ora2.quantize(case2.x, g_a2)
    ora2.linear_w4a4(ac, asf, rows, wc2, ws2, N, K, ora2.alpha_w4a4(g_a2, g_w2))
    t = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {PREFILL_M} prefill rows (quantise + W4A4 against the full 7168x5120 weight), "
                      f"{t:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = oracle.threads()
    ora, case, wc, ws, g_w, g_a = _oracle_prefill_setup(64)
    N, K = case.N, case.K
    # size the per-step sample so the whole run stays within a few minutes
    t0 = time.perf_counter()
    ac, asf = ora.quantize(case.x, g_a)
    ora.linear_w4a4(ac, asf, 64, wc, ws, N, K, ora.alpha_w4a4(g_a, g_w))
    t64 = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    rows = int(max(16, min(PREFILL_M, 64 * budget / max(t64, 1e-3))) // 16 * 16)
    case = synthdata.prefill_case(rows, seed=0)
    alpha = ora.alpha_w4a4(g_a, g_w)

    def step():
        a, s = ora.quantize(case.x, g_a)
        ora.linear_w4a4(a, s, rows, wc, ws, N, K, alpha)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = (time.perf_counter() - t0) / args.steps
    flops = 2.0 * rows * N * K
    v = flops / t / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32 (CPU oracle, IEEE)", "data": "synthetic",
        "config": {"workload": "fused qkv W4A4 prefill M=8192 N=5120+1024+1024 K=5120 (quant + GEMM)",
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(v, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {PREFILL_M} prefill rows per step"},
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_profile(stage: str, reps: int):
    """One stage of the path launched `reps` times, without graphs or timing,
    on inputs larger than the L2: the small case that the ncu summaries under
    profiles/ are captured on."""
    import nvfp4_block_scaled_act_gb300 as nv
    from nvfp4_block_scaled_act_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if stage in ("gemm", "quant"):
        pc = synthdata.prefill_case(PREFILL_M, seed=0, device=dev)
        W = nv.quantize_weight(pc.w_parts)
        g = nv.nvfp4_compute_global(pc.x_calib)
        alpha = nv.nvfp4_make_alpha(g, W.g)
        codes, sf = nv.nvfp4_quantize_act(pc.x, g)
        out = torch.empty(PREFILL_M, W.N, dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            if stage == "quant":
                nv.nvfp4_quantize_act(pc.x, g, codes, sf)
            else:
                nv.nvfp4_linear_w4a4(codes, sf, W.codes, W.scales, alpha, W.N, W.K, out=out)
    elif stage == "gemv":
        N, K = synthdata.DECODE_SHAPES[0]
        d = synthdata.decode_case(1, N, K, seed=1, device=dev)
        W = nv.quantize_weight(d.w_parts)
        alpha = nv.nvfp4_make_alpha(None, W.g)
        copies = [(W.codes, W.scales)] + [(W.codes.clone(), W.scales.clone()) for _ in range(7)]  # 8 x 25 MB
        out = torch.empty(1, N, dtype=torch.bfloat16, device=dev)
        for i in range(reps):
            c, sc = copies[i % len(copies)]
            nv.nvfp4_linear_w4a16(d.x, c, sc, alpha, N, K, out=out)
    elif stage == "moe":
        cfg = synthdata.MOE_SMALL
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        mc = synthdata.moe_case(MOE_T, E, H, I, topk, cfg["skewed"], seed=0, device=dev)
        Wm = nv.quantize_moe_weights(lambda e: mc.w13(e), lambda e: mc.w2(e), E, H, I, dev)
        g1 = nv.nvfp4_compute_global(mc.x_calib)
        a13 = nv.nvfp4_make_alpha(g1, Wm.g13)
        g2, _ = nv.nvfp4_moe_calibrate(mc.x_calib, g1, Wm.w13_codes, Wm.w13_sf, a13, E, I)
        a2 = nv.nvfp4_make_alpha(g2, Wm.g2)
        out = torch.empty(MOE_T, H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_moe_workspace(MOE_T, H, I, E, topk), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            nv.nvfp4_moe_w4a4(mc.x, mc.topk_ids, mc.topk_w, g1, Wm.w13_codes, Wm.w13_sf, a13, g2, Wm.w2_codes,
                              Wm.w2_sf, a2, E, I, out=out, workspace=ws)
    elif stage == "moe_large":
        cfg = synthdata.MOE_LARGE
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        T = 8192
        mc = synthdata.moe_case(T, E, H, I, topk, cfg["skewed"], seed=0, device=dev)
        Wm = nv.quantize_moe_weights(lambda e: mc.w13(e), lambda e: mc.w2(e), E, H, I, dev)
        g1 = nv.nvfp4_compute_global(mc.x_calib)
        a13 = nv.nvfp4_make_alpha(g1, Wm.g13)
        g2, _ = nv.nvfp4_moe_calibrate(mc.x_calib, g1, Wm.w13_codes, Wm.w13_sf, a13, E, I)
        a2 = nv.nvfp4_make_alpha(g2, Wm.g2)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_moe_workspace(T, H, I, E, topk), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            nv.nvfp4_moe_w4a4(mc.x, mc.topk_ids, mc.topk_w, g1, Wm.w13_codes, Wm.w13_sf, a13, g2, Wm.w2_codes,
                              Wm.w2_sf, a2, E, I, out=out, workspace=ws)
    elif stage == "moe16":
        cfg = synthdata.MOE_SMALL
        E, H, I, topk = cfg["E"], cfg["H"], cfg["I"], cfg["topk"]
        mc = synthdata.moe_case(4, E, H, I, topk, cfg["skewed"], seed=4, device=dev)
        Wm = nv.quantize_moe_weights(lambda e: mc.w13(e), lambda e: mc.w2(e), E, H, I, dev)
        a13 = nv.nvfp4_make_alpha(None, Wm.g13)
        a2 = nv.nvfp4_make_alpha(None, Wm.g2)
        out = torch.empty(4, H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(nv.nvfp4_moe_w4a16_workspace(4, H, I, E, topk), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            nv.nvfp4_moe_w4a16(mc.x, mc.topk_ids, mc.topk_w, Wm.w13_codes, Wm.w13_sf, a13, Wm.w2_codes, Wm.w2_sf,
                               a2, E, I, out=out, workspace=ws)
    else:
        raise SystemExit(f"unknown stage {stage}")
    torch.cuda.synchronize()
    print(json.dumps({"profile": stage, "reps": reps, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-config sweep after the timed steps")
    ap.add_argument("--profile", choices=["gemm", "quant", "gemv", "moe", "moe_large", "moe16"],
                    help="launch one stage a few times on a small case (for ncu), print nothing else")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args()
    world, rank, local = _dist()
    if args.profile:
        run_profile(args.profile, args.reps)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
