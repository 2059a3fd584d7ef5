"""Benchmark of the fused attention forward on GB300 (one JSON line on stdout).

A step is one call of the fused forward over one batch of the headline workload
(B=2, H=32, N=4096, d=128, non-causal, bf16 inputs from the seeded generator), inputs resident
in HBM.  ``value`` is whole-job TFLOPS (4*B*H*N^2*d per step, summed over ranks, over the max
rank time).  Timing: W untimed warm-up steps, then K steps timed with CUDA events on the
launching stream, an L2 flush (a 256 MiB write) before each step outside the events, barrier and
synchronize on both sides.  Extra keys: ``e2e`` (the same metric through the public API with
pinned host buffers and every step's host<->device copies inside the timed region, steps
pipelined over two device buffers; the serial loop beside it), ``roofline`` (the
kernel against the measured bf16 tensor peak), ``cpu_baseline`` (the float64 oracle on a bounded
sample), ``unfused`` (the three-kernel comparison path), ``configs`` (the fused forward on each
of the five parity configurations: TFLOPS, achieved HBM GB/s on the algorithmic bytes and both
roofline fractions), the grouped-query, split-KV, FP8, backward and packed-batch extras, and
``clocks``.

``--impl reference`` times the float64 CPU oracle (the only reference this method has) on the
host cores instead, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gen import configs  # noqa: E402
from io_aware_attention_attn_gb300 import accounting as acc  # noqa: E402

METRIC = "fused attention fwd TFLOPS at d=128 N=4096; % of BF16 tensor peak"
L2_FLUSH_BYTES = 256 << 20


# the files that make up the fused forward kernel (every bf16 forward runs on it): a profile
# taken on other contents is stale
KERNEL_SOURCES = {
    "attn_fwd_2sm_kernel": ("attn_fwd_2sm_kernel.cuh", "attn_params.h", "sm103_ptx.cuh",
                            "attn_fwd_2sm.cu"),
}
FUSED_SOURCES = KERNEL_SOURCES["attn_fwd_2sm_kernel"]


def kernel_for(w) -> str:
    """The forward kernel the library runs for a workload (CTA pairs for every bf16 forward)."""
    return "attn_fwd_2sm_kernel"


def _code_only(text: str) -> str:
    """Source text without comments and with whitespace collapsed (a profile stays valid across
    comment edits)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def sources_digest(files=FUSED_SOURCES) -> str:
    """Digest of the kernel's code (comments and whitespace excluded)."""
    h = hashlib.sha256()
    for f in files:
        path = os.path.join(ROOT, "io_aware_attention_attn_gb300", "csrc", f)
        h.update(_code_only(open(path, encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        d["_source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "_source": "fallback"}


def _profile_lookup(pattern: str, digest: str):
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for m in re.finditer(pattern + r":\s*([\d.]+)\s+sources:\s*(\w+)", open(f).read()):
            if m.group(2) == digest:
                return m.group(1)
    return None


def profiled_traffic(kernel_tag: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current sources."""
    v = _profile_lookup(r"traffic_bytes_per_launch\[" + re.escape(kernel_tag) + r"\]",
                        sources_digest())
    return int(v) if v is not None else None


def profiled_tensor_pipe(w):
    """ncu sm__pipe_tensor_cycles_active (percent of peak) of the kernel that serves workload
    ``w``, from a committed single-launch summary taken on that kernel's current sources."""
    kern = kernel_for(w)
    v = _profile_lookup(r"tensor_pipe_active\[" + re.escape(kern) + "@" + re.escape(w.name) +
                        r"\]", sources_digest(KERNEL_SOURCES[kern]))
    return float(v) if v is not None else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.out.flush()
        rows = [r.split(", ") for r in open(self.out.name).read().strip().splitlines() if r]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest of every rank's ``value`` (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def blas_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        blas = [i["num_threads"] for i in info if i.get("user_api") == "blas"]
        if blas:
            return int(max(blas))
    except Exception:
        pass
    return None


def cpu_cores() -> int:
    """Threads the oracle's float64 matmuls use (the BLAS pool), else the host's core count."""
    return blas_threads() or os.cpu_count() or 1


def cpu_info() -> dict:
    return {"cores": cpu_cores(), "host_cpu_count": os.cpu_count(),
            "blas_threads": blas_threads()}


def _head_slices(w, q, k, v):
    """(q, k, v) of each attention problem of the workload, head-major from the first head:
    dense [B, H, N, d] gives one per (b, h); packed [H, T, d] one per (h, sequence)."""
    if not w.varlen:
        for i in range(w.B * w.H):
            b, h = divmod(i, w.H)
            yield q[b, h], k[b, h], v[b, h]
    else:
        cu = w.cu_seqlens()
        for h in range(w.H):
            for s_ in range(len(cu) - 1):
                a, e = int(cu[s_]), int(cu[s_ + 1])
                if e > a:
                    yield q[h, a:e], k[h, a:e], v[h, a:e]


def oracle_sample(w, q, k, v, target_s: float, max_rows: int | None = None):
    """Time the float64 oracle on query rows of the workload (problem by problem from the first
    head) until about ``target_s`` seconds have passed (at least one block of rows); returns
    (TFLOPS, rows, seconds)."""
    from oracle import attention as orc
    rows_done, flops, t_total = 0, 0.0, 0.0
    step = 128
    limit = max_rows or w.H * w.total_tokens()
    problems = _head_slices(w, q, k, v)
    cur, r0 = None, 0
    while rows_done == 0 or (t_total < target_s and rows_done < limit):  # at least one block
        if cur is None or r0 >= cur[0].shape[0]:
            try:
                cur, r0 = next(problems), 0
            except StopIteration:
                break
        qq, kk, vv = cur
        L = qq.shape[0]
        rows = np.arange(r0, min(L, r0 + step))
        t0 = time.perf_counter()
        orc.attention_head_rows(qq, kk, vv, rows, w.causal, w.scale)
        t_total += time.perf_counter() - t0
        vis = [(int(r) + 1) if w.causal else L for r in rows]
        flops += sum(4.0 * x * w.d for x in vis)
        rows_done += len(rows)
        r0 += len(rows)
        step = min(step * 2, 1024)
    return flops / t_total / 1e12, rows_done, t_total


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    q, k, v, _ = w.make()
    cores = cpu_info()
    per_step = max(1.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(w, q, k, v, per_step)
    vals, times, rows = [], [], 0
    for _ in range(args.steps):
        tf, r, t = oracle_sample(w, q, k, v, per_step)
        vals.append(tf)
        times.append(t)
        rows += r
    value = len(vals) / sum(1.0 / x for x in vals)  # flops-weighted mean of equal-time steps
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded splitmix64/Box-Muller, bf16-rounded)",
        "config": {**w.describe(), "l2": "n/a (host)"},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "TFLOPS", **cores, "kind": "oracle",
                         "sample": f"float64 oracle, {rows} query rows (problem by problem "
                                   f"from the first head) of {w.name} over {args.steps} steps"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w, rank, world, dist):
    import torch
    from io_aware_attention_attn_gb300 import attn, build
    build.build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    attn.lib()
    q_np, k_np, v_np, cu_np = w.make()

    def to_dev(x):
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = to_dev(q_np), to_dev(k_np), to_dev(v_np)
    cu = torch.from_numpy(cu_np).to(dev) if w.varlen else None
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    lengths = [int(x) for x in np.diff(cu_np)] if w.varlen else [w.N] * w.B
    flops = acc.attention_flops(w.H, lengths, w.d, w.causal)

    def step():
        attn.attn_fwd(q, k, v, cu_seqlens=cu, causal=w.causal, scale=w.scale, out=o, lse=lse,
                      stream=stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    barrier()
    clock_info = clocks.stop()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms, one kernel launch each
    total_ms = max_over_ranks(sum(per), dist, dev)
    value = flops * args.steps * world / (total_ms * 1e-3) / 1e12
    if attn.last_device_error() != 0:
        raise RuntimeError("device-side pipeline wait timed out during the bench")

    peaks = measured_peaks()
    kernel_ms = statistics.mean(per)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic("attn_fwd_kernel") if w is configs.WORKLOADS[
                    configs.HEADLINE] else None,
                "peak_source": f"{peaks['_source']} bf16 burst (cuBLAS)",
                "tensor_pipe_active": profiled_tensor_pipe(w),
                "kernel": kernel_for(w),
                "algorithmic_bytes": acc.attention_ideal_bytes(w.H, w.total_tokens(), w.d)}

    # ---- end to end through the public API: pinned host -> device, forward, device -> host.
    # Every step copies its own Q, K, V in and its O and LSE out; steps are pipelined over two
    # device buffers (inputs of step i+1 copied in on one stream and outputs of step i-1 copied
    # out on another while step i computes), as a data loader would.  The plain serial loop is
    # reported beside it.
    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(args.steps, 50))
        h_in = [[torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
                 for x in (q_np, k_np, v_np)] for _ in range(2)]
        if w.varlen:
            for hb in h_in:
                hb.append(torch.from_numpy(cu_np).pin_memory())
        h_out = [(torch.empty(o.shape, dtype=torch.bfloat16).pin_memory(),
                  torch.empty(lse.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
        d_in = [[torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)] +
                ([torch.empty_like(cu)] if w.varlen else []) for _ in range(2)]
        d_out = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
        s_h2d = torch.cuda.Stream(dev)
        s_d2h = torch.cuda.Stream(dev)

        def run_pipelined(n):
            ev_in = [torch.cuda.Event() for _ in range(2)]
            ev_done = [torch.cuda.Event() for _ in range(2)]
            ev_out = [torch.cuda.Event() for _ in range(2)]
            used = [False, False]

            def h2d(i):
                b = i % 2
                with torch.cuda.stream(s_h2d):
                    if used[b]:
                        s_h2d.wait_event(ev_done[b])  # the buffer's previous step has computed
                    for dst, src in zip(d_in[b], h_in[b]):
                        dst.copy_(src, non_blocking=True)
                    ev_in[b].record(s_h2d)

            h2d(0)
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    h2d(i + 1)
                stream.wait_event(ev_in[b])
                if used[b]:
                    stream.wait_event(ev_out[b])  # the buffer's previous outputs left the device
                attn.attn_fwd(d_in[b][0], d_in[b][1], d_in[b][2],
                              cu_seqlens=d_in[b][3] if w.varlen else None, causal=w.causal,
                              scale=w.scale, out=d_out[b][0], lse=d_out[b][1], stream=stream)
                ev_done[b].record(stream)
                used[b] = True
                with torch.cuda.stream(s_d2h):
                    s_d2h.wait_event(ev_done[b])
                    h_out[b][0].copy_(d_out[b][0], non_blocking=True)
                    h_out[b][1].copy_(d_out[b][1], non_blocking=True)
                    ev_out[b].record(s_d2h)
            stream.wait_stream(s_h2d)
            stream.wait_stream(s_d2h)

        def run_serial(n):
            for _ in range(n):
                dq_ = h_in[0][0].to(dev, non_blocking=True)
                dk_ = h_in[0][1].to(dev, non_blocking=True)
                dv_ = h_in[0][2].to(dev, non_blocking=True)
                dc_ = h_in[0][3].to(dev, non_blocking=True) if w.varlen else None
                oo, ll = attn.attn_fwd(dq_, dk_, dv_, cu_seqlens=dc_, causal=w.causal,
                                       scale=w.scale)
                h_out[0][0].copy_(oo, non_blocking=True)
                h_out[0][1].copy_(ll, non_blocking=True)

        def timed(fn):
            fn(3)
            barrier()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(n_e2e)
            e1.record(stream)
            barrier()
            return max_over_ranks(e0.elapsed_time(e1), dist, dev)

        e_ms = timed(run_pipelined)
        s_ms = timed(run_serial)
        if not np.array_equal(h_out[(n_e2e - 1) % 2][0].view(torch.int16).numpy(),
                              o.view(torch.int16).cpu().numpy()):
            raise RuntimeError("end-to-end output differs from the device-resident run")
        e2e = {"value": flops * n_e2e * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
               "h2d_bytes_per_step": 3 * q.numel() * 2 + (cu.numel() * 4 if w.varlen else 0),
               "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4, "steps": n_e2e,
               "pipelined": "two device buffers; H2D of step i+1 and D2H of step i-1 overlap step i",
               "serial_value": flops * n_e2e * world / (s_ms * 1e-3) / 1e12}
        del h_in, h_out, d_in, d_out

    # ---- unfused three-kernel comparison path (memory wall)
    unfused = None
    if not args.no_unfused and not w.varlen:  # the comparison path takes dense batches only
        try:
            need = attn.unfused_workspace_bytes(w.B, w.H, w.N, w.d)
            ws = torch.empty(need, dtype=torch.uint8, device=dev)
            ou = torch.empty_like(o)
            lu = torch.empty_like(lse)
            for _ in range(2):
                attn.attn_fwd_unfused(q, k, v, causal=w.causal, scale=w.scale, workspace=ws,
                                      out=ou, lse=lu)
            barrier()
            n_u = 5
            u0 = torch.cuda.Event(enable_timing=True)
            u1 = torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            for _ in range(n_u):
                attn.attn_fwd_unfused(q, k, v, causal=w.causal, scale=w.scale, workspace=ws,
                                      out=ou, lse=lu)
            u1.record(stream)
            barrier()
            u_ms = u0.elapsed_time(u1) / n_u
            ub = acc.unfused_bytes(w.B, w.H, w.N, w.d)
            unfused = {"ms_per_step": u_ms, "tflops": flops / (u_ms * 1e-3) / 1e12,
                       "algorithmic_bytes": ub, "gbs": ub / (u_ms * 1e-3) / 1e9,
                       "hbm_frac": ub / (u_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                       "fused_speedup": u_ms / kernel_ms, "launches_per_step": 3}
            del ws
        except Exception as e:  # reported, never silently replaced
            unfused = {"error": str(e)[:200]}

    # ---- grouped-query variant of the same shape (32 query heads sharing 8 K/V heads)
    gqa = None
    if not args.no_extras:
        g = configs.GQA
        gq, gk, gv, _ = g.make()
        gq, gk, gv = to_dev(gq), to_dev(gk), to_dev(gv)
        go = torch.empty_like(gq)
        gl = torch.empty(gq.shape[:-1], dtype=torch.float32, device=dev)
        for _ in range(3):
            attn.attn_fwd(gq, gk, gv, causal=g.causal, scale=g.scale, out=go, lse=gl)
        barrier()
        n_g = 50
        g_ms = []
        for _ in range(n_g):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.attn_fwd(gq, gk, gv, causal=g.causal, scale=g.scale, out=go, lse=gl)
            e1.record(stream)
            g_ms.append((e0, e1))
        barrier()
        g_ms = statistics.mean(a.elapsed_time(b) for a, b in g_ms)
        g_flops = acc.attention_flops(g.H, [g.N] * g.B, g.d, g.causal)
        gqa = {"workload": g.name, "ms": g_ms, "tflops": g_flops / (g_ms * 1e-3) / 1e12,
               "frac_of_peak": g_flops / (g_ms * 1e-3) / 1e12 / peak,
               "kv_bytes_saved": 2 * (g.H - g.kv_heads) * g.B * g.N * g.d * 2}
        del gq, gk, gv, go, gl

    # ---- split-KV on a few-heads, long-sequence shape (32 query pairs, 64 of the 152 SMs in one
    # slice): the library's slice count against one slice (the plain fused kernel)
    splitkv = None
    if not args.no_extras:
        sw = configs.SPLITKV
        sq, sk, sv, _ = sw.make()
        sq, sk, sv = to_dev(sq), to_dev(sk), to_dev(sv)
        so = torch.empty_like(sq)
        sl = torch.empty(sq.shape[:-1], dtype=torch.float32, device=dev)
        need = attn.splitkv_workspace_bytes(sw.B, sw.H, sw.N, sw.d, 0)
        sws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        s_flops = acc.attention_flops(sw.H, [sw.N] * sw.B, sw.d, sw.causal)

        def time_split(n_splits, n=50):
            for _ in range(3):
                attn.attn_fwd_splitkv(sq, sk, sv, causal=sw.causal, scale=sw.scale,
                                      num_splits=n_splits, workspace=sws, out=so, lse=sl)
            barrier()
            evs = []
            for _ in range(n):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                attn.attn_fwd_splitkv(sq, sk, sv, causal=sw.causal, scale=sw.scale,
                                      num_splits=n_splits, workspace=sws, out=so, lse=sl)
                e1.record(stream)
                evs.append((e0, e1))
            barrier()
            return statistics.mean(a.elapsed_time(b) for a, b in evs)

        ms_auto = time_split(0)
        ms_one = time_split(1)
        chosen = attn.splitkv_slices(sw.B, sw.H, sw.N, sw.d, 0)
        splitkv = {"workload": sw.name, "splits": chosen, "ms": ms_auto,
                   "tflops": s_flops / (ms_auto * 1e-3) / 1e12, "ms_one_slice": ms_one,
                   "tflops_one_slice": s_flops / (ms_one * 1e-3) / 1e12,
                   "speedup": ms_one / ms_auto, "launches_per_step": 2 if chosen > 1 else 1}
        del sq, sk, sv, so, sl, sws

    # ---- FP8 (E4M3) forward on the same shape: quantize once, then time the FP8 kernel; the
    # quantization of Q, K and V (three launches) is timed separately
    fp8 = None
    if not args.no_extras and w.d == 128 and not w.varlen:
        q8, sq = attn.quantize_fp8(q)
        k8, sk = attn.quantize_fp8(k)
        vt8, sv = attn.quantize_fp8(v, transpose=True)
        fo8 = torch.empty_like(o)
        fl8 = torch.empty_like(lse)

        def fp8_step():
            attn.attn_fwd_fp8(q8, sq, k8, sk, vt8, sv, causal=w.causal, scale=w.scale, out=fo8,
                              lse=fl8)

        for _ in range(3):
            fp8_step()
        barrier()
        evs = []
        for _ in range(50):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fp8_step()
            e1.record(stream)
            evs.append((e0, e1))
        barrier()
        f_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        evs = []
        for _ in range(10):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.quantize_fp8(q)
            attn.quantize_fp8(k)
            attn.quantize_fp8(v, transpose=True)
            e1.record(stream)
            evs.append((e0, e1))
        barrier()
        qz_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        fp8_peak = float(peaks["bf16_tflops"]) * 2.0
        fp8 = {"workload": w.name, "ms": f_ms, "tflops": flops / (f_ms * 1e-3) / 1e12,
               "frac_of_fp8_peak": flops / (f_ms * 1e-3) / 1e12 / fp8_peak,
               "fp8_peak": fp8_peak,
               "fp8_peak_source": "measured bf16 burst x 2 (nominal dense fp8/bf16 ratio)",
               "speedup_vs_bf16": kernel_ms / f_ms, "quantize_qkv_ms": qz_ms,
               "launches_per_step": 1}
        del q8, k8, vt8, sq, sk, sv, fo8, fl8

    # ---- backward pass on the same shape (non-causal and causal): dQ, dK, dV from the
    # forward's O and LSE and a random upstream gradient
    backward = None
    if not args.no_extras and not w.varlen:
        backward = {}
        dout = to_dev(w.make_dout())
        bws = torch.empty(max(attn.bwd_workspace_bytes(w.B, w.H, w.N, w.d), 1),
                          dtype=torch.uint8, device=dev)
        gq, gk, gv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        for causal in (False, True):
            fo, fl = attn.attn_fwd(q, k, v, causal=causal, scale=w.scale)

            def bwd_step():
                attn.attn_bwd(q, k, v, fo, fl, dout, causal=causal, scale=w.scale, workspace=bws,
                              dq=gq, dk=gk, dv=gv)

            for _ in range(3):
                bwd_step()
            barrier()
            evs = []
            for _ in range(30):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                bwd_step()
                e1.record(stream)
                evs.append((e0, e1))
            barrier()
            b_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
            b_flops = acc.attention_bwd_flops(w.H, [w.N] * w.B, w.d, causal)
            backward["causal" if causal else "non_causal"] = {
                "ms": b_ms, "tflops": b_flops / (b_ms * 1e-3) / 1e12,
                "frac_of_peak": b_flops / (b_ms * 1e-3) / 1e12 / peak,
                "flops_counted": "2.5x forward (5 matmuls); the kernels execute 7",
                "launches_per_step": 2}
            del fo, fl
        backward["workload"] = w.name
        # grouped-query backward on the GQA shape (dK, dV summed over each group of 4)
        gw = configs.GQA
        gq_np, gk_np, gv_np, _ = gw.make()
        gqd, gkd, gvd = to_dev(gq_np), to_dev(gk_np), to_dev(gv_np)
        gdo = to_dev(gw.make_dout())
        fo, fl = attn.attn_fwd(gqd, gkd, gvd, causal=False, scale=gw.scale)
        for _ in range(3):
            attn.attn_bwd(gqd, gkd, gvd, fo, fl, gdo, scale=gw.scale, workspace=bws)
        barrier()
        evs = []
        for _ in range(30):
            flush.zero_()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            attn.attn_bwd(gqd, gkd, gvd, fo, fl, gdo, scale=gw.scale, workspace=bws)
            e1.record(stream)
            evs.append((e0, e1))
        barrier()
        g_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        g_flops = acc.attention_bwd_flops(gw.H, [gw.N] * gw.B, gw.d, False)
        backward["gqa_non_causal"] = {"workload": gw.name, "ms": g_ms,
                                      "tflops": g_flops / (g_ms * 1e-3) / 1e12}
        del dout, bws, gq, gk, gv, gqd, gkd, gvd, gdo, fo, fl

    # ---- packed variable-length batch (16 sequences of U[128, 4096] rows, H=16, d=128, causal):
    # forward and backward through the cu_seqlens entry points
    varlen = None
    if not args.no_extras:
        vw = configs.WORKLOADS[5]
        vq_np, vk_np, vv_np, vcu = vw.make()
        vq, vk, vv = to_dev(vq_np), to_dev(vk_np), to_dev(vv_np)
        vcu_d = torch.from_numpy(vcu).to(dev)
        vdo = to_dev(configs.custom(vw.index, 1, vw.H, vw.total_tokens(), vw.d, True)
                     .make_dout()[0])
        vo, vl = attn.attn_fwd(vq, vk, vv, cu_seqlens=vcu_d, causal=True, scale=vw.scale)
        vws = torch.empty(max(int(attn.lib().attn_bwd_varlen_workspace_bytes(
            vw.n_seqs, vw.H, vw.total_tokens(), vw.d)), 1), dtype=torch.uint8, device=dev)

        def time_it(fn, n=30):
            for _ in range(3):
                fn()
            barrier()
            evs = []
            for _ in range(n):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                evs.append((e0, e1))
            barrier()
            return statistics.mean(a.elapsed_time(b) for a, b in evs)

        f_ms = time_it(lambda: attn.attn_fwd(vq, vk, vv, cu_seqlens=vcu_d, causal=True,
                                             scale=vw.scale, out=vo, lse=vl))
        b_ms = time_it(lambda: attn.attn_bwd(vq, vk, vv, vo, vl, vdo, cu_seqlens=vcu_d,
                                             causal=True, scale=vw.scale, workspace=vws))
        lens = [int(x) for x in np.diff(vcu)]
        vf = acc.attention_flops(vw.H, lens, vw.d, True)
        varlen = {"workload": vw.name, "lengths": lens, "fwd_ms": f_ms,
                  "fwd_tflops": vf / (f_ms * 1e-3) / 1e12, "bwd_ms": b_ms,
                  "bwd_tflops": 2.5 * vf / (b_ms * 1e-3) / 1e12}
        del vq, vk, vv, vo, vl, vdo, vws

    # ---- every named configuration (the five parity configurations) through the fused forward:
    # time, TFLOPS (causal halved), achieved HBM bandwidth on the algorithmic bytes (read Q, K,
    # V once, write O and LSE once) and both roofline fractions; the small-N cases are bound by
    # latency and bandwidth, not by the tensor cores
    per_config = None
    if not args.no_extras:
        per_config = []
        hbm_peak = float(peaks["hbm_gbs"])
        for idx in sorted(configs.WORKLOADS):
            cw = configs.WORKLOADS[idx]
            made = cw.make()
            cq, ck, cv = to_dev(made[0]), to_dev(made[1]), to_dev(made[2])
            cu_np = made[3] if cw.varlen else None
            cu_d = torch.from_numpy(cu_np).to(dev) if cw.varlen else None
            co, cl = attn.attn_fwd(cq, ck, cv, cu_seqlens=cu_d, causal=cw.causal, scale=cw.scale)

            def call():
                attn.attn_fwd(cq, ck, cv, cu_seqlens=cu_d, causal=cw.causal, scale=cw.scale,
                              out=co, lse=cl)
            for _ in range(3):
                call()
            barrier()
            evs = []
            for _ in range(20):
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                call()
                e1.record(stream)
                evs.append((e0, e1))
            barrier()
            c_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
            lens = [int(x) for x in np.diff(cu_np)] if cw.varlen else [cw.N] * cw.B
            c_flops = acc.attention_flops(cw.H, lens, cw.d, cw.causal)
            c_bytes = acc.attention_ideal_bytes(cw.H, sum(lens), cw.d)
            c_tf = c_flops / (c_ms * 1e-3) / 1e12
            c_gbs = c_bytes / (c_ms * 1e-3) / 1e9
            per_config.append({"workload": cw.name, "ms": c_ms, "tflops": c_tf,
                               "tensor_frac": c_tf / peak, "algorithmic_bytes": c_bytes,
                               "gbs": c_gbs, "hbm_frac": c_gbs / hbm_peak,
                               "kernel": kernel_for(cw),
                               "tensor_pipe_active": profiled_tensor_pipe(cw)})
            del cq, ck, cv, co, cl, cu_d

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tf, rows, secs = oracle_sample(w, q_np, k_np, v_np, args.cpu_seconds)
        cpu = {"value": tf, "unit": "TFLOPS", **cpu_info(), "kind": "oracle",
               "sample": f"float64 oracle, {rows} query rows (problem by problem from the "
                         f"first head) of {w.name}, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded splitmix64/Box-Muller, bf16-rounded)",
            "config": {**w.describe(), "l2": "flushed (256 MiB write) before every step",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_bf16_peak": 100.0 * value / world / peak,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "unfused": unfused,
            "gqa": gqa, "splitkv": splitkv, "backward": backward, "fp8": fp8, "varlen": varlen,
            "configs": per_config,
            "clocks": clock_info, "gpu_launches": args.steps,
            "kernel_ms_median": statistics.median(per),
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=configs.HEADLINE)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-unfused", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the grouped-query, split-KV, FP8, backward and packed-batch measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = configs.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist_mod.init_process_group(backend)
        dist = dist_mod
    if args.impl == "reference":
        run_reference(args, w, rank, world)
    else:
        run_ours(args, w, rank, world, dist)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
