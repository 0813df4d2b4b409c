"""Benchmark of the H3 attention step on GB300.

One step = the whole hot path over one batch of synthetic input: fused Q/K
RMSNorm + bf16 boundary + partial RoPE (in place) and dense prefill
attention, both through libh3attn's C ABI.  Default workload: long video
self-attention, B=1, S=32760, H=24, D=128 (the shape the headline attention
throughput is quoted on), inputs drawn by h3inputs (seed 0).

Prints one JSON line (rank 0).  `value` = attention FLOP (4*B*Sq*Sk*Hq*D)
per step / device time per step, inputs resident in HBM (q, k, v: 603 MB,
larger than the 129 MB L2, so no flush is needed between steps).  `e2e` =
the same metric when every step also copies q, k, v from pinned host memory
and reads o back.  `--impl reference` times the CPU oracle on the host
cores instead (bounded row samples of the same workload).

Multi-GPU: one process per GPU (torchrun); each rank runs its own replica of
the workload (independent problems, no data-path collective); a barrier and
a max-over-ranks of the timings are the only communication.
"""
from __future__ import annotations

import argparse
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

METRIC = "attention TFLOP/s & % of GB300 BF16 peak at S=32k,H=24,D=128; QK-norm+RoPE GB/s"
WORKLOAD = "long_video_h24"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(values, ws, device):
    """Element-wise max of this rank's timings over all ranks (the slowest rank
    sets each time); a no-op on one rank.  `device` is where the process
    group's collectives run ("cuda" for NCCL, "cpu" for gloo)."""
    if ws <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(ws, units_per_step, steps, total_ms):
    """Whole-job throughput: every rank processes units_per_step per step (weak
    scaling), and the slowest rank's time counts."""
    return ws * units_per_step * steps / (total_ms * 1e-3)


def _allowed_pairs(wl, kv_len, causal_b):
    """Allowed (query row, key) pairs summed over samples (structured masks)."""
    total = 0
    for b in range(wl.B):
        L = wl.Sk if kv_len is None else max(0, min(wl.Sk, int(kv_len[b])))
        if causal_b is not None and causal_b[b]:
            # rows i < L attend i+1 keys, rows i >= L attend L keys
            m = min(L, wl.Sq)
            total += m * (m + 1) // 2 + (wl.Sq - m) * L
        else:
            total += wl.Sq * L
    return total


def _workload_numbers(wl):
    flops = 4.0 * wl.B * wl.Sq * wl.Sk * wl.Hq * wl.D
    rows_q = wl.B * wl.Sq * wl.Hq
    rows_k = 0 if wl.cross else wl.B * wl.Sk * wl.Hkv
    half = wl.rotary_dim // 2
    norm_bytes = 2.0 * (rows_q + rows_k) * wl.D * 2 + 2.0 * max(wl.Sq, wl.Sk) * half * 4 + 2.0 * wl.D * 4
    return flops, norm_bytes


class ClockSampler:
    """nvidia-smi clock/throttle sampling; only samples stamped inside the
    timed region (host wall-clock window set by window()) are summarised."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 50

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="h3clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    @staticmethod
    def _epoch(stamp: str):
        from datetime import datetime
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.strptime(stamp, fmt).timestamp()
            except ValueError:
                pass
        return None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        return self.summarise(rows)

    def summarise(self, rows):
        """rows: split CSV lines of QUERY; returns the clocks record."""
        inside = [r for r in rows if self.t0 is not None and (t := self._epoch(r[0])) is not None
                  and self.t0 <= t <= self.t1]
        use = inside if inside else rows

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for r in use if (v := num(r[2])) is not None]
        smax = [v for r in use if (v := num(r[3])) is not None]
        power = [v for r in use if (v := num(r[4])) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole sampler run (no sample inside the timed region)",
                "power_w_median": statistics.median(power) if power else None,
                "power_w_max": max(power) if power else None}


def run_gpu(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import h3inputs as gen
    import video_dit_dense_gb300 as h3

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    h3.build()
    h3.load()
    wl = gen.WORKLOADS[args.workload]
    inp = gen.make_inputs(wl, seed=args.seed + rank)
    flops_nominal, norm_bytes = _workload_numbers(wl)
    # algorithmic flops: 4*D*Hq per allowed (row, key) pair; equals the nominal
    # 4*B*Sq*Sk*Hq*D for unmasked workloads
    flops = 4.0 * wl.D * wl.Hq * _allowed_pairs(wl, inp.kv_len, inp.causal_b)
    peaks = _peaks()

    def pinned(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = pinned(inp.q), pinned(inp.k), pinned(inp.v)
    q, k, v = hq.cuda(), hk.cuda(), hv.cuda()
    o = torch.empty_like(q)
    ho = torch.empty(o.shape, dtype=torch.bfloat16).pin_memory()
    wq = wk = cos = sin = None
    if wl.norm_rope:
        wq, wk = torch.from_numpy(inp.wq).cuda(), torch.from_numpy(inp.wk).cuda()
        cos, sin = torch.from_numpy(inp.cos).cuda(), torch.from_numpy(inp.sin).cuda()
    kn = None if wl.cross else k
    wkn = None if wl.cross else wk
    # The device-resident steps read the raw q, k and write the normalised
    # copies (out-of-place norm/RoPE, the same bytes as in place), so every
    # timed step runs the whole path on the same synthetic batch; in place,
    # step k would attend over inputs normalised and rotated k times.
    qa = torch.empty_like(q) if wl.norm_rope else q
    ka = (torch.empty_like(k) if not wl.cross else k) if wl.norm_rope else k
    kan = None if wl.cross else ka
    mask = None
    if inp.kv_len is not None or inp.causal_b is not None:
        mask = h3.Mask(kv_len=None if inp.kv_len is None else torch.from_numpy(inp.kv_len).cuda(),
                       causal_b=None if inp.causal_b is None else torch.from_numpy(inp.causal_b).cuda())
    stream = torch.cuda.current_stream()
    # the split-key tail's workspace (caller-owned; None when the shape does not split)
    wsp = h3.prefill_workspace(q, k, mask) if args.split else None

    def step():
        if wl.norm_rope:
            h3.h3attn_qk_norm_rope_out(q, kn, qa, kan, wq, wkn, cos, sin, wl.rotary_dim, wl.eps, stream)
        h3.h3attn_prefill(qa, ka, v, o, wl.scale, mask, False, stream, workspace=wsp)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    # ---- device-resident timing --------------------------------------------
    for _ in range(args.warmup):
        step()
    barrier()
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    wall0 = time.time()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        if wl.norm_rope:
            h3.h3attn_qk_norm_rope_out(q, kn, qa, kan, wq, wkn, cos, sin, wl.rotary_dim, wl.eps, stream)
        ev[i][1].record(stream)
        h3.h3attn_prefill(qa, ka, v, o, wl.scale, mask, False, stream, workspace=wsp)
        ev[i][2].record(stream)
    t_end.record(stream)
    barrier()
    clocks.window(wall0, time.time())
    clk = clocks.stop()
    st = h3.h3attn_check_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st}: {h3.h3attn_status_string(st)}")
    total_ms = t_start.elapsed_time(t_end)
    norm_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / args.steps
    attn_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / args.steps

    # ---- end to end through the public API, host buffers -------------------
    # Every step copies its q, k, v from pinned host memory and reads its o
    # back.  Two device buffer sets and three streams let the copies of
    # neighbouring steps run on the copy engines while the kernels of this
    # step run: step i's H2D waits until step i-2's kernels are done with the
    # buffer set, its kernels wait for its H2D and for step i-2's D2H of o.
    bufs = [(q, k, v, o)] + [tuple(torch.empty_like(t) for t in (q, k, v, o))]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i, tev=None):
        # tev: timing events around this step's H2D and D2H on their streams
        bq, bk, bv, bo = bufs[i % 2]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_done[i % 2])
            if tev:
                tev[0].record(s_in)
            bq.copy_(hq, non_blocking=True); bk.copy_(hk, non_blocking=True); bv.copy_(hv, non_blocking=True)
            ev_in[i % 2].record(s_in)
            if tev:
                tev[1].record(s_in)
        stream.wait_event(ev_in[i % 2])
        if i >= 2:
            stream.wait_event(ev_out[i % 2])
        if wl.norm_rope:
            h3.h3attn_qk_norm_rope(bq, None if wl.cross else bk, wq, wkn, cos, sin, wl.rotary_dim, wl.eps, stream)
        h3.h3attn_prefill(bq, bk, bv, bo, wl.scale, mask, False, stream, workspace=wsp)
        ev_done[i % 2].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[i % 2])
            if tev:
                tev[2].record(s_out)
            ho.copy_(bo, non_blocking=True)
            ev_out[i % 2].record(s_out)
            if tev:
                tev[3].record(s_out)

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    barrier()
    # the clocks of this region on their own: the copies draw power too
    clocks_e2e = ClockSampler(local)
    clocks_e2e.start()
    barrier()
    wall_e2e = time.time()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    tevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    e0.record(stream)
    s_in.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i, tevs[i])
    stream.wait_stream(s_out)
    e1.record(stream)
    barrier()
    clocks_e2e.window(wall_e2e, time.time())
    clk_e2e = clocks_e2e.stop()
    e2e_ms = e0.elapsed_time(e1)
    h2d_ms = sum(t[0].elapsed_time(t[1]) for t in tevs) / args.steps
    d2h_ms = sum(t[2].elapsed_time(t[3]) for t in tevs) / args.steps

    mod = _time_rmsnorm_modulate(h3, gen, torch, stream, peaks) if args.modulate else None
    wnd = _time_window(h3, gen, torch, stream, peaks) if args.window else None

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], ws, "cuda")
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return

    ms_per_step = total_ms / args.steps
    value = job_throughput(ws, flops, args.steps, total_ms) / 1e12
    attn_tflops = flops / (attn_ms * 1e-3) / 1e12
    norm_gbs = norm_bytes / (norm_ms * 1e-3) / 1e9 if wl.norm_rope else None
    # recorded traffic is for the default workload's launches only
    traffic = _profiled_traffic() if wl.name == WORKLOAD else {}
    attn_kernel = _attn_kernel_name(wl)
    if wsp is not None:
        attn_kernel += " (split-key tail) + split_combine_kernel<%d>" % wl.D
    attn_launches = 2 if wsp is not None else 1
    # the dense bf16 tensor rate at the clock the kernel ran at: 152 SMs x 8192
    # flop (4096 bf16 FMA) per clock per SM x the median SM clock of the timed region
    sm_mhz = (clk or {}).get("sm_mhz")
    clock_peak = 152 * 8192 * sm_mhz * 1e6 / 1e12 if sm_mhz else None
    masks = []
    if inp.kv_len is not None:
        masks.append("key padding kv_len=%s" % list(map(int, inp.kv_len)))
    if inp.causal_b is not None:
        masks.append("causal per sample %s" % list(map(int, inp.causal_b)))
    what = ("QK-norm + RoPE %d/%d then " % (wl.rotary_dim, wl.D) if wl.norm_rope else "") + \
        ("cross-attention" if wl.cross else "self-attention") + (" with " + ", ".join(masks) if masks else " (dense, non-causal)")
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (h3inputs seed %d: N(0,1) bf16 + N(0,0.5) per-head offsets on q/k)" % args.seed,
        "config": {
            "workload": f"{wl.name}: B={wl.B} Sq={wl.Sq} Sk={wl.Sk} Hq={wl.Hq} Hkv={wl.Hkv} D={wl.D}; {what}",
            "flops_per_step": flops,
            "flops_nominal_per_step": flops_nominal,
            "l2": "no flush: inputs larger than L2 (q,k,v %.0f MB > 129 MB)" % (3 * wl.B * wl.Sq * wl.Hq * wl.D * 2 / 1e6),
            "parallelism": f"replicas x{ws} (independent problems per GPU)",
        },
        "clocks": clk,
        "e2e": {
            "how": "per step: H2D of q,k,v from pinned host memory, both kernels, D2H of o; "
                   "two buffer sets, copies of neighbouring steps overlap kernels on separate streams",
            "value": round(job_throughput(ws, flops, args.steps, e2e_ms) / 1e12, 2),
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2),
            "d2h_bytes_per_step": int(ho.numel() * 2),
            "ms_per_step": round(e2e_ms / args.steps, 4),
            # each step's copies on their own streams (they overlap the kernels)
            "h2d_ms_per_step": round(h2d_ms, 4),
            "d2h_ms_per_step": round(d2h_ms, 4),
            "clocks": {key: clk_e2e.get(key) for key in ("sm_mhz", "power_w_median", "power_w_max", "reasons",
                                                         "samples", "window")},
        },
        "gpu_launches": ((1 if wl.norm_rope else 0) + attn_launches) * args.steps,
        "roofline": {
            "kernel": attn_kernel,
            "bound": "tensor",
            "achieved": round(attn_tflops, 2),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(attn_tflops / peaks["bf16_tflops"], 4),
            "frac_of_sustained": round(attn_tflops / peaks["bf16_tflops_sustained"], 4),
            "frac_of_clock_peak": None if clock_peak is None else round(attn_tflops / clock_peak, 4),
            "clock_peak_how": "152 SMs x 8192 bf16 flop/clk x median SM MHz in the timed region",
            "peak_source": peaks["source"] + " burst bf16 (MEASURED_PEAKS.json)",
            "traffic": traffic.get("attn"),
            "ms_per_launch": round(attn_ms, 4),
        },
        "norm_rope": None if not wl.norm_rope else {
            "kernel": "qk_norm_rope_kernel<%d>" % wl.D,
            "bound": "hbm",
            "achieved": round(norm_gbs, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(norm_gbs / peaks["hbm_gbs"], 4),
            "frac_of_8tbs": round(norm_gbs / 8000.0, 4),
            "algorithmic_bytes": int(norm_bytes),
            "traffic": traffic.get("norm"),
            "ms_per_launch": round(norm_ms, 4),
        },
    }
    if mod is not None:
        line["rmsnorm_modulate"] = mod
    if wnd is not None:
        line["window_attention"] = wnd
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def _time_rmsnorm_modulate(h3, gen, torch, stream, peaks, steps=20, warmup=3):
    """The fused RMSNorm -> indexed AdaLN modulation kernel on its hidden-row
    workload (x and y, 201 MB each, are larger than L2: no flush needed)."""
    import numpy as np
    mw = gen.MOD_WORKLOADS["dit_hidden_adaln"]
    mi = gen.make_modulate_inputs(mw.T, mw.C, mw.frames, seed=0)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()
    x, sc, sh = dev(mi.x), dev(mi.scale), dev(mi.shift)
    y = torch.empty_like(x)
    w, idx = torch.from_numpy(mi.w).cuda(), torch.from_numpy(mi.idx).cuda()
    for _ in range(warmup):
        h3.h3attn_rmsnorm_modulate(x, y, w, sc, sh, idx, mw.eps, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        h3.h3attn_rmsnorm_modulate(x, y, w, sc, sh, idx, mw.eps, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    st = h3.h3attn_check_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after rmsnorm_modulate")
    ms = e0.elapsed_time(e1) / steps
    nbytes = 2.0 * mw.T * mw.C * 2 + 2.0 * mw.frames * mw.C * 2 + mw.C * 4 + mw.T * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    # the shape the library's launcher picks (label only)
    w_mod, staged = _mod_shape(mw.C, with_weight=True)
    return {"kernel": f"rmsnorm_modulate_kernel<{w_mod}>" + (" (weight staged in shared memory)" if staged else ""),
            "workload": f"{mw.name}: T={mw.T} C={mw.C} N={mw.frames}",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": int(nbytes),
            "ms_per_launch": round(ms, 4), "launches": steps + warmup,
            "traffic": _profiled_traffic().get("mod")}


def _window_pairs(S, L, frame_tokens, anchor_frames, chunk_frames, radius):
    """Allowed (query row, key) pairs of one sample under the chunked window
    and key padding L: anchor rows see every key; any other row sees the
    anchor keys and the keys of the chunks within the radius of its own."""
    import numpy as np
    af, ct = anchor_frames * frame_tokens, chunk_frames * frame_tokens
    L = max(0, min(L, S))
    i = np.arange(af, S, dtype=np.int64)
    ci = (i - af) // ct
    lo = np.maximum(af + (ci - radius) * ct, af)
    hi = np.minimum(af + (ci + radius + 1) * ct, L)
    return int(min(af, S) * L + len(i) * min(af, L) + np.maximum(hi - lo, 0).sum())


def _time_window(h3, gen, torch, stream, peaks, steps=5, warmup=3):
    """The chunked-window prefill on the packed clip (q, k, v 641 MB each)."""
    ww = gen.WINDOW_WORKLOADS["packed_clip_window"]

    def dev(bits):
        import numpy as np
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    q = dev(gen.normal_bshd(ww.B, ww.S, ww.H, ww.D, 0, gen.STREAM_Q))
    k = dev(gen.normal_bshd(ww.B, ww.S, ww.H, ww.D, 0, gen.STREAM_K))
    v = dev(gen.normal_bshd(ww.B, ww.S, ww.H, ww.D, 0, gen.STREAM_V))
    o = torch.empty_like(q)
    win = h3.Window(ww.frame_tokens, ww.anchor_frames, ww.chunk_frames, ww.radius)
    for _ in range(warmup):
        h3.h3attn_prefill_window(q, k, v, o, win, None, None, stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        h3.h3attn_prefill_window(q, k, v, o, win, None, None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    st = h3.h3attn_check_device_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the window prefill")
    ms = e0.elapsed_time(e1) / steps
    pairs = ww.B * _window_pairs(ww.S, ww.S, ww.frame_tokens, ww.anchor_frames, ww.chunk_frames, ww.radius)
    flops = 4.0 * ww.D * ww.H * pairs
    tf = flops / (ms * 1e-3) / 1e12
    dense = 4.0 * ww.B * ww.S * ww.S * ww.H * ww.D
    return {"kernel": "attn_pipe_kernel<128,7> (window tile ranges)",
            "workload": f"{ww.name}: B={ww.B} S={ww.S} H={ww.H} D={ww.D}; frames of {ww.frame_tokens} tokens, "
                        f"{ww.anchor_frames} anchor frame, chunks of {ww.chunk_frames} frames, radius {ww.radius}",
            "bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": round(tf / peaks["bf16_tflops"], 4), "flops_per_launch": flops,
            "allowed_fraction": round(flops / dense, 4), "ms_per_launch": round(ms, 4),
            "dense_equivalent_tflops": round(dense / (ms * 1e-3) / 1e12, 1), "launches": steps + warmup}


# The library's choice of attention kernel: one query tile per CTA (Q held in
# tensor memory) for head dim 128 from 1024 keys on; one query tile per CTA
# with two CTAs per SM for head dim 128 below that and for head dim 64; the
# double-buffered-score kernel for head dim 256.  H3ATTN_ATTN_KERNEL forces 1
# (one tile, Q in tensor memory), 2 (two tiles per CTA), 3 (the persistent
# kernel), 4 (two CTAs per SM), 5 (head dim 256) or 6 (the unit-chaining
# kernel, head dim 128) where the head dim has it.
ONE_TILE_MIN_KEYS = 1024


def _attn_kernel_name(wl):
    sel = os.environ.get("H3ATTN_ATTN_KERNEL", "")
    if wl.D == 256:
        return "attn_fwd_kernel<256,1,2,1>" if sel in ("2", "3", "4") else "attn_wide_kernel<5>"
    if sel == "6" and wl.D == 128:
        return "attn_chain_kernel<6>"
    if sel == "3":
        return {64: "attn_persist_kernel<64,12>", 128: "attn_persist_kernel<128,7>"}[wl.D]
    one_tile = sel == "1" or (sel not in ("2", "4") and wl.D == 128 and wl.Sk >= ONE_TILE_MIN_KEYS)
    if one_tile:
        return {64: "attn_pipe_kernel<64,12>", 128: "attn_pipe_kernel<128,7>"}[wl.D]
    if sel == "2":
        return {64: "attn_fwd_kernel<64,2,8,1>", 128: "attn_fwd_kernel<128,2,4,1>"}[wl.D]
    return {64: "attn_fwd_kernel<64,1,4,2>", 128: "attn_fwd_kernel<128,1,2,2>"}[wl.D]


def _mod_shape(C, with_weight):
    """(compute warps per CTA, weight staged) that the library's AdaLN launcher
    picks for C channels: the first (warps, CTAs per SM) shape whose ring holds
    warps + 2 rows of 2C + 16 bytes, with the weight (4C bytes) staged when that
    keeps at least 3/4 of the compute warps per SM.  Used for labels only."""
    shapes = [(16, 2), (14, 2), (8, 4), (8, 3), (16, 1), (8, 2), (8, 1)]

    def pick(extra):
        for w, ctas in shapes:
            if (233472 // ctas - 1040 - extra) // (2 * C + 16) >= w + 2:
                return w, ctas
        return None
    plain = pick(0)
    staged = pick(4 * C) if with_weight else None
    if staged is not None and (plain is None or 4 * staged[0] * staged[1] >= 3 * plain[0] * plain[1]):
        return staged[0], True
    return (plain[0] if plain else 0), False


def _profiled_traffic():
    """DRAM bytes per launch recorded from an ncu capture, per kernel; a kernel
    whose sources changed since the capture (hash mismatch) reports None."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    out = {}
    if not os.path.exists(p):
        return out
    with open(p) as f:
        rec = json.load(f)
    for key in ("attn", "norm", "mod"):
        r = rec.get(key)
        if not r:
            continue
        h = hashlib.sha256()
        for name in r["sources"]:
            with open(os.path.join(ROOT, "video_dit_dense_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        out[key] = r["bytes_per_launch"] if h.hexdigest()[:16] == r["source_sha"] else None
    return out


def cpu_baseline(wl, inp, seconds):
    """The oracle as it stands, on the host cores, on a bounded row sample."""
    import numpy as np

    import oracle
    cores = min(os.cpu_count() or 1, 64)  # the oracle's thread count (one per core, at most 64)
    rng = np.random.default_rng(0)
    # norm/RoPE oracle (fp64) on consecutive token slices of q, then k, for at least a second
    norm_rows, t_norm, tok = 0, 0.0, 0
    while t_norm < 1.0 and wl.norm_rope:
        src = inp.q if (tok // wl.Sq) % 2 == 0 else inp.k
        t_lo = tok % wl.Sq
        n_tok = min(4096, wl.Sq - t_lo)
        x = np.ascontiguousarray(src[:, t_lo:t_lo + n_tok])
        t0 = time.perf_counter()
        oracle.qk_norm_rope_f64(x, inp.wq, inp.cos[t_lo:], inp.sin[t_lo:], wl.rotary_dim, wl.eps)
        t_norm += time.perf_counter() - t0
        norm_rows += x.shape[0] * x.shape[1] * x.shape[2]
        tok += n_tok
    # attention oracle on sampled rows, growing the sample until ~`seconds`
    n = min(8, wl.B * wl.Sq * wl.Hq)
    done_rows, t_att = 0, 0.0
    while t_att < seconds:
        ids = np.sort(rng.choice(wl.B * wl.Sq * wl.Hq, size=n, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attention_f64(inp.q, inp.k, inp.v, wl.scale, row_ids=ids)
        t_att += time.perf_counter() - t0
        done_rows += n
        n = min(n * 2, 4096, wl.B * wl.Sq * wl.Hq)
    flops_per_row = 4.0 * wl.Sk * wl.D
    total_rows = wl.B * wl.Sq * wl.Hq
    return {"value": round(done_rows * flops_per_row / t_att / 1e12, 6), "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"attention rate extrapolated from {done_rows} sampled row evaluations ({wl.name} has "
                      f"{total_rows} output rows; fp64, all {wl.Sk} keys each, {t_att:.1f} s; the full step would "
                      f"take ~{total_rows / done_rows * t_att:.0f} s); norm/RoPE fp64 on {norm_rows} q/k rows "
                      f"in {t_norm:.2f} s",
            "norm_rope_gbs": round(norm_rows * wl.D * 2 * 2 / t_norm / 1e9, 3) if norm_rows else None}


def run_reference(args):
    """Reference arm: the CPU oracle as it stands on the host cores."""
    import numpy as np

    import h3inputs as gen
    import oracle

    ws, rank, _ = _dist()
    if rank != 0:
        return
    wl = gen.WORKLOADS[args.workload]
    inp = gen.make_inputs(wl, seed=args.seed)
    flops_per_row = 4.0 * wl.Sk * wl.D
    rows_per_step = args.ref_rows
    rng = np.random.default_rng(0)

    def one_step():
        ids = np.sort(rng.choice(wl.B * wl.Sq * wl.Hq, size=rows_per_step, replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.qk_norm_rope_f64(np.ascontiguousarray(inp.q[:, :256]), inp.wq, inp.cos, inp.sin, wl.rotary_dim, wl.eps)
        oracle.attention_f64(inp.q, inp.k, inp.v, wl.scale, row_ids=ids)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one_step()
    t = sum(one_step() for _ in range(args.steps))
    value = rows_per_step * args.steps * flops_per_row / t / 1e12
    cores = os.cpu_count() or 1
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name}: B={wl.B} Sq={wl.Sq} Sk={wl.Sk} Hq={wl.Hq} Hkv={wl.Hkv} D={wl.D}; "
                               f"CPU oracle, {rows_per_step} sampled attention rows per step"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_per_step} attention rows (all {wl.Sk} keys) + norm/RoPE of 256 tokens per step"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-baseline", dest="cpu_baseline", action="store_true", default=True)
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--no-modulate", dest="modulate", action="store_false", default=True,
                    help="skip the RMSNorm -> AdaLN modulation measurement")
    ap.add_argument("--no-split", dest="split", action="store_false", default=True,
                    help="run prefill without the split-key tail's workspace")
    ap.add_argument("--no-window", dest="window", action="store_false", default=True,
                    help="skip the chunked-window attention measurement")
    args = ap.parse_args()
    if args.warmup < 3:
        print("bench: at least 3 warm-up steps are required; using 3", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
