"""Benchmark: shifted-window video attention on GB300.

One step = two layers of the alternating schedule on the 1080p-like grid
(T=21, H=68, W=120; nt=4, nh=nw=3; 24 heads x 128; 256 text tokens; bf16):

    window attention, REGULAR layout   (wp_window_attn: tcgen05 kernel + text mean)
    re-layout of the hidden rows [N, 2560] REGULAR -> SHIFTED   (wp_permute)
    window attention, SHIFTED layout
    re-layout of the hidden rows SHIFTED -> REGULAR

Inputs are synthetic N(0,1) (seeded) and resident in HBM before the timed
region; every input is larger than L2, so no flush is needed between steps.
The headline value is attention TFLOP/s over the whole step time (permutes
included); the kernel-level numbers and the roofline are reported beside it.
On one GPU the same line also carries the metric's 720p-like layers
(attn_720p), a bounded run of the re-layout sweep (relayout_sweep) and a
short run of the 32-layer schedule on T=30, 90x160 with the fused re-layout
beside the unfused one (full_schedule); --no-extras leaves them out.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload 1080p|720p|full|sweep] [--no-extras]

--impl reference times the CPU oracle on the host cores (bounded samples of
the same workload, same metric and unit).  Under torchrun every rank runs an
independent replica (the path has nothing to shard); the step time is the
max over ranks.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "window-attn TFLOP/s (% BF16 peak) and re-layout GB/s (% HBM) at 720p/1080p grids"
WORKLOADS = {
    "1080p": dict(T=21, H=68, W=120, nt=4, nh=3, nw=3, heads=24, hd=128, L=256, hidden=2560),
    "720p": dict(T=21, H=45, W=80, nt=4, nh=3, nw=3, heads=24, hd=128, L=256, hidden=2560),
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 129 * 1024 * 1024


def workload_desc(name, w):
    return ("%s-like grid T=%d H=%d W=%d (N=%d), nt=%d nh=%d nw=%d, heads=%d head_dim=%d, text L=%d, "
            "bf16; step = attn(regular) + relayout [N,%d] bf16 regular->shifted + attn(shifted) + "
            "relayout shifted->regular" % (name, w["T"], w["H"], w["W"], w["T"] * w["H"] * w["W"],
                                          w["nt"], w["nh"], w["nw"], w["heads"], w["hd"], w["L"],
                                          w["hidden"]))


def attn_flops(win_sizes, heads, hd, L):
    """4 * heads * hd * sum_w (n_w + L)^2 -- QK^T and PV over real rows only."""
    s = np.asarray(win_sizes, dtype=np.float64) + L
    return 4.0 * heads * hd * float((s * s).sum())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel_file, key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel (sha256 match); else None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = os.path.join(ROOT, "video_dit_shifted_gb300", "csrc", kernel_file)
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == key and f[1] == sha:
            return float(f[2])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc = index, None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) == 7:
                rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][1]) if rows[0][1].replace(".", "").isdigit() else None,
                "power_w_max": max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit()),
                "samples": len(rows), "reasons": reasons}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x, device):
    """Max of a host float over all ranks (the slowest replica sets the time)."""
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return t.item()


# ------------------------------------------------------------------ ours --
class Workload:
    def __init__(self, name, device, hidden=True):
        import video_dit_shifted_gb300 as vds
        from video_dit_shifted_gb300 import synth
        self.vds, self.w, self.name, self.dev = vds, WORKLOADS[name], name, device
        w = self.w
        self.plan = vds.Plan(w["T"], w["H"], w["W"], w["nt"], w["nh"], w["nw"], device=device)
        N, heads, hd, L = self.plan.N, w["heads"], w["hd"], w["L"]
        self.N = N
        x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, device)
        self.qkv = {vds.REGULAR: x["vid_buf"], vds.SHIFTED: torch.empty_like(x["vid_buf"])}
        vds.permute(self.plan, x["vid_buf"].view(N, -1), self.qkv[vds.SHIFTED].view(N, -1),
                    vds.REGULAR, vds.SHIFTED)
        self.txt = x["txt_buf"]
        if hidden:
            self.hidden = synth.hidden(N, w["hidden"], torch.bfloat16, device)
            self.hidden2 = torch.empty_like(self.hidden)
        self.o_vid = {l: torch.empty((N, heads, hd), dtype=torch.bfloat16, device=device)
                      for l in (vds.REGULAR, vds.SHIFTED)}
        self.o_txt = {l: torch.empty((L, heads, hd), dtype=torch.bfloat16, device=device)
                      for l in (vds.REGULAR, vds.SHIFTED)}
        self.ws = {l: vds.make_workspace(self.plan, l, heads, hd, L, vds.BF16, device)
                   for l in (vds.REGULAR, vds.SHIFTED)}
        self.flops = {}
        for l in (vds.REGULAR, vds.SHIFTED):
            off = self.plan.host_tables(l)[0]
            self.flops[l] = attn_flops(np.diff(off), heads, hd, L)
        self.relayout_bytes = 2.0 * N * w["hidden"] * 2  # read + write per re-layout
        torch.cuda.synchronize()

    def attn(self, layout):
        vds, t = self.vds, self.txt
        b = self.qkv[layout]
        vds.window_attn(self.plan, layout, b[:, 0], b[:, 1], b[:, 2], t[:, 0], t[:, 1], t[:, 2],
                        self.o_vid[layout], self.o_txt[layout], self.ws[layout])

    def step(self, ev=None):
        """ev: list of 8 events to bracket the four launches (or None)."""
        vds = self.vds
        rec = (lambda i: ev[i].record()) if ev else (lambda i: None)
        rec(0); self.attn(vds.REGULAR); rec(1)
        rec(2); vds.permute(self.plan, self.hidden, self.hidden2, vds.REGULAR, vds.SHIFTED); rec(3)
        rec(4); self.attn(vds.SHIFTED); rec(5)
        rec(6); vds.permute(self.plan, self.hidden2, self.hidden, vds.SHIFTED, vds.REGULAR); rec(7)

    launches_per_step = 6  # 2 x (attention kernel + text mean) + 2 x permute

    def step_flops(self):
        return self.flops[self.vds.REGULAR] + self.flops[self.vds.SHIFTED]

    def check_status(self):
        for l, ws in self.ws.items():
            st = self.vds.read_status(ws)
            if st != 0:
                raise RuntimeError("device status %d after layout %d" % (st, l))


def run_e2e(wl, steps, warmup):
    """Same step through the public API with host buffers: every step copies
    its inputs in from pinned host memory (q/k/v in the regular layout, text
    q/k/v, hidden rows), derives the shifted q/k/v on the device with
    wp_permute, runs the step, and copies every output back (video and text
    outputs of both layers, hidden rows), all inside the timed region.

    Steps are pipelined the way a serving loop would run them: three device
    buffer sets and three streams, so that the copy-in of step i+1 and the
    copy-out of step i-1 overlap step i's compute (the copy engines of the
    two directions run at once).  Events keep every reuse safe: a set is
    refilled only after the copy-out of its last outputs (the hidden rows
    are both an input and an output), and its compute waits for its inputs."""
    vds = wl.vds
    N = wl.N
    nsets = 3
    sets = [wl] + [Workload(wl.name, wl.dev) for _ in range(nsets - 1)]

    def ins(w):
        return {"qkv_reg": w.qkv[vds.REGULAR], "txt": w.txt, "hidden": w.hidden}

    def outs(w):
        return [w.o_vid[vds.REGULAR], w.o_vid[vds.SHIFTED], w.o_txt[vds.REGULAR], w.o_txt[vds.SHIFTED], w.hidden]

    pinned_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in ins(wl).items()}
    for k, v in ins(wl).items():
        pinned_in[k].copy_(v)
    pinned_out = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs(wl)] for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in pinned_in.values())
    d2h = sum(t.numel() * t.element_size() for t in pinned_out[0])
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = ([ev() for _ in range(nsets)] for _ in range(3))
    for e in out_done:
        e.record(torch.cuda.current_stream())

    copy_ev = []  # per step: (h2d start, h2d end, d2h start, d2h end), timing events

    def one(i, timed=False):
        b = i % nsets
        w = sets[b]
        ev4 = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if timed else None
        s_in.wait_event(out_done[b])           # this set's last outputs (and so its compute) are done
        with torch.cuda.stream(s_in):
            if timed: ev4[0].record(s_in)
            for k, dst in ins(w).items():
                dst.copy_(pinned_in[k], non_blocking=True)
            if timed: ev4[1].record(s_in)
            in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        with torch.cuda.stream(s_comp):
            vds.permute(w.plan, w.qkv[vds.REGULAR].view(N, -1), w.qkv[vds.SHIFTED].view(N, -1),
                        vds.REGULAR, vds.SHIFTED)
            w.step()
            comp_done[b].record(s_comp)
        s_out.wait_event(comp_done[b])
        with torch.cuda.stream(s_out):
            if timed: ev4[2].record(s_out)
            for o, p in zip(outs(w), pinned_out[b]):
                p.copy_(o, non_blocking=True)
            if timed: ev4[3].record(s_out)
            out_done[b].record(s_out)
        if timed: copy_ev.append(ev4)

    def copies_only():
        """The same copies with no compute, both directions at once, every
        buffer set once as the loop uses them: what the host link allows per
        step at that moment (the e2e bound)."""
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0.record(s_in)
        s_out.wait_stream(s_in)
        for r in range(nsets):
            w = sets[r]
            with torch.cuda.stream(s_in):
                for k, dst in ins(w).items():
                    dst.copy_(pinned_in[k], non_blocking=True)
            with torch.cuda.stream(s_out):
                for o, p in zip(outs(w), pinned_out[r]):
                    p.copy_(o, non_blocking=True)
        s_in.wait_stream(s_out)
        l1.record(s_in)
        torch.cuda.synchronize()
        return l0.elapsed_time(l1) / nsets

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    link_before = copies_only()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    s_comp.wait_stream(s_in)
    s_out.wait_stream(s_in)
    for i in range(steps):
        one(i, timed=True)
    s_out.wait_stream(s_comp)
    s_out.wait_stream(s_in)
    end.record(s_out)
    torch.cuda.synchronize()
    for w in sets:
        w.check_status()
    e2e_ms = start.elapsed_time(end) / steps
    # The link during the loop: each step's copies in and out, timed on their streams.
    h2d_ms = statistics.median(e[0].elapsed_time(e[1]) for e in copy_ev)
    d2h_ms = statistics.median(e[2].elapsed_time(e[3]) for e in copy_ev)
    link_after = copies_only()
    del sets[1:]
    return e2e_ms, h2d, d2h, (link_before, link_after), (h2d_ms, d2h_ms)


def oracle_sample(wl_name, budget_s, seed_rows=None):
    """Time the CPU oracle on (window, head) pairs of the REGULAR layer, in
    window order, until budget_s seconds of work.  Inputs are synthetic
    N(0,1) float values drawn on the host (the oracle's cost does not depend
    on the values).  Returns (tflops, pairs, flops, seconds)."""
    from oracle import attention as oa
    from oracle import plan as op
    w = WORKLOADS[wl_name]
    off, ids = op.layout_tables(w["T"], w["H"], w["W"], w["nt"], w["nh"], w["nw"], op.REGULAR)
    rng = np.random.default_rng(0)
    heads, hd, L = w["heads"], w["hd"], w["L"]
    txt = [rng.standard_normal((L, 1, hd)) for _ in range(3)]
    done, flops, t_used = 0, 0.0, 0.0
    nwin = len(off) - 1
    k = 0
    while t_used < budget_s and k < nwin * heads:
        win = k % nwin
        n_w = int(off[win + 1] - off[win])
        q, kk, v = (rng.standard_normal((n_w, 1, hd)) for _ in range(3))
        sub_off = np.array([0, n_w])
        t0 = time.perf_counter()
        oa.window_attention(q, kk, v, *txt, sub_off, np.arange(n_w))
        t_used += time.perf_counter() - t0
        flops += attn_flops([n_w], 1, hd, L)
        done += 1
        k += 1
    return flops / t_used / 1e12, done, flops, t_used


def oracle_relayout_sample(wl_name, reps=3):
    """The oracle's re-layout (a numpy row gather by the inverted id table)
    of the hidden rows [N, 2560] (bf16 bits as uint16) regular -> shifted on
    the workload's grid, timed on the host: GB/s counting 2 * N * 5120 bytes
    per re-layout, like the GPU's figure.  numpy's gather runs on one core."""
    from oracle import permute as opm
    from oracle import plan as op
    w = WORKLOADS[wl_name]
    g = (w["T"], w["H"], w["W"], w["nt"], w["nh"], w["nw"])
    ids_r, ids_s = op.layout_tables(*g, op.REGULAR)[1], op.layout_tables(*g, op.SHIFTED)[1]
    N = ids_r.size
    rows = np.random.default_rng(0).integers(0, 1 << 16, size=(N, w["hidden"]), dtype=np.uint16)
    opm.permute_rows(rows, ids_r, ids_s)                      # warm the pages
    t0 = time.perf_counter()
    for _ in range(reps):
        opm.permute_rows(rows, ids_r, ids_s)
    secs = (time.perf_counter() - t0) / reps
    nbytes = 2.0 * N * w["hidden"] * 2
    return {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "%d re-layouts of [%d, %d] bf16 rows regular -> shifted (%.2f GB each), %.3f s each"
                      % (reps, N, w["hidden"], nbytes / 1e9, secs)}


def host_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("internal_api") in ("openblas", "mkl")]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    if args.workload not in WORKLOADS:
        args.workload = "1080p"  # the oracle is timed on (window, head) samples of the 1080p grid
    w = WORKLOADS[args.workload]
    times, flops_all = [], []
    for i in range(args.warmup + args.steps):
        tf, pairs, fl, secs = oracle_sample(args.workload, args.ref_step_s)
        if i >= args.warmup:
            times.append(secs)
            flops_all.append(fl)
    val = sum(flops_all) / sum(times) / 1e12
    cores = host_threads()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_desc(args.workload, w)},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": "per step: (window, head) pairs of the regular layer in window order "
                                       "until %.0f s of float64 oracle work" % args.ref_step_s},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def full_schedule_measure(dev, steps, warmup):
    """The full 32-layer schedule on T=30, H=90, W=160 (N=432000): layer l
    runs window attention in the regular layout if l is even, else shifted;
    the text output of every layer is mean-reduced.  Three ways to bring the
    rows into the next layer's order between layers (31 transitions), each
    timed as its own 32-layer step:

      qkv      attention (video output in canonical order), then the packed
               q/k/v rows [N, 3, 24, 128] bf16 re-laid out into the next
               layer's order (wp_permute);
      unfused  attention (canonical output), then the video output
               [N, 24, 128] re-laid out canonical -> next layout (wp_permute);
      fused    attention writing its video output straight into the next
               layer's order (wp_window_attn_to): no separate pass.

    In the last two the next layer reads q/k/v already in its own order (a
    model's projections after the attention output would produce them
    there).  Returns a dict of the three measurements."""
    import video_dit_shifted_gb300 as vds
    from video_dit_shifted_gb300 import schedule, synth
    T, H, W, heads, hd, L = 30, 90, 160, 24, 128, 256
    plan = vds.Plan(T, H, W, 4, 3, 3, device=dev)
    N = plan.N
    layouts = schedule.layer_layouts(32)
    trans = schedule.transitions(layouts)
    x = synth.attention_inputs(N, L, heads, hd, torch.bfloat16, dev)
    qkv = {vds.REGULAR: x["vid_buf"], vds.SHIFTED: torch.empty_like(x["vid_buf"])}
    vds.permute(plan, qkv[vds.REGULAR].view(N, -1), qkv[vds.SHIFTED].view(N, -1), vds.REGULAR, vds.SHIFTED)
    ping = [x["vid_buf"], torch.empty_like(x["vid_buf"])]      # qkv variant: starts in REGULAR order
    txt = x["txt_buf"]
    o_vid = [torch.empty((N, heads, hd), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    o_txt = torch.empty((32, L, heads, hd), dtype=torch.bfloat16, device=dev)
    ws = {l: vds.make_workspace(plan, l, heads, hd, L, vds.BF16, dev) for l in (vds.REGULAR, vds.SHIFTED)}
    flops = {l: attn_flops(np.diff(plan.host_tables(l)[0]), heads, hd, L) for l in (vds.REGULAR, vds.SHIFTED)}
    step_flops = sum(flops[l] for l in layouts)
    qkv_row_B = x["vid_buf"][0].numel() * 2
    out_row_B = heads * hd * 2
    ev = lambda: torch.cuda.Event(enable_timing=True)

    fused_out = schedule.output_layouts(layouts)  # the next layer's order; canonical after the last

    def step(variant, rec=None):
        cur = 0
        for l, lay in enumerate(layouts):
            nxt = layouts[l + 1] if l + 1 < len(layouts) else None
            b = ping[cur] if variant == "qkv" else qkv[lay]
            a0, a1 = ev(), ev()
            a0.record()
            out_layout = fused_out[l] if variant == "fused" else vds.CANONICAL
            vds.window_attn(plan, lay, b[:, 0], b[:, 1], b[:, 2], txt[:, 0], txt[:, 1], txt[:, 2], o_vid[0],
                            o_txt[l], ws[lay], out_layout=out_layout)
            a1.record()
            p = None
            if nxt is not None and variant != "fused":
                p0, p1 = ev(), ev()
                p0.record()
                if variant == "qkv":
                    vds.permute(plan, ping[cur].view(N, -1), ping[1 - cur].view(N, -1), lay, nxt)
                    cur = 1 - cur
                else:
                    vds.permute(plan, o_vid[0].view(N, -1), o_vid[1].view(N, -1), vds.CANONICAL, nxt)
                p1.record()
                p = (p0, p1)
            if rec is not None:
                rec.append(((a0, a1), p))

    out = {}
    for variant in ("qkv", "unfused", "fused"):
        for _ in range(warmup):
            step(variant)
        torch.cuda.synchronize()
        for l, w in ws.items():
            if vds.read_status(w) != 0:
                raise RuntimeError("device status set in the full schedule (%s)" % variant)
        s, e = ev(), ev()
        rec = []
        s.record()
        for _ in range(steps):
            step(variant, rec)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e) / steps
        attn_ms = sum(a[0].elapsed_time(a[1]) for a, _ in rec) / steps
        perm = [p[0].elapsed_time(p[1]) for _, p in rec if p is not None]
        perm_ms = sum(perm) / steps
        row_B = {"qkv": qkv_row_B, "unfused": out_row_B, "fused": 0}[variant]
        perm_bytes = len(trans) * 2.0 * N * row_B
        out[variant] = {"ms_per_step": ms, "tflops": step_flops / (ms * 1e-3) / 1e12,
                        "attn_ms_per_step": attn_ms, "attn_tflops": step_flops / (attn_ms * 1e-3) / 1e12,
                        "relayout_ms_per_step": perm_ms, "relayout_gb_per_step": perm_bytes / 1e9,
                        "relayout_gbs": (perm_bytes / (perm_ms * 1e-3) / 1e9) if perm_ms > 0 else None,
                        "gpu_launches_per_step": 2 * len(layouts) + (len(trans) if variant != "fused" else 0)}
    out["attn_tflop_per_step"] = step_flops / 1e12
    out["fused_saves"] = {"ms_per_step": out["unfused"]["ms_per_step"] - out["fused"]["ms_per_step"],
                          "gb_per_step": out["unfused"]["relayout_gb_per_step"]}
    plan.close()
    del x, qkv, ping, o_vid, o_txt, ws
    torch.cuda.empty_cache()
    return out


def run_full_schedule(args):
    """--workload full: the 32-layer schedule (see full_schedule_measure) as
    its own JSON line; value = attention TFLOP of a step / step time of the
    qkv variant."""
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    clocks = ClockSampler(0)
    clocks.start()
    r = full_schedule_measure(dev, args.steps, args.warmup)
    clk = clocks.stop()
    peaks, peak_src = load_peaks()
    q = r["qkv"]
    line = {"metric": METRIC, "value": q["tflops"], "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": q["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "full schedule: 32 alternating regular/shifted layers (31 re-layouts of packed "
                                   "qkv [N,3,24,128] bf16) on T=30 H=90 W=160 (N=432000), nt=4 nh=3 nw=3, "
                                   "heads=24 head_dim=128, text L=256, text mean per layer",
                       "l2": "inputs larger than L2: no flush"},
            "attn_tflops": q["attn_tflops"], "attn_frac_bf16_peak": q["attn_tflops"] / peaks["bf16_tflops"],
            "relayout_gbs": q["relayout_gbs"], "relayout_frac_hbm": q["relayout_gbs"] / peaks["hbm_gbs"],
            "variants": r, "peak_source": peak_src,
            "gpu_launches": args.steps * q["gpu_launches_per_step"], "clocks": clk}
    print(json.dumps(line), flush=True)


def sweep_measure(dev, steps, warmup):
    """The re-layout sweep: hidden rows [N, 2560] bf16 permuted regular ->
    shifted and back on grids 45x80 / 68x120 / 90x160 x T in {5, 21, 30}
    (nt, nh, nw = 4, 3, 3).  Each timed launch follows an L2 flush (a write
    of twice the L2 size); points whose footprint is under four times L2 are
    flagged and left out of the median.  Bytes = 2 * N * 5120 per launch (the
    4-byte table read per row is not counted)."""
    import video_dit_shifted_gb300 as vds
    from video_dit_shifted_gb300 import synth
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    peaks, peak_src = load_peaks()
    points = []
    for (H, W) in ((45, 80), (68, 120), (90, 160)):
        for T in (5, 21, 30):
            plan = vds.Plan(T, H, W, 4, 3, 3, device=dev)
            N = plan.N
            src = synth.hidden(N, 2560, torch.bfloat16, dev)
            dst = torch.empty_like(src)
            back = torch.empty_like(src)
            nbytes = 2.0 * N * 2560 * 2
            res = {}
            for name, a, b, (x, y) in (("regular->shifted", vds.REGULAR, vds.SHIFTED, (src, dst)),
                                       ("shifted->regular", vds.SHIFTED, vds.REGULAR, (dst, back))):
                for _ in range(warmup):
                    vds.permute(plan, x, y, a, b)
                ms = []
                for _ in range(steps):
                    flush.fill_(1)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record()
                    vds.permute(plan, x, y, a, b)
                    e1.record()
                    torch.cuda.synchronize()
                    ms.append(e0.elapsed_time(e1))
                med = statistics.median(ms)
                res[name] = {"ms": med, "gbs": nbytes / (med * 1e-3) / 1e9,
                             "frac": nbytes / (med * 1e-3) / 1e9 / peaks["hbm_gbs"]}
            if not torch.equal(back, src):
                raise RuntimeError("re-layout round trip is not the identity on %dx%dx%d" % (T, H, W))
            points.append({"grid": "%dx%dx%d" % (T, H, W), "N": N, "bytes_per_launch": nbytes,
                           "near_l2": nbytes < 4 * l2, **res})
            plan.close()
            del src, dst, back
    del flush
    torch.cuda.empty_cache()
    big = [p for p in points if not p["near_l2"]]
    gbs = [p[d]["gbs"] for p in big for d in ("regular->shifted", "shifted->regular")]
    med = statistics.median(gbs)
    return {"median_gbs": med, "frac": med / peaks["hbm_gbs"], "peak": peaks["hbm_gbs"], "peak_source": peak_src,
            "min_gbs": min(gbs), "max_gbs": max(gbs), "points_in_median": 2 * len(big), "points": points,
            "l2": "L2 flushed (write of %d MB) before every timed launch" % (2 * l2 // 2**20),
            "gpu_launches": len(points) * 2 * steps}


def run_sweep(args):
    """--workload sweep: the re-layout sweep (see sweep_measure) as its own
    JSON line."""
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    clocks = ClockSampler(0)
    clocks.start()
    r = sweep_measure(dev, args.steps, args.warmup)
    clk = clocks.stop()
    line = {"metric": "re-layout GB/s (% HBM), [N,2560] bf16 sweep", "value": r["median_gbs"],
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "re-layout sweep: hidden rows [N,2560] bf16, grids 45x80/68x120/90x160 x "
                                   "T in {5,21,30}, nt nh nw = 4 3 3, both directions; value = median GB/s "
                                   "over the points above 4x L2",
                       "l2": r["l2"]},
            "peak": r["peak"], "peak_source": r["peak_source"], "frac": r["frac"],
            "points": r["points"], "gpu_launches": r["gpu_launches"], "clocks": clk}
    print(json.dumps(line), flush=True)


def layer_measure(name, dev, reps, warmup):
    """Both attention layers of a workload timed alone (wp_window_attn:
    tcgen05 kernel + text mean), `reps` launches each after `warmup`;
    inputs larger than L2.  Returns per-layout ms and TFLOP/s."""
    import video_dit_shifted_gb300 as vds
    wl = Workload(name, dev, hidden=False)
    peaks, _ = load_peaks()
    out = {}
    for layout, lname in ((vds.REGULAR, "regular"), (vds.SHIFTED, "shifted")):
        for _ in range(warmup):
            wl.attn(layout)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            wl.attn(layout)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tf = wl.flops[layout] / (ms * 1e-3) / 1e12
        out[lname] = {"ms": ms, "tflops": tf, "frac_bf16_peak": tf / peaks["bf16_tflops"],
                      "tflop_per_launch": wl.flops[layout] / 1e12}
    wl.check_status()
    del wl
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    world, rank, local, pg = dist_setup(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    wl = Workload(args.workload, dev)
    vds = wl.vds
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    wl.check_status()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(8)] for _ in range(args.steps)]
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if world == 1 else local)
    clocks.start()
    barrier(pg)
    torch.cuda.synchronize()
    s.record()
    for i in range(args.steps):
        wl.step(evs[i])
    e.record()
    torch.cuda.synchronize()
    barrier(pg)
    clk = clocks.stop()
    wl.check_status()
    total_ms = max_over_ranks(pg, s.elapsed_time(e), dev)
    ms_step = total_ms / args.steps
    attn_reg = [ev[0].elapsed_time(ev[1]) for ev in evs]
    attn_shf = [ev[4].elapsed_time(ev[5]) for ev in evs]
    perm = [ev[2].elapsed_time(ev[3]) for ev in evs] + [ev[6].elapsed_time(ev[7]) for ev in evs]
    f_reg, f_shf = wl.flops[vds.REGULAR], wl.flops[vds.SHIFTED]
    step_flops = f_reg + f_shf
    value = world * step_flops / (ms_step * 1e-3) / 1e12
    attn_ms = (sum(attn_reg) + sum(attn_shf)) / (2 * args.steps)
    attn_tflops = (f_reg + f_shf) / 2 / (attn_ms * 1e-3) / 1e12
    perm_ms = sum(perm) / len(perm)
    relayout_gbs = wl.relayout_bytes / (perm_ms * 1e-3) / 1e9
    peaks, peak_src = load_peaks()
    traffic = recorded_traffic("attn_tc.cu", "attn_tc_1080p") if args.workload == "1080p" else None
    roofline = {"bound": "tensor", "achieved": attn_tflops, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": attn_tflops / peaks["bf16_tflops"], "traffic": traffic,
                "peak_source": peak_src + " (bf16 burst)",
                "kernel": "attn_tc_kernel (+ text_mean_kernel inside the same timed call)",
                "frac_of_sustained": attn_tflops / peaks["bf16_tflops_sustained"],
                "per_layout_ms": {"regular": sum(attn_reg) / args.steps, "shifted": sum(attn_shf) / args.steps},
                "flops_per_launch": {"regular": f_reg, "shifted": f_shf}}
    relayout = {"bound": "hbm", "achieved": relayout_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": relayout_gbs / peaks["hbm_gbs"],
                "traffic": recorded_traffic("permute.cu", "permute_1080p") if args.workload == "1080p" else None,
                "kernel": "permute_rows_kernel", "bytes_per_launch": wl.relayout_bytes, "ms": perm_ms,
                "peak_source": peak_src}
    e2e_ms, h2d, d2h, link_ms, loop_copy_ms = run_e2e(wl, args.e2e_steps, max(3, min(args.warmup, 4)))
    e2e_ms = max_over_ranks(pg, e2e_ms, dev)
    e2e = {"value": world * step_flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "steps": args.e2e_steps,
           "copies_only_ms_per_step": min(link_ms),
           "copies_only_ms_before_after": list(link_ms),
           "in_loop_copies": {"h2d_ms_median": loop_copy_ms[0], "d2h_ms_median": loop_copy_ms[1],
                              "h2d_gbs": h2d / (loop_copy_ms[0] * 1e-3) / 1e9,
                              "d2h_gbs": d2h / (loop_copy_ms[1] * 1e-3) / 1e9,
                              "note": "each step's copies timed on their streams inside the loop; the two "
                                      "directions overlap each other and the compute"},
           "pipelining": "copy-in of step i+1 and copy-out of step i-1 overlap step i (3 device buffer sets, "
                         "3 streams); every step's copies are inside the timed region"}
    # Window-local RoPE of q and k (a separate in-place pass, not part of the
    # step): HBM-bound, 2 tensors x (read + write) x rows x heads x 128 x 2 B.
    b, t = wl.qkv[vds.REGULAR], wl.txt
    rope_bytes = 2 * 2 * (wl.N + wl.w["L"]) * wl.w["heads"] * wl.w["hd"] * 2
    for _ in range(2):
        vds.rope(wl.plan, vds.REGULAR, b[:, 0], b[:, 1], t[:, 0], t[:, 1])
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record()
    for _ in range(10):
        vds.rope(wl.plan, vds.REGULAR, b[:, 0], b[:, 1], t[:, 0], t[:, 1])
    r1.record()
    torch.cuda.synchronize()
    rope_ms = r0.elapsed_time(r1) / 10
    peaks_r, _ = load_peaks()
    rope = {"bound": "hbm", "achieved": rope_bytes / (rope_ms * 1e-3) / 1e9, "peak": peaks_r["hbm_gbs"],
            "unit": "GB/s", "frac": rope_bytes / (rope_ms * 1e-3) / 1e9 / peaks_r["hbm_gbs"], "ms": rope_ms,
            "traffic": recorded_traffic("rope.cu", "rope_1080p") if args.workload == "1080p" else None,
            "bytes_per_launch": rope_bytes, "kernel": "rope_kernel (regular layout, q and k in place)"}
    # The same regular layer with the RoPE applied inside the attention kernel
    # (wp_window_attn_rope, un-rotated q/k in) against the RoPE pass followed
    # by the attention call above.
    ws_rope = vds.make_workspace(wl.plan, vds.REGULAR, wl.w["heads"], wl.w["hd"], wl.w["L"], vds.BF16, dev,
                                 rope=True)
    fused = lambda: vds.window_attn_rope(wl.plan, vds.REGULAR, b[:, 0], b[:, 1], b[:, 2], t[:, 0], t[:, 1],
                                         t[:, 2], wl.o_vid[vds.REGULAR], wl.o_txt[vds.REGULAR], ws_rope)
    for _ in range(2):
        fused()
    r0.record()
    for _ in range(10):
        fused()
    r1.record()
    torch.cuda.synchronize()
    fused_ms = r0.elapsed_time(r1) / 10
    if vds.read_status(ws_rope) != 0:
        raise RuntimeError("device status set by wp_window_attn_rope")
    attn_reg_ms = sum(attn_reg) / args.steps
    rope_fused = {"kernel": "wp_window_attn_rope, regular layer: k rotated once into the workspace "
                            "(rope_k_copy_kernel), Q tiles rotated inside attn_tc_kernel",
                  "ms_fused": fused_ms, "tflops_fused": f_reg / (fused_ms * 1e-3) / 1e12,
                  "ms_rope_then_attn": rope_ms + attn_reg_ms, "ms_attn": attn_reg_ms, "ms_rope": rope_ms}
    del ws_rope
    fp8 = fp8_measure(wl, attn_reg, attn_shf, args.steps)
    # The metric's other grid and the other configurations, measured in the
    # same run (single-GPU runs only; each after its own warm-up).
    extras = None
    if world == 1 and not args.no_extras:
        torch.cuda.empty_cache()

        def clocked(fn):
            c = ClockSampler(dev.index)
            c.start()
            out = fn()
            return out, c.stop()

        a720, clk720 = clocked(lambda: layer_measure("720p", dev, reps=20, warmup=3))
        sw, clksw = clocked(lambda: sweep_measure(dev, steps=5, warmup=3))
        fs, clkfs = clocked(lambda: full_schedule_measure(dev, steps=2, warmup=3))
        a720["clocks"] = clk720
        fs["clocks"] = clkfs
        extras = {
            "attn_720p": a720,
            "relayout_sweep": {k: sw[k] for k in ("median_gbs", "frac", "min_gbs", "max_gbs", "points_in_median",
                                                  "peak", "l2")},
            "full_schedule": fs,
        }
        extras["relayout_sweep"]["clocks"] = clksw
        extras["relayout_sweep"]["workload"] = ("[N,2560] bf16 rows, regular->shifted and back, grids 45x80/68x120/"
                                                "90x160 x T in {5,21,30}; median of 5 launches per point, L2 flushed "
                                                "before each; median over the points above 4x L2")
        extras["relayout_sweep"]["points_gbs"] = {p["grid"]: [round(p[d]["gbs"], 1) for d in
                                                              ("regular->shifted", "shifted->regular")]
                                                  for p in sw["points"]}
        extras["full_schedule"]["workload"] = ("32 alternating layers on T=30 H=90 W=160 (N=432000), 24x128 heads, "
                                               "L=256; 2 steps after 3 per variant (see bench.py "
                                               "full_schedule_measure)")
    cpu = cpu_relayout = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tf, pairs, fl, secs = oracle_sample(args.workload, args.cpu_budget_s)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": host_threads(), "kind": "oracle",
               "sample": "%d (window, head) pairs of the regular layer (%.1f GFLOP, %.1f s), float64 numpy"
                         % (pairs, fl / 1e9, secs)}
        cpu_relayout = oracle_relayout_sample(args.workload)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": workload_desc(args.workload, wl.w),
                           "l2": "inputs larger than L2 (qkv %.2f GB, hidden %.2f GB): no flush"
                                 % (wl.qkv[vds.REGULAR].numel() * 2 / 1e9, wl.hidden.numel() * 2 / 1e9),
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "attn_tflops": attn_tflops, "relayout_gbs": relayout_gbs,
                "roofline": roofline, "roofline_relayout": relayout, "roofline_rope": rope,
                "rope_fused": rope_fused, "fp8_qk": fp8,
                "cpu_baseline": cpu, "cpu_baseline_relayout": cpu_relayout, "e2e": e2e,
                "gpu_launches": wl.launches_per_step * args.steps, "clocks": clk}
        if extras is not None:
            line.update(extras_line(extras))
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def fp8_measure(wl, attn_reg, attn_shf, steps):
    """Both 1080p layers with e4m3 q/k (wp_window_attn_fp8) against the bf16
    call of the timed steps, and the quantise pass (wp_quantize_e4m3 of q and
    k, HBM-bound) that a caller without e4m3 projections would add."""
    vds = wl.vds
    N, heads, hd, L = wl.N, wl.w["heads"], wl.w["hd"], wl.w["L"]
    inv = 64.0
    qk8 = {l: torch.empty((N, 2, heads, hd), dtype=torch.uint8, device=wl.dev) for l in (vds.REGULAR, vds.SHIFTED)}
    qkt8 = torch.empty((L, 2, heads, hd), dtype=torch.uint8, device=wl.dev)

    def quantize(l):
        b = wl.qkv[l]
        for i in range(2):
            vds.quantize_e4m3(b[:, i].reshape(N, heads * hd), qk8[l][:, i].reshape(N, heads * hd), inv)

    for i in range(2):
        vds.quantize_e4m3(wl.txt[:, i].reshape(L, heads * hd), qkt8[:, i].reshape(L, heads * hd), inv)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for l in (vds.REGULAR, vds.SHIFTED, vds.REGULAR, vds.REGULAR):
        quantize(l)
    e0.record()
    for _ in range(5):
        quantize(vds.REGULAR)
    e1.record()
    torch.cuda.synchronize()
    q_ms = e0.elapsed_time(e1) / 5
    q_bytes = 2 * N * heads * hd * (2 + 1)
    out = {"kernel": "attn_tc_kernel<128, e4m3 Q K^T> (wp_window_attn_fp8), q/k codes = e4m3(x * 64)",
           "quantize_ms": q_ms, "quantize_gbs": q_bytes / (q_ms * 1e-3) / 1e9,
           "quantize_bytes": q_bytes}
    t = wl.txt
    for l, name, bf in ((vds.REGULAR, "regular", attn_reg), (vds.SHIFTED, "shifted", attn_shf)):
        run = lambda: vds.window_attn_fp8(wl.plan, l, qk8[l][:, 0], qk8[l][:, 1], wl.qkv[l][:, 2], qkt8[:, 0],
                                          qkt8[:, 1], t[:, 2], 1.0 / inv, 1.0 / inv, wl.o_vid[l], wl.o_txt[l],
                                          wl.ws[l])
        for _ in range(3):
            run()
        e0.record()
        for _ in range(10):
            run()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / 10
        if vds.read_status(wl.ws[l]) != 0:
            raise RuntimeError("device status set by wp_window_attn_fp8")
        bf_ms = sum(bf) / steps
        out[name] = {"ms": ms, "tflops": wl.flops[l] / (ms * 1e-3) / 1e12, "ms_bf16": bf_ms,
                     "speedup_vs_bf16": bf_ms / ms}
    del qk8, qkt8
    return out


def extras_line(x):
    """Keys the default line carries for the other configurations."""
    fs = x["full_schedule"]
    return {"attn_720p": x["attn_720p"], "relayout_sweep": x["relayout_sweep"],
            "full_schedule": {"workload": fs["workload"], "attn_tflop_per_step": fs["attn_tflop_per_step"],
                              "qkv": fs["qkv"], "unfused": fs["unfused"], "fused": fs["fused"],
                              "fused_saves": fs["fused_saves"], "clocks": fs["clocks"]}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS) + ["full", "sweep"], default="1080p")
    ap.add_argument("--e2e-steps", type=int, default=16)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the 720p layers, the re-layout sweep and the 32-layer schedule")
    args = ap.parse_args()
    if args.warmup < 3:
        print("note: --warmup raised to 3 (timing rules)", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "full":
        run_full_schedule(args)
    elif args.workload == "sweep":
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
