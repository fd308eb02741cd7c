#!/usr/bin/env python3
"""Throughput of the routed W4A16 MoE layer (moe_layer_forward) on GB300.

One step = one pass of the whole layer over one batch of the workload:
  decode (default): 48 distinct decode-shaped layers back to back, T=2 tokens
      each (d_model 2048, d_ff 768, 128 experts, top-8, int4 g128 weights);
      15.4 GB of distinct weights, so every layer reads its experts from HBM.
  skew: one skewed prefill layer, P=4096 tokens, Zipf(1.1) expert load.
  (prefill, large_decode, large_prefill, tiny are accepted too.)
Metric: MoE-layer tokens/s = tokens routed through the layer per second
(decode: 2 tokens x 48 layers per step).  The timed region replays a CUDA
graph of the step on inputs already resident in HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
       [--impl ours|reference] [--layers L] [--no-secondary] [--no-cpu-baseline]
The JSON line also carries the dominant kernel's roofline, the CPU oracle's
rate on a bounded sample (cpu_baseline), the parity of the timed step against
the oracle on that sample, an end-to-end rate with host buffers (e2e), the
kernel launch count and the SM clocks seen during the timed region.
Under torchrun (N > 1) every rank runs an independent replica (the layer has
no cross-GPU exchange); value = all ranks' tokens / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth as S  # noqa: E402

METRIC = "MoE-layer tokens/s (decode T=2, prefill P=4096); % HBM BW / % bf16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
WORKLOADS = {
    "decode": ("decode", 48),
    "skew": ("skew", 1),
    "prefill": ("prefill", 1),
    "large_decode": ("large_decode", 1),
    "large_prefill": ("large_prefill", 1),
    "tiny": ("tiny", 1),
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# --------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def job_rate(torch, ms_local, tokens_per_rank_step, world, device):
    """Whole-job throughput of `world` replicas: the step time is the slowest
    rank's (max over ranks), the tokens are every rank's.  Returns (tokens/s,
    max ms per step)."""
    ms = float(ms_local)
    if world > 1:
        tt = torch.tensor([ms], device=device, dtype=torch.float64)
        torch.distributed.all_reduce(tt, op=torch.distributed.ReduceOp.MAX)
        ms = float(tt.item())
    return tokens_per_rank_step * world / (ms / 1e3), ms


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def file_sha(path):
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def traffic_for(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if still current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh).get(kernel_key)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or file_sha(src) != d["source_sha"]:
        return None  # kernel changed since the counters were taken
    return d


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            if self.uuid and f[1] != self.uuid:
                continue
            rows.append(f)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[6:10]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][3]) if rows[0][3].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[4]) for r in rows if r[4].replace(".", "").isdigit()), default=None)}


# --------------------------------------------------------------------------
class Workload:
    """Synthetic layers of one configuration, resident on the device."""

    def __init__(self, M, torch, name, device, layers=None):
        self.cfg_name, self.L = WORKLOADS[name]
        if layers:
            self.L = layers
        self.name = name
        cfg = S.CONFIGS[self.cfg_name]
        self.cfg = cfg
        t0 = time.time()
        self.host_w = [S.layer_weights(cfg, l) for l in range(self.L)]
        self.host_x = [S.activations(cfg, l) for l in range(self.L)]
        self.host_lg = [S.router_logits(cfg, l) for l in range(self.L)]
        log(f"[bench] generated {self.L} layer(s) of {cfg.name} in {time.time() - t0:.1f}s")
        self.layers = [M.Layer.from_numpy(w, device) for w in self.host_w]
        # every layer's activations, logits and outputs in one buffer each (the
        # layers take views), so a step's inputs and outputs move in one copy each
        self.x_all = torch.from_numpy(np.stack(self.host_x).view(np.int16)).to(device).view(torch.bfloat16)
        self.lg_all = torch.from_numpy(np.stack(self.host_lg)).to(device)
        self.out_all = torch.empty((self.L, cfg.T, cfg.d), dtype=torch.bfloat16, device=device)
        self.x = [self.x_all[l] for l in range(self.L)]
        self.lg = [self.lg_all[l] for l in range(self.L)]
        self.out = [self.out_all[l] for l in range(self.L)]
        self.ids = [torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=device) for _ in range(self.L)]
        self.calls = [M.LayerCall(layer, cfg.T, cfg.k, device=device) for layer in self.layers]
        self.weight_bytes = sum(layer.nbytes() for layer in self.layers)

    def step(self, stream, bufs=None):
        x, lg, out = (self.x_all, self.lg_all, self.out_all) if bufs is None else bufs
        for l in range(self.L):
            self.calls[l](x[l], lg[l], out[l], self.ids[l], stream=stream)

    def second_buffers(self, torch):
        """Another set of input and output buffers with the same contents, so a
        step can compute on one set while the next step's inputs arrive in the
        other."""
        return self.x_all.clone(), self.lg_all.clone(), torch.empty_like(self.out_all)

    def tokens_per_step(self):
        return self.cfg.T * self.L


def decode_kernel_name():
    """The one-kernel decode layer the library runs."""
    return "decode_fused_kernel"


def expert_bytes(cfg, which):
    """Algorithmic bytes of one expert's gate_up or down matrix (codes + fp16 scale + zero)."""
    n = (2 * cfg.f * cfg.d) if which == "gate_up" else (cfg.d * cfg.f)
    return n // 2 + 4 * (n // 128)


def measure(M, torch, wl, steps, warmup, rank, world, peaks, peak_src, want_e2e=True):
    dev = torch.device("cuda", torch.cuda.current_device())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    cfg = wl.cfg
    with torch.cuda.stream(s):
        # eager warm-up (also configures kernels and checks the error word)
        for _ in range(max(1, warmup)):
            wl.step(s)
        s.synchronize()
        for c in wl.calls:
            e = M.get_device_error(c.ws, s)
            if e != 0:
                raise RuntimeError(f"device error {M.status_str(e)}")
        # eager timing (host launch cost included)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(steps):
            wl.step(s)
        e1.record(s)
        s.synchronize()
        eager_ms = e0.elapsed_time(e1) / steps
        # one CUDA graph per step
        n0 = M.kernel_launches()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            wl.step(s)
        launches_per_step = M.kernel_launches() - n0
        for _ in range(warmup):
            g.replay()
        s.synchronize()

    # ---------------------------------------------------------- timed region
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not uuid.startswith("GPU-"):
            uuid = "GPU-" + uuid
    except Exception:
        pass
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(uuid)
    with sampler:
        time.sleep(0.3)
        with torch.cuda.stream(s):
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(s)
            for _ in range(steps):
                g.replay()
            t1.record(s)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
    value, ms = job_rate(torch, t0.elapsed_time(t1) / steps, wl.tokens_per_step(), world, dev)
    tokens = wl.tokens_per_step() * world

    # -------------------------------------- stage events of the same step (graph)
    prof = M.StageProfiler(wl.L)
    with torch.cuda.stream(s):
        with prof:
            gp = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gp, stream=s):
                wl.step(s)
        stage_sum = np.zeros(5)
        per_layer = np.zeros((wl.L, 5))
        reps = max(3, min(steps, 10))
        for _ in range(reps):
            gp.replay()
            st = np.array(prof.stage_ms())
            per_layer += st
            stage_sum += st.sum(0)
        per_layer /= reps
        stage_sum /= reps
    uniq = [len(np.unique(i.cpu().numpy())) for i in wl.ids]
    counts_R = cfg.T * cfg.k

    decode_regime = counts_R <= 64
    # the one-kernel decode layer: exactly one launch per layer
    fused = decode_regime and launches_per_step == wl.L
    if fused:
        # dominant (only) kernel: the whole layer.  Bytes = the touched experts'
        # gate_up and down matrices + x, logits, ids and out.  Its average launch
        # duration comes from the timed region itself, which holds exactly L
        # back-to-back launches per step (CUDA events on the launching stream).
        io = cfg.T * cfg.d * 2 * 2 + cfg.T * cfg.E * 4 + cfg.T * cfg.k * 4
        lay_bytes = np.array([u * (expert_bytes(cfg, "gate_up") + expert_bytes(cfg, "down")) + io for u in uniq],
                             dtype=np.float64)
        t_lay = np.full(wl.L, ms / wl.L / 1e3)
        achieved = float(lay_bytes.sum() / t_lay.sum() / 1e9)
        peak = float(peaks["hbm_gbs"])
        tr = traffic_for(decode_kernel_name().replace("_kernel", "") + "_" + wl.name)
        roofline = {"bound": "hbm", "kernel": decode_kernel_name(), "achieved": round(achieved, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": (round(tr["dram_bytes_per_launch"]) if tr else None),
                    "algorithmic_bytes_per_launch": round(float(lay_bytes.mean())),
                    "avg_launch_us": round(float(t_lay.mean() * 1e6), 2),
                    "peak_source": peak_src}
    elif decode_regime:
        # dominant kernel: gate_up GEMV; bytes = touched experts' gate+up rows
        gu_bytes = np.array([u * expert_bytes(cfg, "gate_up") + cfg.T * cfg.d * 2 for u in uniq], dtype=np.float64)
        dn_bytes = np.array([u * expert_bytes(cfg, "down") for u in uniq], dtype=np.float64)
        t_gu = per_layer[:, 2] / 1e3
        t_dn = per_layer[:, 3] / 1e3
        achieved = float(gu_bytes.sum() / t_gu.sum() / 1e9)
        peak = float(peaks["hbm_gbs"])
        pair = float((gu_bytes.sum() + dn_bytes.sum()) / (t_gu.sum() + t_dn.sum()) / 1e9)
        tr = traffic_for("gemv_gateup_decode")
        roofline = {"bound": "hbm", "kernel": "gemv_w4_kernel<gate_up>", "achieved": round(achieved, 1),
                    "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": (round(tr["dram_bytes_per_launch"]) if tr else None),
                    "algorithmic_bytes_per_launch": round(float(gu_bytes.mean())),
                    "avg_launch_us": round(float(t_gu.mean() * 1e6), 2),
                    "peak_source": peak_src,
                    "expert_gemms_pair": {"achieved": round(pair, 1), "frac": round(pair / peak, 4),
                                          "down_avg_us": round(float(t_dn.mean() * 1e6), 2)}}
    else:
        R = counts_R
        fl_gu = 2.0 * R * 2 * cfg.f * cfg.d
        fl_dn = 2.0 * R * cfg.f * cfg.d
        t_gu = per_layer[:, 2].mean() / 1e3
        t_dn = per_layer[:, 3].mean() / 1e3
        achieved = fl_gu / t_gu / 1e12
        peak = float(peaks["bf16_tflops"])
        both = (fl_gu + fl_dn) / (t_gu + t_dn) / 1e12
        tr = traffic_for("tc_gateup_" + wl.name)
        wb_gu = float(sum(uniq) / len(uniq) * expert_bytes(cfg, "gate_up"))
        wb_dn = float(sum(uniq) / len(uniq) * expert_bytes(cfg, "down"))
        # The bound follows the arithmetic intensity: FLOPs per byte of the
        # expert weights the GEMM must read, against the ridge point of the
        # measured peaks.  Few tokens per expert (P=512 over 128 or 256
        # experts) put the grouped GEMM on the HBM side of the ridge.
        hbm_peak = float(peaks["hbm_gbs"])
        intensity = fl_gu / wb_gu
        ridge = peak * 1e12 / (hbm_peak * 1e9)
        if intensity >= ridge:
            roofline = {"bound": "tensor", "kernel": "tc_grouped_kernel<gate_up>", "achieved": round(achieved, 1),
                        "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                        "traffic": (round(tr["dram_bytes_per_launch"]) if tr else None),
                        "flops_per_launch": fl_gu, "avg_launch_us": round(t_gu * 1e6, 2), "peak_source": peak_src,
                        "expert_gemms_pair": {"achieved": round(both, 1), "frac": round(both / peak, 4),
                                              "down_avg_us": round(t_dn * 1e6, 2)}}
        else:
            gbs = wb_gu / t_gu / 1e9
            gbs_pair = (wb_gu + wb_dn) / (t_gu + t_dn) / 1e9
            roofline = {"bound": "hbm", "kernel": "tc_grouped_kernel<gate_up>", "achieved": round(gbs, 1),
                        "peak": hbm_peak, "unit": "GB/s", "frac": round(gbs / hbm_peak, 4),
                        "traffic": (round(tr["dram_bytes_per_launch"]) if tr else None),
                        "algorithmic_bytes_per_launch": wb_gu, "avg_launch_us": round(t_gu * 1e6, 2),
                        "peak_source": peak_src,
                        "tensor": {"achieved_tflops": round(achieved, 1), "frac_of_bf16_peak": round(achieved / peak, 4)},
                        "expert_gemms_pair": {"achieved": round(gbs_pair, 1), "frac": round(gbs_pair / hbm_peak, 4),
                                              "down_avg_us": round(t_dn * 1e6, 2)}}
        roofline["arithmetic_intensity_flop_per_weight_byte"] = round(intensity, 1)
        roofline["ridge_flop_per_byte"] = round(ridge, 1)
        roofline["weight_bytes_touched"] = wb_gu + wb_dn
    if fused:
        # one launch holds every stage: only the bracket around it means
        # anything (its event-record nodes also stop consecutive launches from
        # overlapping, so it reads above the timed region's per-layer time)
        stages = {f"{decode_kernel_name()} (routing .. combine, event-bracketed)":
                  round(float(stage_sum[0]) * 1e3 / wl.L, 2)}
    else:
        stages = {k: round(float(v) * 1e3 / wl.L, 2) for k, v in
                  zip(["route", "permute", "gate_up", "down", "combine"], stage_sum)}

    # ------------------------------------------------------------------ e2e
    e2e = None
    if want_e2e:
        # the step's inputs and outputs as one pinned buffer each: one copy in
        # per tensor kind, one copy out
        hx = torch.from_numpy(np.stack(wl.host_x).view(np.int16)).pin_memory()
        hl = torch.from_numpy(np.stack(wl.host_lg)).pin_memory()
        ho = torch.empty((wl.L, cfg.T, cfg.d), dtype=torch.int16).pin_memory()
        h2d = hx.numel() * hx.element_size() + hl.numel() * hl.element_size()
        d2h = ho.numel() * ho.element_size()
        # serial: copy in, compute, copy out, one step after the other on one stream
        with torch.cuda.stream(s):
            def serial_step():
                wl.x_all.view(torch.int16).copy_(hx, non_blocking=True)
                wl.lg_all.copy_(hl, non_blocking=True)
                g.replay()
                ho.copy_(wl.out_all.view(torch.int16), non_blocking=True)
            for _ in range(warmup):
                serial_step()
            s.synchronize()
            if world > 1:
                torch.distributed.barrier()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(s)
            for _ in range(steps):
                serial_step()
            a1.record(s)
            s.synchronize()
        _, serial_ms = job_rate(torch, a0.elapsed_time(a1) / steps, wl.tokens_per_step(), world, dev)

        # double-buffered, as a serving loop runs it: two input/output buffer
        # sets, one graph per set; step i's inputs are copied in on a copy
        # stream while step i-1 computes, and its outputs copied out on another
        # while step i+1 computes.  Every step still copies all of its inputs
        # in and all of its outputs out inside the timed region.
        bufs = [(wl.x_all, wl.lg_all, wl.out_all), wl.second_buffers(torch)]
        hos = [ho, torch.empty_like(ho).pin_memory()]
        graphs = [g, torch.cuda.CUDAGraph()]
        with torch.cuda.stream(s):
            with torch.cuda.graph(graphs[1], stream=s):
                wl.step(s, bufs[1])
        s.synchronize()
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        in_ready, computed, out_read = ([torch.cuda.Event(), torch.cuda.Event()] for _ in range(3))
        used = [False, False]

        def pipelined_steps(n, start):
            start.record(s)
            cin.wait_event(start)
            for i in range(n):
                b = i & 1
                xb, lb, ob = bufs[b]
                with torch.cuda.stream(cin):
                    if used[b]:
                        cin.wait_event(computed[b])   # step i-2 has read this set's inputs
                    xb.view(torch.int16).copy_(hx, non_blocking=True)
                    lb.copy_(hl, non_blocking=True)
                    in_ready[b].record(cin)
                with torch.cuda.stream(s):
                    s.wait_event(in_ready[b])
                    if used[b]:
                        s.wait_event(out_read[b])     # step i-2's outputs have left
                    graphs[b].replay()
                    computed[b].record(s)
                with torch.cuda.stream(cout):
                    cout.wait_event(computed[b])
                    hos[b].copy_(ob.view(torch.int16), non_blocking=True)
                    out_read[b].record(cout)
                used[b] = True
            for b in range(2):
                if used[b]:
                    s.wait_event(out_read[b])

        pipelined_steps(warmup, torch.cuda.Event())
        s.synchronize()
        if world > 1:
            torch.distributed.barrier()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pipelined_steps(steps, a0)
        a1.record(s)
        s.synchronize()
        for hb in hos[1:]:
            if not torch.equal(hb, hos[0]):
                raise RuntimeError("the two buffer sets' outputs differ")
        e2e_value, ems = job_rate(torch, a0.elapsed_time(a1) / steps, wl.tokens_per_step(), world, dev)
        e2e = {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ems, 4),
               "serial_ms_per_step": round(serial_ms, 4),
               "path": "pinned host x/logits -> device, graph replay of moe_layer_forward x L, out -> pinned "
                       "host; double-buffered (copies of neighbouring steps overlap this step's compute)"}

    return {
        "value": value, "ms_per_step": ms, "eager_ms_per_step": eager_ms, "roofline": roofline,
        "stages_us_per_layer": stages, "gpu_launches": int(launches_per_step * steps),
        "launches_per_step": int(launches_per_step), "clocks": sampler.summary(), "e2e": e2e,
        "uniq_experts_mean": float(np.mean(uniq)),
    }


# --------------------------------------------------------------------------
def bf16_host_to_f64(t):
    """bf16 torch tensor on the host -> float64 numpy (exact)."""
    import torch
    u = t.contiguous().view(torch.int16).numpy().view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def parity_vs_oracle(gpu_out, gpu_ids, oracle_layers):
    """The step's outputs against the oracle's, per layer: max|err| / rms(ref)
    and mean|err| / mean|ref| (the worst layer of each), and whether the
    routing ids match exactly."""
    worst_max, worst_mean, ids_exact = 0.0, 0.0, True
    for l, ref, ids in oracle_layers:
        got = bf16_host_to_f64(gpu_out[l])
        err = np.abs(got - ref)
        rms = float(np.sqrt(np.mean(ref * ref)))
        worst_max = max(worst_max, float(err.max()) / rms)
        worst_mean = max(worst_mean, float(err.mean()) / float(np.mean(np.abs(ref))))
        ids_exact &= bool(np.array_equal(np.asarray(gpu_ids[l]), ids))
    return {"vs": "oracle (fp64), the layers of the CPU baseline's sample", "layers": len(oracle_layers),
            "max_err_over_rms": round(worst_max, 6), "mean_rel_err": round(worst_mean, 6),
            "routing_exact": ids_exact, "bar": {"max_err_over_rms": 2e-2, "mean_rel_err": 5e-3}}


def sampled_parity(wl, ntok):
    """The measured step's outputs of the workload's first layer against the
    oracle: routing ids of every token exactly, outputs of `ntok` sampled
    tokens within the bar (max|err|/rms of the sample, mean relative error)."""
    import oracle as O
    cfg = wl.cfg
    x, lg, W = wl.host_x[0], wl.host_lg[0], wl.host_w[0]
    ids_ref, _ = O.route_topk(lg, cfg.k)
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(cfg.T, size=min(ntok, cfg.T), replace=False))
    ref = O.layer_forward_tokens(x, lg, lambda e: {k: v[e] for k, v in W.items()}, cfg.E, cfg.d, cfg.f, cfg.k, toks)
    got = bf16_host_to_f64(wl.out[0].cpu())[toks]
    err = np.abs(got - ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return {"vs": "oracle (fp64)", "tokens": int(len(toks)), "of": int(cfg.T),
            "max_err_over_rms": round(float(err.max()) / rms, 6),
            "mean_rel_err": round(float(err.mean()) / float(np.mean(np.abs(ref))), 6),
            "routing_exact": bool(np.array_equal(wl.ids[0].cpu().numpy(), ids_ref)),
            "bar": {"max_err_over_rms": 2e-2, "mean_rel_err": 5e-3}}


def cpu_baseline(wl_name, budget_s=15.0, max_units=None, layers=None, keep=None):
    """The oracle, as it stands, on the host cores: a bounded sample of the workload.
    `layers` overrides the workload's layer count; with `keep` (a list) the
    oracle's output and routing of every whole layer it ran are appended as
    (layer, out, ids)."""
    import oracle as O
    cfg_name, L = WORKLOADS[wl_name]
    if layers:
        L = layers
    cfg = S.CONFIGS[cfg_name]
    t_used = 0.0
    tokens = 0
    layers_done = 0
    sample_desc = ""
    t_start = time.time()
    for l in range(L if cfg.T <= 64 else 1):
        W = S.layer_weights(cfg, l)
        x = S.activations(cfg, l)
        lg = S.router_logits(cfg, l)

        def ge(e, W=W):
            return {k: v[e] for k, v in W.items()}
        if cfg.T <= 64:
            t0 = time.perf_counter()
            out, mid = O.layer_forward(x, lg, ge, cfg.E, cfg.d, cfg.f, cfg.k, want_intermediates=True)
            t_used += time.perf_counter() - t0
            if keep is not None:
                keep.append((l, out, mid["ids"]))
            tokens += cfg.T
            layers_done += 1
            sample_desc = f"{layers_done} of {L} {cfg.name} layers (T={cfg.T} each), whole layer"
        else:
            # large batch: a bounded sample of tokens through the same layer
            rng = np.random.default_rng(0)
            n = 16
            toks = np.sort(rng.choice(cfg.T, size=n, replace=False))
            t0 = time.perf_counter()
            O.layer_forward_tokens(x, lg, ge, cfg.E, cfg.d, cfg.f, cfg.k, toks)
            t_used += time.perf_counter() - t0
            tokens += n
            sample_desc = f"{n} of {cfg.T} tokens of one {cfg.name} layer (all their experts)"
        if t_used >= budget_s or time.time() - t_start > 3 * budget_s:
            break
        if max_units and layers_done >= max_units:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(tokens / t_used, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample_desc, "seconds": round(t_used, 2)}


# --------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS))
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="layers per step (default: the workload's own)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    rank, world, local = dist_env()
    cfg_name, L = WORKLOADS[args.workload]
    if args.layers:
        L = args.layers
    cfg = S.CONFIGS[cfg_name]
    config = {"workload": f"{args.workload}: {cfg.name} layer x{L}, T={cfg.T}, d_model={cfg.d}, d_ff={cfg.f}, "
                          f"E={cfg.E}, top-{cfg.k}, int4 g128 (fp16 scale+zero)",
              "T": cfg.T, "layers": L, "d_model": cfg.d, "d_ff": cfg.f, "E": cfg.E, "k": cfg.k,
              "l2": "inputs larger than L2",
              "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        # The reference arm is the CPU oracle, as it stands, on the host cores.
        # Each step is a bounded sample of the same workload: one decode layer
        # (T tokens) per step, or a 16-token sample of a prefill layer.
        if rank != 0:
            return 0
        import oracle as O
        t_wall = time.time()
        big = cfg.T > 64
        rng = np.random.default_rng(0)

        def one_step(i):
            l = i % L
            W = S.layer_weights(cfg, l)
            x = S.activations(cfg, l)
            lg = S.router_logits(cfg, l)

            def ge(e, W=W):
                return {k: v[e] for k, v in W.items()}
            t0 = time.perf_counter()
            if big:
                toks = np.sort(rng.choice(cfg.T, size=16, replace=False))
                O.layer_forward_tokens(x, lg, ge, cfg.E, cfg.d, cfg.f, cfg.k, toks)
                n = 16
            else:
                O.layer_forward(x, lg, ge, cfg.E, cfg.d, cfg.f, cfg.k)
                n = cfg.T
            return time.perf_counter() - t0, n

        for i in range(args.warmup):
            one_step(i)
        times, toks = [], 0
        for i in range(args.steps):
            dt, n = one_step(args.warmup + i)
            times.append(dt)
            toks += n
        value = toks / sum(times)
        cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
        sample = (f"per step: 16 of {cfg.T} tokens of one {cfg.name} layer" if big else
                  f"per step: one of {L} {cfg.name} layers (T={cfg.T}), whole layer")
        line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(1e3 * sum(times) / len(times), 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "wall_s": round(time.time() - t_wall, 1)}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    from bit_quantized_expert_moe_gb300 import build as B
    if rank == 0:
        B.build()
    if world > 1:
        torch.distributed.barrier()
    import bit_quantized_expert_moe_gb300 as M
    peaks, peak_src = load_peaks()
    dev = torch.device("cuda", local)

    wl = Workload(M, torch, args.workload, dev, layers=args.layers or None)
    config["l2"] = (f"inputs larger than L2 ({wl.weight_bytes / 1e9:.1f} GB of distinct expert weights "
                    f"across the step; no flush needed)")
    res = measure(M, torch, wl, args.steps, args.warmup, rank, world, peaks, peak_src)
    want_base = rank == 0 and world == 1 and not args.no_cpu_baseline
    # the step's outputs and routing, compared with the oracle's below
    step_out = ([o.cpu() for o in wl.out], [i.cpu().numpy() for i in wl.ids]) if want_base else None
    n_layers = wl.L
    del wl
    torch.cuda.empty_cache()

    # Every other workload of the suite, each with its own roofline, end-to-end
    # rate, clocks and a sampled parity check against the oracle.  "prefill"
    # keeps the skewed P=4096 layer (the prefill headline); "workloads" holds
    # the 512-token prefill layer and the large decode and prefill layers.
    secondary, others = None, {}
    if not args.no_secondary and args.workload == "decode":
        for name, nl, ntok in (("skew", None, 16), ("prefill", None, 16), ("large_decode", 4, 2),
                               ("large_prefill", None, 4)):
            wl2 = Workload(M, torch, name, dev, layers=nl)
            steps2 = max(5, args.steps)
            r2 = measure(M, torch, wl2, steps2, args.warmup, rank, world, peaks, peak_src, want_e2e=True)
            entry = {"workload": f"{name}: {wl2.cfg.name} layer x{wl2.L}, T={wl2.cfg.T}, d_model={wl2.cfg.d}, "
                                 f"d_ff={wl2.cfg.f}, E={wl2.cfg.E}, top-{wl2.cfg.k}",
                     "value": round(r2["value"], 1), "unit": "tokens/s", "ms_per_step": round(r2["ms_per_step"], 4),
                     "eager_ms_per_step": round(r2["eager_ms_per_step"], 4), "roofline": r2["roofline"],
                     "stages_us_per_layer": r2["stages_us_per_layer"], "gpu_launches": r2["gpu_launches"],
                     "clocks": r2["clocks"], "e2e": r2["e2e"], "uniq_experts_mean": r2["uniq_experts_mean"]}
            if rank == 0 and world == 1 and not args.no_cpu_baseline:
                try:
                    entry["parity"] = sampled_parity(wl2, ntok)
                except Exception as e:  # the line is still printed
                    entry["parity"] = {"error": f"{type(e).__name__}: {e}"}
            if name == "skew":
                secondary = entry
            else:
                others[name] = entry
            del wl2
            torch.cuda.empty_cache()

    base = parity = None
    if want_base:
        kept = []
        base = cpu_baseline(args.workload, budget_s=12.0, layers=n_layers, keep=kept)
        try:
            parity = parity_vs_oracle(step_out[0], step_out[1], kept) if kept else None
        except Exception as e:  # the line is still printed
            parity = {"error": f"{type(e).__name__}: {e}"}

    if rank == 0:
        line = {"metric": METRIC, "value": round(res["value"], 1), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(res["ms_per_step"], 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded int4 codes, fp16 scales, bf16 N(0,1) activations, fp32 logits)",
                "config": config, "roofline": res["roofline"], "cpu_baseline": base, "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
                "eager_ms_per_step": round(res["eager_ms_per_step"], 4),
                "stages_us_per_layer": res["stages_us_per_layer"], "uniq_experts_mean": res["uniq_experts_mean"],
                "parity": parity,
                "timing": "CUDA graph of the step replayed K times between two events on its stream; "
                          "barrier + synchronize on both sides; max over ranks",
                "prefill": secondary, "workloads": others or None}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
