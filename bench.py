"""Benchmark of one wide-beam decode step (beam_select + beam_attn_decode).

Default workload: 4 requests, prompts of 4096 tokens, 16 query / 8 kv heads of
dim 128, bf16 KV, beam_width 512, top_k 512, vocabulary 151936 with SID codes
3 x 8192, a 4M-item Zipf(1.1) catalog, fp32 logits N(0, 2) — the last of the
three decode steps, reached by running the first two for real, so every
request has 512 live beams at trie level 2 and 3 unshared tokens per beam.

One JSON line on rank 0.  `value` is beam rows per second (rows = live beams
processed per step, summed over requests and ranks) with inputs resident in
HBM; `e2e` is the same metric through the C ABI from pinned host buffers with
every step's inputs copied in and its outputs copied out inside the timed
region (as a serving loop: the next step's copy overlaps the current step's
compute; the one-step-at-a-time figure is reported beside it).
With --impl reference the CPU oracle is timed instead on a bounded sample.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "beam-decode step µs & beam-rows/s; attn+select HBM GB/s as fraction of peak"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# FP32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flop x 2.07 GHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _peak_value(d, *names):
    for n in names:
        for k, v in d.items():
            if k == n and isinstance(v, (int, float)):
                return float(v)
    return None


class Clocks:
    """nvidia-smi clock and throttle-reason samples (every 20 ms) taken from
    just before the per-kernel breakdown pass until 0.25 s after the timed
    region: the timed steps alone last only milliseconds, shorter than the
    sampler's start-up, so the samples bracket them under the same load."""

    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.p = None
        self.lines = []
        self.t = None

    def _pump(self):
        for line in self.p.stdout:
            self.lines.append(line)

    def start(self):
        import threading
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                       "-i", str(self.index), "-lms", "20"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
            return
        self.t = threading.Thread(target=self._pump, daemon=True)
        self.t.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5.0:   # the sampler is running once it has printed
            time.sleep(0.01)

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=10)
        except Exception:
            self.p.kill()
        self.t.join(timeout=5)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "every 20 ms from the breakdown pass to 0.25 s after the timed steps"}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------ GPU arm

class Step:
    """Resident inputs and state of the benchmarked decode step."""

    def __init__(self, wl, dev):
        from wide_beam_generative_gb300 import beamdec as bd
        self.bd = bd
        self.wl = wl
        self.dev = dev
        self.items = synth.catalog(wl)
        t0 = time.time()
        self.trie = bd.beam_trie_build(self.items, [wl.C] * wl.levels, wl.token_base(), wl.V) \
            if wl.levels else None
        self.t_trie_build = time.time() - t0
        R, W, T = wl.R, wl.W, wl.T
        self.step = T - 1
        self.attn = synth.attention_inputs(wl, self.step, device=dev)
        self.maxp = int(synth.prompt_lens(wl).max())
        self.ws_sel = bd.workspace(bd.beam_select_workspace_size(R, W, wl.K, wl.V), dev)
        self.ws_att = bd.workspace(bd.beam_attn_workspace_size(R, W, wl.Hq, wl.Hkv, wl.d, self.maxp,
                                                               wl.kv_dtype), dev)
        # the request's prompt K/V is fixed for its decode: e4m3 is
        # dequantised once, as a serving loop does at prefill (no-op otherwise)
        bd.beam_attn_prepare_prompt(self.attn["shared_k"], self.attn["shared_v"], self.attn["prompt_offsets"],
                                    self.maxp, W, wl.Hq, self.ws_att)
        # reach the last step's state with the real chain (untimed)
        st = dict(cum=torch.zeros((R, W), dtype=torch.float32, device=dev),
                  node=torch.zeros((R, W), dtype=torch.int32, device=dev),
                  n_live=torch.ones((R,), dtype=torch.int32, device=dev),
                  slot=torch.full((R, W, T), -1, dtype=torch.int32, device=dev))
        for t in range(self.step):
            lg = synth.logits(wl, t, device=dev)
            res = bd.beam_select(lg, st["cum"], st["node"], st["n_live"], st["slot"], self.trie, t, t,
                                 wl.K, ws=self.ws_sel)
            st = dict(cum=res["cum_out"], node=res["node_out"], n_live=res["n_live_out"],
                      slot=res["slot_out"])
            del lg
        self.state = st
        self.logits = synth.logits(wl, self.step, device=dev)
        self.out_sel = dict(tokens=torch.empty((R, W), dtype=torch.int32, device=dev),
                            parents=torch.empty((R, W), dtype=torch.int32, device=dev),
                            cum_out=torch.empty((R, W), dtype=torch.float32, device=dev),
                            lse_out=None,
                            node_out=torch.empty((R, W), dtype=torch.int32, device=dev),
                            n_live_out=torch.empty((R,), dtype=torch.int32, device=dev),
                            slot_out=torch.empty((R, W, T), dtype=torch.int32, device=dev))
        self.out_att = torch.empty((R, W, wl.Hq, wl.d),
                                   dtype=torch.float32 if wl.q_dtype == synth.F32 else torch.bfloat16,
                                   device=dev)
        torch.cuda.synchronize()

    def run(self, logits=None, q=None, state=None):
        wl, bd, s = self.wl, self.bd, self.state if state is None else state
        lg = self.logits if logits is None else logits
        o = bd.beam_select(lg, s["cum"], s["node"], s["n_live"], s["slot"], self.trie, self.step,
                           self.step, wl.K, out=self.out_sel, ws=self.ws_sel)
        a = self.attn
        bd.beam_attn_decode(a["q"] if q is None else q, a["shared_k"], a["shared_v"], a["prompt_offsets"],
                            self.maxp, a["unshared_k"], a["unshared_v"], o["slot_out"], o["n_live_out"],
                            self.step, k_scale=a["k_scale"], v_scale=a["v_scale"], out=self.out_att,
                            ws=self.ws_att, prepared=True)
        return o

    def rows(self):
        return int(self.state["n_live"].sum().item())


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (no input of the
    previous step stays cached), then read another one, so that the lines
    left in L2 are clean and the timed work does not pay the write-back of
    the flush buffer."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def algorithmic(wl, rows, kernel):
    """Algorithmic bytes or flops of one launch of `kernel` at this step."""
    G = wl.G
    L = wl.T                                   # unshared tokens per beam at the last step
    b_kv = 1 if wl.kv_dtype == synth.E4M3 else (4 if wl.kv_dtype == synth.F32 else 2)
    b_q = 4 if wl.q_dtype == synth.F32 else 2
    P = synth.prompt_lens(wl)
    if kernel == "bd_stream_select_kernel":
        # one read of every live logits row (the children gathers hit L2)
        return rows * wl.V * 4, "bytes"
    if kernel in ("bd_attn_shared_simt_kernel", "bd_attn_shared_tc_kernel"):
        return float(4 * wl.Hkv * wl.W * G * P.sum() * wl.d), "flops"
    if kernel == "bd_attn_merge_kernel":
        unshared = rows * L * wl.Hkv * wl.d * 2 * b_kv
        qo = 2 * rows * wl.Hq * wl.d * b_q
        return unshared + qo, "bytes"
    if kernel == "bd_expand_kernel":
        if not wl.levels:
            # open vocabulary: every live logits row is read in full (its
            # first pass from HBM; a row's later passes mostly hit L2)
            return rows * wl.V * 4, "bytes"
        # trie children windows (code + logit) dominate; a bound, not a count
        return rows * 2 * 4 * min(wl.K, 512), "bytes"
    if kernel == "bd_kv_e4m3_to_bf16_kernel":
        return int(synth.prompt_lens(wl).sum()) * wl.Hkv * wl.d * 2 * 3, "bytes"
    if kernel == "bd_global_kernel":
        return rows * 12, "bytes"
    return 0, "bytes"


def step_roofline(wl, rows, ms_per_step, kernels, pk, unique_slots=None):
    """The metric's second half: algorithmic HBM bytes of attention + selection
    per step (prompt KV counted once per request) over the step time, as a
    fraction of the HBM peak; and the attention alone against its binding
    roof, max(bytes / HBM peak, shared-stage flops / bf16 peak), over the
    attention kernels' time from the per-kernel breakdown."""
    P = synth.prompt_lens(wl)
    b_kv = 1 if wl.kv_dtype == synth.E4M3 else (4 if wl.kv_dtype == synth.F32 else 2)
    b_q = 4 if wl.q_dtype == synth.F32 else 2
    shared = int(P.sum()) * wl.Hkv * wl.d * 2 * b_kv
    unshared = rows * wl.T * wl.Hkv * wl.d * 2 * b_kv
    qo = 2 * rows * wl.Hq * wl.d * b_q
    attn_bytes = shared + unshared + qo
    sel_bytes = rows * wl.V * 4
    flops = 4.0 * wl.Hkv * wl.W * wl.G * P.sum() * wl.d
    hbm = _peak_value(pk, "hbm_gbs", "hbm_GBs", "hbm") or FALLBACK_PEAKS["hbm_gbs"]
    # the attention kernels run on their own (each after the selection, with
    # no other kernel beside them) for tens of microseconds: the burst peak
    tc = _peak_value(pk, "bf16_tflops", "bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops"]
    step_gbs = (attn_bytes + sel_bytes) / (ms_per_step / 1e3) / 1e9
    attn_us = sum(v["us_per_launch"] for k, v in kernels.items()
                  if k.startswith("bd_attn") or k == "bd_kv_e4m3_to_bf16_kernel")
    out = {"attn_select_bytes": attn_bytes + sel_bytes, "attn_select_gbs": round(step_gbs, 1),
           "hbm_peak_gbs": hbm, "hbm_frac": round(step_gbs / hbm, 4)}
    if attn_us > 0:
        roof_hbm_us = attn_bytes / (hbm * 1e9) * 1e6
        roof_tc_us = flops / (tc * 1e12) * 1e6
        out["attention"] = {"us": round(attn_us, 2), "bytes": attn_bytes, "flops": float(flops),
                            "hbm_frac": round(roof_hbm_us / attn_us, 4),
                            "roof_us": {"hbm": round(float(roof_hbm_us), 2), "tensor": round(float(roof_tc_us), 2)},
                            "binding": "tensor" if roof_tc_us > roof_hbm_us else "hbm",
                            "binding_frac": round(float(max(roof_hbm_us, roof_tc_us) / attn_us), 4),
                            "tensor_peak_tflops": tc, "tensor_peak": "bf16 burst (measured)"}
        if unique_slots is not None:
            # the conservative denominator: each distinct unshared K/V row the
            # live beams reference counted once (beams share ancestry)
            uniq = unique_slots * wl.Hkv * wl.d * 2 * b_kv
            ub = shared + uniq + qo
            out["attention"]["unique_slots"] = int(unique_slots)
            out["attention"]["bytes_unique_slots"] = int(ub)
            out["attention"]["hbm_frac_unique_slots"] = round(ub / (hbm * 1e9) * 1e6 / attn_us, 4)
    return out


def workload_dtype(wl):
    """The arithmetic types the step computes in for this workload."""
    names = {synth.F32: "f32", synth.BF16: "bf16", synth.E4M3: "e4m3"}
    return (f"f32 logits; {names[wl.q_dtype]} q / {names[wl.kv_dtype]} KV / {names[wl.out_dtype]} out, "
            f"f32 accumulate")


def read_traffic(kernel, workload):
    """dram bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the current source of that kernel."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.md")
    if not os.path.exists(path):
        return None
    src_for = {"bd_expand_kernel": "select.cu", "bd_global_kernel": "select.cu", "bd_stream_select_kernel": "select.cu",
               "bd_seed_kernel": "select.cu",
               "bd_kv_e4m3_to_bf16_kernel": "attn_tc.cu",
               "bd_attn_shared_simt_kernel": "attn_simt.cu", "bd_attn_shared_tc_kernel": "attn_tc.cu",
               "bd_attn_merge_kernel": "attn_merge.cu"}
    if kernel not in src_for:
        return None
    src = os.path.join(ROOT, "wide_beam_generative_gb300", "csrc", src_for[kernel])
    if not os.path.isfile(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:12]
    for line in open(path):
        f = line.strip().strip("|").split("|")
        f = [x.strip() for x in f]
        if len(f) >= 5 and f[0] == kernel and f[1] == workload and f[3] == sha:
            try:
                return float(f[2])
            except ValueError:
                return None
    return None


def gpu_arm(args, ws, rank, local):
    from wide_beam_generative_gb300 import beamdec as bd
    dev = torch.device("cuda", local)
    wl = synth.WORKLOADS[args.workload]
    if args.requests:
        wl = wl.scaled(R=args.requests, prompt_lens=None if wl.prompt_lens is None else
                       list(wl.prompt_lens[:1]) * args.requests)
    if args.beams:
        wl = wl.scaled(W=args.beams, K=min(wl.K, args.beams))
    step = Step(wl, dev)
    rows = step.rows()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush()
        step.run()
    torch.cuda.synchronize()
    assert bd.read_status(step.ws_sel) == 0 and bd.read_status(step.ws_att) == 0
    clocks = Clocks(local)
    clocks.start()
    # per-kernel breakdown: one pass of the same steps with every kernel
    # bracketed by events (outside the timed region, whose value those
    # events would slow down)
    bd.profile_enable(True)
    for _ in range(args.steps):
        flush()
        step.run()
    torch.cuda.synchronize()
    bd.profile_enable(False)
    breakdown = {k: v for k, v in bd.profile_read().items() if v[1]}
    if not breakdown:
        raise SystemExit("no kernel launches were recorded")
    dom_name = max(breakdown.items(), key=lambda kv: kv[1][0])[0]

    # The timed region: nothing but the steps between their events.  The
    # shared stage launches as a programmatic dependent of the selection
    # kernel, so its CTAs start while the selection drains; an event recorded
    # between the two kernels would make it wait, so the roofline kernel is
    # timed in a second loop of the same steps, its launches bracketed by
    # events (the step times of that loop are reported too).
    def timed_loop(kernel_events):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(ws)
        torch.cuda.synchronize()
        if kernel_events:
            bd.profile_enable(True, kernels=[dom_name])
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            step.run()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        if kernel_events:
            bd.profile_enable(False)
        barrier(ws)
        return [a.elapsed_time(b) for a, b in ev]

    times = timed_loop(False)
    times_kev = timed_loop(True)   # the roofline kernel, timed live
    clk = clocks.stop()
    prof = bd.profile_read()
    total_ms = max_over_ranks(sum(times), ws)
    ms_per_step = total_ms / args.steps
    value = rows * ws / (ms_per_step / 1e3)
    srt = sorted(times)
    dist = {"median_us": round(statistics.median(times) * 1e3, 2),
            "p90_us": round(srt[min(len(srt) - 1, int(0.9 * len(srt)))] * 1e3, 2),
            "min_us": round(srt[0] * 1e3, 2), "max_us": round(srt[-1] * 1e3, 2)}
    # distinct unshared K/V rows the live beams' slot rows reference this step
    so, nlo = step.out_sel["slot_out"], step.out_sel["n_live_out"].tolist()
    unique_slots = sum(int(torch.unique(so[r, :nlo[r], :step.step + 1]).numel()) for r in range(wl.R))
    # launches of our kernels in the timed region: the same steps as the
    # breakdown pass launch the same kernels
    launches = sum(n for _, n in breakdown.values())

    # roofline of the dominant kernel (its events ran inside the timed region)
    kname = dom_name
    kms, kn = prof[kname]
    if not kn:
        raise SystemExit("the roofline kernel was not recorded in its timed loop")
    units, kind = algorithmic(wl, rows, kname)
    pk, src = peaks()
    if kind == "bytes":
        achieved = units / (kms / kn / 1e3) / 1e9
        peak = _peak_value(pk, "hbm_gbs", "hbm_GBs", "hbm") or FALLBACK_PEAKS["hbm_gbs"]
        roof = {"bound": "hbm", "unit": "GB/s"}
    elif kname == "bd_attn_shared_simt_kernel":
        achieved = units / (kms / kn / 1e3) / 1e12
        peak = FP32_ALU_TFLOPS
        roof = {"bound": "alu", "unit": "TFLOP/s"}
        src = "derived: 152 SMs x 128 FP32 lanes x 2 x 2.07 GHz"
    else:
        achieved = units / (kms / kn / 1e3) / 1e12
        peak = _peak_value(pk, "bf16_tflops", "bf16_tflops_sustained") or FALLBACK_PEAKS["bf16_tflops"]
        roof = {"bound": "tensor", "unit": "TFLOP/s", "peak_kind": "bf16 burst"}
    roof.update(kernel=kname, achieved=round(achieved, 2), peak=peak, frac=round(achieved / peak, 4),
                traffic=read_traffic(kname, wl.name), peak_source=src,
                algorithmic_per_launch=units, launch_us=round(kms / kn * 1e3, 2),
                timing=f"CUDA events around each launch of the kernel in a second loop of the {args.steps} "
                       f"timed steps (step {round(statistics.median(times_kev) * 1e3, 2)} us median there: "
                       f"the events keep the next kernel from starting early)")
    kernels = {k: {"us_per_launch": round(ms / n * 1e3, 2), "launches": n,
                   "share": round(ms / max(1e-9, sum(x for x, _ in breakdown.values())), 4)}
               for k, (ms, n) in breakdown.items()}
    step_roof = step_roofline(wl, rows, ms_per_step, kernels, pk, unique_slots=unique_slots)

    # end-to-end through the C ABI from pinned host buffers
    e2e = None if args.no_e2e else e2e_arm(step, args, ws, flush)
    e2e_head = None if args.no_e2e else e2e_lmhead_arm(step, args, ws, flush)
    chain = None if args.no_chain else chain_arm(step, args, flush)
    gumbel = None if args.no_chain else gumbel_arm(step, args, flush)
    lmhead = None if args.no_chain else lmhead_arm(step, args, flush)
    dense = None if args.no_chain else dense_arm(step, args, flush)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "beam-rows/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "step_us": round(ms_per_step * 1e3, 2), "step_us_distribution": dist,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": workload_dtype(wl), "data": "synthetic (seeded; see synth)",
        "config": {"workload": workload_name(wl, step.step),
                   "rows_per_step_per_gpu": rows, "l2": f"flushed before each step: a {L2_FLUSH_BYTES >> 20} MB write, then a "
                         f"{L2_FLUSH_BYTES >> 20} MB read so that no dirty line of the flush is left to "
                         f"write back inside the timed step",
                   "parallelism": f"request-sharded replicas x{ws}",
                   "launch": "the attention's shared stage is a programmatic dependent of the selection "
                             "(its main loop reads only the step's Q and prompt K/V; the slot table and "
                             "live counts after the selection completes)"},
        "roofline": roof, "step_roofline": step_roof, "kernels": kernels,
        "kernels_note": "per-kernel event times from a pass of the same steps just before the timed "
                        "region (events between kernels stop the shared stage from starting while the "
                        "selection drains, so their sum exceeds the step)",
        "gpu_launches": launches, "clocks": clk, "e2e": e2e, "e2e_lmhead": e2e_head,
        "setup": {"catalog_items": int(len(step.items)) if wl.levels else 0,
                  "trie_build_s": round(step.t_trie_build, 3)},
        "chain_graph": chain, "gumbel_select": gumbel,
        "lmhead_select": lmhead, "dense_trie": dense,
    }
    if rank == 0 and not args.no_cpu_baseline:
        crows = args.cpu_rows or default_cpu_rows(wl)
        line["cpu_baseline"] = cpu_baseline(wl, crows, one_thread_rows=max(1, crows // 8))
    return line


def _e2e_loop(step, args, ws, flush, host, compute, host_outs):
    """Times a step through the public API from pinned host buffers: every
    step copies `host` to the device, runs compute(device buffers), which
    queues the device-to-host copies of the results into `host_outs`.  Timed
    two ways: one step at a time (serial), and as a serving loop that copies
    step i + 1's inputs on a second stream into a second set of device
    buffers while step i computes (pipelined; the value).  Every step's
    copies stay inside the timed region."""
    dev = step.dev
    bufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in host_outs)
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream(device=dev)

    def h2d_into(b):
        for k, v in host.items():
            bufs[b][k].copy_(v, non_blocking=True)

    def serial():
        h2d_into(0)
        compute(bufs[0])

    def pipelined(n):
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]
        copy_stream.wait_stream(stream)
        with torch.cuda.stream(copy_stream):
            h2d_into(0)
            copied[0].record(copy_stream)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                nb = b ^ 1
                with torch.cuda.stream(copy_stream):
                    if i >= 1:
                        copy_stream.wait_event(consumed[nb])   # step i - 1 is done with it
                    h2d_into(nb)
                    copied[nb].record(copy_stream)
            stream.wait_event(copied[b])
            compute(bufs[b])
            consumed[b].record(stream)
        stream.wait_stream(copy_stream)

    for _ in range(max(1, min(args.warmup, 3))):
        serial()
    torch.cuda.synchronize()
    n = max(2, min(args.steps, 10))
    times = []
    for _ in range(n):
        flush()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        serial()
        e.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(e))
    ms_serial = max_over_ranks(sum(times) / n, ws)
    pipelined(2)
    torch.cuda.synchronize()
    trials = []
    for _ in range(3):   # the host link's rate varies between runs: the median of three loops
        flush()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pipelined(n)
        e.record(stream)
        torch.cuda.synchronize()
        trials.append(a.elapsed_time(e) / n)
    ms_pipe = max_over_ranks(sorted(trials)[1], ws)
    rows = step.rows()
    # the serving loop runs whichever schedule is faster on this host
    ms = min(ms_pipe, ms_serial)
    mode = (f"pipelined over {n} steps (step i + 1's inputs copied while step i computes), median of 3"
            if ms_pipe <= ms_serial else f"one step at a time over {n} steps (faster than the pipelined loop here)")
    return {"value": round(rows * ws / (ms / 1e3), 1), "unit": "beam-rows/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 3),
            "mode": mode, "pipelined_ms_per_step": [round(x, 3) for x in trials],
            "serial_ms_per_step": round(ms_serial, 3),
            "serial_value": round(rows * ws / (ms_serial / 1e3), 1)}


def e2e_arm(step, args, ws, flush):
    """The benchmarked step end to end: each step copies its inputs (logits,
    queries, beam state) to the device, runs the selection and the
    attention, and reads the selection's outputs and the attention output
    back."""
    s = step.state
    host = {"logits": step.logits.cpu().pin_memory(), "q": step.attn["q"].cpu().pin_memory()}
    for k in ("cum", "node", "n_live", "slot"):
        host[k] = s[k].cpu().pin_memory()
    outs = ["tokens", "parents", "cum_out", "node_out", "n_live_out", "slot_out"]
    host_out = {k: torch.empty_like(step.out_sel[k], device="cpu").pin_memory() for k in outs}
    host_att = torch.empty_like(step.out_att, device="cpu").pin_memory()

    def compute(d):
        st = dict(cum=d["cum"], node=d["node"], n_live=d["n_live"], slot=d["slot"])
        step.run(logits=d["logits"], q=d["q"], state=st)
        for k in outs:
            host_out[k].copy_(step.out_sel[k], non_blocking=True)
        host_att.copy_(step.out_att, non_blocking=True)

    return _e2e_loop(step, args, ws, flush, host, compute, list(host_out.values()) + [host_att])


def e2e_lmhead_arm(step, args, ws, flush, H=2048):
    """The step with the LM head in front (N2), end to end: each step copies
    the beams' hidden states (bf16, hidden size H = 2048 as in Qwen3-1.7B),
    the queries and the beam state to the device; the head GEMM reduces every
    row to its log-sum-exp and writes only the level's window of logits (the
    whole vocabulary without a trie), the selection takes the normalisers
    (lse_in), the attention follows, and the selection's outputs and the
    attention output are read back.  The head's weight [V, H] (random, bf16)
    is resident, like any model weight.  This figure measures the library
    rather than the host link: the per-step input is H x 2 bytes per beam
    instead of V x 4."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl, dev, s = step.wl, step.dev, step.state
    rows, V = wl.R * wl.W, wl.V
    g = torch.Generator(device=dev).manual_seed(5)
    hidden = torch.randn(rows, H, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g, device=dev) * (2.0 / H ** 0.5)).to(torch.bfloat16)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    logits = torch.empty((rows, V), dtype=torch.float32, device=dev)
    ws_head = bd.workspace(bd.beam_lmhead_workspace_size(rows, V), dev)
    tb = int(wl.token_base()[step.step]) if wl.levels else 0
    win = wl.C if wl.levels else V
    host = {"hidden": hidden.cpu().pin_memory(), "q": step.attn["q"].cpu().pin_memory()}
    for k in ("cum", "node", "n_live", "slot"):
        host[k] = s[k].cpu().pin_memory()
    outs = ["tokens", "parents", "cum_out", "node_out", "n_live_out", "slot_out"]
    host_out = {k: torch.empty_like(step.out_sel[k], device="cpu").pin_memory() for k in outs}
    host_att = torch.empty_like(step.out_att, device="cpu").pin_memory()
    a = step.attn

    def compute(d):
        bd.beam_lmhead_lse(d["hidden"], w, tb, win, lse_out=lse, logits_out=logits, ws=ws_head)
        o = bd.beam_select(logits.view(wl.R, wl.W, V), d["cum"], d["node"], d["n_live"], d["slot"], step.trie,
                           step.step, step.step, wl.K, lse_in=lse.view(wl.R, wl.W), out=step.out_sel,
                           ws=step.ws_sel)
        bd.beam_attn_decode(d["q"], a["shared_k"], a["shared_v"], a["prompt_offsets"], step.maxp,
                            a["unshared_k"], a["unshared_v"], o["slot_out"], o["n_live_out"], step.step,
                            k_scale=a["k_scale"], v_scale=a["v_scale"], out=step.out_att, ws=step.ws_att,
                            prepared=True)
        for k in outs:
            host_out[k].copy_(step.out_sel[k], non_blocking=True)
        host_att.copy_(step.out_att, non_blocking=True)

    res = _e2e_loop(step, args, ws, flush, host, compute, list(host_out.values()) + [host_att])
    assert bd.read_status(step.ws_sel) == 0 and bd.read_status(ws_head) == 0
    res.update(hidden=H, window=win)
    del w, logits, ws_head
    torch.cuda.empty_cache()
    return res


def lmhead_arm(step, args, flush, H=2048):
    """The step before the selection folded in: synthetic hidden states [R*W,
    H] and LM head [V, H] (bf16, H = 2048 as in Qwen3-1.7B).  fused: the head
    GEMM reduces each row to its log-sum-exp and writes only the SID level's
    8192 logits, then the selection runs with lse_in.  materialised: the same
    GEMM writes all V logits and the selection streams them (the path of the
    main measurement)."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl, s, dev = step.wl, step.state, step.dev
    rows, V = wl.R * wl.W, wl.V
    g = torch.Generator(device=dev).manual_seed(3)
    h = torch.randn(rows, H, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g, device=dev) * (2.0 / H ** 0.5)).to(torch.bfloat16)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    logits = torch.empty((rows, V), dtype=torch.float32, device=dev)
    ws = bd.workspace(bd.beam_lmhead_workspace_size(rows, V), dev)
    tb = int(wl.token_base()[step.step]) if wl.levels else 0
    win = wl.C if wl.levels else V
    stream = torch.cuda.current_stream()

    def fused():
        bd.beam_lmhead_lse(h, w, tb, win, lse_out=lse, logits_out=logits, ws=ws)
        bd.beam_select(logits.view(wl.R, wl.W, V), s["cum"], s["node"], s["n_live"], s["slot"], step.trie,
                       step.step, step.step, wl.K, lse_in=lse.view(wl.R, wl.W), out=step.out_sel, ws=step.ws_sel)

    def materialised():
        bd.beam_lmhead_lse(h, w, 0, V, lse_out=lse, logits_out=logits, ws=ws)
        bd.beam_select(logits.view(wl.R, wl.W, V), s["cum"], s["node"], s["n_live"], s["slot"], step.trie,
                       step.step, step.step, wl.K, out=step.out_sel, ws=step.ws_sel)

    def head_only():
        bd.beam_lmhead_lse(h, w, tb, win, lse_out=lse, logits_out=logits, ws=ws)

    res = {"hidden": H, "rows": rows, "vocab": V}
    for name, fn in (("fused_us", fused), ("materialised_us", materialised), ("head_gemm_us", head_only)):
        for _ in range(3):
            flush()
            fn()
        n = max(1, min(args.steps, 10))
        times = []
        for _ in range(n):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        res[name] = round(sum(times) / n * 1e3, 1)
    res["head_tflops"] = round(2.0 * rows * H * V / (res["head_gemm_us"] * 1e-6) / 1e12, 1)
    assert bd.read_status(step.ws_sel) == 0 and bd.read_status(ws) == 0
    del h, w, logits, ws
    torch.cuda.empty_cache()
    return res


def dense_arm(step, args, flush):
    """The selection of every decode step given each row's log-sum-exp
    (lse_in, the path the fused LM head feeds), with the trie levels as CSR
    and with dense child masks where they fit (levels whose masks exceed
    1 GiB stay CSR), on resident logits; per-step microseconds.  The
    normalisers come from an untimed one-launch selection of the same step."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl, dev, trie = step.wl, step.dev, step.trie
    if trie is None:
        return None
    R, W, T = wl.R, wl.W, wl.T
    logits = [synth.logits(wl, t, device=dev) for t in range(T - 1)] + [step.logits]
    stream = torch.cuda.current_stream()

    def chain_times():
        st = dict(cum=torch.zeros((R, W), dtype=torch.float32, device=dev),
                  node=torch.zeros((R, W), dtype=torch.int32, device=dev),
                  n_live=torch.ones((R,), dtype=torch.int32, device=dev),
                  slot=torch.full((R, W, T), -1, dtype=torch.int32, device=dev))
        out = []
        for t in range(T):
            lse = bd.beam_select(logits[t], st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t,
                                 wl.K, ws=step.ws_sel)["lse_out"]
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            o = bd.beam_select(logits[t], st["cum"], st["node"], st["n_live"], st["slot"], trie, t, t, wl.K,
                               lse_in=lse, ws=step.ws_sel)
            e1.record(stream)
            torch.cuda.synchronize()
            out.append(e0.elapsed_time(e1) * 1e3)
            st = dict(cum=o["cum_out"], node=o["node_out"], n_live=o["n_live_out"], slot=o["slot_out"])
        return out

    def timed():
        for _ in range(2):
            chain_times()
        n = max(1, min(args.steps, 5))
        acc = [0.0] * T
        for _ in range(n):
            for t, x in enumerate(chain_times()):
                acc[t] += x / n
        return [round(x, 1) for x in acc]

    res = {"csr_us_per_step": timed()}
    dense_levels = []
    for lv in range(wl.levels):
        try:
            trie.make_dense(lv)
            dense_levels.append(lv)
        except bd.BeamdecError:
            pass
    res["dense_levels"] = dense_levels
    res["dense_us_per_step"] = timed()
    for lv in dense_levels:
        trie.drop_dense(lv)
    assert bd.read_status(step.ws_sel) == 0
    del logits
    torch.cuda.empty_cache()
    return res


def lmhead_only(V, rows=2048, H=2048):
    from wide_beam_generative_gb300 import beamdec as bd
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(3)
    h = torch.randn(rows, H, generator=g, device=dev).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g, device=dev) * (2.0 / H ** 0.5)).to(torch.bfloat16)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    logits = torch.empty((rows, V), dtype=torch.float32, device=dev)
    ws = bd.workspace(bd.beam_lmhead_workspace_size(rows, V), dev)
    win0, win = max(0, V - 8192), min(V, 8192)
    bd.beam_lmhead_lse(h, w, win0, win, lse_out=lse, logits_out=logits, ws=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    bd.beam_lmhead_lse(h, w, win0, win, lse_out=lse, logits_out=logits, ws=ws)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3
    assert bd.read_status(ws) == 0
    print(json.dumps({"lmhead_only": {"rows": rows, "hidden": H, "vocab": V, "us": round(us, 1),
                                      "tflops": round(2.0 * rows * H * V / (us * 1e-6) / 1e12, 1)}}))


def gumbel_arm(step, args, flush):
    """The benchmarked step's selection with temperature 1 (Gumbel top-k),
    beside the deterministic one, on the same resident inputs."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl, s = step.wl, step.state
    stream = torch.cuda.current_stream()

    def sel(temp):
        return bd.beam_select(step.logits, s["cum"], s["node"], s["n_live"], s["slot"], step.trie, step.step,
                              step.step, wl.K, out=step.out_sel, ws=step.ws_sel, temperature=temp, seed=12345)

    res = {}
    for name, temp in (("deterministic", 0.0), ("temperature_1", 1.0)):
        for _ in range(3):
            flush()
            sel(temp)
        n = max(1, min(args.steps, 10))
        times = []
        for _ in range(n):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            sel(temp)
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        res[name + "_us"] = round(sum(times) / n * 1e3, 1)
    assert bd.read_status(step.ws_sel) == 0
    return res


def chain_arm(step, args, flush):
    """All T decode steps of the workload (selection + attention each) as one
    CUDA graph replay (DecodeChain), inputs resident: the multi-step loop with
    no host work between steps.  Reported beside the per-step number."""
    from wide_beam_generative_gb300 import beamdec as bd
    wl, dev = step.wl, step.dev
    att = [step.attn] + [synth.attention_inputs(wl, t, device=dev) for t in range(1, wl.T)]
    logits = [synth.logits(wl, t, device=dev) for t in range(wl.T - 1)] + [step.logits]
    a0 = step.attn
    ch = bd.DecodeChain(logits, [x["q"] for x in att], a0["shared_k"], a0["shared_v"], a0["prompt_offsets"],
                        step.maxp, a0["unshared_k"], a0["unshared_v"], step.trie, wl.K,
                        k_scale=a0["k_scale"], v_scale=a0["v_scale"])
    for _ in range(3):
        flush()
        ch.replay()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 10))
    times = []
    stream = torch.cuda.current_stream()
    for _ in range(n):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ch.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    assert ch.status() == (0, 0)
    us = sum(times) / n * 1e3
    del ch, logits, att
    torch.cuda.empty_cache()
    return {"steps": wl.T, "us_per_chain": round(us, 1), "us_per_step": round(us / wl.T, 1),
            "note": "every decode step of the workload (1, then W live beams) as one CUDA graph; "
                    "L2 flushed before each replay"}


# ------------------------------------------------------------------------------ CPU oracle

def cpu_sample(wl, rows):
    """A bounded sample of the workload for the oracle: `rows` beams of the
    last decode step, taken request by request (W beams each), with their
    logits rows, queries and ancestry rows."""
    from oracle import trie as otrie
    items = synth.catalog(wl)
    tr = otrie.build_trie(items, wl.C) if wl.levels else None
    step = wl.T - 1
    rng = np.random.default_rng(1)
    parts = []
    left = rows
    for r in range(wl.R):
        if left <= 0:
            break
        n = min(wl.W, left)
        left -= n
        lg = synth.logit_rows(wl, step, r, 0, n).numpy()[None]
        if tr is not None:
            pick = items[rng.integers(0, len(items), n)]
            node = np.array([[tr.node_of_prefix(p[:step]) for p in pick]], np.int64)
        else:
            node = np.zeros((1, n), np.int64)
        cum = np.zeros((1, n), np.float32)
        slot = np.zeros((1, n, wl.T), np.int32)
        for t in range(step):
            slot[0, :, t] = t * wl.W + rng.integers(0, wl.W, n)
        sub = wl.scaled(R=1, prompt_lens=[int(synth.prompt_lens(wl)[r])], p_range=None)
        a = synth.attention_inputs(sub, step)

        def raw(t):
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            if t.dtype == torch.float8_e4m3fn:
                return t.view(torch.uint8).numpy()
            return t.numpy()
        inp = dict(q=raw(a["q"][:, :n]), shared_k=raw(a["shared_k"]), shared_v=raw(a["shared_v"]),
                   unshared_k=raw(a["unshared_k"]), unshared_v=raw(a["unshared_v"]),
                   k_scale=a["k_scale"].numpy(), v_scale=a["v_scale"].numpy(),
                   prompt_offsets=a["prompt_offsets"].numpy(), q_dtype=wl.q_dtype, kv_dtype=wl.kv_dtype)
        parts.append(dict(lg=lg, node=node, cum=cum, slot=slot, inp=inp, rows=n))
    return dict(parts=parts, tr=tr, step=step, rows=sum(p["rows"] for p in parts))


def cpu_run(wl, s):
    """The oracle's decode step (selection, then attention) on the sample."""
    from oracle import attention as oatt
    from oracle import select as osel
    step = s["step"]
    for p in s["parts"]:
        n = p["rows"]
        sel = osel.beam_select(p["lg"], p["cum"], p["node"], np.array([n]), p["slot"], s["tr"],
                               wl.token_base(), step, step, n, min(wl.K, n))
        oatt.attention_decode(p["inp"], sel["slot_out"], sel["n_live_out"], step)
    return s["rows"]


def default_cpu_rows(wl):
    """Rows of the oracle's timed sample: four requests' worth, bounded so
    that the sample takes about 10-30 s on 16 cores (the oracle spends about
    8 ms per row on a trie step and about 16 ms on an open-vocabulary row,
    whose candidates are the whole vocabulary)."""
    return min(4 * wl.W, 2048 if wl.levels else 1024)


def cpu_baseline(wl, rows, one_thread_rows=None):
    s = cpu_sample(wl, rows)
    t0 = time.time()
    done = cpu_run(wl, s)
    dt = time.time() - t0
    res = {"value": round(done / dt, 2), "unit": "beam-rows/s", "cores": len(os.sched_getaffinity(0)),
           "kind": "oracle", "seconds": round(dt, 2),
           "sample": f"{done} beams ({min(wl.R, (rows + wl.W - 1) // wl.W)} requests x up to {wl.W}) of the "
                     f"last decode step: float64 log-sum-exp + trie children + full sorts, float64 "
                     f"attention over prompt + ancestry (numpy; BLAS matmuls may use every core)"}
    if one_thread_rows:
        res["one_thread"] = cpu_baseline_one_thread(wl, one_thread_rows)
    return res


def cpu_baseline_one_thread(wl, rows):
    """The same oracle step on one core: a child process pinned to one CPU
    with every BLAS / OpenMP pool at one thread (set before numpy loads)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    cpu = sorted(os.sched_getaffinity(0))[0]
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-sample-only", str(rows), "--workload", wl.name,
           "--pin-cpu", str(cpu)]
    try:
        p = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
        line = [x for x in p.stdout.splitlines() if x.startswith("{")][-1]
        return json.loads(line)
    except Exception as e:   # the main figure stands without it
        return {"unavailable": f"one-thread oracle run failed: {type(e).__name__}"}


def workload_name(wl, step_idx):
    """The workload as both arms name it in `config`."""
    return (f"{wl.name}: R{wl.R} P{int(synth.prompt_lens(wl).max())} Hq{wl.Hq} Hkv{wl.Hkv} "
            f"d{wl.d} W{wl.W} K{wl.K} V{wl.V} SID {wl.levels}x{wl.C} "
            f"catalog {wl.n_items} step {step_idx + 1}/{wl.T}")


def reference_arm(args, ws, rank):
    wl = synth.WORKLOADS[args.workload]
    if rank != 0:
        return None
    s = cpu_sample(wl, args.cpu_rows or 128)
    for _ in range(args.warmup):
        cpu_run(wl, s)
    t0 = time.time()
    for _ in range(args.steps):
        cpu_run(wl, s)
    dt = (time.time() - t0) / args.steps
    v = round(s["rows"] / dt, 2)
    return {"metric": METRIC, "value": v, "unit": "beam-rows/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; see synth)",
            "impl": "reference",
            "config": {"workload": workload_name(wl, wl.T - 1),
                       "sample": f"{s['rows']} of the step's beams per timed step (a bounded sample)"},
            "cpu_baseline": {"value": v, "unit": "beam-rows/s", "cores": len(os.sched_getaffinity(0)),
                             "kind": "oracle", "sample": f"{s['rows']} beams of the last decode step"},
            "e2e": {"value": v, "unit": "beam-rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="libbeamdec")
    ap.add_argument("--workload", default="onerec17b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="beams in the oracle's sample (default 512 for cpu_baseline, 128 per reference step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--no-chain", action="store_true", help="skip the whole-chain CUDA-graph replay")
    ap.add_argument("--requests", type=int, default=None,
                    help="override the workload's request count (smaller cases for profiling)")
    ap.add_argument("--beams", type=int, default=None,
                    help="override the workload's beam width (top_k capped to it; smaller cases for profiling)")
    ap.add_argument("--lmhead-only", type=int, default=0, metavar="VOCAB",
                    help="profiling aid: run only the fused LM head (2048 rows, hidden 2048) over VOCAB "
                         "tokens, warm-up + 1 launch, and print its time")
    ap.add_argument("--cpu-sample-only", type=int, default=0, metavar="ROWS",
                    help="internal: time the oracle on ROWS beams of the workload and print one JSON object")
    ap.add_argument("--pin-cpu", type=int, default=None, help="internal: run on this one CPU core")
    args = ap.parse_args()
    if args.cpu_sample_only:
        if args.pin_cpu is not None:
            os.sched_setaffinity(0, {args.pin_cpu})
        wl = synth.WORKLOADS[args.workload]
        s = cpu_sample(wl, args.cpu_sample_only)
        t0 = time.time()
        done = cpu_run(wl, s)
        dt = time.time() - t0
        print(json.dumps({"value": round(done / dt, 2), "unit": "beam-rows/s",
                          "cores": len(os.sched_getaffinity(0)), "threads": 1, "seconds": round(dt, 2),
                          "sample": f"{done} beams of the last decode step"}))
        return
    ws, rank, local = dist_setup()
    if args.lmhead_only:
        lmhead_only(args.lmhead_only)
        return
    if args.impl == "reference":
        line = reference_arm(args, ws, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA GPU")
        line = gpu_arm(args, ws, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
