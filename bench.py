"""Benchmark of the fused MLA hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--quick]

One step = one pass of the hot path over one batch of synthetic input: the causal
bf16 MLA prefill B=4 H=128 S=4096 (the headline ``value``, TFLOP/s) followed by the
absorbed bf16 decode B=64 H=128 L=4096 (reported under ``decode``, KV GB/s).  The fp8
per-token-scale prefill (B=2 H=128 S=8192) and the ragged fp8 decode (B=128 H=16
q_len=2) are timed the same way and reported under ``prefill_fp8`` / ``decode_fp8``.
Inputs are seeded synthetic tensors (numpy PCG64), resident in HBM before timing.

``--impl reference`` times the fp64 CPU oracle instead, on bounded samples of the
same prefill workload, and prints the same JSON line with ``"impl": "reference"``.
With N > 1 (torchrun) every rank runs an independent replica (no collective on the
data path): ``value`` = work of all ranks / max over ranks of the elapsed time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("MLA prefill TFLOP/s (% tensor peak); MLA decode KV GB/s (% of HBM peak), 1 GB300")
HEADLINE = "prefill_b4h128s4096_bf16"
DECODE = "decode_b64h128t1l4096_bf16"
PREFILL_FP8 = "prefill_b2h128s8192_fp8"
DECODE_FP8 = "decode_b128h16t2_ragged_fp8"


def prefill_flops(B, H, S, dqk=192, dv=128, causal=True):
    pairs = S * (S + 1) // 2 if causal else S * S
    return 2.0 * B * H * pairs * (dqk + dv)


def decode_kv_bytes(inp):
    per = (inp.d_latent + inp.d_rope) * (1 if inp.fp8 else 2) + (4 if inp.fp8 else 0)
    return float(inp.cache_lens.astype("int64").sum()) * per


TENSOR_PEAKS = os.path.join(ROOT, "profiles", "tensor_peaks.json")


def peaks():
    """HBM and bf16 peaks from MEASURED_PEAKS.json (else the fallback figures); the fp8 dense
    peak from profiles/tensor_peaks.json (written by --measure-tensor-peaks on a GB300), else
    the nominal fp8:bf16 ratio of 2 times the bf16 peak."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        pk = {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
              "bf16_tflops_sustained": d.get("bf16_tflops_sustained"),
              "peak_sm_mhz": (d.get("clocks_under_load") or {}).get("sm_mhz_median"),
              "source": "measured"}
    else:
        pk = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
              "peak_sm_mhz": None, "source": "fallback"}
    pk["fp8_tflops"], pk["fp8_source"] = 2.0 * pk["bf16_tflops"], "2 x bf16 (nominal ratio)"
    if os.path.exists(TENSOR_PEAKS):
        t = json.load(open(TENSOR_PEAKS))
        if t.get("fp8_e4m3_tflops"):
            pk["fp8_tflops"], pk["fp8_source"] = t["fp8_e4m3_tflops"], "measured (profiles/tensor_peaks.json)"
    return pk


def fp8_prefill_roofline(pairs, ms, pk):
    """Both rooflines of the per-token-scale fp8 prefill.  Per visible (query, key) pair:
    Q_nope K_nope' 2*128 FLOP and P V 2*128 FLOP with fp8 inputs, Q_rope K_rope' 2*64 FLOP in
    bf16.  fp8-input roofline: the fp8 FLOP at the fp8 peak plus the rope FLOP at the bf16
    peak.  Issued-precision roofline: as the kernel issues them -- nope scores on fp8, rope on
    bf16, and P V as one f16 product (P'' = p ks in f16 against V widened to f16), at the
    16-bit rate."""
    f_nope, f_rope, f_pv = 2.0 * 128 * pairs, 2.0 * 64 * pairs, 2.0 * 128 * pairs
    t_in = (f_nope + f_pv) / (pk["fp8_tflops"] * 1e12) + f_rope / (pk["bf16_tflops"] * 1e12)
    t_issued = f_nope / (pk["fp8_tflops"] * 1e12) + (f_rope + f_pv) / (pk["bf16_tflops"] * 1e12)
    t = ms * 1e-3
    return {"flop_split": {"fp8_nope_scores": f_nope, "bf16_rope_scores": f_rope, "fp8_pv": f_pv},
            "roofline_ms_fp8_input": t_in * 1e3, "frac_fp8_input": t_in / t,
            "roofline_ms_issued": t_issued * 1e3, "frac_issued": t_issued / t,
            "target_ms_60pct_issued": t_issued * 1e3 / 0.6,
            "peaks": {"fp8_tflops": pk["fp8_tflops"], "fp8_source": pk["fp8_source"],
                      "bf16_tflops": pk["bf16_tflops"], "bf16_source": pk["source"]}}


def clock_normalised(frac, clocks, pk):
    """The roofline fraction per SM clock: frac x (clock of the peak measurement / clock of this
    run), both the median SM clock under load.  The measured peaks ran power-capped at a lower
    clock than this bench's kernels, so the plain fraction flatters a kernel that runs at the
    maximum clock."""
    if not clocks or not clocks.get("sm_mhz") or not pk.get("peak_sm_mhz"):
        return None
    return {"frac_per_clock": frac * pk["peak_sm_mhz"] / clocks["sm_mhz"],
            "run_sm_mhz": clocks["sm_mhz"], "peak_run_sm_mhz": pk["peak_sm_mhz"]}


def kernel_source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, "mla_flash_attention_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(key, src_files):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(key)
    if not d or d.get("src_sha") != kernel_source_hash(src_files):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms while running.

    Starting nvidia-smi perturbs the GPU for a while (measured: the headline prefill 2 %
    slower when the sampler starts with its timed loop), so `ready()` waits for the first
    sample before the caller times anything, and `mark()` makes the summary count only the
    samples taken after it (the timed region)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.first = 0
        self.path = os.path.join("/tmp", "mla_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def _lines(self):
        try:
            with open(self.path) as fh:
                return sum(1 for _ in fh)
        except OSError:
            return 0

    def ready(self, timeout_s=5.0):
        """Wait (up to timeout_s) until nvidia-smi has written its first sample."""
        t0 = time.time()
        while self.proc is not None and self._lines() == 0 and time.time() - t0 < timeout_s:
            time.sleep(0.05)
        return self

    def mark(self):
        """Count only the samples written from now on."""
        self.first = self._lines()
        return self

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for k, line in enumerate(open(self.path)):
            if k < self.first:
                continue
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
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- ranks

class Ranks:
    """Whole-job aggregation over the ranks of a torchrun launch (or a single process).

    Every rank runs an independent replica; the job's throughput is the work of all ranks
    divided by the slowest rank's time.
    """

    def __init__(self, dist=None, device=None):
        self.dist = dist
        self.device = device

    def _reduce(self, x, op):
        if self.dist is None:
            return float(x)
        import torch

        t = torch.tensor([float(x)], dtype=torch.float64, device=self.device)
        self.dist.all_reduce(t, op=op)
        return float(t.item())

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()
        if self.device is not None and self.device.type == "cuda":
            import torch

            torch.cuda.synchronize(self.device)

    def max(self, x):
        return x if self.dist is None else self._reduce(x, self.dist.ReduceOp.MAX)

    def sum(self, x):
        return x if self.dist is None else self._reduce(x, self.dist.ReduceOp.SUM)

    def rate(self, work_local, ms_local):
        """(sum of work over ranks) / (max over ranks of the elapsed ms), per second."""
        return self.sum(work_local) / (self.max(ms_local) * 1e-3)


# --------------------------------------------------------------------------- GPU arm

def time_calls(fn, steps, warmup, before=None):
    """Per-call CUDA-event times (ms) on the current stream (`before` runs outside the events)."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        if before is not None:
            before()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        evs.append((s, e))
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def time_graph(fn, steps, warmup, per_graph=10):
    """Mean CUDA-event time (ms) per call of `fn`, captured `per_graph` times into one CUDA
    graph that is replayed between the events (host launch cost removed, as in a serving loop
    that replays graphs)."""
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st):
            for _ in range(per_graph):
                fn()
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // per_graph)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(reps):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / (reps * per_graph)


def run_gpu(args):
    import numpy as np
    import torch

    from gen import config_inputs
    from mla_flash_attention_gb300 import binding
    from mla_flash_attention_gb300.testing import decode_to_device, prefill_to_device

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    ranks = Ranks(dist, dev)
    barrier, max_over_ranks = ranks.barrier, ranks.max

    pk = peaks()
    l2_buf = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, about 2 x L2

    def l2_flush():
        l2_buf.zero_()

    # ---------------- headline: bf16 prefill
    inp = config_inputs(HEADLINE)
    t = prefill_to_device(inp, dev)
    flops = prefill_flops(inp.B, inp.H, inp.S)

    def call_prefill():
        binding.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=True)

    barrier()
    with ClockSampler(local) as clk:
        clk.ready()
        for _ in range(args.warmup):
            call_prefill()
        torch.cuda.synchronize()
        clk.mark()
        ms = time_calls(call_prefill, args.steps, 0)
    barrier()
    ms_mean = max_over_ranks(sum(ms) / len(ms))
    clocks = clk.summary()
    launches = args.steps * 1

    # end to end through the C ABI with host buffers (pinned): H2D inputs, call, D2H outputs
    host = prefill_to_device(inp, dev, pin=True)
    dev_in = [None if x is None else torch.empty_like(x, device=dev) for x in host["args"]]
    out_h = torch.empty((inp.B, inp.S, inp.H, inp.d_v), dtype=torch.bfloat16).pin_memory()
    lse_h = torch.empty((inp.B, inp.H, inp.S), dtype=torch.float32).pin_memory()
    out_d = torch.empty_like(out_h, device=dev)
    lse_d = torch.empty_like(lse_h, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in host["args"] if x is not None)
    d2h = out_h.numel() * 2 + lse_h.numel() * 4

    # pipelined per batch element: H2D of element b+1 (copy stream), the kernel on element b
    # (current stream) and the D2H of element b-1 (second copy stream) overlap
    h2d_s, d2h_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def call_e2e():
        cur = torch.cuda.current_stream()
        h2d_s.wait_stream(cur)  # the previous call's kernels are done with the device inputs
        for bi in range(inp.B):
            with torch.cuda.stream(h2d_s):
                for d_, h_ in zip(dev_in, host["args"]):
                    if d_ is not None:
                        d_[bi:bi + 1].copy_(h_[bi:bi + 1], non_blocking=True)
            cur.wait_stream(h2d_s)
            binding.mla_prefill(*[None if x is None else x[bi:bi + 1] for x in dev_in],
                                softmax_scale=inp.softmax_scale, causal=True,
                                out=out_d[bi:bi + 1], lse=lse_d[bi:bi + 1], stream=cur)
            d2h_s.wait_stream(cur)
            with torch.cuda.stream(d2h_s):
                out_h[bi:bi + 1].copy_(out_d[bi:bi + 1], non_blocking=True)
                lse_h[bi:bi + 1].copy_(lse_d[bi:bi + 1], non_blocking=True)
        cur.wait_stream(d2h_s)

    e2e_ms = max_over_ranks(statistics.mean(time_calls(call_e2e, max(2, args.steps // 2), 1)))
    launches += (max(2, args.steps // 2) + 1) * inp.B  # e2e calls (one launch per batch element)
    del host, dev_in, out_d, lse_d, t
    torch.cuda.empty_cache()

    res = {
        "metric": METRIC, "value": ranks.rate(flops, ms_mean) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_mean,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded PCG64 N(0,1) rounded to bf16 (no dataset)",
        "config": {"workload": HEADLINE, "B": inp.B, "H": inp.H, "S": inp.S, "d_nope": 128,
                   "d_rope": 64, "d_v": 128, "causal": True, "softmax_scale": inp.softmax_scale,
                   "l2": "inputs (1.6 GB) larger than L2; no flush",
                   "parallelism": "replicas (dp%d, no collective)" % world},
    }
    src = ["prefill_sm103.cu", "sm103_ptx.cuh"]
    achieved = flops / (ms_mean * 1e-3) / 1e12
    res["roofline"] = {"kernel": "prefill", "bound": "tensor", "achieved": achieved,
                       "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                       "frac": achieved / pk["bf16_tflops"],
                       "traffic": recorded_traffic("prefill_bf16", src),
                       "peak_source": pk["source"] + " (bf16 dense, burst; of measured)"}
    res["e2e"] = {"value": ranks.rate(flops, e2e_ms) / 1e12, "unit": "TFLOP/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                  "schedule": "pinned host buffers; per batch element H2D / mla_prefill / D2H "
                              "pipelined over two copy streams"}
    res["clocks"] = clocks
    res["roofline"]["clock_normalised"] = clock_normalised(res["roofline"]["frac"], clocks, pk)

    # ---------------- decode (bf16) and the fp8 workloads
    def decode_entry(name, with_append=False):
        dinp = config_inputs(name)
        d = decode_to_device(dinp, dev)
        ws = torch.empty(binding.decode_workspace_size(dinp.B, dinp.H, dinp.T), dtype=torch.uint8,
                         device=dev)
        out = torch.empty((dinp.B, dinp.T, dinp.H, dinp.d_latent), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((dinp.B, dinp.H, dinp.T), dtype=torch.float32, device=dev)

        def call():
            binding.mla_decode(*d["args"], **d["kwargs"], softmax_scale=dinp.softmax_scale,
                               causal=True, out=out, lse=lse, workspace=ws)

        barrier()
        dms = max_over_ranks(time_graph(call, args.steps, args.warmup))
        # the same call timed one by one with L2 flushed before each (a 256 MB write outside
        # the events): per-call events include the launch of the two kernels of a call
        fms = max_over_ranks(statistics.mean(time_calls(call, args.steps, args.warmup, before=l2_flush)))
        kv = decode_kv_bytes(dinp)
        gbs = kv / (dms * 1e-3) / 1e9
        binding.check_device_error()
        res_d = {"workload": name, "ms": dms, "kv_bytes": kv, "kv_gbs": world * gbs,
                 "frac_hbm": gbs / pk["hbm_gbs"],
                 "l2": "cache (%.0f MB) larger than L2" % (kv / 1e6),
                 "timing": "CUDA graph of 10 calls replayed back to back between events (no flush)",
                 "l2_flushed": {"ms": fms, "kv_gbs": world * kv / (fms * 1e-3) / 1e9,
                                "frac_hbm": kv / (fms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                "timing": "per-call CUDA events, 256 MB written before each call"},
                 "launches_per_call": 2}
        nonlocal launches
        launches += 2 * (max(1, args.steps // 10) * 10 + args.steps)
        if with_append:
            # the step before decode: the q_len new rows of every sequence into the same cache
            c_new = torch.randn((dinp.B, dinp.T, dinp.d_latent + dinp.d_rope), device=dev).to(torch.bfloat16)
            cache, pt, lens = d["args"][2], d["args"][3], d["args"][4]

            def append():
                binding.mla_cache_append(c_new, cache, pt, lens, kv_scale=d["kwargs"]["kv_scale"])

            ams = max_over_ranks(time_graph(append, args.steps, args.warmup))
            binding.check_device_error()
            rows = dinp.B * dinp.T
            moved = rows * ((dinp.d_latent + dinp.d_rope) * (2 + (1 if dinp.fp8 else 2)) + (4 if dinp.fp8 else 0))
            res_d["cache_append"] = {"us": ams * 1e3, "rows": rows, "bytes": moved,
                                     "gbs": moved / (ams * 1e-3) / 1e9, "launches_per_call": 1}
        return res_d

    def prefill_entry(name):
        pinp = config_inputs(name)
        pt = prefill_to_device(pinp, dev)

        def call():
            binding.mla_prefill(*pt["args"], softmax_scale=pinp.softmax_scale, causal=True)

        barrier()
        pms = max_over_ranks(statistics.mean(time_calls(call, args.steps, args.warmup)))
        f = prefill_flops(pinp.B, pinp.H, pinp.S)
        tf = f / (pms * 1e-3) / 1e12
        pairs = pinp.B * pinp.H * pinp.S * (pinp.S + 1) / 2
        rl = fp8_prefill_roofline(pairs, pms, pk)
        return {"workload": name, "ms": pms, "flops": f, "tflops": world * tf, "out_dtype": "fp32",
                "roofline": {"bound": "tensor", "achieved": tf, "unit": "TFLOP/s", **rl}}

    res["decode"] = decode_entry(DECODE)

    def backward_entry():
        # gradients of the headline prefill (B4 H128 S4096 causal) for a random upstream dO:
        # the forward runs once outside the timed region, then prep + backward per call
        binp = config_inputs(HEADLINE)
        bt = prefill_to_device(binp, dev)["args"][:5]
        out, lse = binding.mla_prefill(*bt, None, None, softmax_scale=binp.softmax_scale, causal=True)
        d_out = torch.randn_like(out, dtype=torch.float32).to(torch.bfloat16)
        B_, S_, H_ = binp.B, binp.S, binp.H
        grads = (torch.empty((B_, S_, H_, 128), dtype=torch.bfloat16, device=dev),
                 torch.empty((B_, S_, H_, 64), dtype=torch.bfloat16, device=dev),
                 torch.empty((B_, S_, H_, 128), dtype=torch.bfloat16, device=dev),
                 torch.empty((B_, S_, 64), dtype=torch.float32, device=dev),
                 torch.empty((B_, S_, H_, 128), dtype=torch.bfloat16, device=dev))
        ws = torch.empty(binding.prefill_backward_workspace_size(B_, H_, S_), dtype=torch.uint8,
                         device=dev)

        def call():
            binding.mla_prefill_backward(*bt, out, lse, d_out, softmax_scale=binp.softmax_scale,
                                         causal=True, grads=grads, workspace=ws)

        barrier()
        bms = max_over_ranks(statistics.mean(time_calls(call, args.steps, args.warmup)))
        binding.check_device_error()
        # algorithmic FLOP per visible (query, key) pair: S = Q K' (192), dP = dO V' (128),
        # dV (128), dQ (192), dK (192), two FLOP per multiply-add
        f = prefill_flops(B_, H_, S_) * (192 + 128 + 128 + 192 + 192) / (192 + 128)
        tf = f / (bms * 1e-3) / 1e12
        return {"workload": "backward of " + HEADLINE, "ms": bms, "flops": f,
                "tflops": world * tf, "frac_bf16_peak": tf / pk["bf16_tflops"],
                "flop_per_pair": 2 * (192 + 128 + 128 + 192 + 192),
                "issued_flop_per_pair": 2 * (2 * 192 + 2 * 128 + 128 + 192 + 192),
                "l2": "inputs (2.7 GB) larger than L2; no flush", "launches_per_call": 3}

    res["prefill_backward"] = backward_entry()
    launches += args.steps * 3  # prep, zero fill, main
    torch.cuda.empty_cache()

    def chunked_entry():
        # chunked prefill in absorbed form: 4 sequences of 4096 tokens whose last 64 are the
        # new chunk (rows 64 x 128 heads = 64 query tiles per sequence), bf16 cache
        from gen import make_decode

        cinp = make_decode(4, 128, 64, 4096, seed=1005)
        cd = decode_to_device(cinp, dev)
        out = torch.empty((cinp.B, cinp.T, cinp.H, cinp.d_latent), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((cinp.B, cinp.H, cinp.T), dtype=torch.float32, device=dev)
        ws = torch.empty(binding.decode_workspace_size(cinp.B, cinp.H, cinp.T), dtype=torch.uint8,
                         device=dev)

        def call():
            binding.mla_decode(*cd["args"], **cd["kwargs"], softmax_scale=cinp.softmax_scale,
                               causal=True, out=out, lse=lse, workspace=ws)

        cms = max_over_ranks(time_graph(call, args.steps, args.warmup))
        binding.check_device_error()
        L = cinp.cache_lens.astype(np.int64)
        pairs = sum(int(sum(l - cinp.T + t + 1 for t in range(cinp.T))) for l in L) * cinp.H
        f = 2.0 * pairs * (cinp.d_latent + cinp.d_rope + cinp.d_latent)
        return {"workload": "chunk of 64 new tokens on 4032 cached, B4 H128, bf16 cache",
                "timing": "CUDA graph of 10 calls replayed back to back between events", "ms": cms, "flops_absorbed": f, "tflops": world * f / (cms * 1e-3) / 1e12,
                "launches_per_call": 2}

    # the absorption products either side of the bf16 decode workload (B64 T1 H128)
    evict = torch.ones(64 << 20, dtype=torch.float32, device=dev)  # 256 MB, read to evict L2

    def absorb_entry(R, H, K, N):
        x = torch.randn((R, H, K), device=dev).to(torch.bfloat16)
        w = (torch.randn((H, K, N), device=dev) / K ** 0.5).to(torch.bfloat16)
        y = torch.empty((R, H, N), dtype=torch.bfloat16, device=dev)
        ams = max_over_ranks(statistics.mean(time_calls(lambda: binding.mla_absorb(x, w, out=y),
                                                        args.steps, args.warmup, before=evict.sum)))
        moved = 2 * (R * H * K + H * K * N + R * H * N)
        return {"shape": "x [%d,%d,%d] w [%d,%d,%d]" % (R, H, K, H, K, N), "us": ams * 1e3,
                "bytes": moved, "gbs": moved / (ams * 1e-3) / 1e9,
                "frac_hbm": moved / (ams * 1e-3) / 1e9 / pk["hbm_gbs"],
                "l2": "256 MB read before each call (weights not L2-resident)"}

    res["absorb"] = {"q_nope_W_UK": absorb_entry(64, 128, 128, 512),
                     "O_latent_W_UV": absorb_entry(64, 128, 512, 128)}
    binding.check_device_error()
    launches += args.steps * 2
    if not args.quick:
        res["prefill_fp8"] = prefill_entry(PREFILL_FP8)
        res["decode_fp8"] = decode_entry(DECODE_FP8, with_append=True)
        launches += args.steps * 1 + max(1, args.steps // 10) * 10  # fp8 prefill, cache append
        res["chunked_prefill"] = chunked_entry()
        launches += 2 * max(1, args.steps // 10) * 10
    res["gpu_launches"] = launches
    if rank == 0:
        res["cpu_baseline"] = cpu_baseline(inp_name=HEADLINE, budget_s=args.cpu_seconds)
        print(json.dumps(res))
    if dist is not None:
        dist.destroy_process_group()


# --------------------------------------------------------------------------- CPU oracle

def _cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(inp_name=HEADLINE, budget_s=15.0, inp=None):
    """Time the fp64 oracle on (batch, head) slices of the prefill workload for ~budget_s."""
    import numpy as np

    import oracle
    from gen import CONFIGS, make_prefill

    c = CONFIGS[inp_name]
    if inp is None:
        # one (batch, head) slice of the workload's shape: same S, depths and distribution
        inp = make_prefill(1, 1, c["S"], fp8=c["fp8"], seed=c["seed"])
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.prefill_bh(inp, 0, 0)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    f = n * prefill_flops(1, 1, inp.S)
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": _cpu_cores(), "kind": "oracle",
            "sample": "%d x one (batch, head) slice S=%d of %s (%.1f s, numpy fp64)" % (
                n, inp.S, inp_name, dt)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from gen import CONFIGS, make_prefill

    c = CONFIGS[HEADLINE]
    inp = make_prefill(1, 1, c["S"], seed=c["seed"])
    import oracle

    for _ in range(args.warmup):
        oracle.prefill_bh(inp, 0, 0, rows=range(0, c["S"], 64))
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.prefill_bh(inp, 0, 0)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    f = prefill_flops(1, 1, c["S"])
    v = f / (ms * 1e-3) / 1e12
    world = int(os.environ.get("WORLD_SIZE", "1"))
    res = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic: seeded PCG64 N(0,1) rounded to bf16 (no dataset)",
           "config": {"workload": HEADLINE, "B": c["B"], "H": c["H"], "S": c["S"],
                      "sample": "one (batch, head) slice per step"},
           "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": _cpu_cores(),
                            "kind": "oracle",
                            "sample": "one (batch, head) slice S=%d per step, numpy fp64" % c["S"]},
           "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(res))


PROFILE_CASES = {
    # reduced workloads for ncu captures: same shapes per (batch, head) / per sequence, a few
    # hundred MB of inputs (larger than L2), 1 warm-up + 2 launches
    "prefill": dict(kind="prefill", B=1, H=64, S=4096, fp8=False, seed=1001),
    "prefill_fp8": dict(kind="prefill", B=1, H=64, S=8192, fp8=True, seed=1002),
    "decode": dict(kind="decode", B=32, H=128, T=1, lens=4096, fp8=False, seed=1003),
    "decode_fp8": dict(kind="decode", B=64, H=16, T=2, lens=("uniform", 1, 8192), fp8=True,
                       seed=1004),
    "backward": dict(kind="backward", B=1, H=64, S=4096, fp8=False, seed=1001),
}


def run_profile_case(name):
    """Run one reduced workload (for ncu); no timing, no JSON."""
    import torch

    from gen import make_decode, make_prefill
    from mla_flash_attention_gb300 import binding
    from mla_flash_attention_gb300.testing import decode_to_device, prefill_to_device

    c = PROFILE_CASES[name]
    dev = torch.device("cuda", 0)
    if c["kind"] == "prefill":
        inp = make_prefill(c["B"], c["H"], c["S"], fp8=c["fp8"], seed=c["seed"])
        t = prefill_to_device(inp, dev)
        for _ in range(3):
            binding.mla_prefill(*t["args"], softmax_scale=inp.softmax_scale, causal=True)
    elif c["kind"] == "backward":
        inp = make_prefill(c["B"], c["H"], c["S"], seed=c["seed"])
        t = prefill_to_device(inp, dev)["args"][:5]
        out, lse = binding.mla_prefill(*t, None, None, softmax_scale=inp.softmax_scale, causal=True)
        d_out = torch.randn_like(out, dtype=torch.float32).to(torch.bfloat16)
        for _ in range(3):
            binding.mla_prefill_backward(*t, out, lse, d_out, softmax_scale=inp.softmax_scale)
    else:
        inp = make_decode(c["B"], c["H"], c["T"], c["lens"], fp8=c["fp8"], seed=c["seed"])
        d = decode_to_device(inp, dev)
        for _ in range(3):
            binding.mla_decode(*d["args"], **d["kwargs"], softmax_scale=inp.softmax_scale)
    torch.cuda.synchronize()
    binding.check_device_error()


def measure_tensor_peaks():
    """Dense library-GEMM peaks on cuda:0 (8192^3, best of 10 CUDA-event timings after warm-up;
    clocks untouched and sampled): bf16 torch.matmul and fp8 e4m3 torch._scaled_mm with
    bf16 output.  Writes profiles/tensor_peaks.json."""
    import datetime

    import torch

    dev = torch.device("cuda", 0)
    n = 8192
    a = torch.randn((n, n), device=dev)
    b = torch.randn((n, n), device=dev)
    ab, bb = a.to(torch.bfloat16), b.to(torch.bfloat16)
    a8 = (a / 4).to(torch.float8_e4m3fn)
    b8 = (b / 4).to(torch.float8_e4m3fn).t()  # column-major operand
    one = torch.tensor(1.0, device=dev)

    def best(fn):
        for _ in range(5):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(10):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            ts.append(s.elapsed_time(e))
        return min(ts)

    with ClockSampler(0) as clk:
        t_bf16 = best(lambda: torch.matmul(ab, bb))
        t_fp8 = best(lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one, out_dtype=torch.bfloat16))
    f = 2.0 * n ** 3
    res = {"bf16_tflops": f / (t_bf16 * 1e-3) / 1e12, "fp8_e4m3_tflops": f / (t_fp8 * 1e-3) / 1e12,
           "how": "torch.matmul bf16 and torch._scaled_mm e4m3 (bf16 out), %d^3, best of 10 CUDA-event "
                  "timings after 5 warm-ups; clocks not changed" % n,
           "command": "python bench.py --measure-tensor-peaks",
           "clocks": clk.summary(), "torch": torch.__version__,
           "gpu": torch.cuda.get_device_name(dev),
           "when": datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%dT%H:%M:%SZ")}
    os.makedirs(os.path.dirname(TENSOR_PEAKS), exist_ok=True)
    with open(TENSOR_PEAKS, "w") as fh:
        json.dump(res, fh, indent=1)
    print(json.dumps(res))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile", choices=sorted(PROFILE_CASES),
                    help="run one reduced workload for an ncu capture and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline prefill + bf16 decode only")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--measure-tensor-peaks", action="store_true",
                    help="measure dense bf16 / fp8 library-GEMM peaks into profiles/tensor_peaks.json")
    args = ap.parse_args()
    if args.measure_tensor_peaks:
        measure_tensor_peaks()
        return
    if args.profile:
        run_profile_case(args.profile)
        return
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
