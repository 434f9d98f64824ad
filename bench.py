"""Decode-throughput benchmark of the fused layer stack (one JSON line on rank 0).

Workload: the 7B-shaped GPT-style stack (32 pre-LN layers, hidden 4096, 32
heads, FFN 16384, fp16 weights ~ N(0, 0.02), seeded synthetic), batch 1, a KV
cache of 512 positions ~ N(0, 1); each step decodes one token through all 32
layers.  Steps cycle over cache positions 512..575 (64 decode positions),
resetting the device-side sequence length every 64 steps.

A step is one ds_stack_decode_step (160 kernels, replayed as one CUDA graph).
`value` = tokens/s over the timed steps with every input already in HBM;
`e2e` = the same through ds_stack_decode_host (host input copied in, output
copied back and the stream synchronised every step).  `roofline` is the
dominant region kernel (FFN) timed alone in profile mode; `step_roofline` is
the whole step's algorithmic bytes over its time.

--impl reference times the float64 CPU oracle (oracle/) on this machine's host
cores: whole decode steps of the same stack (every layer sharing one layer's
float64 weights; the oracle's time does not depend on their values).  The
`cpu_baseline` leg does the same on a bounded number of steps.

--prefill T times a prompt chunk of T new tokens per sequence through the
7B-shaped stack (ds_stack_forward over an empty cache): tokens/s, and the
tensor-core roofline of the dominant GEMM and of the whole chunk against the
measured bf16 dense peak.

`host_us_per_call` is the host time of one ds_stack_decode_step call with the
input buffer rotating (the captured graph's x_in node is updated in place).

Multi-GPU (torchrun, N > 1): every rank runs an independent replica (its own
weights and caches; decode of independent sequences needs no exchange), the
timed region is bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
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

METRIC = "decode tokens/sec at batch 1 (7B-shaped fp16 stack); % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0
CYCLE = 64  # decode positions per pass over the cache

# Stack shapes: hidden, heads, FFN, depth, cached positions, weight bytes per
# weight (int8: one code byte + a 2-byte fp16 scale per group; `--quant-group`
# and `--mlp-extra-grouping` change the groups of the int8 stack).
MODELS = {
    "7b": dict(H=4096, nh=32, F=16384, layers=32, past=512, wbytes=2.0, wname="fp16",
               title="7B-shaped GPT-style stack"),
    "13b-int8": dict(H=5120, nh=40, F=20480, layers=40, past=1024, wbytes=1.0 + 2.0 / 64, wname="int8",
                     title="13B-shaped GPT-style stack, MoQ int8 weights"),
    "neo-2.7b": dict(H=2560, nh=20, F=10240, layers=32, past=128, wbytes=2.0, wname="fp16",
                     title="GPT-Neo-2.7B-shaped stack"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=4)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--layers", type=int, default=None, help="default: the model's depth")
    ap.add_argument("--model", default="7b", choices=sorted(MODELS),
                    help="7b: the headline fp16 stack; 13b-int8: the MoQ int8 stack; neo-2.7b: the "
                         "GPT-Neo-2.7B-shaped fp16 stack (the last two without CPU baseline)")
    ap.add_argument("--bf16", action="store_true",
                    help="bf16 weights and activations (fp16 stacks only); default fp16")
    ap.add_argument("--quant-group", type=int, default=64, choices=[64, 128],
                    help="13b-int8: MoQ group length along K of the attention matrices")
    ap.add_argument("--mlp-extra-grouping", action="store_true",
                    help="13b-int8: FFN matrices in groups of half that length")
    ap.add_argument("--prefill", type=int, default=0,
                    help="prompt chunk of this many new tokens per sequence through the 7B-shaped stack "
                         "(ds_stack_forward, empty cache); 0 = decode (the headline)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=4)
    return ap.parse_args()


def workload_config(B, layers, model="7b", wname=None, wbytes=None):
    m = MODELS[model]
    wname = wname or m["wname"]
    H, nh, F, past = m["H"], m["nh"], m["F"], m["past"]
    gb = layers * layer_bytes(H, F, wbytes if wbytes is not None else m["wbytes"]) / 1e9
    return {
        "workload": f"{m['title']}: {layers} pre-LN layers, hidden {H}, {nh} heads "
                    f"(head_dim {H // nh}), FFN {F}, GeLU(tanh), {wname} weights; batch {B}; KV cache "
                    f"{past} cached positions + {CYCLE} decode positions",
        "batch": B, "layers": layers, "hidden": H, "heads": nh, "ffn": F,
        "past": past, "decode_positions": CYCLE,
        "l2": f"inputs larger than L2: {gb:.1f} GB of weights streamed per step (L2 is 129 MB)",
        "parallelism": "replicas",
    }


def load_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBps", "hbm_copy_gbs"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def csrc_hash():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "transformer_layer_gb300", "csrc", "*"))):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, or None
    when the kernels changed since that capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        if d.get("csrc_hash") != csrc_hash():
            return None
        v = d.get("per_launch_dram_bytes", {}).get(kernel_key)
        return float(v) if v is not None else None
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [ln.strip().split(",") for ln in self.f.read().splitlines() if ln.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for i, n in enumerate(names):
                    if r[5 + i].strip().lower() == "active":
                        reasons.add(n)
            except Exception:
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def _wb(wbytes):
    """(attention matrices, FFN matrices) bytes per weight."""
    return tuple(wbytes) if isinstance(wbytes, (tuple, list)) else (wbytes, wbytes)


def layer_bytes(H, F, wbytes=2.0):
    wa, wm = _wb(wbytes)
    n_small = 3 * H + H + F + H + 4 * H
    return wa * 4 * H * H + wm * 2 * F * H + 2 * n_small


def step_bytes(H, F, layers, B, past, steps, wbytes=2.0):
    """Average algorithmic bytes of one decode step over positions past..past+CYCLE-1:
    weights + biases + LN params, K/V read (S = past + 1 + i keys), K/V write."""
    kv = 0.0
    for i in range(steps):
        S = past + 1 + (i % CYCLE)
        kv += B * layers * 2 * S * H * 2 + B * layers * 2 * H * 2
    return layers * layer_bytes(H, F, wbytes) + kv / steps


def region_bytes(H, F, B, past, wbytes=2.0):
    """Algorithmic bytes of one launch of each region kernel (weights + vectors in/out)."""
    S = past + 1 + CYCLE // 2
    wa, wm = _wb(wbytes)
    return {
        "ln_qkv": 3 * H * H * wa + 3 * H * 2 + 4 * H + B * (H * 2 + H * 4 + 2 * H * 2),
        "attention": B * (2 * S * H * 2 + H * 4 + H * 4),
        "oproj_res": H * H * wa + 2 * H + B * (H * 4 + H * 2 + H * 4),
        "ffn_up": F * H * wm + 2 * F + 4 * H + B * (H * 4 + F * 4),
        "ffn_down": H * F * wm + 2 * H + B * (F * 4 + H * 4 + H * 2),
    }


REGIONS = ("ln_qkv", "attention", "oproj_res", "ffn_up", "ffn_down")


class OracleStack:
    """The float64 CPU oracle (oracle/) running whole decode steps of the
    7B-shaped stack: every layer has its own KV cache and the output of layer l
    feeds layer l + 1.  All layers share one layer's float64 weights, converted
    once: the oracle's time does not depend on the weight values."""

    def __init__(self, B, layers):
        import numpy as np
        from transformer_layer_gb300 import inputs
        H, F, nh, d, past = 4096, 16384, 32, 128, 512
        self.B, self.layers, self.nh, self.past, self.H = B, layers, nh, past, H
        self.p = {k: v.double().numpy() for k, v in inputs.layer_params(H, F, 1002, 0, device="cpu").items()}
        self.K, self.V = [], []
        for l in range(layers):
            kc, vc = inputs.kv_cache(B, nh, past + CYCLE, d, 1002, layer=l, device="cpu")
            self.K.append(kc.double().numpy())
            self.V.append(vc.double().numpy())
        self.xs = [inputs.hidden(B, 1, H, 1002, step=i, device="cpu").double().numpy() for i in range(4)]
        self.np = np

    def step(self, i):
        """One decode step (cache position past + i % 64); returns seconds."""
        import oracle
        t0 = time.perf_counter()
        h = self.xs[i % 4]
        for l in range(self.layers):
            h = oracle.layer_forward(h, self.p, self.K[l], self.V[l], [self.past + (i % CYCLE)] * self.B, self.nh)["y"]
        return time.perf_counter() - t0


def cpu_baseline_sample(B, budget_s=10.0, layers=32):
    """The oracle, as it stands, running whole decode steps of the 7B-shaped
    stack on this host's cores; returns (tokens/s, cores, sample description)."""
    st = OracleStack(B, layers)
    times = []
    t_end = time.perf_counter() + budget_s
    while not times or (time.perf_counter() < t_end and len(times) < 16):
        times.append(st.step(len(times)))
    per_step = statistics.median(times)
    cores = len(os.sched_getaffinity(0))
    sample = (f"{len(times)} whole decode steps ({layers} layers, batch {B}, 512 cached positions) of the "
              f"float64 oracle (numpy; BLAS threads over {cores} host cores), median {per_step:.3f} s/step")
    return B / per_step, cores, sample


def max_over_ranks(x, world, device="cpu"):
    """The largest value of x over the ranks (every rank receives it)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step, steps, world, seconds):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank_step * steps * world / seconds


def run_reference(args):
    """--impl reference: the float64 CPU oracle on this host's cores (rank 0
    only), whole decode steps of the 7B-shaped stack."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    B = args.batch
    layers = args.layers if args.layers is not None else MODELS["7b"]["layers"]
    st = OracleStack(B, layers)
    for i in range(max(args.warmup, 0)):
        st.step(i)
    ts = [st.step(args.warmup + i) for i in range(args.steps)]
    per_step = sum(ts) / len(ts)
    value = B / per_step
    cores = len(os.sched_getaffinity(0))
    sample = (f"each step = one whole decode step of the float64 oracle through {layers} 7B-shaped layers "
              f"(one layer's weights shared by all layers), batch {B}, cache 512 + i positions")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1000.0, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(B, layers),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefill_flops(H, F, nh, layers, B, T, past=0):
    """FLOPs of one prompt chunk: the four GEMMs (2 per multiply-add) and
    attention (QK^T and PV: 4 d per query-key pair and head) of every layer,
    query t seeing past + t + 1 keys; per region kernel and in total."""
    M = B * T
    pairs = B * (T * past + T * (T + 1) // 2)
    reg = {"ln_qkv": 2.0 * M * 3 * H * H, "attention": 4.0 * H * pairs, "oproj_res": 2.0 * M * H * H,
           "ffn_up": 2.0 * M * F * H, "ffn_down": 2.0 * M * H * F}
    return reg, layers * sum(reg.values())


def load_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def check_device(ws, stream, what):
    """A run in which a device-side check fired (a bounded wait that gave up,
    a bounds or cache check) produced no valid result: stop without a line."""
    from transformer_layer_gb300 import ds
    code, flags = ds.ds_workspace_status(ws, stream)
    if flags != 0:
        raise SystemExit(f"bench: device status flags 0x{flags:x} after {what} (code {code}): no result reported")


def run_prefill(args, torch, dist, world, rank, local, dev):
    """--prefill T: one step = a prompt chunk of T new tokens per sequence
    through the 7B-shaped stack (ds_stack_forward; cache empty)."""
    from transformer_layer_gb300 import ds, inputs
    m = MODELS["7b"]
    B, T = args.batch, args.prefill
    L = args.layers if args.layers is not None else m["layers"]
    H, nh, F = m["H"], m["nh"], m["F"]
    act = torch.bfloat16 if args.bf16 else torch.float16
    seed = 1002 + rank
    stream = torch.cuda.Stream(device=dev)
    layers, params, kcs, vcs = [], [], [], []
    for l in range(L):
        p = inputs.layer_params(H, F, seed, l, dtype=act, device=dev)
        params.append(p)
        layers.append(ds.ds_layer_create(H, nh, F, p, act, act))
        k, v = inputs.kv_cache(B, nh, T, H // nh, seed, l, dtype=act, device=dev)
        kcs.append(k)
        vcs.append(v)
    stack = ds.ds_stack_create(layers)
    nbytes = ds.ds_layer_workspace_bytes(layers[0], B, T)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ds.ds_workspace_init(ws, nbytes, stream)
    past = torch.zeros((B,), dtype=torch.int32, device=dev)
    xs = [inputs.hidden(B, T, H, seed, step=i, dtype=act, device=dev) for i in range(2)]
    out = torch.empty_like(xs[0])
    torch.cuda.synchronize(dev)

    def step(i):
        ds.ds_stack_forward(stack, xs[i % 2], out, B, T, kcs, vcs, T, past, ws, nbytes, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = ds.ds_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
    stream.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    launches = ds.ds_launch_count() - launches0
    check_device(ws, stream, "the timed prompt chunks")
    ms_max = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    value = job_throughput(B * T, args.steps, world, ms_max / 1000.0)
    # end to end: prompt from pinned host memory, result back, synchronised
    xh = [x.cpu().pin_memory() for x in xs]
    yh = torch.empty(out.shape, dtype=act).pin_memory()
    xd = torch.empty_like(xs[0])
    torch.cuda.synchronize(dev)
    e2e_steps = max(4, min(args.steps, 16))
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        with torch.cuda.stream(stream):
            xd.copy_(xh[i % 2], non_blocking=True)
        ds.ds_stack_forward(stack, xd, out, B, T, kcs, vcs, T, past, ws, nbytes, stream)
        with torch.cuda.stream(stream):
            yh.copy_(out, non_blocking=True)
        stream.synchronize()
    e2e_value = job_throughput(B * T, e2e_steps, world, max_over_ranks(time.perf_counter() - t0, world, dev))
    check_device(ws, stream, "the end-to-end prompt chunks")
    # region kernels alone (profile mode)
    ds.ds_stack_set_profiling(stack, True)
    ds.ds_stack_region_times(stack)
    with torch.cuda.stream(stream):
        for i in range(max(1, args.profile_steps // 2)):
            step(i)
    us, _ = ds.ds_stack_region_times(stack)
    ds.ds_stack_set_profiling(stack, False)
    check_device(ws, stream, "the profiled prompt chunks")
    reg, total = prefill_flops(H, F, nh, L, B, T)
    burst, sustained, kind = load_tensor_peak()
    shares = {r: us[i] for i, r in enumerate(REGIONS)}
    dom = max(("ffn_up", "ffn_down", "ln_qkv", "oproj_res"), key=lambda r: shares[r])
    achieved = reg[dom] / (shares[dom] * 1e-6) / 1e12
    step_tf = total / (ms_max / args.steps / 1000.0) / 1e12
    line = {
        "metric": f"prefill tokens/sec ({m['title']}, prompt chunk of {T} tokens, batch {B})",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.bf16 else "f16",
        "data": "synthetic (seeded: weights N(0,0.02), biases N(0,0.01), LN gamma 1+N(0,0.1), beta N(0,0.1), "
                "inputs N(0,1))",
        "config": {"workload": f"{m['title']}: {L} pre-LN layers, hidden {H}, {nh} heads, FFN {F}; prompt "
                               f"chunk of {T} new tokens per sequence over an empty cache, batch {B}",
                   "batch": B, "layers": L, "new_tokens": T,
                   "l2": f"inputs larger than L2: {L * layer_bytes(H, F) / 1e9:.1f} GB of weights per step"},
        "roofline": {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                     "frac": achieved / burst, "peak_source": f"{kind} bf16 dense (burst; fp16 runs at the same "
                     f"tensor rate)", "flops_per_launch": reg[dom], "us_per_launch": shares[dom],
                     "traffic": None},
        "step_roofline": {"flops_per_step": total, "achieved": step_tf, "peak": sustained, "unit": "TFLOP/s",
                          "frac": step_tf / sustained, "peak_source": f"{kind} bf16 dense (sustained)"},
        "region_us": shares,
        "cpu_baseline": None,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": B * T * H * 2,
                "d2h_bytes_per_step": B * T * H * 2, "steps": e2e_steps},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ds.ds_stack_destroy(stack)
    for l in layers:
        ds.ds_layer_destroy(l)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from transformer_layer_gb300 import ds, inputs
    if args.prefill > 0:
        run_prefill(args, torch, dist, world, rank, local, dev)
        if world > 1:
            dist.destroy_process_group()
        return

    m = MODELS[args.model]
    B = args.batch
    L = args.layers if args.layers is not None else m["layers"]
    H, nh, F, past, wbytes = m["H"], m["nh"], m["F"], m["past"], m["wbytes"]
    d = H // nh
    int8 = m["wname"] == "int8"
    if args.bf16 and int8:
        raise SystemExit("--bf16 applies to the fp16 stacks")
    ga = args.quant_group
    gm = ga // 2 if args.mlp_extra_grouping else ga
    if int8:
        if gm < 64:
            raise SystemExit("--mlp-extra-grouping needs --quant-group 128")
        wbytes = (1.0 + 2.0 / ga, 1.0 + 2.0 / gm)
    elif ga != 64 or args.mlp_extra_grouping:
        raise SystemExit("--quant-group / --mlp-extra-grouping apply to the int8 stack")
    act = torch.bfloat16 if args.bf16 else torch.float16
    wname = "bf16" if args.bf16 else m["wname"]
    if int8:
        wname = f"int8 (MoQ groups of {ga}" + (f", FFN groups of {gm})" if gm != ga else ")")
    max_len = past + CYCLE
    seed = 1002 + rank
    stream = torch.cuda.Stream(device=dev)

    # ---- weights, caches, workspace (all resident in HBM before timing)
    layers, params, kcs, vcs = [], [], [], []
    for l in range(L):
        p = inputs.layer_params(H, F, seed, l, dtype=act, device=dev)
        if int8:   # MoQ codes and fp16 group scales, quantised on the device
            for k, sk, g in (("w_qkv", "s_qkv", ga), ("w_o", "s_o", ga), ("w_fc1", "s_fc1", gm),
                             ("w_fc2", "s_fc2", gm)):
                w = p[k]
                q = torch.empty(w.shape, dtype=torch.int8, device=dev)
                sc = torch.empty((w.shape[0], w.shape[1] // g), dtype=torch.float16, device=dev)
                ds.ds_quantize_int8(w, q, sc, group=g)
                p[k], p[sk] = q, sc
            torch.cuda.synchronize(dev)
        params.append(p)
        layers.append(ds.ds_layer_create(H, nh, F, p, act, torch.int8 if int8 else act, quant_group=ga,
                                         mlp_extra_grouping=int(args.mlp_extra_grouping)))
        k, v = inputs.kv_cache(B, nh, max_len, d, seed, l, dtype=act, device=dev)
        kcs.append(k)
        vcs.append(v)
    stack = ds.ds_stack_create(layers)
    nbytes = ds.ds_stack_workspace_bytes(stack, B)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    ds.ds_workspace_init(ws, nbytes, stream)
    seq = torch.full((B,), past, dtype=torch.int32, device=dev)
    seq0 = seq.clone()
    n_x = 8
    xs = [inputs.hidden(B, 1, H, seed, step=i, dtype=act, device=dev).reshape(B, H) for i in range(n_x)]
    out = torch.empty(B, H, dtype=act, device=dev)
    torch.cuda.synchronize(dev)

    def step(i):
        if i % CYCLE == 0:
            seq.copy_(seq0)
        ds.ds_stack_decode_step(stack, xs[i % n_x], out, B, kcs, vcs, max_len, seq, ws, nbytes, stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()

    # ---- timed region
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = ds.ds_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    launches = ds.ds_launch_count() - launches0
    ms = ev0.elapsed_time(ev1)
    check_device(ws, stream, "the timed decode steps")
    # host cost of one ds_stack_decode_step call (graph replay; the inputs
    # rotate over 8 buffers, so the graph's x_in node is updated each call)
    host_us = []
    with torch.cuda.stream(stream):
        for i in range(16):
            if i % CYCLE == 0:
                seq.copy_(seq0)
            t0 = time.perf_counter()
            ds.ds_stack_decode_step(stack, xs[i % n_x], out, B, kcs, vcs, max_len, seq, ws, nbytes, stream)
            host_us.append((time.perf_counter() - t0) * 1e6)
    stream.synchronize()
    ms_max = max_over_ranks(ms, world, dev)
    value = job_throughput(B, args.steps, world, ms_max / 1000.0)

    # ---- end to end through the host-buffer entry point
    xh = [x.cpu().pin_memory() for x in xs]
    yh = torch.empty(B, H, dtype=act).pin_memory()
    xd, yd = torch.empty_like(xs[0]), torch.empty_like(out)
    seq.copy_(seq0)
    torch.cuda.synchronize(dev)
    e2e_steps = max(8, min(args.steps, 64))
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        if i % CYCLE == 0 and i > 0:
            seq.copy_(seq0)
        ds.ds_stack_decode_host(stack, xh[i % n_x], yh, xd, yd, B, kcs, vcs, max_len, seq, ws, nbytes,
                                stream)
    e2e_s = time.perf_counter() - t0
    e2e_value = job_throughput(B, e2e_steps, world, max_over_ranks(e2e_s, world, dev))
    check_device(ws, stream, "the end-to-end decode steps")

    # ---- per-region kernel times (profile mode: no graph, no PDL; each kernel alone)
    ds.ds_stack_set_profiling(stack, True)
    seq.copy_(seq0)
    torch.cuda.synchronize(dev)
    ds.ds_stack_region_times(stack)
    with torch.cuda.stream(stream):
        for i in range(args.profile_steps):
            step(i + 1)   # avoid the seq reset at i % 64 == 0 on the first profiled step
    us, counts = ds.ds_stack_region_times(stack)
    ds.ds_stack_set_profiling(stack, False)
    check_device(ws, stream, "the profiled decode steps")

    peak, peak_kind = load_peak()
    rbytes = region_bytes(H, F, B, past, wbytes)
    shares = {r: us[i] for i, r in enumerate(REGIONS)}
    dom = max(("ffn_up", "ffn_down", "ln_qkv", "oproj_res"), key=lambda r: shares[r])
    dom_us = shares[dom]
    achieved = rbytes[dom] / (dom_us * 1e-6) / 1e9
    sbytes = step_bytes(H, F, L, B, past, args.steps, wbytes)
    step_gbs = sbytes / (ms_max / args.steps / 1000.0) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.model == "7b" and not args.bf16:
        v, cores, sample = cpu_baseline_sample(B, layers=L)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}

    line = {
        "metric": METRIC if (args.model == "7b" and not args.bf16) else
                  f"decode tokens/sec at batch {B} ({m['title']}, {wname}); % of HBM roofline",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if args.bf16 else "f16",
        "data": "synthetic (seeded: weights N(0,0.02), biases N(0,0.01), LN gamma 1+N(0,0.1), "
                "beta N(0,0.1), KV cache and inputs N(0,1))",
        "config": workload_config(B, L, args.model, wname, wbytes),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} HBM copy",
                     "bytes_per_launch": rbytes[dom], "us_per_launch": dom_us,
                     "traffic": ncu_traffic(dom) if args.model == "7b" and B == 1 and not args.bf16 else None},
        "step_roofline": {"bytes_per_step": sbytes, "achieved": step_gbs, "peak": peak, "unit": "GB/s",
                          "frac": step_gbs / peak, "peak_source": f"{peak_kind} HBM copy"},
        "region_us": {r: shares[r] for r in REGIONS},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": B * H * 2,
                "d2h_bytes_per_step": B * H * 2, "steps": e2e_steps},
        "gpu_launches": launches,
        "host_us_per_call": statistics.median(host_us),
        "graph_captures": ds.ds_stack_graph_captures(stack),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ds.ds_stack_destroy(stack)
    for l in layers:
        ds.ds_layer_destroy(l)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
