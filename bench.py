#!/usr/bin/env python
"""Throughput of the block-FP8 fused MoE layer on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one moe_fp8_block_forward over one batch of synthetic tokens (routing,
expert sort, activation quantisation, both grouped GEMMs with their fused
epilogues, bf16 output), inputs already resident in HBM.  The default workload
is the DeepSeek-V3-shaped prefill layer (T=4096, H=7168, I=2048, E=256, top-8,
sigmoid grouped routing); its 11.3 GB of expert weights exceed the 129 MB L2, so
no flush is needed between steps.  Under torchrun each rank runs its own replica
on its own batch (no collective on the data path): scaling is weak.

--impl reference times the CPU oracle (oracle/) on a bounded token sample of the
same workload on the host cores; it needs no GPU.
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

import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

FP8_OVER_BF16 = 2.0        # nominal dense fp8 / bf16 tensor throughput ratio
CSRC = os.path.join(ROOT, "block_fp8_mixture_topk_gb300", "csrc")
# DRAM traffic of each w13 kernel from an ncu capture (a JSON record beside the profile's summary)
# and the sources it was taken on: tile GEMM, block-scaled tile GEMM, decode-path GEMM (FP8, NVFP4)
PROFILES = {
    "tile": (os.path.join(ROOT, "profiles", "gemm_w13_dsv3.json"),
             [os.path.join(CSRC, f) for f in ("gemm.cu", "common.cuh")]),
    "tile_bs": (os.path.join(ROOT, "profiles", "gemm_bs_w13_dsv3.json"),
                [os.path.join(CSRC, f) for f in ("gemm.cu", "common.cuh")]),
    "decode": (os.path.join(ROOT, "profiles", "decode_mlp_dsv3_decode.json"),
               [os.path.join(CSRC, f) for f in ("decode.cu", "common.cuh")]),
    "nvfp4": (os.path.join(ROOT, "profiles", "decode_mlp_nvfp4_dsv3_decode.json"),
              [os.path.join(CSRC, f) for f in ("decode.cu", "common.cuh")]),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="dsv3", choices=sorted(mi.WORKLOADS))
    p.add_argument("--tokens", type=int, default=None, help="override T (decode sweeps)")
    p.add_argument("--experts", type=int, default=None, help="override E (smaller profiling cases)")
    p.add_argument("--cpu-sample", type=int, default=None, help="tokens the oracle computes")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layout", choices=["routed", "masked"], default="routed",
                   help="routed: the whole layer (default); masked: moe_fp8_block_forward_masked on rows "
                        "grouped by expert, counts from routing the workload's tokens")
    p.add_argument("--max-tokens", type=int, default=None, help="masked layout: rows per expert (default: max count)")
    p.add_argument("--scale-fmt", choices=["f32", "ue8m0", "ue8m0_packed", "mxfp8"], default="f32",
                   help="block scales: fp32 amax/448, rounded up to a power of two (FLOAT32_CEIL_UE8M0), those "
                        "UE8M0 scales packed for the block-scaled tensor-core MMA, or MXFP8 (1x32 groups and blocks, "
                        "UE8M0; block-scaled MMA); the last two on the tile GEMMs only")
    p.add_argument("--decode", choices=["auto", "off", "on"], default="auto",
                   help="expert GEMMs of small steps: decode-path kernels for up to 8 tokens (auto), never, "
                        "or whenever the step qualifies")
    p.add_argument("--no-variants", action="store_true",
                   help="skip the extra timings of the default run (the block-scaled formats on the same "
                        "workload, and the tensor-bound Qwen3-shaped workload in every FP8 scale format)")
    p.add_argument("--weights", choices=["tiled", "nk", "nvfp4"], default="tiled",
                   help="expert weights: e4m3 tile-packed at load time (default), e4m3 in the pages' [E, N, K], "
                        "or NVFP4 (e2m1 codes with e4m3 16-blocks and a global scale, packed; decode-path kernel)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d.get("bf16_tflops_sustained"),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


def describe(wl, world):
    routing = ("sigmoid + bias, n_group=%d topk_group=%d, scaling %.1f" % (wl.n_group, wl.topk_group,
                                                                           wl.routed_scaling)
               if wl.scoring == mi.SIGMOID else "softmax")
    wbytes = wl.E * 3 * wl.H * wl.I
    return {"workload": f"{wl.name}: MoE layer T={wl.T} H={wl.H} I={wl.I} E={wl.E} top-{wl.topk}, {routing}"
                        + (", renormalize" if wl.renormalize else "")
                        + (f", Zipf s={wl.zipf_s} router offsets" if wl.zipf_s else ""),
            "T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "topk": wl.topk,
            "expert_weight_bytes": wbytes,
            "l2": "inputs larger than L2" if wbytes > 129e6 else "L2 flushed between steps",
            "parallelism": f"replicas x{world}"}


def describe_weights(args):
    fmt = {"ue8m0": ", scales rounded up to powers of two (ue8m0)",
           "ue8m0_packed": ", UE8M0 scales packed for the block-scaled MMA (ue8m0_packed)",
           "mxfp8": ", MXFP8: 1x32 blocks with UE8M0 scales (block-scaled MMA)"}.get(args.scale_fmt, ", fp32 scales")
    if args.weights == "nvfp4":
        return ("NVFP4: e2m1 codes, e4m3 scale per 16 along K, fp32 global scale per expert, packed at load "
                "time (moe_nvfp4_pack_weights); activations e4m3 1x128 groups" + fmt)
    return ("e4m3 128x128 blocks, tile-packed at load time (moe_fp8_block_pack_weights)"
            if args.weights == "tiled" else "e4m3 128x128 blocks, [E, N, K] layout") + fmt


def touched_per_pass(ids, tokens_per_pass):
    """Experts touched, summed over passes of `tokens_per_pass` consecutive tokens (ids [T, k])."""
    return sum(int(torch.unique(ids[t0:t0 + tokens_per_pass]).numel())
               for t0 in range(0, ids.shape[0], tokens_per_pass))


def expert_weight_bytes(wl, nvfp4=False, packed_scales=False, mxfp8=False):
    """Bytes one expert's w13 and w2 occupy (codes and scales): (w13, both)."""
    H, I = wl.H, wl.I
    if mxfp8:
        # one UE8M0 byte per 32 weights
        w13 = 2 * I * H + 2 * I * H // 32
        return w13, w13 + H * I + H * I // 32
    if packed_scales:
        # UE8M0 scale tiles: 512 bytes per 128 weight rows and 4 K blocks
        w13 = 2 * I * H + (2 * I // 128) * -(-H // 512) * 512
        return w13, w13 + H * I + (H // 128) * -(-I // 512) * 512
    if nvfp4:
        w13 = 2 * I * H // 2 + 2 * I * H // 16 + 4
        return w13, w13 + H * I // 2 + H * I // 16 + 4
    w13 = 2 * I * H + (2 * I // 128) * (H // 128) * 4
    return w13, 3 * H * I + ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) * 4


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        self.index = ids[device_index] if device_index < len(ids) and ids[device_index].isdigit() else str(device_index)
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", self.index, "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- replicas (N > 1)
# The layer is data-parallel over tokens: every rank runs its own replica on its own batch
# (no collective on the data path); only the step time is reduced, as the maximum over ranks.

def replica_workload(wl, rank):
    """The batch rank `rank` processes: the same shapes and weights, its own seeded tokens."""
    return wl.with_(number=wl.number + 100 * rank) if rank else wl


def max_over_ranks(values, dist, device):
    """Element-wise maximum of a list of floats over all ranks (no-op without a process group)."""
    if dist is None:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(world, units_per_rank, ms):
    """Units per second processed by all ranks together in `ms` milliseconds."""
    return world * units_per_rank / (ms / 1e3)


# ----------------------------------------------------------------------------- oracle (CPU)
def oracle_inputs(wl, tokens, device, nvfp4=False):
    """CPU copies of the workload's inputs and the oracle's own quantisation of the experts
    the sampled tokens use (untimed preparation)."""
    import numpy as np
    import oracle
    if nvfp4:
        return oracle_inputs_nvfp4(wl, tokens, device)
    hidden, logits = mi.hidden(wl, device), mi.router_logits(wl, device)
    bias = mi.expert_bias(wl, device)
    okw = dict(scoring=wl.scoring, bias=None if bias is None else bias.cpu().numpy(), n_group=wl.n_group,
               topk_group=wl.topk_group, routed_scaling=wl.routed_scaling)
    ids, _ = oracle.route(logits.cpu().numpy(), wl.topk, wl.renormalize, **okw)
    experts = sorted(set(ids[tokens].reshape(-1).tolist()))
    E, H, I = wl.E, wl.H, wl.I
    w13q = np.zeros((E, 2 * I, H), np.uint8)
    w13s = np.zeros((E, 2 * I // 128, H // 128), np.float32)
    w2q = np.zeros((E, H, I), np.uint8)
    w2s = np.zeros((E, H // 128, I // 128), np.float32)
    for e in experts:
        q, s = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w13_bf16(wl, device, [e])))
        w13q[e], w13s[e] = q[0], s[0]
        q, s = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w2_bf16(wl, device, [e])))
        w2q[e], w2s[e] = q[0], s[0]
    args = (mi.bf16_bits(hidden), logits.cpu().numpy(), w13q, w13s, w2q, w2s, wl.topk, wl.renormalize)
    return args, okw, len(experts)


def oracle_inputs_nvfp4(wl, tokens, device):
    import numpy as np
    import oracle
    hidden, logits = mi.hidden(wl, device), mi.router_logits(wl, device)
    bias = mi.expert_bias(wl, device)
    okw = dict(scoring=wl.scoring, bias=None if bias is None else bias.cpu().numpy(), n_group=wl.n_group,
               topk_group=wl.topk_group, routed_scaling=wl.routed_scaling)
    ids, _ = oracle.route(logits.cpu().numpy(), wl.topk, wl.renormalize, **okw)
    experts = sorted(set(ids[tokens].reshape(-1).tolist()))
    E, H, I = wl.E, wl.H, wl.I
    w = [np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // 16), np.uint8), np.ones(E, np.float32),
         np.zeros((E, H, I // 2), np.uint8), np.zeros((E, H, I // 16), np.uint8), np.ones(E, np.float32)]
    for e in experts:
        for i, t in ((0, mi.w13_bf16(wl, device, [e])), (3, mi.w2_bf16(wl, device, [e]))):
            q, sf, gs = oracle.quant_nvfp4_bf16(mi.bf16_bits(t))
            w[i][e], w[i + 1][e], w[i + 2][e] = q[0], sf[0], gs[0]
    args = (mi.bf16_bits(hidden), logits.cpu().numpy(), *w, wl.topk, wl.renormalize)
    return args, okw, len(experts)


def default_sample(wl):
    return max(1, min(wl.T, 2 if wl.E * wl.H * wl.I > 1e9 else 16))


def time_oracle(wl, n_tokens, device, runs=1, warmup=0, nvfp4=False):
    import oracle
    tokens = list(range(n_tokens))
    args, okw, n_exp = oracle_inputs(wl, tokens, device, nvfp4)
    layer = oracle.moe_forward_nvfp4 if nvfp4 else oracle.moe_forward
    for _ in range(warmup):
        layer(*args, tokens=tokens, **okw)
    times = []
    for _ in range(runs):
        t0 = time.perf_counter()
        layer(*args, tokens=tokens, **okw)
        times.append(time.perf_counter() - t0)
    sample = (f"first {n_tokens} of {wl.T} tokens ({n_tokens * wl.topk} routed pairs over {n_exp} experts); "
              f"routing, sort and quantisation of all {wl.T} tokens included")
    return times, sample, oracle.num_threads()


def run_reference(args, wl):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    n = args.cpu_sample or default_sample(wl)
    times, sample, cores = time_oracle(wl, n, "cpu", runs=args.steps, warmup=args.warmup,
                                       nvfp4=args.weights == "nvfp4")
    ms = 1000.0 * sum(times) / len(times)
    value = n / (ms / 1000.0)
    line = {"impl": "reference", "metric": "block-FP8 fused-MoE tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": ("synthetic (seeded; weights N(0,0.02) quantised to NVFP4)" if args.weights == "nvfp4" else
                     "synthetic (seeded; weights N(0,0.02) quantised to 128x128 e4m3 blocks)"),
            "config": describe(wl, 1),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- ours (GPU)
def gemm_source_sha(mode="tile"):
    h = hashlib.sha256()
    for f in PROFILES[mode][1]:
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(wl, mode="tile", scale_fmt="f32"):
    """dram bytes per launch of the w13 GEMM (tile GEMM, block-scaled tile GEMM, decode-path kernel,
    or the decode-path kernel on NVFP4 weights) from the committed ncu record, if it was taken on the
    current kernel source for this workload and scale format; else None."""
    path = PROFILES[mode][0]
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != gemm_source_sha(mode) or rec.get("workload") != wl.name:
        return None
    if rec.get("tokens") not in (None, wl.T) or rec.get("scale_fmt", "f32") != scale_fmt:
        return None
    # a record without a token count holds the named workload's own sizes; the expert counts it
    # holds for are listed, else the named workload's
    canon = mi.WORKLOADS.get(wl.name)
    if rec.get("tokens") is None and canon is not None and wl.T != canon.T:
        return None
    if wl.E not in rec.get("experts", [canon.E if canon is not None else wl.E]):
        return None
    try:
        return float(rec["dram_bytes_per_launch_full"])
    except (KeyError, TypeError, ValueError):
        return None


def run_ours(args, wl):
    import numpy as np
    import block_fp8_mixture_topk_gb300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # inputs: each rank its own batch (seed offset by rank), weights quantised on the GPU (untimed)
    wl_r = replica_workload(wl, rank)
    hidden, logits = mi.hidden(wl_r, dev), mi.router_logits(wl_r, dev)
    bias = mi.expert_bias(wl, dev)
    rp = (moe.RoutingParams("sigmoid", wl.n_group, wl.topk_group, wl.routed_scaling, bias)
          if wl.scoring == mi.SIGMOID else moe.RoutingParams("softmax", 1, 1, wl.routed_scaling))
    E, H, I = wl.E, wl.H, wl.I
    nvfp4 = args.weights == "nvfp4"
    if nvfp4:
        # NVFP4: quantised and packed at load time, a few experts at a time (untimed)
        unit = 16 * 64 + 16 * 8
        w13q = torch.empty(E, 2 * I // 16, H // 128, unit, dtype=torch.uint8, device=dev)
        w2q = torch.empty(E, H // 16, I // 128, unit, dtype=torch.uint8, device=dev)
        w13s = torch.empty(E, dtype=torch.float32, device=dev)
        w2s = torch.empty(E, dtype=torch.float32, device=dev)
        for e0 in range(0, E, 8):
            ex = range(e0, min(E, e0 + 8))
            n = len(ex)
            q, sf, w13s[e0:e0 + n] = moe.moe_nvfp4_quant_weight(mi.w13_bf16(wl, dev, ex))
            w13q[e0:e0 + n] = moe.moe_nvfp4_pack_weights(q, sf)
            q, sf, w2s[e0:e0 + n] = moe.moe_nvfp4_quant_weight(mi.w2_bf16(wl, dev, ex))
            w2q[e0:e0 + n] = moe.moe_nvfp4_pack_weights(q, sf)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    else:
        w13q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
        w13s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        w2q = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
        w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
        wfmt = "ue8m0" if args.scale_fmt == "ue8m0_packed" else args.scale_fmt
        if args.scale_fmt == "mxfp8":
            # MXFP8 weights: 1x32 blocks, UE8M0 scale bytes, packed for the MMA (untimed, load time)
            w13s = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=dev)
            w2s = torch.empty(E, H, I // 32, dtype=torch.uint8, device=dev)
        for e0 in range(0, E, 8):
            ex = range(e0, min(E, e0 + 8))
            quant = moe.moe_mxfp8_quant_weight if args.scale_fmt == "mxfp8" else \
                (lambda w: moe.fp8_block_quant_weight(w, wfmt))
            w13q[e0:e0 + len(ex)], w13s[e0:e0 + len(ex)] = quant(mi.w13_bf16(wl, dev, ex))
            w2q[e0:e0 + len(ex)], w2s[e0:e0 + len(ex)] = quant(mi.w2_bf16(wl, dev, ex))
        if args.scale_fmt == "mxfp8":
            w13s, w2s = moe.moe_mxfp8_pack_scales(w13s), moe.moe_mxfp8_pack_scales(w2s)
        if args.scale_fmt == "ue8m0_packed":
            # load-time packing of the UE8M0 block scales for the block-scaled MMA (untimed)
            w13s, w2s = moe.moe_fp8_block_pack_scales(w13s), moe.moe_fp8_block_pack_scales(w2s)
    if args.weights == "tiled":
        # load-time conversion into the kernels' tile-packed layout (untimed, like the quantisation)
        w13q = moe.moe_fp8_block_pack_weights(w13q)
        w2q = moe.moe_fp8_block_pack_weights(w2q)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out = torch.empty(wl.T, H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, H, I, E, wl.topk), dtype=torch.uint8, device=dev)
    ids, _ = moe.moe_route_topk(logits, wl.topk, wl.renormalize, rp)
    touched = int(torch.unique(ids).numel())
    # NVFP4 steps of more than 8 tokens run 8 tokens at a time: each pass streams the experts
    # its own tokens touch
    touched_streamed = touched_per_pass(ids, 8) if args.weights == "nvfp4" else touched
    P = wl.P
    packed_scales = args.scale_fmt in ("ue8m0_packed", "mxfp8")
    if packed_scales and (nvfp4 or args.decode == "on"):
        raise SystemExit(f"--scale-fmt {args.scale_fmt} runs on the tile GEMMs: not with NVFP4 weights or --decode on")
    decode = moe.moe_fp8_block_decode_path(wl.T, H, I, wl.topk, args.decode) and not packed_scales
    if nvfp4:
        if args.decode == "off":
            raise SystemExit("NVFP4 weights run on the decode-path kernel: --decode off does not apply")
        decode = True
    # kernels per step, as the library counts them for these routing parameters and options
    layout = {"nk": moe.ops.MOE_WEIGHTS_NK, "tiled": moe.ops.MOE_WEIGHTS_TILED,
              "nvfp4": moe.ops.MOE_WEIGHTS_NVFP4}[args.weights]
    launches_per_step = moe.moe_fp8_block_forward_kernel_count(wl.T, H, I, E, wl.topk, rp, layout, args.scale_fmt,
                                                               args.decode)

    def step(events=None):
        moe.moe_fp8_block_forward(hidden, logits, w13q, w13s, w2q, w2s, wl.topk, wl.renormalize, rp, out=out,
                                  workspace=ws, events=events, scale_fmt=args.scale_fmt, decode=args.decode)

    def barrier():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        step()
    n_ev = len(moe.ops.FORWARD_STAGES) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local) if rank == 0 else None
    barrier()
    if clocks:
        clocks.start()
    torch.cuda.nvtx.range_push("moe_timed")
    t0.record()
    for i in range(args.steps):
        step(evs[i])
    t1.record()
    torch.cuda.nvtx.range_pop()
    barrier()
    eager_ms = t0.elapsed_time(t1) / args.steps
    stage_ms = {name: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs)
                for j, name in enumerate(moe.ops.FORWARD_STAGES)}

    # the same step captured once in a CUDA graph and replayed: identical kernels and work,
    # without the host's per-launch cost (the way a serving loop issues a decode step)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    barrier()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.nvtx.range_push("moe_timed_graph")
    g0.record()
    for _ in range(args.steps):
        graph.replay()
    g1.record()
    torch.cuda.nvtx.range_pop()
    barrier()
    graph_ms = g0.elapsed_time(g1) / args.steps
    clk = clocks.stop() if clocks else None
    ms = min(eager_ms, graph_ms)
    launch = "cuda_graph" if graph_ms <= eager_ms else "eager"
    if moe.moe_get_device_status(clear=True):
        raise RuntimeError("device status word set during the benchmark")

    # end to end through the public API: every step uploads its inputs from pinned host memory
    # and downloads its bf16 output, all inside the timed region.  As a serving loop would, the
    # uploads and downloads run on their own streams, double-buffered, so that step i+1's
    # upload and step i-1's download overlap step i's forward.
    comp, up, down = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    nbuf = 2
    hid_h, log_h = hidden.cpu().pin_memory(), logits.cpu().pin_memory()
    hid_d = [torch.empty_like(hidden) for _ in range(nbuf)]
    log_d = [torch.empty_like(logits) for _ in range(nbuf)]
    out_d = [torch.empty_like(out) for _ in range(nbuf)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nbuf)]
    h2d_done = [torch.cuda.Event() for _ in range(nbuf)]
    fwd_done = [torch.cuda.Event() for _ in range(nbuf)]
    d2h_done = [torch.cuda.Event() for _ in range(nbuf)]

    def e2e_run(n, start_event):
        up.wait_event(start_event)
        for i in range(n):
            b = i % nbuf
            with torch.cuda.stream(up):
                if i >= nbuf:
                    up.wait_event(fwd_done[b])          # the forward that read buffer b is done
                hid_d[b].copy_(hid_h, non_blocking=True)
                log_d[b].copy_(log_h, non_blocking=True)
                h2d_done[b].record(up)
            comp.wait_event(h2d_done[b])
            if i >= nbuf:
                comp.wait_event(d2h_done[b])            # output buffer b was downloaded
            moe.moe_fp8_block_forward(hid_d[b], log_d[b], w13q, w13s, w2q, w2s, wl.topk, wl.renormalize, rp,
                                      out=out_d[b], workspace=ws, scale_fmt=args.scale_fmt, decode=args.decode)
            fwd_done[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(fwd_done[b])
                out_h[b].copy_(out_d[b], non_blocking=True)
                d2h_done[b].record(down)
        for b in range(min(n, nbuf)):
            comp.wait_event(d2h_done[b])

    w0 = torch.cuda.Event()
    w0.record(comp)
    e2e_run(max(3, args.warmup), w0)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    e2e_run(args.steps, e0)
    e1.record(comp)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if not torch.equal(out_h[(args.steps - 1) % nbuf].to(dev), out):
        raise RuntimeError("end-to-end output differs from the device-resident run")

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    pk = peaks()
    tokens_s = whole_job_rate(world, wl.T, ms)
    flops = wl.flops()
    per_expert_w13, per_expert = expert_weight_bytes(wl, nvfp4, packed_scales, args.scale_fmt == "mxfp8")
    layer_bytes = touched * per_expert + wl.T * H * 2 * 2 + wl.T * E * 4
    # algorithmic bytes of one w13 GEMM launch: touched experts' w13 + scales, the sorted activation
    # rows and scales read once, the requantised intermediate and its scales written once
    gemm_bytes = touched * per_expert_w13 + P * (H + H // 128 * 4) + P * (I + I // 128 * 4)
    if packed_scales:
        # one scale byte per row and 128 (packed UE8M0) or 32 (MXFP8) activations
        g_act = 32 if args.scale_fmt == "mxfp8" else 128
        gemm_bytes = touched * per_expert_w13 + P * (H + H // g_act) + P * (I + I // g_act)
    gemm_flops = 4 * P * H * I
    g_ms = stage_ms["gemm_w13"]
    if decode:
        # the decode path runs both GEMMs in one kernel (timed as the w13 stage): both GEMMs'
        # weights, the activation rows read, the intermediate written and read once, the
        # weighted bf16 rows written
        gemm_bytes = (touched_streamed * per_expert + P * (H + H // 128 * 4) + 2 * P * (I + I // 128 * 4) +
                      P * H * 2)
        gemm_flops = 6 * P * H * I
        g_ms = stage_ms["gemm_w13"] + stage_ms["gemm_w2"]
    fp8_peak = pk["bf16"] * FP8_OVER_BF16
    ridge = fp8_peak * 1e12 / (pk["hbm"] * 1e9)
    if gemm_flops / gemm_bytes > ridge:
        roof = {"bound": "tensor", "achieved": gemm_flops / (g_ms / 1e3) / 1e12, "peak": fp8_peak,
                "unit": "TFLOP/s", "peak_source": f"{pk['source']} bf16 burst x {FP8_OVER_BF16} (fp8/bf16 nominal)"}
    else:
        roof = {"bound": "hbm", "achieved": gemm_bytes / (g_ms / 1e3) / 1e9, "peak": pk["hbm"], "unit": "GB/s",
                "peak_source": f"{pk['source']} copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = ("decode_mlp_kernel<nvfp4> (both GEMMs, decode path, NVFP4 weights)" if nvfp4
                      else "decode_mlp_kernel (both GEMMs, decode path)" if decode
                      else "grouped_gemm_bs_kernel<silu_mul_quant> (w13 GEMM, block-scaled MMA)" if packed_scales
                      else "grouped_gemm_kernel<silu_mul_quant> (w13 GEMM)")
    roof["algorithmic_bytes_per_launch"] = gemm_bytes
    if nvfp4 and wl.T > 8:
        # passes of 8 tokens: each pass streams the experts its own tokens touch
        roof["bytes_basis"] = "weights streamed: each 8-token pass's touched experts"
    roof["ms_per_launch"] = g_ms
    roof["traffic"] = profiled_traffic(wl, "nvfp4" if nvfp4 else "decode" if decode else "tile_bs" if packed_scales
                                       else "tile", args.scale_fmt)

    line = {"metric": "block-FP8 fused-MoE tokens/s", "value": tokens_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e4m3 (f16 MMA)" if nvfp4 else "e4m3",
            "data": ("synthetic (seeded; weights N(0,0.02) quantised to NVFP4)" if nvfp4 else
                     "synthetic (seeded; weights N(0,0.02) quantised to 128x128 e4m3 blocks)"),
            "config": describe(wl, world), "weights_layout": describe_weights(args),
            "tflops": world * flops / (ms / 1e3) / 1e12,
            "pct_fp8_peak": world * flops / (ms / 1e3) / 1e12 / fp8_peak,
            "layer_gbs": world * layer_bytes / (ms / 1e3) / 1e9,
            "ms_per_step_eager": eager_ms, "ms_per_step_graph": graph_ms, "launch": launch,
            "experts_touched": touched, "weight_bytes_touched": touched * per_expert, "decode_path": decode,
            "weight_gbs_unique": world * touched * per_expert / (ms / 1e3) / 1e9,
            "stage_ms": stage_ms, "clocks": clk,
            "e2e": {"value": whole_job_rate(world, wl.T, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": hidden.numel() * 2 + logits.numel() * 4,
                    "d2h_bytes_per_step": out.numel() * 2},
            "gpu_launches": launches_per_step * args.steps,
            "roofline": roof}
    if (world == 1 and not args.no_variants and args.scale_fmt == "f32" and args.weights == "tiled"
            and args.layout == "routed" and wl == mi.WORKLOADS["dsv3"]):
        # the same layer in the pages' Blackwell scale format (packed UE8M0) and MXFP8, both on the
        # block-scaled tensor-core MMA; and the tensor-bound Qwen3-shaped batch in every FP8 format
        del w13q, w13s, w2q, w2s
        torch.cuda.empty_cache()
        var = {}
        for fmt in ("ue8m0_packed", "mxfp8"):
            var[f"dsv3/{fmt}"] = time_variant(moe, wl, dev, fmt, args.steps, args.warmup, fp8_peak)
        q3 = mi.WORKLOADS["qwen3_skew"]
        for fmt in ("f32", "ue8m0_packed", "mxfp8"):
            var[f"qwen3_skew/{fmt}"] = time_variant(moe, q3, dev, fmt, args.steps, args.warmup, fp8_peak)
        line["variants"] = var
    if world == 1 and not args.no_cpu_baseline:
        n = args.cpu_sample or default_sample(wl)
        times, sample, cores = time_oracle(wl, n, dev, runs=1, nvfp4=nvfp4)
        line["cpu_baseline"] = {"value": n / times[0], "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    _ = np


def build_weights(moe, wl, dev, fmt):
    """Tile-packed e4m3 expert weights of a workload and their scales in scale format `fmt` (load time)."""
    E, H, I = wl.E, wl.H, wl.I
    w13q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
    w2q = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
    if fmt == "mxfp8":
        w13s = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=dev)
        w2s = torch.empty(E, H, I // 32, dtype=torch.uint8, device=dev)
        quant = moe.moe_mxfp8_quant_weight
    else:
        w13s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
        w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
        wfmt = "ue8m0" if fmt == "ue8m0_packed" else fmt
        quant = (lambda w: moe.fp8_block_quant_weight(w, wfmt))
    for e0 in range(0, E, 8):
        ex = range(e0, min(E, e0 + 8))
        w13q[e0:e0 + len(ex)], w13s[e0:e0 + len(ex)] = quant(mi.w13_bf16(wl, dev, ex))
        w2q[e0:e0 + len(ex)], w2s[e0:e0 + len(ex)] = quant(mi.w2_bf16(wl, dev, ex))
    if fmt == "mxfp8":
        w13s, w2s = moe.moe_mxfp8_pack_scales(w13s), moe.moe_mxfp8_pack_scales(w2s)
    elif fmt == "ue8m0_packed":
        w13s, w2s = moe.moe_fp8_block_pack_scales(w13s), moe.moe_fp8_block_pack_scales(w2s)
    w13q, w2q = moe.moe_fp8_block_pack_weights(w13q), moe.moe_fp8_block_pack_weights(w2q)
    torch.cuda.synchronize()
    return w13q, w13s, w2q, w2s


def time_variant(moe, wl, dev, fmt, steps, warmup, fp8_peak):
    """One workload in one scale format: CUDA-graph replay time per step, and each stage's time from
    one eager pass with events.  The weights are freed before returning."""
    w13q, w13s, w2q, w2s = build_weights(moe, wl, dev, fmt)
    hidden, logits = mi.hidden(wl, dev), mi.router_logits(wl, dev)
    bias = mi.expert_bias(wl, dev)
    rp = (moe.RoutingParams("sigmoid", wl.n_group, wl.topk_group, wl.routed_scaling, bias)
          if wl.scoring == mi.SIGMOID else moe.RoutingParams("softmax", 1, 1, wl.routed_scaling))
    out = torch.empty(wl.T, wl.H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(moe.moe_fp8_block_workspace_size(wl.T, wl.H, wl.I, wl.E, wl.topk), dtype=torch.uint8, device=dev)

    def step(events=None):
        moe.moe_fp8_block_forward(hidden, logits, w13q, w13s, w2q, w2s, wl.topk, wl.renormalize, rp, out=out,
                                  workspace=ws, events=events, scale_fmt=fmt)

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(moe.ops.FORWARD_STAGES) + 1)]
    for _ in range(warmup):
        step()
    step(evs)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    if moe.moe_get_device_status(clear=True):
        raise RuntimeError(f"device status word set during the {fmt} variant")
    stage = {name: evs[j].elapsed_time(evs[j + 1]) for j, name in enumerate(moe.ops.FORWARD_STAGES)}
    flops = wl.flops()
    res = {"ms_per_step": ms, "tokens_per_s": wl.T / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
           "pct_fp8_peak": flops / (ms / 1e3) / 1e12 / fp8_peak,
           "w13_pct_fp8_peak": 4 * wl.P * wl.H * wl.I / (stage["gemm_w13"] / 1e3) / 1e12 / fp8_peak,
           "w2_pct_fp8_peak": 2 * wl.P * wl.H * wl.I / (stage["gemm_w2"] / 1e3) / 1e12 / fp8_peak,
           "stage_ms_eager": stage}
    del w13q, w13s, w2q, w2s, ws, graph
    torch.cuda.empty_cache()
    return res


def run_masked(args, wl):
    """The expert MLP on the masked batched layout [E, M, H] (rows already grouped by expert, as
    expert-parallel dispatch delivers them): counts from routing the workload's tokens, M the
    largest count (or --max-tokens), timed as CUDA-graph replays; one GPU."""
    import numpy as np
    import block_fp8_mixture_topk_gb300 as moe
    import oracle

    if args.weights == "nvfp4":
        raise SystemExit("the masked layout takes FP8 weights (--weights tiled or nk)")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E, H, I = wl.E, wl.H, wl.I
    bias = mi.expert_bias(wl, dev)
    rp = (moe.RoutingParams("sigmoid", wl.n_group, wl.topk_group, wl.routed_scaling, bias)
          if wl.scoring == mi.SIGMOID else moe.RoutingParams("softmax", 1, 1, wl.routed_scaling))
    ids, _ = moe.moe_route_topk(mi.router_logits(wl, dev), wl.topk, wl.renormalize, rp)
    counts = torch.bincount(ids.reshape(-1).long(), minlength=E).to(torch.int32)
    M = args.max_tokens or int(counts.max().item())
    counts = counts.clamp(max=M)
    rows = int(counts.sum().item())
    touched = int((counts > 0).sum().item())
    g = torch.Generator(device=dev).manual_seed(wl.seed + 7)
    hidden = torch.randn(E, M, H, generator=g, device=dev).to(torch.bfloat16)
    w13q = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=dev)
    w13s = torch.empty(E, 2 * I // 128, H // 128, dtype=torch.float32, device=dev)
    w2q = torch.empty(E, H, I, dtype=torch.uint8, device=dev)
    w2s = torch.empty(E, H // 128, I // 128, dtype=torch.float32, device=dev)
    wfmt = "ue8m0" if args.scale_fmt == "ue8m0_packed" else args.scale_fmt
    if args.scale_fmt == "mxfp8":
        w13s = torch.empty(E, 2 * I, H // 32, dtype=torch.uint8, device=dev)
        w2s = torch.empty(E, H, I // 32, dtype=torch.uint8, device=dev)
    quant = moe.moe_mxfp8_quant_weight if args.scale_fmt == "mxfp8" else (lambda w: moe.fp8_block_quant_weight(w, wfmt))
    for e0 in range(0, E, 8):
        ex = range(e0, min(E, e0 + 8))
        w13q[e0:e0 + len(ex)], w13s[e0:e0 + len(ex)] = quant(mi.w13_bf16(wl, dev, ex))
        w2q[e0:e0 + len(ex)], w2s[e0:e0 + len(ex)] = quant(mi.w2_bf16(wl, dev, ex))
    if args.scale_fmt == "mxfp8":
        w13s, w2s = moe.moe_mxfp8_pack_scales(w13s), moe.moe_mxfp8_pack_scales(w2s)
    if args.scale_fmt == "ue8m0_packed":
        w13s, w2s = moe.moe_fp8_block_pack_scales(w13s), moe.moe_fp8_block_pack_scales(w2s)
    w13p, w2p = (moe.moe_fp8_block_pack_weights(w13q), moe.moe_fp8_block_pack_weights(w2q)) \
        if args.weights == "tiled" else (w13q, w2q)
    out = torch.empty(E, M, H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(moe.moe_fp8_block_masked_workspace_size(E, M, H, I), dtype=torch.uint8, device=dev)

    def step():
        moe.moe_fp8_block_forward_masked(hidden, counts, w13p, w13s, w2p, w2s, out=out, workspace=ws,
                                         scale_fmt=args.scale_fmt)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        graph.replay()
    t1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if moe.moe_get_device_status(clear=True):
        raise RuntimeError("device status word set during the benchmark")
    pk = peaks()
    per_expert = 3 * H * I + ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) * 4
    layer_bytes = touched * per_expert + rows * H * 2 * 2
    line = {"metric": "block-FP8 masked-layout expert rows/s", "value": rows / (ms / 1e3), "unit": "rows/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
            "data": "synthetic (seeded; counts from routing the workload's tokens)",
            "config": {**describe(wl, 1), "layout": f"masked [E={E}, M={M}, H={H}], {rows} valid rows"},
            "weights_layout": describe_weights(args), "launch": "cuda_graph",
            "tflops": 6 * rows * H * I / (ms / 1e3) / 1e12, "layer_gbs": layer_bytes / (ms / 1e3) / 1e9,
            "hbm_frac": layer_bytes / (ms / 1e3) / 1e9 / pk["hbm"], "experts_touched": touched,
            "clocks": clk, "gpu_launches": 4 * args.steps}
    if not args.no_cpu_baseline:
        # the oracle on the rows of the first two touched experts
        cnt = counts.cpu().numpy()
        sample = [int(e) for e in np.nonzero(cnt)[0][:2]]
        sub = np.zeros(E, dtype=np.int64)
        sub[sample] = cnt[sample]
        w13o = np.zeros((E, 2 * I, H), np.uint8)
        w13so = np.zeros((E, 2 * I // 128, H // 128), np.float32)
        w2o = np.zeros((E, H, I), np.uint8)
        w2so = np.zeros((E, H // 128, I // 128), np.float32)
        for e in sample:
            q, s_ = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w13_bf16(wl, dev, [e])))
            w13o[e], w13so[e] = q[0], s_[0]
            q, s_ = oracle.quant_128x128_bf16(mi.bf16_bits(mi.w2_bf16(wl, dev, [e])))
            w2o[e], w2so[e] = q[0], s_[0]
        hb = mi.bf16_bits(hidden.cpu())
        t_start = time.perf_counter()
        oracle.moe_forward_masked(hb, sub, w13o, w13so, w2o, w2so)
        dt = time.perf_counter() - t_start
        line["cpu_baseline"] = {"value": int(sub.sum()) / dt, "unit": "rows/s", "cores": oracle.num_threads(),
                                "kind": "oracle", "sample": f"{int(sub.sum())} rows of experts {sample}"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    wl = mi.WORKLOADS[args.workload]
    if args.tokens:
        wl = wl.with_tokens(args.tokens)
    if args.experts:
        wl = wl.with_(E=args.experts)
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.layout == "masked":
        run_masked(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
