#!/usr/bin/env python3
"""Benchmark of the MoE decode layer on B300 (one JSON line on rank 0).

Default workload: full-width single MoE layer at batch 1 -- hidden 4096, 512
experts, top-4 routed (softmax renormalised over the 4) + 1 shared expert,
expert intermediate 1024, 4-bit codes with bf16 scale/bias per 64 inputs,
bf16 router; 1000 decode tokens with x ~ N(0, 1).  One step = those 1000
tokens, each one moe_layer_decode call at B = 1 (one fused kernel launch),
replayed from a CUDA graph.  Inputs: 3.6 GB of routed experts (far larger than
L2); the shared expert and the router (11 MB) are rotated over 16 copies so
that consecutive tokens do not find them in L2, as in a model whose other
layers evict them.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 2|3|4|5] [--batch B]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FULL = dict(hidden=4096, inter=1024, n_experts=512, top_k=4)
TOKENS = 1000
STACK_LAYERS = 40
STACK_TOKENS = 256
COPIES = 16
FALLBACK_HBM_GBS = 6400.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5],
                   help="2 full-width layer; 3 skewed routing (use --batch); 4 2-bit routed experts; 5 40-layer stack")
    p.add_argument("--batch", type=int, default=1)
    p.add_argument("--tokens", type=int, default=TOKENS)
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--experts", type=int, default=512, help="routed experts (smaller pools for profiling runs)")
    p.add_argument("--pdl", type=int, default=1, help="programmatic dependent launch between decode calls")
    p.add_argument("--stack", action="store_true",
                   help="40-layer stack: one moe_stack_decode call per token (every layer in one launch) instead of one "
                        "moe_layer_decode call per layer (PDL-chained launches, the faster form on B300)")
    p.add_argument("--tensor-cores", action="store_true",
                   help="B > 1: expert contractions on the tensor cores (MOE_TENSOR_CORES)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value: the job's time is its slowest rank's."""
    if world <= 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        mx = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


def _code_only(text: str) -> str:
    """A source file without its comments and with runs of blank space made one
    space: a change of wording in a comment leaves a profile valid, any change
    of code does not."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", " ", text).strip()


def kernel_source_sha(files=("moe_decode_b1.cu", "moe_device.cuh", "moe_kernels.cu"), root=None):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(root or ROOT, "bit_expert_matvec_moe_b300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name, algorithmic_bytes_per_launch):
    """dram bytes of one launch of the bench's workload: the committed ncu
    capture's DRAM bytes per algorithmic byte (taken on a smaller expert pool,
    whose layers differ only in the router's rows) times the launch's
    algorithmic bytes, if the capture was taken on the current kernel sources;
    else None."""
    try:
        with open(os.path.join(ROOT, "profiles", f"{name}.json")) as f:
            p = json.load(f)
        if p.get("source_sha") == kernel_source_sha():
            return int(round(p["dram_over_algorithmic"] * algorithmic_bytes_per_launch))
    except Exception:  # noqa: BLE001
        pass
    return None


TC_SOURCES = ("moe_tc.cu", "moe_tc.cuh", "moe_device.cuh")


def profiled_tc_traffic(experts_per_call):
    """dram bytes of one call's two contraction launches (gate/up + down), from
    the committed small-pool capture scaled by the experts the call streams
    (each expert's tiles are read once per call), if it was taken on the
    current sources; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "tc_contract_b128.json")) as f:
            p = json.load(f)
        if p.get("source_sha") == kernel_source_sha(TC_SOURCES):
            return int(round(p["dram_bytes_per_expert_per_call"] * experts_per_call))
    except Exception:  # noqa: BLE001
        pass
    return None


# ----------------------------------------------------------------------------- workload
def build_full_layer(torch, M, bits=4, copies=COPIES, n_experts=512):
    """Full-width layer on the device: 512 routed experts, `copies` copies of the
    shared expert and router (identical bytes, distinct addresses)."""
    from synth import device as SD
    from synth import generate as G

    d = M.Dims(bits=bits, flags=M.MOE_HAS_SHARED, **{**FULL, "n_experts": n_experts})
    H, I, E = d.hidden, d.inter, d.n_experts
    stride = M.moe_packed_expert_bytes(d, bits)
    experts = torch.empty((E, stride), dtype=torch.uint8, device="cuda")

    def pack(canon, b, dst):
        M.moe_pack_weights(M.Dims(bits=b, flags=M.MOE_HAS_SHARED, **{**FULL, "n_experts": n_experts}), b,
                           [canon[m][0] for m in ("gate", "up", "down")],
                           [canon[m][1] for m in ("gate", "up", "down")],
                           [canon[m][2] for m in ("gate", "up", "down")], dst)

    for e in range(E):
        pack(SD.expert(G.SEED, 0, e, H, I, bits), bits, experts[e])
    sbytes = M.moe_packed_expert_bytes(d, 4)
    shared = torch.empty((copies, sbytes), dtype=torch.uint8, device="cuda")
    pack(SD.expert(G.SEED, 0, G.SHARED_EXPERT, H, I, 4), 4, shared[0])
    router_np = G.router(G.SEED, 0, E, H)
    router = torch.from_numpy(router_np.view(np.int16)).cuda().unsqueeze(0).repeat(copies, 1, 1).contiguous()
    for c in range(1, copies):
        shared[c].copy_(shared[0])
    torch.cuda.synchronize()
    return d, experts, stride, shared, router


def run_ours(args, rank, world, local):
    import torch

    import bit_expert_matvec_moe_b300 as M

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    from synth import generate as G

    bits = 2 if args.config == 4 else 4
    d, experts, stride, shared, router = build_full_layer(torch, M, bits=bits, n_experts=args.experts)
    if args.pdl:
        d.flags |= M.MOE_PDL
    tc = bool(args.tensor_cores) and args.batch > 1
    if tc:
        d.flags |= M.MOE_TENSOR_CORES
    B = args.batch
    T = args.tokens
    nsteps_tok = T // B
    layers = [M.make_layer(d, experts, stride, router[c], shared=shared[c], shared_bits=4) for c in range(COPIES)]
    offsets = None
    if args.config == 3:
        # skewed routing: per-expert popularity offsets o_e ~ N(0, 1.5) added to every token's logits
        o = torch.from_numpy(G.popularity_offsets(G.SEED, 0, d.n_experts)).cuda()
        offsets = o.unsqueeze(0).expand(B, d.n_experts).contiguous()
    h_host = G.hidden_states(G.SEED, 100 + rank, T, d.hidden)
    h0 = torch.from_numpy(h_host).cuda()
    h = h0.clone()
    ws = torch.empty(M.moe_workspace_bytes(d, B), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def one_step():
        for t in range(nsteps_tok):
            sl = slice(t * B, (t + 1) * B)
            M.moe_layer_decode(layers[t % COPIES], h[sl], ws, logit_offset=offsets, idx_out=idx[sl], w_out=w[sl],
                               stream=stream)

    # correctness smoke of the configuration (status word) before timing
    with torch.cuda.stream(stream):
        one_step()
    assert M.moe_get_device_status(ws, stream) == 0
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                one_step()
        except Exception as exc:  # noqa: BLE001
            print(f"# CUDA graph capture failed ({exc}); timing eager launches", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()
    run = (lambda: graph.replay()) if graph is not None else one_step

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            h.copy_(h0)
            run()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms = []
    with torch.cuda.stream(stream):
        # h is updated in place; resetting it (16 MB) is outside the event pair of each step
        for _ in range(args.steps):
            h.copy_(h0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    ck = clocks.stop()
    assert M.moe_get_device_status(ws, stream) == 0
    ms = max_over_ranks(float(np.mean(step_ms)), world, "cuda")

    # end to end through the public API with host buffers: H2D of the step's
    # hidden states from pinned memory, the decode calls, D2H of the outputs
    h_pin = torch.from_numpy(h_host).pin_memory()
    y_pin = torch.empty_like(h_pin).pin_memory()
    idx_pin = torch.empty((T, d.top_k), dtype=torch.int32).pin_memory()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for it in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            h.copy_(h_pin, non_blocking=True)
            run()
            y_pin.copy_(h, non_blocking=True)
            idx_pin.copy_(idx, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
    e2e = max_over_ranks(float(np.mean(e2e_ms)), world, "cuda")

    # unique routed experts per call (each streamed once for all of the call's tokens)
    idx_h = idx[: nsteps_tok * B].cpu().numpy().reshape(nsteps_tok, B * d.top_k)
    uniq = float(np.mean([len(np.unique(r)) for r in idx_h]))
    T = nsteps_tok * B
    expert_bytes = d.top_k * M.moe_packed_expert_bytes(d, bits) + M.moe_packed_expert_bytes(d, 4)
    call_bytes = uniq * M.moe_packed_expert_bytes(d, bits) + M.moe_packed_expert_bytes(d, 4)
    router_bytes = d.n_experts * d.hidden * 2
    launches_per_step = nsteps_tok
    per_launch_s = ms / 1e3 / launches_per_step
    tok_s = job_throughput(T, world, ms)
    peak, peak_kind = measured_hbm_peak()
    alg = int(call_bytes + router_bytes)
    achieved = (call_bytes + router_bytes) / per_launch_s / 1e9
    out = {
        "metric": "MoE layer decode tokens/s; expert-weight HBM GB/s vs ~8 TB/s peak",
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": (f"u{bits} codes dequantised to fp16 x fp16 hi/lo activations (tcgen05 kind::f16, fp32 accumulate)"
                  if tc else f"u{bits} codes x 23-bit block-floating-point activations (3 byte limbs per 64-group, "
                             "exact int32 dp4a group sums), fp32 scale/bias and accumulation"),
        "data": "synthetic (seeded SplitMix64; random-init weights of the stated shape)",
        "config": {
            "workload": (f"full-width single MoE layer, batch {B}: hidden 4096, {d.n_experts} experts, top-4 routed + 1 shared, "
                         f"inter 1024, {bits}-bit group-64 affine quant, bf16 router, {T} decode tokens"
                         + (", per-expert popularity offsets N(0, 1.5)" if offsets is not None else "")),
            "batch": B, "tokens_per_step": T, "launches_per_step": launches_per_step,
            "l2": f"inputs larger than L2 (3.6 GB routed experts); shared expert + router rotated over {COPIES} copies",
            "graph": graph is not None, "parallelism": f"replicas x{world}", "tensor_cores": tc,
        },
        "expert_gbs": round(call_bytes / per_launch_s / 1e9, 1),
        "unique_experts_per_call": round(uniq, 2),
        "us_per_token": round(ms * 1e3 / T, 3),
        "roofline": {
            "bound": "hbm",
            "kernel": ("decode_b1_kernel" if B == 1 else
                       "tc_contract_kernel, gate/up + down (batched path)" if tc else
                       "gateup_kernel + down_kernel (batched path)"),
            "achieved": round(achieved, 1) if achieved else None,
            "peak": peak,
            "peak_kind": peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4) if achieved else None,
            "algorithmic_bytes_per_launch": alg,
            "traffic": (profiled_traffic("decode_b1_full_b1", alg) if (B == 1 and bits == 4) else
                        profiled_tc_traffic(uniq + 1) if (tc and bits == 4) else None),
        },
        "e2e": {"value": round(job_throughput(T, world, e2e), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_pin.numel() * 4), "d2h_bytes_per_step": int(y_pin.numel() * 4 + idx_pin.numel() * 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
    }
    print(f"# {tok_s:.1f} tokens/s, {ms * 1e3 / T:.3f} us/token, e2e {e2e:.3f} ms/step", file=sys.stderr, flush=True)
    if rank == 0 and args.cpu_seconds > 0:
        # the oracle decodes token by token: batching does not change its tokens/s
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds, bits=bits)
        ncpu = os.cpu_count() or 1
        if ncpu > 1 and args.config == 2 and B == 1:  # the same oracle with its rows split over every host core
            mt = cpu_baseline(args.cpu_seconds / 2, threads=ncpu)
            out["cpu_baseline"]["all_cores"] = {"value": mt["value"], "cores": mt["cores"], "sample": mt["sample"]}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------- 40-layer stack
def run_stack(args, rank, world, local):
    """40 full-width 4-bit layers resident in HBM; each token passes all of them
    (RMSNorm before, residual after each), one moe_layer_decode call per layer
    (PDL-chained launches replayed from a graph), or with --stack one
    moe_stack_decode call per token (every layer in one launch).  Every layer
    has its own copy of the 512-expert pool, shared expert and router (identical
    bytes, distinct addresses: 145 GB of experts), so nothing a token reads is
    left in L2 by the previous token.  Routing follows a reuse trace (token t's
    slot j keeps token t-1's expert with probability 0.27), imposed through a
    +30 logit offset on the traced experts, which leaves the routing weights
    unchanged."""
    import torch

    import bit_expert_matvec_moe_b300 as M
    from synth import generate as G

    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    Lyr = STACK_LAYERS
    T = args.tokens if args.tokens != TOKENS else STACK_TOKENS
    d, experts0, stride, shared0, router0 = build_full_layer(torch, M, bits=4, copies=1, n_experts=args.experts)
    if args.pdl:
        d.flags |= M.MOE_PDL
    E, K = d.n_experts, d.top_k
    pools = [experts0] + [experts0.clone() for _ in range(Lyr - 1)]
    shared = [shared0[0]] + [shared0[0].clone() for _ in range(Lyr - 1)]
    routers = [router0[0]] + [router0[0].clone() for _ in range(Lyr - 1)]
    layers = [M.make_layer(d, pools[l], stride, routers[l], shared=shared[l], shared_bits=4) for l in range(Lyr)]
    trace = np.stack([G.reuse_trace(G.SEED, l, T, E, K) for l in range(Lyr)])  # [L, T, K]
    offs_h = np.zeros((T, Lyr, E), dtype=np.float32)  # token t's rows: one per layer
    for l in range(Lyr):
        for t in range(T):
            offs_h[t, l] = G.trace_offsets(trace[l, t], E)
    offs = torch.from_numpy(offs_h).cuda()
    h_host = G.hidden_states(G.SEED, 100 + rank, T, d.hidden)
    h0 = torch.from_numpy(h_host).cuda()
    h = h0.clone()
    ws = torch.empty(M.moe_workspace_bytes(d, 1), dtype=torch.uint8, device="cuda")
    M.moe_workspace_init(ws)
    idx = torch.empty((T, Lyr, K), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def one_step():
        for t in range(T):
            if not args.stack:
                for l in range(Lyr):
                    M.moe_layer_decode(layers[l], h[t:t + 1], ws, logit_offset=offs[t, l:l + 1],
                                       idx_out=idx[t, l:l + 1], stream=stream)
            else:
                M.moe_stack_decode(layers, h[t:t + 1], ws, logit_offset=offs[t], idx_out=idx[t], stream=stream)

    with torch.cuda.stream(stream):
        one_step()
    assert M.moe_get_device_status(ws, stream) == 0
    got = np.sort(idx.cpu().numpy(), axis=-1)
    assert np.array_equal(got, np.sort(trace.transpose(1, 0, 2), axis=-1)), "routing does not follow the imposed trace"
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        one_step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            h.copy_(h0)
            graph.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    step_ms = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            h.copy_(h0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    ck = clocks.stop()
    assert M.moe_get_device_status(ws, stream) == 0
    ms = max_over_ranks(float(np.mean(step_ms)), world, "cuda")
    # end to end: H2D of the step's hidden states, the 40-layer pass of every token, D2H of the outputs
    h_pin = torch.from_numpy(h_host).pin_memory()
    y_pin = torch.empty_like(h_pin).pin_memory()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for it in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            h.copy_(h_pin, non_blocking=True)
            graph.replay()
            y_pin.copy_(h, non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if it >= args.warmup:
                e2e_ms.append(e0.elapsed_time(e1))
    e2e = max_over_ranks(float(np.mean(e2e_ms)), world, "cuda")
    layer_bytes = (K + 1) * M.moe_packed_expert_bytes(d, 4) + E * d.hidden * 2
    launches = T * -(-Lyr // 64) if args.stack else T * Lyr
    tok_s = job_throughput(T, world, ms)
    per_launch_s = ms / 1e3 / (T * Lyr)
    peak, peak_kind = measured_hbm_peak()
    achieved = layer_bytes / per_launch_s / 1e9
    out = {
        "metric": "MoE layer decode tokens/s; expert-weight HBM GB/s vs ~8 TB/s peak",
        "value": round(tok_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("u4 codes x 23-bit block-floating-point activations (3 byte limbs per 64-group, exact int32 dp4a "
                  "group sums), fp32 scale/bias and accumulation"),
        "data": "synthetic (seeded SplitMix64; random-init weights of the stated shape)",
        "config": {
            "workload": (f"{Lyr}-layer MoE decode stack resident in HBM: full-width 4-bit layers (hidden 4096, {E} experts, "
                         f"top-4 + 1 shared, inter 1024), {T} tokens, top-4 reuse trace p=0.27"),
            "batch": 1, "tokens_per_step": T, "layers": Lyr, "launches_per_step": launches,
            "entry": "moe_stack_decode per token" if args.stack else "moe_layer_decode per layer",
            "l2": "no reuse: every layer has its own expert pool, shared expert and router (145 GB of experts)",
            "graph": True, "parallelism": f"replicas x{world}",
        },
        "expert_gbs": round((K + 1) * M.moe_packed_expert_bytes(d, 4) / per_launch_s / 1e9, 1),
        "us_per_layer": round(per_launch_s * 1e6, 3),
        "bytes_per_token": int(layer_bytes * Lyr),
        "roofline": {
            "bound": "hbm", "kernel": "decode_stack_kernel" if args.stack else "decode_b1_kernel",
            "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "algorithmic_bytes_per_launch": int(layer_bytes * (T * Lyr // launches)),
            "traffic": profiled_traffic("decode_stack_full_b1" if args.stack else "decode_b1_full_b1",
                                        layer_bytes * (T * Lyr // launches)),
        },
        "e2e": {"value": round(job_throughput(T, world, e2e), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h_pin.numel() * 4), "d2h_bytes_per_step": int(y_pin.numel() * 4)},
        "gpu_launches": launches * args.steps,
        "clocks": ck,
    }
    print(f"# {tok_s:.1f} tokens/s through {Lyr} layers, {per_launch_s * 1e6:.3f} us/layer", file=sys.stderr, flush=True)
    if rank == 0 and args.cpu_seconds > 0:
        # one token through the stack = Lyr single-layer decodes of the same shape for the oracle
        cb = cpu_baseline(args.cpu_seconds)
        out["cpu_baseline"] = {"value": round(cb["value"] / Lyr, 5), "unit": "tokens/s", "cores": cb["cores"],
                               "kind": "oracle", "sample": cb["sample"] + f"; extrapolated x{Lyr} layers per token"}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# ----------------------------------------------------------------------------- oracle (CPU) timing
def cpu_baseline(seconds: float, tokens_max: int = 64, threads: int = 1, bits: int = 4):
    """The fp64 oracle as it stands on a bounded sample of the same workload,
    run in a child process on `threads` host threads (1: one core; more: the
    rows of every matvec split over a thread pool, each BLAS call on one
    thread)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", str(seconds),
                          str(tokens_max), str(threads), str(bits)], capture_output=True, text=True, env=env,
                         timeout=600)
    if res.returncode != 0:
        raise RuntimeError("oracle timing failed: " + res.stderr[-2000:])
    return json.loads(res.stdout.strip().splitlines()[-1])


def _expert_forward_rows(O, ex, xn, H, I, pool, threads):
    """O.expert_forward with the rows of each matvec split over `threads`
    threads: the oracle's own dequant and SiLU on row blocks (every row of a
    matvec is independent, so the result is the oracle's)."""
    bits, group = ex["bits"], ex["group"]

    def rows(m, n_cols, x, lo, hi):
        c, sc, bi = ex[m]
        return O.dequant(c[lo:hi], sc[lo:hi], bi[lo:hi], bits, group, n_cols) @ x

    def split(n):
        step = (n + threads - 1) // threads
        return [(i, min(n, i + step)) for i in range(0, n, step)]

    g = np.concatenate(list(pool.map(lambda r: rows("gate", H, xn, *r), split(I))))
    u = np.concatenate(list(pool.map(lambda r: rows("up", H, xn, *r), split(I))))
    a = O.silu(g) * u
    return np.concatenate(list(pool.map(lambda r: rows("down", I, a, *r), split(H))))


def _cpu_baseline_child(seconds: float, tokens_max: int, threads: int = 1, bits: int = 4):
    """Tokens are decoded one by one until `seconds` of oracle time pass.  The
    touched experts are generated before each token's timing (input generation
    is not oracle work).  With one thread this is O.layer_decode as it stands;
    with several, the same layer with the rows of every matvec split over a
    thread pool (numpy releases the interpreter lock in its kernels)."""
    from concurrent.futures import ThreadPoolExecutor

    from oracle import moe_oracle as O
    from synth import generate as G

    H, I, E, K = FULL["hidden"], FULL["inter"], FULL["n_experts"], FULL["top_k"]
    R = G.router(G.SEED, 0, E, H)
    h = G.hidden_states(G.SEED, 100, tokens_max, H)
    shared = G.expert(G.SEED, 0, G.SHARED_EXPERT, H, I, 4)
    cache = {}

    def get(e):
        if e not in cache:
            cache[e] = G.expert(G.SEED, 0, e, H, I, bits)
        return cache[e]

    pool = ThreadPoolExecutor(max_workers=threads) if threads > 1 else None

    def decode(hh):
        if pool is None:
            return O.layer_decode(hh, experts=get, shared=shared, router_bits=R, top_k=K, hidden=H, inter=I)["y"]
        xn = O.rmsnorm(hh, None, 1e-6)
        logits = O.router_logits(R, xn)
        chosen = O.topk(logits, K)
        w = O.routing_weights(logits, chosen)
        y = np.asarray(hh, dtype=np.float64).copy()
        for wk, e in zip(w, chosen):
            y = y + wk * _expert_forward_rows(O, get(int(e)), xn, H, I, pool, threads)
        return y + _expert_forward_rows(O, shared, xn, H, I, pool, threads)

    done, spent = 0, 0.0
    while done < tokens_max and spent < seconds:
        xn = O.rmsnorm(h[done], None, 1e-6)
        for e in O.topk(O.router_logits(R, xn), K):
            get(int(e))  # generation outside the timed region
        t0 = time.perf_counter()
        decode(h[done])
        spent += time.perf_counter() - t0
        done += 1
    if pool is not None:
        pool.shutdown()
    how = ("fp64 numpy, 1 thread" if threads == 1 else
           f"fp64 numpy, rows of every matvec split over {threads} threads")
    return {"value": round(done / spent, 3), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} of the {TOKENS} decode tokens of the same layer ({bits}-bit routed experts), {how}"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import time as _t

    t_all = []
    for it in range(args.warmup + args.steps):
        cb = cpu_baseline(max(2.0, args.cpu_seconds / max(1, args.steps)), tokens_max=8)
        if it >= args.warmup:
            t_all.append(cb)
    vals = [c["value"] for c in t_all]
    v = float(np.mean(vals))
    out = {
        "impl": "reference",
        "metric": "MoE layer decode tokens/s; expert-weight HBM GB/s vs ~8 TB/s peak",
        "value": round(v, 3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 / v, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded SplitMix64; random-init weights of the stated shape)",
        "config": {"workload": ("full-width single MoE layer, batch 1: hidden 4096, 512 experts, top-4 routed + 1 "
                                "shared, inter 1024, 4-bit group-64 affine quant, bf16 router; each step a bounded "
                                "sample of its decode tokens"), "parallelism": "host cores, 1 thread"},
        "cpu_baseline": {"value": round(v, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": t_all[-1]["sample"]},
        "e2e": {"value": round(v, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)
    _t.sleep(0)


def main():
    if len(sys.argv) == 6 and sys.argv[1] == "--cpu-baseline-child":
        print(json.dumps(_cpu_baseline_child(float(sys.argv[2]), int(sys.argv[3]), int(sys.argv[4]), int(sys.argv[5]))))
        return
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.config == 5:
        run_stack(args, rank, world, local)
        return
    run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
