#!/usr/bin/env python
"""Benchmark of the DSA layer hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
lightning-indexer scores -> top-k -> sparse attention forward -> backward
(the backward only for workloads that have one). Inputs are resident in HBM
when the timed region starts; L2 is flushed (256 MiB write) between steps.

Prints ONE JSON line (rank 0). `value` is whole-job tokens/s (B*S tokens per
step per GPU); `e2e` is the same metric through the public API with the inputs
copied from pinned host memory and the outputs copied back inside the timed
region. `--impl reference` times the fp64 CPU oracle instead (on the host
cores, bounded row samples of the same workload).

Multi-GPU (torchrun): every rank runs an independent batch of the same
workload (weak scaling, no data-path collective); the step time is the max
over ranks.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "DSA layer fwd+bwd tokens/s and TFLOP/s on 1 GB300, % of tensor/HBM roofline"
DEFAULT_WORKLOAD = "v32_671b_s16k"
L2_FLUSH_BYTES = 256 << 20


# ------------------------------------------------------------------ work model

def pair_counts(wl: synth.Workload):
    """(valid causal pairs, selected pairs) per step, exact, from the segment layout."""
    S, k = wl.S, wl.topk
    if wl.ndocs:
        seg = synth.segments(wl.B, wl.S, wl.ndocs, wl.seed)
        causal = sel = 0
        for b in range(wl.B):
            _, counts = np.unique(seg[b], return_counts=True)
            for n in counts:
                n = int(n)
                causal += n * (n + 1) // 2
                m = min(n, k)
                sel += m * (m + 1) // 2 + (n - m) * k
        return causal, sel
    m = min(S, k)
    causal = wl.B * S * (S + 1) // 2
    sel = wl.B * (m * (m + 1) // 2 + (S - m) * k)
    return causal, sel


def stage_work(wl: synth.Workload, indexer_loss: bool = False):
    """Algorithmic work per step: FLOP for the contractions, bytes for top-k (the causal
    scores read, idx written, and with the indexer loss the selected scores written too).

    The indexer loss: its forward is the target's logit product (H x Dqk per selected
    pair); its backward the three products Z, dq and dk (Hi x Di each per selected pair).
    """
    causal, sel = pair_counts(wl)
    slots = wl.topk * wl.B * wl.S
    return {
        "indexer": {"flop": 2.0 * wl.Hi * wl.Di * causal},
        "indexer_topk": {"flop": 2.0 * wl.Hi * wl.Di * causal},
        "topk": {"bytes": 4.0 * causal + 4.0 * slots * (2 if indexer_loss else 1)},
        "attn_fwd": {"flop": 2.0 * wl.H * (wl.Dqk + wl.Dv) * sel},
        "attn_bwd": {"flop": 2.0 * wl.H * (3 * wl.Dqk + 2 * wl.Dv) * sel} if wl.backward else None,
        "loss_fwd": {"flop": 2.0 * wl.H * wl.Dqk * sel},
        "loss_bwd": {"flop": 3 * 2.0 * wl.Hi * wl.Di * sel},
    }


def step_flop(wl: synth.Workload, stages) -> float:
    """Whole-step FLOP: the contractions of the stages that ran, each counted once."""
    work = stage_work(wl)
    return sum(work[s]["flop"] for s in stages if "flop" in work[s])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash(stage: str) -> str:
    files = {"indexer": ["indexer.cu"], "topk": ["topk.cu"],
             "attn_fwd": ["attn_fwd.cu", "attn_fwd_tc.cu"],
             "attn_bwd": ["attn_bwd.cu", "attn_bwd_tc.cu"],
             "loss_fwd": ["iloss.cu"], "loss_bwd": ["iloss.cu"]}[stage]
    h = hashlib.sha256()
    for f in files + ["dsa_common.cuh", "dsa_attn_common.cuh"]:
        with open(os.path.join(ROOT, "sparse_attention_index_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(stage: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(f"{stage}/{workload}")
    if not e or e.get("source_hash") != kernel_source_hash(stage):
        return None
    return e.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = f"/tmp/dsa_clocks_{os.getpid()}.csv"

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- distributed

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, world: int) -> float:
    """Max of a host float over ranks (host metadata only, not the data path)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    backend = dist.get_backend()
    t = torch.tensor([value], dtype=torch.float64,
                     device="cuda" if backend == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ our arm

def make_inputs(wl):
    ind = synth.indexer_inputs(wl)
    att = synth.attention_inputs(wl)
    return ind, att


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import sparse_attention_index_gb300 as dsa

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    wl_r = wl.replace(seed=wl.seed + 1000 * rank) if rank else wl
    ind, att = make_inputs(wl_r)
    fp8 = args.indexer_dtype == "e4m3"

    def to_dev(a, bf16=False):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if bf16 else a)
        t = t.to(device)
        return t.view(torch.bfloat16) if bf16 else t

    if fp8:   # the same dyadic values as e4m3 bytes (exact)
        ind8 = synth.indexer_inputs_fp8(wl_r, "none")
        q_idx, k_idx = to_dev(ind8["q_idx"]), to_dev(ind8["k_idx"])
    else:
        q_idx, k_idx = to_dev(ind["q_idx"], True), to_dev(ind["k_idx"], True)
    w = to_dev(ind["w"])
    seg = None if ind["seg"] is None else to_dev(ind["seg"])
    Q, K, V = to_dev(att["Q"], True), to_dev(att["K"], True), to_dev(att["V"], True)
    dO = to_dev(att["dO"], True) if wl.backward else None
    B, S, k = wl.B, wl.S, wl.topk
    ld = (S + 3) // 4 * 4
    fused = args.fused_topk > 0 or args.stream_topk > 0
    stream_form = args.stream_topk > 0
    if fused:   # one block of query rows of scores (or none) instead of the [B, S, S] matrix
        R = args.stream_topk if stream_form else args.fused_topk
        wsb = (dsa.index_topk_stream_workspace_bytes(B, S, R) if stream_form
               else dsa.index_topk_workspace_bytes(B, S, R))
        topk_ws = torch.empty((wsb,), dtype=torch.uint8, device=device)
        scores = None
    else:
        scores = torch.empty((B, S, ld), dtype=torch.float32, device=device)
    idx = torch.empty((B, S, k), dtype=torch.int32, device=device)
    count = torch.empty((B, S), dtype=torch.int32, device=device)
    O = torch.empty((B, S, wl.H, wl.Dv), dtype=torch.bfloat16, device=device)
    lse = torch.empty((B, S, wl.H), dtype=torch.float32, device=device)
    fwd_ws = torch.empty((max(dsa.fwd_workspace_bytes(B, S, wl.H, wl.Hkv, wl.Dqk, wl.Dv), 16),),
                         dtype=torch.uint8, device=device)
    if wl.backward:
        dQ = torch.empty_like(Q)
        dK = torch.empty_like(K)
        dV = torch.empty_like(V)
        ws = torch.empty((dsa.bwd_workspace_bytes(B, S, wl.H, wl.Hkv, wl.Dqk, wl.Dv),), dtype=torch.uint8,
                         device=device)
    flush = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    stages = (["indexer_topk"] if fused else ["indexer", "topk"]) + ["attn_fwd"] + \
        (["attn_bwd"] if wl.backward else [])
    loss = args.indexer_loss
    if loss:
        # the indexer's auxiliary loss and its gradient into the indexer inputs
        stages += ["loss_fwd", "loss_bwd"]
        kl = torch.empty((B, S), dtype=torch.float32, device=device)
        dI = torch.empty((B, S, k), dtype=torch.float32, device=device)
        dq_idx = torch.empty((B, S, wl.Hi, wl.Di), dtype=torch.float32, device=device)
        dk_idx = torch.empty((B, S, wl.Di), dtype=torch.float32, device=device)
        dw = torch.empty((B, S, wl.Hi), dtype=torch.float32, device=device)
        # the top-k hands the loss the selected scores slot by slot (read contiguously)
        sel = torch.empty((B, S, k), dtype=torch.float32, device=device)
    else:
        sel = None
    # indexer, top-k, the forward (two launches on the dense-tile kernel: bitmap build +
    # attention), the backward and its finalize (four on the dense-tile kernels: bitmap,
    # dQ pass, dK / dV pass, finalize)
    fwd_launches = 2 if dsa.dsa_sparse_attn_fwd_kernel(B, S, wl.H, wl.Hkv, wl.Dqk, wl.Dv, k, wl.scale) \
        == dsa.DSA_FWD_DENSE_TC else 1
    bwd_launches = (4 if dsa.dsa_sparse_attn_bwd_kernel(B, S, wl.H, wl.Hkv, wl.Dqk, wl.Dv, k, wl.scale)
                    == dsa.DSA_BWD_DENSE_TC else 2) if wl.backward else 0
    if stream_form:   # sample, window, emit, finish; then per block two gated launches
        idx_launches = 4 + 2 * ((S + R - 1) // R)
    elif fused:   # per block of query rows: the indexer, the staged and / or the long-row top-k
        idx_launches = sum(1 + (t_lo < 16384) + (min(t_lo + R, S) > 16384)
                           for t_lo in range(0, S, R))
    else:
        idx_launches = 2
    launches_per_step = idx_launches + fwd_launches + bwd_launches + (2 if loss else 0)

    def step(ev):
        ev[0].record(stream)
        e = 1
        if stream_form:
            dsa.dsa_index_topk_stream(q_idx, k_idx, w, k, seg, block_rows=R, idx=idx,
                                      count=count, ws=topk_ws, stream=stream, vals=sel)
        elif fused:
            dsa.dsa_index_topk(q_idx, k_idx, w, k, seg, block_rows=R, idx=idx, count=count,
                               ws=topk_ws, stream=stream, vals=sel)   # e4m3: the fp8 indexer
        else:
            if fp8:
                dsa.dsa_index_scores_fp8(q_idx, k_idx, w, seg, scores=scores, stream=stream)
            else:
                dsa.dsa_index_scores(q_idx, k_idx, w, seg, scores=scores, stream=stream)
            ev[e].record(stream)
            e += 1
            dsa.dsa_topk(scores, k, seg, idx=idx, count=count, vals=sel, stream=stream)
        ev[e].record(stream)
        e += 1
        dsa.dsa_sparse_attn_fwd(Q, K, V, idx, wl.scale, O=O, lse=lse, ws=fwd_ws, stream=stream)
        ev[e].record(stream)
        e += 1
        if wl.backward:
            dsa.dsa_sparse_attn_bwd(Q, K, V, idx, O, lse, dO, wl.scale, dQ=dQ, dK=dK, dV=dV, ws=ws,
                                    stream=stream)
            ev[e].record(stream)
            e += 1
        if loss:
            dsa.dsa_indexer_loss(Q, K, idx, lse, None, wl.scale, 1.0 / (B * S), kl=kl, dI=dI,
                                 stream=stream, sel_scores=sel)
            ev[e].record(stream)
            dsa.dsa_indexer_loss_bwd(q_idx, k_idx, w, idx, dI, dq_idx=dq_idx, dk_idx=dk_idx,
                                     dw=dw, stream=stream)
            ev[e + 1].record(stream)

    n_ev = len(stages) + 1
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step([torch.cuda.Event(enable_timing=True) for _ in range(n_ev)])
            flush.zero_()
        torch.cuda.synchronize(device)
        if dsa.dsa_get_last_device_error(stream) != 0:
            raise RuntimeError("device error during warm-up")
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
                  for _ in range(args.steps)]
        clocks = ClockSampler(local_rank)
        barrier(world)
        torch.cuda.synchronize(device)
        clocks.start()
        for i in range(args.steps):
            step(events[i])
            flush.zero_()   # between timed steps, outside their events
        torch.cuda.synchronize(device)
        clk = clocks.stop()
        barrier(world)
    stage_ms = {s: 0.0 for s in stages}
    for ev in events:
        for j, s in enumerate(stages):
            stage_ms[s] += ev[j].elapsed_time(ev[j + 1])
    stage_ms = {s: v / args.steps for s, v in stage_ms.items()}
    ms_step = sum(stage_ms.values())
    ms_step_max = reduce_max(ms_step, world)
    err = dsa.dsa_get_last_device_error(stream)

    # ---- end to end through the public API: pinned host in, host out
    e2e = None
    if not args.no_e2e:
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        src = ind8 if fp8 else ind   # e4m3 bytes of the same dyadic values
        h_in = {"q_idx": pin(src["q_idx"]), "k_idx": pin(src["k_idx"]), "w": pin(ind["w"]),
                "Q": pin(att["Q"]), "K": pin(att["K"]), "V": pin(att["V"])}
        if seg is not None:
            h_in["seg"] = pin(ind["seg"])
        if wl.backward:
            h_in["dO"] = pin(att["dO"])
        # the public host-to-host API: copies in, the four stages and copies out on
        # three streams, overlapped (sparse_attention_index_gb300.HostPipeline)
        pipe = dsa.HostPipeline(B, S, wl.Hi, wl.Di, wl.H, wl.Dqk, wl.Dv, k, wl.scale,
                                backward=wl.backward, segments=seg is not None, device=device,
                                Hkv=wl.Hkv, indexer_loss=loss,
                                indexer_dtype="e4m3" if fp8 else "bf16",
                                fused_block_rows=R if fused else 0, stream_form=stream_form)
        h_out = {n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in pipe.out.items()}
        h2d = sum(t.numel() * t.element_size() for t in h_in.values())
        d2h = sum(t.numel() * t.element_size() for t in h_out.values())
        for _ in range(max(1, min(args.warmup, 3))):
            pipe.step(h_in, h_out)
        torch.cuda.synchronize(device)
        # as many timed steps as the device-side measurement: the first step's copies in and
        # the last step's copies out overlap no other step, so fewer steps overstate them
        n_e2e = max(1, args.steps)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record(pipe.s_in)   # every stream's work of the timed steps follows this
        for _ in range(n_e2e):
            pipe.step(h_in, h_out)
        e1.record(pipe.s_out)  # the last copy-out follows every kernel of the last step
        torch.cuda.synchronize(device)
        if dsa.dsa_get_last_device_error(stream) != 0:
            raise RuntimeError("device error during the end-to-end steps")
        e2e_ms = reduce_max(e0.elapsed_time(e1) / n_e2e, world)
        e2e = {"value": world * B * S / (e2e_ms / 1e3), "unit": "tokens/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e}

    return {"stage_ms": stage_ms, "ms_step": ms_step_max, "clocks": clk, "device_error": err,
            "launches_per_step": launches_per_step, "e2e": e2e, "stages": stages}


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(wl, ind, att, rows, loss=False):
    """The oracle's full per-row work (scores, top-k, fwd, bwd; with loss, the indexer loss
    and its gradient) on the listed query rows."""
    import oracle
    S, k = wl.S, wl.topk
    sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], ind["seg"], rows=rows)
    idx_rows, _ = oracle.topk(sc, ind["seg"], S, k, rows=rows, B=wl.B)
    idx = np.full((wl.B * S, k), -1, dtype=np.int32)
    idx[rows] = idx_rows
    idx = idx.reshape(wl.B, S, k)
    oracle.attn_fwd(att["Q"], att["K"], att["V"], idx, wl.scale, rows=rows)
    if wl.backward:
        oracle.attn_bwd(att["Q"], att["K"], att["V"], idx, att["dO"], wl.scale, rows=rows)
    if loss:
        _, dI = oracle.indexer_loss(att["Q"], att["K"], idx, sc, wl.scale, 1.0 / wl.tokens,
                                    rows=rows)
        oracle.indexer_loss_bwd(ind["q_idx"], ind["k_idx"], ind["w"], idx, dI, rows=rows)


def sample_rows(wl, n, salt):
    rng = np.random.default_rng(wl.seed * 7919 + salt)
    return np.sort(rng.choice(wl.B * wl.S, size=min(n, wl.B * wl.S), replace=False)).astype(np.int64)


def cpu_baseline(wl, n_rows, loss=False):
    import oracle
    ind, att = make_inputs(wl)
    rows = sample_rows(wl, n_rows, 1)
    t0 = time.perf_counter()
    oracle_sample(wl, ind, att, rows, loss)
    dt = time.perf_counter() - t0
    return {"value": rows.size / dt, "unit": "tokens/s", "cores": oracle.default_threads(),
            "kind": "oracle", "seconds": dt,
            "sample": f"{rows.size} uniformly drawn query rows of {wl.name} (B*S={wl.tokens}); "
                      "each row gets its full indexer, top-k, forward"
                      + (" and backward" if wl.backward else "")
                      + (" and indexer-loss" if loss else "") + " work; tokens/s = rows / s"}


def run_reference(args, wl, rank, world):
    import oracle
    if rank != 0:
        return 0
    ind, att = make_inputs(wl)
    per_step = args.cpu_rows_per_step
    for i in range(args.warmup):
        oracle_sample(wl, ind, att, sample_rows(wl, per_step, 100 + i), args.indexer_loss)
    times = []
    for i in range(args.steps):
        rows = sample_rows(wl, per_step, 1000 + i)
        t0 = time.perf_counter()
        oracle_sample(wl, ind, att, rows, args.indexer_loss)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * per_step / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, args),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle",
                         "cores": oracle.default_threads(),
                         "sample": f"each step: {per_step} uniformly drawn query rows of {wl.name}, "
                                   "full per-row work of every stage, on the host cores"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, args=None):
    cfg = {"workload": f"{wl.name}: {wl.description}", "B": wl.B, "S": wl.S,
           "index_heads": wl.Hi, "index_head_dim": wl.Di, "index_topk": wl.topk,
           "heads": wl.H, "kv_heads": wl.Hkv, "qk_dim": wl.Dqk, "v_dim": wl.Dv,
           "backward": wl.backward, "segments": wl.ndocs,
           "l2": "flushed between steps (256 MiB write outside the timed events)"}
    if args is not None and getattr(args, "indexer_dtype", "bf16") == "e4m3":
        cfg["indexer_dtype"] = "e4m3"
    if args is not None and getattr(args, "indexer_loss", False):
        cfg["indexer_loss"] = True
    if args is not None and getattr(args, "fused_topk", 0):
        cfg["fused_topk_block_rows"] = args.fused_topk
    if args is not None and getattr(args, "stream_topk", 0):
        cfg["stream_topk_block_rows"] = args.stream_topk
    return cfg


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--indexer-dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="e4m3: the indexer runs on fp8 inputs (the same dyadic values)")
    ap.add_argument("--fused-topk", type=int, default=0, metavar="BLOCK_ROWS",
                    help="run the indexer and the top-k fused through blocks of this many query "
                         "rows (a multiple of 256): no [B, S, S] score matrix")
    ap.add_argument("--stream-topk", type=int, default=0, metavar="BLOCK_ROWS",
                    help="run the indexer and the top-k in the streaming form (no score rows; "
                         "blocks of this many query rows, a multiple of 256, for rows it leaves)")
    ap.add_argument("--indexer-loss", action="store_true",
                    help="add the indexer auxiliary loss and its gradient to every step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=0,
                    help="rows in the CPU-baseline sample (default: 24 per host core)")
    ap.add_argument("--cpu-rows-per-step", type=int, default=0,
                    help="rows per reference-arm step (default: 4 per host core)")
    args = ap.parse_args(argv)
    for opt, val in (("--fused-topk", args.fused_topk), ("--stream-topk", args.stream_topk)):
        if val and val % 256:
            ap.error(f"{opt} takes a multiple of 256")
    if args.fused_topk and args.stream_topk:
        ap.error("--fused-topk and --stream-topk are two forms of the same stage: pick one")
    if args.indexer_loss:
        if args.indexer_dtype != "bf16":
            ap.error("--indexer-loss takes the bf16 indexer (its backward reads bf16 inputs)")
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    wl = synth.WORKLOADS[args.workload]
    import oracle
    cores = oracle.default_threads()
    args.cpu_rows = args.cpu_rows or 24 * cores
    args.cpu_rows_per_step = args.cpu_rows_per_step or 4 * cores
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")

    if args.impl == "reference":
        rc = run_reference(args, wl, rank, world)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc

    r = run_ours(args, wl, rank, world, local_rank)
    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    work = stage_work(wl, args.indexer_loss)
    tokens = wl.B * wl.S
    total_flop = step_flop(wl, r["stages"])
    stages_out = {}
    for s in r["stages"]:
        ms = r["stage_ms"][s]
        wk = work[s]
        if "flop" in wk:
            tf = wk["flop"] / (ms / 1e3) / 1e12
            # e4m3 contractions: the measured bf16 peak x the nominal fp8 / bf16 ratio (2)
            pk = peaks["bf16_tflops_sustained"] * (2.0 if s in ("indexer", "indexer_topk") and
                                                   args.indexer_dtype == "e4m3" else 1.0)
            stages_out[s] = {"ms": ms, "tflops": tf, "bound": "tensor", "frac": tf / pk}
        else:
            gbs = wk["bytes"] / (ms / 1e3) / 1e9
            stages_out[s] = {"ms": ms, "gbs": gbs, "bound": "hbm", "frac": gbs / peaks["hbm_gbs"]}
    dom = max(r["stages"], key=lambda s: r["stage_ms"][s])
    d = stages_out[dom]
    if d["bound"] == "tensor":
        roof = {"kernel": dom, "bound": "tensor", "achieved": d["tflops"],
                "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s", "frac": d["frac"],
                "peak_kind": f"{peaks['source']} bf16 sustained (kernel timed inside a repeated step)"}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": d["gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": d["frac"], "peak_kind": f"{peaks['source']} HBM copy"}
    roof["traffic"] = measured_traffic(dom, wl.name)

    line = {
        "metric": METRIC, "value": world * tokens / (r["ms_step"] / 1e3), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded: dyadic indexer inputs, N(0,1) bf16 attention inputs)",
        "config": workload_config(wl, args),
        "tflops": total_flop / (r["ms_step"] / 1e3) / 1e12,
        "stages": stages_out,
        "roofline": roof,
        "clocks": r["clocks"],
        "e2e": r["e2e"],
        "gpu_launches": r["launches_per_step"] * args.steps,
        "device_error": r["device_error"],
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_rows, args.indexer_loss)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
