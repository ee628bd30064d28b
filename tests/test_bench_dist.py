"""Multi-rank host logic of bench.py, as world_size-2 gloo process groups on the CPU.

bench.py shards by batch: every rank runs its own seeded batch and the step time
is the maximum over ranks. What needs no GPU is checked here: the rank/world
environment, the max-over-ranks reduction and the barrier, and the reference arm
under two ranks (rank 0 alone runs and prints; rank 1 exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(args_per_rank, world=2, timeout=300):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable] + args_per_rank(rank), cwd=ROOT, env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=timeout)
            outs.append((p.returncode, out, err))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    return outs


def test_reduce_max_and_barrier_over_two_ranks():
    code = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import torch.distributed as dist
        import bench
        rank, world, local_rank = bench.dist_env()
        dist.init_process_group("gloo")
        bench.barrier(world)
        v = bench.reduce_max(10.0 * rank + 0.25, world)
        bench.barrier(world)
        print(rank, world, local_rank, v)
        dist.destroy_process_group()
    """)
    outs = _launch(lambda r: ["-c", code])
    for rank, (rc, out, err) in enumerate(outs):
        assert rc == 0, err
        r, w, lr, v = out.split()
        assert (int(r), int(w), int(lr)) == (rank, 2, rank)
        assert float(v) == 10.25   # the max over ranks, on every rank


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)


def test_reference_arm_under_two_ranks():
    args = ["bench.py", "--impl", "reference", "--gpus", "2", "--workload", "tiny_s128",
            "--steps", "1", "--warmup", "0", "--cpu-rows-per-step", "4"]
    outs = _launch(lambda r: args)
    (rc0, out0, err0), (rc1, out1, err1) = outs
    assert rc0 == 0, err0
    assert rc1 == 0, err1
    assert out1.strip() == ""          # only rank 0 prints
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_step_flop_counts_each_stage_that_ran_once():
    """The whole-step TFLOP/s of the bench line: the fused indexer + top-k counts the indexer's
    contraction once, and the loss stages count only when they run."""
    import bench
    import synth
    wl = synth.WORKLOADS["v32_671b_s16k"]
    causal, sel = bench.pair_counts(wl)
    unfused = bench.step_flop(wl, ["indexer", "topk", "attn_fwd", "attn_bwd"])
    assert unfused == (2.0 * wl.Hi * wl.Di * causal + 2.0 * wl.H * (wl.Dqk + wl.Dv) * sel
                       + 2.0 * wl.H * (3 * wl.Dqk + 2 * wl.Dv) * sel)
    assert bench.step_flop(wl, ["indexer_topk", "attn_fwd", "attn_bwd"]) == unfused
    with_loss = bench.step_flop(wl, ["indexer", "topk", "attn_fwd", "attn_bwd", "loss_fwd",
                                     "loss_bwd"])
    assert with_loss == unfused + 2.0 * wl.H * wl.Dqk * sel + 3 * 2.0 * wl.Hi * wl.Di * sel
