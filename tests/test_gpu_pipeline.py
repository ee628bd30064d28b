"""HostPipeline: host -> device copies, the four stages and device -> host copies on
three streams. Its host outputs must equal the device-resident path's results (the
same kernels: bit-exact, except dK / dV, whose fp32 atomic order is unspecified),
also over consecutive overlapped steps."""
import numpy as np
import pytest
import torch

import synth
from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["packed_s489", "small2b_s4096"])
def test_host_pipeline_matches_device_path(name):
    import sparse_attention_index_gb300 as dsa
    wl = synth.WORKLOADS[name]
    if name == "small2b_s4096":
        wl = wl.replace(B=1, S=1500)
    ind = synth.indexer_inputs(wl)
    att = synth.attention_inputs(wl)
    seg = None if ind["seg"] is None else dev(ind["seg"])
    ref = dsa.dsa_layer(bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"]),
                        bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]), wl.topk,
                        wl.scale, seg=seg, dO=bf16_dev(att["dO"]) if wl.backward else None)
    torch.cuda.synchronize()

    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_in = {n: pin(ind[n]) for n in ("q_idx", "k_idx", "w")}
    h_in.update({n: pin(att[n]) for n in ("Q", "K", "V")})
    if seg is not None:
        h_in["seg"] = pin(ind["seg"])
    if wl.backward:
        h_in["dO"] = pin(att["dO"])
    pipe = dsa.HostPipeline(wl.B, wl.S, wl.Hi, wl.Di, wl.H, wl.Dqk, wl.Dv, wl.topk, wl.scale,
                            backward=wl.backward, segments=seg is not None)
    h_out = {n: torch.zeros(t.shape, dtype=t.dtype).pin_memory() for n, t in pipe.out.items()}
    for _ in range(3):   # overlapped consecutive steps over the same inputs
        pipe.step(h_in, h_out)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0

    for n in ("idx", "count", "O", "lse") + (("dQ",) if wl.backward else ()):
        assert torch.equal(h_out[n], ref[n].cpu()), n
    if wl.backward:
        for n in ("dK", "dV"):
            assert rel_err(host_f64(h_out[n]), host_f64(ref[n])) <= TOL, n


def test_host_pipeline_with_indexer_loss():
    """The pipeline's loss stage (it reads the top-k's selected scores, Q, K and the indexer
    inputs, so the next step's copies wait for it) gives the device-resident path's dq_idx
    exactly, and kl, dw and dk_idx within the rounding of their atomic fp32 sums, over
    consecutive overlapped steps."""
    import sparse_attention_index_gb300 as dsa
    wl = synth.WORKLOADS["packed_s489"]
    ind = synth.indexer_inputs(wl)
    att = synth.attention_inputs(wl)
    seg = dev(ind["seg"])
    qd, kd, wd = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"])
    ref = dsa.dsa_layer(qd, kd, wd, bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]),
                        wl.topk, wl.scale, seg=seg, dO=bf16_dev(att["dO"]))
    g = 1.0 / (wl.B * wl.S)
    kl, dI = dsa.dsa_indexer_loss(bf16_dev(att["Q"]), bf16_dev(att["K"]), ref["idx"], ref["lse"],
                                  ref["scores"], wl.scale, g)
    dq, dk, dw = dsa.dsa_indexer_loss_bwd(qd, kd, wd, ref["idx"], dI)
    torch.cuda.synchronize()

    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    h_in = {n: pin(ind[n]) for n in ("q_idx", "k_idx", "w", "seg")}
    h_in.update({n: pin(att[n]) for n in ("Q", "K", "V", "dO")})
    pipe = dsa.HostPipeline(wl.B, wl.S, wl.Hi, wl.Di, wl.H, wl.Dqk, wl.Dv, wl.topk, wl.scale,
                            backward=True, segments=True, indexer_loss=True)
    h_out = {n: torch.zeros(t.shape, dtype=t.dtype).pin_memory() for n, t in pipe.out.items()}
    for _ in range(3):
        pipe.step(h_in, h_out)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(h_out["idx"], ref["idx"].cpu())
    assert rel_err(host_f64(h_out["kl"]), host_f64(kl)) <= 1e-6       # atomic order of the sum
    assert torch.equal(h_out["dq_idx"], dq.cpu())
    assert rel_err(host_f64(h_out["dw"]), host_f64(dw)) <= 1e-6
    assert rel_err(host_f64(h_out["dk_idx"]), host_f64(dk)) <= 1e-5


@pytest.mark.parametrize("form", [("e4m3", 0), ("bf16", 256), ("e4m3", 512)])
def test_host_pipeline_fp8_and_fused_indexer(form):
    """The pipeline with e4m3 indexer inputs and / or the indexer and top-k fused through
    blocks of query rows: on the dyadic inputs (exact in e4m3) its index lists, O and dQ equal
    the bf16, unfused device-resident path bit for bit."""
    import sparse_attention_index_gb300 as dsa
    dtype, block = form
    wl = synth.WORKLOADS["packed_s489"]
    ind = synth.indexer_inputs(wl)
    ind8 = synth.indexer_inputs_fp8(wl, "none")
    att = synth.attention_inputs(wl)
    seg = dev(ind["seg"])
    ref = dsa.dsa_layer(bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"]),
                        bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]), wl.topk,
                        wl.scale, seg=seg, dO=bf16_dev(att["dO"]))
    torch.cuda.synchronize()
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    src = ind8 if dtype == "e4m3" else ind
    h_in = {"q_idx": pin(src["q_idx"]), "k_idx": pin(src["k_idx"]), "w": pin(ind["w"]),
            "seg": pin(ind["seg"])}
    h_in.update({n: pin(att[n]) for n in ("Q", "K", "V", "dO")})
    pipe = dsa.HostPipeline(wl.B, wl.S, wl.Hi, wl.Di, wl.H, wl.Dqk, wl.Dv, wl.topk, wl.scale,
                            backward=True, segments=True, indexer_dtype=dtype,
                            fused_block_rows=block)
    h_out = {n: torch.zeros(t.shape, dtype=t.dtype).pin_memory() for n, t in pipe.out.items()}
    for _ in range(3):
        pipe.step(h_in, h_out)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    for n in ("idx", "count", "O", "lse", "dQ"):
        assert torch.equal(h_out[n], ref[n].cpu()), n


@pytest.mark.parametrize("form", ["memory", "stream"])
def test_host_pipeline_distinct_consecutive_steps(form):
    """Two input sets taken in turns over four overlapped steps, each step into its own host
    outputs: every step's results are those of its own inputs (a step's kernels overwrite the
    device outputs only once the previous step's copies of them have left; the index lists,
    O, LSE and dQ match the device-resident path bit for bit), with the indexer loss on (kl
    and dw, from the top-k's selected scores, within the rounding of their atomic sums)."""
    import sparse_attention_index_gb300 as dsa
    base = synth.WORKLOADS["packed_s489"]
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
    sets, refs = [], []
    for seed in (4, 5):
        wl = base.replace(seed=seed)
        ind, att = synth.indexer_inputs(wl), synth.attention_inputs(wl)
        qd, kd, wd, seg = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"]), dev(ind["seg"])
        ref = dsa.dsa_layer(qd, kd, wd, bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]),
                            wl.topk, wl.scale, seg=seg, dO=bf16_dev(att["dO"]))
        kl, dI = dsa.dsa_indexer_loss(bf16_dev(att["Q"]), bf16_dev(att["K"]), ref["idx"],
                                      ref["lse"], ref["scores"], wl.scale, 1.0 / (wl.B * wl.S))
        _, _, dw = dsa.dsa_indexer_loss_bwd(qd, kd, wd, ref["idx"], dI)
        ref = {n: ref[n].cpu() for n in ("idx", "count", "O", "lse", "dQ")}
        ref["kl"], ref["dw"] = kl.cpu(), dw.cpu()
        refs.append(ref)
        h_in = {n: pin(ind[n]) for n in ("q_idx", "k_idx", "w", "seg")}
        h_in.update({n: pin(att[n]) for n in ("Q", "K", "V", "dO")})
        sets.append(h_in)
    torch.cuda.synchronize()
    wl = base
    pipe = dsa.HostPipeline(wl.B, wl.S, wl.Hi, wl.Di, wl.H, wl.Dqk, wl.Dv, wl.topk, wl.scale,
                            backward=True, segments=True, indexer_loss=True,
                            fused_block_rows=512 if form == "stream" else 0,
                            stream_form=form == "stream")
    outs = [{n: torch.zeros(t.shape, dtype=t.dtype).pin_memory() for n, t in pipe.out.items()}
            for _ in range(4)]
    for i in range(4):
        pipe.step(sets[i % 2], outs[i])
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    for i in range(4):
        ref, got = refs[i % 2], outs[i]
        for n in ("idx", "count", "O", "lse", "dQ"):
            assert torch.equal(got[n], ref[n]), (i, n)
        # kl and dw: fp32 sums whose order across warps (atomics) is unspecified
        assert rel_err(host_f64(got["kl"]), host_f64(ref["kl"])) <= 1e-6, i
        assert rel_err(host_f64(got["dw"]), host_f64(ref["dw"])) <= 1e-6, i
