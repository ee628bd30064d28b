"""Full-size workloads, run exactly as bench.py launches them, checked on samples.

At these sizes the oracle cannot recompute everything, so the checks are:
* index scores and top-k sets: bit-exact on sampled query rows
  (t = 0, k-1, k, S-1 and uniform draws, per batch row);
* attention output / LSE and dQ: within 2e-2 * max|ref| on the sampled rows;
* dK / dV: exact reference for the last keys of every batch row (key s only
  receives gradient from queries t >= s, so the oracle over the last rows
  gives those keys completely);
* sum over keys of dV equals the sum over queries and heads of dO (softmax
  weights sum to one), at any size.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TOL, bf16_dev, dev, host_f64, rel_err

pytestmark = pytest.mark.gpu

TAIL = 48


def _run(wl):
    import sparse_attention_index_gb300 as dsa
    ind = synth.indexer_inputs(wl)
    att = synth.attention_inputs(wl)
    seg = None if ind["seg"] is None else dev(ind["seg"])
    out = dsa.dsa_layer(bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"]),
                        bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"]), wl.topk,
                        wl.scale, seg=seg, dO=bf16_dev(att["dO"]) if wl.backward else None)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    return ind, att, out


def _check(wl, n_uniform):
    ind, att, out = _run(wl)
    rows = synth.sample_rows(wl, n_uniform)
    S, k = wl.S, wl.topk

    # index scores, bit-exact on the sampled rows (and on the last TAIL rows of every batch
    # row, whose selections give the oracle's dK / dV of the last keys)
    tail_rows = np.concatenate([b * S + np.arange(S - TAIL, S) for b in range(wl.B)]) \
        if wl.backward else np.zeros(0, dtype=np.int64)
    all_rows = np.union1d(rows, tail_rows).astype(np.int64)
    ref_sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], ind["seg"], rows=all_rows)
    ab, at = all_rows // S, all_rows % S
    gsc = out["scores"][torch.as_tensor(ab), torch.as_tensor(at), :S].double().cpu().numpy()
    for r in range(all_rows.size):
        t = at[r]
        g, o = gsc[r, : t + 1], ref_sc[r, : t + 1]
        assert np.array_equal(np.isneginf(g), np.isneginf(o))
        fin = np.isfinite(o)
        assert np.array_equal(g[fin], o[fin]), (int(all_rows[r]),)

    # top-k sets, bit-exact; the oracle's own lists feed every oracle call below
    ref_idx, ref_cnt = oracle.topk(ref_sc, ind["seg"], S, k, rows=all_rows, B=wl.B)
    gidx = out["idx"].cpu().numpy().reshape(-1, k)
    assert np.array_equal(gidx[all_rows], ref_idx)
    assert np.array_equal(out["count"].cpu().numpy().reshape(-1)[all_rows], ref_cnt)
    idx = np.full((wl.B * S, k), -1, dtype=np.int32)
    idx[all_rows] = ref_idx
    idx = idx.reshape(wl.B, S, k)

    # attention forward on the sampled rows
    O_ref, lse_ref = oracle.attn_fwd(att["Q"], att["K"], att["V"], idx, wl.scale, rows=rows)
    O = out["O"].reshape(wl.B * S, wl.H, wl.Dv)[torch.as_tensor(rows)]
    lse = out["lse"].reshape(wl.B * S, wl.H)[torch.as_tensor(rows)]
    assert rel_err(host_f64(O), O_ref) <= TOL
    assert rel_err(host_f64(lse), lse_ref) <= TOL

    if not wl.backward:
        return
    dQ_ref, _, _ = oracle.attn_bwd(att["Q"], att["K"], att["V"], idx, att["dO"], wl.scale,
                                   rows=rows)
    dQ = out["dQ"].reshape(wl.B * S, wl.H, wl.Dqk)[torch.as_tensor(rows)]
    assert rel_err(host_f64(dQ), dQ_ref) <= TOL
    _, dK_ref, dV_ref = oracle.attn_bwd(att["Q"], att["K"], att["V"], idx, att["dO"], wl.scale,
                                        rows=tail_rows)
    dK = host_f64(out["dK"][:, S - TAIL:])
    dV = host_f64(out["dV"][:, S - TAIL:])
    assert rel_err(dK, dK_ref[:, S - TAIL:]) <= TOL
    assert rel_err(dV, dV_ref[:, S - TAIL:]) <= TOL
    # sum_s dV[s] = sum_{t,h} dO[t,h]
    dv_sum = out["dV"].double().sum(dim=(1, 2)).cpu().numpy()
    do_sum = bf16_dev(att["dO"]).double().sum(dim=(1, 2)).cpu().numpy()
    assert rel_err(dv_sum, do_sum) <= TOL


@pytest.mark.parametrize("name", ["tiny_s128", "packed_s489", "small2b_s4096", "packed_s4096",
                                  "v32_671b_s16k", "mla_perhead_s4096"])
def test_workload(name):
    _check(synth.WORKLOADS[name], n_uniform=12)


@pytest.mark.slow
def test_long_context_workload():
    _check(synth.WORKLOADS["long_s128k"], n_uniform=6)


def test_indexer_loss_full_size():
    """The indexer loss and its gradient at v32_671b_s16k, the step bench.py --indexer-loss times.

    Sampled rows against the oracle (its own scores and selection); dk_idx, which gathers every
    row, through an identity that holds at any size: I is positively homogeneous of degree 1 in
    q_idx and in k_idx, so sum_s <dk_s, k_s> = sum_{t,h} <dq_th, q_th> = sum_{t,h} w dw
    = sum_{t,j} dI_tj I[t, s_tj]."""
    import sparse_attention_index_gb300 as dsa
    wl = synth.WORKLOADS["v32_671b_s16k"]
    ind = synth.indexer_inputs(wl)
    att = synth.attention_inputs(wl, with_grad=False)
    S, k, g = wl.S, wl.topk, 1.0 / wl.S
    qd, kd, wd = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"])
    Qd, Kd, Vd = bf16_dev(att["Q"]), bf16_dev(att["K"]), bf16_dev(att["V"])
    scores = dsa.dsa_index_scores(qd, kd, wd)
    idx, _ = dsa.dsa_topk(scores, k)
    _, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idx, wl.scale)
    kl, dI = dsa.dsa_indexer_loss(Qd, Kd, idx, lse, scores, wl.scale, g)
    dq, dk, dw = dsa.dsa_indexer_loss_bwd(qd, kd, wd, idx, dI)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0

    rows = synth.sample_rows(wl, 8)
    sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], None, rows=rows)
    ref_idx, _ = oracle.topk(sc, None, S, k, rows=rows, B=wl.B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k)[rows], ref_idx)
    full_idx = np.full((wl.B * S, k), -1, dtype=np.int32)
    full_idx[rows] = ref_idx
    full_idx = full_idx.reshape(wl.B, S, k)
    kl_ref, dI_ref = oracle.indexer_loss(att["Q"], att["K"], full_idx, sc, wl.scale, g, rows=rows)
    rt = torch.as_tensor(rows)
    assert rel_err(host_f64(kl.reshape(-1)[rt]), kl_ref) <= 1e-3
    assert rel_err(host_f64(dI.reshape(-1, k)[rt]), dI_ref) <= 1e-3
    dq_ref, _, dw_ref = oracle.indexer_loss_bwd(ind["q_idx"], ind["k_idx"], ind["w"], full_idx,
                                                dI_ref, rows=rows)
    assert rel_err(host_f64(dq.reshape(wl.B * S, wl.Hi, wl.Di)[rt]), dq_ref) <= TOL
    # dw from the GPU's dI (within 1e-3 of the oracle's); its sum over keys can cancel
    assert rel_err(host_f64(dw.reshape(wl.B * S, wl.Hi)[rt]), dw_ref) <= TOL

    sel = idx.long().clamp(min=0)
    I_sel = torch.gather(scores[:, :, :S], 2, sel).double() * (idx >= 0)
    rhs = (dI.double() * I_sel).sum().item()
    via_dk = (dk.double() * kd.double()).sum().item()
    via_dq = (dq.double() * qd.double()).sum().item()
    via_dw = (dw.double() * wd.double()).sum().item()
    assert abs(via_dw - rhs) <= 1e-4 * abs(rhs)
    assert abs(via_dk - rhs) <= 2e-3 * abs(rhs)      # G in bf16 (2^-9) in the dk, dq products
    assert abs(via_dq - rhs) <= 2e-3 * abs(rhs)


@pytest.mark.slow
def test_index_topk_stream_long_context():
    """The streaming form (no score rows) at the long-context shape S = 131072: every row equal
    to the memory form's (block-fused indexer + top-k), and sampled rows (t = 0, k-1, k, S-1
    and uniform draws) equal to the oracle's top-k of the oracle's scores."""
    import sparse_attention_index_gb300 as dsa
    wl = synth.WORKLOADS["long_s128k"]
    ind = synth.indexer_inputs(wl)
    qd, kd, wd = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"])
    S, k = wl.S, wl.topk
    idx_s, cnt_s = dsa.dsa_index_topk_stream(qd, kd, wd, k)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    idx_m, cnt_m = dsa.dsa_index_topk(qd, kd, wd, k, block_rows=8192)
    torch.cuda.synchronize()
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(idx_s, idx_m) and torch.equal(cnt_s, cnt_m)
    del idx_m, cnt_m
    rows = synth.sample_rows(wl, 6)
    sc = oracle.index_scores(ind["q_idx"], ind["k_idx"], ind["w"], None, rows=rows)
    ref_idx, ref_cnt = oracle.topk(sc, None, S, k, rows=rows, B=wl.B)
    assert np.array_equal(idx_s.cpu().numpy().reshape(-1, k)[rows], ref_idx)
    assert np.array_equal(cnt_s.cpu().numpy().reshape(-1)[rows], ref_cnt)
