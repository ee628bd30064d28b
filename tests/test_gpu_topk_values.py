"""The top-k's selected scores (`vals`): each slot of idx with the score of its key and -inf
at slots without a key, from the unfused top-k (short rows, k > 2048, long rows), the fused
memory form and the streaming form; and the indexer loss reading them slot by slot
(ld_scores = 0) instead of gathering them from the score rows."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import bf16_dev, dev, host_f64, rel_err
from test_gpu_parity import INDEXER_CASES, _check_topk, _dsa, _fp8_inputs, _indexer_case, _run_scores

pytestmark = pytest.mark.gpu


def _expected_vals(idx, rows_scores):
    """vals of rows: the row's score at each selected key, -inf where idx is -1."""
    idx = np.asarray(idx)
    safe = np.where(idx >= 0, idx, 0)
    got = np.take_along_axis(np.asarray(rows_scores, dtype=np.float32), safe, axis=1)
    return np.where(idx >= 0, got, np.float32(-np.inf)).astype(np.float32)


def _check_vals(idx_gpu, vals_gpu, rows_scores, rows):
    """vals_gpu / idx_gpu flattened to [B*S, k]; rows_scores[r] is the score row of rows[r]."""
    k = idx_gpu.shape[-1]
    idx = idx_gpu.reshape(-1, k)[rows]
    vals = vals_gpu.reshape(-1, k)[rows]
    exp = _expected_vals(idx, rows_scores)
    assert np.array_equal(np.isneginf(vals), idx < 0)
    bad = np.argwhere(vals != exp)
    assert bad.size == 0, (bad[:5], vals[tuple(bad[0])], exp[tuple(bad[0])])


@pytest.mark.parametrize("case", INDEXER_CASES[:5])
@pytest.mark.parametrize("k", [37, 300])
def test_topk_values_short_rows(case, k):
    """Staged rows, with and without documents, rows with at most k keys among them."""
    dsa = _dsa()
    B, S, Hi, Di, ndocs, w_kind = case
    inp = _indexer_case(B, S, Hi, Di, seed=900 + S, ndocs=ndocs, w_kind=w_kind)
    sc = _run_scores(inp)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    idx, cnt, vals = dsa.dsa_topk(sc, k, seg, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.arange(B * S)
    sc32 = sc[:, :, :S].cpu().numpy().reshape(B * S, S)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc32.astype(np.float64), inp["seg"], S, k,
                rows)
    _check_vals(idx.cpu().numpy(), vals.cpu().numpy(), sc32, rows)


@pytest.mark.parametrize("ndocs", [0, 3])
def test_topk_values_wide_k(ndocs):
    """k = 3000 > 2048: the short-row kernel writes the slots straight to global memory."""
    dsa = _dsa()
    B, S, k = 1, 5000, 3000
    rng = np.random.default_rng(31 + ndocs)
    sc = rng.standard_normal((B, S, S), dtype=np.float32)
    seg = synth.segments(B, S, ndocs, 5) if ndocs else None
    idx, cnt, vals = dsa.dsa_topk(dev(sc), k, None if seg is None else dev(seg), vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    rows = np.array([0, 2999, 3000, 3001, 4500, S - 1], dtype=np.int64)
    _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc[0][rows].astype(np.float64), seg, S, k,
                rows)
    _check_vals(idx.cpu().numpy(), vals.cpu().numpy(), sc[0][rows], rows)


def test_topk_values_long_rows():
    """Rows past the shared stage (the long-row kernel), with packed documents and rows
    whose document is shorter than k."""
    dsa = _dsa()
    S, k = 20000, 300
    rng = np.random.default_rng(13)
    sc = rng.standard_normal((1, S, S), dtype=np.float32)
    seg = np.zeros((1, S), dtype=np.int32)
    seg[0, 9000:] = 1
    seg[0, 19800:] = 2
    for sg in (None, seg):
        idx, cnt, vals = dsa.dsa_topk(dev(sc), k, None if sg is None else dev(sg), vals=True)
        assert dsa.dsa_get_last_device_error() == 0
        rows = np.array([100, 16383, 16384, 16385, 19799, 19800, 19850, S - 1], dtype=np.int64)
        _check_topk(idx.cpu().numpy(), cnt.cpu().numpy(), sc[0][rows].astype(np.float64), sg,
                    S, k, rows)
        _check_vals(idx.cpu().numpy(), vals.cpu().numpy(), sc[0][rows], rows)


def test_index_topk_values_match_unfused_path():
    """The memory form's vals equal the unfused top-k's on the same scores, bit for bit,
    across blocks and the 16384-key boundary."""
    dsa = _dsa()
    for B, S, Hi, Di, k, ndocs, R in ((2, 1500, 4, 32, 200, 3, 256),
                                      (1, 17000, 64, 128, 2048, 0, 4096)):
        inp = _indexer_case(B, S, Hi, Di, seed=950 + S, ndocs=ndocs)
        q, kk, w = bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), dev(inp["w"])
        seg = None if inp["seg"] is None else dev(inp["seg"])
        idx_f, cnt_f, vals_f = dsa.dsa_index_topk(q, kk, w, k, seg, block_rows=R, vals=True)
        scores = dsa.dsa_index_scores(q, kk, w, seg)
        idx_u, cnt_u, vals_u = dsa.dsa_topk(scores, k, seg, vals=True)
        assert dsa.dsa_get_last_device_error() == 0
        assert torch.equal(idx_f, idx_u) and torch.equal(cnt_f, cnt_u)
        assert torch.equal(vals_f, vals_u)
        del scores


@pytest.mark.parametrize("case", [
    # B, S, Hi, Di, k, ndocs, block_rows
    (1, 128, 4, 32, 4, 0, 256),
    (2, 3000, 64, 128, 300, 0, 512),
    (2, 2000, 16, 64, 100, 3, 512),
    (1, 489, 64, 128, 512, 3, 256),    # every row has at most k keys
])
def test_index_topk_stream_values_match_oracle(case):
    """The streaming form's vals (the keys >= U carry theirs from the emit pass, the window
    keys from the window list) against the oracle's scores at the oracle's selection."""
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs, R = case
    inp = _indexer_case(B, S, Hi, Di, seed=830 + S + Hi, ndocs=ndocs)
    seg = None if inp["seg"] is None else dev(inp["seg"])
    idx, cnt, vals = dsa.dsa_index_topk_stream(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]),
                                               dev(inp["w"]), k, seg, block_rows=R, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"])
    ref_idx, ref_cnt = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    assert np.array_equal(cnt.cpu().numpy().reshape(-1), ref_cnt)
    rows = np.arange(B * S)
    _check_vals(idx.cpu().numpy(), vals.cpu().numpy(), sc.reshape(B * S, S).astype(np.float32),
                rows)


def test_index_topk_stream_values_match_unfused_path_at_v32_shape():
    dsa = _dsa()
    wl = synth.WORKLOADS["v32_671b_s16k"].replace(S=6000)
    ind = synth.indexer_inputs(wl)
    q, kk, w = bf16_dev(ind["q_idx"]), bf16_dev(ind["k_idx"]), dev(ind["w"])
    idx_s, cnt_s, vals_s = dsa.dsa_index_topk_stream(q, kk, w, wl.topk, vals=True)
    idx_u, cnt_u, vals_u = dsa.dsa_topk(dsa.dsa_index_scores(q, kk, w), wl.topk, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(idx_s, idx_u) and torch.equal(cnt_s, cnt_u)
    assert torch.equal(vals_s, vals_u)


def test_index_topk_stream_values_rows_left_to_the_memory_form():
    """All scores tied (each is 64 * 0.0625 * 128 * 0.125^2 = 8): rows past 4096 keys
    overflow the window list and their block goes through the memory form."""
    dsa = _dsa()
    B, S, Hi, Di, k = 1, 6000, 64, 128, 100
    one = torch.full((B, S, Hi, Di), 0.125, dtype=torch.bfloat16, device="cuda")
    kk = torch.full((B, S, Di), 0.125, dtype=torch.bfloat16, device="cuda")
    w = torch.full((B, S, Hi), 0.0625, dtype=torch.float32, device="cuda")
    idx, cnt, vals = dsa.dsa_index_topk_stream(one, kk, w, k, block_rows=2048, vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    t = np.arange(S)
    sel = np.arange(k)[None, :] <= t[:, None]
    ref = np.where(sel, np.float32(8.0), np.float32(-np.inf))
    assert np.array_equal(vals.cpu().numpy().reshape(S, k), ref)


def test_index_topk_stream_fp8_values_match_oracle():
    dsa = _dsa()
    B, S, Hi, Di, k, ndocs = 1, 2600, 64, 128, 256, 2
    _, inp = _fp8_inputs(B, S, Hi, Di, ndocs, "pow2", seed=871)
    idx, cnt, vals = dsa.dsa_index_topk_stream(dev(inp["q_idx"]), dev(inp["k_idx"]),
                                               dev(inp["w"]), k, dev(inp["seg"]), block_rows=512,
                                               k_scale=dev(inp["k_scale"]), vals=True)
    assert dsa.dsa_get_last_device_error() == 0
    sc = oracle.index_scores_fp8(inp["q_idx"], inp["k_idx"], inp["w"], inp["seg"], inp["k_scale"])
    ref_idx, _ = oracle.topk(sc, inp["seg"], S, k, B=B)
    assert np.array_equal(idx.cpu().numpy().reshape(-1, k), ref_idx)
    _check_vals(idx.cpu().numpy(), vals.cpu().numpy(), sc.reshape(B * S, S).astype(np.float32),
                np.arange(B * S))


@pytest.mark.parametrize("H, Hkv", [(128, 1), (8, 2)])   # the tensor-core and CUDA-core kernels
def test_indexer_loss_reads_selected_scores_by_slot(H, Hkv):
    """dsa_indexer_loss on the top-k's vals (ld_scores = 0) gives the same dI, bit for bit,
    as on the score rows, and the same loss up to the order of its atomic sum."""
    dsa = _dsa()
    B, S, Dqk, k, seed = 1, 700, 128, 256, 41
    Q = synth.normal_bf16((B, S, H, Dqk), seed, synth.STREAM_Q)
    K = synth.normal_bf16((B, S, Hkv, Dqk), seed, synth.STREAM_K)
    V = synth.normal_bf16((B, S, Hkv, 128), seed, synth.STREAM_V)
    inp = _indexer_case(B, S, 64, 128, seed=seed, ndocs=2)
    seg = dev(inp["seg"])
    scores = dsa.dsa_index_scores(bf16_dev(inp["q_idx"]), bf16_dev(inp["k_idx"]), dev(inp["w"]),
                                  seg)
    idx, _, vals = dsa.dsa_topk(scores, k, seg, vals=True)
    Qd, Kd, Vd = bf16_dev(Q), bf16_dev(K), bf16_dev(V)
    scale = Dqk ** -0.5
    _, lse = dsa.dsa_sparse_attn_fwd(Qd, Kd, Vd, idx, scale)
    kl_a, dI_a = dsa.dsa_indexer_loss(Qd, Kd, idx, lse, scores, scale, 0.5)
    kl_b, dI_b = dsa.dsa_indexer_loss(Qd, Kd, idx, lse, None, scale, 0.5, sel_scores=vals)
    assert dsa.dsa_get_last_device_error() == 0
    assert torch.equal(dI_a, dI_b)
    assert rel_err(host_f64(kl_b), host_f64(kl_a)) <= 1e-6
